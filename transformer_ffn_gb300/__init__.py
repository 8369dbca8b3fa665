"""GB300-native fused Transformer FFN and MoE-FFN (placeholder until the binding lands)."""
