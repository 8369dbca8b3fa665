"""The seeded input generators: shapes, dtypes, reproducibility and the
router skew distributions of the MoE workloads (host only)."""
import numpy as np
import pytest
import torch

import oracle
from transformer_ffn_gb300 import synth


def test_ffn_inputs_shapes_and_reproducible():
    a = synth.ffn_inputs(5, 16, 24, 8, seed=3)
    b = synth.ffn_inputs(5, 16, 24, 8, seed=3)
    assert a.X.shape == (5, 16) and a.W1.shape == (16, 24) and a.W2.shape == (24, 8)
    assert a.X.dtype == torch.bfloat16 and a.b2.shape == (8,)
    for x, y in zip((a.X, a.W1, a.b1, a.W2, a.b2), (b.X, b.W1, b.b1, b.W2, b.b2)):
        assert torch.equal(x, y)


def test_router_offsets_keep_the_balanced_draw():
    # the skewed logits are the balanced ones plus a per-expert offset
    bal = synth.moe_inputs(64, 8, 8, 8, 4, seed=5)
    for router in ("moderate", "stress"):
        sk = synth.moe_inputs(64, 8, 8, 8, 4, seed=5, router=router)
        assert torch.equal(sk.X, bal.X)
        assert torch.allclose(sk.logits - bal.logits, synth.router_offsets(4, router).expand(64, 4))
    with pytest.raises(ValueError):
        synth.router_offsets(4, "bogus")


@pytest.mark.parametrize("router", synth.ROUTERS)
def test_router_distributions_have_their_skew(router):
    T, E, k = 8192, 8, 2
    g = torch.Generator().manual_seed(0)
    logits = torch.randn((T, E), generator=g) + synth.router_offsets(E, router)
    idx, _ = oracle.moe_route(logits.numpy(), k)
    share = np.bincount(idx.ravel(), minlength=E) / T     # fraction of tokens per expert
    if router == "balanced":
        assert np.all(np.abs(share - k / E) < 0.03)
    elif router == "moderate":
        assert np.all(np.diff(share) < 0)                    # strictly decreasing popularity
        assert share[0] > 0.6 and share[-1] < 0.1
    else:
        assert share[0] > 0.95
        assert np.all(np.abs(share[1:] - (k - share[0]) / (E - 1)) < 0.03)
