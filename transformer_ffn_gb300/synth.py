"""Seeded synthetic inputs for the FFN and MoE-FFN workloads.

This module draws random tensors and nothing else: it holds none of the FFN's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Distributions (the workloads of the fused-FFN benchmarks: bf16 activations and
weights with the dimensions of Llama/Mixtral-class FFNs):
  X  ~ N(0, 1)               bf16, M x N (row-major)
  W1 ~ N(0, 1/N)             bf16, N x O
  b1 ~ U(-0.1, 0.1)          bf16, O
  W2 ~ N(0, 1/O)             bf16, O x P
  b2 ~ U(-0.1, 0.1)          bf16, P
  W3 ~ N(0, 1/N)             bf16, N x O   (gated FFN only; no biases there)
  gate logits ~ N(0, 1)      fp32, T x E   (MoE only), plus a per-expert
                             offset beta_e that sets the router's skew:
      balanced   beta_e = 0                 (~T*k/E rows per expert)
      moderate   beta_e = -ln(1 + e)        (Zipf-like popularity: E=8, top-2
                                             gives ~36/22/14/9/7/5/4/3 %)
      stress     beta_0 = 3, others 0       (expert 0 is in ~98 % of tokens)
Each tensor is drawn in fp32 from one torch.Generator seeded with ``seed`` in
the fixed order X, W1, b1, W2, b2 (experts in index order), logits, then
rounded to bf16 (round to nearest even).
"""
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def _uniform(shape, lo, hi, g, device):
    t = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(hi - lo).add_(lo)
    return t.to(torch.bfloat16)


@dataclass
class FFNInputs:
    X: torch.Tensor
    W1: torch.Tensor
    b1: torch.Tensor
    W2: torch.Tensor
    b2: torch.Tensor


@dataclass
class GLUInputs:
    X: torch.Tensor
    W1: torch.Tensor
    W3: torch.Tensor
    W2: torch.Tensor


@dataclass
class MoEInputs:
    X: torch.Tensor
    logits: torch.Tensor
    W1: List[torch.Tensor]
    b1: List[torch.Tensor]
    W2: List[torch.Tensor]
    b2: List[torch.Tensor]


def ffn_inputs(M, N, O, P, seed=0, device="cpu", x_std=1.0) -> FFNInputs:
    g = _gen(device, seed)
    X = _normal((M, N), x_std, g, device)
    W1 = _normal((N, O), (1.0 / N) ** 0.5, g, device)
    b1 = _uniform((O,), -0.1, 0.1, g, device)
    W2 = _normal((O, P), (1.0 / O) ** 0.5, g, device)
    b2 = _uniform((P,), -0.1, 0.1, g, device)
    return FFNInputs(X, W1, b1, W2, b2)


def glu_inputs(M, N, O, P, seed=0, device="cpu") -> GLUInputs:
    """Gated FFN operands, drawn in the order X, W1, W3, W2 (no biases); W3 is
    distributed like W1."""
    g = _gen(device, seed)
    X = _normal((M, N), 1.0, g, device)
    W1 = _normal((N, O), (1.0 / N) ** 0.5, g, device)
    W3 = _normal((N, O), (1.0 / N) ** 0.5, g, device)
    W2 = _normal((O, P), (1.0 / O) ** 0.5, g, device)
    return GLUInputs(X, W1, W3, W2)


ROUTERS = ("balanced", "moderate", "stress")


def router_offsets(E, router="balanced") -> torch.Tensor:
    """Per-expert logit offsets beta_e of the named router distribution."""
    if router == "balanced":
        return torch.zeros(E)
    if router == "moderate":
        return -torch.log1p(torch.arange(E, dtype=torch.float32))
    if router == "stress":
        b = torch.zeros(E)
        b[0] = 3.0
        return b
    raise ValueError(f"unknown router distribution {router!r}")


def moe_inputs(T, N, O, P, E, seed=0, device="cpu",
               logits: Optional[torch.Tensor] = None, router="balanced") -> MoEInputs:
    g = _gen(device, seed)
    X = _normal((T, N), 1.0, g, device)
    W1, b1, W2, b2 = [], [], [], []
    for _ in range(E):
        W1.append(_normal((N, O), (1.0 / N) ** 0.5, g, device))
        b1.append(_uniform((O,), -0.1, 0.1, g, device))
        W2.append(_normal((O, P), (1.0 / O) ** 0.5, g, device))
        b2.append(_uniform((P,), -0.1, 0.1, g, device))
    if logits is None:
        logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
        if router != "balanced":
            logits += router_offsets(E, router).to(device)
    return MoEInputs(X, logits, W1, b1, W2, b2)


@dataclass
class MoEGLUInputs:
    X: torch.Tensor
    logits: torch.Tensor
    W1: List[torch.Tensor]
    W3: List[torch.Tensor]
    W2: List[torch.Tensor]


def moe_glu_inputs(T, N, O, P, E, seed=0, device="cpu", router="balanced") -> MoEGLUInputs:
    """Gated-expert MoE operands: X, then W1, W3, W2 of each expert in index
    order (no biases), then the logits (with the router's offsets)."""
    g = _gen(device, seed)
    X = _normal((T, N), 1.0, g, device)
    W1, W3, W2 = [], [], []
    for _ in range(E):
        W1.append(_normal((N, O), (1.0 / N) ** 0.5, g, device))
        W3.append(_normal((N, O), (1.0 / N) ** 0.5, g, device))
        W2.append(_normal((O, P), (1.0 / O) ** 0.5, g, device))
    logits = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if router != "balanced":
        logits += router_offsets(E, router).to(device)
    return MoEGLUInputs(X, logits, W1, W3, W2)


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_u16(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
