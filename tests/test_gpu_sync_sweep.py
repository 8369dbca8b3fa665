"""Synchronisation sweep over random shapes.

The fused engine hands H from layer-1 to layer-2 tiles inside one launch:
per-tile ready flags, per-band tallies, tasks claimed one ahead and handed to
the peer CTA ("Kernel fusion and tensor parallelism", section "Step 1": a
tile of H feeds its row of W2 as soon as it is ready).  The two-launch path
computes the same tiles with the same arithmetic and no hand-over inside a
launch (the kernel boundary orders the layers), so the two must agree bit
for bit; a layer-2 tile that read H too early would differ.  Each call runs
on a caller workspace whose data region is refilled with 0xFF bytes (NaN as
bf16) before it, so stale bytes cannot pass for the right ones.  The MoE form
is swept the same way, its combine fused into the layer-2 epilogue against
the separate combine kernel (bit-equal by construction: both sum a token's
expert rows in slot order).  Shapes, activations and routers come from a
fixed seed; the sizes span one to twelve row bands and several raster groups.
"""
import random

import pytest
import torch

from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

SYNC_BYTES = 5 << 20   # control block, flags and counters: initialised by the library, not poisoned
ACTS = ["none", "relu", "gelu_tanh", "silu"]


def _dense_cases():
    rnd = random.Random(20240611)
    cases = []
    for _ in range(16):
        M = rnd.choice([rnd.randint(1, 300), rnd.randint(257, 1300), rnd.randint(1000, 3000)])
        N = 8 * rnd.randint(1, 160)
        O = 8 * rnd.randint(1, 320)
        P = 8 * rnd.randint(1, 160)
        cases.append((M, N, O, P, rnd.choice(ACTS), rnd.choice(ACTS)))
    return cases


def _moe_cases():
    rnd = random.Random(777)
    cases = []
    for _ in range(6):
        E = rnd.choice([1, 2, 4, 8, 16])
        cases.append((rnd.randint(1, 4000), E, rnd.randint(1, min(4, E)), 8 * rnd.randint(2, 64),
                      8 * rnd.randint(2, 128), 8 * rnd.randint(2, 64)))
    return cases


def _equal_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.fixture
def lib(cuda_lib):
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 0)
    yield cuda_lib
    cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.set_workspace(None)


def test_fused_equals_two_launches_on_random_shapes(lib):
    for i, (M, N, O, P, a1, a2) in enumerate(_dense_cases()):
        inp = synth.ffn_inputs(M, N, O, P, seed=i, device="cuda")
        results = {}
        for path in (1, 3):
            lib.set_option(lib.OPT_PATH, path)
            need = lib.workspace_bytes(M, N, O, P)
            buf = torch.full(((need + 255) // 256 * 256,), 0xFF, dtype=torch.uint8, device="cuda")
            lib.set_workspace(buf)
            ys = []
            for _ in range(2):
                if need > SYNC_BYTES:
                    buf[SYNC_BYTES:].fill_(0xFF)
                Y = lib.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, a1, a2)
                lib.check()
                ys.append(Y.clone())
            lib.set_workspace(None)
            results[path] = ys
        ref = results[3][0]
        assert torch.isfinite(ref.float()).all(), (M, N, O, P, a1, a2)
        for path, ys in results.items():
            for rep, y in enumerate(ys):
                assert _equal_bits(y, ref), f"{(M, N, O, P, a1, a2)}: path {path}, call {rep} differs"


def test_moe_fused_combine_equals_kernel_on_random_shapes(cuda_lib):
    for i, (T, E, k, N, O, P) in enumerate(_moe_cases()):
        inp = synth.moe_inputs(T, N, O, P, E, seed=100 + i, device="cuda")
        ys = {}
        for fused in (1, 0):
            old = cuda_lib.set_option(cuda_lib.OPT_MOE_COMBINE, fused)
            try:
                y = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                             "gelu_tanh", "none")
                cuda_lib.check()
                ys[fused] = y.clone()
            finally:
                cuda_lib.set_option(cuda_lib.OPT_MOE_COMBINE, old)
        assert torch.isfinite(ys[1].float()).all(), (T, E, k, N, O, P)
        assert _equal_bits(ys[0], ys[1]), f"MoE {(T, E, k, N, O, P)}: fused combine differs"
