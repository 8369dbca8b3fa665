"""Parity of moe_glu_forward (gated experts, SwiGLU with act = SiLU) through
the C ABI with the CPU oracle: routing bit-exact, outputs within
|y - y_ref| <= 1e-2 + 1e-2 |y_ref|."""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
       "silu": oracle.ACT_SILU}


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bad = err > 1e-2 + 1e-2 * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"


def _oracle(inp, k, act, tokens=None):
    u = synth.to_u16
    return oracle.moe_glu_ffn(u(inp.X), inp.logits.cpu().numpy(), k, [u(w) for w in inp.W1],
                              [u(w) for w in inp.W3], [u(w) for w in inp.W2], ACT[act], tokens=tokens)


@pytest.mark.parametrize("T,N,O,P,E,k,act,router", [
    (300, 64, 256, 128, 8, 2, "silu", "balanced"),
    (129, 128, 328, 200, 4, 1, "gelu_tanh", "moderate"),   # hidden tail of 72 columns, 2-D maps
    (400, 256, 512, 256, 8, 2, "silu", "stress"),
    (64, 64, 128, 64, 4, 4, "relu", "balanced"),            # top_k = E
    (200, 1024, 256, 128, 4, 2, "silu", "balanced"),        # N > O
])
def test_moe_glu_small_full(cuda_lib, T, N, O, P, E, k, act, router):
    inp = synth.moe_glu_inputs(T, N, O, P, E, seed=T + E, device="cuda", router=router)
    Y, r = cuda_lib.moe_glu_forward(inp.X, inp.logits, k, inp.W1, inp.W3, inp.W2, act, routing=True)
    cuda_lib.check()
    idx, _ = oracle.moe_route(inp.logits.cpu().numpy(), k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), idx)
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, k, act), f"moe glu {router}")


def test_moe_glu_single_expert_equals_dense_gated_ffn(cuda_lib):
    T, N, O, P = 300, 128, 512, 192
    inp = synth.moe_glu_inputs(T, N, O, P, 1, seed=2, device="cuda")
    Y = cuda_lib.moe_glu_forward(inp.X, inp.logits, 1, inp.W1, inp.W3, inp.W2, "silu")
    D = cuda_lib.ffn_glu_forward(inp.X, inp.W1[0], inp.W3[0], inp.W2[0], "silu")
    cuda_lib.check()
    # the grouped engine keeps expert outputs in fp32 and rounds once after the
    # gate weight (1.0 here); the dense engine rounds its fp32 output once
    assert torch.equal(Y, D)


def test_moe_glu_full_size_sampled_tokens(cuda_lib):
    # Mixtral-class expert layer: T 8192, N 4096, 8 experts of O 14336, P 4096, top-2, SwiGLU
    T, N, O, P, E, k = 8192, 4096, 14336, 4096, 8, 2
    inp = synth.moe_glu_inputs(T, N, O, P, E, seed=0, device="cuda")
    Y, r = cuda_lib.moe_glu_forward(inp.X, inp.logits, k, inp.W1, inp.W3, inp.W2, "silu", routing=True)
    cuda_lib.check()
    assert torch.isfinite(Y.float()).all()
    # tokens in every expert's zero-padded last band, plus random ones
    tail = parity.moe_tail_tokens(r["perm"].cpu().numpy(), r["expert_offsets"].cpu().numpy(), k)
    tokens = parity.with_random(set([0, T - 1] + tail), T, 64, seed=3)
    u = synth.to_u16
    host = (u(inp.X), inp.logits.cpu().numpy(), [u(w) for w in inp.W1], [u(w) for w in inp.W3],
            [u(w) for w in inp.W2])
    want = parity.oracle_rows(lambda t: oracle.moe_glu_ffn(*host[:2], k, *host[2:], oracle.ACT_SILU, tokens=t),
                              tokens)
    parity.assert_close(Y[tokens].float().cpu().numpy(), want, "moe glu full size")
