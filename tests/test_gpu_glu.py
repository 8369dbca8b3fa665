"""Parity of ffn_glu_forward (the gated FFN, SwiGLU with act = SiLU) through
the C ABI with the CPU oracle: |y - y_ref| <= 1e-2 + 1e-2 |y_ref|."""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
       "silu": oracle.ACT_SILU}


def _inputs(M, N, O, P, seed):
    g = synth.glu_inputs(M, N, O, P, seed=seed, device="cuda")
    return g.X, g.W1, g.W3, g.W2


def _oracle(X, W1, W3, W2, act, rows=None):
    u = synth.to_u16
    return oracle.glu_ffn(u(X), u(W1), u(W3), u(W2), ACT[act], rows=rows)


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bad = err > 1e-2 + 1e-2 * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"


@pytest.mark.parametrize("M,N,O,P,act", [
    (64, 256, 1024, 256, "silu"),        # several layer-1 tiles, one band
    (300, 136, 328, 200, "silu"),        # ragged rows, hidden tail of 72 columns, no 3-D maps
    (513, 64, 384, 64, "gelu_tanh"),     # three bands, GeGLU
    (200, 128, 256, 128, "relu"),        # ReGLU
    (96, 64, 128, 64, "none"),           # bilinear
    (16, 512, 640, 256, "silu"),         # decode-sized batch (engine path)
    (64, 2048, 256, 256, "silu"),        # N > O: more layer-1 k-blocks than H tiles
])
def test_glu_small_full(cuda_lib, M, N, O, P, act):
    X, W1, W3, W2 = _inputs(M, N, O, P, seed=M + O)
    Y = cuda_lib.ffn_glu_forward(X, W1, W3, W2, act)
    cuda_lib.check()
    _assert_close(Y.float().cpu().numpy(), _oracle(X, W1, W3, W2, act), f"glu {act}")


def test_glu_fused_equals_two_launches_and_is_deterministic(cuda_lib):
    X, W1, W3, W2 = _inputs(700, 256, 1152, 320, seed=3)
    a = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
    b = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 3)
    try:
        c = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
        assert cuda_lib.last_launch_count() == 2
    finally:
        cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.check()
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
def test_glu_with_unit_linear_branch_equals_dense_ffn(cuda_lib, act):
    # X W3 == 1 exactly (a column of ones selected by W3): the gated FFN is the
    # dense FFN without biases, and the two GPU paths agree bit for bit
    M, N, O, P = 300, 128, 512, 192
    X, W1, _, W2 = _inputs(M, N, O, P, seed=8)
    X = X.clone()
    X[:, 5] = 1.0
    W3 = torch.zeros((N, O), dtype=torch.bfloat16, device="cuda")
    W3[5, :] = 1.0
    g = cuda_lib.ffn_glu_forward(X, W1, W3, W2, act)
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 1)
    try:
        d = cuda_lib.ffn_forward(X, W1, None, W2, None, act, "none")
    finally:
        cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.check()
    assert torch.equal(g, d)


def test_glu_empty_and_validation(cuda_lib):
    X, W1, W3, W2 = _inputs(8, 64, 128, 64, seed=1)
    assert cuda_lib.ffn_glu_forward(X[:0], W1, W3, W2, "silu").shape == (0, 64)
    with pytest.raises(Exception):
        cuda_lib.ffn_glu_forward(X, W1, W3[:, :64].contiguous(), W2, "silu")


def test_glu_full_size_sampled_rows(cuda_lib):
    # the Llama 3 8B FFN shape: M 4096, N 4096, O 14336, P 4096, SwiGLU
    M, N, O, P = 4096, 4096, 14336, 4096
    X, W1, W3, W2 = _inputs(M, N, O, P, seed=0)
    Y = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
    cuda_lib.check()
    assert torch.isfinite(Y.float()).all()
    # every 256-row band (both CTAs of the pair tile, the band edges) and so
    # every raster group
    rows = parity.band_rows(M)
    u = synth.to_u16
    host = (u(X), u(W1), u(W3), u(W2))
    want = parity.oracle_rows(lambda r: oracle.glu_ffn(*host, oracle.ACT_SILU, rows=r), rows)
    parity.assert_close(Y[rows].float().cpu().numpy(), want, "glu full size")


def test_dense_ffn_with_silu_on_both_paths(cuda_lib):
    # SiLU as the dense FFN's activation, on the weight-streaming path (M <= 64)
    # and on the engine
    for M in (16, 200):
        inp = synth.ffn_inputs(M, 256, 512, 128, seed=M, device="cuda")
        Y = cuda_lib.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "silu", "silu")
        cuda_lib.check()
        u = synth.to_u16
        want = oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), oracle.ACT_SILU,
                          oracle.ACT_SILU)
        _assert_close(Y.float().cpu().numpy(), want, f"silu M={M}")


# ------------------------------------------------ weight-streaming path, M <= 64

@pytest.mark.parametrize("M,N,O,P,act", [
    (1, 256, 384, 136, "silu"),
    (5, 136, 200, 264, "silu"),          # hidden tail: 200 = 3 x 64 + 8
    (16, 2048, 136, 4096, "gelu_tanh"),  # N > O, narrow hidden
    (32, 1024, 2048, 512, "silu"),       # two 16-row tiles
    (8, 4096, 8192, 1024, "relu"),       # long split-K ranges
    (64, 1024, 2048, 512, "silu"),       # the 64-row instance
    (8, 512, 20480, 256, "silu"),        # 320 hidden blocks, more than two per CTA: split layer 1, no window
])
def test_glu_decode_path_full(cuda_lib, M, N, O, P, act):
    X, W1, W3, W2 = _inputs(M, N, O, P, seed=3 * M + O)
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 2)
    try:
        Y = cuda_lib.ffn_glu_forward(X, W1, W3, W2, act)
        assert cuda_lib.last_launch_count() == 1
    finally:
        cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.check()
    _assert_close(Y.float().cpu().numpy(), _oracle(X, W1, W3, W2, act), f"glu decode {act}")


def test_glu_decode_deterministic_and_close_to_engine(cuda_lib):
    X, W1, W3, W2 = _inputs(24, 1024, 3072, 1024, seed=12)
    a = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")      # auto: the weight stream at M <= 64
    b = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 1)
    try:
        e = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
    finally:
        cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.check()
    assert torch.equal(a, b)
    d = (a.float() - e.float()).abs()
    assert torch.all(d <= 2e-2 + 2e-2 * e.float().abs())


def test_glu_decode_llama3_8b_full(cuda_lib):
    # decode step of the Llama 3 8B SwiGLU FFN: M 16, N 4096, O 14336, P 4096
    X, W1, W3, W2 = _inputs(16, 4096, 14336, 4096, seed=0)
    Y = cuda_lib.ffn_glu_forward(X, W1, W3, W2, "silu")
    cuda_lib.check()
    _assert_close(Y.float().cpu().numpy(), _oracle(X, W1, W3, W2, "silu"), "glu decode 8B")
