"""Parity of the tensor-core weight stream (TFFN_OPT_PATH = 6: up to 256 rows;
the weights as the MMA's M side) with the CPU oracle, through the
C ABI: |y - y_ref| <= 1e-2 + 1e-2 |y_ref| elementwise.  Small shapes in full
(several slices, split-K parts and ragged tails; layer 1 as per-CTA windows
and, for hidden widths past two blocks per CTA, as split slices), the Llama 3
8B shapes on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

PATH = 6
ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
       "silu": oracle.ACT_SILU}


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bound = 1e-2 + 1e-2 * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def _with_path(tffn, path, fn):
    old = tffn.set_option(tffn.OPT_PATH, path)
    try:
        out = fn()
        tffn.check()
    finally:
        tffn.set_option(tffn.OPT_PATH, old)
    return out


def _dense(tffn, inp, act1, act2, path=PATH):
    return _with_path(tffn, path, lambda: tffn.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, act1, act2))


def _dense_oracle(inp, act1, act2, rows=None):
    u = synth.to_u16
    return oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), ACT[act1], ACT[act2], rows=rows)


def _glu(tffn, g, act, path=PATH):
    return _with_path(tffn, path, lambda: tffn.ffn_glu_forward(g.X, g.W1, g.W3, g.W2, act))


def _glu_oracle(g, act, rows=None):
    u = synth.to_u16
    return oracle.glu_ffn(u(g.X), u(g.W1), u(g.W3), u(g.W2), ACT[act], rows=rows)


@pytest.mark.parametrize("shape,acts", [
    ((128, 512, 1024, 256), ("gelu_tanh", "none")),     # 128-row instance, split-K in both layers
    ((65, 136, 520, 264), ("relu", "gelu_tanh")),       # one row past the mma.sync path; ragged N, O, P
    ((100, 4096, 1024, 256), ("gelu_tanh", "none")),    # N > O: long layer-1 ranges
    ((129, 256, 384, 136), ("gelu_tanh", "relu")),      # 256-row instance, one row past 128
    ((256, 1024, 2048, 512), ("relu", "none")),         # full 256 rows
    ((200, 64, 128, 64), ("none", "none")),             # one K chunk, one slice per layer
    ((1, 256, 264, 72), ("gelu_tanh", "none")),         # a single row through the 32-row instance
    ((16, 512, 1024, 256), ("relu", "none")),           # decode-sized batch, 32-row instance
    ((48, 136, 520, 264), ("gelu_tanh", "relu")),       # 64-row instance, ragged
    ((32, 4096, 1024, 256), ("gelu_tanh", "none")),     # N > O at 32 rows
])
def test_stream_dense_full(cuda_lib, shape, acts):
    M, N, O, P = shape
    inp = synth.ffn_inputs(M, N, O, P, seed=31 + sum(shape), device="cuda")
    Y = _dense(cuda_lib, inp, *acts)
    _assert_close(Y.float().cpu().numpy(), _dense_oracle(inp, *acts), f"stream {shape}")


@pytest.mark.parametrize("shape,glu", [
    ((64, 512, 20480, 512), False),     # 320 hidden blocks, 2-3 per CTA: four-block windows (two tiles)
    ((48, 256, 40960, 264), False),     # 640 blocks, more than 4 per CTA: Stream-K layer 1, ragged P
    ((100, 256, 20480, 264), True),     # gated past 2 blocks per CTA: Stream-K layer 1, ragged P
])
def test_stream_wide_hidden(cuda_lib, shape, glu):
    M, N, O, P = shape
    if glu:
        g = synth.glu_inputs(M, N, O, P, seed=M + 3, device="cuda")
        Y = _glu(cuda_lib, g, "silu")
        _assert_close(Y.float().cpu().numpy(), _glu_oracle(g, "silu"), f"wide hidden glu {shape}")
    else:
        inp = synth.ffn_inputs(M, N, O, P, seed=M + 5, device="cuda")
        Y = _dense(cuda_lib, inp, "gelu_tanh", "none")
        _assert_close(Y.float().cpu().numpy(), _dense_oracle(inp, "gelu_tanh", "none"), f"wide hidden {shape}")


@pytest.mark.parametrize("M,glu", [(200, False), (160, True)])
def test_stream_is_the_default_to_256_rows(cuda_lib, M, glu):
    # 129-256 rows take the stream automatically while its window layer 1
    # applies; the result matches the oracle and the forced stream bit for bit
    N, O, P = 512, 2048, 512
    if glu:
        g = synth.glu_inputs(M, N, O, P, seed=9, device="cuda")
        auto = _glu(cuda_lib, g, "silu", path=0)
        forced = _glu(cuda_lib, g, "silu")
        _assert_close(auto.float().cpu().numpy(), _glu_oracle(g, "silu"), "auto glu")
    else:
        inp = synth.ffn_inputs(M, N, O, P, seed=9, device="cuda")
        auto = _dense(cuda_lib, inp, "gelu_tanh", "none", path=0)
        forced = _dense(cuda_lib, inp, "gelu_tanh", "none")
        _assert_close(auto.float().cpu().numpy(), _dense_oracle(inp, "gelu_tanh", "none"), "auto dense")
    assert torch.equal(auto, forced)


def test_stream_dense_no_bias(cuda_lib):
    inp = synth.ffn_inputs(96, 256, 640, 192, seed=8, device="cuda")
    Y = _with_path(cuda_lib, PATH, lambda: cuda_lib.ffn_forward(inp.X, inp.W1, None, inp.W2, None, "gelu_tanh"))
    u = synth.to_u16
    want = oracle.ffn(u(inp.X), u(inp.W1), None, u(inp.W2), None, oracle.ACT_GELU_TANH, oracle.ACT_NONE)
    _assert_close(Y.float().cpu().numpy(), want, "stream no bias")


@pytest.mark.parametrize("M,N,O,P,act", [
    (128, 512, 1024, 256, "silu"),       # SwiGLU, split-K in both layers
    (72, 136, 328, 200, "gelu_tanh"),    # GeGLU, ragged everything
    (100, 2048, 256, 512, "silu"),       # N > O
    (65, 64, 128, 64, "relu"),           # ReGLU, one slice
    (200, 256, 640, 392, "silu"),        # 256-row instance (one accumulator buffer), ragged P
    (16, 512, 1024, 256, "silu"),        # 32-row instance
    (40, 136, 328, 200, "gelu_tanh"),    # 64-row instance, ragged
])
def test_stream_glu_full(cuda_lib, M, N, O, P, act):
    g = synth.glu_inputs(M, N, O, P, seed=M + N, device="cuda")
    Y = _glu(cuda_lib, g, act)
    _assert_close(Y.float().cpu().numpy(), _glu_oracle(g, act), f"stream glu {act}")


def test_stream_deterministic_and_close_to_engine(cuda_lib):
    inp = synth.ffn_inputs(160, 512, 2048, 512, seed=12, device="cuda")
    a = _dense(cuda_lib, inp, "gelu_tanh", "relu")
    b = _dense(cuda_lib, inp, "gelu_tanh", "relu")
    assert torch.equal(a, b)
    e = _dense(cuda_lib, inp, "gelu_tanh", "relu", path=1)
    _assert_close(a.float().cpu().numpy(), e.float().cpu().numpy(), "stream vs engine")


def test_stream_rows_past_its_limit_run_the_engine(cuda_lib):
    # 257 rows are past the stream's instances: the option falls back to the
    # engine, which still gives the oracle's result
    inp = synth.ffn_inputs(257, 64, 256, 64, seed=4, device="cuda")
    Y = _dense(cuda_lib, inp, "relu", "none")
    _assert_close(Y.float().cpu().numpy(), _dense_oracle(inp, "relu", "none"), "257 rows")
    g = synth.glu_inputs(257, 64, 256, 64, seed=5, device="cuda")
    Y = _glu(cuda_lib, g, "silu")
    _assert_close(Y.float().cpu().numpy(), _glu_oracle(g, "silu"), "257 gated rows")


@pytest.mark.parametrize("M", [128, 256])
def test_stream_llama3_8b_all_rows(cuda_lib, M):
    # batched decode of the Llama 3 8B FFN shape (dense form, GELU)
    N, O, P = 4096, 14336, 4096
    inp = synth.ffn_inputs(M, N, O, P, seed=0, device="cuda")
    Y = _dense(cuda_lib, inp, "gelu_tanh", "none")
    u = synth.to_u16
    host = (u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2))
    want = parity.oracle_rows(
        lambda r: oracle.ffn(*host, oracle.ACT_GELU_TANH, oracle.ACT_NONE, rows=r), range(M))
    parity.assert_close(Y.float().cpu().numpy(), want, f"8B M={M}")


@pytest.mark.parametrize("M", [128, 256])
def test_stream_swiglu_llama3_8b_all_rows(cuda_lib, M):
    N, O, P = 4096, 14336, 4096
    g = synth.glu_inputs(M, N, O, P, seed=0, device="cuda")
    Y = _glu(cuda_lib, g, "silu")
    u = synth.to_u16
    host = (u(g.X), u(g.W1), u(g.W3), u(g.W2))
    want = parity.oracle_rows(lambda r: oracle.glu_ffn(*host, oracle.ACT_SILU, rows=r), range(M))
    parity.assert_close(Y.float().cpu().numpy(), want, f"SwiGLU 8B M={M}")
