"""The allocation-free decode entry point, ffn_forward_decode_noalloc.

For callers that cannot allocate device memory (a host framework that owns
all of HBM, code that must not trigger cudaMalloc's device-wide
synchronisation): the library keeps this entry point's scratch in a static
device array.  Its output must match ffn_forward's on the same inputs, call
after call, since every call reuses (and must re-clear) the same array.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

ORACLE_ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH}


def _entry(tffn):
    L = tffn.load()
    fn = L.ffn_forward_decode_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i64, i64, i64, vp, vp]
    fn.restype = i32
    return fn


def _check_entry(tffn):
    L = tffn.load()
    fn = L.tffn_check_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    fn.restype = ctypes.c_int
    return fn


def _oracle(inp, a1, a2):
    u = synth.to_u16
    return oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), ORACLE_ACT[a1], ORACLE_ACT[a2])


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_matches_ffn_forward_on_consecutive_calls(cuda_lib):
    tffn = cuda_lib
    fn = _entry(tffn)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    shapes = [(16, 1024, 2048, 512, "relu", "none"), (5, 520, 1032, 264, "gelu_tanh", "relu"),
              (32, 256, 384, 136, "gelu_tanh", "none")]
    acts = {"none": 0, "relu": 1, "gelu_tanh": 2}
    for call, (M, N, O, P, a1, a2) in enumerate(shapes + shapes[:1]):
        inp = synth.ffn_inputs(M, N, O, P, seed=100 + call, device="cuda")
        old = tffn.set_option(tffn.OPT_PATH, 2)
        try:
            want = tffn.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, a1, a2)
            tffn.check()
        finally:
            tffn.set_option(tffn.OPT_PATH, old)
        got = torch.full((M, P), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = fn(_p(inp.X), _p(inp.W1), _p(inp.b1), _p(inp.W2), _p(inp.b2), acts[a1], acts[a2],
                M, N, O, P, _p(got), stream)
        assert rc == 0
        torch.cuda.synchronize()
        g = got.float().cpu().numpy()
        w = want.float().cpu().numpy()
        assert np.all(np.abs(g - w) <= 1e-2 + 1e-2 * np.abs(w)), f"call {call}"
        # and against the oracle itself, not only against the other GPU path
        parity.assert_close(g, _oracle(inp, a1, a2), f"call {call} vs oracle")


def test_noalloc_timeout_is_reported_and_cleared(cuda_lib):
    # A device wait that runs out of time is reported by tffn_check_noalloc
    # (which reads the static array's control block), and the next call runs
    # normally.  The failure is made on the host side of the protocol: with
    # the fault-injection option set, the flags of one H slice are never
    # published, so the layer-2 work that reads it waits out a 200 ms limit.
    tffn = cuda_lib
    fn, check = _entry(tffn), _check_entry(tffn)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    M, N, O, P = 16, 1024, 2048, 512
    inp = synth.ffn_inputs(M, N, O, P, seed=7, device="cuda")
    want = _oracle(inp, "relu", "none")
    detail = (ctypes.c_int32 * 4)()
    Y = torch.empty((M, P), dtype=torch.bfloat16, device="cuda")
    args = lambda: (_p(inp.X), _p(inp.W1), _p(inp.b1), _p(inp.W2), _p(inp.b2), 1, 0, M, N, O, P, _p(Y), stream)
    assert check(stream, detail) == 0          # nothing pending before the test
    old_wait = tffn.set_option(tffn.OPT_WAIT_LIMIT_MS, 200)
    old_skip = tffn.set_option(tffn.OPT_SKIP_FLAG, 3)
    try:
        assert fn(*args()) == 0
        assert check(stream, detail) == -4
        assert detail[0] == -4 and detail[1] != 0
    finally:
        tffn.set_option(tffn.OPT_SKIP_FLAG, old_skip)
        tffn.set_option(tffn.OPT_WAIT_LIMIT_MS, old_wait)
    assert check(stream, detail) == 0          # the record was cleared by the first query
    for _ in range(2):
        assert fn(*args()) == 0
        assert check(stream, detail) == 0
        parity.assert_close(Y.float().cpu().numpy(), want, "after the timeout")


def test_noalloc_rejects_what_it_cannot_hold(cuda_lib):
    fn = _entry(cuda_lib)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    p = _p(t)
    # more rows than the decode path handles
    assert fn(p, p, None, p, None, 1, 0, 33, 64, 64, 64, p, stream) == -1
    # partial sums of a 131072-wide hidden layer exceed the static scratch
    assert fn(p, p, None, p, None, 1, 0, 16, 8192, 131072, 8192, p, stream) == -2
    torch.cuda.synchronize()
