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

from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu


def _entry(tffn):
    L = tffn.load()
    fn = L.ffn_forward_decode_noalloc
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, i64, i64, i64, vp, vp]
    fn.restype = i32
    return fn


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
