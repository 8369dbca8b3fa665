"""Caller-owned workspace (tffn_set_workspace) of exactly the size
tffn_workspace_bytes reports, on every path: results match the oracle, the
bytes just past the workspace are untouched, and a smaller buffer is refused
with TFFN_ERR_NO_WORKSPACE before anything runs."""
import numpy as np
import pytest
import torch

import oracle
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 1 << 20
ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
       "silu": oracle.ACT_SILU}


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bad = err > 1e-2 + 1e-2 * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"


class _Workspace:
    """A workspace of `need` bytes followed by a guard region with a pattern."""

    def __init__(self, lib, need):
        self.lib, self.need = lib, need
        n = (need + 255) // 256 * 256 + GUARD
        self.buf = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.buf[need:].fill_(0xA5)
        lib.set_workspace(self.buf[:need])

    def guard_intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[self.need:] == 0xA5).all())

    def close(self):
        self.lib.set_workspace(None)


@pytest.fixture
def lib_path(cuda_lib):
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 0)
    yield cuda_lib
    cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.set_workspace(None)


@pytest.mark.parametrize("path,M,N,O,P", [
    (0, 16, 2048, 3072, 1024),      # weight stream (split-K partials sized for every SM)
    (0, 300, 256, 1152, 320),       # fused engine
    (3, 300, 256, 1152, 320),       # engine as two launches
    (4, 300, 256, 1152, 320),       # reduce-add form (fp32 Y accumulator)
    (5, 300, 256, 1152, 320),       # back-to-back form
    (0, 100, 1024, 2048, 520),      # tensor-core weight stream (split-slice partial sums)
    (6, 200, 512, 1152, 264),       # the same at 256 rows
])
def test_dense_with_exact_caller_workspace(lib_path, path, M, N, O, P):
    lib_path.set_option(lib_path.OPT_PATH, path)
    inp = synth.ffn_inputs(M, N, O, P, seed=M + path, device="cuda")
    ws = _Workspace(lib_path, lib_path.workspace_bytes(M, N, O, P))
    try:
        Y = lib_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
        lib_path.check()
        assert ws.guard_intact(), "the call wrote past the workspace it was given"
    finally:
        ws.close()
    u = synth.to_u16
    want = oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), oracle.ACT_GELU_TANH,
                      oracle.ACT_NONE)
    _assert_close(Y.float().cpu().numpy(), want, f"path {path}")


@pytest.mark.parametrize("M", [16, 100, 300])
def test_glu_with_exact_caller_workspace(lib_path, M):
    N, O, P = 1024, 2560, 512
    g = synth.glu_inputs(M, N, O, P, seed=M, device="cuda")
    ws = _Workspace(lib_path, lib_path.workspace_bytes(M, N, O, P))
    try:
        Y = lib_path.ffn_glu_forward(g.X, g.W1, g.W3, g.W2, "silu")
        lib_path.check()
        assert ws.guard_intact()
    finally:
        ws.close()
    u = synth.to_u16
    _assert_close(Y.float().cpu().numpy(), oracle.glu_ffn(u(g.X), u(g.W1), u(g.W3), u(g.W2), oracle.ACT_SILU),
                  f"glu M={M}")


def test_moe_with_exact_caller_workspace(lib_path):
    T, N, O, P, E, k = 300, 128, 384, 192, 8, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=6, device="cuda", router="moderate")
    ws = _Workspace(lib_path, lib_path.workspace_bytes(T, N, O, P, E, k))
    try:
        Y = lib_path.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
        lib_path.check()
        assert ws.guard_intact()
    finally:
        ws.close()
    u = synth.to_u16
    want = oracle.moe_ffn(u(inp.X), inp.logits.cpu().numpy(), k, [u(w) for w in inp.W1], [u(b) for b in inp.b1],
                          [u(w) for w in inp.W2], [u(b) for b in inp.b2], oracle.ACT_GELU_TANH, oracle.ACT_NONE)
    _assert_close(Y.float().cpu().numpy(), want, "moe")


def test_too_small_caller_workspace_is_refused(lib_path):
    M, N, O, P = 300, 256, 1152, 320
    inp = synth.ffn_inputs(M, N, O, P, seed=1, device="cuda")
    need = lib_path.workspace_bytes(M, N, O, P)
    buf = torch.zeros(need, dtype=torch.uint8, device="cuda")
    lib_path.set_workspace(buf[: need - 4096])
    try:
        with pytest.raises(lib_path.TffnError) as e:
            lib_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
        assert e.value.code == -5
    finally:
        lib_path.set_workspace(None)
