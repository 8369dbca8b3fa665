"""Race detector: every path run on a caller workspace whose data region is
filled with 0xFF bytes (NaN as bf16 and as fp32) before each call, with the
output tensor pre-filled with NaN too.

A kernel that reads H before its ready flag, a split-K partial sum before its
counter, a grouped row before the gather wrote it, or that leaves part of Y
unwritten, would now produce NaN (or a wrong value) instead of silently
reusing plausible bytes from an earlier call.  Each case runs twice on the
same workspace, re-poisoned in between, and both results must be finite and
match the oracle.  Fusion changes what is read when ("Kernel fusion",
tirogla.com, section "Pitfalls"), and the layers hand H over with release /
acquire flags ("CUDA graphs and megakernels", section "3. Megakernel"), so
this checks the hand-over itself rather than the arithmetic.

The workspace's first 5 MiB (control block, ready flags, split-K counters) are
initialised by the library when a workspace is handed in and are not
poisoned: they hold the synchronisation state, not data.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

SYNC_BYTES = 5 << 20   # control block, flags and counters precede the data region
GUARD = 1 << 20
ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
       "silu": oracle.ACT_SILU}


class _PoisonedWorkspace:
    def __init__(self, lib, need):
        self.lib, self.need = lib, need
        self.buf = torch.full(((need + 255) // 256 * 256 + GUARD,), 0xFF, dtype=torch.uint8, device="cuda")
        lib.set_workspace(self.buf[:need])

    def repoison(self):
        if self.need > SYNC_BYTES:
            self.buf[SYNC_BYTES:self.need].fill_(0xFF)

    def guard_intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[self.need:] == 0xFF).all())

    def close(self):
        self.lib.set_workspace(None)


def _nan_out(M, P):
    return torch.full((M, P), float("nan"), dtype=torch.bfloat16, device="cuda")


@pytest.fixture
def lib(cuda_lib):
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 0)
    yield cuda_lib
    cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.set_workspace(None)


def _twice(lib, ws, call, want, what):
    for i in range(2):
        ws.repoison()
        Y = call()
        lib.check()
        parity.assert_close(Y.float().cpu().numpy(), want, f"{what}, call {i}")
    assert ws.guard_intact(), f"{what}: wrote past the workspace"


@pytest.mark.parametrize("path,M,N,O,P,acts", [
    (1, 300, 256, 1152, 320, ("gelu_tanh", "relu")),    # fused engine: layer 2 reads H by flags
    (3, 300, 256, 1152, 320, ("gelu_tanh", "none")),    # engine as two launches
    (2, 16, 2048, 3072, 1024, ("relu", "none")),        # mma.sync stream: split-K partials + H flags
    (2, 32, 4096, 1024, 256, ("gelu_tanh", "none")),    # N > O, long split-K ranges
    (6, 100, 1024, 2048, 520, ("gelu_tanh", "none")),   # tensor-core stream: window H + split layer 2
    (6, 200, 512, 1152, 264, ("relu", "gelu_tanh")),    # the same at 200 rows
    (4, 300, 256, 1152, 320, ("gelu_tanh", "none")),    # reduce-add form: fp32 Y accumulator
    (5, 300, 256, 1152, 320, ("gelu_tanh", "none")),    # back-to-back form
])
def test_dense_paths_on_poisoned_workspace(lib, path, M, N, O, P, acts):
    lib.set_option(lib.OPT_PATH, path)
    inp = synth.ffn_inputs(M, N, O, P, seed=M + N + path, device="cuda")
    u = synth.to_u16
    want = oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), ACT[acts[0]], ACT[acts[1]])
    ws = _PoisonedWorkspace(lib, lib.workspace_bytes(M, N, O, P))
    try:
        _twice(lib, ws, lambda: lib.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, *acts, out=_nan_out(M, P)),
               want, f"path {path}")
    finally:
        ws.close()


@pytest.mark.parametrize("M", [16, 100, 300])
def test_gated_paths_on_poisoned_workspace(lib, M):
    # the decode window (16), the tensor-core stream (100), the engine (300)
    N, O, P = 1024, 2560, 512
    g = synth.glu_inputs(M, N, O, P, seed=M + 1, device="cuda")
    u = synth.to_u16
    want = oracle.glu_ffn(u(g.X), u(g.W1), u(g.W3), u(g.W2), oracle.ACT_SILU)
    ws = _PoisonedWorkspace(lib, lib.workspace_bytes(M, N, O, P))
    try:
        _twice(lib, ws, lambda: lib.ffn_glu_forward(g.X, g.W1, g.W3, g.W2, "silu", out=_nan_out(M, P)),
               want, f"gated M={M}")
    finally:
        ws.close()


@pytest.mark.parametrize("router", ["balanced", "stress"])
def test_moe_on_poisoned_workspace(lib, router):
    # routing tables, grouped rows (with zero padding), H and the fp32 expert
    # outputs all live in the poisoned data region
    T, N, O, P, E, k = 600, 128, 384, 192, 8, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=31, device="cuda", router=router)
    u = synth.to_u16
    want = oracle.moe_ffn(u(inp.X), inp.logits.cpu().numpy(), k, [u(w) for w in inp.W1], [u(b) for b in inp.b1],
                          [u(w) for w in inp.W2], [u(b) for b in inp.b2], oracle.ACT_GELU_TANH, oracle.ACT_NONE)
    ws = _PoisonedWorkspace(lib, lib.workspace_bytes(T, N, O, P, E, k))
    try:
        _twice(lib, ws, lambda: lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                                    "gelu_tanh", "none", out=_nan_out(T, P)), want, router)
    finally:
        ws.close()


def test_moe_gated_on_poisoned_workspace(lib):
    T, N, O, P, E, k = 500, 128, 384, 192, 4, 2
    inp = synth.moe_glu_inputs(T, N, O, P, E, seed=32, device="cuda")
    u = synth.to_u16
    want = oracle.moe_glu_ffn(u(inp.X), inp.logits.cpu().numpy(), k, [u(w) for w in inp.W1],
                              [u(w) for w in inp.W3], [u(w) for w in inp.W2], oracle.ACT_SILU)
    ws = _PoisonedWorkspace(lib, lib.workspace_bytes(T, N, O, P, E, k))
    try:
        _twice(lib, ws, lambda: lib.moe_glu_forward(inp.X, inp.logits, k, inp.W1, inp.W3, inp.W2, "silu",
                                                    out=_nan_out(T, P)), want, "moe gated")
    finally:
        ws.close()


def test_poison_is_nan():
    # the fill pattern reads as NaN in both data types of the workspace
    b = np.frombuffer(bytes([0xFF] * 4), dtype=np.uint32)[0]
    assert np.isnan(np.array([b], dtype=np.uint32).view(np.float32)[0])
    assert np.isnan(torch.tensor([0xFFFF], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()[0])
