"""Engine band counts.

A fused engine launch tallies, per 256-row band and CTA rank, how many
layer-1 epilogue warps have published their rows of H; a layer-2 producer
that finds its band's tally complete starts its copies after one load instead
of polling every ready flag of the band ("Kernel fusion and tensor
parallelism", section "Step 1": a tile of H feeds the row of Y tiles once it
is ready).  The tallies are plain counters, so every launch must find them at
zero: the last CTA out of each fused launch zeroes them, including a launch
that gave up on a wait.  These tests run on a caller workspace so that the
counter region can be read back, and check the results against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

# sync-region layout of the library's workspace: control block, 4 MiB of
# ready flags, 256 KiB of split-K counters, then the 64 KiB of band counts
OFF_BCOUNT = 256 + (4 << 20) + (256 << 10)
BCOUNT_BYTES = 64 << 10
ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH}


class _Workspace:
    def __init__(self, lib, need):
        self.lib = lib
        self.buf = torch.empty((need + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
        lib.set_workspace(self.buf)

    # (the library zeroes a newly handed-in workspace's sync region when the
    # next call starts, so the counts are read only after calls)
    def counts(self):
        torch.cuda.synchronize()
        return self.buf[OFF_BCOUNT:OFF_BCOUNT + BCOUNT_BYTES].view(torch.int32).cpu().numpy()

    def close(self):
        self.lib.set_workspace(None)


@pytest.fixture
def fused(cuda_lib):
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 1)
    yield cuda_lib
    cuda_lib.set_option(cuda_lib.OPT_PATH, prev)
    cuda_lib.set_workspace(None)


def _ffn_oracle(inp, rows, act1="gelu_tanh", act2="none"):
    u = synth.to_u16
    host = (u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2))
    return parity.oracle_rows(lambda r: oracle.ffn(*host, ACT[act1], ACT[act2], rows=r), rows)


@pytest.mark.parametrize("M,N,O,P", [
    (2304, 512, 2304, 512),     # 9 bands in raster groups of 4: the last group is short
    (4096, 1024, 4096, 1024),   # 16 bands, layer-2 tiles mostly start on complete bands
    (1000, 256, 1280, 264),     # ragged last band and ragged columns
])
def test_counts_zero_after_each_launch_and_results_match(fused, M, N, O, P):
    inp = synth.ffn_inputs(M, N, O, P, seed=M + O, device="cuda")
    ws = _Workspace(fused, fused.workspace_bytes(M, N, O, P))
    try:
        rows = parity.band_rows(M)
        want = _ffn_oracle(inp, rows)
        for rep in range(3):
            Y = fused.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2)
            fused.check()
            got = ws.counts()
            assert not got.any(), f"launch {rep}: {int(np.count_nonzero(got))} band counts left non-zero"
            parity.assert_close(Y[rows].float().cpu().numpy(), want, f"launch {rep}")
    finally:
        ws.close()


def test_counts_zero_after_a_launch_that_timed_out(fused):
    M, N, O, P = 1024, 256, 1024, 256
    inp = synth.ffn_inputs(M, N, O, P, seed=11, device="cuda")
    ws = _Workspace(fused, fused.workspace_bytes(M, N, O, P))
    old_wait = fused.set_option(fused.OPT_WAIT_LIMIT_MS, 200)
    old_skip = fused.set_option(fused.OPT_SKIP_FLAG, 0)     # band 0's first tile is never published
    try:
        fused.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2)
        with pytest.raises(fused.TffnError) as ei:
            fused.check()
        assert ei.value.code == -4
        got = ws.counts()
        assert not got.any(), f"{int(np.count_nonzero(got))} band counts left non-zero by the aborted launch"
    finally:
        fused.set_option(fused.OPT_SKIP_FLAG, old_skip)
        fused.set_option(fused.OPT_WAIT_LIMIT_MS, old_wait)
    try:
        Y = fused.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2)
        fused.check()
        assert not ws.counts().any()
        rows = parity.band_rows(M)
        parity.assert_close(Y[rows].float().cpu().numpy(), _ffn_oracle(inp, rows), "after the timeout")
    finally:
        ws.close()


def test_counts_zero_after_gated_launches(fused):
    # gated layer-1 tiles hold 128 hidden columns (their W1 and W3 halves):
    # a band has O / 128 of them, each counted by its eight epilogue warps
    M, N, O, P = 1280, 512, 1536, 512
    g = synth.glu_inputs(M, N, O, P, seed=9, device="cuda")
    ws = _Workspace(fused, fused.workspace_bytes(M, N, O, P))
    try:
        u = synth.to_u16
        host = (u(g.X), u(g.W1), u(g.W3), u(g.W2))
        rows = parity.band_rows(M)
        want = parity.oracle_rows(lambda r: oracle.glu_ffn(*host, oracle.ACT_SILU, rows=r), rows)
        for rep in range(2):
            Y = fused.ffn_glu_forward(g.X, g.W1, g.W3, g.W2, "silu")
            fused.check()
            assert not ws.counts().any(), f"gated launch {rep}"
            parity.assert_close(Y[rows].float().cpu().numpy(), want, f"gated launch {rep}")
    finally:
        ws.close()


def test_counts_zero_after_moe_launches(cuda_lib):
    T, N, O, P, E, k = 1500, 256, 768, 256, 4, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=5, device="cuda")
    ws = _Workspace(cuda_lib, cuda_lib.workspace_bytes(T, N, O, P, E, k))
    try:
        u = synth.to_u16
        host = (u(inp.X), inp.logits.cpu().numpy())
        ws_ = ([u(w) for w in inp.W1], [u(b) for b in inp.b1], [u(w) for w in inp.W2], [u(b) for b in inp.b2])
        tokens = list(range(0, T, 7)) + [T - 1]
        want = parity.oracle_rows(
            lambda t: oracle.moe_ffn(*host, k, *ws_, ACT["gelu_tanh"], ACT["none"], tokens=t), tokens)
        for rep in range(2):
            Y = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2)
            cuda_lib.check()
            assert not ws.counts().any(), f"launch {rep}"
            parity.assert_close(Y[tokens].float().cpu().numpy(), want, f"moe launch {rep}")
    finally:
        ws.close()
