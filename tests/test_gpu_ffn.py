"""Parity of ffn_forward (through the C ABI) with the CPU oracle.

Tolerance, elementwise: |y - y_ref| <= 1e-2 + 1e-2 |y_ref|, y_ref the oracle's
fp64 output (H rounded to bf16 between the layers, as the kernels store it).
Small shapes are compared in full; the full-size workloads on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH}


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def _run(tffn, inp, act1, act2, path=0):
    old = tffn.set_option(tffn.OPT_PATH, path)
    try:
        Y = tffn.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, act1, act2)
        tffn.check()
    finally:
        tffn.set_option(tffn.OPT_PATH, old)
    return Y


def _oracle(inp, act1, act2, rows=None):
    u = synth.to_u16
    return oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), ACT[act1], ACT[act2],
                      rows=rows)


def _case(M, N, O, P, seed, device="cuda"):
    return synth.ffn_inputs(M, N, O, P, seed=seed, device=device)


# ------------------------------------------------------------- small, in full

@pytest.mark.parametrize("path", [0, 1, 2, 3, 6])
def test_tiny_config_full(cuda_lib, path):
    # 64 x 256 x 1024 x 256, GELU-tanh, no second activation, seed 0; path 0 is
    # the library's own choice at 64 rows (the tensor-core weight stream)
    inp = _case(64, 256, 1024, 256, seed=0)
    Y = _run(cuda_lib, inp, "gelu_tanh", "none", path=path)
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, "gelu_tanh", "none"), "tiny")


@pytest.mark.parametrize("shape,acts", [
    ((200, 136, 520, 264), ("relu", "gelu_tanh")),      # ragged rows, columns, K
    ((129, 64, 256, 128), ("gelu_tanh", "relu")),       # one row past a band
    ((384, 512, 768, 520), ("gelu_tanh", "none")),      # several bands and tiles
    ((33, 8, 8, 8), ("none", "none")),                  # minimum widths
    ((1, 256, 264, 72), ("gelu_tanh", "none")),         # one row through the engine
])
def test_engine_ragged_shapes(cuda_lib, shape, acts):
    M, N, O, P = shape
    inp = _case(M, N, O, P, seed=sum(shape))
    Y = _run(cuda_lib, inp, acts[0], acts[1], path=1)
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, *acts), f"engine {shape}")


@pytest.mark.parametrize("shape,acts", [
    ((16, 512, 1024, 256), ("relu", "none")),
    ((1, 256, 384, 136), ("gelu_tanh", "relu")),
    ((5, 136, 520, 264), ("gelu_tanh", "none")),
    ((17, 1024, 2048, 512), ("relu", "gelu_tanh")),     # two m tiles
    ((32, 64, 128, 64), ("gelu_tanh", "none")),
    ((8, 4096, 8192, 1024), ("relu", "none")),          # long split-K ranges
    ((16, 4096, 1024, 256), ("gelu_tanh", "none")),     # N > O: more layer-1 k than hidden columns
    ((4, 2048, 136, 4096), ("relu", "none")),           # N > O, narrow ragged hidden, wide output
    ((48, 512, 1024, 256), ("gelu_tanh", "none")),      # four 16-row tiles (64-row instance)
    ((64, 1024, 2048, 512), ("relu", "gelu_tanh")),
    ((33, 136, 520, 264), ("gelu_tanh", "relu")),       # one row past the 32-row instance, ragged
])
def test_decode_path_full(cuda_lib, shape, acts):
    M, N, O, P = shape
    inp = _case(M, N, O, P, seed=7 + sum(shape))
    Y = _run(cuda_lib, inp, acts[0], acts[1], path=2)
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, *acts), f"decode {shape}")


@pytest.mark.parametrize("path", [1, 3])
@pytest.mark.parametrize("shape", [(16, 4096, 1024, 256), (64, 2048, 256, 512), (300, 1024, 136, 200)])
def test_engine_input_wider_than_hidden(cuda_lib, path, shape):
    # N > O: a layer-1 tile has more k-blocks than there are H tiles (a
    # down-projecting FFN); layer-1 tasks must not wait on H flags
    inp = _case(*shape, seed=sum(shape))
    Y = _run(cuda_lib, inp, "gelu_tanh", "none", path=path)
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, "gelu_tanh", "none"), f"N > O {shape}")


def test_fused_equals_two_launches_bitwise(cuda_lib):
    inp = _case(300, 256, 1024, 384, seed=3)
    a = _run(cuda_lib, inp, "gelu_tanh", "none", path=1)
    b = _run(cuda_lib, inp, "gelu_tanh", "none", path=3)
    assert torch.equal(a, b)


@pytest.mark.parametrize("path,M", [(1, 520), (2, 24)])
def test_deterministic(cuda_lib, path, M):
    inp = _case(M, 512, 2048, 512, seed=11)
    a = _run(cuda_lib, inp, "gelu_tanh", "relu", path=path)
    b = _run(cuda_lib, inp, "gelu_tanh", "relu", path=path)
    assert torch.equal(a, b)


def test_empty_rows(cuda_lib):
    inp = _case(0, 64, 128, 64, seed=1)
    Y = cuda_lib.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2)
    assert Y.shape == (0, 64)
    assert cuda_lib.last_launch_count() == 0


def test_no_bias(cuda_lib):
    inp = _case(150, 128, 512, 256, seed=5)
    Y = cuda_lib.ffn_forward(inp.X, inp.W1, None, inp.W2, None, "gelu_tanh", "none")
    cuda_lib.check()
    u = synth.to_u16
    want = oracle.ffn(u(inp.X), u(inp.W1), None, u(inp.W2), None, oracle.ACT_GELU_TANH, oracle.ACT_NONE)
    _assert_close(Y.float().cpu().numpy(), want, "no bias")


@pytest.mark.parametrize("G", [2, 4])
def test_megatron_shards_sum_to_full(cuda_lib, G):
    # W1 split by columns and W2 by rows: the shards' partial outputs (b2 and
    # act2 left out) summed, then b2 and act2, match the unsplit FFN.
    M, N, O, P = 256, 256, 1024, 256
    inp = _case(M, N, O, P, seed=21)
    s = O // G
    acc = torch.zeros((M, P), dtype=torch.float32, device="cuda")
    for g in range(G):
        part = cuda_lib.ffn_forward(inp.X, inp.W1[:, g * s:(g + 1) * s].contiguous(),
                                    inp.b1[g * s:(g + 1) * s].contiguous(),
                                    inp.W2[g * s:(g + 1) * s].contiguous(), None, "gelu_tanh", "none")
        acc += part.float()
    cuda_lib.check()
    y = torch.relu(acc + inp.b2.float())
    want = _oracle(inp, "gelu_tanh", "relu")
    # each partial is rounded to bf16 once more than the unsplit output
    err = np.abs(y.cpu().numpy() - want)
    assert np.all(err <= 2e-2 + 2e-2 * np.abs(want))


# --------------------------------------------------- full-size, sampled rows
# Rows are compared with the oracle one by one (computed over host threads).
# Prefill: rows 0, 127, 128 and 255 of every 256-row band (both CTAs of the
# pair tile, the band edges), so every band and every raster group of four
# bands is checked.  Large: one row per band at a varying offset, plus the
# band edges of every fourth band.  Decode: all 16 rows.

def _large_rows(M):
    rows = {b * 256 + (b * 37) % 256 for b in range(M // 256)}
    for b in range(0, M // 256, 4):
        rows |= {b * 256 + 127, b * 256 + 128, b * 256 + 255}
    rows |= {0, M - 1}
    return sorted(rows)


@pytest.mark.parametrize("name,shape,acts", [
    ("prefill", (4096, 4096, 16384, 4096), ("gelu_tanh", "none")),
    ("decode", (16, 8192, 28672, 8192), ("relu", "none")),
    ("large", (16384, 8192, 28672, 8192), ("gelu_tanh", "relu")),
])
def test_full_size_rows(cuda_lib, name, shape, acts):
    M, N, O, P = shape
    inp = _case(M, N, O, P, seed=0)
    Y = _run(cuda_lib, inp, acts[0], acts[1], path=0)
    assert torch.isfinite(Y.float()).all()
    if name == "decode":
        rows = list(range(M))
    elif name == "prefill":
        rows = parity.band_rows(M)
    else:
        rows = _large_rows(M)
    assert len(rows) >= min(M, 64)
    u = synth.to_u16
    host = (u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2))
    want = parity.oracle_rows(
        lambda r: oracle.ffn(*host, ACT[acts[0]], ACT[acts[1]], rows=r), rows)
    parity.assert_close(Y[rows].float().cpu().numpy(), want, name)


# ---------------------------------------------------------- failure report

def test_wait_timeout_is_reported_and_recovered(cuda_lib):
    tffn = cuda_lib
    inp = _case(256, 256, 512, 256, seed=2)
    old_wait = tffn.set_option(tffn.OPT_WAIT_LIMIT_MS, 200)
    old_skip = tffn.set_option(tffn.OPT_SKIP_FLAG, 0)    # tile 0's flag is never published
    old_path = tffn.set_option(tffn.OPT_PATH, 1)
    try:
        tffn.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2)
        with pytest.raises(tffn.TffnError) as ei:
            tffn.check()
        assert ei.value.code == -4
    finally:
        tffn.set_option(tffn.OPT_SKIP_FLAG, old_skip)
        tffn.set_option(tffn.OPT_WAIT_LIMIT_MS, old_wait)
    try:
        # the next call runs normally on the re-initialised workspace
        Y = tffn.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2)
        tffn.check()
    finally:
        tffn.set_option(tffn.OPT_PATH, old_path)
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, "gelu_tanh", "none"), "after timeout")
