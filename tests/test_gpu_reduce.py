"""The reduce-add form of the fused FFN (TFFN_OPT_PATH = 4): each H tile is
multiplied by its row of W2 tiles and the products are reduced into an fp32
Y with asynchronous tile reductions ("Kernel fusion and tensor parallelism",
section "Step 1").  Parity with the CPU oracle: |y - y_ref| <= 1e-2 + 1e-2 |y_ref|.
The reduction order varies, so results are compared within the tolerance, not
bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH,
       "silu": oracle.ACT_SILU}


@pytest.fixture
def reduce_path(cuda_lib):
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 4)
    yield cuda_lib
    cuda_lib.set_option(cuda_lib.OPT_PATH, prev)


def _oracle(inp, acts, rows=None):
    u = synth.to_u16
    return oracle.ffn(u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2), ACT[acts[0]], ACT[acts[1]],
                      rows=rows)


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bad = err > 1e-2 + 1e-2 * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"


@pytest.mark.parametrize("M,N,O,P,acts", [
    (64, 256, 1024, 256, ("gelu_tanh", "none")),     # one band, four hidden tiles
    (300, 136, 328, 200, ("gelu_tanh", "relu")),     # ragged rows, hidden and output tails, 2-D maps
    (513, 64, 512, 576, ("relu", "gelu_tanh")),      # three bands, three output tiles
    (16, 512, 256, 128, ("silu", "none")),           # one hidden tile: a single contribution
])
def test_reduce_form_small_full(reduce_path, M, N, O, P, acts):
    inp = synth.ffn_inputs(M, N, O, P, seed=M + P, device="cuda")
    Y = reduce_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, *acts)
    reduce_path.check()
    assert reduce_path.last_launch_count() == 1
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, acts), "reduce form")


def test_reduce_form_repeated_calls_start_from_zero(reduce_path):
    # the accumulator and counters are cleared by every call
    inp = synth.ffn_inputs(400, 128, 768, 320, seed=5, device="cuda")
    a = reduce_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    b = reduce_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    reduce_path.check()
    want = _oracle(inp, ("gelu_tanh", "none"))
    _assert_close(a.float().cpu().numpy(), want, "first call")
    _assert_close(b.float().cpu().numpy(), want, "second call")


def test_reduce_form_agrees_with_engine(reduce_path):
    inp = synth.ffn_inputs(1024, 512, 2048, 1024, seed=2, device="cuda")
    r = reduce_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    reduce_path.set_option(reduce_path.OPT_PATH, 1)
    e = reduce_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    reduce_path.check()
    d = (r.float() - e.float()).abs()
    assert torch.all(d <= 2e-2 + 2e-2 * e.float().abs())


def test_reduce_form_full_size_band_rows(reduce_path):
    # the prefill workload: M 4096, N 4096, O 16384, P 4096, GELU-tanh
    M, N, O, P = 4096, 4096, 16384, 4096
    inp = synth.ffn_inputs(M, N, O, P, seed=0, device="cuda")
    Y = reduce_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    reduce_path.check()
    assert torch.isfinite(Y.float()).all()
    rows = parity.band_rows(M)
    u = synth.to_u16
    host = (u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2))
    want = parity.oracle_rows(lambda r: oracle.ffn(*host, oracle.ACT_GELU_TANH, oracle.ACT_NONE, rows=r), rows)
    parity.assert_close(Y[rows].float().cpu().numpy(), want, "full size")


# ------------------------------------------------- back-to-back form (path 5)
# Each task walks the hidden tiles of one band for one Y tile; H lives only in
# shared memory and the products are summed in tensor memory (no reductions),
# so the results are bit-reproducible.

@pytest.fixture
def b2b_path(cuda_lib):
    prev = cuda_lib.set_option(cuda_lib.OPT_PATH, 5)
    yield cuda_lib
    cuda_lib.set_option(cuda_lib.OPT_PATH, prev)


@pytest.mark.parametrize("M,N,O,P,acts", [
    (64, 256, 1024, 256, ("gelu_tanh", "none")),     # the tiny FFN: one task
    (300, 136, 328, 200, ("gelu_tanh", "relu")),     # ragged rows, hidden and output tails, 2-D maps
    (513, 64, 512, 576, ("relu", "gelu_tanh")),      # three bands x three Y tiles
    (16, 512, 256, 128, ("silu", "none")),           # one hidden tile
    (8, 64, 4096, 64, ("gelu_tanh", "none")),        # sixteen hidden tiles summed in tensor memory
])
def test_b2b_form_small_full(b2b_path, M, N, O, P, acts):
    inp = synth.ffn_inputs(M, N, O, P, seed=M + O, device="cuda")
    Y = b2b_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, *acts)
    b2b_path.check()
    assert b2b_path.last_launch_count() == 1
    _assert_close(Y.float().cpu().numpy(), _oracle(inp, acts), "b2b form")


def test_b2b_form_deterministic_and_close_to_engine(b2b_path):
    inp = synth.ffn_inputs(700, 256, 1536, 512, seed=4, device="cuda")
    a = b2b_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    b = b2b_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    b2b_path.set_option(b2b_path.OPT_PATH, 1)
    e = b2b_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    b2b_path.check()
    assert torch.equal(a, b)
    d = (a.float() - e.float()).abs()
    assert torch.all(d <= 2e-2 + 2e-2 * e.float().abs())


def test_b2b_form_full_size_band_rows(b2b_path):
    # the prefill workload through the back-to-back form (H recomputed for each
    # of the 16 Y tiles of a band): slow, but exact
    M, N, O, P = 4096, 4096, 16384, 4096
    inp = synth.ffn_inputs(M, N, O, P, seed=0, device="cuda")
    Y = b2b_path.ffn_forward(inp.X, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    b2b_path.check()
    rows = parity.band_rows(M)
    u = synth.to_u16
    host = (u(inp.X), u(inp.W1), u(inp.b1), u(inp.W2), u(inp.b2))
    want = parity.oracle_rows(lambda r: oracle.ffn(*host, oracle.ACT_GELU_TANH, oracle.ACT_NONE, rows=r), rows)
    parity.assert_close(Y[rows].float().cpu().numpy(), want, "b2b full size")
