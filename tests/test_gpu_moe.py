"""Parity of moe_ffn_forward (through the C ABI) with the CPU oracle.

Routing indices, the expert-grouped permutation and the expert offsets must
match the oracle bit for bit; gate weights and outputs within the floating
point tolerance |y - y_ref| <= 1e-2 + 1e-2 |y_ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
from transformer_ffn_gb300 import synth

pytestmark = pytest.mark.gpu

ACT = {"none": oracle.ACT_NONE, "relu": oracle.ACT_RELU, "gelu_tanh": oracle.ACT_GELU_TANH}


def _assert_close(got, want, what=""):
    err = np.abs(got - want)
    bound = 1e-2 + 1e-2 * np.abs(want)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} out of tolerance, max err {err.max():.3e}"


def _inputs(T, N, O, P, E, seed, logits=None, device="cuda"):
    return synth.moe_inputs(T, N, O, P, E, seed=seed, device=device, logits=logits)


def _oracle_y(inp, k, act1, act2, tokens=None):
    u = synth.to_u16
    return oracle.moe_ffn(u(inp.X), inp.logits.cpu().numpy(), k, [u(w) for w in inp.W1],
                          [u(b) for b in inp.b1], [u(w) for w in inp.W2], [u(b) for b in inp.b2],
                          ACT[act1], ACT[act2], tokens=tokens)


def _check_routing(r, logits, k, E):
    lg = logits.cpu().numpy()
    idx, w = oracle.moe_route(lg, k)
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy(), idx)
    np.testing.assert_allclose(r["topk_w"].cpu().numpy(), w, rtol=1e-5, atol=1e-6)
    perm, offs = oracle.moe_permute(idx, E)
    np.testing.assert_array_equal(r["perm"].cpu().numpy(), perm)
    np.testing.assert_array_equal(r["expert_offsets"].cpu().numpy(), offs)


@pytest.mark.parametrize("T,N,O,P,E,k,acts", [
    (300, 64, 256, 128, 8, 2, ("gelu_tanh", "none")),
    (77, 128, 136, 72, 4, 1, ("relu", "relu")),
    (129, 64, 512, 264, 16, 4, ("gelu_tanh", "gelu_tanh")),
    (1, 64, 128, 64, 8, 2, ("gelu_tanh", "none")),
    (40, 64, 128, 64, 1, 1, ("relu", "none")),
    (50, 64, 128, 64, 4, 4, ("gelu_tanh", "none")),      # top_k = E
    (200, 1024, 256, 128, 4, 2, ("gelu_tanh", "none")),  # N > O
    (5000, 64, 128, 64, 40, 2, ("relu", "none")),        # 40 token blocks, more experts than warps in the plan
])
def test_moe_small_full(cuda_lib, T, N, O, P, E, k, acts):
    inp = _inputs(T, N, O, P, E, seed=T + E)
    Y, r = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                    acts[0], acts[1], routing=True)
    cuda_lib.check()
    _check_routing(r, inp.logits, k, E)
    _assert_close(Y.float().cpu().numpy(), _oracle_y(inp, k, *acts), "moe")


def test_moe_skewed_routing(cuda_lib):
    # one expert nobody picks, one expert every token picks, exact ties
    T, N, O, P, E, k = 200, 64, 256, 128, 8, 2
    g = torch.Generator(device="cpu").manual_seed(9)
    logits = torch.randn((T, E), generator=g)
    logits[:, 5] = -50.0
    logits[:, 2] = 50.0
    logits[::4, 0] = logits[::4, 1]
    inp = _inputs(T, N, O, P, E, seed=4, logits=logits.cuda())
    Y, r = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                    "gelu_tanh", "none", routing=True)
    cuda_lib.check()
    _check_routing(r, inp.logits, k, E)
    offs = r["expert_offsets"].cpu().numpy()
    assert offs[6] - offs[5] == 0 and offs[3] - offs[2] == T
    _assert_close(Y.float().cpu().numpy(), _oracle_y(inp, k, "gelu_tanh", "none"), "skewed")


def test_moe_equal_gates_top_all_is_mean_of_experts(cuda_lib):
    T, N, O, P, E = 64, 64, 128, 64, 4
    inp = _inputs(T, N, O, P, E, seed=8, logits=torch.zeros((T, E), device="cuda"))
    Y = cuda_lib.moe_ffn_forward(inp.X, inp.logits, E, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "none")
    cuda_lib.check()
    dense = sum(cuda_lib.ffn_forward(inp.X, inp.W1[e], inp.b1[e], inp.W2[e], inp.b2[e], "gelu_tanh",
                                     "none").float() for e in range(E)) / E
    cuda_lib.check()
    err = (Y.float() - dense).abs()
    assert torch.all(err <= 2e-2 + 2e-2 * dense.abs())


def test_moe_deterministic(cuda_lib):
    inp = _inputs(500, 128, 512, 256, 8, seed=12)
    a = cuda_lib.moe_ffn_forward(inp.X, inp.logits, 2, inp.W1, inp.b1, inp.W2, inp.b2)
    b = cuda_lib.moe_ffn_forward(inp.X, inp.logits, 2, inp.W1, inp.b1, inp.W2, inp.b2)
    cuda_lib.check()
    assert torch.equal(a, b)


def _oracle_tokens(inp, k, act1, act2, tokens):
    """The oracle on the given tokens, computed over host threads."""
    u = synth.to_u16
    host = (u(inp.X), inp.logits.cpu().numpy(), [u(w) for w in inp.W1], [u(b) for b in inp.b1],
            [u(w) for w in inp.W2], [u(b) for b in inp.b2])
    return parity.oracle_rows(lambda t: oracle.moe_ffn(*host[:2], k, *host[2:], ACT[act1], ACT[act2], tokens=t),
                              tokens)


def _full_size_tokens(r, T, k, n, seed):
    """n or more tokens to compare at full size: the first and last, tokens
    whose grouped row lies in an expert's zero-padded last band, and random
    ones."""
    tail = parity.moe_tail_tokens(r["perm"].cpu().numpy(), r["expert_offsets"].cpu().numpy(), k)
    return parity.with_random(set([0, T - 1] + tail), T, n, seed=seed), tail


def test_moe_full_size_tokens(cuda_lib):
    # T 8192, N 4096, E 8 experts of O 14336, P 4096, softmax top-2, GELU-tanh
    T, N, O, P, E, k = 8192, 4096, 14336, 4096, 8, 2
    inp = _inputs(T, N, O, P, E, seed=0)
    Y, r = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                    "gelu_tanh", "none", routing=True)
    cuda_lib.check()
    _check_routing(r, inp.logits, k, E)
    assert torch.isfinite(Y.float()).all()
    tokens, tail = _full_size_tokens(r, T, k, 64, seed=1)
    assert len(tokens) >= 64 and len(tail) >= E
    parity.assert_close(Y[tokens].float().cpu().numpy(), _oracle_tokens(inp, k, "gelu_tanh", "none", tokens),
                        "moe full size")


@pytest.mark.parametrize("router", ["balanced", "moderate", "stress"])
def test_moe_router_skew_and_segment_order(cuda_lib, router):
    # Routing skew of the MoE benchmarks (balanced / moderate / stress) under
    # both segment orders: identical routing, identical outputs bit for bit
    # (each grouped row is computed the same way wherever its band sits).
    T, N, O, P, E, k = 700, 64, 256, 128, 8, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=21, device="cuda", router=router)
    outs = []
    prev = cuda_lib.set_option(cuda_lib.OPT_MOE_ORDER, 0)
    try:
        for order in (0, 1):
            cuda_lib.set_option(cuda_lib.OPT_MOE_ORDER, order)
            Y, r = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                            "gelu_tanh", "none", routing=True)
            cuda_lib.check()
            _check_routing(r, inp.logits, k, E)
            outs.append(Y)
    finally:
        cuda_lib.set_option(cuda_lib.OPT_MOE_ORDER, prev)
    assert torch.equal(outs[0], outs[1])
    _assert_close(outs[1].float().cpu().numpy(), _oracle_y(inp, k, "gelu_tanh", "none"), router)


def test_moe_full_size_stress_skew_sampled_tokens(cuda_lib):
    # the MoE workload with expert 0 in ~98 % of the tokens
    T, N, O, P, E, k = 8192, 4096, 14336, 4096, 8, 2
    inp = synth.moe_inputs(T, N, O, P, E, seed=0, device="cuda", router="stress")
    Y, r = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2,
                                    "gelu_tanh", "none", routing=True)
    cuda_lib.check()
    _check_routing(r, inp.logits, k, E)
    offs = r["expert_offsets"].cpu().numpy()
    assert offs[1] - offs[0] > 0.95 * T
    tokens, _ = _full_size_tokens(r, T, k, 32, seed=2)
    parity.assert_close(Y[tokens].float().cpu().numpy(), _oracle_tokens(inp, k, "gelu_tanh", "none", tokens),
                        "moe stress full size")


@pytest.mark.parametrize("T,N,O,P,E,k,router", [
    (300, 64, 256, 128, 8, 2, "balanced"),
    (700, 128, 384, 264, 8, 2, "stress"),     # one expert in most tokens; ragged last Y tile
    (129, 64, 512, 520, 16, 4, "moderate"),   # top-4, three Y tiles
    (50, 64, 128, 64, 4, 4, "balanced"),      # top_k = E
    (40, 64, 128, 64, 1, 1, "balanced"),      # a single expert
])
def test_moe_fused_combine_equals_combine_kernel(cuda_lib, T, N, O, P, E, k, router):
    # The gate-weighted sum formed in the expert FFN's layer-2 epilogue (by the
    # last of a token's rows to finish) and by the separate combine kernel are
    # the same fp32 arithmetic in slot order: bit-equal, and equal to the oracle.
    inp = synth.moe_inputs(T, N, O, P, E, seed=T + k, device="cuda", router=router)
    prev = cuda_lib.set_option(cuda_lib.OPT_MOE_COMBINE, 1)
    try:
        fused = [cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "relu")
                 for _ in range(2)]
        assert cuda_lib.last_launch_count() == 5
        cuda_lib.set_option(cuda_lib.OPT_MOE_COMBINE, 0)
        sep = cuda_lib.moe_ffn_forward(inp.X, inp.logits, k, inp.W1, inp.b1, inp.W2, inp.b2, "gelu_tanh", "relu")
        assert cuda_lib.last_launch_count() == 6
    finally:
        cuda_lib.set_option(cuda_lib.OPT_MOE_COMBINE, prev)
    cuda_lib.check()
    assert torch.equal(fused[0], sep) and torch.equal(fused[1], sep)
    _assert_close(sep.float().cpu().numpy(), _oracle_y(inp, k, "gelu_tanh", "relu"), "combine")
