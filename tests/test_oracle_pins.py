"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one part of the oracle to something fixed outside it: exact
rational arithmetic on tiny inputs, closed forms of the activations, an
independent integer rounding routine, library routines for special cases, and
the identities the fused-FFN page states (the Megatron-LM split, the collapse
of two linear layers).  A dropped term, a wrong sign, a transposed operand or
a misplaced rounding in the oracle fails at least one of them.
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import ACT_GELU_TANH, ACT_NONE, ACT_RELU
from transformer_ffn_gb300 import synth

# ----------------------------------------------------------------- bf16 ----


def _int_round_f32_bits_to_bf16(bits):
    """Independent RNE of binary32 bit patterns to bf16 by integer arithmetic."""
    bits = bits.astype(np.uint64)
    return ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)


def test_bf16_widening_exhaustive():
    L = oracle.lib()
    for h in range(0, 1 << 16):
        if (h & 0x7F80) == 0x7F80 and (h & 0x007F):
            continue  # NaN payloads
        ref = np.array([h << 16], dtype=np.uint32).view(np.float32)[0]
        assert L.tffn_oracle_bf16_to_f64(h) == float(ref), hex(h)


@pytest.mark.parametrize("exp_field", [0, 1, 100, 126, 127, 128, 200, 254])
def test_bf16_rounding_matches_integer_rne_on_fp32_patterns(exp_field):
    # Every 7th mantissa plus every pattern whose low half sits at or next to
    # the tie point 0x8000, for one binary32 exponent, both signs.
    mant = np.arange(0, 1 << 23, 7, dtype=np.uint32)
    ties = (np.arange(0, 1 << 7, dtype=np.uint32)[:, None] << 16) + \
        np.array([0x7FFF, 0x8000, 0x8001, 0x0000, 0xFFFF], dtype=np.uint32)[None, :]
    mant = np.unique(np.concatenate([mant, ties.ravel()]))
    for sign in (0, 1):
        bits = (np.uint32(sign) << 31) | (np.uint32(exp_field) << 23) | mant
        vals = bits.view(np.float32).astype(np.float64)
        want = _int_round_f32_bits_to_bf16(bits)
        L = oracle.lib()
        got = np.fromiter((L.tffn_oracle_f64_to_bf16(float(v)) for v in vals[::53]),
                          dtype=np.uint16)
        np.testing.assert_array_equal(got, want[::53])
        # the tie neighbourhood in full
        sel = np.isin(bits & 0xFFFF, [0x7FFF, 0x8000, 0x8001])
        got_t = np.fromiter((L.tffn_oracle_f64_to_bf16(float(v)) for v in vals[sel]),
                            dtype=np.uint16)
        np.testing.assert_array_equal(got_t, want[sel])


@pytest.mark.parametrize("x, want", [
    (1.0, 0x3F80),
    (1.0 + 2**-8, 0x3F80),              # tie -> even (mantissa 0)
    (1.0 + 3 * 2**-8, 0x3F82),          # tie -> even (mantissa 2)
    (1.0 + 2**-8 + 2**-30, 0x3F81),     # above the tie; rounding via fp32 first would give 0x3F80
    (-(1.0 + 2**-8 + 2**-30), 0xBF81),
    (2.0**-133, 0x0001),                # smallest bf16 subnormal
    (2.0**-134, 0x0000),                # tie between 0 and the smallest subnormal -> 0
    (3 * 2.0**-134, 0x0002),            # tie -> even subnormal
    ((2 - 2**-7) * 2.0**127, 0x7F7F),   # largest finite bf16
    ((2 - 2**-8) * 2.0**127, 0x7F80),   # tie at the top rounds to infinity
    ((2 - 2**-8 - 2**-20) * 2.0**127, 0x7F7F),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (math.inf, 0x7F80),
    (-math.inf, 0xFF80),
])
def test_bf16_rounding_special_values(x, want):
    assert oracle.f64_to_bf16(x) == want


# ---------------------------------------------------------- activations ----


def test_relu_closed_form():
    assert oracle.act(ACT_RELU, -1.0) == 0.0
    assert oracle.act(ACT_RELU, 2.0) == 2.0
    assert oracle.act(ACT_RELU, 0.0) == 0.0
    assert oracle.act(ACT_RELU, -1e-300) == 0.0
    assert oracle.act(ACT_NONE, -3.25) == -3.25


def test_gelu_tanh_special_values_and_identities():
    assert oracle.act(ACT_GELU_TANH, 0.0) == 0.0
    for x in (0.1, 0.5, 1.0, 2.0, 3.7, 8.0):
        # tanh is odd, so GELU(x) - GELU(-x) = x exactly up to rounding
        d = oracle.act(ACT_GELU_TANH, x) - oracle.act(ACT_GELU_TANH, -x)
        assert abs(d - x) <= 4e-16 * max(1.0, abs(x))
    assert abs(oracle.act(ACT_GELU_TANH, 30.0) - 30.0) < 1e-12
    assert abs(oracle.act(ACT_GELU_TANH, -30.0)) < 1e-12


def test_gelu_tanh_matches_library_routine():
    xs = torch.linspace(-12, 12, 4001, dtype=torch.float64)
    ref = torch.nn.functional.gelu(xs, approximate="tanh")
    got = torch.tensor([oracle.act(ACT_GELU_TANH, float(x)) for x in xs], dtype=torch.float64)
    assert torch.allclose(got, ref, rtol=1e-14, atol=1e-15)


def test_gelu_tanh_is_close_to_exact_gelu():
    # the tanh form approximates x * Phi(x); its error stays below 1e-3
    for i in range(-800, 801):
        x = i / 100.0
        exact = 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))
        assert abs(oracle.act(ACT_GELU_TANH, x) - exact) < 1e-3


# ------------------------------------------------- FFN by brute force ----


def _frac_to_bf16(q: Fraction) -> Fraction:
    """Nearest bf16 value of an exact rational (ties to even), finite range."""
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # 2^(e-1) <= a < 2^e after correction
    while Fraction(2) ** e <= a:
        e += 1
    while Fraction(2) ** (e - 1) > a:
        e -= 1
    ulp = Fraction(2) ** max(e - 8, -133)
    n = a / ulp
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return s * fl * ulp


def _u16_of_values(vals):
    out = np.array([np.float32(v) for v in vals], dtype=np.float32).view(np.uint32)
    assert np.all(out & 0xFFFF == 0), "values must be exact bf16"
    return (out >> 16).astype(np.uint16)


def _bf16_values(rng, count, choices):
    return [rng.choice(choices) for _ in range(count)]


def _exact_ffn(X, W1, b1, W2, b2, act1, act2, M, N, O, P, round_h=True):
    def actq(kind, v):
        if kind == ACT_NONE:
            return v
        if kind == ACT_RELU:
            return v if v > 0 else Fraction(0)
        raise ValueError
    Y = []
    for i in range(M):
        h = []
        for j in range(O):
            s = sum((Fraction(X[i * N + n]) * Fraction(W1[n * O + j]) for n in range(N)),
                    Fraction(0))
            v = actq(act1, s + Fraction(b1[j]))
            h.append(_frac_to_bf16(v) if round_h else v)
        row = []
        for k in range(P):
            s = sum((h[o] * Fraction(W2[o * P + k]) for o in range(O)), Fraction(0))
            row.append(actq(act2, s + Fraction(b2[k])))
        Y.append(row)
    return Y


@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 3, 4, 5), (7, 9, 13, 5)])
@pytest.mark.parametrize("acts", [(ACT_RELU, ACT_NONE), (ACT_NONE, ACT_RELU), (ACT_RELU, ACT_RELU)])
def test_ffn_brute_force_integer_values(shape, acts):
    # integer inputs with |x| <= 3: every sum is an exactly representable integer
    M, N, O, P = shape
    rng = random.Random(hash(shape) & 0xFFFF)
    ints = [-3, -2, -1, 0, 1, 2, 3]
    X = _bf16_values(rng, M * N, ints)
    W1 = _bf16_values(rng, N * O, [-1, 0, 1])
    b1 = _bf16_values(rng, O, ints)
    W2 = _bf16_values(rng, O * P, [-1, 0, 1])
    b2 = _bf16_values(rng, P, ints)
    want = _exact_ffn(X, W1, b1, W2, b2, acts[0], acts[1], M, N, O, P)
    got = oracle.ffn(_u16_of_values(X).reshape(M, N), _u16_of_values(W1).reshape(N, O),
                     _u16_of_values(b1), _u16_of_values(W2).reshape(O, P),
                     _u16_of_values(b2), acts[0], acts[1])
    assert got.tolist() == [[float(v) for v in r] for r in want]


@pytest.mark.parametrize("shape", [(2, 3, 4, 5), (7, 9, 13, 5), (3, 17, 33, 6)])
@pytest.mark.parametrize("acts", [(ACT_RELU, ACT_NONE), (ACT_NONE, ACT_NONE), (ACT_RELU, ACT_RELU)])
def test_ffn_brute_force_fractional_values(shape, acts):
    # bf16 fractions; H is rounded to bf16 with exact rational arithmetic, so
    # the rounding point between the layers is checked too
    M, N, O, P = shape
    rng = random.Random(sum(shape) * 31 + acts[0] * 7 + acts[1])
    cnt = M * N + N * O + O + O * P + P
    raw = np.array([rng.uniform(-2, 2) for _ in range(cnt)], dtype=np.float32)
    vals = (raw.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64).tolist()
    it = iter(vals)
    X = [next(it) for _ in range(M * N)]
    W1 = [next(it) for _ in range(N * O)]
    b1 = [next(it) for _ in range(O)]
    W2 = [next(it) for _ in range(O * P)]
    b2 = [next(it) for _ in range(P)]
    want = _exact_ffn(X, W1, b1, W2, b2, acts[0], acts[1], M, N, O, P)
    Yo, Ho = oracle.ffn(_u16_of_values(X).reshape(M, N), _u16_of_values(W1).reshape(N, O),
                        _u16_of_values(b1), _u16_of_values(W2).reshape(O, P),
                        _u16_of_values(b2), acts[0], acts[1], want_h=True)
    for i in range(M):
        for k in range(P):
            w = float(want[i][k])
            assert abs(Yo[i, k] - w) <= 1e-12 * max(1.0, abs(w)), (i, k)
    # the H rows match the exact rational rounding bit for bit
    for i in range(M):
        for j in range(O):
            s = sum((Fraction(X[i * N + n]) * Fraction(W1[n * O + j]) for n in range(N)),
                    Fraction(0)) + Fraction(b1[j])
            if acts[0] == ACT_RELU and s < 0:
                s = Fraction(0)
            assert oracle.bf16_to_f64(int(Ho[i, j])) == float(_frac_to_bf16(s))


def test_ffn_row_subset_matches_full():
    inp = synth.ffn_inputs(9, 24, 40, 16, seed=3)
    a = [synth.to_u16(t) for t in (inp.X, inp.W1, inp.b1, inp.W2, inp.b2)]
    full = oracle.ffn(*a, ACT_GELU_TANH, ACT_RELU)
    rows = [8, 0, 5]
    sub = oracle.ffn(*a, ACT_GELU_TANH, ACT_RELU, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])


# --------------------------------------------- identities from the pages ----


@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("acts", [(ACT_GELU_TANH, ACT_NONE), (ACT_RELU, ACT_RELU),
                                  (ACT_GELU_TANH, ACT_GELU_TANH)])
def test_megatron_split_reproduces_unsplit(G, acts):
    # W1 split by columns, W2 by rows: the partial outputs summed, then b2 and
    # the second activation, equal the unsplit FFN.
    M, N, O, P = 6, 32, 64, 24
    inp = synth.ffn_inputs(M, N, O, P, seed=11 + G)
    X, W1, b1, W2, b2 = (synth.to_u16(t) for t in (inp.X, inp.W1, inp.b1, inp.W2, inp.b2))
    full = oracle.ffn(X, W1, b1, W2, b2, acts[0], acts[1])
    s = O // G
    acc = np.zeros((M, P))
    for g in range(G):
        acc += oracle.ffn(X, np.ascontiguousarray(W1[:, g * s:(g + 1) * s]),
                          np.ascontiguousarray(b1[g * s:(g + 1) * s]),
                          np.ascontiguousarray(W2[g * s:(g + 1) * s, :]), None,
                          acts[0], ACT_NONE)
    b2d = np.array([oracle.bf16_to_f64(int(v)) for v in b2])
    split = np.vectorize(lambda v: oracle.act(acts[1], v))(acc + b2d[None, :])
    np.testing.assert_allclose(split, full, rtol=1e-12, atol=1e-12)


def test_megatron_split_detects_bias_before_sum():
    # applying b2 to each partial (the error the page warns about) is caught
    M, N, O, P = 4, 16, 32, 8
    inp = synth.ffn_inputs(M, N, O, P, seed=5)
    X, W1, b1, W2, b2 = (synth.to_u16(t) for t in (inp.X, inp.W1, inp.b1, inp.W2, inp.b2))
    full = oracle.ffn(X, W1, b1, W2, b2, ACT_RELU, ACT_NONE)
    wrong = sum(oracle.ffn(X, np.ascontiguousarray(W1[:, g * 16:(g + 1) * 16]),
                           np.ascontiguousarray(b1[g * 16:(g + 1) * 16]),
                           np.ascontiguousarray(W2[g * 16:(g + 1) * 16, :]), b2,
                           ACT_RELU, ACT_NONE) for g in range(2))
    assert np.max(np.abs(wrong - full)) > 1e-3


def test_linear_collapse_without_activation():
    # (X W1 + b1) W2 + b2 = X (W1 W2) + (b1 W2 + b2) when nothing sits between
    M, N, O, P = 5, 24, 40, 12
    inp = synth.ffn_inputs(M, N, O, P, seed=7)
    X, W1, b1, W2, b2 = (synth.to_u16(t) for t in (inp.X, inp.W1, inp.b1, inp.W2, inp.b2))
    got = oracle.ffn(X, W1, b1, W2, b2, ACT_NONE, ACT_NONE, round_h=False)

    def f(a):
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Xd, W1d, b1d, W2d, b2d = f(X), f(W1), f(b1), f(W2), f(b2)
    want = Xd @ (W1d @ W2d) + (b1d @ W2d + b2d)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------ MoE ----


def _brute_topk(l, k):
    return sorted(range(len(l)), key=lambda e: (-float(l[e]), e))[:k]


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 8, 2), (64, 8, 8), (50, 16, 4), (20, 64, 6)])
def test_routing_matches_brute_force_sort(T, E, k):
    rng = np.random.default_rng(T * 1000 + E * 10 + k)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # plant exact ties
    logits[::3, : E // 2] = logits[::3, :1]
    idx, w = oracle.moe_route(logits, k)
    for t in range(T):
        assert list(idx[t]) == _brute_topk(logits[t], k)
        assert abs(w[t].sum() - 1.0) < 1e-15
        assert np.all(w[t] > 0) and np.all(np.diff(w[t]) <= 0)
        # weights are the softmax over E restricted to the kept experts, renormalised
        full = np.exp(logits[t].astype(np.float64) - logits[t].max())
        full /= full.sum()
        kept = full[idx[t]] / full[idx[t]].sum()
        np.testing.assert_allclose(w[t], kept, rtol=1e-13)


def test_permutation_order_and_offsets():
    rng = np.random.default_rng(0)
    T, E, k = 300, 8, 2
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:40, 3] = 50.0       # a crowded expert
    logits[:, 6] = -50.0        # an expert nobody picks
    idx, _ = oracle.moe_route(logits, k)
    perm, offs = oracle.moe_permute(idx, E)
    assert offs[0] == 0 and offs[E] == T * k
    assert np.all(np.diff(offs) >= 0)
    assert offs[7] - offs[6] == 0
    want = sorted(((int(idx[t, s]), t, s) for t in range(T) for s in range(k)))
    assert [int(p) for p in perm] == [t * k + s for (_, t, s) in want]
    counts = np.bincount(idx.ravel(), minlength=E)
    np.testing.assert_array_equal(np.diff(offs), counts)


def _moe_case(T, N, O, P, E, seed, logits=None):
    inp = synth.moe_inputs(T, N, O, P, E, seed=seed,
                           logits=None if logits is None else torch.from_numpy(logits))
    u = synth.to_u16
    return (u(inp.X), inp.logits.numpy(), [u(w) for w in inp.W1], [u(b) for b in inp.b1],
            [u(w) for w in inp.W2], [u(b) for b in inp.b2])


def test_moe_all_experts_equal_gates_is_mean_of_experts():
    T, N, O, P, E = 5, 16, 32, 8, 4
    X, _, W1, b1, W2, b2 = _moe_case(T, N, O, P, E, seed=1)
    logits = np.zeros((T, E), dtype=np.float32)
    got = oracle.moe_ffn(X, logits, E, W1, b1, W2, b2, ACT_GELU_TANH, ACT_NONE)
    dense = [oracle.ffn(X, W1[e], b1[e], W2[e], b2[e], ACT_GELU_TANH, ACT_NONE) for e in range(E)]
    np.testing.assert_allclose(got, sum(dense) / E, rtol=1e-13, atol=1e-14)


def test_moe_top1_is_the_argmax_expert():
    T, N, O, P, E = 12, 16, 32, 8, 4
    X, logits, W1, b1, W2, b2 = _moe_case(T, N, O, P, E, seed=2)
    got = oracle.moe_ffn(X, logits, 1, W1, b1, W2, b2, ACT_RELU, ACT_RELU)
    for t in range(T):
        e = int(np.argmax(logits[t]))
        want = oracle.ffn(X, W1[e], b1[e], W2[e], b2[e], ACT_RELU, ACT_RELU, rows=[t])
        np.testing.assert_array_equal(got[t], want[0])


def test_moe_single_expert_is_dense_ffn():
    T, N, O, P = 6, 16, 24, 8
    X, logits, W1, b1, W2, b2 = _moe_case(T, N, O, P, 1, seed=4)
    got = oracle.moe_ffn(X, logits, 1, W1, b1, W2, b2, ACT_GELU_TANH, ACT_NONE)
    want = oracle.ffn(X, W1[0], b1[0], W2[0], b2[0], ACT_GELU_TANH, ACT_NONE)
    np.testing.assert_array_equal(got, want)


def test_moe_top2_is_weighted_sum_of_two_experts():
    T, N, O, P, E = 8, 16, 32, 8, 8
    X, logits, W1, b1, W2, b2 = _moe_case(T, N, O, P, E, seed=6)
    got = oracle.moe_ffn(X, logits, 2, W1, b1, W2, b2, ACT_GELU_TANH, ACT_NONE, tokens=[3, 7])
    for r, t in enumerate([3, 7]):
        e = _brute_topk(logits[t], 2)
        l0, l1 = float(logits[t][e[0]]), float(logits[t][e[1]])
        g1 = 1.0 / (1.0 + math.exp(l0 - l1))       # softmax over the two kept logits
        g0 = 1.0 - g1
        y0 = oracle.ffn(X, W1[e[0]], b1[e[0]], W2[e[0]], b2[e[0]], ACT_GELU_TANH, ACT_NONE, rows=[t])
        y1 = oracle.ffn(X, W1[e[1]], b1[e[1]], W2[e[1]], b2[e[1]], ACT_GELU_TANH, ACT_NONE, rows=[t])
        np.testing.assert_allclose(got[r], g0 * y0[0] + g1 * y1[0], rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------ gated FFN ----
# "Kernel fusion and tensor parallelism", section "Results": the SwiGLU FFN of
# the benchmarked models has a third weight matrix that gates the activation
# and no biases; written out as H = act(X W1) * (X W3), Y = H W2.

ACT_SILU = oracle.ACT_SILU


def test_silu_closed_forms_and_identities():
    assert oracle.act(ACT_SILU, 0.0) == 0.0
    for x in (0.1, 0.5, 1.0, 2.0, 5.5, 20.0):
        # sigma(x) + sigma(-x) = 1, so silu(x) - silu(-x) = x
        d = oracle.act(ACT_SILU, x) - oracle.act(ACT_SILU, -x)
        assert abs(d - x) <= 4e-16 * max(1.0, abs(x))
    assert oracle.act(ACT_SILU, 1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert abs(oracle.act(ACT_SILU, 40.0) - 40.0) < 1e-15
    assert abs(oracle.act(ACT_SILU, -40.0)) < 1e-15
    v = oracle.act(ACT_SILU, -1000.0)
    assert v == 0.0 and not math.isnan(v)


def test_silu_matches_library_routine():
    xs = torch.linspace(-30, 30, 6001, dtype=torch.float64)
    ref = torch.nn.functional.silu(xs)
    got = torch.tensor([oracle.act(ACT_SILU, float(x)) for x in xs], dtype=torch.float64)
    assert torch.allclose(got, ref, rtol=1e-14, atol=1e-300)


def _exact_glu(X, W1, W3, W2, act, M, N, O, P):
    """Exact rational gated FFN for act in {NONE, RELU}, H rounded to bf16."""
    Y, Hs = [], []
    for i in range(M):
        h = []
        for j in range(O):
            g = sum((Fraction(X[i * N + n]) * Fraction(W1[n * O + j]) for n in range(N)), Fraction(0))
            u = sum((Fraction(X[i * N + n]) * Fraction(W3[n * O + j]) for n in range(N)), Fraction(0))
            if act == ACT_RELU and g < 0:
                g = Fraction(0)
            h.append(_frac_to_bf16(g * u))
        Hs.append(h)
        Y.append([sum((h[o] * Fraction(W2[o * P + k]) for o in range(O)), Fraction(0)) for k in range(P)])
    return Y, Hs


def _bf16_fracs(rng, count):
    raw = np.array([rng.uniform(-2, 2) for _ in range(count)], dtype=np.float32)
    return (raw.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64).tolist()


@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (2, 3, 4, 5), (5, 9, 13, 6)])
@pytest.mark.parametrize("act", [ACT_RELU, ACT_NONE])
def test_glu_brute_force_exact(shape, act):
    # ReGLU and the bilinear form are rational, so the exact answer is known;
    # the gate and linear operands get different matrices, so swapping them
    # (or the operand the activation goes on) fails
    M, N, O, P = shape
    rng = random.Random(sum(shape) * 17 + act)
    X, W1, W3, W2 = (_bf16_fracs(rng, c) for c in (M * N, N * O, N * O, O * P))
    want, want_h = _exact_glu(X, W1, W3, W2, act, M, N, O, P)
    Yo, Ho = oracle.glu_ffn(_u16_of_values(X).reshape(M, N), _u16_of_values(W1).reshape(N, O),
                            _u16_of_values(W3).reshape(N, O), _u16_of_values(W2).reshape(O, P),
                            act, want_h=True)
    for i in range(M):
        for j in range(O):
            assert oracle.bf16_to_f64(int(Ho[i, j])) == float(want_h[i][j])
        for k in range(P):
            w = float(want[i][k])
            assert abs(Yo[i, k] - w) <= 1e-12 * max(1.0, abs(w))


def test_swiglu_brute_force_python():
    # SiLU is transcendental: pure-Python loops with math.exp on a tiny case
    M, N, O, P = 3, 5, 7, 4
    rng = random.Random(99)
    X, W1, W3, W2 = (_bf16_fracs(rng, c) for c in (M * N, N * O, N * O, O * P))
    Yo = oracle.glu_ffn(_u16_of_values(X).reshape(M, N), _u16_of_values(W1).reshape(N, O),
                        _u16_of_values(W3).reshape(N, O), _u16_of_values(W2).reshape(O, P), ACT_SILU,
                        round_h=False)
    for i in range(M):
        h = []
        for j in range(O):
            g = math.fsum(X[i * N + n] * W1[n * O + j] for n in range(N))
            u = math.fsum(X[i * N + n] * W3[n * O + j] for n in range(N))
            h.append(g / (1.0 + math.exp(-g)) * u)
        for k in range(P):
            want = math.fsum(h[o] * W2[o * P + k] for o in range(O))
            assert abs(Yo[i, k] - want) <= 1e-13 * max(1.0, abs(want))


@pytest.mark.parametrize("act", [ACT_SILU, ACT_GELU_TANH, ACT_RELU])
def test_glu_with_unit_linear_branch_is_the_dense_ffn(act):
    # a column of ones in X selected by W3 makes X W3 == 1 everywhere: the
    # gated FFN is then the two-layer FFN with no biases, bit for bit
    M, N, O, P = 6, 16, 40, 12
    inp = synth.ffn_inputs(M, N, O, P, seed=31)
    X, W1, W2 = (synth.to_u16(t) for t in (inp.X, inp.W1, inp.W2))
    X = X.copy()
    X[:, 3] = 0x3F80                              # 1.0
    W3 = np.zeros((N, O), dtype=np.uint16)
    W3[3, :] = 0x3F80
    np.testing.assert_array_equal(oracle.glu_ffn(X, W1, W3, W2, act),
                                  oracle.ffn(X, W1, None, W2, None, act, ACT_NONE))


@pytest.mark.parametrize("G", [2, 4])
def test_glu_megatron_split_reproduces_unsplit(G):
    # W1 and W3 split by columns, W2 by rows: each H column depends on one
    # column of each, so the partial outputs sum to the unsplit result
    M, N, O, P = 5, 24, 64, 16
    a = synth.ffn_inputs(M, N, O, P, seed=40 + G)
    b = synth.ffn_inputs(M, N, O, P, seed=50 + G)
    X, W1, W2 = (synth.to_u16(t) for t in (a.X, a.W1, a.W2))
    W3 = synth.to_u16(b.W1)
    full = oracle.glu_ffn(X, W1, W3, W2, ACT_SILU)
    s = O // G
    acc = sum(oracle.glu_ffn(X, np.ascontiguousarray(W1[:, g * s:(g + 1) * s]),
                             np.ascontiguousarray(W3[:, g * s:(g + 1) * s]),
                             np.ascontiguousarray(W2[g * s:(g + 1) * s, :]), ACT_SILU) for g in range(G))
    np.testing.assert_allclose(acc, full, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- gated-expert MoE ----

def _glu_experts(E, N, O, P, seed):
    exps = [synth.glu_inputs(1, N, O, P, seed=seed + e) for e in range(E)]
    u = synth.to_u16
    return [u(g.W1) for g in exps], [u(g.W3) for g in exps], [u(g.W2) for g in exps]


def test_moe_glu_single_expert_is_the_gated_ffn():
    T, N, O, P = 9, 16, 24, 8
    X = synth.to_u16(synth.glu_inputs(T, N, O, P, seed=3).X)
    W1, W3, W2 = _glu_experts(1, N, O, P, seed=10)
    logits = np.zeros((T, 1), dtype=np.float32)
    np.testing.assert_array_equal(oracle.moe_glu_ffn(X, logits, 1, W1, W3, W2),
                                  oracle.glu_ffn(X, W1[0], W3[0], W2[0], ACT_SILU))


def test_moe_glu_top2_is_the_weighted_sum_of_two_gated_experts():
    T, N, O, P, E = 7, 16, 24, 8, 4
    X = synth.to_u16(synth.glu_inputs(T, N, O, P, seed=4).X)
    W1, W3, W2 = _glu_experts(E, N, O, P, seed=20)
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    got = oracle.moe_glu_ffn(X, logits, 2, W1, W3, W2)
    idx, w = oracle.moe_route(logits, 2)
    for t in range(T):
        want = sum(w[t, s] * oracle.glu_ffn(X[t:t + 1], W1[idx[t, s]], W3[idx[t, s]], W2[idx[t, s]], ACT_SILU)[0]
                   for s in range(2))
        np.testing.assert_allclose(got[t], want, rtol=1e-13, atol=1e-13)


def test_moe_glu_equal_gates_all_experts_is_their_mean():
    T, N, O, P, E = 5, 16, 24, 8, 3
    X = synth.to_u16(synth.glu_inputs(T, N, O, P, seed=6).X)
    W1, W3, W2 = _glu_experts(E, N, O, P, seed=30)
    got = oracle.moe_glu_ffn(X, np.zeros((T, E), dtype=np.float32), E, W1, W3, W2)
    want = sum(oracle.glu_ffn(X, W1[e], W3[e], W2[e], ACT_SILU) for e in range(E)) / E
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)
