/*
 * tffn_oracle.c -- the CPU oracle for the fused Transformer FFN and its
 * Mixture-of-Experts form.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference arm of bench.py use it.  It shares no code, header,
 * table or constant with the CUDA library under transformer_ffn_gb300/.
 *
 * Plain, slow, single-threaded C99.  Inputs are bf16 bit patterns (uint16_t),
 * widened exactly to double; every sum is accumulated in double in ascending
 * index order; the hidden tensor H is rounded to bf16 (round to nearest, ties
 * to even) between the two layers, which is the precision the fused kernel
 * stores H in.  The output is returned in double, unrounded.
 *
 * What each function follows:
 *   ffn          "Kernel fusion and tensor parallelism" (brunomaga.github.io),
 *                section "Megatron-LM tensor parallelism", the FFN equation
 *                H = act(X W1 + b1), Y = act(H W2 + b2), with X in R^{MxN},
 *                W1 in R^{NxO}, b1 in R^O, W2 in R^{OxP}, b2 in R^P; the second
 *                activation optional.
 *   activations  The page names no formula.  GELU is the tanh form
 *                0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) of Hendrycks
 *                and Gimpel, "Gaussian Error Linear Units"; ReLU is max(x, 0).
 *   glu_ffn      "Kernel fusion and tensor parallelism", section "Results": a
 *                SwiGLU FFN has a third weight matrix whose product with the
 *                input gates the activation, and no biases.  Written out as in
 *                Shazeer, "GLU Variants Improve Transformer" (2020):
 *                H = act(X W1) * (X W3) elementwise, Y = H W2, with W1, W3 in
 *                R^{NxO}, W2 in R^{OxP}; SwiGLU takes act = SiLU (Swish with
 *                beta 1), x sigma(x) = x / (1 + exp(-x)).  H is rounded to bf16
 *                after the product, as in the two-layer FFN.
 *   moe_route    "Fine-Grained Compute-Communication Overlap for MoE" review
 *                (zhongzhuzhou.org), section 2.1: the router turns logits into a
 *                distribution over E experts and keeps the top k; the kept
 *                weights are renormalised to sum to one (softmax over the k
 *                kept logits).  Ties between equal logits go to the lower
 *                expert index.
 *   moe_permute  same page, section 4.2: rows grouped contiguously by expert;
 *                single-GPU order is (expert ascending, token ascending).
 *   moe_glu_ffn  moe_ffn with gated experts (each expert the glu_ffn above,
 *                no biases): the SwiGLU experts of the MoE models the
 *                fused-FFN page benchmarks.
 *   moe_ffn      same page, sections 2.1-2.2, steps 3 and 5: every kept
 *                expert runs the FFN above on the token; the layer output is
 *                the gate-weighted sum of those outputs.  Expert outputs are
 *                not rounded before the weighted sum.
 *
 * Parity pins: every function above is pinned by tests/test_oracle_pins.py
 * (brute force with exact rational arithmetic, closed forms, the Megatron
 * split identity, the linear-collapse identity, MoE invariants).
 */
#include "tffn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

double tffn_oracle_bf16_to_f64(uint16_t h)
{
    /* bf16 is the top half of an IEEE binary32; the widening is exact. */
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

uint16_t tffn_oracle_f64_to_bf16(double x)
{
    /*
     * Round a double straight to bf16 (8 significant bits, exponent range of
     * binary32), to nearest, ties to even.  No intermediate rounding to
     * binary32, so no double rounding.
     */
    if (isnan(x))
        return 0x7FC0;
    double ax = fabs(x);
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isinf(x))
        return sign | 0x7F80;
    if (ax == 0.0)
        return sign;

    /* ulp of bf16 at |x|: 2^(e-8) for |x| in [2^(e-1), 2^e); subnormals
     * (|x| < 2^-126) have the fixed ulp 2^-133. */
    int e;
    frexp(ax, &e);
    int ulp_exp = e - 8;
    if (ulp_exp < -133)
        ulp_exp = -133;
    double q = ldexp(ax, -ulp_exp);        /* exact: power-of-two scaling */
    double r = nearbyint(q);               /* default mode: nearest, ties to even */
    double v = ldexp(r, ulp_exp);          /* exact */
    if (v >= ldexp(1.0, 128))              /* overflow of the binary32 range */
        return sign | 0x7F80;
    float vf = (float)v;                   /* exact: v has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &vf, sizeof bits);
    return sign | (uint16_t)(bits >> 16);
}

/* --------------------------------------------------------- activations -- */

double tffn_oracle_act(int act, double x)
{
    switch (act) {
    case TFFN_ORACLE_ACT_NONE:
        return x;
    case TFFN_ORACLE_ACT_RELU:
        return x > 0.0 ? x : 0.0;
    case TFFN_ORACLE_ACT_GELU_TANH: {
        const double k0 = sqrt(2.0 / M_PI);
        const double k1 = 0.044715;
        return 0.5 * x * (1.0 + tanh(k0 * (x + k1 * x * x * x)));
    }
    case TFFN_ORACLE_ACT_SILU:
        /* x sigma(x); for x below about -745 exp(-x) overflows to +inf and
         * the quotient is -0, the limit of x sigma(x). */
        return x / (1.0 + exp(-x));
    default:
        return NAN;
    }
}

static int act_ok(int act)
{
    return act == TFFN_ORACLE_ACT_NONE || act == TFFN_ORACLE_ACT_RELU ||
           act == TFFN_ORACLE_ACT_GELU_TANH || act == TFFN_ORACLE_ACT_SILU;
}

static double bias_at(const uint16_t *b, int64_t j)
{
    return b ? tffn_oracle_bf16_to_f64(b[j]) : 0.0;
}

/* ----------------------------------------------------------------- FFN -- */

int tffn_oracle_ffn(const uint16_t *X, const uint16_t *W1, const uint16_t *b1,
                    const uint16_t *W2, const uint16_t *b2, int act1, int act2,
                    int64_t M, int64_t N, int64_t O, int64_t P,
                    const int64_t *rows, int64_t nrows, int round_h,
                    double *Y, uint16_t *H)
{
    if (!X || !W1 || !W2 || !Y || M < 0 || N < 1 || O < 1 || P < 1 ||
        !act_ok(act1) || !act_ok(act2))
        return -1;
    if (!rows)
        nrows = M;

    double *acc1 = malloc(sizeof(double) * (size_t)O);   /* one row of X W1 */
    double *hrow = malloc(sizeof(double) * (size_t)O);   /* one row of H    */
    double *acc2 = malloc(sizeof(double) * (size_t)P);   /* one row of H W2 */
    if (!acc1 || !hrow || !acc2) {
        free(acc1); free(hrow); free(acc2);
        return -2;
    }

    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) {
            free(acc1); free(hrow); free(acc2);
            return -1;
        }
        /* Layer 1: acc1[j] = sum_n X[i,n] W1[n,j], n ascending for every j.
         * The n loop is outermost so W1 is read row by row; each acc1[j]
         * still receives its terms in ascending n. */
        for (int64_t j = 0; j < O; ++j)
            acc1[j] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double x = tffn_oracle_bf16_to_f64(X[i * N + n]);
            const uint16_t *w = W1 + n * O;
            for (int64_t j = 0; j < O; ++j)
                acc1[j] += x * tffn_oracle_bf16_to_f64(w[j]);
        }
        /* H[i,j] = act1(acc1 + b1[j]), rounded to bf16 between the layers. */
        for (int64_t j = 0; j < O; ++j) {
            double h = tffn_oracle_act(act1, acc1[j] + bias_at(b1, j));
            if (round_h) {
                uint16_t hb = tffn_oracle_f64_to_bf16(h);
                if (H)
                    H[r * O + j] = hb;
                h = tffn_oracle_bf16_to_f64(hb);
            }
            hrow[j] = h;
        }
        /* Layer 2: acc2[k] = sum_o H[i,o] W2[o,k], o ascending. */
        for (int64_t k = 0; k < P; ++k)
            acc2[k] = 0.0;
        for (int64_t o = 0; o < O; ++o) {
            double h = hrow[o];
            const uint16_t *w = W2 + o * P;
            for (int64_t k = 0; k < P; ++k)
                acc2[k] += h * tffn_oracle_bf16_to_f64(w[k]);
        }
        /* Y = act2(acc2 + b2): the bias and the second activation come after
         * the full sum over the hidden dimension. */
        for (int64_t k = 0; k < P; ++k)
            Y[r * P + k] = tffn_oracle_act(act2, acc2[k] + bias_at(b2, k));
    }
    free(acc1); free(hrow); free(acc2);
    return 0;
}

/* ------------------------------------------------------------ gated FFN -- */

int tffn_oracle_glu_ffn(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                        const uint16_t *W2, int act, int64_t M, int64_t N, int64_t O,
                        int64_t P, const int64_t *rows, int64_t nrows, int round_h,
                        double *Y, uint16_t *H)
{
    if (!X || !W1 || !W3 || !W2 || !Y || M < 0 || N < 1 || O < 1 || P < 1 || !act_ok(act))
        return -1;
    if (!rows)
        nrows = M;

    double *gate = malloc(sizeof(double) * (size_t)O);   /* one row of X W1 */
    double *lin = malloc(sizeof(double) * (size_t)O);    /* one row of X W3 */
    double *acc2 = malloc(sizeof(double) * (size_t)P);   /* one row of H W2 */
    if (!gate || !lin || !acc2) {
        free(gate); free(lin); free(acc2);
        return -2;
    }
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= M) {
            free(gate); free(lin); free(acc2);
            return -1;
        }
        /* The two input products, each summed over n in ascending order. */
        for (int64_t j = 0; j < O; ++j) {
            gate[j] = 0.0;
            lin[j] = 0.0;
        }
        for (int64_t n = 0; n < N; ++n) {
            double x = tffn_oracle_bf16_to_f64(X[i * N + n]);
            const uint16_t *w1 = W1 + n * O;
            const uint16_t *w3 = W3 + n * O;
            for (int64_t j = 0; j < O; ++j) {
                gate[j] += x * tffn_oracle_bf16_to_f64(w1[j]);
                lin[j] += x * tffn_oracle_bf16_to_f64(w3[j]);
            }
        }
        /* H[i,j] = act(gate) * lin, rounded to bf16; reuse gate[] for H. */
        for (int64_t j = 0; j < O; ++j) {
            double h = tffn_oracle_act(act, gate[j]) * lin[j];
            if (round_h) {
                uint16_t hb = tffn_oracle_f64_to_bf16(h);
                if (H)
                    H[r * O + j] = hb;
                h = tffn_oracle_bf16_to_f64(hb);
            }
            gate[j] = h;
        }
        /* Y[i,k] = sum_o H[i,o] W2[o,k], o ascending; no bias, no second
         * activation. */
        for (int64_t k = 0; k < P; ++k)
            acc2[k] = 0.0;
        for (int64_t o = 0; o < O; ++o) {
            double h = gate[o];
            const uint16_t *w = W2 + o * P;
            for (int64_t k = 0; k < P; ++k)
                acc2[k] += h * tffn_oracle_bf16_to_f64(w[k]);
        }
        for (int64_t k = 0; k < P; ++k)
            Y[r * P + k] = acc2[k];
    }
    free(gate); free(lin); free(acc2);
    return 0;
}

/* ----------------------------------------------------------------- MoE -- */

int tffn_oracle_moe_route(const float *logits, int64_t T, int E, int k,
                          int32_t *topk_idx, double *topk_w)
{
    if (!logits || !topk_idx || T < 0 || E < 1 || k < 1 || k > E)
        return -1;
    int *taken = malloc(sizeof(int) * (size_t)E);
    if (!taken)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        for (int e = 0; e < E; ++e)
            taken[e] = 0;
        /* Selection: slot s receives the largest remaining logit; among equal
         * logits the lowest expert index wins (strict '>' scanning upward). */
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e;
            }
            taken[best] = 1;
            topk_idx[t * k + s] = best;
        }
        if (topk_w) {
            /* Softmax over all E logits, keep the top k, divide by the kept
             * mass.  Written as the softmax over the k kept logits, which is
             * the same quantity. */
            double lmax = (double)l[topk_idx[t * k + 0]];
            double sum = 0.0;
            for (int s = 0; s < k; ++s)
                sum += exp((double)l[topk_idx[t * k + s]] - lmax);
            for (int s = 0; s < k; ++s)
                topk_w[t * k + s] = exp((double)l[topk_idx[t * k + s]] - lmax) / sum;
        }
    }
    free(taken);
    return 0;
}

int tffn_oracle_moe_permute(const int32_t *topk_idx, int64_t T, int E, int k,
                            int32_t *perm, int32_t *expert_offsets)
{
    if (!topk_idx || !perm || !expert_offsets || T < 0 || E < 1 || k < 1)
        return -1;
    /* Rows grouped by expert, experts ascending; inside an expert, tokens
     * ascending (then slot ascending, which cannot tie since a token picks an
     * expert at most once).  perm[row] = t*k + s. */
    int64_t row = 0;
    for (int e = 0; e < E; ++e) {
        expert_offsets[e] = (int32_t)row;
        for (int64_t t = 0; t < T; ++t)
            for (int s = 0; s < k; ++s)
                if (topk_idx[t * k + s] == e)
                    perm[row++] = (int32_t)(t * k + s);
    }
    expert_offsets[E] = (int32_t)row;
    return row == T * k ? 0 : -3;
}

int tffn_oracle_moe_ffn(const uint16_t *X, const float *logits, int top_k,
                        const uint16_t *const *W1, const uint16_t *const *b1,
                        const uint16_t *const *W2, const uint16_t *const *b2,
                        int64_t T, int64_t N, int64_t O, int64_t P, int E,
                        int act1, int act2, const int64_t *tokens, int64_t ntok,
                        double *Y)
{
    if (!X || !logits || !W1 || !W2 || !Y || T < 0 || E < 1 || top_k < 1 ||
        top_k > E)
        return -1;
    if (!tokens)
        ntok = T;
    int32_t *idx = malloc(sizeof(int32_t) * (size_t)top_k);
    double *w = malloc(sizeof(double) * (size_t)top_k);
    double *ye = malloc(sizeof(double) * (size_t)P);
    if (!idx || !w || !ye) {
        free(idx); free(w); free(ye);
        return -2;
    }
    int rc = 0;
    for (int64_t r = 0; r < ntok && rc == 0; ++r) {
        int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) { rc = -1; break; }
        rc = tffn_oracle_moe_route(logits + t * E, 1, E, top_k, idx, w);
        for (int64_t c = 0; c < P; ++c)
            Y[r * P + c] = 0.0;
        for (int s = 0; s < top_k && rc == 0; ++s) {
            int e = idx[s];
            int64_t one = 0;
            /* The token's row alone, through expert e's FFN. */
            rc = tffn_oracle_ffn(X + t * N, W1[e], b1 ? b1[e] : NULL, W2[e],
                                 b2 ? b2[e] : NULL, act1, act2, 1, N, O, P,
                                 &one, 1, 1, ye, NULL);
            for (int64_t c = 0; c < P; ++c)
                Y[r * P + c] += w[s] * ye[c];
        }
    }
    free(idx); free(w); free(ye);
    return rc;
}

int tffn_oracle_moe_glu_ffn(const uint16_t *X, const float *logits, int top_k,
                            const uint16_t *const *W1, const uint16_t *const *W3,
                            const uint16_t *const *W2, int64_t T, int64_t N, int64_t O,
                            int64_t P, int E, int act, const int64_t *tokens, int64_t ntok,
                            double *Y)
{
    if (!X || !logits || !W1 || !W3 || !W2 || !Y || T < 0 || E < 1 || top_k < 1 ||
        top_k > E)
        return -1;
    if (!tokens)
        ntok = T;
    int32_t *idx = malloc(sizeof(int32_t) * (size_t)top_k);
    double *w = malloc(sizeof(double) * (size_t)top_k);
    double *ye = malloc(sizeof(double) * (size_t)P);
    if (!idx || !w || !ye) {
        free(idx); free(w); free(ye);
        return -2;
    }
    int rc = 0;
    for (int64_t r = 0; r < ntok && rc == 0; ++r) {
        int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) { rc = -1; break; }
        rc = tffn_oracle_moe_route(logits + t * E, 1, E, top_k, idx, w);
        for (int64_t c = 0; c < P; ++c)
            Y[r * P + c] = 0.0;
        for (int s = 0; s < top_k && rc == 0; ++s) {
            int e = idx[s];
            int64_t one = 0;
            /* The token's row alone, through expert e's gated FFN. */
            rc = tffn_oracle_glu_ffn(X + t * N, W1[e], W3[e], W2[e], act, 1, N, O, P,
                                     &one, 1, 1, ye, NULL);
            for (int64_t c = 0; c < P; ++c)
                Y[r * P + c] += w[s] * ye[c];
        }
    }
    free(idx); free(w); free(ye);
    return rc;
}
