/*
 * tffn_oracle.h -- declarations of the CPU oracle (test infrastructure only;
 * see tffn_oracle.c).  Shares nothing with the CUDA library's headers.
 */
#ifndef TFFN_ORACLE_H
#define TFFN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    TFFN_ORACLE_ACT_NONE = 0,
    TFFN_ORACLE_ACT_RELU = 1,
    TFFN_ORACLE_ACT_GELU_TANH = 2,
    TFFN_ORACLE_ACT_SILU = 3
};

double   tffn_oracle_bf16_to_f64(uint16_t h);
uint16_t tffn_oracle_f64_to_bf16(double x);
double   tffn_oracle_act(int act, double x);

/* Y[r, :] for the rows listed in rows[0..nrows) (all M rows when rows is
 * NULL); H (nullable) receives the bf16 hidden rows.  b1/b2 may be NULL
 * (zero).  round_h = 0 skips the bf16 rounding of H (identity tests only). */
int tffn_oracle_ffn(const uint16_t *X, const uint16_t *W1, const uint16_t *b1,
                    const uint16_t *W2, const uint16_t *b2, int act1, int act2,
                    int64_t M, int64_t N, int64_t O, int64_t P,
                    const int64_t *rows, int64_t nrows, int round_h,
                    double *Y, uint16_t *H);

/* Gated FFN: Y = (act(X W1) * (X W3)) W2 for the listed rows (all M when
 * rows is NULL); SwiGLU is act = SILU.  H (nullable) receives the bf16 rows. */
int tffn_oracle_glu_ffn(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                        const uint16_t *W2, int act, int64_t M, int64_t N, int64_t O,
                        int64_t P, const int64_t *rows, int64_t nrows, int round_h,
                        double *Y, uint16_t *H);

/* topk_idx[T*k], topk_w[T*k] (nullable) from fp32 logits[T*E]. */
int tffn_oracle_moe_route(const float *logits, int64_t T, int E, int k,
                          int32_t *topk_idx, double *topk_w);

/* perm[T*k] (row -> t*k+s) and expert_offsets[E+1]. */
int tffn_oracle_moe_permute(const int32_t *topk_idx, int64_t T, int E, int k,
                            int32_t *perm, int32_t *expert_offsets);

/* Y[r, :] for the tokens listed (all T when tokens is NULL). */
int tffn_oracle_moe_ffn(const uint16_t *X, const float *logits, int top_k,
                        const uint16_t *const *W1, const uint16_t *const *b1,
                        const uint16_t *const *W2, const uint16_t *const *b2,
                        int64_t T, int64_t N, int64_t O, int64_t P, int E,
                        int act1, int act2, const int64_t *tokens, int64_t ntok,
                        double *Y);

/* MoE with gated experts: expert e is glu_ffn(W1[e], W3[e], W2[e], act). */
int tffn_oracle_moe_glu_ffn(const uint16_t *X, const float *logits, int top_k,
                            const uint16_t *const *W1, const uint16_t *const *W3,
                            const uint16_t *const *W2, int64_t T, int64_t N, int64_t O,
                            int64_t P, int E, int act, const int64_t *tokens, int64_t ntok,
                            double *Y);

#ifdef __cplusplus
}
#endif
#endif
