/*
 * Oracle for absorbed-MLA verify attention -- TEST INFRASTRUCTURE ONLY.
 * fp64 CPU reference used by the tests, the smoke check and the bench's CPU
 * baseline.  Shares no code with the CUDA library.
 *
 * Inputs are bf16 bit patterns (uint16), read exactly into fp64:
 *   q_nope [B, q, H, Dl], q_rope [B, q, H, Dr], kv [B, Smax, Dl+Dr]
 *   seq_lens [B] (prefix + q, q <= seq_lens[b] <= Smax)
 *   tree_mask [B, q, ceil(q/32)] uint32, bit j of row i: draft i sees draft j
 * Outputs are fp64: out [B, q, H, Dl], lse [B, q, H] (natural log).
 */
#ifndef MLA_ORACLE_H
#define MLA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { MLA_ORACLE_OK = 0, MLA_ORACLE_ERR_ARG = -1, MLA_ORACLE_ERR_SEQLEN = -2,
       MLA_ORACLE_ERR_ALLOC = -3 };

int mla_oracle_verify_attn(const uint16_t *q_nope, const uint16_t *q_rope, const uint16_t *kv,
                           const int32_t *seq_lens, const uint32_t *tree_mask, int B, int q, int H,
                           int Smax, int Dl, int Dr, double scale, double *out, double *lse,
                           int nthreads);

/* Same, for query rows [row_begin, row_begin + row_count) of the flattened
 * (b, i, h) order only; out/lse keep their full [B*q*H] indexing. */
int mla_oracle_verify_attn_rows(const uint16_t *q_nope, const uint16_t *q_rope,
                                const uint16_t *kv, const int32_t *seq_lens,
                                const uint32_t *tree_mask, int B, int q, int H, int Smax, int Dl,
                                int Dr, double scale, long row_begin, long row_count, double *out,
                                double *lse, int nthreads);

/* Unnormalised partial state over keys [k0[b], k1[b]) of each stream:
 * acc [B*q*H, Dl], m, l [B*q*H].  Empty window: acc = 0, m = -inf, l = 0. */
int mla_oracle_partial(const uint16_t *q_nope, const uint16_t *q_rope, const uint16_t *kv,
                       const int32_t *seq_lens, const uint32_t *tree_mask, int B, int q, int H,
                       int Smax, int Dl, int Dr, double scale, const int32_t *k0, const int32_t *k1,
                       double *acc, double *m, double *l, int nthreads);

/* Merge nsplit partial states laid out [nsplit][nrows](x Dl for acc). */
void mla_oracle_combine(const double *acc, const double *m, const double *l, int nsplit,
                        long nrows, int Dl, double *out, double *lse);

/* Normalised softmax weights of one query row over keys [0, Smax). */
int mla_oracle_row_weights(const uint16_t *q_nope, const uint16_t *q_rope, const uint16_t *kv,
                           const int32_t *seq_lens, const uint32_t *tree_mask, int B, int q, int H,
                           int Smax, int Dl, int Dr, double scale, int b, int i, int h,
                           double *weights);

#ifdef __cplusplus
}
#endif
#endif
