/*
 * qmm_oracle.h -- CPU oracle (test infrastructure only; see qmm_oracle.c).
 * Its own types: nothing here is shared with the CUDA library.
 */
#ifndef QMM_ORACLE_H
#define QMM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A quantised weight W[N,K]: codes int8 (stored q-128) [N*K] or packed uint8
 * [N*K/2] (low nibble = even column), scales fp32 [N, K/group], zps int32
 * [N, K/group]. */
typedef struct orc_qweight {
  int32_t bits, group;
  int64_t N, K;
  const void *codes;
  const float *scales;
  const int32_t *zps;
} orc_qweight;

int orc_quantize(const float *w, int64_t N, int64_t K, int bits, int group,
                 void *codes, float *scales, int32_t *zps);
int32_t orc_code_at(const orc_qweight *w, int64_t n, int64_t k);
void orc_dequantize(const orc_qweight *w, float *out);
void orc_linear_fused(const float *x, int64_t M, const orc_qweight *w, double *y);
void orc_linear_two_step(const float *x, int64_t M, const orc_qweight *w, double *y);
void orc_linear_bound(const float *x, int64_t M, const orc_qweight *w, double *bound);
void orc_router_logits(const float *x, int64_t M, int64_t H, const float *wr,
                       const float *bias, int32_t E, float *logits);
void orc_topk(const float *logits, int64_t M, int32_t E, int32_t k, int32_t *idx,
              float *w);
int orc_load_stats(const int32_t *idx, int64_t M, int32_t k, int32_t E,
                   int64_t threshold, int64_t *stats);
/* gate/up/down: arrays of E descriptors (only experts named in idx are read).
 * dw: bound on |w_gpu - w_oracle| of the routing weights (0 when both sides
 * use the same weights).  y and bound are [M, H] doubles. */
int orc_moe_ffn(const float *x, int64_t M, int64_t H, int64_t I,
                const int32_t *idx, const float *tw, int32_t k, int32_t E,
                const orc_qweight *gate, const orc_qweight *up,
                const orc_qweight *down, double dw, double *y, double *bound);

/* Decode attention [P1 section 3.4] (readings in qmm_oracle.c).  RoPE table
 * cos/sin [max_seq, head_dim/2] fp32; rope_apply rotates n_vec head vectors
 * (double) at position pos; attention: q [n_head*hd] double, caches fp32
 * [n_kv, max_seq, hd], rows t < T (row T-1 from k_last / v_last when they are
 * not NULL), bounds dq / dk_last / dv_last may be NULL; out, bound
 * [n_head*hd].  attn_decode: one token through q/k/v projections, RoPE, the
 * cache (cache_in [2][n_kv][max_seq][hd], rows < pos), attention over
 * 0..pos and the output projection; kv_new / kv_bound [2][n_kv*hd] (NULL
 * allowed) get the key/value row written at pos; y, bound [wo->N]. */
void orc_rope_table(int64_t max_seq, int32_t head_dim, double base, float *cos_t, float *sin_t);
void orc_rope_apply(const double *x, int32_t n_vec, int32_t head_dim, int64_t pos,
                    const float *cos_t, const float *sin_t, double *out);
void orc_attention(const double *q, const double *dq, const float *k_cache, const float *v_cache,
                   const double *k_last, const double *v_last, const double *dk_last,
                   const double *dv_last, int32_t n_head, int32_t n_kv, int32_t head_dim,
                   int64_t max_seq, int64_t T, double *out, double *bound);
int orc_attn_decode(const float *x, int64_t pos, int32_t n_head, int32_t n_kv, int32_t head_dim,
                    int64_t max_seq, const orc_qweight *wq, const orc_qweight *wk,
                    const orc_qweight *wv, const orc_qweight *wo, const float *cos_t,
                    const float *sin_t, const float *cache_in, double *kv_new, double *kv_bound,
                    double *y, double *bound);

#ifdef __cplusplus
}
#endif

#endif
