/*
 * qmm.h -- C ABI of the group-wise quantised linear / routed MoE library
 * (libqmm.so, CUDA kernels for sm_103a).
 *
 * What the library computes is defined on three web pages:
 *  [P1] "Why I hand-wrote a DeepSeek inference engine in pure C" (hnwysp.cn,
 *       news 134870): section 2.3 (group-wise INT8/INT4 quantisation, group
 *       size 64/128, dequantise as (q - zero_point) * scale), section 3.2
 *       (quantize_group; dequantisation fused into the matmul inner loop; two
 *       INT4 codes per byte), section 3.3 (the matmul), section 3.4 (softmax
 *       with the maximum subtracted) and section 3.5 (MoE router = linear +
 *       softmax + top-k; tokens grouped by expert; weighted sum of expert
 *       outputs).  Section 3.4 also defines the decode attention step
 *       (rotary positions from a precomputed table, KV cache, softmax).
 *  [P2] "ds4 code walkthrough", Trace 2 (256 experts, 6 per token, width 4096)
 *       and Trace 3 (opaque C API style), the allocation guard (no allocation
 *       inside the generation loop).
 *  [P3] "I ran a 284B-parameter LLM from 3.2GB of RAM in plain C" (batched
 *       prefill with expert reuse is the missing piece).
 *
 * Conventions shared by every entry point:
 *  - Tensor pointers are DEVICE memory owned by the caller; the library never
 *    frees or keeps them.  Descriptor structs are HOST memory, read only during
 *    the call.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are detected on the host and returned
 *    before anything is enqueued.  Launch failures return QMM_ERR_CUDA.
 *    Conditions only visible on the device (an expert index out of range, a
 *    copy that never completed) set bits in the device status word, read with
 *    qmm_device_status().
 *  - Nothing here allocates device memory; scratch space is passed in by the
 *    caller (moe_ffn_forward's workspace).
 *  - On any non-zero return, qmm_last_error() gives a message (per thread).
 *  - Weight layout: W is [N, K] row-major (each output row's K inputs are
 *    contiguous).  Groups are `group` consecutive elements along K of one row;
 *    G = K / group groups per row.  INT8 codes are int8[N*K] holding q - 128;
 *    INT4 codes are uint8[N*K/2], byte j of a row holding column 2j in its low
 *    nibble and column 2j+1 in its high nibble.  scales are fp32 [N, G], zero
 *    points int32 [N, G].  The dequantised weight is (q - zp) * scale.
 *  - Supported: bits 8 or 4; group 32, 64, 128 or 256; K a positive multiple
 *    of group.  Codes, scales, zero points and activations must start on a
 *    16-byte boundary (QMM_ERR_ALIGN otherwise).
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
enum {
  QMM_OK = 0,
  QMM_ERR_INVALID_ARG = 1, /* null pointer, bad dtype, bad bits, k > E ... */
  QMM_ERR_SHAPE = 2,       /* K % group != 0, K == 0, mismatched sizes      */
  QMM_ERR_ALIGN = 3,       /* a pointer or stride is not 16-byte aligned    */
  QMM_ERR_WORKSPACE = 4,   /* workspace missing or too small                */
  QMM_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed          */
  QMM_ERR_UNSUPPORTED = 6  /* a valid configuration the library does not run */
};

/* Activation / output element types. */
enum { QMM_F32 = 0, QMM_BF16 = 1 };

/* Device status bits (qmm_device_status). */
enum {
  QMM_DEV_WAIT_TIMEOUT = 1u, /* an asynchronous copy or MMA did not complete
                                within the kernel's time limit; that kernel's
                                output is incomplete                        */
  QMM_DEV_BAD_EXPERT = 2u,   /* topk_idx held an index outside [0, E); that
                                assignment contributed nothing              */
  QMM_DEV_EXPERT_OVERLOAD = 4u /* moe_route_load_stats found an expert chosen
                                more often than its threshold             */
};

typedef void *qmm_stream_t; /* a cudaStream_t */

/* A quantised weight W[N, K] (device pointers, layout above). */
typedef struct qmm_weight {
  int32_t bits;          /* 8 or 4                                          */
  int32_t group;         /* elements per group along K                      */
  int64_t N, K;          /* output features, input features                 */
  const void *codes;     /* int8 [N*K] (q-128) or uint8 [N*K/2] (packed)     */
  const float *scales;   /* [N, K/group]                                    */
  const int32_t *zps;    /* [N, K/group]                                    */
} qmm_weight;

/*
 * Group-wise quantisation of w[N, K] (fp32, device) [P1 section 3.2].
 * Per group: mn = min, mx = max, s = (mx - mn) / (2^bits - 1) (fp32, IEEE
 * division); a zero range gives s = max(|mn|, |mx|), or 1 when that is 0;
 * zp = roundf(-mn / s); q = clamp(roundf(v / s) + zp, 0, 2^bits - 1) with
 * roundf = half away from zero, float->int conversions saturating to int32 and
 * the sum formed in 64 bits.  Writes codes / scales / zps in the layout above
 * (INT8 stores q - 128; INT4 packs the low nibble first).  Inputs must be
 * finite.
 */
int qmm_quantize_groupwise(const float *w, int64_t N, int64_t K, int32_t bits,
                           int32_t group, void *codes, float *scales,
                           int32_t *zps, qmm_stream_t stream);

/*
 * Fused dequantise-matmul [P1 sections 3.2-3.3]:
 *   y[m, n] = sum_k x[m, k] * (q[n, k] - zp[n, k/g]) * s[n, k/g]
 * x: [M, K] fp32 or bf16 (x_dtype), y: [M, N] fp32 or bf16 (y_dtype; a bf16
 * output is the fp32 result rounded to nearest even).  The codes are
 * dequantised in registers inside the inner loop; accumulation in fp32.
 * Error: fp32 rounding, of order 2^-24 relative to sum_k |x_k w^_k|; with one
 * or two rows and K in {2048, 4096} (integer byte dot products of the codes
 * with fixed-point activations) also the activations' representation: each
 * lane's slice of 16 or 32 activations is held to 2^-22 of its largest |x|,
 * or to 2^-38 when that largest exceeds 128 times the mean |x| around it (a
 * "massive" channel).  The library's tests hold every output to
 * 1e-5 * sum_k |x_k w^_k| + 1e-6.  A NaN or infinite activation gives NaN
 * outputs.  M == 0 or N == 0 is a no-op.
 */
int qmm_linear(const void *x, int32_t x_dtype, int64_t M, const qmm_weight *w,
               void *y, int32_t y_dtype, qmm_stream_t stream);

/*
 * The same linear layer for batches of rows [P1 sections 3.2-3.3; P3: reusing
 * each weight read for many tokens is the batched-prefill piece the pages'
 * engines lack].  With bf16 activations, M >= 9, INT8 codes, group >= 64,
 * K a multiple of 64 and K / group a multiple of 4, it runs on the tensor
 * cores: each row of x is copied to fp16 scaled by the power of two that
 * puts its largest |x| into [2^14, 2^15), each weight row is dequantised to
 * fp16 with its own power-of-two scale (inexact zero points as
 * (float)(q - zp) * s rounded once), fp32 accumulation, the K range split so
 * that every SM gets work and the splits' partial sums added in a fixed
 * order (results are reproducible bit for bit).  Accuracy: the fp16 operand
 * rounding, a relative L2 error per row within 1e-2 of the exact result.
 * Any other call is qmm_linear's (workspace unused).  N may be any positive
 * size.  workspace: device scratch of at least
 * qmm_linear_batched_workspace_bytes(M, w) bytes, 256-byte aligned (the fp16
 * rows and, with more than one split, the partial sums).
 */
size_t qmm_linear_batched_workspace_bytes(int64_t M, const qmm_weight *w);

int qmm_linear_batched(const void *x, int32_t x_dtype, int64_t M, const qmm_weight *w,
                       void *y, int32_t y_dtype, void *workspace, size_t workspace_bytes,
                       qmm_stream_t stream);

/*
 * MoE router [P1 sections 3.4-3.5]:
 *   logits[m, e] = sum_h x[m, h] * w_router[e, h]  (+ bias[e] when bias != NULL)
 * in fp32 with a fixed summation order: 128 partial sums (partial p takes
 * h = p, p+128, p+256, ... with one correctly rounded fma per term), the four
 * adjacent partials of each 32-partial lane added as (a + b) + (c + d), then a
 * halving tree t[l] = t[l] + t[l + o] for o = 16, 8, 4, 2, 1, then + bias.
 * topk_idx[m, :] = the k experts with the largest logits, larger first, equal
 * logits -> lower index first.  topk_w[m, i] = softmax probability of expert
 * topk_idx[m, i] renormalised over the k selected experts (sums to 1).
 * expert_counts (optional, [E] int32): number of tokens that selected each
 * expert.  x: [M, H] fp32 or bf16; w_router: [E, H] fp32; bias: [E] fp32 or
 * NULL.  workspace: device scratch of at least moe_route_workspace_bytes(M, E)
 * bytes (holds the logits), 256-byte aligned.  Requires 1 <= k <= min(E, 16),
 * E <= 1024, H % 4 == 0, M < 2^31 and H <= 2^24 (moe_route_workspace_bytes
 * returns SIZE_MAX for sizes beyond these).
 */
size_t moe_route_workspace_bytes(int64_t M, int32_t E);

int moe_route_topk(const void *x, int32_t x_dtype, int64_t M, int64_t H,
                   const float *w_router, const float *bias, int32_t E,
                   int32_t k, int32_t *topk_idx, float *topk_w,
                   int32_t *expert_counts, void *workspace,
                   size_t workspace_bytes, qmm_stream_t stream);

/* E quantised matrices of one shape [rows, cols], stacked: expert e's codes
 * start at codes + e * codes_stride (bytes), its scales / zps at
 * scales + e * groups_stride, zps + e * groups_stride (elements). */
typedef struct qmm_expert_weights {
  int32_t bits, group;
  int64_t rows, cols;
  const void *codes;
  int64_t codes_stride;   /* bytes between experts, multiple of 16          */
  const float *scales;
  const int32_t *zps;
  int64_t groups_stride;  /* elements between experts, multiple of 4        */
} qmm_expert_weights;

/* The routed experts of one MoE layer: E experts, width H, inner width I.
 * gate and up are [I, H] per expert, down is [H, I]; all three share bits and
 * group, and H / group and I / group must be multiples of 4 (each tile's
 * scales and zero points are copied as whole 16-byte units). */
typedef struct moe_experts {
  int32_t E;
  int32_t H, I;
  qmm_expert_weights gate, up, down;
} moe_experts;

/* Bytes of device workspace moe_ffn_forward needs for M tokens, k slots. */
size_t moe_ffn_workspace_bytes(int64_t M, int32_t k, const moe_experts *ex);

/*
 * Routed SwiGLU MoE feed-forward layer [P1 section 3.5; P2 Trace 2]:
 *   y[m, :] = sum_{i<k} topk_w[m, i] * FFN_{topk_idx[m, i]}(x[m, :])
 *   FFN_e(v) = Wd_e . (silu(Wg_e . v) * (Wu_e . v)),  silu(a) = a / (1 + e^-a)
 * Tokens are first grouped by expert (each expert's weights are then read
 * once for all its tokens).  x: [M, H] fp32 or bf16; y: [M, H] fp32 or bf16
 * (y_dtype).  topk_idx / topk_w: [M, k] as produced by moe_route_topk.
 * workspace: device scratch of at least moe_ffn_workspace_bytes(M, k, ex)
 * bytes, 256-byte aligned; its contents on entry do not matter.
 *
 * Which arithmetic runs (all of it on the GPU):
 *  - fp32 activations, any M, and bf16 activations with M <= 8 (decode): the
 *    CUDA-core kernels, codes dequantised in registers, fp32 accumulation;
 *    every output is within 1e-5 * sum |x w^| + 1e-6 per linear stage of the
 *    exact result (propagated through SwiGLU and the weighted sum).
 *  - bf16 activations with M > 8 and INT8 experts (batched prefill, H and I
 *    multiples of 128, group >= 64, gate and up with the same groups_stride):
 *    experts with three or more tokens run on the tensor cores with fp16
 *    operands and fp32 accumulation.  Each token
 *    row, each SwiGLU row and each weight row is scaled by its own power of
 *    two so that its largest magnitude lies in [2^14, 2^15) (no overflow,
 *    fp16's full 11-bit precision for every value within 2^28 of its row's
 *    largest, for tokens and weights of any fp32 magnitude); groups whose
 *    zero point lies outside [-1793, 1024] (q - zp not exact in fp16) are
 *    dequantised as (float)(q - zp) * s rounded once to fp16.  Accuracy: per
 *    token row a relative L2 error within 1e-2 of the exact result (the
 *    operands' fp16 rounding, about 2^-11 relative per value).  Experts
 *    with one or two tokens in such a batch run on the CUDA-core kernels.
 *  - bf16 activations with M > 8 whose experts do not qualify: the CUDA-core
 *    kernels, with the fp32 bound of the first case.
 */
int moe_ffn_forward(const void *x, int32_t x_dtype, int64_t M,
                    const int32_t *topk_idx, const float *topk_w, int32_t k,
                    const moe_experts *ex, void *y, int32_t y_dtype,
                    void *workspace, size_t workspace_bytes,
                    qmm_stream_t stream);

/*
 * Rotary-position table [P1 section 3.4: RoPE rotates pairs of Q/K
 * dimensions by position-dependent angles, from a cos/sin table
 * [max_seq_len, head_dim/2] precomputed once]:
 *   cos_t[p, i] = cos(p * base^(-2i / head_dim)),  sin_t[p, i] = sin(...)
 * for 0 <= p < max_seq, 0 <= i < head_dim / 2, evaluated in double and
 * rounded to fp32.  The page gives no base; 10000 is the usual one.
 * cos_t, sin_t: device, fp32 [max_seq, head_dim / 2].  head_dim even.
 */
int qmm_rope_table(int64_t max_seq, int32_t head_dim, double base, float *cos_t, float *sin_t,
                   qmm_stream_t stream);

/* One attention layer for decoding (device pointers in the weights and
 * tables).  Query heads n_head, key/value heads n_head_kv (n_head a multiple
 * of it: query head h reads key/value head h / (n_head / n_head_kv)),
 * head_dim a multiple of 4 in [4, 512], max_seq cache rows (<= 2^31).
 * wq [n_head * head_dim, D], wk and wv [n_head_kv * head_dim, D],
 * wo [D_out, n_head * head_dim]: quantised weights as for qmm_linear.
 * rope_cos / rope_sin: tables from qmm_rope_table for max_seq and head_dim. */
typedef struct qmm_attn_layer {
  int32_t n_head, n_head_kv, head_dim;
  int64_t max_seq;
  qmm_weight wq, wk, wv, wo;
  const float *rope_cos, *rope_sin;
} qmm_attn_layer;

/* Bytes of device workspace qmm_attn_decode needs (0 for an invalid layer). */
size_t qmm_attn_decode_workspace_bytes(const qmm_attn_layer *L);

/*
 * One decode step of an attention layer for one token at position pos
 * [P1 section 3.4], with the projections as fused dequantised linear layers
 * (qmm_linear):
 *   q = x Wq^T, k = x Wk^T, v = x Wv^T (fp32);
 *   pairs (2i, 2i+1) of every head of q and k rotated by the angles of row pos
 *   of the table: (a, b) -> (a cos - b sin, a sin + b cos);
 *   kv_cache row pos <- rotated k (keys) and v (values);
 *   for each query head: s_t = q . k_t / sqrt(head_dim) over rows 0..pos,
 *   p = softmax(s) with the maximum subtracted first, o = sum_t p_t v_t;
 *   y = o Wo^T.
 * kv_cache: device fp32 [2][n_head_kv][max_seq][head_dim] (keys, then values:
 * one layer of the page's [layers, 2, heads, max_seq, head_dim] cache),
 * 16-byte aligned; rows < pos must hold the earlier steps' keys and values,
 * rows > pos are neither read nor written.  x: [D] fp32 or bf16; y: [D_out]
 * fp32 or bf16.  workspace: device scratch of qmm_attn_decode_workspace_bytes
 * bytes, 256-byte aligned; contents on entry do not matter.  The softmax is
 * split over chunks of 64 rows whose partial results are merged in a fixed
 * order (results reproducible bit for bit).  Accuracy: fp32 arithmetic; the
 * tests hold every stage to 1e-5 * sum |terms| + 1e-6 and propagate it to y.
 * Requires 0 <= pos < max_seq.  When wk and wv follow wq in memory as rows of
 * one [(n_head + 2 n_head_kv) head_dim, D] matrix (codes, scales and zero
 * points each contiguous, same bits and group), the three projections run as
 * one launch: three kernel launches in all (else five), one more when
 * pos >= 512 (the chunks' merge), asynchronous on `stream`.
 */
int qmm_attn_decode(const void *x, int32_t x_dtype, int64_t pos, const qmm_attn_layer *L,
                    float *kv_cache, void *y, int32_t y_dtype, void *workspace,
                    size_t workspace_bytes, qmm_stream_t stream);

/*
 * The routed MoE layer of a decode batch in one launch [P1 section 3.5: the
 * router, the grouping of tokens by expert and the experts' weighted sum as
 * one step]: computes exactly what moe_route_topk followed by
 * moe_ffn_forward compute (the same fixed-order logits, so the same expert
 * indices, weights and histogram bit for bit; the same expert arithmetic),
 * as one cooperative kernel whose phases (logits, top-k, grouping, gate/up,
 * down, combine) are separated by grid-wide barriers instead of launches.
 * Takes 1..8 tokens, E <= 256, H = 4096, I = 2048 (the decode shape of the
 * DeepSeek layer this library targets), INT8 or INT4 experts with
 * group >= 64 and H / group, I / group multiples of 4; anything else
 * returns QMM_ERR_UNSUPPORTED (use the two calls).  x: [M, H] fp32 or bf16;
 * w_router [E, H] fp32, bias [E] or NULL; y: [M, H] fp32 or bf16.
 * topk_idx [M, k] int32, topk_w [M, k] fp32 and expert_counts [E] int32 are
 * optional outputs (NULL to skip).  workspace: moe_decode_workspace_bytes
 * bytes, 256-byte aligned, contents on entry do not matter (a counter in it
 * is cleared by an asynchronous memset before the kernel).  Every barrier
 * wait is bounded (QMM_DEV_WAIT_TIMEOUT on expiry).  Needs all of its CTAs
 * resident at once (two per SM): it returns QMM_ERR_CUDA if the device
 * cannot hold them.
 */
size_t moe_decode_workspace_bytes(int64_t M, int32_t k, const moe_experts *ex);

int moe_decode_forward(const void *x, int32_t x_dtype, int64_t M, const float *w_router,
                       const float *bias, int32_t k, const moe_experts *ex, void *y,
                       int32_t y_dtype, int32_t *topk_idx, float *topk_w,
                       int32_t *expert_counts, void *workspace, size_t workspace_bytes,
                       qmm_stream_t stream);

/*
 * Allocation-free router (no counterpart on the pages: it is a calling
 * convention, not part of the method).  Computes exactly what moe_route_topk
 * computes, with the same arguments minus the workspace, for callers that
 * cannot create device allocations themselves -- hosts whose device memory is
 * owned by another allocator (a serving arena, a framework plugin limited to
 * the buffers it is handed) or loops that must not pay for cudaMalloc and its
 * implicit synchronisation.  The caller still passes all inputs and outputs.
 * The logits scratch is a fixed array of device memory inside the library,
 * QMM_NOALLOC_MAX_LOGITS fp32 values (1 MiB), which every GPU that loads the
 * library holds until the process exits; M * E above that limit returns
 * QMM_ERR_WORKSPACE.  The first call on a device looks up the array's device
 * address (one-time set-up; make that first call before any stream capture;
 * after cudaDeviceReset the looked-up address is stale, so do not call this
 * entry point again on a device the process has reset).
 * All calls on a device share the array and it keeps the last call's
 * contents (every value read is written first, so nothing needs clearing);
 * calls whose kernels may overlap on the GPU race on it.  Nothing here calls
 * cudaMalloc, cudaFree or any allocating routine.
 */
#define QMM_NOALLOC_MAX_LOGITS 262144

int moe_route_topk_noalloc(const void *x, int32_t x_dtype, int64_t M, int64_t H,
                           const float *w_router, const float *bias, int32_t E,
                           int32_t k, int32_t *topk_idx, float *topk_w,
                           int32_t *expert_counts, qmm_stream_t stream);

/*
 * Routing load statistics [P1 section 3.5, last paragraph: grouped expert
 * work degrades towards serial when one expert gets most tokens, so the
 * engine checks how often each expert was chosen and warns above a
 * threshold].  Reads expert_counts[E] (device, int32, e.g. the histogram
 * moe_route_topk writes) and writes stats[4] (device, int64): the largest
 * count, its expert (the lowest index among equal counts), the number of
 * experts with at least one token and the sum of the counts (M * k for a
 * histogram of M tokens and k slots).  The imbalance of the routing is
 * stats[0] * stats[2] / stats[3] (largest over mean count per touched
 * expert).  When the largest count exceeds `threshold`, QMM_DEV_EXPERT_OVERLOAD
 * is set in the device status word.  Requires 1 <= E <= 1024; asynchronous on
 * `stream`.
 */
int moe_route_load_stats(const int32_t *expert_counts, int32_t E, int64_t threshold,
                         int64_t *stats, qmm_stream_t stream);

/*
 * Diagnostic of the library's bounded waits (no counterpart on the pages).
 * Launches one kernel whose single thread waits on a barrier that nothing
 * completes, using the same bounded wait as the library's kernels but with a
 * limit of limit_ns (1 ns .. 10 s; the kernels themselves use 2 s).  When the
 * limit passes, the wait gives up, QMM_DEV_WAIT_TIMEOUT is set in the device
 * status word and the kernel returns; nothing else is in flight, so the
 * device stays usable.  It shows that an expired wait is reported rather than
 * hanging the GPU.
 */
int qmm_diag_wait_timeout(uint64_t limit_ns, qmm_stream_t stream);

/* Message for the last non-zero return on this thread ("" if none). */
const char *qmm_last_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t qmm_launch_count(void);

/*
 * Timing of the tensor-core prefill GEMMs (a profiling aid; no counterpart on
 * the pages).  After qmm_tc_timing(1), every moe_ffn_forward on the current
 * device that takes the tensor-core path records CUDA events owned by the
 * library around its gate/up GEMM launch and around its down GEMM launch (the
 * launches then no longer overlap the tails of the kernels before them);
 * qmm_tc_timing(0) stops it.  qmm_tc_timing_ms waits for the events of the
 * last such call and returns the two launches' durations in milliseconds;
 * QMM_ERR_INVALID_ARG if no call was recorded since timing was enabled.
 * Not for concurrent use from several threads' streams (one set of events).
 */
int qmm_tc_timing(int32_t enable);
int qmm_tc_timing_ms(float *gateup_ms, float *down_ms);

/* Reads (and, if clear != 0, resets) the device status word of the current
 * device.  Synchronises the device.  Returns QMM_OK or QMM_ERR_CUDA. */
int qmm_device_status(uint32_t *status, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
