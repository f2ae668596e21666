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
 *       outputs).
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
  QMM_DEV_BAD_EXPERT = 2u    /* topk_idx held an index outside [0, E); that
                                assignment contributed nothing              */
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
 * x: [M, K] fp32 or bf16 (x_dtype), y: [M, N] fp32.  The codes are
 * dequantised in registers inside the inner loop; accumulation in fp32.
 * M == 0 or N == 0 is a no-op.
 */
int qmm_linear(const void *x, int32_t x_dtype, int64_t M, const qmm_weight *w,
               float *y, qmm_stream_t stream);

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
 * E <= 1024, H % 4 == 0.
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
 * Every expert runs on the fp32 CUDA-core path (dequantisation in registers,
 * fp32 accumulation).
 */
int moe_ffn_forward(const void *x, int32_t x_dtype, int64_t M,
                    const int32_t *topk_idx, const float *topk_w, int32_t k,
                    const moe_experts *ex, void *y, int32_t y_dtype,
                    void *workspace, size_t workspace_bytes,
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
 * address (one-time set-up; make that first call before any stream capture).
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

/* Message for the last non-zero return on this thread ("" if none). */
const char *qmm_last_error(void);

/* Number of kernels this library has launched in this process. */
uint64_t qmm_launch_count(void);

/* Reads (and, if clear != 0, resets) the device status word of the current
 * device.  Synchronises the device.  Returns QMM_OK or QMM_ERR_CUDA. */
int qmm_device_status(uint32_t *status, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
