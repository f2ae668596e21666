// qmm_internal.h -- host-side interfaces between the C ABI layer (qmm_abi.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qmm {

// One quantised matrix family: E matrices [rows, cols] stacked with strides
// (a single matrix is E = 1).
struct QMat {
  const uint8_t *codes;
  int64_t codes_stride;   // bytes between experts
  const float *scales;
  const int32_t *zps;
  int64_t groups_stride;  // elements between experts
  int64_t rows, cols;
  int32_t bits, group;
};

// Workspace of the routed MoE layer (device pointers into the caller's
// buffer).
struct MoeWork {
  int32_t *counts;      // [E]
  int32_t *offsets;     // [E + 1]
  int32_t *active;      // [E] expert ids with at least one token, ascending
  int32_t *num_active;  // [1]
  int32_t *assign;      // [M*k] assignment ids a = m*k + i, grouped by expert
  int32_t *pos;         // [M*k] position of assignment a inside `assign`
  float *h;             // [M*k, I] SwiGLU activations (fp32)
  float *out;           // [M*k, H] per-assignment expert outputs (fp32)
  int32_t *tile_start;  // [E + 1] prefix of 128-token tiles per expert (light experts: none)
  int32_t *active_light;  // [E] experts with 1..light_max tokens, ascending
  int32_t *num_light;     // [1]
  __half *xg;           // [M*k, H] tokens in expert order, fp16 (tensor-core path)
  __half *hh;           // [M*k, I] SwiGLU activations, fp16 (tensor-core path)
  float *xs;            // [M*k] power of two that undoes the scaling of xg's row
  float *hs;            // [M*k] the same for hh's row
};

// Counts one kernel launch (for qmm_launch_count).
void count_launch();

// Launches `kernel` with programmatic stream serialization (see pdl_wait in
// qmm_device.cuh) and counts the launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  count_launch();
  return e;
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Device status word of the current device.
uint32_t *device_status();

// Raises a kernel's dynamic shared memory limit to at least `bytes` on the
// current device (the attribute is set once per kernel and device, not on
// every launch).
cudaError_t ensure_smem(const void *kernel, int bytes);

cudaError_t launch_quantize(const float *w, int64_t N, int64_t K, int bits, int group,
                            void *codes, float *scales, int32_t *zps, cudaStream_t s);

cudaError_t launch_gemv(const void *x, bool x_bf16, int64_t M, const QMat &w, void *y,
                        bool y_bf16, cudaStream_t s);

cudaError_t launch_router(const void *x, bool x_bf16, int64_t M, int64_t H,
                          const float *wr, const float *bias, int E, int k,
                          float *logits_scratch, int32_t *idx, float *w, int32_t *counts,
                          cudaStream_t s);

cudaError_t launch_moe_dispatch(const int32_t *idx, int64_t M, int k, int E, int light_max,
                                const MoeWork &ws, cudaStream_t s);

cudaError_t launch_moe_gateup(const void *x, bool x_bf16, int64_t M, int k, int E,
                              const QMat &gate, const QMat &up, const MoeWork &ws,
                              cudaStream_t s);

cudaError_t launch_moe_down(int64_t M, int k, int E, const QMat &down, const MoeWork &ws,
                            cudaStream_t s);

// Tensor-core (tcgen05) path of the routed experts for bf16 activations.
bool moe_tc_supported(const QMat &gate, const QMat &up, const QMat &down, int64_t H, int64_t I);
cudaError_t launch_moe_tc(const void *x, int64_t M, int k, int E, const QMat &gate, const QMat &up,
                          const QMat &down, const MoeWork &ws, cudaStream_t s);

// Linear layer with bf16 rows on the tensor cores (INT8, group >= 64):
// workspace bytes for M rows, and the launch (gather, GEMM with K splits,
// ordered reduction of the splits).
bool linear_tc_supported(const QMat &w);
// Timing of the tensor-core MoE GEMM launches (qmm_tc_timing).
cudaError_t tc_timing_enable(bool on);
cudaError_t tc_timing_read(float *gateup_ms, float *down_ms, bool *have);
size_t linear_tc_workspace_bytes(int64_t M, const QMat &w);
cudaError_t launch_linear_tc(const void *x, int64_t M, const QMat &w, void *y, bool y_bf16,
                             void *workspace, cudaStream_t s);

cudaError_t launch_moe_combine(int64_t M, int k, int64_t H, const float *topk_w,
                               const MoeWork &ws, void *y, bool y_bf16, cudaStream_t s);

}  // namespace qmm

namespace qmm {
// The routed MoE layer of a decode batch in one cooperative launch
// (moe_decode.cu): router, top-k, grouping, gate/up, down and combine.
// ws: the moe_ffn_forward workspace of (M, k); logits [M, E]; bar: one
// counter (zeroed by the launcher).  Outputs topk_idx / topk_w / counts
// may be NULL.
bool moe_decode_supported(const QMat &gate, const QMat &down, int64_t M, int E, int k, int64_t H,
                          int64_t I);
cudaError_t launch_moe_decode(const void *x, bool x_bf16, int64_t M, const float *wr,
                              const float *bias, int E, int k, const QMat &gate, const QMat &up,
                              const QMat &down, const MoeWork &ws, float *logits,
                              unsigned *bar, int32_t *topk_idx, float *topk_w, int32_t *counts,
                              void *y, bool y_bf16, cudaStream_t s);
}  // namespace qmm

namespace qmm {
// Decode attention (attn.cu): the RoPE table, and the steps between the
// projections (rotation, cache write and chunked softmax-weighted sums in
// one kernel, their merge in a second).  q, k, v: the projections
// (unrotated); part: [n_head, attn_chunks(pos + 1), head_dim + 2] fp32.
int attn_chunks(int64_t T);
cudaError_t launch_rope_table(int64_t max_seq, int head_dim, double base, float *cos_t,
                              float *sin_t, cudaStream_t s);
cudaError_t launch_attn_decode_core(const float *q, const float *k, const float *v, int n_head,
                                    int n_kv, int head_dim, int64_t max_seq, int64_t pos,
                                    const float *cos_t, const float *sin_t, float *cache,
                                    float *part, float *attn_out, cudaStream_t s);
}  // namespace qmm

namespace qmm {
// Rows of `copies` matrices (row = `rowbytes` of codes + G groups) one copy
// slot of the CUDA-core kernels holds per tile; 0 if a row does not fit.
int gemv_rows_per_tile(int64_t rowbytes, int64_t G, int copies);
// Bytes of router logits for M tokens and E experts.
size_t router_logits_bytes(int64_t M, int E);
// Largest token count and width the router takes (every size computed from
// them then fits in 64 bits and every grid in 2^31 blocks).
constexpr int64_t kMaxRouteTokens = 2147483647;
constexpr int64_t kMaxRouteWidth = int64_t(1) << 24;
}  // namespace qmm

namespace qmm {
// Small-M fused dequantise-matmul (1..8 activation rows per matrix, more in
// passes of 8): K in {2048, 4096}, group >= 64 with K / group a multiple of 4.
bool smallm_supported(int bits, int group, int64_t K);
cudaError_t launch_smallm_linear(const void *x, bool x_bf16, int64_t M, const QMat &w, void *y,
                                 bool y_bf16, cudaStream_t s);
// The routed experts on the small-M kernels, one token per pass (32
// columns per lane): decode batches, and the experts of a prefill batch with
// one or two tokens (two passes for two: the second reads the expert's tiles
// from L2, and still beats the two-token kernel on those experts).
// idx (decode batches, M k <= 128 assignments): the kernels group the
// assignments by expert themselves from the top-k indices instead of reading
// the dispatch kernel's lists; gate/up writes ws.pos for the combine.
cudaError_t launch_smallm_gateup(const void *x, bool x_bf16, int k, int E, const QMat &gate,
                                 const QMat &up, const MoeWork &ws, cudaStream_t s,
                                 const int32_t *idx = nullptr, int64_t MK = 0);
cudaError_t launch_smallm_down(int k, int E, const QMat &down, const MoeWork &ws, cudaStream_t s,
                               const int32_t *idx = nullptr, int64_t MK = 0);
}  // namespace qmm

namespace qmm {
// Sets this thread's qmm_last_error() message (printf-style; "" clears it).
void record_error(const char *fmt, ...);
// Routing load statistics over an expert histogram (E <= 1024).
cudaError_t launch_load_stats(const int32_t *counts, int E, int64_t threshold, int64_t *stats,
                              cudaStream_t s);
// One thread waiting on a barrier nothing completes, bounded by limit_ns.
cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t s);
}  // namespace qmm
