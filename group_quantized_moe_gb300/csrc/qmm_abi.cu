// qmm_abi.cu -- the library's extern "C" entry points: argument validation on
// the host, workspace carving, kernel selection and launch on the caller's
// stream.  Declared in include/qmm.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "../../include/qmm.h"
#include "qmm_internal.h"

namespace qmm {
namespace {

thread_local char g_err[512] = "";
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
uint32_t *g_status_ptr[kMaxDevices] = {nullptr};
std::mutex g_mu;

// One status word per device (a module-scope device variable; its address on
// each device is looked up once).
__device__ uint32_t g_status_word;

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char *where) {
  return fail(QMM_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

bool group_ok(int g) { return g == 32 || g == 64 || g == 128 || g == 256; }

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

// Common checks of one quantised matrix (bits, group, shape).
int check_qshape(int bits, int group, int64_t rows, int64_t cols, const char *what) {
  if (bits != 8 && bits != 4) return fail(QMM_ERR_INVALID_ARG, "%s: bits must be 8 or 4 (got %d)", what, bits);
  if (!group_ok(group))
    return fail(QMM_ERR_UNSUPPORTED, "%s: group must be 32, 64, 128 or 256 (got %d)", what, group);
  if (rows < 0) return fail(QMM_ERR_SHAPE, "%s: negative row count", what);
  if (cols <= 0 || cols % group != 0)
    return fail(QMM_ERR_SHAPE, "%s: K=%lld must be a positive multiple of group %d", what,
                static_cast<long long>(cols), group);
  return QMM_OK;
}

}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void record_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

cudaError_t ensure_smem(const void *kernel, int bytes) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t key = reinterpret_cast<uintptr_t>(kernel) ^ (static_cast<uint64_t>(dev) << 56);
  std::lock_guard<std::mutex> lk(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[key] = bytes;
  return e;
}

int sm_count() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 1;
  if (g_sms[d] == 0) {
    int v = 1;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

uint32_t *device_status() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[d]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[d] = static_cast<uint32_t *>(p);
  }
  return g_status_ptr[d];
}

}  // namespace qmm

using namespace qmm;

extern "C" {

const char *qmm_last_error(void) { return g_err; }

uint64_t qmm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int qmm_tc_timing(int32_t enable) {
  cudaError_t e = tc_timing_enable(enable != 0);
  if (e != cudaSuccess) return cuda_fail(e, "qmm_tc_timing");
  return QMM_OK;
}

int qmm_tc_timing_ms(float *gateup_ms, float *down_ms) {
  if (!gateup_ms || !down_ms) return fail(QMM_ERR_INVALID_ARG, "qmm_tc_timing_ms: NULL output");
  bool have = false;
  cudaError_t e = tc_timing_read(gateup_ms, down_ms, &have);
  if (e != cudaSuccess) return cuda_fail(e, "qmm_tc_timing_ms");
  if (!have)
    return fail(QMM_ERR_INVALID_ARG,
                "qmm_tc_timing_ms: no tensor-core launch recorded since timing was enabled");
  return QMM_OK;
}

int qmm_device_status(uint32_t *status, int32_t clear) {
  if (!status) return fail(QMM_ERR_INVALID_ARG, "qmm_device_status: status is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "qmm_device_status");
  e = cudaMemcpyFromSymbol(status, g_status_word, sizeof(uint32_t));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_device_status");
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "qmm_device_status");
  }
  return QMM_OK;
}

int qmm_quantize_groupwise(const float *w, int64_t N, int64_t K, int32_t bits, int32_t group,
                           void *codes, float *scales, int32_t *zps, qmm_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_qshape(bits, group, N, K, "qmm_quantize_groupwise");
  if (rc) return rc;
  if (N == 0) return QMM_OK;
  if (!w || !codes || !scales || !zps)
    return fail(QMM_ERR_INVALID_ARG, "qmm_quantize_groupwise: null pointer");
  if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(zps))
    return fail(QMM_ERR_ALIGN, "qmm_quantize_groupwise: w, codes, scales and zps must be 16-byte aligned");
  cudaError_t e = launch_quantize(w, N, K, bits, group, codes, scales, zps,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_quantize_groupwise");
  return QMM_OK;
}

int qmm_linear(const void *x, int32_t x_dtype, int64_t M, const qmm_weight *w, void *y,
               int32_t y_dtype, qmm_stream_t stream) {
  g_err[0] = '\0';
  if (!w) return fail(QMM_ERR_INVALID_ARG, "qmm_linear: weight descriptor is NULL");
  int rc = check_qshape(w->bits, w->group, w->N, w->K, "qmm_linear");
  if (rc) return rc;
  if (x_dtype != QMM_F32 && x_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "qmm_linear: x_dtype must be QMM_F32 or QMM_BF16");
  if (y_dtype != QMM_F32 && y_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "qmm_linear: y_dtype must be QMM_F32 or QMM_BF16");
  if (M < 0) return fail(QMM_ERR_SHAPE, "qmm_linear: negative M");
  if (M == 0 || w->N == 0) return QMM_OK;
  if (!x || !y || !w->codes || !w->scales || !w->zps)
    return fail(QMM_ERR_INVALID_ARG, "qmm_linear: null pointer");
  if (!aligned16(x) || !aligned16(w->codes) || !aligned16(w->scales) || !aligned16(w->zps))
    return fail(QMM_ERR_ALIGN, "qmm_linear: x, codes, scales and zps must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(y) & (y_dtype == QMM_BF16 ? 1u : 3u)) != 0)
    return fail(QMM_ERR_ALIGN, "qmm_linear: y must be aligned to its element size");
  const int64_t rowbytes = w->K * w->bits / 8;
  if (gemv_rows_per_tile(rowbytes, w->K / w->group, 1) < 1)
    return fail(QMM_ERR_UNSUPPORTED, "qmm_linear: K=%lld is longer than one weight tile holds",
                static_cast<long long>(w->K));
  QMat q{static_cast<const uint8_t *>(w->codes), 0, w->scales, w->zps, 0, w->N, w->K,
         w->bits, w->group};
  cudaError_t e;
  // The small-M kernel (integer dot products, K split over the warps) for
  // 1..8 rows of the shapes it takes; the per-warp row kernel otherwise.
  const bool small = smallm_supported(w->bits, w->group, w->K) && M >= 1 && M <= 8;
  if (small)
    e = launch_smallm_linear(x, x_dtype == QMM_BF16, M, q, y, y_dtype == QMM_BF16,
                             static_cast<cudaStream_t>(stream));
  else
    e = launch_gemv(x, x_dtype == QMM_BF16, M, q, y, y_dtype == QMM_BF16,
                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_linear");
  return QMM_OK;
}

// Rows from which bf16 activations take the tensor-core linear path.
constexpr int64_t kLinearTcMinRows = 9;

size_t qmm_linear_batched_workspace_bytes(int64_t M, const qmm_weight *w) {
  if (!w || M < kLinearTcMinRows || M > 2147483647 || w->N <= 0 || w->K <= 0 || w->group <= 0)
    return 256;
  QMat q{static_cast<const uint8_t *>(w->codes), 0, w->scales, w->zps, 0, w->N, w->K,
         w->bits, w->group};
  if (!linear_tc_supported(q)) return 256;
  return linear_tc_workspace_bytes(M, q);
}

int qmm_linear_batched(const void *x, int32_t x_dtype, int64_t M, const qmm_weight *w, void *y,
                       int32_t y_dtype, void *workspace, size_t workspace_bytes,
                       qmm_stream_t stream) {
  g_err[0] = '\0';
  if (!w) return fail(QMM_ERR_INVALID_ARG, "qmm_linear_batched: weight descriptor is NULL");
  QMat q{static_cast<const uint8_t *>(w->codes), 0, w->scales, w->zps, 0, w->N, w->K,
         w->bits, w->group};
  const bool tc = x_dtype == QMM_BF16 && M >= kLinearTcMinRows && M <= 2147483647 &&
                  check_qshape(w->bits, w->group, w->N, w->K, "qmm_linear_batched") == QMM_OK &&
                  w->N > 0 && linear_tc_supported(q);
  g_err[0] = '\0';
  if (!tc)  // the CUDA-core paths of qmm_linear (the workspace is not used)
    return qmm_linear(x, x_dtype, M, w, y, y_dtype, stream);
  if (y_dtype != QMM_F32 && y_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "qmm_linear_batched: y_dtype must be QMM_F32 or QMM_BF16");
  if (!x || !y || !w->codes || !w->scales || !w->zps)
    return fail(QMM_ERR_INVALID_ARG, "qmm_linear_batched: null pointer");
  if (!aligned16(x) || !aligned16(w->codes) || !aligned16(w->scales) || !aligned16(w->zps))
    return fail(QMM_ERR_ALIGN, "qmm_linear_batched: x, codes, scales and zps must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(y) & (y_dtype == QMM_BF16 ? 1u : 3u)) != 0)
    return fail(QMM_ERR_ALIGN, "qmm_linear_batched: y must be aligned to its element size");
  const size_t need = linear_tc_workspace_bytes(M, q);
  if (!workspace || workspace_bytes < need)
    return fail(QMM_ERR_WORKSPACE, "qmm_linear_batched: workspace needs %zu bytes", need);
  if (!aligned256(workspace))
    return fail(QMM_ERR_ALIGN, "qmm_linear_batched: workspace must be 256-byte aligned");
  cudaError_t e = launch_linear_tc(x, M, q, y, y_dtype == QMM_BF16, workspace,
                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_linear_batched");
  return QMM_OK;
}

size_t moe_route_workspace_bytes(int64_t M, int32_t E) {
  if (M <= 0 || E <= 0) return 256;
  // sizes the router refuses (M >= 2^31 or E > 1024) cannot be given a
  // workspace: report the largest size so that no allocation succeeds
  if (M > kMaxRouteTokens || E > 1024) return SIZE_MAX;
  return round256(router_logits_bytes(M, E));
}

int moe_route_topk(const void *x, int32_t x_dtype, int64_t M, int64_t H, const float *w_router,
                   const float *bias, int32_t E, int32_t k, int32_t *topk_idx, float *topk_w,
                   int32_t *expert_counts, void *workspace, size_t workspace_bytes,
                   qmm_stream_t stream) {
  g_err[0] = '\0';
  if (x_dtype != QMM_F32 && x_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "moe_route_topk: x_dtype must be QMM_F32 or QMM_BF16");
  if (E < 1 || E > 1024) return fail(QMM_ERR_INVALID_ARG, "moe_route_topk: E must be in [1, 1024]");
  if (k < 1 || k > 16 || k > E)
    return fail(QMM_ERR_INVALID_ARG, "moe_route_topk: k must be in [1, min(E, 16)]");
  if (M < 0 || H <= 0 || H % 4 != 0)
    return fail(QMM_ERR_SHAPE, "moe_route_topk: need M >= 0 and H a positive multiple of 4");
  if (M > kMaxRouteTokens || H > kMaxRouteWidth)
    return fail(QMM_ERR_UNSUPPORTED, "moe_route_topk: need M < 2^31 and H <= 2^24");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {
    if (expert_counts) {
      cudaError_t e = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s);
      if (e != cudaSuccess) return cuda_fail(e, "moe_route_topk");
    }
    return QMM_OK;
  }
  if (!x || !w_router || !topk_idx || !topk_w)
    return fail(QMM_ERR_INVALID_ARG, "moe_route_topk: null pointer");
  if (!aligned16(x) || !aligned16(w_router))
    return fail(QMM_ERR_ALIGN, "moe_route_topk: x and w_router must be 16-byte aligned");
  if (!workspace || workspace_bytes < moe_route_workspace_bytes(M, E))
    return fail(QMM_ERR_WORKSPACE, "moe_route_topk: workspace needs %zu bytes",
                moe_route_workspace_bytes(M, E));
  if (!aligned256(workspace))
    return fail(QMM_ERR_ALIGN, "moe_route_topk: workspace must be 256-byte aligned");
  cudaError_t e = launch_router(x, x_dtype == QMM_BF16, M, H, w_router, bias, E, k,
                                static_cast<float *>(workspace), topk_idx, topk_w, expert_counts, s);
  if (e != cudaSuccess) return cuda_fail(e, "moe_route_topk");
  return QMM_OK;
}

int moe_route_load_stats(const int32_t *expert_counts, int32_t E, int64_t threshold,
                         int64_t *stats, qmm_stream_t stream) {
  g_err[0] = '\0';
  if (E < 1 || E > 1024) return fail(QMM_ERR_INVALID_ARG, "moe_route_load_stats: E must be in [1, 1024]");
  if (!expert_counts || !stats) return fail(QMM_ERR_INVALID_ARG, "moe_route_load_stats: null pointer");
  if ((reinterpret_cast<uintptr_t>(expert_counts) & 3u) || (reinterpret_cast<uintptr_t>(stats) & 7u))
    return fail(QMM_ERR_ALIGN, "moe_route_load_stats: counts and stats must be aligned to their elements");
  cudaError_t e = launch_load_stats(expert_counts, E, threshold, stats,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_route_load_stats");
  return QMM_OK;
}

int qmm_diag_wait_timeout(uint64_t limit_ns, qmm_stream_t stream) {
  g_err[0] = '\0';
  if (limit_ns < 1 || limit_ns > 10000000000ull)
    return fail(QMM_ERR_INVALID_ARG, "qmm_diag_wait_timeout: limit must be in [1 ns, 10 s]");
  cudaError_t e = launch_wait_timeout(limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_diag_wait_timeout");
  return QMM_OK;
}

}  // extern "C"

namespace {

int check_experts(const moe_experts *ex) {
  if (!ex) return fail(QMM_ERR_INVALID_ARG, "moe_experts descriptor is NULL");
  if (ex->E < 1 || ex->E > 1024) return fail(QMM_ERR_INVALID_ARG, "moe_experts: E must be in [1, 1024]");
  if (ex->H <= 0 || ex->I <= 0) return fail(QMM_ERR_SHAPE, "moe_experts: H and I must be positive");
  const qmm_expert_weights *m[3] = {&ex->gate, &ex->up, &ex->down};
  const char *names[3] = {"gate", "up", "down"};
  for (int i = 0; i < 3; ++i) {
    const int64_t rows = i < 2 ? ex->I : ex->H;
    const int64_t cols = i < 2 ? ex->H : ex->I;
    if (m[i]->rows != rows || m[i]->cols != cols)
      return fail(QMM_ERR_SHAPE, "moe_experts.%s: shape [%lld, %lld], expected [%lld, %lld]", names[i],
                  static_cast<long long>(m[i]->rows), static_cast<long long>(m[i]->cols),
                  static_cast<long long>(rows), static_cast<long long>(cols));
    int rc = check_qshape(m[i]->bits, m[i]->group, rows, cols, names[i]);
    if (rc) return rc;
    if (m[i]->bits != ex->gate.bits || m[i]->group != ex->gate.group)
      return fail(QMM_ERR_UNSUPPORTED, "moe_experts: gate, up and down must share bits and group");
    if (!m[i]->codes || !m[i]->scales || !m[i]->zps)
      return fail(QMM_ERR_INVALID_ARG, "moe_experts.%s: null pointer", names[i]);
    if ((cols / m[i]->group) % 4 != 0)
      return fail(QMM_ERR_UNSUPPORTED,
                  "moe_experts.%s: groups per row (%lld) must be a multiple of 4", names[i],
                  static_cast<long long>(cols / m[i]->group));
    if (!aligned16(m[i]->codes) || !aligned16(m[i]->scales) || !aligned16(m[i]->zps) ||
        m[i]->codes_stride % 16 != 0 || m[i]->groups_stride % 4 != 0)
      return fail(QMM_ERR_ALIGN, "moe_experts.%s: pointers and strides must be 16-byte aligned",
                  names[i]);
    if (m[i]->codes_stride < 0 || m[i]->groups_stride < 0)
      return fail(QMM_ERR_INVALID_ARG, "moe_experts.%s: negative stride", names[i]);
  }
  // Gate and up rows are staged together, two per copy slot.
  if (gemv_rows_per_tile(static_cast<int64_t>(ex->H) * ex->gate.bits / 8, ex->H / ex->gate.group, 2) < 1 ||
      gemv_rows_per_tile(static_cast<int64_t>(ex->I) * ex->down.bits / 8, ex->I / ex->down.group, 1) < 1)
    return fail(QMM_ERR_UNSUPPORTED, "moe_experts: rows too long for the expert kernels");
  return QMM_OK;
}

struct WsLayout {
  size_t counts, offsets, active, num_active, assign, pos, h, out, tile_start, xg, light,
      num_light, hh, xs, hs, total;
};

WsLayout ws_layout(int64_t M, int k, const moe_experts *ex) {
  WsLayout L;
  const size_t MK = static_cast<size_t>(M) * k;
  size_t o = 0;
  L.counts = o;     o += round256(sizeof(int32_t) * ex->E);
  L.offsets = o;    o += round256(sizeof(int32_t) * (ex->E + 1));
  L.active = o;     o += round256(sizeof(int32_t) * ex->E);
  L.num_active = o; o += 256;
  L.assign = o;     o += round256(sizeof(int32_t) * MK);
  L.pos = o;        o += round256(sizeof(int32_t) * MK);
  L.h = o;          o += round256(sizeof(float) * MK * ex->I);
  L.out = o;        o += round256(sizeof(float) * MK * ex->H);
  L.tile_start = o; o += round256(sizeof(int32_t) * (ex->E + 1));
  L.xg = o;         o += round256(2 * MK * ex->H);  // fp16 gathered tokens
  L.light = o;      o += round256(sizeof(int32_t) * ex->E);
  L.num_light = o;  o += 256;
  L.hh = o;         o += round256(2 * MK * ex->I);  // fp16 SwiGLU activations
  L.xs = o;         o += round256(sizeof(float) * MK);
  L.hs = o;         o += round256(sizeof(float) * MK);
  L.total = o;
  return L;
}

QMat qmat(const qmm_expert_weights &w) {
  return QMat{static_cast<const uint8_t *>(w.codes), w.codes_stride, w.scales, w.zps,
              w.groups_stride, w.rows, w.cols, w.bits, w.group};
}

}  // namespace

extern "C" {

size_t moe_ffn_workspace_bytes(int64_t M, int32_t k, const moe_experts *ex) {
  if (!ex || M < 0 || k < 1 || ex->E < 1) return 0;
  return ws_layout(M, k, ex).total;
}

int moe_ffn_forward(const void *x, int32_t x_dtype, int64_t M, const int32_t *topk_idx,
                    const float *topk_w, int32_t k, const moe_experts *ex, void *y,
                    int32_t y_dtype, void *workspace, size_t workspace_bytes,
                    qmm_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_experts(ex);
  if (rc) return rc;
  if (x_dtype != QMM_F32 && x_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "moe_ffn_forward: x_dtype must be QMM_F32 or QMM_BF16");
  if (y_dtype != QMM_F32 && y_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "moe_ffn_forward: y_dtype must be QMM_F32 or QMM_BF16");
  if (k < 1 || k > 16 || k > ex->E)
    return fail(QMM_ERR_INVALID_ARG, "moe_ffn_forward: k must be in [1, min(E, 16)]");
  if (M < 0) return fail(QMM_ERR_SHAPE, "moe_ffn_forward: negative M");
  if (M == 0) return QMM_OK;
  if (!x || !topk_idx || !topk_w || !y)
    return fail(QMM_ERR_INVALID_ARG, "moe_ffn_forward: null pointer");
  if (!aligned16(x) || !aligned16(y))
    return fail(QMM_ERR_ALIGN, "moe_ffn_forward: x and y must be 16-byte aligned");
  const WsLayout L = ws_layout(M, k, ex);
  if (!workspace || workspace_bytes < L.total)
    return fail(QMM_ERR_WORKSPACE, "moe_ffn_forward: workspace needs %zu bytes", L.total);
  if (!aligned256(workspace))
    return fail(QMM_ERR_ALIGN, "moe_ffn_forward: workspace must be 256-byte aligned");

  uint8_t *base = static_cast<uint8_t *>(workspace);
  MoeWork ws;
  ws.counts = reinterpret_cast<int32_t *>(base + L.counts);
  ws.offsets = reinterpret_cast<int32_t *>(base + L.offsets);
  ws.active = reinterpret_cast<int32_t *>(base + L.active);
  ws.num_active = reinterpret_cast<int32_t *>(base + L.num_active);
  ws.assign = reinterpret_cast<int32_t *>(base + L.assign);
  ws.pos = reinterpret_cast<int32_t *>(base + L.pos);
  ws.h = reinterpret_cast<float *>(base + L.h);
  ws.out = reinterpret_cast<float *>(base + L.out);
  ws.tile_start = reinterpret_cast<int32_t *>(base + L.tile_start);
  ws.xg = reinterpret_cast<__half *>(base + L.xg);
  ws.hh = reinterpret_cast<__half *>(base + L.hh);
  ws.xs = reinterpret_cast<float *>(base + L.xs);
  ws.hs = reinterpret_cast<float *>(base + L.hs);
  ws.active_light = reinterpret_cast<int32_t *>(base + L.light);
  ws.num_light = reinterpret_cast<int32_t *>(base + L.num_light);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool xb = x_dtype == QMM_BF16;
  // Decode batches (at most 8 tokens, so at most 8 per expert unless the
  // caller repeats an expert within a token) use the small-M kernels.
  const bool small_gu = M <= 8 && smallm_supported(ex->gate.bits, ex->gate.group, ex->H);
  const bool small_dn = M <= 8 && smallm_supported(ex->down.bits, ex->down.group, ex->I);
  const bool tc = xb && !small_gu && moe_tc_supported(qmat(ex->gate), qmat(ex->up), qmat(ex->down),
                                                             ex->H, ex->I);
  // On the tensor-core path, experts with one or two tokens skip the
  // dequantise -> fp16 -> MMA pipeline (a 16-row token tile for two tokens at
  // most) and stream their weights through the small-M integer kernels, one
  // token per pass (for two tokens the second pass reads the tiles from L2;
  // on the prefill workload this beat the two-tokens-per-pass kernel by 3.5 %
  // of the layer, and moving three- or four-token experts here lost 5-6 %).
  const int light_max = (tc && smallm_supported(ex->gate.bits, ex->gate.group, ex->H) &&
                         smallm_supported(ex->down.bits, ex->down.group, ex->I))
                            ? 2
                            : 0;
  // Decode batches on the small-M kernels group their (at most 128)
  // assignments themselves; everything else goes through the dispatch kernel.
  const bool self_grouped = !tc && small_gu && small_dn;
  cudaError_t e = cudaSuccess;
  if (!self_grouped) {
    e = launch_moe_dispatch(topk_idx, M, k, ex->E, light_max, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (dispatch)");
  }
  if (tc) {
    // bf16 activations: tensor-core grouped GEMMs (fp16 operands, fp32 accumulate)
    e = launch_moe_tc(x, M, k, ex->E, qmat(ex->gate), qmat(ex->up), qmat(ex->down), ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (tensor-core experts)");
    if (light_max > 0) {
      // the experts with one or two tokens (their rows of the fp32 h
      // buffer are disjoint from the tensor-core experts' rows)
      MoeWork wl = ws;
      wl.active = ws.active_light;
      wl.num_active = ws.num_light;
      e = launch_smallm_gateup(x, xb, k, ex->E, qmat(ex->gate), qmat(ex->up), wl, s);
      if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (few-token gate/up)");
      e = launch_smallm_down(k, ex->E, qmat(ex->down), wl, s);
      if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (few-token down)");
    }
  } else if (self_grouped) {
    const int64_t MK = M * k;
    e = launch_smallm_gateup(x, xb, k, ex->E, qmat(ex->gate), qmat(ex->up), ws, s, topk_idx, MK);
    if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (gate/up)");
    e = launch_smallm_down(k, ex->E, qmat(ex->down), ws, s, topk_idx, MK);
    if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (down)");
  } else {
    e = launch_moe_gateup(x, xb, M, k, ex->E, qmat(ex->gate), qmat(ex->up), ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (gate/up)");
    e = launch_moe_down(M, k, ex->E, qmat(ex->down), ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (down)");
  }
  e = launch_moe_combine(M, k, ex->H, topk_w, ws, y, y_dtype == QMM_BF16, s);
  if (e != cudaSuccess) return cuda_fail(e, "moe_ffn_forward (combine)");
  return QMM_OK;
}

}  // extern "C"

// ------------------------------------------------------- one-launch decode layer

extern "C" {

size_t moe_decode_workspace_bytes(int64_t M, int32_t k, const moe_experts *ex) {
  if (!ex || M < 1 || M > 8 || k < 1 || ex->E < 1) return 0;
  return ws_layout(M, k, ex).total + round256(sizeof(float) * M * ex->E) + 256;
}

int moe_decode_forward(const void *x, int32_t x_dtype, int64_t M, const float *w_router,
                       const float *bias, int32_t k, const moe_experts *ex, void *y,
                       int32_t y_dtype, int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                       void *workspace, size_t workspace_bytes, qmm_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_experts(ex);
  if (rc) return rc;
  if (x_dtype != QMM_F32 && x_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "moe_decode_forward: x_dtype must be QMM_F32 or QMM_BF16");
  if (y_dtype != QMM_F32 && y_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "moe_decode_forward: y_dtype must be QMM_F32 or QMM_BF16");
  if (k < 1 || k > 16 || k > ex->E)
    return fail(QMM_ERR_INVALID_ARG, "moe_decode_forward: k must be in [1, min(E, 16)]");
  if (M < 0) return fail(QMM_ERR_SHAPE, "moe_decode_forward: negative M");
  if (M == 0) return QMM_OK;
  if (!x || !w_router || !y)
    return fail(QMM_ERR_INVALID_ARG, "moe_decode_forward: null pointer");
  if (!aligned16(x) || !aligned16(y) || !aligned16(w_router))
    return fail(QMM_ERR_ALIGN, "moe_decode_forward: x, w_router and y must be 16-byte aligned");
  if (!moe_decode_supported(qmat(ex->gate), qmat(ex->down), M, ex->E, k, ex->H, ex->I))
    return fail(QMM_ERR_UNSUPPORTED,
                "moe_decode_forward: takes 1..8 tokens, E <= 256, H = 4096, I = 2048 and "
                "group >= 64 with H / group and I / group multiples of 4");
  const WsLayout L = ws_layout(M, k, ex);
  const size_t logits_off = L.total, bar_off = L.total + round256(sizeof(float) * M * ex->E);
  if (!workspace || workspace_bytes < bar_off + 256)
    return fail(QMM_ERR_WORKSPACE, "moe_decode_forward: workspace needs %zu bytes",
                bar_off + 256);
  if (!aligned256(workspace))
    return fail(QMM_ERR_ALIGN, "moe_decode_forward: workspace must be 256-byte aligned");
  uint8_t *base = static_cast<uint8_t *>(workspace);
  MoeWork ws{};
  ws.pos = reinterpret_cast<int32_t *>(base + L.pos);
  ws.h = reinterpret_cast<float *>(base + L.h);
  ws.out = reinterpret_cast<float *>(base + L.out);
  const cudaError_t e = launch_moe_decode(
      x, x_dtype == QMM_BF16, M, w_router, bias, ex->E, k, qmat(ex->gate), qmat(ex->up),
      qmat(ex->down), ws, reinterpret_cast<float *>(base + logits_off),
      reinterpret_cast<unsigned *>(base + bar_off), topk_idx, topk_w, expert_counts, y,
      y_dtype == QMM_BF16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_decode_forward");
  return QMM_OK;
}

}  // extern "C"

// ------------------------------------------------------------ decode attention

namespace {

struct AttnLayout {
  size_t q, k, v, attn, part, total;
};

AttnLayout attn_layout(const qmm_attn_layer *L) {
  AttnLayout a;
  const size_t nq = static_cast<size_t>(L->n_head) * L->head_dim;
  const size_t nk = static_cast<size_t>(L->n_head_kv) * L->head_dim;
  size_t o = 0;
  // q, k, v back to back (one linear layer fills all three when the weights
  // are stacked)
  a.q = o;
  a.k = a.q + 4 * nq;
  a.v = a.k + 4 * nk;
  o = round256(a.v + 4 * nk);
  a.attn = o; o += round256(4 * nq);
  a.part = o; o += round256(4 * static_cast<size_t>(L->n_head) * attn_chunks(L->max_seq) *
                            (L->head_dim + 2));
  a.total = o;
  return a;
}

int check_attn_layer(const qmm_attn_layer *L, const char *who) {
  if (!L) return fail(QMM_ERR_INVALID_ARG, "%s: layer descriptor is NULL", who);
  if (L->n_head < 1 || L->n_head_kv < 1 || L->n_head % L->n_head_kv != 0)
    return fail(QMM_ERR_INVALID_ARG, "%s: n_head must be a positive multiple of n_head_kv", who);
  if (L->head_dim < 4 || L->head_dim > 512 || L->head_dim % 4 != 0)
    return fail(QMM_ERR_UNSUPPORTED, "%s: head_dim must be a multiple of 4 in [4, 512]", who);
  if (L->max_seq < 1 || L->max_seq > (int64_t(1) << 31))
    return fail(QMM_ERR_INVALID_ARG, "%s: max_seq must be in [1, 2^31]", who);
  const int64_t nq = int64_t(L->n_head) * L->head_dim, nk = int64_t(L->n_head_kv) * L->head_dim;
  const int64_t D = L->wq.K;
  if (L->wq.N != nq || L->wk.N != nk || L->wv.N != nk || L->wk.K != D || L->wv.K != D ||
      L->wo.K != nq || L->wo.N < 1 || D < 1)
    return fail(QMM_ERR_SHAPE,
                "%s: need wq [n_head*head_dim, D], wk / wv [n_head_kv*head_dim, D], "
                "wo [D_out, n_head*head_dim]", who);
  if (!L->rope_cos || !L->rope_sin)
    return fail(QMM_ERR_INVALID_ARG, "%s: null RoPE table", who);
  return QMM_OK;
}

// Whether wk and wv follow wq in memory as rows of one [Nq + 2 Nk, D]
// matrix (codes, scales and zero points each contiguous, one scheme).
bool qkv_stacked(const qmm_attn_layer *L) {
  const qmm_weight &a = L->wq, &b = L->wk, &c = L->wv;
  if (a.bits != b.bits || a.bits != c.bits || a.group != b.group || a.group != c.group ||
      a.K != b.K || a.K != c.K || a.group <= 0)
    return false;
  const int64_t rb = a.K * a.bits / 8, G = a.K / a.group;
  auto at = [](const void *p, int64_t off) { return static_cast<const uint8_t *>(p) + off; };
  return b.codes == at(a.codes, a.N * rb) && c.codes == at(b.codes, b.N * rb) &&
         b.scales == a.scales + a.N * G && c.scales == b.scales + b.N * G &&
         b.zps == a.zps + a.N * G && c.zps == b.zps + b.N * G;
}

}  // namespace

extern "C" {

int qmm_rope_table(int64_t max_seq, int32_t head_dim, double base, float *cos_t, float *sin_t,
                   qmm_stream_t stream) {
  g_err[0] = '\0';
  if (max_seq < 1 || head_dim < 2 || head_dim % 2 != 0 || max_seq > (int64_t(1) << 31) ||
      head_dim > 65536)
    return fail(QMM_ERR_INVALID_ARG, "qmm_rope_table: need max_seq >= 1 and an even head_dim");
  if (!(base > 0.0)) return fail(QMM_ERR_INVALID_ARG, "qmm_rope_table: base must be positive");
  if (!cos_t || !sin_t) return fail(QMM_ERR_INVALID_ARG, "qmm_rope_table: null pointer");
  if ((reinterpret_cast<uintptr_t>(cos_t) & 3u) || (reinterpret_cast<uintptr_t>(sin_t) & 3u))
    return fail(QMM_ERR_ALIGN, "qmm_rope_table: tables must be 4-byte aligned");
  const cudaError_t e =
      launch_rope_table(max_seq, head_dim, base, cos_t, sin_t, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_rope_table");
  return QMM_OK;
}

size_t qmm_attn_decode_workspace_bytes(const qmm_attn_layer *L) {
  if (!L || L->n_head < 1 || L->n_head_kv < 1 || L->head_dim < 4 || L->head_dim > 512 ||
      L->max_seq < 1 || L->max_seq > (int64_t(1) << 31))
    return 0;
  return attn_layout(L).total;
}

int qmm_attn_decode(const void *x, int32_t x_dtype, int64_t pos, const qmm_attn_layer *L,
                    float *kv_cache, void *y, int32_t y_dtype, void *workspace,
                    size_t workspace_bytes, qmm_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_attn_layer(L, "qmm_attn_decode");
  if (rc) return rc;
  if (x_dtype != QMM_F32 && x_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "qmm_attn_decode: x_dtype must be QMM_F32 or QMM_BF16");
  if (y_dtype != QMM_F32 && y_dtype != QMM_BF16)
    return fail(QMM_ERR_INVALID_ARG, "qmm_attn_decode: y_dtype must be QMM_F32 or QMM_BF16");
  if (pos < 0 || pos >= L->max_seq)
    return fail(QMM_ERR_INVALID_ARG, "qmm_attn_decode: pos must be in [0, max_seq)");
  if (!x || !kv_cache || !y)
    return fail(QMM_ERR_INVALID_ARG, "qmm_attn_decode: null pointer");
  if (!aligned16(kv_cache))
    return fail(QMM_ERR_ALIGN, "qmm_attn_decode: kv_cache must be 16-byte aligned");
  const AttnLayout A = attn_layout(L);
  if (!workspace || workspace_bytes < A.total)
    return fail(QMM_ERR_WORKSPACE, "qmm_attn_decode: workspace needs %zu bytes", A.total);
  if (!aligned256(workspace))
    return fail(QMM_ERR_ALIGN, "qmm_attn_decode: workspace must be 256-byte aligned");
  uint8_t *base = static_cast<uint8_t *>(workspace);
  float *q = reinterpret_cast<float *>(base + A.q), *k = reinterpret_cast<float *>(base + A.k);
  float *v = reinterpret_cast<float *>(base + A.v);
  float *attn = reinterpret_cast<float *>(base + A.attn);
  float *part = reinterpret_cast<float *>(base + A.part);
  // the three projections, fused dequantised linear layers: one launch over
  // the stacked rows when the weights are stored as one matrix, else three
  if (qkv_stacked(L)) {
    qmm_weight w = L->wq;
    w.N = L->wq.N + L->wk.N + L->wv.N;
    rc = qmm_linear(x, x_dtype, 1, &w, q, QMM_F32, stream);
  } else {
    rc = qmm_linear(x, x_dtype, 1, &L->wq, q, QMM_F32, stream);
    if (rc == QMM_OK) rc = qmm_linear(x, x_dtype, 1, &L->wk, k, QMM_F32, stream);
    if (rc == QMM_OK) rc = qmm_linear(x, x_dtype, 1, &L->wv, v, QMM_F32, stream);
  }
  if (rc != QMM_OK) return rc;
  const cudaError_t e = launch_attn_decode_core(
      q, k, v, L->n_head, L->n_head_kv, L->head_dim, L->max_seq, pos, L->rope_cos, L->rope_sin,
      kv_cache, part, attn, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmm_attn_decode");
  // output projection
  return qmm_linear(attn, QMM_F32, 1, &L->wo, y, y_dtype, stream);
}

}  // extern "C"
