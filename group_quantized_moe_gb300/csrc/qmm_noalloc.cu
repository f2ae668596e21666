// qmm_noalloc.cu -- moe_route_topk_noalloc: the router without a caller
// workspace, for callers that cannot allocate device memory themselves.
//
// Some hosts of this library cannot create device allocations: their device
// memory belongs to someone else's allocator (an inference server's arena, a
// framework plugin that may only use buffers handed to it), or they run loops
// that must not pay for cudaMalloc and the device synchronisation it implies.
// Such callers still own their inputs and outputs but have no way to supply
// the router's scratch (the [M, E] fp32 logits).  This entry point keeps that
// scratch in a fixed-size array of device memory that belongs to the library
// itself: every GPU that loads the library holds it until the process exits.
//
// The array is shared by every call on a device and keeps the previous call's
// contents.  The router writes every logit it later reads, so nothing has to
// be cleared first; two calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race on the array and must be avoided.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/qmm.h"
#include "qmm_internal.h"

namespace qmm {
namespace {

// Largest M * E the allocation-free router accepts (1 MiB of fp32 logits).
constexpr int64_t kNoallocLogits = QMM_NOALLOC_MAX_LOGITS;

static __device__ __align__(256) float g_noalloc_logits[kNoallocLogits];

constexpr int kMaxDevices = 64;
std::atomic<float *> g_scratch_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device with that device current (in host code the array's name is only
// a host-side stand-in, not a device address).  Later calls read the cached
// address without taking the lock.  The address belongs to the device's
// primary context: after cudaDeviceReset it is stale, so a process that
// resets a device must not call this entry point on it again.
cudaError_t scratch_for_current_device(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  float *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      void *a = nullptr;
      e = cudaGetSymbolAddress(&a, g_noalloc_logits);
      if (e != cudaSuccess) return e;
      p = static_cast<float *>(a);
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace qmm

extern "C" {

int moe_route_topk_noalloc(const void *x, int32_t x_dtype, int64_t M, int64_t H,
                           const float *w_router, const float *bias, int32_t E, int32_t k,
                           int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                           qmm_stream_t stream) {
  // Same argument rules as moe_route_topk, plus the scratch size limit.
  qmm::record_error("");
  if (x_dtype != QMM_F32 && x_dtype != QMM_BF16) {
    qmm::record_error(
             "moe_route_topk_noalloc: x_dtype must be QMM_F32 or QMM_BF16");
    return QMM_ERR_INVALID_ARG;
  }
  if (E < 1 || E > 1024 || k < 1 || k > 16 || k > E) {
    qmm::record_error(
             "moe_route_topk_noalloc: need 1 <= E <= 1024 and 1 <= k <= min(E, 16)");
    return QMM_ERR_INVALID_ARG;
  }
  if (M < 0 || H <= 0 || H % 4 != 0) {
    qmm::record_error(
             "moe_route_topk_noalloc: need M >= 0 and H a positive multiple of 4");
    return QMM_ERR_SHAPE;
  }
  if (H > qmm::kMaxRouteWidth) {
    qmm::record_error("moe_route_topk_noalloc: need H <= 2^24");
    return QMM_ERR_UNSUPPORTED;
  }
  // M > limit / E rather than M * E > limit: the product of a huge M could
  // wrap around.
  if (M > qmm::kNoallocLogits / E) {
    qmm::record_error(
             "moe_route_topk_noalloc: M = %lld tokens times E = %d experts exceeds the "
             "built-in scratch of %lld logits; use moe_route_topk with a workspace",
             static_cast<long long>(M), E, static_cast<long long>(qmm::kNoallocLogits));
    return QMM_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0) {
    if (expert_counts) {
      cudaError_t e = cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, s);
      if (e != cudaSuccess) {
        qmm::record_error("moe_route_topk_noalloc: %s", cudaGetErrorString(e));
        return QMM_ERR_CUDA;
      }
    }
    return QMM_OK;
  }
  if (!x || !w_router || !topk_idx || !topk_w) {
    qmm::record_error(
             "moe_route_topk_noalloc: null pointer");
    return QMM_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w_router) & 15u)) {
    qmm::record_error(
             "moe_route_topk_noalloc: x and w_router must be 16-byte aligned");
    return QMM_ERR_ALIGN;
  }
  float *scratch = nullptr;
  cudaError_t e = qmm::scratch_for_current_device(&scratch);
  if (e == cudaSuccess)
    e = qmm::launch_router(x, x_dtype == QMM_BF16, M, H, w_router, bias, E, k, scratch, topk_idx,
                           topk_w, expert_counts, s);
  if (e != cudaSuccess) {
    qmm::record_error( "moe_route_topk_noalloc: %s",
             cudaGetErrorString(e));
    return QMM_ERR_CUDA;
  }
  return QMM_OK;
}

}  // extern "C"
