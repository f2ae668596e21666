// quantize.cu -- group-wise INT8 / INT4 quantiser.
//
// Follows the quantize_group routine of "Why I hand-wrote a DeepSeek inference
// engine in pure C" (section 3.2): per group of `group` consecutive columns of
// one row, scale = (max - min) / (2^bits - 1), zp = round(-min / scale),
// q = clamp(round(v / scale) + zp, 0, 2^bits - 1); INT8 stores q - 128, INT4
// packs two codes per byte (even column in the low nibble).
//
// GPU mapping: a group is owned by LPG = min(32, group/4) lanes, each lane
// holding group/LPG values loaded as float4 (fully coalesced 16-byte loads).
// min/max are reduced with xor shuffles inside the lane group; every lane then
// computes the same scale and zero point and writes its own codes (4 or 8
// bytes for INT8, 2 or 4 bytes for INT4).  The kernel is HBM-bound: it reads
// 4 bytes per weight and writes bits/8 bytes plus 8 bytes per group.
#include <climits>
#include <cstdint>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

// roundf (half away from zero) then a saturating conversion to int32.
__device__ __forceinline__ int32_t round_sat_i32(float v) {
  const float r = roundf(v);
  if (r != r) return 0;
  if (r >= 2147483648.0f) return INT_MAX;
  if (r <= -2147483648.0f) return INT_MIN;
  return static_cast<int32_t>(r);
}

template <int BITS, int GROUP>
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ w, int64_t N,
                                                       int64_t K, uint8_t *__restrict__ codes,
                                                       float *__restrict__ scales,
                                                       int32_t *__restrict__ zps) {
  // Waits for the preceding kernel but lets no successor start early: the
  // codes it writes may be read by a successor's early weight prefetch.
  pdl_wait();
  constexpr int LPG = (GROUP / 4) < 32 ? (GROUP / 4) : 32;  // lanes per group
  constexpr int VPL = GROUP / LPG;                          // values per lane
  constexpr int NV4 = VPL / 4;                              // float4 per lane
  constexpr int GPW = 32 / LPG;                             // groups per warp
  constexpr int32_t QMAX = (1 << BITS) - 1;

  const int lane = threadIdx.x & 31;
  const int sub = lane / LPG;   // which group of the warp
  const int sl = lane % LPG;    // lane inside the group
  const int64_t G = K / GROUP;
  const int64_t total_groups = N * G;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t gb = warp_id * GPW; gb < total_groups; gb += nwarps * GPW) {
    const int64_t gi = gb + sub;  // global group index = row * G + j
    const bool live = gi < total_groups;
    float v[VPL];
    float mn = 3.402823466e38f, mx = -3.402823466e38f;
    if (live) {
      // Element offset of this lane's values: lane-major inside the group so
      // that consecutive lanes read consecutive 16-byte words.
      const float *src = w + gi * GROUP;  // rows are contiguous: row*K + j*GROUP = gi*GROUP
#pragma unroll
      for (int t = 0; t < NV4; ++t) {
        const float4 f = ldg_f4(src + (t * LPG + sl) * 4);
        v[4 * t + 0] = f.x;
        v[4 * t + 1] = f.y;
        v[4 * t + 2] = f.z;
        v[4 * t + 3] = f.w;
      }
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        mn = fminf(mn, v[i]);
        mx = fmaxf(mx, v[i]);
      }
    }
#pragma unroll
    for (int o = LPG / 2; o >= 1; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    if (!live) continue;
    float s = __fdiv_rn(mx - mn, static_cast<float>(QMAX));
    if (s == 0.0f) {  // zero range: scale = max(|min|, |max|), or 1
      s = fmaxf(fabsf(mn), fabsf(mx));
      if (s == 0.0f) s = 1.0f;
    }
    const int32_t zp = round_sat_i32(__fdiv_rn(-mn, s));
    if (sl == 0) {
      scales[gi] = s;
      zps[gi] = zp;
    }
    int32_t q[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      int64_t t = static_cast<int64_t>(round_sat_i32(__fdiv_rn(v[i], s))) + zp;
      t = t < 0 ? 0 : (t > QMAX ? QMAX : t);
      q[i] = static_cast<int32_t>(t);
    }
    if constexpr (BITS == 8) {
      uint8_t *dst = codes + gi * GROUP;
#pragma unroll
      for (int t = 0; t < NV4; ++t) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) word |= (static_cast<uint32_t>(q[4 * t + b] - 128) & 0xFFu) << (8 * b);
        *reinterpret_cast<uint32_t *>(dst + (t * LPG + sl) * 4) = word;
      }
    } else {
      uint8_t *dst = codes + gi * (GROUP / 2);
#pragma unroll
      for (int t = 0; t < NV4; ++t) {
        const uint32_t lo = static_cast<uint32_t>(q[4 * t + 0] | (q[4 * t + 1] << 4));
        const uint32_t hi = static_cast<uint32_t>(q[4 * t + 2] | (q[4 * t + 3] << 4));
        *reinterpret_cast<uint16_t *>(dst + (t * LPG + sl) * 2) =
            static_cast<uint16_t>(lo | (hi << 8));
      }
    }
  }
}

template <int BITS, int GROUP>
cudaError_t launch_q(const float *w, int64_t N, int64_t K, void *codes, float *scales,
                     int32_t *zps, cudaStream_t s) {
  constexpr int LPG = (GROUP / 4) < 32 ? (GROUP / 4) : 32;
  constexpr int GPW = 32 / LPG;
  const int64_t groups = N * (K / GROUP);
  const int64_t warps_needed = (groups + GPW - 1) / GPW;
  int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(quantize_kernel<BITS, GROUP>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                    s, w, N, K, static_cast<uint8_t *>(codes), scales, zps);
}

}  // namespace

cudaError_t launch_quantize(const float *w, int64_t N, int64_t K, int bits, int group,
                            void *codes, float *scales, int32_t *zps, cudaStream_t s) {
#define QMM_Q_CASE(B, GR) \
  if (bits == B && group == GR) return launch_q<B, GR>(w, N, K, codes, scales, zps, s);
  QMM_Q_CASE(8, 32) QMM_Q_CASE(8, 64) QMM_Q_CASE(8, 128) QMM_Q_CASE(8, 256)
  QMM_Q_CASE(4, 32) QMM_Q_CASE(4, 64) QMM_Q_CASE(4, 128) QMM_Q_CASE(4, 256)
#undef QMM_Q_CASE
  return cudaErrorInvalidValue;
}

}  // namespace qmm
