// moe_common.cuh -- shared pieces of the routed-expert kernels of the MoE layer on the CUDA cores:
// gate + up projections with the SwiGLU epilogue, and the down projection.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5:
// tokens routed to the same expert are gathered so the expert's weights are
// read once for all of them.  Work items are (expert with tokens, tile of
// weight rows); each warp streams its items' weight tiles through the
// bulk-copy pipeline of stream_tile.cuh and applies them to the expert's
// token list (1-4 tokens per pass).
#pragma once

#include <cstdint>

#include "stream_tile.cuh"

namespace qmm {
namespace moe {
using namespace tile;

// Expert metadata staged in shared memory after the copy slots: the list of
// experts with tokens and the token-list offsets (E <= 1024).
__device__ __forceinline__ void stage_meta(uint8_t *smem, const MoeWork &ws, int E, int &na,
                                           const int32_t *&s_active, const int32_t *&s_off) {
  int32_t *act = reinterpret_cast<int32_t *>(smem + kSmemBytes);
  int32_t *off = act + E;
  na = *ws.num_active;
  for (int i = threadIdx.x; i < na; i += blockDim.x) act[i] = ws.active[i];
  for (int i = threadIdx.x; i <= E; i += blockDim.x) off[i] = ws.offsets[i];
  __syncthreads();
  s_active = act;
  s_off = off;
}

// Loads one activation row into registers in the lane-owned chunk order of
// tile_dot_xr.
template <bool XBF16, int NCL, int CH>
__device__ __forceinline__ void load_xr(const void *row, int lane, float (&xr)[NCL][CH]) {
#pragma unroll
  for (int i = 0; i < NCL; ++i)
#pragma unroll
    for (int e = 0; e < CH; e += 4) {
      const float4 v = load_x4<XBF16>(row, (lane + 32 * i) * CH + e);
      xr[i][e] = v.x;
      xr[i][e + 1] = v.y;
      xr[i][e + 2] = v.z;
      xr[i][e + 3] = v.w;
    }
}

inline size_t meta_bytes(int E) { return static_cast<size_t>(2 * E + 1) * sizeof(int32_t); }

template <typename Kern>
cudaError_t prep_meta(Kern k, int E) {
  return ensure_smem(reinterpret_cast<const void *>(k),
                     static_cast<int>(kSmemBytes + meta_bytes(E)));
}

// Activation chunks per lane when a row of K values fits in registers (at
// most 128 floats per lane), else 0.
template <int BITS>
inline int ncl_for(int K) {
  constexpr int CH = (BITS == 8) ? 16 : 32;
  for (int n : {4, 2, 1})
    if (K == 32 * CH * n && n * CH <= 128) return n;
  return 0;
}

}  // namespace moe
}  // namespace qmm
