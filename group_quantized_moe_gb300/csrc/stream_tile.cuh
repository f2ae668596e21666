// stream_tile.cuh -- the streaming-tile machinery shared by the CUDA-core
// fused dequantise-matmul kernels (qmm_linear and the routed-expert kernels).
//
// The operation is the one "Why I hand-wrote a DeepSeek inference engine in
// pure C" fuses in section 3.2: the codes are dequantised, (q - zp) * scale,
// inside the matmul's inner loop instead of materialising the fp32 weights.
//
// GB300 design (HBM-bound, one weight byte is used by at most a few tokens):
//  * Each warp streams its own weight tiles (RT full rows of W, contiguous in
//    HBM) into shared memory with 1-D bulk async copies (cp.async.bulk),
//    double buffered, completion tracked by one mbarrier per slot.  The same
//    transaction also brings the tile rows' scales and zero points (contiguous
//    [rows, G] blocks), so no dependent global load sits in the inner loop.
//    A slot holds up to 12 KB; with 8 warps per SM that keeps 96-192 KB of
//    reads in flight per SM, enough to cover HBM latency.
//  * Lanes read 16-byte code chunks from shared memory (consecutive lanes,
//    consecutive chunks: no bank conflicts).  A chunk (16 INT8 or 32 INT4
//    codes) never straddles a group, so its scale and zero point are read
//    once per chunk.
//  * Dequantisation in registers: byte_perm places each code under the
//    exponent byte 0x4B (value 2^23 + q), one packed f32x2 subtract of
//    2^23 + zp gives (q - zp) exactly, then packed f32x2 FMAs with the
//    activations.  The chunk's partial sum is scaled once: y += s * sum.
#pragma once

#include <cstdint>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace tile {

constexpr int kWarps = 8;
constexpr int kSlots = 2;
constexpr int kSlotBytes = 12288;
constexpr int kSmemBytes = kWarps * kSlots * kSlotBytes;

struct Pipe {
  uint32_t slot0;  // shared address of this warp's first slot
  uint32_t bar0;   // shared address of this warp's first mbarrier
};

__device__ __forceinline__ uint32_t slot_addr(const Pipe &p, int s) {
  return p.slot0 + s * kSlotBytes;
}
__device__ __forceinline__ uint32_t bar_addr(const Pipe &p, int s) { return p.bar0 + 8 * s; }

// Lays out this warp's slots and barriers and initialises the barriers.
__device__ __forceinline__ Pipe pipe_setup(uint8_t *smem, uint64_t (*bars)[kSlots], int warp,
                                           int lane) {
  Pipe p;
  p.slot0 = smem_addr(smem) + warp * kSlots * kSlotBytes;
  p.bar0 = smem_addr(&bars[warp][0]);
  if (lane == 0) {
    for (int s = 0; s < kSlots; ++s) mbar_init(bar_addr(p, s), 1);
    mbar_fence_init();
  }
  __syncwarp();
  return p;
}

// Waits (bounded) for every copy issued for iterations [from, to) whose item
// exists; used when giving up after a timeout so that no copy is still
// writing into shared memory when the warp exits.
template <typename Exists>
__device__ void drain(const Pipe &p, int64_t from, int64_t to, Exists exists, uint32_t *status) {
  for (int64_t j = from; j < to; ++j) {
    if (!exists(j)) continue;
    mbar_wait_bounded(bar_addr(p, static_cast<int>(j % kSlots)),
                      static_cast<uint32_t>((j / kSlots) & 1), status);
  }
}

// ---------------------------------------------------------------------------
// Where a tile row's scales and zero points are read from: shared memory
// (staged by the same bulk copy as the codes; needs G % 4 == 0 so that a
// [rows, G] block is a whole number of 16-byte units) or, for other shapes,
// global memory.
template <bool GSM>
struct GroupSrc {
  uint32_t s_sc, s_zp;       // shared addresses (GSM)
  const float *g_sc;         // global pointers (!GSM)
  const int32_t *g_zp;
  __device__ __forceinline__ float scale(int gi) const {
    if constexpr (GSM) return lds_f32(s_sc + 4 * gi);
    else return __ldg(g_sc + gi);
  }
  __device__ __forceinline__ int32_t zp(int gi) const {
    if constexpr (GSM) return lds_s32(s_zp + 4 * gi);
    else return __ldg(g_zp + gi);
  }
};

// Tile dot product: R weight rows (16-byte aligned rows of `rowbytes` bytes in
// shared memory starting at `tile`) against up to MT activation rows.
// yacc[r][m] += sum_k x_m[k] * (q_r[k] - zp_r[k/g]) * s_r[k/g]  (per lane,
// partial over this lane's chunks; reduced across the warp by the caller).
template <int BITS, int R, int MT, bool XBF16, bool GSM>
__device__ __forceinline__ void tile_dot(uint32_t tile, int rowbytes, int rows,
                                         const GroupSrc<GSM> (&gs)[R], int group_shift,
                                         const void *const (&xrow)[MT], int mt, int K, int lane,
                                         float (&yacc)[R][MT]) {
  constexpr int CH = (BITS == 8) ? 16 : 32;  // columns per 16-byte chunk
  const int nch = K / CH;
  for (int c = lane; c < nch; c += 32) {
    const int k0 = c * CH;
    const int gi = k0 >> group_shift;
    uint4 cw[R];
    float s[R];
    f32x2 mz[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < rows) {
        cw[r] = lds128(tile + r * rowbytes + c * 16);
        s[r] = gs[r].scale(gi);
        const float m = zp_magic(gs[r].zp(gi));
        mz[r] = pack2(m, m);
      } else {
        cw[r] = make_uint4(0, 0, 0, 0);
        s[r] = 0.0f;
        mz[r] = pack2(0.0f, 0.0f);
      }
    }
    f32x2 acc[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = 0ull;

    if constexpr (BITS == 8) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f32x2 d[R][2];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t w = j == 0 ? cw[r].x : j == 1 ? cw[r].y : j == 2 ? cw[r].z : cw[r].w;
          deq8_word(w, mz[r], d[r][0], d[r][1]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < mt) {
            const float4 xv = load_x4<XBF16>(xrow[m], k0 + 4 * j);
            const f32x2 x01 = pack2(xv.x, xv.y), x23 = pack2(xv.z, xv.w);
#pragma unroll
            for (int r = 0; r < R; ++r) {
              acc[r][m] = fma2(x01, d[r][0], acc[r][m]);
              acc[r][m] = fma2(x23, d[r][1], acc[r][m]);
            }
          }
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f32x2 d[R][4];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t w = j == 0 ? cw[r].x : j == 1 ? cw[r].y : j == 2 ? cw[r].z : cw[r].w;
          deq4_word(w, mz[r], d[r]);
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < mt) {
            const float4 xa = load_x4<XBF16>(xrow[m], k0 + 8 * j);
            const float4 xb = load_x4<XBF16>(xrow[m], k0 + 8 * j + 4);
            const f32x2 x0 = pack2(xa.x, xa.y), x1 = pack2(xa.z, xa.w);
            const f32x2 x2 = pack2(xb.x, xb.y), x3 = pack2(xb.z, xb.w);
#pragma unroll
            for (int r = 0; r < R; ++r) {
              acc[r][m] = fma2(x0, d[r][0], acc[r][m]);
              acc[r][m] = fma2(x1, d[r][1], acc[r][m]);
              acc[r][m] = fma2(x2, d[r][2], acc[r][m]);
              acc[r][m] = fma2(x3, d[r][3], acc[r][m]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        float a, b;
        unpack2(acc[r][m], a, b);
        yacc[r][m] = fmaf(s[r], a + b, yacc[r][m]);
      }
  }
}

// Decode (one activation row) with the row held in registers: lane l owns
// chunks l, l + 32, ..., l + 32 (NCL - 1) of every weight row for the whole
// kernel, so the inner loop has no activation loads and the NCL chunks are
// independent chains the scheduler can interleave.
template <int BITS, int R, int NCL, bool GSM>
__device__ __forceinline__ void tile_dot_xr(uint32_t tile, int rowbytes, int rows,
                                            const GroupSrc<GSM> (&gs)[R], int group_shift,
                                            const float (&xr)[NCL][BITS == 8 ? 16 : 32], int lane,
                                            float (&yacc)[R]) {
  constexpr int CH = (BITS == 8) ? 16 : 32;
#pragma unroll
  for (int i = 0; i < NCL; ++i) {
    const int c = lane + 32 * i;
    const int gi = (c * CH) >> group_shift;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r >= rows) continue;
      const uint4 cw = lds128(tile + r * rowbytes + c * 16);
      const float s = gs[r].scale(gi);
      const float m = zp_magic(gs[r].zp(gi));
      const f32x2 mz = pack2(m, m);
      f32x2 acc = 0ull;
      if constexpr (BITS == 8) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = j == 0 ? cw.x : j == 1 ? cw.y : j == 2 ? cw.z : cw.w;
          f32x2 d01, d23;
          deq8_word(w, mz, d01, d23);
          acc = fma2(pack2(xr[i][4 * j], xr[i][4 * j + 1]), d01, acc);
          acc = fma2(pack2(xr[i][4 * j + 2], xr[i][4 * j + 3]), d23, acc);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = j == 0 ? cw.x : j == 1 ? cw.y : j == 2 ? cw.z : cw.w;
          f32x2 d[4];
          deq4_word(w, mz, d);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            acc = fma2(pack2(xr[i][8 * j + 2 * t], xr[i][8 * j + 2 * t + 1]), d[t], acc);
        }
      }
      float a, b;
      unpack2(acc, a, b);
      yacc[r] = fmaf(s, a + b, yacc[r]);
    }
  }
}

template <int R, int MT>
__device__ __forceinline__ void zero_acc(float (&y)[R][MT]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) y[r][m] = 0.0f;
}

template <int R, int MT>
__device__ __forceinline__ void reduce_acc(float (&y)[R][MT]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) y[r][m] = warp_sum(y[r][m]);
}

// One matrix stream of a tile: RT rows of codes plus (GSM) their scales and
// zero points, at fixed offsets of the slot.
struct TileLayout {
  int rowbytes;   // bytes of codes per row
  int G;          // groups per row
  int codes_off;  // byte offsets inside the slot
  int sc_off;
  int zp_off;
};

// Issues the copies of `rows` rows starting at row n0 of one matrix.
template <bool GSM>
__device__ __forceinline__ uint32_t issue_rows(uint32_t slot, uint32_t bar, const TileLayout &L,
                                               const uint8_t *codes, const float *scales,
                                               const int32_t *zps, int64_t n0, int rows) {
  const uint32_t cb = static_cast<uint32_t>(rows * L.rowbytes);
  bulk_g2s(slot + L.codes_off, codes + n0 * L.rowbytes, cb, bar);
  if constexpr (GSM) {
    const uint32_t gb = static_cast<uint32_t>(rows * L.G * 4);
    bulk_g2s(slot + L.sc_off, scales + n0 * L.G, gb, bar);
    bulk_g2s(slot + L.zp_off, zps + n0 * L.G, gb, bar);
    return cb + 2 * gb;
  }
  return cb;
}

template <int R, bool GSM>
__device__ __forceinline__ void group_srcs(GroupSrc<GSM> (&gs)[R], int first, int count,
                                           uint32_t slot, const TileLayout &L,
                                           const float *scales, const int32_t *zps, int64_t n0,
                                           int rows) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r < first || r >= first + count) continue;
    const int rr = r - first;
    const int rc = rr < rows ? rr : 0;
    gs[r].s_sc = slot + L.sc_off + 4 * rc * L.G;
    gs[r].s_zp = slot + L.zp_off + 4 * rc * L.G;
    gs[r].g_sc = scales + (n0 + rc) * L.G;
    gs[r].g_zp = zps + (n0 + rc) * L.G;
  }
}

inline int log2i(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return s;
}

// Rows per tile (1, 2 or 4): as many rows (codes, plus scales and zero points
// when staged) of `copies` matrices as fit in one slot.
inline int rows_per_tile(int rowbytes, int G, bool gsm, int copies) {
  const int per_row = rowbytes + (gsm ? 8 * G : 0);
  const int fit = kSlotBytes / (per_row * copies);
  return fit >= 4 ? 4 : fit >= 2 ? 2 : fit;
}

// Slot layout for `copies` matrices of RT rows each.
inline void layouts(int rowbytes, int G, int RT, int copies, TileLayout *out) {
  const int codes = RT * rowbytes, groups = RT * G * 4;
  for (int c = 0; c < copies; ++c) {
    out[c].rowbytes = rowbytes;
    out[c].G = G;
    out[c].codes_off = c * codes;
    out[c].sc_off = copies * codes + c * groups;
    out[c].zp_off = copies * codes + copies * groups + c * groups;
  }
}

template <typename Kern>
cudaError_t prep(Kern k) {
  return ensure_smem(reinterpret_cast<const void *>(k), kSmemBytes);
}

}  // namespace tile
}  // namespace qmm
