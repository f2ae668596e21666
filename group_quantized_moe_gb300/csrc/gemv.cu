// gemv.cu -- fused dequantise-matmul for decode-sized batches (CUDA cores) and
// the routed-expert kernels built on it.
//
// The operation is the one "Why I hand-wrote a DeepSeek inference engine in
// pure C" fuses in section 3.2: the codes are dequantised, (q - zp) * scale,
// inside the matmul's inner loop instead of materialising the fp32 weights.
// Section 3.5 of the same article gives the expert grouping used by the MoE
// kernels here (gather the tokens of one expert, then read its weights once).
//
// GB300 design (HBM-bound, one weight byte is used by at most a few tokens):
//  * Each warp streams its own weight tiles (RT full rows of W, contiguous in
//    HBM) into shared memory with 1-D bulk async copies (cp.async.bulk),
//    double buffered, completion tracked by one mbarrier per slot.  A tile is
//    one copy of up to 8 KB; with 8 warps per SM that keeps 64-128 KB of reads
//    in flight per SM, enough to cover HBM latency.
//  * Lanes read 16-byte code chunks from shared memory (consecutive lanes,
//    consecutive chunks: no bank conflicts).  A chunk (16 INT8 or 32 INT4
//    codes) never straddles a group, so its scale and zero point are read
//    once per chunk.
//  * Dequantisation in registers: byte_perm places each code under the
//    exponent byte 0x4B (value 2^23 + q), one packed f32x2 subtract of
//    2^23 + zp gives (q - zp) exactly, then packed f32x2 FMAs with the
//    activations.  The chunk's partial sum is scaled once: y += s * sum.
//  * Activations are read with 16-byte read-only loads (L1-resident: at most
//    a few rows of K floats).  Each activation load feeds RT weight rows.
//  * Grid = one block of 8 warps per SM; tiles are dealt round-robin over all
//    warps of the grid.
#include <cstdint>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kWarps = 8;
constexpr int kSlots = 2;
constexpr int kSlotBytes = 8192;
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
// Tile dot product: R weight rows (16-byte aligned rows of `rowbytes` bytes in
// shared memory starting at `tile`) against up to MT activation rows.
// yacc[r][m] += sum_k x_m[k] * (q_r[k] - zp_r[k/g]) * s_r[k/g]  (per lane,
// partial over this lane's chunks; reduced across the warp by the caller).
template <int BITS, int R, int MT, bool XBF16>
__device__ __forceinline__ void tile_dot(uint32_t tile, int rowbytes, int rows,
                                         const float *const (&scp)[R],
                                         const int32_t *const (&zpp)[R], int group_shift,
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
        s[r] = __ldg(scp[r] + gi);
        const float m = zp_magic(__ldg(zpp[r] + gi));
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

// ---------------------------------------------------------------------------
// qmm_linear: y[M, N] = x[M, K] . deq(W)^T.  Tile = RT rows of W.
struct GemvArgs {
  const void *x;
  int64_t M;
  const uint8_t *codes;
  const float *scales;
  const int32_t *zps;
  int64_t N;
  int K;
  int G;
  int group_shift;
  int rowbytes;
  float *y;
  uint32_t *status;
};

template <int BITS, int RT, int MT, bool XBF16>
__global__ void __launch_bounds__(kWarps * 32, 1) gemv_kernel(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Pipe p = pipe_setup(smem, bars, warp, lane);

  const int64_t ntiles = (a.N + RT - 1) / RT;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  auto tile_of = [&](int64_t it) { return gw + it * nw; };
  auto exists = [&](int64_t it) { return tile_of(it) < ntiles; };
  auto issue = [&](int64_t it) {
    const int64_t t = tile_of(it);
    const int64_t n0 = t * RT;
    const int rows = static_cast<int>(min64(RT, a.N - n0));
    const uint32_t bytes = static_cast<uint32_t>(rows * a.rowbytes);
    const int s = static_cast<int>(it % kSlots);
    mbar_arrive_expect_tx(bar_addr(p, s), bytes);
    bulk_g2s(slot_addr(p, s), a.codes + n0 * a.rowbytes, bytes, bar_addr(p, s));
  };

  if (lane == 0)
    for (int s = 0; s < kSlots; ++s)
      if (exists(s)) issue(s);

  for (int64_t it = 0; exists(it); ++it) {
    const int s = static_cast<int>(it % kSlots);
    if (!mbar_wait_bounded(bar_addr(p, s), static_cast<uint32_t>((it / kSlots) & 1), a.status)) {
      drain(p, it + 1, it + kSlots, exists, a.status);
      return;
    }
    const int64_t n0 = tile_of(it) * RT;
    const int rows = static_cast<int>(min64(RT, a.N - n0));
    const float *scp[RT];
    const int32_t *zpp[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int64_t n = n0 + (r < rows ? r : 0);
      scp[r] = a.scales + n * a.G;
      zpp[r] = a.zps + n * a.G;
    }
    for (int64_t m0 = 0; m0 < a.M; m0 += MT) {
      const int mt = static_cast<int>(min64(MT, a.M - m0));
      const void *xrow[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int64_t mm = m0 + (m < mt ? m : 0);
        xrow[m] = XBF16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.x) + mm * a.K)
                        : static_cast<const void *>(static_cast<const float *>(a.x) + mm * a.K);
      }
      float yacc[RT][MT];
      zero_acc(yacc);
      tile_dot<BITS, RT, MT, XBF16>(slot_addr(p, s), a.rowbytes, rows, scp, zpp, a.group_shift,
                                    xrow, mt, a.K, lane, yacc);
      reduce_acc(yacc);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (r < rows && m < mt) a.y[(m0 + m) * a.N + n0 + r] = yacc[r][m];
      }
    }
    __syncwarp();
    if (lane == 0 && exists(it + kSlots)) {
      fence_proxy_async_smem();
      issue(it + kSlots);
    }
  }
}

// ---------------------------------------------------------------------------
// Routed experts, gate + up projections with the SwiGLU epilogue.
// Work item = (active expert, RT rows of gate and the same RT rows of up).
struct GateUpArgs {
  const void *x;  // [M, H]
  int k;
  QMat gate, up;  // [I, H] per expert
  int group_shift;
  int rowbytes;   // H * bits / 8
  int G;          // H / group
  MoeWork ws;
  uint32_t *status;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <int BITS, int RT, int MT, bool XBF16>
__global__ void __launch_bounds__(kWarps * 32, 1) moe_gateup_kernel(GateUpArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Pipe p = pipe_setup(smem, bars, warp, lane);

  const int I = static_cast<int>(a.gate.rows);
  const int H = static_cast<int>(a.gate.cols);
  const int tiles_per_expert = (I + RT - 1) / RT;
  const int64_t nitems = static_cast<int64_t>(*a.ws.num_active) * tiles_per_expert;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  auto item_of = [&](int64_t it) { return gw + it * nw; };
  auto exists = [&](int64_t it) { return item_of(it) < nitems; };
  auto issue = [&](int64_t it) {
    const int64_t item = item_of(it);
    const int e = a.ws.active[item / tiles_per_expert];
    const int n0 = static_cast<int>(item % tiles_per_expert) * RT;
    const int rows = min(RT, I - n0);
    const uint32_t bytes = static_cast<uint32_t>(rows * a.rowbytes);
    const int s = static_cast<int>(it % kSlots);
    mbar_arrive_expect_tx(bar_addr(p, s), 2 * bytes);
    bulk_g2s(slot_addr(p, s), a.gate.codes + e * a.gate.codes_stride + int64_t(n0) * a.rowbytes,
             bytes, bar_addr(p, s));
    bulk_g2s(slot_addr(p, s) + RT * a.rowbytes,
             a.up.codes + e * a.up.codes_stride + int64_t(n0) * a.rowbytes, bytes,
             bar_addr(p, s));
  };

  if (lane == 0)
    for (int s = 0; s < kSlots; ++s)
      if (exists(s)) issue(s);

  for (int64_t it = 0; exists(it); ++it) {
    const int s = static_cast<int>(it % kSlots);
    if (!mbar_wait_bounded(bar_addr(p, s), static_cast<uint32_t>((it / kSlots) & 1), a.status)) {
      drain(p, it + 1, it + kSlots, exists, a.status);
      return;
    }
    const int64_t item = item_of(it);
    const int e = a.ws.active[item / tiles_per_expert];
    const int n0 = static_cast<int>(item % tiles_per_expert) * RT;
    const int rows = min(RT, I - n0);
    // Rows 0..RT-1 are gate rows, RT..2RT-1 the matching up rows.
    const float *scp[2 * RT];
    const int32_t *zpp[2 * RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int64_t n = n0 + (r < rows ? r : 0);
      scp[r] = a.gate.scales + e * a.gate.groups_stride + n * a.G;
      zpp[r] = a.gate.zps + e * a.gate.groups_stride + n * a.G;
      scp[RT + r] = a.up.scales + e * a.up.groups_stride + n * a.G;
      zpp[RT + r] = a.up.zps + e * a.up.groups_stride + n * a.G;
    }
    const int base = a.ws.offsets[e];
    const int cnt = a.ws.offsets[e + 1] - base;
    for (int t0 = 0; t0 < cnt; t0 += MT) {
      const int mt = min(MT, cnt - t0);
      const void *xrow[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const int tok = a.ws.assign[base + t0 + (m < mt ? m : 0)] / a.k;
        xrow[m] = XBF16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.x) +
                                                    int64_t(tok) * H)
                        : static_cast<const void *>(static_cast<const float *>(a.x) +
                                                    int64_t(tok) * H);
      }
      float yacc[2 * RT][MT];
      zero_acc(yacc);
      // Gate rows and up rows are laid out as 2*RT consecutive rows only when
      // the tile is full; otherwise the up rows start at RT * rowbytes.
      if (rows == RT) {
        tile_dot<BITS, 2 * RT, MT, XBF16>(slot_addr(p, s), a.rowbytes, 2 * RT, scp, zpp,
                                          a.group_shift, xrow, mt, H, lane, yacc);
      } else {
        // Ragged last tile: gate rows and up rows separately.
        float yg[RT][MT], yu[RT][MT];
        zero_acc(yg);
        zero_acc(yu);
        const float *scg[RT], *scu[RT];
        const int32_t *zpg[RT], *zpu[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          scg[r] = scp[r];
          zpg[r] = zpp[r];
          scu[r] = scp[RT + r];
          zpu[r] = zpp[RT + r];
        }
        tile_dot<BITS, RT, MT, XBF16>(slot_addr(p, s), a.rowbytes, rows, scg, zpg,
                                      a.group_shift, xrow, mt, H, lane, yg);
        tile_dot<BITS, RT, MT, XBF16>(slot_addr(p, s) + RT * a.rowbytes, a.rowbytes, rows, scu,
                                      zpu, a.group_shift, xrow, mt, H, lane, yu);
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            yacc[r][m] = yg[r][m];
            yacc[RT + r][m] = yu[r][m];
          }
      }
      reduce_acc(yacc);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (r < rows && m < mt)
              a.ws.h[int64_t(base + t0 + m) * I + n0 + r] = silu_f(yacc[r][m]) * yacc[RT + r][m];
      }
    }
    __syncwarp();
    if (lane == 0 && exists(it + kSlots)) {
      fence_proxy_async_smem();
      issue(it + kSlots);
    }
  }
}

// ---------------------------------------------------------------------------
// Routed experts, down projection: out[a, :] = h[a, :] . Wd_e^T for every
// assignment a of expert e.  Work item = (active expert, RT rows of Wd).
struct DownArgs {
  QMat down;  // [H, I] per expert
  int group_shift;
  int rowbytes;  // I * bits / 8
  int G;         // I / group
  MoeWork ws;
  uint32_t *status;
};

template <int BITS, int RT, int MT>
__global__ void __launch_bounds__(kWarps * 32, 1) moe_down_kernel(DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Pipe p = pipe_setup(smem, bars, warp, lane);

  const int H = static_cast<int>(a.down.rows);
  const int I = static_cast<int>(a.down.cols);
  const int tiles_per_expert = (H + RT - 1) / RT;
  const int64_t nitems = static_cast<int64_t>(*a.ws.num_active) * tiles_per_expert;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  auto item_of = [&](int64_t it) { return gw + it * nw; };
  auto exists = [&](int64_t it) { return item_of(it) < nitems; };
  auto issue = [&](int64_t it) {
    const int64_t item = item_of(it);
    const int e = a.ws.active[item / tiles_per_expert];
    const int n0 = static_cast<int>(item % tiles_per_expert) * RT;
    const int rows = min(RT, H - n0);
    const uint32_t bytes = static_cast<uint32_t>(rows * a.rowbytes);
    const int s = static_cast<int>(it % kSlots);
    mbar_arrive_expect_tx(bar_addr(p, s), bytes);
    bulk_g2s(slot_addr(p, s), a.down.codes + e * a.down.codes_stride + int64_t(n0) * a.rowbytes,
             bytes, bar_addr(p, s));
  };

  if (lane == 0)
    for (int s = 0; s < kSlots; ++s)
      if (exists(s)) issue(s);

  for (int64_t it = 0; exists(it); ++it) {
    const int s = static_cast<int>(it % kSlots);
    if (!mbar_wait_bounded(bar_addr(p, s), static_cast<uint32_t>((it / kSlots) & 1), a.status)) {
      drain(p, it + 1, it + kSlots, exists, a.status);
      return;
    }
    const int64_t item = item_of(it);
    const int e = a.ws.active[item / tiles_per_expert];
    const int n0 = static_cast<int>(item % tiles_per_expert) * RT;
    const int rows = min(RT, H - n0);
    const float *scp[RT];
    const int32_t *zpp[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const int64_t n = n0 + (r < rows ? r : 0);
      scp[r] = a.down.scales + e * a.down.groups_stride + n * a.G;
      zpp[r] = a.down.zps + e * a.down.groups_stride + n * a.G;
    }
    const int base = a.ws.offsets[e];
    const int cnt = a.ws.offsets[e + 1] - base;
    for (int t0 = 0; t0 < cnt; t0 += MT) {
      const int mt = min(MT, cnt - t0);
      const void *xrow[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        xrow[m] = a.ws.h + int64_t(base + t0 + (m < mt ? m : 0)) * I;
      float yacc[RT][MT];
      zero_acc(yacc);
      tile_dot<BITS, RT, MT, false>(slot_addr(p, s), a.rowbytes, rows, scp, zpp, a.group_shift,
                                    xrow, mt, I, lane, yacc);
      reduce_acc(yacc);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (r < rows && m < mt) a.ws.out[int64_t(base + t0 + m) * H + n0 + r] = yacc[r][m];
      }
    }
    __syncwarp();
    if (lane == 0 && exists(it + kSlots)) {
      fence_proxy_async_smem();
      issue(it + kSlots);
    }
  }
}

int log2i(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return s;
}

// Rows per tile: as many full rows as fit in a slot, at most 4.
int rows_per_tile(int rowbytes, int copies) {
  const int fit = kSlotBytes / (rowbytes * copies);
  return fit >= 4 ? 4 : fit >= 2 ? 2 : fit;
}

template <typename Kern>
cudaError_t prep(Kern k) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

template <int BITS, int RT, int MT, bool XBF16>
cudaError_t run_gemv(const GemvArgs &a, cudaStream_t s) {
  auto k = gemv_kernel<BITS, RT, MT, XBF16>;
  cudaError_t e = prep(k);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (a.N + RT - 1) / RT;
  int64_t blocks = (ntiles + kWarps - 1) / kWarps;
  if (blocks > sm_count()) blocks = sm_count();
  k<<<static_cast<unsigned>(blocks), kWarps * 32, kSmemBytes, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BITS, int RT, bool XBF16>
cudaError_t run_gemv_m(const GemvArgs &a, cudaStream_t s) {
  if (a.M == 1) return run_gemv<BITS, RT, 1, XBF16>(a, s);
  if (a.M == 2) return run_gemv<BITS, RT, 2, XBF16>(a, s);
  return run_gemv<BITS, RT, 4, XBF16>(a, s);
}

template <int BITS, bool XBF16>
cudaError_t run_gemv_rt(const GemvArgs &a, int rt, cudaStream_t s) {
  if (rt >= 4) return run_gemv_m<BITS, 4, XBF16>(a, s);
  if (rt == 2) return run_gemv_m<BITS, 2, XBF16>(a, s);
  return run_gemv_m<BITS, 1, XBF16>(a, s);
}

template <int BITS, int RT, int MT, bool XBF16>
cudaError_t run_gateup(const GateUpArgs &a, cudaStream_t s) {
  auto k = moe_gateup_kernel<BITS, RT, MT, XBF16>;
  cudaError_t e = prep(k);
  if (e != cudaSuccess) return e;
  k<<<sm_count(), kWarps * 32, kSmemBytes, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BITS, bool XBF16>
cudaError_t run_gateup_rt(const GateUpArgs &a, int rt, int mt, cudaStream_t s) {
  if (rt >= 2) {
    if (mt == 1) return run_gateup<BITS, 2, 1, XBF16>(a, s);
    return run_gateup<BITS, 2, 2, XBF16>(a, s);
  }
  if (mt == 1) return run_gateup<BITS, 1, 1, XBF16>(a, s);
  return run_gateup<BITS, 1, 4, XBF16>(a, s);
}

template <int BITS, int RT, int MT>
cudaError_t run_down(const DownArgs &a, cudaStream_t s) {
  auto k = moe_down_kernel<BITS, RT, MT>;
  cudaError_t e = prep(k);
  if (e != cudaSuccess) return e;
  k<<<sm_count(), kWarps * 32, kSmemBytes, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BITS>
cudaError_t run_down_rt(const DownArgs &a, int rt, int mt, cudaStream_t s) {
  if (rt >= 4) {
    if (mt == 1) return run_down<BITS, 4, 1>(a, s);
    return run_down<BITS, 4, 2>(a, s);
  }
  if (rt == 2) {
    if (mt == 1) return run_down<BITS, 2, 1>(a, s);
    return run_down<BITS, 2, 2>(a, s);
  }
  if (mt == 1) return run_down<BITS, 1, 1>(a, s);
  return run_down<BITS, 1, 4>(a, s);
}

}  // namespace

int gemv_max_rowbytes() { return kSlotBytes; }

cudaError_t launch_gemv(const void *x, bool x_bf16, int64_t M, const QMat &w, float *y,
                        cudaStream_t s) {
  GemvArgs a;
  a.x = x;
  a.M = M;
  a.codes = w.codes;
  a.scales = w.scales;
  a.zps = w.zps;
  a.N = w.rows;
  a.K = static_cast<int>(w.cols);
  a.G = static_cast<int>(w.cols / w.group);
  a.group_shift = log2i(w.group);
  a.rowbytes = static_cast<int>(w.cols * w.bits / 8);
  a.y = y;
  a.status = device_status();
  const int rt = rows_per_tile(a.rowbytes, 1);
  if (rt < 1) return cudaErrorInvalidValue;
  if (w.bits == 8) return x_bf16 ? run_gemv_rt<8, true>(a, rt, s) : run_gemv_rt<8, false>(a, rt, s);
  return x_bf16 ? run_gemv_rt<4, true>(a, rt, s) : run_gemv_rt<4, false>(a, rt, s);
}

cudaError_t launch_moe_gateup(const void *x, bool x_bf16, int64_t M, int k, int E,
                              const QMat &gate, const QMat &up, const MoeWork &ws,
                              cudaStream_t s) {
  (void)E;
  GateUpArgs a;
  a.x = x;
  a.k = k;
  a.gate = gate;
  a.up = up;
  a.group_shift = log2i(gate.group);
  a.rowbytes = static_cast<int>(gate.cols * gate.bits / 8);
  a.G = static_cast<int>(gate.cols / gate.group);
  a.ws = ws;
  a.status = device_status();
  const int rt = rows_per_tile(a.rowbytes, 2);
  if (rt < 1) return cudaErrorInvalidValue;
  // Tokens per pass: decode batches route 1-2 tokens to an expert.
  const int mt = (M * k <= 2 * 256) ? 1 : 4;
  if (gate.bits == 8)
    return x_bf16 ? run_gateup_rt<8, true>(a, rt, mt, s) : run_gateup_rt<8, false>(a, rt, mt, s);
  return x_bf16 ? run_gateup_rt<4, true>(a, rt, mt, s) : run_gateup_rt<4, false>(a, rt, mt, s);
}

cudaError_t launch_moe_down(int64_t M, int k, int E, const QMat &down, const MoeWork &ws,
                            cudaStream_t s) {
  (void)E;
  DownArgs a;
  a.down = down;
  a.group_shift = log2i(down.group);
  a.rowbytes = static_cast<int>(down.cols * down.bits / 8);
  a.G = static_cast<int>(down.cols / down.group);
  a.ws = ws;
  a.status = device_status();
  const int rt = rows_per_tile(a.rowbytes, 1);
  if (rt < 1) return cudaErrorInvalidValue;
  const int mt = (M * k <= 2 * 256) ? 1 : 2;
  if (down.bits == 8) return run_down_rt<8>(a, rt, mt, s);
  return run_down_rt<4>(a, rt, mt, s);
}

}  // namespace qmm
