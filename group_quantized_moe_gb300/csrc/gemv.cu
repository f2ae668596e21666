// gemv.cu -- qmm_linear: fused dequantise-matmul y = x . deq(W)^T for
// decode-sized batches on the CUDA cores (see stream_tile.cuh for the tile
// pipeline and the in-register dequantisation).  Grid = one block of 8
// warps per SM; tiles of RT weight rows are dealt round-robin over all warps.
#include <cstdint>

#include "stream_tile.cuh"

namespace qmm {
namespace {
using namespace tile;

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
  int group_shift;
  TileLayout L;
  void *y;          // [M, N] fp32, or bf16 when y_bf16
  bool y_bf16;
  uint32_t *status;
};

template <int BITS, int RT, int MT, bool XBF16, bool GSM, int NCL>
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
    const int64_t n0 = tile_of(it) * RT;
    const int rows = static_cast<int>(min64(RT, a.N - n0));
    const int s = static_cast<int>(it % kSlots);
    const uint32_t bytes = static_cast<uint32_t>(rows * a.L.rowbytes) +
                           (GSM ? static_cast<uint32_t>(rows * a.L.G * 8) : 0u);
    mbar_arrive_expect_tx(bar_addr(p, s), bytes);
    issue_rows<GSM>(slot_addr(p, s), bar_addr(p, s), a.L, a.codes, a.scales, a.zps, n0, rows);
  };

  // The first weight tiles are requested before waiting for the preceding
  // kernel: no kernel of a launch sequence writes the quantised weights
  // (the quantiser lets no successor start early), so their HBM latency
  // overlaps the previous kernel's tail.  Activations and outputs are only
  // touched after the wait.
  if (lane == 0)
    for (int s = 0; s < kSlots; ++s)
      if (exists(s)) issue(s);
  pdl_enter();

  // Register-resident activation row (M == 1 and K == 32 * CH * NCL).
  constexpr int CH = (BITS == 8) ? 16 : 32;
  float xr[NCL > 0 ? NCL : 1][CH];
  if constexpr (NCL > 0) {
#pragma unroll
    for (int i = 0; i < NCL; ++i)
#pragma unroll
      for (int e = 0; e < CH; e += 4) {
        const float4 v = load_x4<XBF16>(a.x, (lane + 32 * i) * CH + e);
        xr[i][e] = v.x;
        xr[i][e + 1] = v.y;
        xr[i][e + 2] = v.z;
        xr[i][e + 3] = v.w;
      }
  }

  for (int64_t it = 0; exists(it); ++it) {
    const int s = static_cast<int>(it % kSlots);
    if (!mbar_wait_bounded(bar_addr(p, s), static_cast<uint32_t>((it / kSlots) & 1), a.status)) {
      drain(p, it + 1, it + kSlots, exists, a.status);
      return;
    }
    const int64_t n0 = tile_of(it) * RT;
    const int rows = static_cast<int>(min64(RT, a.N - n0));
    GroupSrc<GSM> gs[RT];
    group_srcs<RT, GSM>(gs, 0, RT, slot_addr(p, s), a.L, a.scales, a.zps, n0, rows);
    if constexpr (NCL > 0) {
      float yr[RT];
#pragma unroll
      for (int r = 0; r < RT; ++r) yr[r] = 0.0f;
      tile_dot_xr<BITS, RT, NCL, GSM>(slot_addr(p, s) + a.L.codes_off, a.L.rowbytes, rows, gs,
                                      a.group_shift, xr, lane, yr);
#pragma unroll
      for (int r = 0; r < RT; ++r) yr[r] = warp_sum(yr[r]);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
          if (r < rows) store_y(a.y, n0 + r, yr[r], a.y_bf16);
      }
    } else
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
      tile_dot<BITS, RT, MT, XBF16, GSM>(slot_addr(p, s) + a.L.codes_off, a.L.rowbytes, rows, gs,
                                         a.group_shift, xrow, mt, a.K, lane, yacc);
      reduce_acc(yacc);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
          for (int m = 0; m < MT; ++m)
            if (r < rows && m < mt) store_y(a.y, (m0 + m) * a.N + n0 + r, yacc[r][m], a.y_bf16);
      }
    }
    __syncwarp();
    if (lane == 0 && exists(it + kSlots)) {
      fence_proxy_async_smem();
      issue(it + kSlots);
    }
  }
}

template <int BITS, int RT, int MT, bool XBF16, bool GSM, int NCL = 0>
cudaError_t run_gemv(GemvArgs a, cudaStream_t s) {
  auto k = gemv_kernel<BITS, RT, MT, XBF16, GSM, NCL>;
  cudaError_t e = prep(k);
  if (e != cudaSuccess) return e;
  layouts(a.L.rowbytes, a.L.G, RT, 1, &a.L);
  const int64_t ntiles = (a.N + RT - 1) / RT;
  int64_t blocks = (ntiles + kWarps - 1) / kWarps;
  if (blocks > sm_count()) blocks = sm_count();
  return launch_pdl(k, dim3(static_cast<unsigned>(blocks)), dim3(kWarps * 32), kSmemBytes, s, a);
}

template <int BITS, int RT, bool XBF16, bool GSM>
cudaError_t run_gemv_m(const GemvArgs &a, cudaStream_t s) {
  constexpr int CH = (BITS == 8) ? 16 : 32;
  if (a.M == 1) {
    // Activation row in registers when K is 32 * CH * NCL (NCL = 2, 4, 8).
    // (INT4 with 8 chunks per lane would need 256 activation registers.)
    if constexpr (BITS == 8)
      if (a.K == 32 * CH * 8) return run_gemv<BITS, RT, 1, XBF16, GSM, 8>(a, s);
    if (a.K == 32 * CH * 4) return run_gemv<BITS, RT, 1, XBF16, GSM, 4>(a, s);
    if (a.K == 32 * CH * 2) return run_gemv<BITS, RT, 1, XBF16, GSM, 2>(a, s);
    return run_gemv<BITS, RT, 1, XBF16, GSM>(a, s);
  }
  if (a.M == 2) return run_gemv<BITS, RT, 2, XBF16, GSM>(a, s);
  return run_gemv<BITS, RT, 4, XBF16, GSM>(a, s);
}

template <int BITS, bool XBF16, bool GSM>
cudaError_t run_gemv_rt(const GemvArgs &a, int rt, cudaStream_t s) {
  if (rt >= 4) return run_gemv_m<BITS, 4, XBF16, GSM>(a, s);
  if (rt == 2) return run_gemv_m<BITS, 2, XBF16, GSM>(a, s);
  return run_gemv_m<BITS, 1, XBF16, GSM>(a, s);
}

template <int BITS, bool GSM>
cudaError_t run_gemv_x(const GemvArgs &a, bool xbf16, int rt, cudaStream_t s) {
  return xbf16 ? run_gemv_rt<BITS, true, GSM>(a, rt, s) : run_gemv_rt<BITS, false, GSM>(a, rt, s);
}

}  // namespace

int gemv_rows_per_tile(int64_t rowbytes, int64_t G, int copies) {
  if (rowbytes <= 0 || rowbytes > kSlotBytes || G <= 0 || G > kSlotBytes) return 0;
  return rows_per_tile(static_cast<int>(rowbytes), static_cast<int>(G), G % 4 == 0, copies);
}

cudaError_t launch_gemv(const void *x, bool x_bf16, int64_t M, const QMat &w, void *y, bool y_bf16,
                        cudaStream_t s) {
  GemvArgs a;
  a.x = x;
  a.M = M;
  a.codes = w.codes;
  a.scales = w.scales;
  a.zps = w.zps;
  a.N = w.rows;
  a.K = static_cast<int>(w.cols);
  a.group_shift = log2i(w.group);
  a.L.rowbytes = static_cast<int>(w.cols * w.bits / 8);
  a.L.G = static_cast<int>(w.cols / w.group);
  a.y = y;
  a.y_bf16 = y_bf16;
  a.status = device_status();
  const bool gsm = a.L.G % 4 == 0;
  int rt = rows_per_tile(a.L.rowbytes, a.L.G, gsm, 1);
  if (rt < 1) return cudaErrorInvalidValue;
  if (w.bits == 8)
    return gsm ? run_gemv_x<8, true>(a, x_bf16, rt, s) : run_gemv_x<8, false>(a, x_bf16, rt, s);
  return gsm ? run_gemv_x<4, true>(a, x_bf16, rt, s) : run_gemv_x<4, false>(a, x_bf16, rt, s);
}

}  // namespace qmm
