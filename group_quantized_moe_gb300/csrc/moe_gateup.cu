// moe_gateup.cu -- routed experts on the CUDA cores: gate + up projections
// of each expert's tokens with the SwiGLU epilogue, h = silu(x Wg^T) * (x Wu^T)
// ("Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5:
// gather the tokens of one expert, then read its weights once).
#include <cstdint>

#include "moe_common.cuh"

namespace qmm {
namespace {
using namespace moe;

constexpr int kItemBlock = 4;

// ---------------------------------------------------------------------------
// Routed experts, gate + up projections with the SwiGLU epilogue.
// Work item = (active expert, RT rows of gate and the same RT rows of up);
// each warp takes blocks of 4 consecutive items, so consecutive items mostly
// belong to the same expert.  Experts with one token (the common decode
// case) keep that token's row in registers (NCL > 0) until the expert
// changes; others read activations through L1 a chunk at a time.
// Slot: [gate codes | up codes | gate scales | up scales | gate zps | up zps].
struct GateUpArgs {
  const void *x;  // [M, H]
  int k;
  int E;
  QMat gate, up;  // [I, H] per expert
  int group_shift;
  TileLayout Lg, Lu;
  MoeWork ws;
  uint32_t *status;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <int BITS, int RT, int MT, bool XBF16, bool GSM, int NCL>
__global__ void __launch_bounds__(kWarps * 32, 1) moe_gateup_kernel(GateUpArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kSlots];
  constexpr int CH = (BITS == 8) ? 16 : 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int na;
  const int32_t *s_active, *s_off;
  stage_meta(smem, a.ws, a.E, na, s_active, s_off);
  const Pipe p = pipe_setup(smem, bars, warp, lane);

  const int I = static_cast<int>(a.gate.rows);
  const int H = static_cast<int>(a.gate.cols);
  const int tiles_per_expert = (I + RT - 1) / RT;
  const int64_t nitems = static_cast<int64_t>(na) * tiles_per_expert;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarps;
  // Blocks of kItemBlock consecutive items, dealt round-robin over the warps:
  // the grid's reads stay within a compact window of HBM while a warp's
  // consecutive items mostly share an expert (and its token row).
  auto item_of = [&](int64_t it) {
    return ((it / kItemBlock) * nw + gw) * kItemBlock + (it % kItemBlock);
  };
  auto exists = [&](int64_t it) { return item_of(it) < nitems; };
  auto issue = [&](int64_t it) {
    const int64_t item = item_of(it);
    const int e = s_active[item / tiles_per_expert];
    const int n0 = static_cast<int>(item % tiles_per_expert) * RT;
    const int rows = min(RT, I - n0);
    const int s = static_cast<int>(it % kSlots);
    const uint32_t bytes = static_cast<uint32_t>(rows * a.Lg.rowbytes) +
                           (GSM ? static_cast<uint32_t>(rows * a.Lg.G * 8) : 0u);
    mbar_arrive_expect_tx(bar_addr(p, s), 2 * bytes);
    issue_rows<GSM>(slot_addr(p, s), bar_addr(p, s), a.Lg, a.gate.codes + e * a.gate.codes_stride,
                    a.gate.scales + e * a.gate.groups_stride,
                    a.gate.zps + e * a.gate.groups_stride, n0, rows);
    issue_rows<GSM>(slot_addr(p, s), bar_addr(p, s), a.Lu, a.up.codes + e * a.up.codes_stride,
                    a.up.scales + e * a.up.groups_stride, a.up.zps + e * a.up.groups_stride, n0,
                    rows);
  };

  if (lane == 0)
    for (int s = 0; s < kSlots; ++s)
      if (exists(s)) issue(s);

  float xr[NCL > 0 ? NCL : 1][CH];
  int cur_e = -1;

  for (int64_t it = 0; exists(it); ++it) {
    const int s = static_cast<int>(it % kSlots);
    if (!mbar_wait_bounded(bar_addr(p, s), static_cast<uint32_t>((it / kSlots) & 1), a.status)) {
      drain(p, it + 1, it + kSlots, exists, a.status);
      return;
    }
    const int64_t item = item_of(it);
    const int e = s_active[item / tiles_per_expert];
    const int n0 = static_cast<int>(item % tiles_per_expert) * RT;
    const int rows = min(RT, I - n0);
    const uint32_t slot = slot_addr(p, s);
    GroupSrc<GSM> gs[2 * RT];
    group_srcs<2 * RT, GSM>(gs, 0, RT, slot, a.Lg, a.gate.scales + e * a.gate.groups_stride,
                            a.gate.zps + e * a.gate.groups_stride, n0, rows);
    group_srcs<2 * RT, GSM>(gs, RT, RT, slot, a.Lu, a.up.scales + e * a.up.groups_stride,
                            a.up.zps + e * a.up.groups_stride, n0, rows);
    GroupSrc<GSM> gg[RT], gu[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      gg[r] = gs[r];
      gu[r] = gs[RT + r];
    }
    const int base = s_off[e];
    const int cnt = s_off[e + 1] - base;
    bool done = false;
    if constexpr (NCL > 0) {
      if (cnt == 1) {
        if (e != cur_e) {
          const int tok = a.ws.assign[base] / a.k;
          const void *row = XBF16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.x) +
                                                              int64_t(tok) * H)
                                  : static_cast<const void *>(static_cast<const float *>(a.x) +
                                                              int64_t(tok) * H);
          load_xr<XBF16, NCL, CH>(row, lane, xr);
          cur_e = e;
        }
        float yg[2 * RT];
#pragma unroll
        for (int r = 0; r < 2 * RT; ++r) yg[r] = 0.0f;
        if (rows == RT) {
          tile_dot_xr<BITS, 2 * RT, NCL, GSM>(slot + a.Lg.codes_off, a.Lg.rowbytes, 2 * RT, gs,
                                              a.group_shift, xr, lane, yg);
        } else {
          float yy[RT], yu[RT];
#pragma unroll
          for (int r = 0; r < RT; ++r) yy[r] = yu[r] = 0.0f;
          tile_dot_xr<BITS, RT, NCL, GSM>(slot + a.Lg.codes_off, a.Lg.rowbytes, rows, gg,
                                          a.group_shift, xr, lane, yy);
          tile_dot_xr<BITS, RT, NCL, GSM>(slot + a.Lu.codes_off, a.Lu.rowbytes, rows, gu,
                                          a.group_shift, xr, lane, yu);
#pragma unroll
          for (int r = 0; r < RT; ++r) {
            yg[r] = yy[r];
            yg[RT + r] = yu[r];
          }
        }
#pragma unroll
        for (int r = 0; r < 2 * RT; ++r) yg[r] = warp_sum(yg[r]);
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < RT; ++r)
            if (r < rows) a.ws.h[int64_t(base) * I + n0 + r] = silu_f(yg[r]) * yg[RT + r];
        }
        done = true;
      }
    }
    if (!done) {
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
        if (rows == RT) {
          tile_dot<BITS, 2 * RT, MT, XBF16, GSM>(slot + a.Lg.codes_off, a.Lg.rowbytes, 2 * RT, gs,
                                                 a.group_shift, xrow, mt, H, lane, yacc);
        } else {
          float yg[RT][MT], yu[RT][MT];
          zero_acc(yg);
          zero_acc(yu);
          tile_dot<BITS, RT, MT, XBF16, GSM>(slot + a.Lg.codes_off, a.Lg.rowbytes, rows, gg,
                                             a.group_shift, xrow, mt, H, lane, yg);
          tile_dot<BITS, RT, MT, XBF16, GSM>(slot + a.Lu.codes_off, a.Lu.rowbytes, rows, gu,
                                             a.group_shift, xrow, mt, H, lane, yu);
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
    }
    __syncwarp();
    if (lane == 0 && exists(it + kSlots)) {
      fence_proxy_async_smem();
      issue(it + kSlots);
    }
  }
}

template <int BITS, int RT, int MT, bool XBF16, bool GSM, int NCL>
cudaError_t run_gateup(GateUpArgs a, cudaStream_t s) {
  auto k = moe_gateup_kernel<BITS, RT, MT, XBF16, GSM, NCL>;
  cudaError_t e = prep_meta(k, a.E);
  if (e != cudaSuccess) return e;
  TileLayout L[2];
  layouts(a.Lg.rowbytes, a.Lg.G, RT, 2, L);
  a.Lg = L[0];
  a.Lu = L[1];
  return launch_pdl(k, dim3(sm_count()), dim3(kWarps * 32), kSmemBytes + meta_bytes(a.E), s, a);
}

template <int BITS, int RT, int MT, bool XBF16, bool GSM>
cudaError_t run_gateup_ncl(const GateUpArgs &a, int ncl, cudaStream_t s) {
  if (ncl == 4) return run_gateup<BITS, RT, MT, XBF16, GSM, 4>(a, s);
  if (ncl == 2) return run_gateup<BITS, RT, MT, XBF16, GSM, 2>(a, s);
  return run_gateup<BITS, RT, MT, XBF16, GSM, 0>(a, s);
}

template <int BITS, bool XBF16, bool GSM>
cudaError_t run_gateup_rt(const GateUpArgs &a, int rt, int mt, int ncl, cudaStream_t s) {
  if (rt >= 2) {
    if (mt == 1) return run_gateup_ncl<BITS, 2, 1, XBF16, GSM>(a, ncl, s);
    return run_gateup_ncl<BITS, 2, 2, XBF16, GSM>(a, ncl, s);
  }
  if (mt == 1) return run_gateup_ncl<BITS, 1, 1, XBF16, GSM>(a, ncl, s);
  return run_gateup_ncl<BITS, 1, 4, XBF16, GSM>(a, ncl, s);
}

template <int BITS>
cudaError_t run_gateup_x(const GateUpArgs &a, bool xbf16, int rt, int mt, int ncl,
                         cudaStream_t s) {
  return xbf16 ? run_gateup_rt<BITS, true, true>(a, rt, mt, ncl, s)
               : run_gateup_rt<BITS, false, true>(a, rt, mt, ncl, s);
}

}  // namespace

cudaError_t launch_moe_gateup(const void *x, bool x_bf16, int64_t M, int k, int E,
                              const QMat &gate, const QMat &up, const MoeWork &ws,
                              cudaStream_t s) {
  GateUpArgs a;
  a.x = x;
  a.k = k;
  a.E = E;
  a.gate = gate;
  a.up = up;
  a.group_shift = log2i(gate.group);
  a.Lg.rowbytes = static_cast<int>(gate.cols * gate.bits / 8);
  a.Lg.G = static_cast<int>(gate.cols / gate.group);
  a.Lu = a.Lg;
  a.ws = ws;
  a.status = device_status();
  // Expert scales / zero points are always staged (G % 4 == 0 is required).
  if (a.Lg.G % 4 != 0) return cudaErrorInvalidValue;
  const int rt = rows_per_tile(a.Lg.rowbytes, a.Lg.G, true, 2);
  if (rt < 1) return cudaErrorInvalidValue;
  // Tokens per pass for experts with several tokens.
  const int mt = (M * k <= 2 * 256) ? 2 : 4;
  const int H = static_cast<int>(gate.cols);
  if (gate.bits == 8) {
    const int ncl = ncl_for<8>(H);
    return run_gateup_x<8>(a, x_bf16, rt, mt, ncl, s);
  }
  const int ncl = ncl_for<4>(H);
  return run_gateup_x<4>(a, x_bf16, rt, mt, ncl, s);
}

}  // namespace qmm
