// moe_down.cu -- routed experts on the CUDA cores: down projection of each
// expert's SwiGLU activations, out[a] = h[a] Wd_e^T per assignment a.
#include <cstdint>

#include "moe_common.cuh"

namespace qmm {
namespace {
using namespace moe;

constexpr int kItemBlock = 4;

// ---------------------------------------------------------------------------
// Routed experts, down projection: out[a, :] = h[a, :] . Wd_e^T for every
// assignment a of expert e.  Work item = (active expert, RT rows of Wd);
// blocks of 4 consecutive items per warp and the register-resident
// activation row for single-token experts, as in moe_gateup.cu.
struct DownArgs {
  int E;
  QMat down;  // [H, I] per expert
  int group_shift;
  TileLayout L;
  MoeWork ws;
  uint32_t *status;
};

template <int BITS, int RT, int MT, bool GSM, int NCL>
__global__ void __launch_bounds__(kWarps * 32, 1) moe_down_kernel(DownArgs a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kSlots];
  constexpr int CH = (BITS == 8) ? 16 : 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int na;
  const int32_t *s_active, *s_off;
  stage_meta(smem, a.ws, a.E, na, s_active, s_off);
  const Pipe p = pipe_setup(smem, bars, warp, lane);

  const int H = static_cast<int>(a.down.rows);
  const int I = static_cast<int>(a.down.cols);
  const int tiles_per_expert = (H + RT - 1) / RT;
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
    const int rows = min(RT, H - n0);
    const int s = static_cast<int>(it % kSlots);
    const uint32_t bytes = static_cast<uint32_t>(rows * a.L.rowbytes) +
                           (GSM ? static_cast<uint32_t>(rows * a.L.G * 8) : 0u);
    mbar_arrive_expect_tx(bar_addr(p, s), bytes);
    issue_rows<GSM>(slot_addr(p, s), bar_addr(p, s), a.L, a.down.codes + e * a.down.codes_stride,
                    a.down.scales + e * a.down.groups_stride,
                    a.down.zps + e * a.down.groups_stride, n0, rows);
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
    const int rows = min(RT, H - n0);
    GroupSrc<GSM> gs[RT];
    group_srcs<RT, GSM>(gs, 0, RT, slot_addr(p, s), a.L, a.down.scales + e * a.down.groups_stride,
                        a.down.zps + e * a.down.groups_stride, n0, rows);
    const int base = s_off[e];
    const int cnt = s_off[e + 1] - base;
    bool done = false;
    if constexpr (NCL > 0) {
      if (cnt == 1) {
        if (e != cur_e) {
          load_xr<false, NCL, CH>(a.ws.h + int64_t(base) * I, lane, xr);
          cur_e = e;
        }
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
            if (r < rows) a.ws.out[int64_t(base) * H + n0 + r] = yr[r];
        }
        done = true;
      }
    }
    if (!done) {
      for (int t0 = 0; t0 < cnt; t0 += MT) {
        const int mt = min(MT, cnt - t0);
        const void *xrow[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m)
          xrow[m] = a.ws.h + int64_t(base + t0 + (m < mt ? m : 0)) * I;
        float yacc[RT][MT];
        zero_acc(yacc);
        tile_dot<BITS, RT, MT, false, GSM>(slot_addr(p, s) + a.L.codes_off, a.L.rowbytes, rows,
                                           gs, a.group_shift, xrow, mt, I, lane, yacc);
        reduce_acc(yacc);
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
              if (r < rows && m < mt) a.ws.out[int64_t(base + t0 + m) * H + n0 + r] = yacc[r][m];
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

template <int BITS, int RT, int MT, bool GSM, int NCL>
cudaError_t run_down(DownArgs a, cudaStream_t s) {
  auto k = moe_down_kernel<BITS, RT, MT, GSM, NCL>;
  cudaError_t e = prep_meta(k, a.E);
  if (e != cudaSuccess) return e;
  layouts(a.L.rowbytes, a.L.G, RT, 1, &a.L);
  return launch_pdl(k, dim3(sm_count()), dim3(kWarps * 32), kSmemBytes + meta_bytes(a.E), s, a);
}

template <int BITS, int RT, int MT, bool GSM>
cudaError_t run_down_ncl(const DownArgs &a, int ncl, cudaStream_t s) {
  if (ncl == 4) return run_down<BITS, RT, MT, GSM, 4>(a, s);
  if (ncl == 2) return run_down<BITS, RT, MT, GSM, 2>(a, s);
  return run_down<BITS, RT, MT, GSM, 0>(a, s);
}

template <int BITS, bool GSM>
cudaError_t run_down_rt(const DownArgs &a, int rt, int mt, int ncl, cudaStream_t s) {
  if (rt >= 4) {
    if (mt == 1) return run_down_ncl<BITS, 4, 1, GSM>(a, ncl, s);
    return run_down_ncl<BITS, 4, 2, GSM>(a, ncl, s);
  }
  if (rt == 2) {
    if (mt == 1) return run_down_ncl<BITS, 2, 1, GSM>(a, ncl, s);
    return run_down_ncl<BITS, 2, 2, GSM>(a, ncl, s);
  }
  if (mt == 1) return run_down_ncl<BITS, 1, 1, GSM>(a, ncl, s);
  return run_down_ncl<BITS, 1, 4, GSM>(a, ncl, s);
}

}  // namespace

cudaError_t launch_moe_down(int64_t M, int k, int E, const QMat &down, const MoeWork &ws,
                            cudaStream_t s) {
  DownArgs a;
  a.E = E;
  a.down = down;
  a.group_shift = log2i(down.group);
  a.L.rowbytes = static_cast<int>(down.cols * down.bits / 8);
  a.L.G = static_cast<int>(down.cols / down.group);
  a.ws = ws;
  a.status = device_status();
  if (a.L.G % 4 != 0) return cudaErrorInvalidValue;
  const int rt = rows_per_tile(a.L.rowbytes, a.L.G, true, 1);
  if (rt < 1) return cudaErrorInvalidValue;
  const int mt = (M * k <= 2 * 256) ? 1 : 2;
  const int I = static_cast<int>(down.cols);
  if (down.bits == 8) {
    const int ncl = ncl_for<8>(I);
    return run_down_rt<8, true>(a, rt, mt, ncl, s);
  }
  const int ncl = ncl_for<4>(I);
  return run_down_rt<4, true>(a, rt, mt, ncl, s);
}

}  // namespace qmm
