// moe_experts.cu -- routed-expert kernels of the MoE layer on the CUDA cores:
// gate + up projections with the SwiGLU epilogue, and the down projection.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5:
// tokens routed to the same expert are gathered so the expert's weights are
// read once for all of them.  Work items are (expert with tokens, tile of
// weight rows); each warp streams its items' weight tiles through the
// bulk-copy pipeline of stream_tile.cuh and applies them to the expert's
// token list (1-4 tokens per pass).
#include <cstdint>

#include "stream_tile.cuh"

namespace qmm {
namespace {
using namespace tile;

// ---------------------------------------------------------------------------
// Routed experts, gate + up projections with the SwiGLU epilogue.
// Work item = (active expert, RT rows of gate and the same RT rows of up).
// Slot: [gate codes | up codes | gate scales | up scales | gate zps | up zps].
struct GateUpArgs {
  const void *x;  // [M, H]
  int k;
  QMat gate, up;  // [I, H] per expert
  int group_shift;
  TileLayout Lg, Lu;
  MoeWork ws;
  uint32_t *status;
};

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <int BITS, int RT, int MT, bool XBF16, bool GSM>
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
    const int s = static_cast<int>(it % kSlots);
    const uint32_t per = static_cast<uint32_t>(rows * a.Lg.rowbytes) +
                         (GSM ? static_cast<uint32_t>(rows * a.Lg.G * 8) : 0u);
    mbar_arrive_expect_tx(bar_addr(p, s), 2 * per);
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
    const uint32_t slot = slot_addr(p, s);
    GroupSrc<GSM> gs[2 * RT];
    group_srcs<2 * RT, GSM>(gs, 0, RT, slot, a.Lg, a.gate.scales + e * a.gate.groups_stride,
                            a.gate.zps + e * a.gate.groups_stride, n0, rows);
    group_srcs<2 * RT, GSM>(gs, RT, RT, slot, a.Lu, a.up.scales + e * a.up.groups_stride,
                            a.up.zps + e * a.up.groups_stride, n0, rows);
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
      if (rows == RT) {
        // Full tile: gate rows and up rows are 2*RT consecutive rows.
        tile_dot<BITS, 2 * RT, MT, XBF16, GSM>(slot + a.Lg.codes_off, a.Lg.rowbytes, 2 * RT, gs,
                                               a.group_shift, xrow, mt, H, lane, yacc);
      } else {
        // Ragged last tile: up rows start at RT * rowbytes.
        float yg[RT][MT], yu[RT][MT];
        zero_acc(yg);
        zero_acc(yu);
        GroupSrc<GSM> gg[RT], gu[RT];
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          gg[r] = gs[r];
          gu[r] = gs[RT + r];
        }
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
  TileLayout L;
  MoeWork ws;
  uint32_t *status;
};

template <int BITS, int RT, int MT, bool GSM>
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
    GroupSrc<GSM> gs[RT];
    group_srcs<RT, GSM>(gs, 0, RT, slot_addr(p, s), a.L, a.down.scales + e * a.down.groups_stride,
                        a.down.zps + e * a.down.groups_stride, n0, rows);
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
      tile_dot<BITS, RT, MT, false, GSM>(slot_addr(p, s) + a.L.codes_off, a.L.rowbytes, rows, gs,
                                         a.group_shift, xrow, mt, I, lane, yacc);
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

template <int BITS, int RT, int MT, bool XBF16, bool GSM>
cudaError_t run_gateup(GateUpArgs a, cudaStream_t s) {
  auto k = moe_gateup_kernel<BITS, RT, MT, XBF16, GSM>;
  cudaError_t e = prep(k);
  if (e != cudaSuccess) return e;
  TileLayout L[2];
  layouts(a.Lg.rowbytes, a.Lg.G, RT, 2, L);
  a.Lg = L[0];
  a.Lu = L[1];
  k<<<sm_count(), kWarps * 32, kSmemBytes, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BITS, bool XBF16, bool GSM>
cudaError_t run_gateup_rt(const GateUpArgs &a, int rt, int mt, cudaStream_t s) {
  if (rt >= 2) {
    if (mt == 1) return run_gateup<BITS, 2, 1, XBF16, GSM>(a, s);
    return run_gateup<BITS, 2, 2, XBF16, GSM>(a, s);
  }
  if (mt == 1) return run_gateup<BITS, 1, 1, XBF16, GSM>(a, s);
  return run_gateup<BITS, 1, 4, XBF16, GSM>(a, s);
}

template <int BITS, bool GSM>
cudaError_t run_gateup_x(const GateUpArgs &a, bool xbf16, int rt, int mt, cudaStream_t s) {
  return xbf16 ? run_gateup_rt<BITS, true, GSM>(a, rt, mt, s)
               : run_gateup_rt<BITS, false, GSM>(a, rt, mt, s);
}

template <int BITS, int RT, int MT, bool GSM>
cudaError_t run_down(DownArgs a, cudaStream_t s) {
  auto k = moe_down_kernel<BITS, RT, MT, GSM>;
  cudaError_t e = prep(k);
  if (e != cudaSuccess) return e;
  layouts(a.L.rowbytes, a.L.G, RT, 1, &a.L);
  k<<<sm_count(), kWarps * 32, kSmemBytes, s>>>(a);
  count_launch();
  return cudaGetLastError();
}

template <int BITS, bool GSM>
cudaError_t run_down_rt(const DownArgs &a, int rt, int mt, cudaStream_t s) {
  if (rt >= 4) {
    if (mt == 1) return run_down<BITS, 4, 1, GSM>(a, s);
    return run_down<BITS, 4, 2, GSM>(a, s);
  }
  if (rt == 2) {
    if (mt == 1) return run_down<BITS, 2, 1, GSM>(a, s);
    return run_down<BITS, 2, 2, GSM>(a, s);
  }
  if (mt == 1) return run_down<BITS, 1, 1, GSM>(a, s);
  return run_down<BITS, 1, 4, GSM>(a, s);
}

}  // namespace

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
  a.Lg.rowbytes = static_cast<int>(gate.cols * gate.bits / 8);
  a.Lg.G = static_cast<int>(gate.cols / gate.group);
  a.Lu = a.Lg;
  a.ws = ws;
  a.status = device_status();
  const bool gsm = a.Lg.G % 4 == 0;
  const int rt = rows_per_tile(a.Lg.rowbytes, a.Lg.G, gsm, 2);
  if (rt < 1) return cudaErrorInvalidValue;
  // Tokens per pass: decode batches route 1-2 tokens to an expert.
  const int mt = (M * k <= 2 * 256) ? 1 : 4;
  if (gate.bits == 8)
    return gsm ? run_gateup_x<8, true>(a, x_bf16, rt, mt, s)
               : run_gateup_x<8, false>(a, x_bf16, rt, mt, s);
  return gsm ? run_gateup_x<4, true>(a, x_bf16, rt, mt, s)
             : run_gateup_x<4, false>(a, x_bf16, rt, mt, s);
}

cudaError_t launch_moe_down(int64_t M, int k, int E, const QMat &down, const MoeWork &ws,
                            cudaStream_t s) {
  (void)E;
  DownArgs a;
  a.down = down;
  a.group_shift = log2i(down.group);
  a.L.rowbytes = static_cast<int>(down.cols * down.bits / 8);
  a.L.G = static_cast<int>(down.cols / down.group);
  a.ws = ws;
  a.status = device_status();
  const bool gsm = a.L.G % 4 == 0;
  const int rt = rows_per_tile(a.L.rowbytes, a.L.G, gsm, 1);
  if (rt < 1) return cudaErrorInvalidValue;
  const int mt = (M * k <= 2 * 256) ? 1 : 2;
  if (down.bits == 8) return gsm ? run_down_rt<8, true>(a, rt, mt, s) : run_down_rt<8, false>(a, rt, mt, s);
  return gsm ? run_down_rt<4, true>(a, rt, mt, s) : run_down_rt<4, false>(a, rt, mt, s);
}

}  // namespace qmm
