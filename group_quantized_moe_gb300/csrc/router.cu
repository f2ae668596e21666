// router.cu -- MoE router (logits, top-k, renormalised weights), token
// grouping by expert, and the weighted combine of expert outputs.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5: the
// router is a linear layer followed by a softmax and a top-k; tokens routed to
// the same expert are gathered so that the expert's weights are read once;
// the selected experts' outputs are combined by a weighted sum.  Section 3.4
// (same article): subtract the maximum before exponentiating.
//
// Logits use a fixed fp32 summation order so that the selected experts are
// bit-identical to any other implementation of the same order:
//   partial p (p = 0..127) = fma chain over h = p, p+128, p+256, ...
//   t_l = (P[4l] + P[4l+1]) + (P[4l+2] + P[4l+3]),       l = 0..31
//   t_l = t_l + t_{l+o} for o = 16, 8, 4, 2, 1;  logit = t_0 (+ bias)
// GPU mapping: a block of 128 threads owns the 128 partials (thread p holds
// partial p) for a register tile of MB tokens x EB experts, reading x and the
// router rows as coalesced 512-byte rows per step.  The tree runs in the
// order above: adjacent-partial sums by xor shuffles 1 and 2, the o = 16 and
// o = 8 stages across warps through shared memory, the rest by xor shuffles
// 16, 8, 4 inside warp 0.  Decode batches (M <= 8) use two tokens and one
// expert per block with the router row preloaded; batches above 64 tokens
// stage 16-token x 8-expert tiles through shared memory
// (router_logits_tiled_kernel).
#include <cstdint>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kMaxK = 16;
constexpr int kMaxE = 1024;

// NS > 0 (H == 128 NS): the block's router rows are loaded into registers
// before waiting for the preceding kernel (no kernel writes router weights),
// so their latency overlaps that kernel's tail; small batches use it.
template <int MB, int EB, bool XBF16, int NS>
__global__ void __launch_bounds__(128) router_logits_kernel(const void *__restrict__ x, int64_t M,
                                                            int64_t H,
                                                            const float *__restrict__ wr,
                                                            const float *__restrict__ bias, int E,
                                                            float *__restrict__ logits,
                                                            int32_t *__restrict__ counts) {
  __shared__ float xch[2][32][MB * EB + 1];
  const int p = threadIdx.x;  // partial index
  const int warp = p >> 5, lane = p & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * MB;
  const int e0 = blockIdx.x * EB;
  const int mb = static_cast<int>(min64(MB, M - m0));
  const int eb = min(EB, E - e0);
  float wpre[NS > 0 ? NS : 1][EB];
  if constexpr (NS > 0) {
#pragma unroll
    for (int j = 0; j < NS; ++j)
#pragma unroll
      for (int e = 0; e < EB; ++e)
        wpre[j][e] = __ldg(wr + int64_t(e0 + (e < eb ? e : 0)) * H + p + 128 * j);
  }
  pdl_enter();
  // The expert histogram is accumulated by the top-k kernel that follows.
  if (counts && blockIdx.x == 0 && blockIdx.y == 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = 0;

  float acc[MB][EB];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int e = 0; e < EB; ++e) acc[m][e] = 0.0f;

  static_assert(NS == 0 || MB * NS <= 64, "preloaded rows are for a few tokens");
  if constexpr (NS > 0) {
    // few tokens: the thread's activation loads are independent of each
    // other and of the chains, so they can all be in flight together (same
    // chain order per partial)
    float xv[NS][MB];
#pragma unroll
    for (int j = 0; j < NS; ++j)
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const int64_t mm = m0 + (m < mb ? m : 0);
        const int64_t hh = p + 128 * j;
        if constexpr (XBF16) {
          const uint16_t b = static_cast<const uint16_t *>(x)[mm * H + hh];
          xv[j][m] = __uint_as_float(static_cast<uint32_t>(b) << 16);
        } else {
          xv[j][m] = __ldg(static_cast<const float *>(x) + mm * H + hh);
        }
      }
#pragma unroll
    for (int j = 0; j < NS; ++j)
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int e = 0; e < EB; ++e) acc[m][e] = __fmaf_rn(xv[j][m], wpre[j][e], acc[m][e]);
  }

  // Four h-steps per iteration: all their loads issue before the FMAs, so a
  // thread keeps 4 * (MB + EB) loads in flight (the chain order per partial
  // is unchanged).
  int64_t h = NS > 0 ? H : p;
  for (; h + 3 * 128 < H; h += 4 * 128) {
    float xv[4][MB], wv[4][EB];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        const int64_t mm = m0 + (m < mb ? m : 0);
        if constexpr (XBF16) {
          const uint16_t b = static_cast<const uint16_t *>(x)[mm * H + h + 128 * u];
          xv[u][m] = __uint_as_float(static_cast<uint32_t>(b) << 16);
        } else {
          xv[u][m] = __ldg(static_cast<const float *>(x) + mm * H + h + 128 * u);
        }
      }
#pragma unroll
      for (int e = 0; e < EB; ++e)
        wv[u][e] = __ldg(wr + int64_t(e0 + (e < eb ? e : 0)) * H + h + 128 * u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int e = 0; e < EB; ++e) acc[m][e] = __fmaf_rn(xv[u][m], wv[u][e], acc[m][e]);
  }
  for (; h < H; h += 128) {
    float xv[MB], wv[EB];
#pragma unroll
    for (int m = 0; m < MB; ++m) {
      const int64_t mm = m0 + (m < mb ? m : 0);
      if constexpr (XBF16) {
        const uint16_t b = static_cast<const uint16_t *>(x)[mm * H + h];
        xv[m] = __uint_as_float(static_cast<uint32_t>(b) << 16);
      } else {
        xv[m] = __ldg(static_cast<const float *>(x) + mm * H + h);
      }
    }
#pragma unroll
    for (int e = 0; e < EB; ++e) wv[e] = __ldg(wr + int64_t(e0 + (e < eb ? e : 0)) * H + h);
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int e = 0; e < EB; ++e) acc[m][e] = __fmaf_rn(xv[m], wv[e], acc[m][e]);
  }

  // Level 1: t = (P0 + P1) + (P2 + P3) inside each group of 4 lanes.
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int e = 0; e < EB; ++e) {
      float v = acc[m][e];
      v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
      v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
      acc[m][e] = v;  // valid at lanes with lane % 4 == 0: t_l, l = p / 4
    }
  // o = 16: t_l += t_{l+16}; l in 0..15 lives in warps 0-1, l+16 in warps 2-3.
  if (warp >= 2 && (lane & 3) == 0) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int e = 0; e < EB; ++e) xch[warp - 2][lane][m * EB + e] = acc[m][e];
  }
  __syncthreads();
  if (warp < 2 && (lane & 3) == 0) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int e = 0; e < EB; ++e) acc[m][e] = __fadd_rn(acc[m][e], xch[warp][lane][m * EB + e]);
  }
  __syncthreads();
  // o = 8: t_l += t_{l+8}; l in 0..7 is warp 0, l+8 is warp 1.
  if (warp == 1 && (lane & 3) == 0) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int e = 0; e < EB; ++e) xch[0][lane][m * EB + e] = acc[m][e];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int e = 0; e < EB; ++e) {
        float v = acc[m][e];
        if ((lane & 3) == 0) v = __fadd_rn(v, xch[0][lane][m * EB + e]);
        // o = 4, 2, 1 <-> lanes 4l and 4(l+o): xor 16, 8, 4.
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 16));
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
        if (lane == 0 && m < mb && e < eb) {
          if (bias) v = __fadd_rn(v, bias[e0 + e]);
          logits[(m0 + m) * E + e0 + e] = v;
        }
      }
  }
}

// ---------------------------------------------------------------------------
// Batched logits (many tokens).  The kernel above reads its operands straight
// from L2 with no reuse inside the block, which leaves a 512-token batch
// bound by L2 traffic.  Here a block owns a tile of kTM tokens x TE experts
// for all 128 partials: the tile's token rows and router rows stream through
// shared memory in chunks of kCH columns (1-D bulk copies, a ring of kNST
// stages), thread (p, half) keeps partial p of 8 tokens x TE experts in
// registers, and every staged value feeds 8 or TE FMAs.  TE = 8 keeps the
// registers under 128 so that two blocks share an SM: the FMA chains wait on
// shared-memory loads, and the second block's warps fill those waits.  The summation order
// is the one above: each partial is one fma chain in increasing h; the
// first tree level ((P0 + P1) + (P2 + P3)) runs as two halving exchanges
// between adjacent lanes; the last five levels run per output from shared
// memory.
namespace tiled {
constexpr int kTM = 16, kTE = 8, kCH = 512, kNST = 3, kThreads = 256;
template <bool XBF16, int TE>
__host__ __device__ constexpr int stage_bytes() {
  return kTM * kCH * (XBF16 ? 2 : 4) + TE * kCH * 4;
}
template <bool XBF16, int TE>
__host__ __device__ constexpr int smem_bytes() {
  return kNST * stage_bytes<XBF16, TE>();
}
}  // namespace tiled

template <bool XBF16, int TE>
__global__ void __launch_bounds__(tiled::kThreads, TE <= 8 ? 2 : 1)
    router_logits_tiled_kernel(const void *__restrict__ x, int64_t M, int64_t H,
                               const float *__restrict__ wr, const float *__restrict__ bias,
                               int E, float *__restrict__ logits, int32_t *__restrict__ counts,
                               uint32_t *status) {
  using namespace tiled;
  constexpr int XB = XBF16 ? 2 : 4;
  constexpr int SB = stage_bytes<XBF16, TE>();
  constexpr int V = 8 * TE;          // values per thread (8 tokens x TE experts)
  constexpr int TS = V + 1;          // padded row of the level-1 sums in shared memory
  static_assert(2 * 32 * TS * 4 <= kNST * SB, "level-1 sums reuse the ring");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kNST];
  const int tid = threadIdx.x, p = tid & 127, half = tid >> 7;
  const int lane = tid & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kTM;
  const int e0 = blockIdx.x * TE;
  const int mv = static_cast<int>(min64(kTM, M - m0));
  const int ev = min(TE, E - e0);
  const int nch = static_cast<int>(H / kCH);
  const uint32_t base = smem_addr(smem);
  auto bar = [&](int s) { return smem_addr(&full[s]); };

  if (tid == 0) {
    for (int s = 0; s < kNST; ++s) mbar_init(bar(s), 1);
    mbar_fence_init();
  }
  __syncthreads();
  // Warp 0 requests chunk c into stage c % kNST: the router rows (no
  // kernel of this library writes them, so the first chunks go out before
  // the wait for the preceding kernel) and the token rows, one row per lane
  // (a thread issues a bulk copy only every few hundred cycles, and a chunk
  // is up to TE + kTM copies).  Lane 0 registers the stage's bytes first.
  static_assert(TE + kTM <= 32, "one copy per lane of warp 0");
  auto expect = [&](int c) {
    if (lane == 0)
      mbar_arrive_expect_tx(bar(c % kNST), static_cast<uint32_t>(mv * kCH * XB + ev * kCH * 4));
    __syncwarp();
  };
  auto issue_w = [&](int c) {  // lanes [0, ev)
    const int s = c % kNST;
    const uint32_t ws = base + s * SB + kTM * kCH * XB;
    if (lane < ev)
      bulk_g2s(ws + lane * kCH * 4, wr + int64_t(e0 + lane) * H + int64_t(c) * kCH, kCH * 4,
               bar(s));
  };
  auto issue_x = [&](int c) {  // lanes [TE, TE + mv)
    const int s = c % kNST;
    const uint32_t xs = base + s * SB;
    const int m = lane - TE;
    if (m >= 0 && m < mv)
      bulk_g2s(xs + m * kCH * XB,
               static_cast<const uint8_t *>(x) + ((m0 + m) * H + int64_t(c) * kCH) * XB,
               kCH * XB, bar(s));
  };
  const int npre = min(kNST, nch);
  if (tid < 32)
    for (int c = 0; c < npre; ++c) {
      expect(c);
      issue_w(c);
    }
  pdl_enter();
  if (counts && blockIdx.x == 0 && blockIdx.y == 0)
    for (int e = tid; e < E; e += blockDim.x) counts[e] = 0;
  if (tid < 32)
    for (int c = 0; c < npre; ++c) issue_x(c);

  float acc[8][TE];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < TE; ++e) acc[i][e] = 0.0f;

  int issued = npre, c = 0;
  bool aborted = false;
  for (; c < nch; ++c) {
    const int s = c % kNST;
    const bool ok = mbar_wait_bounded(bar(s), static_cast<uint32_t>((c / kNST) & 1), status);
    if (ok) {
      const uint8_t *st = smem + s * SB;
      const float *ws = reinterpret_cast<const float *>(st + kTM * kCH * XB);
#pragma unroll
      for (int j = 0; j < kCH / 128; ++j) {
        const int hl = p + 128 * j;
        float xv[8], wv[TE];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if constexpr (XBF16) {
            const uint16_t b = reinterpret_cast<const uint16_t *>(st)[(8 * half + i) * kCH + hl];
            xv[i] = __uint_as_float(static_cast<uint32_t>(b) << 16);
          } else {
            xv[i] = reinterpret_cast<const float *>(st)[(8 * half + i) * kCH + hl];
          }
        }
#pragma unroll
        for (int e = 0; e < TE; ++e) wv[e] = ws[e * kCH + hl];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int e = 0; e < TE; ++e) acc[i][e] = __fmaf_rn(xv[i], wv[e], acc[i][e]);
      }
    }
    // one barrier per chunk: every thread is done with stage s, and all
    // learn whether any wait gave up
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid < 32 && issued < nch) {
      // every thread's reads of the stage (generic proxy) before the copies'
      // writes (async proxy)
      fence_proxy_async_smem();
      expect(issued);
      issue_w(issued);
      issue_x(issued);
      ++issued;
    }
  }
  if (aborted) {
    // Wait (bounded) for the copies still landing, then leave.
    if (tid == 0)
      for (int u = c; u < issued; ++u)
        mbar_wait_bounded(bar(u % kNST), static_cast<uint32_t>((u / kNST) & 1), status);
    return;
  }

  // Level 1 inside groups of four lanes (partials 4l .. 4l+3): at offset 1 a
  // lane keeps half of its V values and adds the neighbour's copy of that
  // half (P0 + P1, P2 + P3), at offset 2 half again ((P0+P1) + (P2+P3)).
  // Lane bits (b1 b0) end with the V / 4 sums of value index
  // (V / 2) b0 + (V / 4) b1 + i.
  float v[V];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < TE; ++e) v[i * TE + e] = acc[i][e];
  {
    const bool up = (lane & 1) != 0;
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      const float send = up ? v[i] : v[i + V / 2];
      const float keep = up ? v[i + V / 2] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 1));
    }
  }
  {
    const bool up = (lane & 2) != 0;
#pragma unroll
    for (int i = 0; i < V / 4; ++i) {
      const float send = up ? v[i] : v[i + V / 4];
      const float keep = up ? v[i + V / 4] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 2));
    }
  }
  // t_l (l = p / 4) of value index vi lives at tb[half][l][vi ^ 8 (vi >> 5)]
  // (rows padded to TS; the four value blocks a warp writes at one step,
  // offsets {0, V/2, V/4, 3V/4}, land 8 banks apart after the swizzle).
  float *tb = reinterpret_cast<float *>(smem);
  const int l = p >> 2;
  const int vb = (V / 2) * (lane & 1) + (V / 4) * ((lane >> 1) & 1);
#pragma unroll
  for (int i = 0; i < V / 4; ++i) {
    const int vi = vb + i;
    tb[(half * 32 + l) * TS + (vi ^ ((vi >> 5) << 3))] = v[i];
  }
  __syncthreads();
  if (tid < 2 * V) {
    // Output o = tid: half o / V, value vi = o % V = token offset vi / TE,
    // expert vi % TE.
    const int oh = tid / V, vi = tid % V;
    const int col = vi ^ ((vi >> 5) << 3);
    float t[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) t[j] = tb[(oh * 32 + j) * TS + col];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int j = 0; j < o; ++j) t[j] = __fadd_rn(t[j], t[j + o]);
    const int m = 8 * oh + vi / TE, e = vi % TE;
    if (m < mv && e < ev) {
      float r = t[0];
      if (bias) r = __fadd_rn(r, bias[e0 + e]);
      logits[(m0 + m) * E + e0 + e] = r;
    }
  }
}

// a beats b: larger logit, or equal logit and lower index.
__device__ __forceinline__ bool beats(float la, int a, float lb, int b) {
  return la > lb || (la == lb && a < b);
}

// One warp per token: top-k by repeated warp arg-max, then the weights as a
// softmax over the selected logits (equal to the full softmax renormalised
// over the selection), expert histogram by atomics.
template <int EPL>  // logits per lane = ceil(E / 32)
__global__ void __launch_bounds__(256) router_topk_kernel(const float *__restrict__ logits,
                                                          int64_t M, int E, int k,
                                                          int32_t *__restrict__ idx,
                                                          float *__restrict__ w,
                                                          int32_t *__restrict__ counts) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t m = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (m >= M) return;
  float v[EPL];
#pragma unroll
  for (int t = 0; t < EPL; ++t) {
    const int e = lane + 32 * t;
    v[t] = e < E ? logits[m * E + e] : 0.0f;
  }
  uint32_t taken = 0;  // bit t: expert lane + 32t already selected
  float sel_l[kMaxK];
  int sel_e[kMaxK];
  for (int i = 0; i < k; ++i) {
    float bl = 0.0f;
    int be = -1;
#pragma unroll
    for (int t = 0; t < EPL; ++t) {
      const int e = lane + 32 * t;
      if (e < E && !((taken >> t) & 1u) && (be < 0 || beats(v[t], e, bl, be))) {
        bl = v[t];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ol = __shfl_xor_sync(0xFFFFFFFFu, bl, o);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
      if (oe >= 0 && (be < 0 || beats(ol, oe, bl, be))) {
        bl = ol;
        be = oe;
      }
    }
    sel_l[i] = bl;
    sel_e[i] = be;
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
  }
  if (lane == 0) {
    const float mx = sel_l[0];
    float z = 0.0f;
    float ex[kMaxK];
    for (int i = 0; i < k; ++i) {
      ex[i] = expf(sel_l[i] - mx);
      z += ex[i];
    }
    for (int i = 0; i < k; ++i) {
      idx[m * k + i] = sel_e[i];
      w[m * k + i] = ex[i] / z;
      if (counts) atomicAdd(counts + sel_e[i], 1);
    }
  }
}

// ---------------------------------------------------------------------------
// Grouping by expert (one block): counts, exclusive offsets, the ascending
// list of experts with tokens, and the assignments a = m*k + i sorted by
// (expert, a) -- a stable counting sort, so the layout is deterministic.
// Experts with at most light_max tokens (light_max > 0) also go to a second
// ascending list and get no 128-token tiles in the tile prefix: the
// tensor-core path skips them and the small-M kernels take them.
__global__ void __launch_bounds__(1024) moe_dispatch_kernel(const int32_t *__restrict__ idx,
                                                            int64_t MK, int E, int light_max,
                                                            MoeWork ws, uint32_t *status) {
  pdl_enter();
  extern __shared__ int32_t sm[];
  int32_t *cnt = sm;                 // [E]
  int32_t *cursor = sm + E;          // [E]
  int32_t *wcnt = sm + 2 * E;        // [32][E] per-warp counts of the current chunk
  __shared__ int32_t warp_c[32], warp_f[32], warp_t[32], warp_l[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int nwarps = nthreads >> 5;

  for (int e = tid; e < E; e += nthreads) cnt[e] = 0;
  __syncthreads();
  for (int64_t a = tid; a < MK; a += nthreads) {
    const int e = idx[a];
    if (e >= 0 && e < E) {
      atomicAdd(cnt + e, 1);
    } else {
      atomicOr(status, kDevBadExpert);
    }
  }
  __syncthreads();
  // Exclusive scan of counts (E <= blockDim: one element per thread) and of
  // the "has tokens" flags for the active-expert list.
  {
    // Also the tile prefix: ceil(count / 128) token tiles per expert (the
    // tensor-core path's work list; 128 = its largest token tile).
    const int e = tid;
    const int c = (e < E) ? cnt[e] : 0;
    const int f = c > 0 ? 1 : 0;
    const int lf = (c > 0 && c <= light_max) ? 1 : 0;
    const int tl = lf ? 0 : (c + 127) / 128;
    int sc = c, sf = f, st = tl, sl = lf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yc = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      const int yf = __shfl_up_sync(0xFFFFFFFFu, sf, o);
      const int yt = __shfl_up_sync(0xFFFFFFFFu, st, o);
      const int yl = __shfl_up_sync(0xFFFFFFFFu, sl, o);
      if (lane >= o) {
        sc += yc;
        sf += yf;
        st += yt;
        sl += yl;
      }
    }
    if (lane == 31) {
      warp_c[warp] = sc;
      warp_f[warp] = sf;
      warp_t[warp] = st;
      warp_l[warp] = sl;
    }
    __syncthreads();
    if (warp == 0) {
      int tc = lane < nwarps ? warp_c[lane] : 0;
      int tf = lane < nwarps ? warp_f[lane] : 0;
      int tt = lane < nwarps ? warp_t[lane] : 0;
      int tg = lane < nwarps ? warp_l[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xFFFFFFFFu, tc, o);
        const int yf = __shfl_up_sync(0xFFFFFFFFu, tf, o);
        const int yt = __shfl_up_sync(0xFFFFFFFFu, tt, o);
        const int yl = __shfl_up_sync(0xFFFFFFFFu, tg, o);
        if (lane >= o) {
          tc += yc;
          tf += yf;
          tt += yt;
          tg += yl;
        }
      }
      if (lane < nwarps) {  // inclusive over warps
        warp_c[lane] = tc;
        warp_f[lane] = tf;
        warp_t[lane] = tt;
        warp_l[lane] = tg;
      }
    }
    __syncthreads();
    const int exc = (warp > 0 ? warp_c[warp - 1] : 0) + sc - c;
    const int exf = (warp > 0 ? warp_f[warp - 1] : 0) + sf - f;
    const int ext = (warp > 0 ? warp_t[warp - 1] : 0) + st - tl;
    const int exl = (warp > 0 ? warp_l[warp - 1] : 0) + sl - lf;
    if (e < E) {
      ws.offsets[e] = exc;
      cursor[e] = exc;
      if (f) ws.active[exf] = e;
      if (lf) ws.active_light[exl] = e;
      ws.counts[e] = c;
      ws.tile_start[e] = ext;
    }
    if (e == E - 1) {
      ws.offsets[E] = exc + c;
      *ws.num_active = exf + f;
      *ws.num_light = exl + lf;
      ws.tile_start[E] = ext + tl;
    }
  }
  __syncthreads();
  // Stable placement, chunk by chunk in assignment order.
  for (int64_t base = 0; base < MK; base += nthreads) {
    for (int i = tid; i < nwarps * E; i += nthreads) wcnt[i] = 0;
    __syncthreads();
    const int64_t a = base + tid;
    int e = -1;
    if (a < MK) {
      e = idx[a];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int ee = tid; ee < E; ee += nthreads) {
      int run = 0;
      for (int w2 = 0; w2 < nwarps; ++w2) {
        const int t = wcnt[w2 * E + ee];
        wcnt[w2 * E + ee] = run;
        run += t;
      }
      wcnt[nwarps * E + ee] = run;  // chunk total (scratch row)
    }
    __syncthreads();
    if (e >= 0) {
      const int p = cursor[e] + wcnt[warp * E + e] + rank;
      ws.assign[p] = static_cast<int32_t>(a);
      ws.pos[a] = p;
    } else if (a < MK) {
      ws.pos[a] = -1;
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += nthreads) cursor[ee] += wcnt[nwarps * E + ee];
    __syncthreads();
  }
}

// y[m, n] = sum_{i<k} w[m, i] * out[pos(m, i), n], slot order, fp32.
template <bool YBF16>
__global__ void __launch_bounds__(256) moe_combine_kernel(int64_t M, int k, int64_t H,
                                                          const float *__restrict__ tw,
                                                          const int32_t *__restrict__ pos,
                                                          const float *__restrict__ out,
                                                          void *__restrict__ y) {
  pdl_enter();
  const int64_t H4 = H / 4;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= M * H4) return;
  const int64_t m = t / H4, n4 = t % H4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < k; ++i) {
    const int p = pos[m * k + i];
    if (p < 0) continue;
    const float wi = tw[m * k + i];
    const float4 o = ldg_f4(out + int64_t(p) * H + 4 * n4);
    acc.x = fmaf(wi, o.x, acc.x);
    acc.y = fmaf(wi, o.y, acc.y);
    acc.z = fmaf(wi, o.z, acc.z);
    acc.w = fmaf(wi, o.w, acc.w);
  }
  if constexpr (YBF16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t *>(&lo);
    v.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(y)[m * H4 + n4] = v;
  } else {
    reinterpret_cast<float4 *>(y)[m * H4 + n4] = acc;
  }
}

template <int MB, int EB, bool XBF16, int NS = 0>
cudaError_t run_logits(const void *x, int64_t M, int64_t H, const float *wr, const float *bias,
                       int E, float *logits, int32_t *counts, cudaStream_t s) {
  dim3 grid((E + EB - 1) / EB, static_cast<unsigned>((M + MB - 1) / MB));
  return launch_pdl(router_logits_kernel<MB, EB, XBF16, NS>, grid, dim3(128), 0, s, x, M, H, wr,
                    bias, E, logits, counts);
}

template <bool XBF16>
cudaError_t run_logits_tiled(const void *x, int64_t M, int64_t H, const float *wr,
                             const float *bias, int E, float *logits, int32_t *counts,
                             cudaStream_t s) {
  constexpr int TE = tiled::kTE;
  constexpr int smem = tiled::smem_bytes<XBF16, TE>();
  const cudaError_t err =
      ensure_smem(reinterpret_cast<const void *>(router_logits_tiled_kernel<XBF16, TE>), smem);
  if (err != cudaSuccess) return err;
  dim3 grid((E + TE - 1) / TE, static_cast<unsigned>((M + tiled::kTM - 1) / tiled::kTM));
  return launch_pdl(router_logits_tiled_kernel<XBF16, TE>, grid, dim3(tiled::kThreads), smem, s, x, M,
                    H, wr, bias, E, logits, counts, device_status());
}

template <int EPL>
cudaError_t run_topk(const float *logits, int64_t M, int E, int k, int32_t *idx, float *w,
                     int32_t *counts, cudaStream_t s) {
  const int64_t threads = M * 32;
  return launch_pdl(router_topk_kernel<EPL>, dim3(static_cast<unsigned>((threads + 255) / 256)),
                    dim3(256), 0, s, static_cast<const float *>(logits), M, E, k, idx, w, counts);
}

}  // namespace

size_t router_logits_bytes(int64_t M, int E) { return static_cast<size_t>(M) * E * 4; }

cudaError_t launch_router(const void *x, bool x_bf16, int64_t M, int64_t H, const float *wr,
                          const float *bias, int E, int k, float *logits, int32_t *idx,
                          float *w, int32_t *counts, cudaStream_t s) {
  cudaError_t err;
  // Small batches: fewer experts per block so that the 4 MB router matrix is
  // spread over more SMs.
  if (M <= 8 && H == 4096) {
    // decode: one expert and two tokens per block, the router row preloaded
    // in registers and all of the two token rows' loads in flight at once
    err = x_bf16 ? run_logits<2, 1, true, 32>(x, M, H, wr, bias, E, logits, counts, s)
                 : run_logits<2, 1, false, 32>(x, M, H, wr, bias, E, logits, counts, s);
  } else if (M > 64 && H % tiled::kCH == 0 && (M + tiled::kTM - 1) / tiled::kTM <= 65535) {
    // larger batches: tiles staged through shared memory
    err = x_bf16 ? run_logits_tiled<true>(x, M, H, wr, bias, E, logits, counts, s)
                 : run_logits_tiled<false>(x, M, H, wr, bias, E, logits, counts, s);
  } else if (M <= 64) {
    err = x_bf16 ? run_logits<8, 2, true>(x, M, H, wr, bias, E, logits, counts, s)
                 : run_logits<8, 2, false>(x, M, H, wr, bias, E, logits, counts, s);
  } else {
    err = x_bf16 ? run_logits<8, 8, true>(x, M, H, wr, bias, E, logits, counts, s)
                 : run_logits<8, 8, false>(x, M, H, wr, bias, E, logits, counts, s);
  }
  if (err != cudaSuccess) return err;
  const int epl = (E + 31) / 32;
  if (epl <= 1) return run_topk<1>(logits, M, E, k, idx, w, counts, s);
  if (epl <= 2) return run_topk<2>(logits, M, E, k, idx, w, counts, s);
  if (epl <= 4) return run_topk<4>(logits, M, E, k, idx, w, counts, s);
  if (epl <= 8) return run_topk<8>(logits, M, E, k, idx, w, counts, s);
  if (epl <= 16) return run_topk<16>(logits, M, E, k, idx, w, counts, s);
  return run_topk<32>(logits, M, E, k, idx, w, counts, s);
}

size_t moe_dispatch_smem(int E) {
  // cnt + cursor + (32 warps + 1 total row) x E
  return static_cast<size_t>(2 * E + 33 * E) * sizeof(int32_t);
}

cudaError_t launch_moe_dispatch(const int32_t *idx, int64_t M, int k, int E, int light_max,
                                const MoeWork &ws, cudaStream_t s) {
  const int64_t MK = M * k;
  int threads = 1024;
  if (MK < 1024) threads = static_cast<int>(((MK + 31) / 32) * 32);
  if (threads < E) threads = ((E + 31) / 32) * 32;  // the scan needs one thread per expert
  if (threads > 1024) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(2 * E + (threads / 32 + 1) * E) * sizeof(int32_t);
  cudaError_t err = ensure_smem(reinterpret_cast<const void *>(moe_dispatch_kernel),
                                static_cast<int>(moe_dispatch_smem(E)));
  if (err != cudaSuccess) return err;
  return launch_pdl(moe_dispatch_kernel, dim3(1), dim3(threads), smem, s, idx, MK, E, light_max,
                    ws, device_status());
}

cudaError_t launch_moe_combine(int64_t M, int k, int64_t H, const float *topk_w,
                               const MoeWork &ws, void *y, bool y_bf16, cudaStream_t s) {
  const int64_t threads = M * (H / 4);
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  const int32_t *pos = ws.pos;
  const float *out = ws.out;
  if (y_bf16)
    return launch_pdl(moe_combine_kernel<true>, dim3(blocks), dim3(256), 0, s, M, k, H, topk_w, pos,
                      out, y);
  return launch_pdl(moe_combine_kernel<false>, dim3(blocks), dim3(256), 0, s, M, k, H, topk_w, pos,
                    out, y);
}

}  // namespace qmm
