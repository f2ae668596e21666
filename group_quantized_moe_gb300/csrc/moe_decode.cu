// moe_decode.cu -- the routed MoE layer of a decode batch (at most 8 tokens)
// in one launch: router logits, top-k and weights, grouping by expert,
// gate/up with SwiGLU, down, weighted combine.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5: the
// router is a linear layer, a softmax and a top-k; the tokens of an expert
// are grouped so that its weights are read once; the outputs are combined by
// a weighted sum.  The same page's engine runs the whole step as one loop;
// on the GPU the step is otherwise five dependent launches, each paying a
// launch and a pipeline fill.
//
// One cooperative launch of the small-M expert kernel's configuration (two
// CTAs of eight warps per SM, all resident at once), in phases separated by
// grid barriers (a counter in the workspace, zeroed before the launch; every
// wait bounded):
//   1. logits: each half-CTA (128 threads) computes (expert, token pair)
//      units in the fixed order of moe_route_topk (128 fma partial sums, the
//      same reduction tree, then the bias), so indices and weights are those
//      of moe_route_topk bit for bit;
//      -- barrier --
//   2. top-k: every CTA selects the k experts of every token itself (one
//      warp per token, larger logit first, lower index on ties) and the
//      weights (softmax over the selection); CTA 0 also writes the optional
//      outputs (indices, weights, histogram);
//   3. gate/up: the small-M kernel body (one token per pass), which groups
//      the assignments in its prologue from the CTA's own top-k;
//   4. down: the same body; its first weight tiles are requested before the
//      barrier that waits for every CTA's h rows;
//      -- barriers (h complete, then expert outputs complete) --
//   5. combine: y[m, n] = sum_i w[m, i] out[pos(m, i), n], slots in order.
#include "smallm_kernel.cuh"

namespace qmm {
namespace {

constexpr int kDecMaxTok = 8;    // tokens
constexpr int kDecMaxK = 16;     // slots per token
constexpr int kDecEPL = 8;       // logits per lane in the top-k: E <= 256

struct DecodeArgs {
  smallm::Args gu, dn;  // the two expert phases (grouped from the kernel's own top-k)
  const void *x;        // [M, H] fp32 or bf16
  const float *wr;      // [E, H]
  const float *bias;    // [E] or NULL
  float *logits;        // [M, E] (workspace)
  int32_t *topk_idx;    // [M, k] or NULL
  float *topk_w;        // [M, k] or NULL
  int32_t *counts;      // [E] or NULL
  void *y;              // [M, H]
  unsigned *bar;        // grid barrier counter, zero at launch
  uint32_t *status;
  int M, H, E, k;
  bool y_bf16;
};

// Grid barrier number `n` (1, 2, ...): returns when every CTA has arrived n
// times, or false after the wait limit (QMM_DEV_WAIT_TIMEOUT set).  All
// threads of the CTA call it; they all get the same answer.
__device__ bool grid_sync(unsigned *bar, unsigned n, uint32_t *status, volatile int *flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const unsigned target = n * gridDim.x;
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    while (true) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= target) break;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        atomicOr(status, kDevWaitTimeout);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    *flag = ok;
  }
  __syncthreads();
  return *flag != 0;
}

// a beats b: larger logit, or equal logit and lower index.
__device__ __forceinline__ bool dec_beats(float la, int a, float lb, int b) {
  return la > lb || (la == lb && a < b);
}

template <bool XBF16>
__device__ __forceinline__ float dec_x(const void *x, int64_t i) {
  if constexpr (XBF16)
    return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(x)[i]) << 16);
  else
    return __ldg(static_cast<const float *>(x) + i);
}

template <int BITS, int KWG, int KWD, bool XBF16>
__global__ void __launch_bounds__(smallm::kThreads, 2) moe_decode_kernel(const DecodeArgs f) {
  __shared__ float xch[2][2][32][2];  // [half][slot][lane][token]
  __shared__ int32_t s_topk[kDecMaxTok * kDecMaxK];
  __shared__ float s_topw[kDecMaxTok * kDecMaxK];
  __shared__ int bar_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = threadIdx.x >> 7, p = threadIdx.x & 127, hw = warp & 3;
  const int M = f.M, H = f.H, E = f.E, k = f.k;

  // ---- 1. router logits: unit u = (expert u / NP, tokens 2 (u mod NP) +
  // 0..1), partial p of a unit sums columns p, p + 128, ... with fma in
  // order; (P0 + P1) + (P2 + P3) over each lane quad; then t_l += t_(l+o)
  // for o = 16, 8, 4, 2, 1; then the bias.
  if (f.counts && blockIdx.x == 0)
    for (int e = threadIdx.x; e < E; e += blockDim.x) f.counts[e] = 0;
  const int NP = (M + 1) / 2, U = E * NP;
  for (int ub = 2 * blockIdx.x; ub < U; ub += 2 * gridDim.x) {
    const int u = ub + half;
    const bool live = u < U;
    const int e = live ? u / NP : 0, m0 = live ? 2 * (u - (u / NP) * NP) : 0;
    const int m1 = m0 + 1 < M ? m0 + 1 : m0;
    float a0 = 0.0f, a1 = 0.0f;
    const float *wrow = f.wr + static_cast<int64_t>(e) * H;
#pragma unroll 8
    for (int h = p; h < H; h += 128) {
      const float w = __ldg(wrow + h);
      a0 = __fmaf_rn(dec_x<XBF16>(f.x, static_cast<int64_t>(m0) * H + h), w, a0);
      a1 = __fmaf_rn(dec_x<XBF16>(f.x, static_cast<int64_t>(m1) * H + h), w, a1);
    }
    a0 = __fadd_rn(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, 1));
    a1 = __fadd_rn(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 1));
    a0 = __fadd_rn(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, 2));
    a1 = __fadd_rn(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 2));
    // o = 16: t_l (warps 0-1 of the half) += t_(l+16) (warps 2-3)
    if (hw >= 2 && (lane & 3) == 0) {
      xch[half][hw - 2][lane][0] = a0;
      xch[half][hw - 2][lane][1] = a1;
    }
    __syncthreads();
    if (hw < 2 && (lane & 3) == 0) {
      a0 = __fadd_rn(a0, xch[half][hw][lane][0]);
      a1 = __fadd_rn(a1, xch[half][hw][lane][1]);
    }
    __syncthreads();
    // o = 8: warp 0 of the half += warp 1
    if (hw == 1 && (lane & 3) == 0) {
      xch[half][0][lane][0] = a0;
      xch[half][0][lane][1] = a1;
    }
    __syncthreads();
    if (hw == 0) {
      if ((lane & 3) == 0) {
        a0 = __fadd_rn(a0, xch[half][0][lane][0]);
        a1 = __fadd_rn(a1, xch[half][0][lane][1]);
      }
      // o = 4, 2, 1 between lanes 4l and 4(l + o)
      a0 = __fadd_rn(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, 16));
      a1 = __fadd_rn(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 16));
      a0 = __fadd_rn(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, 8));
      a1 = __fadd_rn(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 8));
      a0 = __fadd_rn(a0, __shfl_xor_sync(0xFFFFFFFFu, a0, 4));
      a1 = __fadd_rn(a1, __shfl_xor_sync(0xFFFFFFFFu, a1, 4));
      if (lane == 0 && live) {
        const float b = f.bias ? f.bias[e] : 0.0f;
        f.logits[static_cast<int64_t>(m0) * E + e] = f.bias ? __fadd_rn(a0, b) : a0;
        if (m0 + 1 < M) f.logits[static_cast<int64_t>(m0 + 1) * E + e] = f.bias ? __fadd_rn(a1, b) : a1;
      }
    }
    __syncthreads();
  }
  if (!grid_sync(f.bar, 1, f.status, &bar_flag)) return;

  // ---- 2. top-k of every token (warp m), weights as a softmax over the
  // selected logits
  if (warp < M) {
    const int m = warp;
    float v[kDecEPL];
#pragma unroll
    for (int t = 0; t < kDecEPL; ++t) {
      const int e = lane + 32 * t;
      v[t] = e < E ? __ldcg(f.logits + static_cast<int64_t>(m) * E + e) : 0.0f;
    }
    uint32_t taken = 0;
    float sel_l[kDecMaxK];
    int sel_e[kDecMaxK];
    for (int i = 0; i < k; ++i) {
      float bl = 0.0f;
      int be = -1;
#pragma unroll
      for (int t = 0; t < kDecEPL; ++t) {
        const int e = lane + 32 * t;
        if (e < E && !((taken >> t) & 1u) && (be < 0 || dec_beats(v[t], e, bl, be))) {
          bl = v[t];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ol = __shfl_xor_sync(0xFFFFFFFFu, bl, o);
        const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
        if (oe >= 0 && (be < 0 || dec_beats(ol, oe, bl, be))) {
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
      float ex[kDecMaxK];
      for (int i = 0; i < k; ++i) {
        ex[i] = expf(sel_l[i] - mx);
        z += ex[i];
      }
      for (int i = 0; i < k; ++i) {
        const float w = ex[i] / z;
        s_topk[m * k + i] = sel_e[i];
        s_topw[m * k + i] = w;
        if (blockIdx.x == 0) {
          if (f.topk_idx) f.topk_idx[m * k + i] = sel_e[i];
          if (f.topk_w) f.topk_w[m * k + i] = w;
          if (f.counts) atomicAdd(f.counts + sel_e[i], 1);
        }
      }
    }
  }
  __syncthreads();

  // ---- 3. gate/up (h rows of every assignment), grouped from s_topk
  smallm::smallm_body<BITS, 32, KWG, smallm::kGateUp, XBF16, 1>(f.gu, s_topk, []() { return true; });

  // ---- 4. down, after every CTA's h rows (barrier 2)
  bool ok = true;
  smallm::smallm_body<BITS, 32, KWD, smallm::kDown, false, 1>(f.dn, s_topk, [&]() {
    ok = grid_sync(f.bar, 2, f.status, &bar_flag);
    return ok;
  });
  if (!ok || !grid_sync(f.bar, 3, f.status, &bar_flag)) return;

  // ---- 5. combine, slots in order
  const int64_t total = static_cast<int64_t>(M) * H;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(i / H);
    const int64_t n = i - static_cast<int64_t>(m) * H;
    float acc = 0.0f;
    for (int s = 0; s < k; ++s) {
      const int pp = __ldcg(f.gu.pos_out + m * k + s);
      acc = fmaf(s_topw[m * k + s], __ldcg(f.dn.ws.out + static_cast<int64_t>(pp) * H + n), acc);
    }
    store_y(f.y, i, acc, f.y_bf16);
  }
}

template <int BITS, bool XBF16>
cudaError_t launch_decode(const DecodeArgs &f, cudaStream_t s) {
  auto kern = moe_decode_kernel<BITS, 4, 2, XBF16>;  // H = 4096: four warps per row; I = 2048: two
  const int smem = smallm::Cfg<1>::smem_bytes(f.E, f.gu.MK);
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(kern), smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, smallm::kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  per_sm = per_sm > 2 ? 2 : per_sm;
  e = cudaMemsetAsync(f.bar, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(per_sm * sm_count());
  cfg.blockDim = dim3(smallm::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, f);
  count_launch();
  return e;
}

}  // namespace

bool moe_decode_supported(const QMat &gate, const QMat &down, int64_t M, int E, int k, int64_t H,
                          int64_t I) {
  return M >= 1 && M <= kDecMaxTok && k >= 1 && k <= kDecMaxK && E >= k && E <= 32 * kDecEPL &&
         H == 4096 && I == 2048 && gate.bits == down.bits &&
         smallm_supported(gate.bits, gate.group, H) && smallm_supported(down.bits, down.group, I);
}

cudaError_t launch_moe_decode(const void *x, bool x_bf16, int64_t M, const float *wr,
                              const float *bias, int E, int k, const QMat &gate, const QMat &up,
                              const QMat &down, const MoeWork &ws, float *logits,
                              unsigned *bar, int32_t *topk_idx, float *topk_w, int32_t *counts,
                              void *y, bool y_bf16, cudaStream_t s) {
  DecodeArgs f{};
  const int64_t MK = M * k;
  f.gu = smallm::base_args(gate, 2);
  f.gu.w1 = up;
  f.gu.E = E;
  f.gu.k = k;
  f.gu.ws = ws;
  f.gu.x = x;
  f.gu.MK = MK;
  f.gu.pos_out = ws.pos;
  f.dn = smallm::base_args(down, 1);
  f.dn.E = E;
  f.dn.k = k;
  f.dn.ws = ws;
  f.dn.MK = MK;
  f.x = x;
  f.wr = wr;
  f.bias = bias;
  f.logits = logits;
  f.topk_idx = topk_idx;
  f.topk_w = topk_w;
  f.counts = counts;
  f.y = y;
  f.y_bf16 = y_bf16;
  f.bar = bar;
  f.status = device_status();
  f.M = static_cast<int>(M);
  f.H = static_cast<int>(gate.cols);
  f.E = E;
  f.k = k;
  if (gate.bits == 4)
    return x_bf16 ? launch_decode<4, true>(f, s) : launch_decode<4, false>(f, s);
  return x_bf16 ? launch_decode<8, true>(f, s) : launch_decode<8, false>(f, s);
}

}  // namespace qmm
