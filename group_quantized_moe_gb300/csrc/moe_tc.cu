// moe_tc.cu -- routed experts on the 5th-generation tensor cores (tcgen05)
// for batched prefill: grouped GEMMs over the experts' token lists with the
// weights dequantised on the fly.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5:
// tokens routed to the same expert are gathered so that the expert's weights
// are read once for all of them; section 3.2: dequantise (q - zp) * scale
// inside the matmul instead of materialising the weights.  "I ran a
// 284B-parameter LLM from 3.2GB of RAM in plain C" names batched prefill with
// expert reuse as the missing piece.
//
// Formulation (per expert e with tokens T_e, features tiled by 128):
//   D[f, t] = sum_k W_e[f, k] * X[t, k]       (swap-AB: features on the MMA M
//                                               side, tokens on N = 16..128)
//   gate/up: D_g, D_u in TMEM, epilogue h = silu(D_g) * D_u -> fp16 [tok, I]
//   down:    D_d in TMEM, epilogue -> fp32 out[tok, H]
//
// CTA = 17 warps, one CTA per SM, persistent over work items
// (token tile of an expert, 128-feature tile):
//   warp 12 (one lane): TMA producer of weight codes [128 rows x 64 K] into a
//     ring (64B swizzle for INT8).
//   warp 13 (one lane): TMA producer of token rows [npad x 64 K] fp16 into
//     the B stages (128B swizzle, the canonical K-major operand layout), one
//     box of 16, 32, 64 or 128 rows per stage.
//   warps 0-11 = three dequant warpgroups; warpgroup g converts the stages
//     whose global number is g (mod 3), thread t the whole 64-K row t % 128
//     of each weight tile, so three stages are being converted at once (one
//     stage's conversion is latency bound; stages pipeline).  A stage's codes
//     are read into registers and its code slot released at once; they are
//     converted to fp16 (q - zp) * s, exact up to the final fp16 rounding,
//     and stored with tcgen05.st straight into tensor memory, where the MMA
//     reads its A operand (row = TMEM lane, two K values per 32-bit column);
//     this keeps shared memory for the TMA rings.  After an item's last stage
//     all three run the epilogue (tcgen05.ld from TMEM, 16-token column
//     blocks in turn).
//   warps 14 and 15 (one lane each): issue the tcgen05.mma (kind::f16, fp32
//     accumulate) of one weight matrix each (gate, up; down uses the first),
//     every stage in order, with one tcgen05.commit per stage; a stage's A
//     and B slots are free once both commits have arrived.  Warp 14 also
//     allocates TMEM.
//   warp 16: the row exponents of each item's weight tile (see below), one
//     item ahead.
// Every wait is bounded; on a timeout the CTA raises QMM_DEV_WAIT_TIMEOUT,
// stops issuing work, waits (bounded) for what is in flight, frees its TMEM
// and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M)
constexpr int kBN = 128;        // max tokens per tile (MMA N)
constexpr int kBK = 64;         // K per stage
constexpr int kDequantGroups = 3;  // warpgroups converting stages round-robin
constexpr int kDequantWarps = 4 * kDequantGroups;  // warps 0-11
constexpr int kWarpCodes = kDequantWarps;          // TMA producer of weight codes
constexpr int kWarpRows = kDequantWarps + 1;       // TMA producer of token rows
constexpr int kWarpMma = kDequantWarps + 2;        // MMA issuers (one per matrix)
constexpr int kWarpRexp = kDequantWarps + 4;       // row exponents, one item ahead
constexpr int kThreads = (kDequantWarps + 5) * 32;
constexpr int kACols = kBK / 2;         // TMEM columns of one A tile stage
constexpr int kBTile = kBN * kBK * 2;   // 16 KB fp16
constexpr int kCTile = kBM * kBK;       // 8 KB INT8 codes (64B swizzle)

template <int NT>
struct Ring;  // NT = weight tiles sharing one token tile (2: gate+up, 1: down)
// Three independent rings: codes (TMA -> dequant), A (dequant -> MMA) and
// B (TMA -> MMA), each with its own depth.
// TMEM: accumulators in columns [0, 256) (gate at 0 and up at 128 for NT=2,
// one at 0 for NT=1), then the A stages: NT=2 uses 256 + 4*2*32 = 512
// columns, NT=1 uses 256 + 4*32 = 384 (allocation 512).
// The A and B rings have the same depth, so that the MMA issuers' commits
// free the A and B slots of a stage together.  The code ring's depth is a multiple of
// the three dequant warpgroups: stage gs goes to code slot gs mod kC and to
// warpgroup gs mod 3, so every use of a slot belongs to the same warpgroup,
// in order.  Its wait on the slot's barrier can then never see a phase two
// uses old (which the parity test would take as complete: with a depth that
// is not a multiple of 3, a warpgroup that runs ahead could read a slot whose
// copy is still landing and arrive on the wrong phase of its free barrier).
// A warpgroup releases its slot as soon as it has read the codes, so nearly
// the whole ring is loading at any time (deeper rings measured slower).
template <>
struct Ring<2> {
  static constexpr int kA = 4, kB = 4, kC = 6;
  static constexpr uint32_t kTmemCols = 512;
};
template <>
struct Ring<1> {
  static constexpr int kA = 4, kB = 4, kC = 9;
  static constexpr uint32_t kTmemCols = 512;
};
static_assert(Ring<2>::kC % kDequantGroups == 0 && Ring<1>::kC % kDequantGroups == 0,
              "each code slot must belong to one dequant warpgroup");

template <int NT>
struct Smem {
  static constexpr int kA = Ring<NT>::kA, kB = Ring<NT>::kB, kC = Ring<NT>::kC;
  static constexpr int b_off = 0;
  static constexpr int c_off = b_off + kB * kBTile;
  static constexpr int bar_off = c_off + kC * NT * kCTile;
  // barriers: c_full[kC], c_free[kC], a_full[kA], ab_free[kA], b_full[kB],
  // acc_full, acc_free, rexp_full[2], rexp_free[2], drain[2]
  static constexpr int nbar = 2 * kC + 2 * kA + kB + 2 + 4 + 2;
  static constexpr int misc_off = bar_off + nbar * 8;
  static constexpr int rexp_off = misc_off + 16;  // int32 [2 slots][NT][128 rows]
  static constexpr int cs_off = rexp_off + 2 * NT * kBM * 4;  // fp32 [2 slots][128 tokens]
  static constexpr int meta_off = cs_off + 2 * kBN * 4;  // offsets[E+1], tile_start[E+1]
  static constexpr int bytes_for(int E) { return meta_off + 8 * (E + 1) + 1024; }
};

struct TcArgs {
  int E, k;
  int64_t rows;          // weight rows per expert (I for gate/up, H for down)
  int64_t K;             // reduction length (H for gate/up, I for down)
  int G;                 // groups per row
  int group_shift;
  const float *sc[2];    // scales of the NT matrices (stacked)
  const int32_t *zp[2];
  int64_t gstride[2];    // elements between experts
  const int32_t *offsets;      // [E + 1] token-list offsets (sorted order)
  const int32_t *tile_start;   // [E + 1] prefix of 128-token tiles per expert
  const float *colscale;       // [MK] power of two that undoes the scaling of
                               // each fp16 token row (gate/up: x, down: h)
  float *out;            // gate/up: fp32 h [MK, I]; down: fp32 out [MK, H]
  int64_t out_ld;        // elements per output row
  uint32_t *status;
  // Linear layer (one matrix, M token rows, rows = N may be ragged): lin_M > 0
  // replaces offsets / tile_start ({0, M} and one expert); the K range is
  // split nsplit ways, split s writing its partial sums at out + s out_split.
  int lin_M;
  int nsplit;
  int64_t out_split;
};

// ------------------------------------------------------------ PTX wrappers

// L2 cache policies: weight codes stream through L2 once per token tile
// (evict first); the gathered token rows are re-read by every feature tile
// of their expert (evict last), so the code stream must not push them out.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16, cta_group::1.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (asynchronous;
// tmem_wait_st() waits for all of this thread's stores).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 16 columns at each of two TMEM addresses of this thread's lane, both loads
// in flight before the single wait (one asm statement, so no use of the
// outputs can be scheduled before the wait).
__device__ __forceinline__ void tmem_ld16x2(uint32_t a0, uint32_t a1, float (&v0)[16],
                                            float (&v1)[16]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v0[i] = __uint_as_float(r[i]);
    v1[i] = __uint_as_float(r[16 + i]);
  }
}

// 16 columns at one TMEM address of this thread's lane.
__device__ __forceinline__ void tmem_ld16x1(uint32_t a0, float (&v0)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(a0)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v0[i] = __uint_as_float(r[i]);
}

// Shared-memory operand descriptor: K-major, 128B swizzle, 8-row groups 1024 B
// apart (SBO), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor: fp16 x fp16 -> fp32, both K-major, M = 128, N.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
}

// Bounded wait that also gives up at once when the CTA has aborted.
__device__ __forceinline__ bool wait_ok(uint32_t bar, uint32_t parity, uint32_t *status,
                                        volatile int *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kDevWaitTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// Work item -> (expert, token tile, feature tile).
struct Item {
  int e, t0, ntok, f, ks;
};

// s_off / s_ts: the token-list offsets and tile prefix, staged in shared
// memory.  Items are ordered (token tile, feature tile, K split), the split
// fastest.
__device__ __forceinline__ Item decode_item(const int32_t *s_off, const int32_t *s_ts, int E,
                                            int64_t item, int ftiles, int nsplit) {
  Item it;
  const int64_t tf = item / nsplit;
  it.ks = static_cast<int>(item % nsplit);
  const int tau = static_cast<int>(tf / ftiles);
  it.f = static_cast<int>(tf % ftiles);
  // last expert whose first tile index is <= tau
  int lo = 0, hi = E;  // s_ts[lo] <= tau < s_ts[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_ts[mid] <= tau) lo = mid;
    else hi = mid;
  }
  it.e = lo;
  const int tt = tau - s_ts[lo];
  const int base = s_off[lo];
  const int cnt = s_off[lo + 1] - base;
  it.t0 = base + tt * kBN;
  it.ntok = min(kBN, cnt - tt * kBN);
  return it;
}

// SwiGLU's silu for a result that is rounded to fp16 before the down GEMM:
// the fast exponential and division (a few ulp of fp32) are far inside fp16
// rounding; the exponent is clamped so that the divisor stays finite (silu(g)
// for g < -80 is below 1e-33 |g|).
__device__ __forceinline__ float silu_f(float g) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f)));
}

// INT8 codes (stored q - 128) of one 16-byte chunk -> 16 fp16 weights
// (q - zp) * s, packed two per 32-bit word in K order.
__device__ __forceinline__ void dequant16(uint4 v, __half2 mz2, __half2 s2, uint4 &o0, uint4 &o1) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;               // q in each byte
    const uint32_t h01 = __byte_perm(u, 0x64646464u, 0x4140u);  // {1024+q0, 1024+q1}
    const uint32_t h23 = __byte_perm(u, 0x64646464u, 0x4342u);  // {1024+q2, 1024+q3}
    __half2 d01 = __hsub2(*reinterpret_cast<const __half2 *>(&h01), mz2);  // exact q - zp
    __half2 d23 = __hsub2(*reinterpret_cast<const __half2 *>(&h23), mz2);
    d01 = __hmul2(d01, s2);
    d23 = __hmul2(d23, s2);
    r[2 * i] = *reinterpret_cast<uint32_t *>(&d01);
    r[2 * i + 1] = *reinterpret_cast<uint32_t *>(&d23);
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// The same for a group outside the fast form's exact range: each weight
// (q - zp) s' formed as the oracle forms it in fp32 (the difference in 64
// bits, one conversion, one product) and rounded to fp16 once.
__device__ __forceinline__ void dequant16_exact(uint4 v, int32_t zp, float s, uint4 &o0,
                                                uint4 &o1) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t u = w[i] ^ 0x80808080u;
    float f[4];
#pragma unroll
    for (int b = 0; b < 4; ++b)
      f[b] = __ll2float_rn(static_cast<int64_t>((u >> (8 * b)) & 0xFFu) - zp) * s;
    __half2 d01 = __floats2half2_rn(f[0], f[1]);
    __half2 d23 = __floats2half2_rn(f[2], f[3]);
    r[2 * i] = *reinterpret_cast<uint32_t *>(&d01);
    r[2 * i + 1] = *reinterpret_cast<uint32_t *>(&d23);
  }
  o0 = make_uint4(r[0], r[1], r[2], r[3]);
  o1 = make_uint4(r[4], r[5], r[6], r[7]);
}

// One matrix's 64 codes of a thread's weight row (four 16-byte chunks in K
// order) -> 64 fp16 weights stored into 32 TMEM columns of the thread's lane
// at taddr (asynchronous: tmem_wait_st() waits for the stores).  kChoose:
// the fast or the exact form per this thread's `fast`; otherwise the fast
// form.  Every lane of the warp must call it (the stores are warp-collective).
template <bool kChoose>
__device__ __forceinline__ void convert_row(const uint4 (&cv)[4], __half2 mz2, __half2 s2,
                                            int32_t zp, float s, bool fast, uint32_t taddr) {
  uint32_t packed[32];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 o0, o1;
    if (!kChoose || fast)
      dequant16(cv[j], mz2, s2, o0, o1);
    else
      dequant16_exact(cv[j], zp, s, o0, o1);
    packed[8 * j + 0] = o0.x;
    packed[8 * j + 1] = o0.y;
    packed[8 * j + 2] = o0.z;
    packed[8 * j + 3] = o0.w;
    packed[8 * j + 4] = o1.x;
    packed[8 * j + 5] = o1.y;
    packed[8 * j + 6] = o1.z;
    packed[8 * j + 7] = o1.w;
  }
  tmem_st16(taddr, packed);
  tmem_st16(taddr + 16, packed + 16);
}

// 2^s and 2^-s for the power of two s that puts a positive magnitude m into
// [2^14, 2^15) (s clamped to [-126, 126], so that both are normal fp32; m = 0
// gives the largest s).  Read from m's exponent bits.
__device__ __forceinline__ void pow2_to_fp16_range(float m, float &up, float &down) {
  const int e = ((__float_as_int(m) >> 23) & 0xFF) - 127;
  const int sh = max(-126, min(126, 14 - e));
  up = __int_as_float((127 + sh) << 23);
  down = __int_as_float((127 - sh) << 23);
}

// NT = 2: gate/up with SwiGLU epilogue (fp32 h); NT = 1: down (fp32 out).
template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    moe_tc_kernel(const __grid_constant__ CUtensorMap tm_codes0,
                  const __grid_constant__ CUtensorMap tm_codes1,
                  const __grid_constant__ CUtensorMap tm_x16,
                  const __grid_constant__ CUtensorMap tm_x32,
                  const __grid_constant__ CUtensorMap tm_x64,
                  const __grid_constant__ CUtensorMap tm_x128, TcArgs a) {
  pdl_enter();
  using S = Smem<NT>;
  constexpr int kA = S::kA, kB = S::kB, kC = S::kC;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (swizzled tiles).
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  const uint32_t sB = base + S::b_off, sC = base + S::c_off;
  const uint32_t bar0 = base + S::bar_off;
  static_assert(kA == kB, "A and B slots are freed together");
  auto c_full = [&](int i) { return bar0 + 8 * i; };
  auto c_free = [&](int i) { return bar0 + 8 * (kC + i); };
  auto a_full = [&](int i) { return bar0 + 8 * (2 * kC + i); };
  // A and B slot s are freed together by the stage's MMA commits
  auto ab_free = [&](int slot) { return bar0 + 8 * (2 * kC + kA + slot); };
  auto b_full = [&](int i) { return bar0 + 8 * (2 * kC + 2 * kA + i); };
  const uint32_t acc_full = bar0 + 8 * (2 * kC + 2 * kA + kB);
  const uint32_t acc_free = acc_full + 8;
  // row-exponent slots: filled by the exponent warp one item ahead
  auto rexp_full = [&](int i) { return acc_free + 8 + 8 * i; };
  auto rexp_free = [&](int i) { return acc_free + 24 + 8 * i; };
  // per MMA issuer: tracks its MMAs in flight after an abort
  auto drain_bar = [&](int i) { return acc_free + 40 + 8 * i; };
  int32_t *s_rexp = reinterpret_cast<int32_t *>(gbase + S::rexp_off);
  float *s_cs = reinterpret_cast<float *>(gbase + S::cs_off);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + S::misc_off);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(gbase + S::misc_off + 4);
  // written, never read: see the release of a code slot below
  const uint32_t sink = base + S::misc_off + 8;
  int32_t *s_off = reinterpret_cast<int32_t *>(gbase + S::meta_off);
  int32_t *s_ts = s_off + a.E + 1;
  if (a.lin_M > 0) {
    if (threadIdx.x == 0) {  // one "expert" holding the M rows of x
      s_off[0] = 0;
      s_off[1] = a.lin_M;
      s_ts[0] = 0;
      s_ts[1] = (a.lin_M + kBN - 1) / kBN;
    }
  } else {
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) {
      s_off[i] = a.offsets[i];
      s_ts[i] = a.tile_start[i];
    }
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t kTmemCols = Ring<NT>::kTmemCols;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kC; ++i) {
      mbar_init(c_full(i), 1);
      mbar_init(c_free(i), 4);  // one arrival per warp of the converting warpgroup
    }
    for (int i = 0; i < kA; ++i) mbar_init(a_full(i), 4);
    // two commits per gate/up stage, one per down stage (see the MMA issuers)
    for (int i = 0; i < kA; ++i) mbar_init(ab_free(i), NT);  // one commit per issuer
    for (int i = 0; i < kB; ++i) mbar_init(b_full(i), 1);
    mbar_init(acc_full, NT);
    mbar_init(acc_free, kDequantWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(rexp_full(i), 32);             // every lane of the exponent warp
      mbar_init(rexp_free(i), kDequantWarps);  // one arrival per dequant warp
    }
    mbar_init(drain_bar(0), 1);
    mbar_init(drain_bar(1), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kWarpMma) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM column of A stage slot s, tile t (after the NT accumulators)
  auto a_col = [&](int slot, int t) {
    return static_cast<uint32_t>(2 * kBN + (slot * NT + t) * kACols);
  };

  const int ftiles = static_cast<int>((a.rows + kBM - 1) / kBM);  // last tile may be ragged
  const int kps = static_cast<int>(a.K / kBK) / a.nsplit;          // stages per item
  const int64_t nitems = static_cast<int64_t>(s_ts[a.E]) * ftiles * a.nsplit;

  if (warp == kWarpCodes) {
    // ------------------------------------------- TMA producer: weight codes
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int64_t gs = 0;  // global stage counter
      for (int64_t item = blockIdx.x; item < nitems && !*abort_flag; item += gridDim.x) {
        const Item it = decode_item(s_off, s_ts, a.E, item, ftiles, a.nsplit);
        for (int kb = it.ks * kps; kb < (it.ks + 1) * kps; ++kb, ++gs) {
          const int c = static_cast<int>(gs % kC);
          const uint32_t cu = static_cast<uint32_t>(gs / kC);
          if (!wait_ok(c_free(c), (cu & 1u) ^ 1u, a.status, abort_flag)) break;
          // the converting warps' reads of the slot (generic proxy) before
          // the copy's writes into it (async proxy)
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(c_full(c), NT * kCTile);
          tma_load_3d(sC + (c * NT + 0) * kCTile, &tm_codes0, kb * kBK, it.f * kBM, it.e, c_full(c),
                      pol);
          if (NT == 2)
            tma_load_3d(sC + (c * NT + 1) * kCTile, &tm_codes1, kb * kBK, it.f * kBM, it.e,
                        c_full(c), pol);
        }
      }
      // After an abort, wait (bounded) for the copies still landing.
      if (*abort_flag)
        for (int64_t j = (gs > kC ? gs - kC : 0); j < gs; ++j)
          mbar_wait_bounded(c_full(static_cast<int>(j % kC)),
                            static_cast<uint32_t>((j / kC) & 1), a.status);
    }
  } else if (warp == kWarpRows) {
    // -------------------------------------------- TMA producer: token rows
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      int64_t gs = 0;
      for (int64_t item = blockIdx.x; item < nitems && !*abort_flag; item += gridDim.x) {
        const Item it = decode_item(s_off, s_ts, a.E, item, ftiles, a.nsplit);
        const int npad = (it.ntok + 15) & ~15;
        const int box_rows = npad <= 16 ? 16 : npad <= 32 ? 32 : npad <= 64 ? 64 : kBN;
        const CUtensorMap *box = npad <= 16   ? &tm_x16
                                 : npad <= 32 ? &tm_x32
                                 : npad <= 64 ? &tm_x64
                                              : &tm_x128;
        for (int kb = it.ks * kps; kb < (it.ks + 1) * kps; ++kb, ++gs) {
          const int s = static_cast<int>(gs % kB);
          const uint32_t su = static_cast<uint32_t>(gs / kB);
          if (!wait_ok(ab_free(s), (su & 1u) ^ 1u, a.status, abort_flag)) break;
          // one box of 16, 32, 64 or 128 rows (a thread issues one TMA copy
          // per few hundred cycles); rows past the item's tokens are never
          // used, rows past the buffer are filled with zeros
          mbar_arrive_expect_tx(b_full(s), box_rows * kBK * 2);
          tma_load_2d(sB + s * kBTile, box, kb * kBK, it.t0, b_full(s), pol);
        }
      }
      if (*abort_flag)
        for (int64_t j = (gs > kB ? gs - kB : 0); j < gs; ++j)
          mbar_wait_bounded(b_full(static_cast<int>(j % kB)),
                            static_cast<uint32_t>((j / kB) & 1), a.status);
    }
  } else if (warp == kWarpRexp) {
    // ------------------------------------------------ row exponents
    // For every item in turn, the power of two r of each weight row (and
    // matrix) that puts the row's largest dequantised magnitude,
    // max over groups of s max(|zp|, |255 - zp|), into [2^14, 2^15), so that
    // every (q - zp) s 2^r is finite in fp16 and uses its full precision
    // whatever the weights' size.  Written to a two-slot ring one item ahead
    // of the dequant warpgroups (lane l takes rows l, l + 32, l + 64, l + 96).
    int64_t n = 0;
    for (int64_t item = blockIdx.x; item < nitems && !*abort_flag; item += gridDim.x, ++n) {
      const int slot = static_cast<int>(n & 1);
      const uint32_t use = static_cast<uint32_t>(n >> 1);
      if (!__all_sync(0xFFFFFFFFu, wait_ok(rexp_free(slot), (use & 1u) ^ 1u, a.status, abort_flag)))
        break;
      const Item it = decode_item(s_off, s_ts, a.E, item, ftiles, a.nsplit);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        for (int rr = lane; rr < kBM; rr += 32) {
          const int64_t wrow = static_cast<int64_t>(it.f) * kBM + rr;
          const float *sp = a.sc[t] + it.e * a.gstride[t] + wrow * a.G;
          const int32_t *zq = a.zp[t] + it.e * a.gstride[t] + wrow * a.G;
          float m = 0.0f;
          // the groups of this item's K range (each K split accumulates and
          // rescales its own partial sums); rows past the matrix (a ragged
          // last tile) read nothing
          const int g0 = ((it.ks * kps * kBK) >> a.group_shift) & ~3;
          const int g1 = wrow < a.rows ? min(a.G, ((((it.ks + 1) * kps * kBK) >> a.group_shift) + 3) & ~3) : g0;
          for (int g = g0; g < g1; g += 4) {
            const float4 s4 = __ldg(reinterpret_cast<const float4 *>(sp + g));
            const int4 z4 = __ldg(reinterpret_cast<const int4 *>(zq + g));
            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
            const int32_t zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              // max(|zp|, |255 - zp|) = |zp - 127.5| + 127.5
              const float zw = fabsf(static_cast<float>(zv[u]) - 127.5f) + 127.5f;
              m = fmaxf(m, sv[u] * zw);
            }
          }
          const int e = ((__float_as_int(m) >> 23) & 0xFF) - 127;
          s_rexp[(slot * NT + t) * kBM + rr] = max(-126, min(126, 14 - e));
        }
      }
      // the item's token column scales, which the epilogue applies
      for (int i = lane; i < it.ntok; i += 32) s_cs[slot * kBN + i] = __ldg(a.colscale + it.t0 + i);
      mbar_arrive(rexp_full(slot));
    }
  } else if (warp == kWarpMma || warp == kWarpMma + 1) {
    // ---------------------------------------------------- MMA issuers
    // Issuer t (one per weight matrix: gate and up, or down alone) issues
    // that matrix's MMAs of every stage, in stage order, into its own
    // accumulator (gate at column 0, up at kBN, down at 0; npad columns),
    // and commits once per stage: a stage's A and B slots are free when
    // every issuer's commit has arrived.  One thread issues back-to-back
    // MMAs about every 70 cycles and spends about as long again per stage on
    // its barrier waits, so the gate/up stage's eight MMAs go to two
    // threads (the down stage's four to one: splitting them by K step was
    // slower).  Each issuer walks every stage in order, so it sees every
    // phase of the rings' barriers in order.
    const int t = warp - kWarpMma;
    if (lane == 0 && t < NT) {
      int64_t gs = 0;
      uint32_t nitem_done = 0;
      const uint32_t d = tmem + kBN * static_cast<uint32_t>(t);
      for (int64_t item = blockIdx.x; item < nitems && !*abort_flag; item += gridDim.x) {
        const Item it = decode_item(s_off, s_ts, a.E, item, ftiles, a.nsplit);
        const int npad = (it.ntok + 15) & ~15;
        const uint32_t idesc = idesc_f16(npad);
        // the previous item's epilogue has drained the accumulators
        if (!wait_ok(acc_free, (nitem_done & 1u) ^ 1u, a.status, abort_flag)) break;
        tc_fence_after();
        bool ok = true;
        uint32_t acc = 0;  // the item's first MMA into the accumulator overwrites it
        for (int kb = 0; kb < kps; ++kb, ++gs) {
          const int sa = static_cast<int>(gs % kA), sb = static_cast<int>(gs % kB);
          const uint32_t ua = static_cast<uint32_t>(gs / kA), ub = static_cast<uint32_t>(gs / kB);
          if (!wait_ok(b_full(sb), ub & 1u, a.status, abort_flag) ||
              !wait_ok(a_full(sa), ua & 1u, a.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = smem_desc_sw128(sB + sb * kBTile);
          const uint32_t a0 = tmem + a_col(sa, t);
          // the descriptor's start address is in 16-byte units: +2 per 16 K
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            tc_mma_ts(d, a0 + kk * 8, bd + 2 * kk, idesc, acc);
            acc = 1u;
          }
          tc_commit(ab_free(sa));
        }
        if (!ok) break;
        tc_commit(acc_full);
        ++nitem_done;
      }
      // After an abort, wait (bounded) for this issuer's MMAs in flight.
      if (*abort_flag) {
        tc_commit(drain_bar(t));
        mbar_wait_bounded(drain_bar(t), 0u, a.status);
      }
    }
  } else {
    // ------------------------------------------ dequantisation + epilogue
    const int row = threadIdx.x & (kBM - 1);  // weight row of the tile (= TMEM lane)
    const int wg = warp >> 2;                  // converts stages kb = wg (mod kDequantGroups)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int64_t gs = 0;
    uint32_t nitem_done = 0;
    // Scale / zero point of this warpgroup's next stage, loaded one of its
    // stages ahead; those of an item's first stage are loaded before the
    // previous item's epilogue (a row past the matrix, in a ragged last
    // tile, dequantises to zero and reads no scales).
    float s_nx[NT];
    int32_t z_nx[NT];
    auto load_first = [&](int64_t nx_item, int64_t nx_gs) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        s_nx[t] = 0.0f;
        z_nx[t] = 0;
      }
      if (nx_item >= nitems) return;
      const Item nx = decode_item(s_off, s_ts, a.E, nx_item, ftiles, a.nsplit);
      const int64_t nx_row = static_cast<int64_t>(nx.f) * kBM + row;
      const int nx_kbs = nx.ks * kps;
      const int nx_kb0 = nx_kbs + static_cast<int>((wg - nx_gs % kDequantGroups + kDequantGroups) %
                                                   kDequantGroups);
      if (nx_kb0 < nx_kbs + kps && nx_row < a.rows) {
        const int64_t off = nx.e * a.gstride[0] + nx_row * a.G + ((nx_kb0 * kBK) >> a.group_shift);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          s_nx[t] = __ldg(a.sc[t] + off);
          z_nx[t] = __ldg(a.zp[t] + off);
        }
      }
    };
    load_first(blockIdx.x, 0);
    for (int64_t item = blockIdx.x; item < nitems && !*abort_flag; item += gridDim.x) {
      const Item it = decode_item(s_off, s_ts, a.E, item, ftiles, a.nsplit);
      const int64_t wrow = static_cast<int64_t>(it.f) * kBM + row;
      // element offset of this row's groups in matrix t's scale and
      // zero-point arrays (the matrices of one launch have the same shape)
      const int64_t goff = it.e * a.gstride[0] + wrow * a.G;
      // Row scale 2^r of each matrix (from the exponent warp) and its inverse,
      // which the epilogue applies; the slot (with the item's token column
      // scales) is released after the epilogue.
      const int rslot = static_cast<int>(nitem_done & 1u);
      float rup[NT], rdn[NT];
      {
        const uint32_t use = nitem_done >> 1;
        if (!__all_sync(0xFFFFFFFFu, wait_ok(rexp_full(rslot), use & 1u, a.status, abort_flag)))
          break;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int sh = s_rexp[(rslot * NT + t) * kBM + row];
          rup[t] = __int_as_float((127 + sh) << 23);
          rdn[t] = __int_as_float((127 - sh) << 23);
        }
      }
      // the item's stages [kbs, kbe); this warpgroup's first one (stages are
      // dealt by their global number gs)
      const int kbs = it.ks * kps, kbe = kbs + kps;
      const bool row_ok = wrow < a.rows;
      const int kb0 =
          kbs + static_cast<int>((wg - gs % kDequantGroups + kDequantGroups) % kDequantGroups);
      bool ok = true;
      // This warpgroup's stages of the item, directly (stage kb has global
      // number gs_item + kb - kbs).
      const int64_t gs_item = gs;
      gs += kps;
      for (int kb = kb0; kb < kbe; kb += kDequantGroups) {
        const int64_t g = gs_item + (kb - kbs);
        // Fast form (q - zp exact in fp16, times the fp16 scale) while the
        // zero point keeps 1024 + zp and every q - zp (|.| <= 2048) exact in
        // fp16 and the scaled scale is a normal fp16; the exact form otherwise.
        __half2 s2[NT], mz2[NT];
        float sx[NT];
        int32_t zx[NT];
        bool fast[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          sx[t] = s_nx[t] * rup[t];
          zx[t] = z_nx[t];
          fast[t] = zx[t] >= -1793 && zx[t] <= 1024 && sx[t] >= 6.103515625e-05f;
          s2[t] = __float2half2_rn(sx[t]);
          mz2[t] = __float2half2_rn(1024.0f + static_cast<float>(zx[t]));
        }
        if (kb + kDequantGroups < kbe && row_ok) {
          const int gi = ((kb + kDequantGroups) * kBK) >> a.group_shift;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            s_nx[t] = __ldg(a.sc[t] + goff + gi);
            z_nx[t] = __ldg(a.zp[t] + goff + gi);
          }
        }
        const int c = static_cast<int>(g % kC);
        const uint32_t cu = static_cast<uint32_t>(g / kC);
        const int s = static_cast<int>(g % kA);
        const uint32_t su = static_cast<uint32_t>(g / kA);
        if (!__all_sync(0xFFFFFFFFu, wait_ok(c_full(c), cu & 1u, a.status, abort_flag))) {
          ok = false;  // warp-uniform exit
          break;
        }
        // Every code chunk of the stage is read before any is converted, and
        // the fast / exact choice is made once per matrix and stage: with a
        // branch per chunk each read waited behind the previous chunk's
        // conversion.
        uint4 cv[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          // codes row `row`: 64 bytes, 16-byte chunk j stored at j ^ ((row >> 1) & 3)
          const uint32_t crow = sC + (c * NT + t) * kCTile + row * kBK;
#pragma unroll
          for (int j = 0; j < 4; ++j) cv[t][j] = lds128(crow + ((j ^ ((row >> 1) & 3)) << 4));
        }
        // The code slot is released as soon as its reads have returned (not
        // after the conversion), so that its refill from HBM overlaps this
        // warpgroup's conversion: the slots then spend their time loading.
        // A store of a value computed from every word read cannot issue
        // before all the reads have completed; the arrive follows it.
        {
          uint32_t dep = 0;
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) dep ^= cv[t][j].x ^ cv[t][j].y ^ cv[t][j].z ^ cv[t][j].w;
          sts_u32(sink, dep);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(c_free(c));
        if (!__all_sync(0xFFFFFFFFu, wait_ok(ab_free(s), (su & 1u) ^ 1u, a.status, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool all_fast = true;
#pragma unroll
        for (int t = 0; t < NT; ++t) all_fast = all_fast && fast[t];
        // A[row][k] -> TMEM lane row, column k / 2 of the stage slot.  The
        // branch is warp-uniform (the TMEM stores are warp-collective); a
        // warp with any row outside the fast form's range chooses per chunk.
        if (__all_sync(0xFFFFFFFFu, all_fast)) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            convert_row<false>(cv[t], mz2[t], s2[t], zx[t], sx[t], true,
                               tmem + lane_base + a_col(s, t));
        } else {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            convert_row<true>(cv[t], mz2[t], s2[t], zx[t], sx[t], fast[t],
                              tmem + lane_base + a_col(s, t));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(a_full(s));
      }
      if (!ok) break;
      load_first(item + gridDim.x, gs);  // gs: the next item's first stage
      // ---------------------------------------------------- epilogue
      if (!__all_sync(0xFFFFFFFFu, wait_ok(acc_full, nitem_done & 1u, a.status, abort_flag)))
        break;
      tc_fence_after();
      const int feat = it.f * kBM + row;
      // Accumulators (see the MMA issuers): gate at column 0 and up at kBN
      // (gate/up), or the down projection's at column 0.
      for (int c0 = 16 * wg; c0 < it.ntok; c0 += 16 * kDequantGroups) {
        float v0[16], v1[16];
        if constexpr (NT == 2)
          tmem_ld16x2(tmem + lane_base + c0, tmem + lane_base + kBN + c0, v0, v1);
        else
          tmem_ld16x1(tmem + lane_base + c0, v0);
        // accumulators x (token row's 2^c) x (weight row's 2^-r): exact
        // power-of-two rescaling back to the true products
        const float *cs = s_cs + rslot * kBN + c0;
        float *const outp = a.out + it.ks * a.out_split;
        const bool feat_ok = feat < a.rows;
        if constexpr (NT == 2) {
          // v0 = gate, v1 = up; h in fp32 (rounded to fp16 with its own row
          // scale once every feature tile of the token is done)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < it.ntok && feat_ok) {
              const float c = cs[j];
              outp[static_cast<int64_t>(it.t0 + c0 + j) * a.out_ld + feat] =
                  silu_f(v0[j] * c * rdn[0]) * (v1[j] * c * rdn[1]);
            }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < it.ntok && feat_ok)
              outp[static_cast<int64_t>(it.t0 + c0 + j) * a.out_ld + feat] =
                  v0[j] * cs[j] * rdn[0];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acc_free);
        mbar_arrive(rexp_free(rslot));
      }
      ++nitem_done;
    }
  }

  // Teardown (every role has drained what it issued), then free TMEM.
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Largest of the per-thread values v over a 256-thread block (every thread
// gets it).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v) {
  __shared__ uint32_t part[8];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  v = part[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) v = max(v, part[w]);
  return v;
}

// Gathers the tokens of every assignment in expert-sorted order into fp16
// rows (one block per sorted position p).  Each row is scaled by the power
// of two 2^s that puts its largest magnitude into [2^14, 2^15), so that
// bf16 -> fp16 is exact for every element within 2^28 of the row's largest
// and never overflows, whatever the tokens' size; xs[p] = 2^-s undoes it in
// the epilogue.  Only the first offsets[E] positions hold assignments
// (out-of-range expert indices are left out by the grouping).  Without an
// assignment list (a linear layer) position p is row p of x's nrows rows.
__global__ void __launch_bounds__(256) gather_x_kernel(const uint16_t *__restrict__ x, int k,
                                                       int64_t H, int E,
                                                       const int32_t *__restrict__ offsets,
                                                       const int32_t *__restrict__ assign,
                                                       int64_t nrows, __half *__restrict__ xg,
                                                       float *__restrict__ xs) {
  pdl_enter();
  const int64_t p = blockIdx.x;
  if (p >= (assign ? static_cast<int64_t>(offsets[E]) : nrows)) return;
  const int64_t tok = assign ? assign[p] / k : p;
  const uint4 *src = reinterpret_cast<const uint4 *>(x + tok * H);
  const int64_t H8 = H / 8;
  // magnitudes as bit patterns: non-negative floats order like integers
  uint32_t mb = 0;
  for (int64_t c = threadIdx.x; c < H8; c += blockDim.x) {
    const uint4 v = __ldg(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) mb = max(mb, max((w[i] << 16) & 0x7FFF0000u, w[i] & 0x7FFF0000u));
  }
  mb = block_max_u32(mb);
  float up, down;
  pow2_to_fp16_range(__uint_as_float(mb), up, down);
  if (threadIdx.x == 0) xs[p] = down;
  for (int64_t c = threadIdx.x; c < H8; c += blockDim.x) {
    const uint4 v = __ldg(src + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
      __half2 h = __floats2half2_rn(lo * up, hi * up);
      o[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    reinterpret_cast<uint4 *>(xg + p * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Rounds the tensor-core experts' fp32 SwiGLU rows to fp16 for the down GEMM
// (one block per sorted position p), each row scaled like the token rows
// above; hs[p] undoes the scaling.  Rows of experts without token tiles (the
// few-token experts, which run on the small-M kernels) are skipped.
__global__ void __launch_bounds__(256) h_convert_kernel(const float *__restrict__ h, int64_t I,
                                                        int E, const int32_t *__restrict__ offsets,
                                                        const int32_t *__restrict__ tile_start,
                                                        __half *__restrict__ hh,
                                                        float *__restrict__ hs) {
  pdl_enter();
  const int p = blockIdx.x;
  if (p >= offsets[E]) return;
  int lo = 0, hi = E;  // the expert of position p: offsets[lo] <= p < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= p) lo = mid;
    else hi = mid;
  }
  if (tile_start[lo + 1] == tile_start[lo]) return;
  const float4 *src = reinterpret_cast<const float4 *>(h + static_cast<int64_t>(p) * I);
  const int64_t I4 = I / 4;
  uint32_t mb = 0;
  for (int64_t c = threadIdx.x; c < I4; c += blockDim.x) {
    const float4 v = src[c];
    mb = max(mb, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                     max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
  }
  mb = block_max_u32(mb);
  float up, down;
  pow2_to_fp16_range(__uint_as_float(mb), up, down);
  if (threadIdx.x == 0) hs[p] = down;
  for (int64_t c = threadIdx.x; c < I4; c += blockDim.x) {
    const float4 v = src[c];
    __half2 a = __floats2half2_rn(v.x * up, v.y * up);
    __half2 b = __floats2half2_rn(v.z * up, v.w * up);
    reinterpret_cast<uint2 *>(hh + static_cast<int64_t>(p) * I)[c] =
        make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
  }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Codes of E stacked [rows, K] INT8 matrices as a 3-D map, box [64 B, 128
// rows, 1], 64-byte swizzle.
bool make_codes_map(CUtensorMap *m, const QMat &w, int E) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t rowbytes = static_cast<cuuint64_t>(w.cols);  // INT8
  cuuint64_t dims[3] = {rowbytes, static_cast<cuuint64_t>(w.rows), static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {rowbytes, static_cast<cuuint64_t>(w.codes_stride)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBM), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(w.codes), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp16 token rows [MK, K] as a 2-D map, box [64, box_rows], 128-byte swizzle.
// Maps of one fp16 row buffer with boxes of 16, 32, 64 and 128 rows.
struct RowMaps {
  CUtensorMap m[4];
};

bool make_rows_map(CUtensorMap *m, const __half *p, int64_t MK, int64_t K, int box_rows);

bool make_row_maps(RowMaps *r, const __half *p, int64_t MK, int64_t K) {
  return make_rows_map(&r->m[0], p, MK, K, 16) && make_rows_map(&r->m[1], p, MK, K, 32) &&
         make_rows_map(&r->m[2], p, MK, K, 64) && make_rows_map(&r->m[3], p, MK, K, kBN);
}

bool make_rows_map(CUtensorMap *m, const __half *p, int64_t MK, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(MK)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half *>(p), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT>
cudaError_t run_tc(const CUtensorMap &c0, const CUtensorMap &c1, const RowMaps &x,
                   const TcArgs &a, cudaStream_t s) {
  auto k = moe_tc_kernel<NT>;
  const int bytes = Smem<NT>::bytes_for(a.E);
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k), bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(sm_count()), dim3(kThreads), bytes, s, c0, c1, x.m[0], x.m[1],
                    x.m[2], x.m[3], a);
}

// y = the sum of the nsplit partial results of the split K range, added in
// split order (deterministic), written as fp32 or bf16.
template <bool YBF16>
__global__ void __launch_bounds__(256) split_reduce_kernel(const float *__restrict__ part,
                                                           int nsplit, int64_t n, void *y) {
  pdl_enter();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float acc = part[i];
  for (int sidx = 1; sidx < nsplit; ++sidx) acc += part[sidx * n + i];
  if constexpr (YBF16)
    static_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(acc);
  else
    static_cast<float *>(y)[i] = acc;
}

// K splits of a linear layer with M rows on the tensor cores: the smallest
// divisor of the number of 64-wide K stages that gives work items for about
// every SM (each item pays a pipeline fill and an epilogue, so one long item
// per CTA beats two short ones), with at least four stages per split.
int linear_tc_splits(int64_t M, int64_t N, int64_t K) {
  const int64_t items = ((M + kBN - 1) / kBN) * ((N + kBM - 1) / kBM);
  const int kst = static_cast<int>(K / kBK);
  const int64_t target = (4 * static_cast<int64_t>(sm_count())) / 5;
  for (int d = 1; d <= kst / 4; ++d)
    if (kst % d == 0 && items * d >= target) return d;
  int best = 1;
  for (int d = 1; d <= kst / 4; ++d)
    if (kst % d == 0) best = d;
  return best;
}

}  // namespace

bool linear_tc_supported(const QMat &w) {
  return w.bits == 8 && w.group >= 64 && w.cols % kBK == 0 && (w.cols / w.group) % 4 == 0 &&
         w.rows >= 1 && encode_fn() != nullptr;
}

size_t linear_tc_workspace_bytes(int64_t M, const QMat &w) {
  const int S = linear_tc_splits(M, w.rows, w.cols);
  auto r256 = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  return r256(2 * static_cast<size_t>(M) * w.cols) + r256(4 * static_cast<size_t>(M)) +
         r256(4 * static_cast<size_t>(S) * M * w.rows);
}

cudaError_t launch_linear_tc(const void *x, int64_t M, const QMat &w, void *y, bool y_bf16,
                             void *workspace, cudaStream_t s) {
  const int64_t N = w.rows, K = w.cols;
  const int S = linear_tc_splits(M, N, K);
  auto r256 = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  uint8_t *base = static_cast<uint8_t *>(workspace);
  __half *xg = reinterpret_cast<__half *>(base);
  float *xs = reinterpret_cast<float *>(base + r256(2 * static_cast<size_t>(M) * K));
  float *part = reinterpret_cast<float *>(base + r256(2 * static_cast<size_t>(M) * K) +
                                          r256(4 * static_cast<size_t>(M)));
  // 1) rows of x -> scaled fp16 rows
  cudaError_t e = launch_pdl(gather_x_kernel, dim3(static_cast<unsigned>(M)), dim3(256), 0, s,
                             static_cast<const uint16_t *>(x), 1, K, 1,
                             static_cast<const int32_t *>(nullptr),
                             static_cast<const int32_t *>(nullptr), M, xg, xs);
  if (e != cudaSuccess) return e;
  CUtensorMap mw;
  RowMaps mx;
  QMat w1 = w;
  w1.codes_stride = N * K;  // one matrix: any positive stride of whole 16-byte units
  if (!make_codes_map(&mw, w1, 1) || !make_row_maps(&mx, xg, M, K))
    return cudaErrorInvalidValue;
  // 2) the GEMM: partial sums of each K split (fp32 y directly when there is
  // one split)
  const bool direct = S == 1 && !y_bf16;
  TcArgs a{};
  a.E = 1;
  a.k = 1;
  a.rows = N;
  a.K = K;
  a.G = static_cast<int>(K / w.group);
  a.group_shift = 0;
  while ((1 << a.group_shift) < w.group) ++a.group_shift;
  a.sc[0] = w.scales;
  a.zp[0] = w.zps;
  a.gstride[0] = 0;
  a.sc[1] = nullptr;
  a.zp[1] = nullptr;
  a.gstride[1] = 0;
  a.colscale = xs;
  a.out = direct ? static_cast<float *>(y) : part;
  a.out_ld = N;
  a.status = device_status();
  a.lin_M = static_cast<int>(M);
  a.nsplit = S;
  a.out_split = M * N;
  e = run_tc<1>(mw, mw, mx, a, s);
  if (e != cudaSuccess || direct) return e;
  // 3) the splits added in order
  const int64_t n = M * N;
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  if (y_bf16)
    return launch_pdl(split_reduce_kernel<true>, dim3(blocks), dim3(256), 0, s,
                      static_cast<const float *>(part), S, n, y);
  return launch_pdl(split_reduce_kernel<false>, dim3(blocks), dim3(256), 0, s,
                    static_cast<const float *>(part), S, n, y);
}

// Timing of the two GEMM launches (off unless enabled): events of the
// device that was current when timing was switched on, recorded around the
// gate/up and the down launch of every tensor-core moe_ffn_forward.
namespace {
struct TcTiming {
  std::mutex mu;
  bool on = false;
  bool recorded = false;
  int dev = -1;
  cudaEvent_t ev[4] = {};
};
TcTiming &tc_timing() {
  static TcTiming t;
  return t;
}
// Records event i on s when timing is on for the current device.
cudaError_t tc_mark(int i, cudaStream_t s) {
  TcTiming &t = tc_timing();
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.on) return cudaSuccess;
  int d = -1;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess || d != t.dev) return e;
  e = cudaEventRecord(t.ev[i], s);
  if (e == cudaSuccess && i == 3) t.recorded = true;
  return e;
}
}  // namespace

cudaError_t tc_timing_enable(bool on) {
  TcTiming &t = tc_timing();
  std::lock_guard<std::mutex> lock(t.mu);
  if (on && t.ev[0] == nullptr) {
    cudaError_t e = cudaGetDevice(&t.dev);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = cudaEventCreate(&t.ev[i]);
    if (e != cudaSuccess) return e;
  }
  t.on = on;
  t.recorded = false;
  return cudaSuccess;
}

cudaError_t tc_timing_read(float *gateup_ms, float *down_ms, bool *have) {
  TcTiming &t = tc_timing();
  std::lock_guard<std::mutex> lock(t.mu);
  *have = t.recorded;
  if (!t.recorded) return cudaSuccess;
  cudaError_t e = cudaEventSynchronize(t.ev[3]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(gateup_ms, t.ev[0], t.ev[1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(down_ms, t.ev[2], t.ev[3]);
  return e;
}

bool moe_tc_supported(const QMat &gate, const QMat &up, const QMat &down, int64_t H, int64_t I) {
  // gate and up share one scale / zero-point offset per dequantising thread
  const bool same_layout = up.groups_stride == gate.groups_stride && up.group == gate.group &&
                           up.rows == gate.rows && up.cols == gate.cols;
  return gate.bits == 8 && up.bits == 8 && down.bits == 8 && gate.group >= 64 && same_layout &&
         H % kBM == 0 && I % kBM == 0 && H % kBK == 0 && I % kBK == 0 && encode_fn() != nullptr;
}

cudaError_t launch_moe_tc(const void *x, int64_t M, int k, int E, const QMat &gate, const QMat &up,
                          const QMat &down, const MoeWork &ws, cudaStream_t s) {
  const int64_t MK = M * k;
  const int64_t H = gate.cols, I = gate.rows;
  // 1) tokens -> scaled fp16 rows in expert order
  {
    cudaError_t e = launch_pdl(gather_x_kernel, dim3(static_cast<unsigned>(MK)), dim3(256), 0, s,
                               static_cast<const uint16_t *>(x), k, H, E,
                               static_cast<const int32_t *>(ws.offsets),
                               static_cast<const int32_t *>(ws.assign), MK, ws.xg, ws.xs);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mg, mu, md;
  RowMaps mx, mh;
  if (!make_codes_map(&mg, gate, E) || !make_codes_map(&mu, up, E) ||
      !make_codes_map(&md, down, E) || !make_row_maps(&mx, ws.xg, MK, H) ||
      !make_row_maps(&mh, ws.hh, MK, I))
    return cudaErrorInvalidValue;
  // 2) gate + up with SwiGLU -> fp32 h
  TcArgs a{};
  a.E = E;
  a.k = k;
  a.rows = I;
  a.K = H;
  a.G = static_cast<int>(H / gate.group);
  a.group_shift = 0;
  while ((1 << a.group_shift) < gate.group) ++a.group_shift;
  a.sc[0] = gate.scales;
  a.zp[0] = gate.zps;
  a.gstride[0] = gate.groups_stride;
  a.sc[1] = up.scales;
  a.zp[1] = up.zps;
  a.gstride[1] = up.groups_stride;
  a.offsets = ws.offsets;
  a.tile_start = ws.tile_start;
  a.colscale = ws.xs;
  a.out = ws.h;
  a.out_ld = I;
  a.status = device_status();
  a.lin_M = 0;
  a.nsplit = 1;
  a.out_split = 0;
  cudaError_t e = tc_mark(0, s);
  if (e == cudaSuccess) e = run_tc<2>(mg, mu, mx, a, s);
  if (e == cudaSuccess) e = tc_mark(1, s);
  if (e != cudaSuccess) return e;
  // 3) h -> scaled fp16 rows
  e = launch_pdl(h_convert_kernel, dim3(static_cast<unsigned>(MK)), dim3(256), 0, s,
                 static_cast<const float *>(ws.h), I, E, static_cast<const int32_t *>(ws.offsets),
                 static_cast<const int32_t *>(ws.tile_start), ws.hh, ws.hs);
  if (e != cudaSuccess) return e;
  // 4) down -> fp32 per-assignment outputs
  TcArgs d = a;
  d.rows = H;
  d.K = I;
  d.G = static_cast<int>(I / down.group);
  d.group_shift = 0;
  while ((1 << d.group_shift) < down.group) ++d.group_shift;
  d.sc[0] = down.scales;
  d.zp[0] = down.zps;
  d.gstride[0] = down.groups_stride;
  d.sc[1] = nullptr;
  d.zp[1] = nullptr;
  d.gstride[1] = 0;
  d.colscale = ws.hs;
  d.out = ws.out;
  d.out_ld = H;
  e = tc_mark(2, s);
  if (e == cudaSuccess) e = run_tc<1>(md, md, mh, d, s);
  if (e == cudaSuccess) e = tc_mark(3, s);
  return e;
}

}  // namespace qmm

