// qmm_device.cuh -- device-side helpers shared by the library's kernels:
// inline-PTX wrappers (mbarrier, 1-D bulk async copy, packed f32x2 math),
// bounded waits that report through the device status word, and the
// in-register dequantisation primitives.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace qmm {

// Status bits (mirrors the public QMM_DEV_* values).
constexpr uint32_t kDevWaitTimeout = 1u;
constexpr uint32_t kDevBadExpert = 2u;
constexpr uint32_t kDevExpertOverload = 4u;

// Upper bound of any single wait inside a kernel (ns of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------- programmatic dependent launch
//
// Every kernel of the library is launched with programmatic stream
// serialization: it may be scheduled while the preceding kernel on the
// stream is still running, waits here for that kernel's completion (and
// memory flush) before it touches anything a preceding kernel may write,
// and lets the next kernel be scheduled early in turn.  Without a
// preceding kernel (or launched without the attribute) both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// limit_ns (kWaitLimitNs unless a caller passes another), sets
// kDevWaitTimeout in *status and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint32_t *status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(status, kDevWaitTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------- bulk copies

// 1-D bulk copy global -> shared (this CTA), completion signalled on `bar` as
// transaction bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// L2 policy "evict first" for all of an access's lines: they become the
// preferred victims of their L2 set (for data read for the last time).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ int32_t lds_s32(uint32_t addr) {
  int32_t v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 ldg_f4(const float *p) {
  return __ldg(reinterpret_cast<const float4 *>(p));
}

// ------------------------------------------------------ packed f32x2 math

typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(f32x2 v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// d = a * b + c, each half rounded once.
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ------------------------------------------------ in-register dequantisation
//
// A code byte b placed under the exponent byte 0x4B forms the fp32 value
// 2^23 + b exactly.  Subtracting the per-group constant 2^23 + zp (exact for
// |zp| < 2^23) leaves (q - zp) exactly, so no int->float conversion is needed.

// 2^23 + zp as fp32.
__device__ __forceinline__ float zp_magic(int32_t zp) { return 8388608.0f + (float)zp; }

// Byte `B` of `u` as 2^23 + byte.
template <int B>
__device__ __forceinline__ float byte_as_magic(uint32_t u) {
  return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u | B));
}

// INT8: one 32-bit word of stored codes (q - 128, columns c..c+3) ->
// two packed pairs {q0-zp, q1-zp}, {q2-zp, q3-zp}.
__device__ __forceinline__ void deq8_word(uint32_t w, f32x2 mzp2, f32x2 &d01, f32x2 &d23) {
  const uint32_t u = w ^ 0x80808080u;  // q - 128 -> q in each byte
  d01 = sub2(pack2(byte_as_magic<0>(u), byte_as_magic<1>(u)), mzp2);
  d23 = sub2(pack2(byte_as_magic<2>(u), byte_as_magic<3>(u)), mzp2);
}

// INT4: one 32-bit word (columns c..c+7, low nibble first) -> four pairs
// {q(c+2j) - zp, q(c+2j+1) - zp}, j = 0..3.
__device__ __forceinline__ void deq4_word(uint32_t w, f32x2 mzp2, f32x2 d[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu;         // even columns
  const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // odd columns
  d[0] = sub2(pack2(byte_as_magic<0>(lo), byte_as_magic<0>(hi)), mzp2);
  d[1] = sub2(pack2(byte_as_magic<1>(lo), byte_as_magic<1>(hi)), mzp2);
  d[2] = sub2(pack2(byte_as_magic<2>(lo), byte_as_magic<2>(hi)), mzp2);
  d[3] = sub2(pack2(byte_as_magic<3>(lo), byte_as_magic<3>(hi)), mzp2);
}

// Activation loads (fp32 or bf16 source), 4 consecutive elements.
template <bool BF16>
__device__ __forceinline__ float4 load_x4(const void *base, int64_t idx) {
  if constexpr (BF16) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(
        reinterpret_cast<const uint16_t *>(base) + idx));
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                       __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  } else {
    return ldg_f4(reinterpret_cast<const float *>(base) + idx);
  }
}

// Output element i of a linear layer, fp32 or rounded to bf16 (nearest even).
__device__ __forceinline__ void store_y(void *y, int64_t i, float v, bool bf16) {
  if (bf16)
    static_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float *>(y)[i] = v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

}  // namespace qmm
