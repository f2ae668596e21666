// smallm_kernel.cuh -- the small-M fused dequantise-matmul kernel template
// (design notes in smallm.cuh), instantiated by smallm_one.cu (one
// activation row per pass: the decode experts), smallm_lo.cu (two rows per
// pass; both two CTAs per SM, balanced-digit integer arithmetic) and
// smallm_hi.cu (eight fp32 rows per pass, one CTA per SM; the linear layer
// with 3..8 rows and small INT4 matrices with one row).
#pragma once

#include <cstdint>

#include "smallm.cuh"

namespace qmm {
namespace smallm {
namespace {

typedef unsigned long long f32x2_t;

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// NW consecutive 32-bit words of shared memory (one lane's codes of a row).
template <int NW>
__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t (&w)[NW]) {
  if constexpr (NW == 8) {
    const uint4 v0 = lds128(addr), v1 = lds128(addr + 16);
    w[0] = v0.x;
    w[1] = v0.y;
    w[2] = v0.z;
    w[3] = v0.w;
    w[4] = v1.x;
    w[5] = v1.y;
    w[6] = v1.z;
    w[7] = v1.w;
  } else if constexpr (NW == 4) {
    const uint4 v = lds128(addr);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else if constexpr (NW == 2) {
    const uint2 v = lds64(addr);
    w[0] = v.x;
    w[1] = v.y;
  } else {
    static_assert(NW == 1, "1, 2, 4 or 8 words");
    w[0] = lds32(addr);
  }
}

// CTA barrier that also ORs a predicate over the threads, so that every
// thread takes the same decision after it.
__device__ __forceinline__ bool consumers_sync_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.or.pred b, 1, %2, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"(p ? 1u : 0u), "n"(kCW * 32)
      : "memory");
  return r != 0;
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

// A byte of u placed under the exponent byte 0x4B: the fp32 value 2^23 + byte.
template <int B>
__device__ __forceinline__ float mag(uint32_t u) {
  return __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u | B));
}

// Dot products of this lane's XPL codes of one row with TB activation rows.
//
// INT8: a stored byte is q - 128; xor 0x80 gives q, read as 2^23 + q.
// INT4: a byte holds column 2j (low nibble) and 2j + 1 (high nibble).  The
// masks 0x0F0F0F0F and 0xF0F0F0F0 leave q and 16 q in each byte, read as
// 2^23 + q and 2^23 + 16 q; one packed subtract of (2^23 + zp, 2^23 + 16 zp)
// gives (q - zp, 16 (q - zp)) exactly.  The odd columns' activations are
// held divided by 16 (a power-of-two scaling), so every product is the
// product of the pages' formula.
// xp[t][p] holds columns (2p, 2p + 1) of activation row t.
template <int BITS, int XPL, int TB, int TBMAX>
__device__ __forceinline__ void row_dot(uint32_t caddr, float zf,
                                        const f32x2_t (&xp)[TBMAX][XPL / 2], float (&d)[TB]) {
  f32x2_t acc[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) acc[t] = 0ull;
  if constexpr (BITS == 4) {
    constexpr int NW = XPL / 8;
    uint32_t w[NW];
    lds_words<NW>(caddr, w);
    const f32x2_t off = pack2(8388608.0f + zf, fmaf(16.0f, zf, 8388608.0f));
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = w[i] & 0xF0F0F0F0u;
      f32x2_t dq[4];
      dq[0] = sub2(pack2(mag<0>(lo), mag<0>(hi)), off);
      dq[1] = sub2(pack2(mag<1>(lo), mag<1>(hi)), off);
      dq[2] = sub2(pack2(mag<2>(lo), mag<2>(hi)), off);
      dq[3] = sub2(pack2(mag<3>(lo), mag<3>(hi)), off);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int t = 0; t < TB; ++t) acc[t] = fma2(dq[j], xp[t][4 * i + j], acc[t]);
    }
  } else {
    constexpr int NW = XPL / 4;
    uint32_t w[NW];
    lds_words<NW>(caddr, w);
    const float m = 8388608.0f + zf;
    const f32x2_t off = pack2(m, m);
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const uint32_t u = w[i] ^ 0x80808080u;
      const f32x2_t d01 = sub2(pack2(mag<0>(u), mag<1>(u)), off);
      const f32x2_t d23 = sub2(pack2(mag<2>(u), mag<3>(u)), off);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        acc[t] = fma2(d01, xp[t][2 * i], acc[t]);
        acc[t] = fma2(d23, xp[t][2 * i + 1], acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    float lo, hi;
    unpack2(acc[t], lo, hi);
    d[t] = lo + hi;
  }
}

// Butterfly reduce-scatter of C values over the lanes: at offset O a lane
// keeps one half of its values (the upper half if its bit O is set) and adds
// the partner's copy of that half; once one value is left the remaining
// offsets are plain sums.  With V values at the start (V <= 32, a power of
// two), lane l ends with the full sum of value l >> (5 - log2 V).
template <int C, int O>
__device__ __forceinline__ void bfly(float *v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (C > 1) {
      constexpr int H = C / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, O);
      }
      bfly<H, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], O);
      bfly<1, O / 2>(v, lane);
    }
  }
}

template <int V>
__host__ __device__ constexpr int log2c() {
  return V <= 1 ? 0 : 1 + log2c<V / 2>();
}

// One tile for TB tokens: the NRW rows row0 .. row0 + NRW - 1 of a stage of
// NR rows (the warp's row group) against the lane's slice of the
// activations; lane partials reduced per block of NRS rows and written to
// this warp's row of the reduction buffer (index row * TB + token).
template <int BITS, int XPL, int NR, int NRW, int TB, int TBMAX>
__device__ __forceinline__ void tile_compute(uint32_t stage, int rowbytes, int G, int gi,
                                             uint32_t lane_off, int row0,
                                             const f32x2_t (&xp)[TBMAX][XPL / 2],
                                             float *red_w, int lane) {
  constexpr int NRS = (NRW * TB <= 32) ? NRW : 32 / TB;
  constexpr int V = NRS * TB;
  constexpr int LV = log2c<V>();
  const uint32_t sc0 = stage + NR * rowbytes + 4 * gi;
  const uint32_t zp0 = sc0 + NR * G * 4;
#pragma unroll
  for (int sb = 0; sb < NRW; sb += NRS) {
    float v[V];
#pragma unroll
    for (int r = 0; r < NRS; ++r) {
      const int row = row0 + sb + r;
      const float s = lds_f32(sc0 + row * G * 4);
      const float zf = static_cast<float>(lds_s32(zp0 + row * G * 4));
      float d[TB];
      row_dot<BITS, XPL, TB, TBMAX>(stage + row * rowbytes + lane_off, zf, xp, d);
#pragma unroll
      for (int t = 0; t < TB; ++t) v[r * TB + t] = s * d[t];
    }
    bfly<V, 16>(v, lane);
    if ((lane & ((32 >> LV) - 1)) == 0) red_w[sb * TB + (lane >> (5 - LV))] = v[0];
  }
}

// This lane's activation slice of up to TBMAX rows: rows[t] for t < T,
// zeros after.  INT4 keeps odd columns divided by 16 (see row_dot).
// The XPL activations of this lane's slice of one row as fp32 (bf16 is
// widened exactly); zeros when `use` is false (a token slot past the pass).
template <bool XBF16, int XPL>
__device__ __forceinline__ void load_slice(const void *row, bool use, int col0, float (&v)[XPL]) {
  if (use) {
    if constexpr (XBF16) {
      const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(row) + col0);
#pragma unroll
      for (int c = 0; c < XPL / 8; ++c) {
        const uint4 u = __ldg(p + c);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          v[8 * c + 2 * h] = __uint_as_float(wv[h] << 16);
          v[8 * c + 2 * h + 1] = __uint_as_float(wv[h] & 0xFFFF0000u);
        }
      }
    } else {
      const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(row) + col0);
#pragma unroll
      for (int c = 0; c < XPL / 4; ++c) {
        const float4 f = __ldg(p + c);
        v[4 * c] = f.x;
        v[4 * c + 1] = f.y;
        v[4 * c + 2] = f.z;
        v[4 * c + 3] = f.w;
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < XPL; ++c) v[c] = 0.0f;
  }
}

template <int BITS, int XPL, bool XBF16, int TBMAX>
__device__ __forceinline__ void load_x(const void *const (&rows)[TBMAX], int T, int col0,
                                       f32x2_t (&xp)[TBMAX][XPL / 2]) {
  const float odd = BITS == 4 ? 0.0625f : 1.0f;
#pragma unroll
  for (int t = 0; t < TBMAX; ++t) {
    float v[XPL];
    load_slice<XBF16, XPL>(rows[t], t < T, col0, v);
#pragma unroll
    for (int p = 0; p < XPL / 2; ++p) xp[t][p] = pack2(v[2 * p], v[2 * p + 1] * odd);
  }
}

__device__ __forceinline__ int32_t dp4a_us(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ------------------------------------------- balanced-digit integer form
//
// Each activation of the lane's slice is held as one 38-bit integer,
// x = X 2^-F with F chosen so that the slice's largest |x| times 2^F lies in
// [2^37, 2^38): every activation within 2^14 of the slice's largest is exact
// (its fp32 ulp is a multiple of 2^-F) and every other one is within
// 2^-38 of the largest.  X is split into five balanced byte digits,
// X = sum_i L_i 2^8i with L_i in [-128, 127] (each digit is the residue of
// the remaining value in [-128, 128) and the next one takes the carry), so
// that a small |X| has small digits and the zero digits of a small value stay
// zero.  Per row, with the codes centred (INT8: the stored q - 128; INT4: the
// nibble q) and z' the zero point centred the same way,
//   c_i = sum_k (q_k - zp) L_i,k = sum_k q'_k L_i,k - z' sum_k L_i,k
// is an exact 32-bit integer (one signed byte dot product per four codes and
// digit, the zero point applied once per digit), and
//   sum_k (q_k - zp) x_k = 2^-F sum_i 256^i c_i
// is formed in fp32 from the most significant digit down (Horner's rule, one
// rounding per step).  Balanced digits keep every partial sum within twice
// sum_k |(q_k - zp) X_k|, so the rounding stays relative to the terms of
// the dot product itself however strongly its terms cancel.  A zero point
// beyond +-2^17 of the centre (single-signed groups far from zero) forms the
// c_i in 64 bits instead.

constexpr int kDigits = 5;
// A slice whose largest |x| exceeds this many times the mean |x| of the
// warp's columns makes the warp use all five digits.
constexpr float kWideRatio = 128.0f;

__device__ __forceinline__ int32_t dp4a_ss(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Shared-memory address of 16-byte unit u of low digit p (0 or 1) of row t
// in this warp's low-digit area: consecutive lanes hold consecutive units,
// so a warp's 16-byte accesses are free of bank conflicts.
template <int XPL, int TBMAX>
__device__ __forceinline__ uint32_t low_addr(uint32_t low, int t, int p, int u, int lane) {
  constexpr int NU = XPL / 16;  // 16-byte units per digit and row
  return low + static_cast<uint32_t>((((t * 2 + p) * NU + u) * 32 + lane) * 16);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Fills the digit planes of this lane's slice of up to TBMAX rows (zeros
// after T) and returns, the same in every lane of the warp, whether some
// lane's slice of some row is wide: its largest |x| more than kWideRatio
// times the mean |x| over the warp's columns of that row.  X is formed as
// X = 2^16 Xh + Xl with Xh = round(x 2^(F-16)) (22 bits) and Xl the rounded
// remainder (|Xl| <= 2^15), so all arithmetic stays in 32 bits; the two low
// digits (from Xl, with their carry into Xh) are formed only when the warp
// needs them.
template <int BITS, int XPL, bool XBF16, int TBMAX>
__device__ __forceinline__ bool load_x_digits(const void *const (&rows)[TBMAX], int T, int col0,
                                              uint32_t (&xl)[TBMAX][3][XPL / 4],
                                              uint32_t low, int lane,
                                              int32_t (&sl)[TBMAX][kDigits],
                                              float (&xsc)[TBMAX]) {
  // raw slice words: XPL fp32 values, or XPL / 2 words of two bf16 each
  // (expanded when used, which keeps fewer registers live)
  constexpr int RW = XBF16 ? XPL / 2 : XPL;
  auto val = [](const uint32_t (&raw)[RW], int c) {
    if constexpr (XBF16)
      return __uint_as_float((c & 1) ? (raw[c >> 1] & 0xFFFF0000u) : (raw[c >> 1] << 16));
    else
      return __uint_as_float(raw[c]);
  };
  // the lane's slice of row t (zeros for t >= T)
  auto load = [&](int t, uint32_t (&raw)[RW]) {
    if (t < T) {
      const uint4 *p = reinterpret_cast<const uint4 *>(
          static_cast<const uint8_t *>(rows[t]) + static_cast<int64_t>(col0) * (XBF16 ? 2 : 4));
#pragma unroll
      for (int c = 0; c < RW / 4; ++c) {
        const uint4 u = __ldg(p + c);
        raw[4 * c] = u.x;
        raw[4 * c + 1] = u.y;
        raw[4 * c + 2] = u.z;
        raw[4 * c + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < RW; ++c) raw[c] = 0u;
    }
  };
  float mxs[TBMAX];
  bool wide = false;
  uint32_t raw[TBMAX][RW];
#pragma unroll
  for (int t = 0; t < TBMAX; ++t) load(t, raw[t]);
#pragma unroll
  for (int t = 0; t < TBMAX; ++t) {
    float mx = 0.0f, sa = 0.0f;
#pragma unroll
    for (int c = 0; c < XPL; ++c) {
      mx = fmaxf(mx, fabsf(val(raw[t], c)));
      sa += fabsf(val(raw[t], c));
    }
    mxs[t] = mx;
    const float warp_sa = warp_sum(sa);  // sum of |x| over the warp's 32 XPL columns
    wide = wide || mx * static_cast<float>(32 * XPL) > kWideRatio * warp_sa;
    // an infinity reaches mx, a NaN the sum (fmaxf skips NaNs)
    xsc[t] = (mx <= 3.40282347e38f && sa == sa) ? 0.0f : __int_as_float(0x7FC00000);
  }
  wide = __any_sync(0xFFFFFFFFu, wide);
#pragma unroll
  for (int t = 0; t < TBMAX; ++t) {
    // F = 37 - floor(log2 mx) (exponent bits; power-of-two scalings exact)
    const float mx = mxs[t];
    const int e = mx > 0.0f ? ((__float_as_int(mx) >> 23) & 0xFF) - 127 : 0;
    const int F = max(-110, min(126, 37 - e));
    const float uph = __int_as_float((F - 16 + 127) << 23);  // 2^(F-16)
    // 2^-F; a NaN or infinite activation makes the slice's results NaN, as
    // they would be in fp32 arithmetic (its digits would be meaningless)
    xsc[t] = xsc[t] == 0.0f ? __int_as_float((127 - F) << 23) : xsc[t];
    int32_t sum[kDigits];
#pragma unroll
    for (int i = 0; i < kDigits; ++i) sum[i] = 0;
    // word w holds, for INT8, columns 4w .. 4w + 3; for INT4, word 2j the
    // even columns 8j, 8j + 2, 8j + 4, 8j + 6 and word 2j + 1 the odd ones
#pragma unroll
    // A balanced digit of v is the low byte of v read as a signed byte,
    // d = v - 256 ((v + 128) >> 8), and the rest (v + 128) >> 8 carries on;
    // the words hold the digits' low bytes (their two's complement).
    auto pack4 = [](const int32_t (&v)[4]) {
      return __byte_perm(__byte_perm(v[0], v[1], 0x0040), __byte_perm(v[2], v[3], 0x0040),
                         0x5410);
    };
    uint32_t lw[2][4];  // the low digits' words, four at a time to shared memory
#pragma unroll
    for (int w = 0; w < XPL / 4; ++w) {
      const int c0 = BITS == 4 ? 8 * (w >> 1) + (w & 1) : 4 * w;
      const int st = BITS == 4 ? 2 : 1;
      int32_t v2[4], v3[4], v4[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float xs = val(raw[t], c0 + st * b) * uph;  // exact
        int32_t xh = __float2int_rn(xs);                  // |xh| <= 2^22
        if (wide) {
          // remainder in units of 2^-F: |.| <= 2^15, exact in fp32
          const int32_t xl16 = __float2int_rn((xs - static_cast<float>(xh)) * 65536.0f);
          const int32_t c1 = (xl16 + 128) >> 8;   // in [-128, 128]
          const int32_t c2 = (c1 + 128) >> 8;     // carry into xh: 0 or +-1
          v2[b] = xl16;                            // digit 0 = low byte of xl16
          v3[b] = c1;                              // digit 1 = low byte of c1
          xh += c2;
        }
        v4[b] = xh;
      }
      if (wide) {
        lw[0][w & 3] = pack4(v2);
        lw[1][w & 3] = pack4(v3);
        // a digit sum is the byte dot product of its word with ones
        sum[0] = dp4a_ss(lw[0][w & 3], 0x01010101u, sum[0]);
        sum[1] = dp4a_ss(lw[1][w & 3], 0x01010101u, sum[1]);
        if ((w & 3) == 3) {
#pragma unroll
          for (int p = 0; p < 2; ++p)
            sts128(low_addr<XPL, TBMAX>(low, t, p, w >> 2, lane),
                   make_uint4(lw[p][0], lw[p][1], lw[p][2], lw[p][3]));
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int32_t xh = v4[b];
        const int32_t c3 = (xh + 128) >> 8;
        const int32_t c4 = (c3 + 128) >> 8;   // the top digit, |.| <= 65
        v2[b] = xh;
        v3[b] = c3;
        v4[b] = c4;
      }
      xl[t][0][w] = pack4(v2);
      xl[t][1][w] = pack4(v3);
      xl[t][2][w] = pack4(v4);
#pragma unroll
      for (int i = 0; i < 3; ++i) sum[i + 2] = dp4a_ss(xl[t][i][w], 0x01010101u, sum[i + 2]);
    }
#pragma unroll
    for (int i = 0; i < kDigits; ++i) sl[t][i] = sum[i];
  }
  return wide;
}

// Exact digit sums c_i = a_i - z' SL_i of one row and token, combined into
// sum_k (q_k - zp) X_k in fp32 from the top digit down (digits D0..4).
template <int D0>
__device__ __forceinline__ float combine_digits(const int32_t (&a)[kDigits], int32_t zc,
                                                const int32_t (&sl)[kDigits]) {
  // Bounds (XPL <= 32): |a_i| <= 32 * 255 * 128 < 2^21, |sum L_i| <= 2^12,
  // |sum (L_i + 256 L_i+1)| <= 2^20.  With |z'| <= 1024 the pairs
  // c_i + 256 c_i+1 = (a_i + 256 a_i+1) - z' (sum L_i + 256 sum L_i+1) are
  // exact in 32 bits (|.| < 2^31); otherwise every c_i is formed in 64 bits.
  if (zc >= -1024 && zc <= 1024) {
    // pairs of digits (2, 3) and (0, 1), then the top digit
    const int32_t c4 = a[4] - zc * sl[4];
    const int32_t c23 = (a[2] + 256 * a[3]) - zc * (sl[2] + 256 * sl[3]);
    float f = fmaf(static_cast<float>(c4), 65536.0f, static_cast<float>(c23));
    if constexpr (D0 == 0) {
      const int32_t c01 = (a[0] + 256 * a[1]) - zc * (sl[0] + 256 * sl[1]);
      f = fmaf(f, 65536.0f, static_cast<float>(c01));
    }
    return f;
  }
  float cf[kDigits];
#pragma unroll
  for (int i = D0; i < kDigits; ++i)
    cf[i] = __ll2float_rn(static_cast<int64_t>(a[i]) - static_cast<int64_t>(zc) * sl[i]);
  float f = cf[kDigits - 1];
#pragma unroll
  for (int i = kDigits - 2; i >= D0; --i) f = fmaf(f, 256.0f, cf[i]);
  return f;
}

// Balanced-digit dot products of this lane's XPL codes of one row with TB
// rows, returned as sum_k (q_k - zp) x_k.  The three top digits (held in
// registers) serve every row; a wide warp adds the two low digits (from
// shared memory), one row at a time.
template <bool WIDE, int BITS, int XPL, int TB, int TBMAX>
__device__ __forceinline__ void row_dot_digits(uint32_t caddr, int32_t zp,
                                               const uint32_t (&xl)[TBMAX][3][XPL / 4],
                                               uint32_t low, int lane,
                                               const int32_t (&sl)[TBMAX][kDigits],
                                               const float (&xsc)[TBMAX], float (&d)[TB]) {
  static_assert(XPL <= 32, "digit sums must fit in 32 bits");
  constexpr int NW = XPL * BITS / 32;  // code words per lane per row
  uint32_t w[NW];
  lds_words<NW>(caddr, w);
  const int32_t zc = BITS == 8 ? zp - 128 : zp;
  // one code word against one digit word (INT4: the word's low nibbles
  // against the even columns' digits, its high nibbles against the odd ones)
  auto dot = [&](int j, const uint32_t *dw, int32_t acc) {
    if constexpr (BITS == 4) {
      const uint32_t lo = w[j] & 0x0F0F0F0Fu, hi = (w[j] >> 4) & 0x0F0F0F0Fu;
      return dp4a_us(hi, dw[2 * j + 1], dp4a_us(lo, dw[2 * j], acc));
    } else {
      return dp4a_ss(w[j], dw[j], acc);  // the stored bytes are the centred codes q - 128
    }
  };
  if constexpr (!WIDE) {
    int32_t a[TB][kDigits];
#pragma unroll
    for (int t = 0; t < TB; ++t)
#pragma unroll
      for (int i = 0; i < kDigits; ++i) a[t][i] = 0;
#pragma unroll
    for (int j = 0; j < NW; ++j)
#pragma unroll
      for (int t = 0; t < TB; ++t)
#pragma unroll
        for (int i = 0; i < 3; ++i) a[t][i + 2] = dot(j, xl[t][i], a[t][i + 2]);
#pragma unroll
    for (int t = 0; t < TB; ++t)
      // the top three digits are X rounded to a multiple of 2^16 (balanced
      // digits: the dropped |L1 2^8 + L0| is at most 2^15 + 2^7)
      d[t] = combine_digits<2>(a[t], zc, sl[t]) * (xsc[t] * 65536.0f);
  } else {
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      int32_t a[kDigits] = {0, 0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < NW; ++j)
#pragma unroll
        for (int i = 0; i < 3; ++i) a[i + 2] = dot(j, xl[t][i], a[i + 2]);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t lw[XPL / 4];
#pragma unroll
        for (int u = 0; u < XPL / 16; ++u) {
          const uint4 v = lds128(low_addr<XPL, TBMAX>(low, t, p, u, lane));
          lw[4 * u] = v.x;
          lw[4 * u + 1] = v.y;
          lw[4 * u + 2] = v.z;
          lw[4 * u + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < NW; ++j) a[p] = dot(j, lw, a[p]);
      }
      d[t] = combine_digits<0>(a, zc, sl[t]) * xsc[t];
    }
  }
}

template <bool WIDE, int BITS, int XPL, int NR, int NRW, int TB, int TBMAX>
__device__ __forceinline__ void tile_compute_digits(uint32_t stage, int rowbytes, int G, int gi,
                                                    uint32_t lane_off, int row0,
                                                    const uint32_t (&xl)[TBMAX][3][XPL / 4],
                                                    uint32_t low,
                                                    const int32_t (&sl)[TBMAX][kDigits],
                                                    const float (&xsc)[TBMAX], float *red_w,
                                                    int lane) {
  if constexpr (WIDE) {
    // All five digits (rare): one row per iteration and a plain warp sum per
    // row and token, which keeps this path's code small next to the
    // unrolled common path.
    const uint32_t sc0 = stage + NR * rowbytes + 4 * gi;
    const uint32_t zp0 = sc0 + NR * G * 4;
#pragma unroll 1
    for (int r = 0; r < NRW; ++r) {
      const int row = row0 + r;
      const float s = lds_f32(sc0 + row * G * 4);
      const int32_t zp = lds_s32(zp0 + row * G * 4);
      float d[TB];
      row_dot_digits<true, BITS, XPL, TB, TBMAX>(stage + row * rowbytes + lane_off, zp, xl, low,
                                                 lane, sl, xsc, d);
#pragma unroll
      for (int t = 0; t < TB; ++t) {
        const float v = warp_sum(s * d[t]);
        if (lane == 0) red_w[r * TB + t] = v;
      }
    }
    return;
  }
  // at most 16 row x token values per butterfly (fewer live registers)
  constexpr int NRS = (NRW * TB <= 16) ? NRW : 16 / TB;
  constexpr int V = NRS * TB;
  constexpr int LV = log2c<V>();
  const uint32_t sc0 = stage + NR * rowbytes + 4 * gi;
  const uint32_t zp0 = sc0 + NR * G * 4;
#pragma unroll
  for (int sb = 0; sb < NRW; sb += NRS) {
    float v[V];
#pragma unroll
    for (int r = 0; r < NRS; ++r) {
      const int row = row0 + sb + r;
      const float s = lds_f32(sc0 + row * G * 4);
      const int32_t zp = lds_s32(zp0 + row * G * 4);
      float d[TB];
      row_dot_digits<WIDE, BITS, XPL, TB, TBMAX>(stage + row * rowbytes + lane_off, zp, xl, low,
                                                 lane, sl, xsc, d);
#pragma unroll
      for (int t = 0; t < TB; ++t) v[r * TB + t] = s * d[t];
    }
    bfly<V, 16>(v, lane);
    if ((lane & ((32 >> LV) - 1)) == 0) red_w[sb * TB + (lane >> (5 - LV))] = v[0];
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ int64_t ceil_div(int64_t n, int64_t d) {
  return n <= 0 ? -((-n) / d) : (n + d - 1) / d;
}

}  // namespace
}  // namespace smallm
}  // namespace qmm


namespace qmm {
namespace smallm {
namespace {

// Segment s of the work: expert s_active[s], whose tokens sit at sorted
// positions s_off[e] .. s_off[e + 1] (the linear layer: one segment of M
// rows).  s_cs[s] = sum of the per-tile cost of the earlier segments.
// Tile j of a segment covers rows [j * RT, j * RT + RT) of each matrix.
// A segment with more than TBMAX tokens is applied in passes of TBMAX
// tokens; each pass sweeps the CTA's tiles of the segment (the tiles are
// streamed again, the pass's activations load once).  The work sequence is
// (segment, pass, tile).
struct TileIt {
  int s, b, nb;  // segment, pass, passes of the segment
  int64_t j, jlo, jhi;
  bool valid;
};

// KW warps split the K range of a row (K = 32 KW XPL); the kCW / KW row
// groups of a CTA take disjoint rows of every stage (KW = 4: two groups).
// The body of smallm_kernel, also run as two phases of the one-launch decode
// layer (moe_decode.cu).  `a` is read in place (a kernel parameter: a copy
// would live in local memory); idx replaces a.idx (the decode layer passes
// its top-k in shared memory).  before_act() is called by every thread once
// the first weight tiles have been requested and before anything a
// preceding step writes is read (the down projection and the linear layer;
// gate/up waits at its start); it returns false to abandon the work (every
// thread gets the same answer), after which the kernel only drains its
// copies.
template <int BITS, int XPL, int KW, int MODE, bool XBF16, int TBMAX, class BeforeAct>
__device__ __forceinline__ void smallm_body(const Args &a, const int32_t *idx,
                                            BeforeAct before_act) {
  // Gate/up needs the routing of the immediately preceding kernel (the
  // dispatch) before anything else.  The linear layer and the down
  // projection first request their leading weight tiles (see gemv_kernel)
  // and wait just before loading activations: the down projection's
  // grouping comes from the dispatch two launches back, which has completed
  // by the time it starts (the gate/up kernel between them starts dependents
  // only after its own wait), and only its activations (h) come from the
  // gate/up kernel.
  if constexpr (MODE == kGateUp) pdl_enter();
  static_assert(KW == kCW || (KW < kCW && TBMAX <= 2), "row groups: one or two rows per pass");
  using C = Cfg<TBMAX>;
  constexpr int STAGES = C::kStages, RED = C::kRedMax;
  constexpr int NR = rows_per_tile<BITS, XPL * KW / kCW>();
  constexpr int RG = kCW / KW;   // row groups
  constexpr int NRG = NR / RG;   // rows of a stage per row group
  constexpr int RT = (MODE == kGateUp) ? NR / 2 : NR;  // rows per matrix per tile
  constexpr int NM = (MODE == kGateUp) ? 2 : 1;
  constexpr int LB = XPL * BITS / 8;                   // code bytes per lane per row
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ int abort_s, nseg_s;
  volatile int *abort_flag = &abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *red = reinterpret_cast<float *>(smem + C::kRingBytes);
  int32_t *s_active =
      reinterpret_cast<int32_t *>(smem + C::kRingBytes + C::kRedBytes + C::kLowBytes);
  int32_t *s_off = s_active + a.E;
  int32_t *s_cs = s_off + a.E + 1;
  int32_t *s_idx = s_cs + a.E + 1;   // in-CTA grouping: expert of each assignment
  int32_t *s_asg = s_idx + a.MK;     //   sorted position -> assignment
  int32_t *s_cnt = s_asg + a.MK;     //   tokens per expert
  __shared__ int32_t scan_w[kCW][2];
  const uint32_t ring = smem_addr(smem);

  // Segments: the experts with tokens, in expert order (the linear layer:
  // one segment of M rows).
  if constexpr (MODE == kLinear) {
    if (threadIdx.x == 0) {
      s_active[0] = 0;
      s_off[0] = 0;
      s_off[1] = static_cast<int32_t>(a.M);
      nseg_s = 1;
    }
  } else if (idx) {
    // Decode batch: group the assignments by expert here (a stable counting
    // sort, the dispatch kernel's order: expert, then assignment).
    const int MK = static_cast<int>(a.MK), E = a.E;
    for (int t = threadIdx.x; t < MK; t += blockDim.x) {
      const int e = idx[t];
      const bool valid = e >= 0 && e < E;
      s_idx[t] = valid ? e : -1;
      if (!valid && MODE == kGateUp && blockIdx.x == 0) atomicOr(a.status, kDevBadExpert);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < MK; t += blockDim.x)
      if (s_idx[t] >= 0) atomicAdd(&s_cnt[s_idx[t]], 1);
    __syncthreads();
    {
      // exclusive scans of the counts and of the "has tokens" flags: four
      // consecutive experts per thread (E <= 1024), then warp and block scans
      constexpr int PER = 1024 / kThreads;
      const int e0 = PER * threadIdx.x;
      int c[PER], f[PER], sc = 0, sf = 0;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        c[u] = e0 + u < E ? s_cnt[e0 + u] : 0;
        f[u] = c[u] > 0 ? 1 : 0;
        sc += c[u];
        sf += f[u];
      }
      int ic = sc, jf = sf;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const int yf = __shfl_up_sync(0xFFFFFFFFu, jf, o);
        if (lane >= o) {
          ic += yc;
          jf += yf;
        }
      }
      if (lane == 31) {
        scan_w[warp][0] = ic;
        scan_w[warp][1] = jf;
      }
      __syncthreads();
      int bc = 0, bf = 0;
      for (int w = 0; w < warp; ++w) {
        bc += scan_w[w][0];
        bf += scan_w[w][1];
      }
      int xc = bc + ic - sc, xf = bf + jf - sf;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        if (e0 + u < E) {
          s_off[e0 + u] = xc;
          if (f[u]) s_active[xf] = e0 + u;
        }
        xc += c[u];
        xf += f[u];
      }
      if (threadIdx.x == kThreads - 1) {
        s_off[E] = xc;
        nseg_s = xf;
      }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < MK; t += blockDim.x) {
      const int e = s_idx[t];
      int p = -1;
      if (e >= 0) {
        int r = 0;
        for (int u = 0; u < t; ++u) r += s_idx[u] == e ? 1 : 0;
        p = s_off[e] + r;
        s_asg[p] = t;
      }
      if (a.pos_out && blockIdx.x == 0) a.pos_out[t] = p;
    }
  } else {
    const int n = *a.ws.num_active;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_active[i] = a.ws.active[i];
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_off[i] = a.ws.offsets[i];
    if (threadIdx.x == 0) nseg_s = n;
  }
  if (threadIdx.x == 0) {
    abort_s = 0;
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (warp == 0) {
    // Per-tile cost prefix over the segments: a run of segments per lane,
    // then a warp scan of the run totals.
    const int nseg = *static_cast<volatile int *>(&nseg_s);
    const int per = (nseg + 31) / 32;
    const int lo = min(nseg, lane * per), hi = min(nseg, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) {
      const int e = s_active[i];
      sum += tile_cost(s_off[e + 1] - s_off[e], TBMAX);
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - sum;
    for (int i = lo; i < hi; ++i) {
      s_cs[i] = run;
      const int e = s_active[i];
      run += tile_cost(s_off[e + 1] - s_off[e], TBMAX);
    }
    if (lane == 31) s_cs[nseg] = incl;
  }
  __syncthreads();
  const int na = nseg_s;

  // This CTA's tiles: those whose start cost c satisfies
  // blockIdx.x * total <= c * gridDim.x < (blockIdx.x + 1) * total.
  const int64_t Gd = gridDim.x;
  const int64_t tiles = a.tiles;
  const int64_t total = tiles * s_cs[na];
  const int64_t lo_c = static_cast<int64_t>(blockIdx.x) * total;
  const int64_t hi_c = lo_c + total;
  int s_first;
  {
    int l = 0, h = na;  // smallest s whose cost range ends beyond lo_c
    while (l < h) {
      const int m = (l + h) >> 1;
      if (tiles * s_cs[m + 1] * Gd > lo_c) h = m;
      else l = m + 1;
    }
    s_first = l;
  }
  // Tile range [jlo, jhi) of segment s; false once the segment starts at or
  // beyond the end of this CTA's range.
  auto seg_range = [&](int s, int64_t &jlo, int64_t &jhi) -> bool {
    if (s >= na) return false;
    const int64_t base = tiles * s_cs[s] * Gd;
    if (base >= hi_c) return false;
    const int e = s_active[s];
    const int64_t c = tile_cost(s_off[e + 1] - s_off[e], TBMAX) * Gd;
    jlo = ceil_div(lo_c - base, c);
    jhi = ceil_div(hi_c - base, c);
    jlo = jlo < 0 ? 0 : (jlo > tiles ? tiles : jlo);
    jhi = jhi < 0 ? 0 : (jhi > tiles ? tiles : jhi);
    return true;
  };
  auto passes = [&](int s) {
    const int e = s_active[s];
    return (s_off[e + 1] - s_off[e] + TBMAX - 1) / TBMAX;
  };
  auto it_settle = [&](TileIt &it) {  // move to the next (segment, pass) with a tile left
    while (it.j >= it.jhi) {
      if (++it.b < it.nb) {
        it.j = it.jlo;
        continue;
      }
      ++it.s;
      it.b = 0;
      if (!seg_range(it.s, it.jlo, it.jhi)) {
        it.valid = false;
        return;
      }
      it.nb = passes(it.s);
      it.j = it.jlo;
    }
  };
  auto it_begin = [&]() {
    TileIt it{s_first, 0, 0, 0, 0, 0, true};
    if (!seg_range(it.s, it.jlo, it.jhi)) {
      it.valid = false;
      return it;
    }
    it.nb = passes(it.s);
    it.j = it.jlo;
    it_settle(it);
    return it;
  };
  auto it_next = [&](TileIt &it) {
    ++it.j;
    it_settle(it);
  };
  const int64_t rows = a.rows;
  const int rowbytes = a.rowbytes, G = a.G;

  // Thread 0 streams the tiles: codes, scales and zero points of RT rows of
  // each matrix, three bulk copies per matrix completing on the stage's
  // barrier.  Experts: a tile that a later pass of its segment reads again
  // (an expert with more tokens than one pass takes) keeps the normal L2
  // priority; every other read is the tile's last and goes in as "evict
  // first", so the tiles still to be re-read stay in L2 while the rest of
  // the weights stream past them.
  auto issue = [&](const TileIt &it, int st) {
    const int e = s_active[it.s];
    const int64_t n0 = it.j * RT;
    const int rv = static_cast<int>(min64(RT, rows - n0));
    const uint32_t fb = smem_addr(&full_bar[st]);
    const uint32_t stage = ring + st * kStageBytes;
    const bool hint = MODE != kLinear && it.b + 1 >= it.nb;
    const uint64_t pol = hint ? l2_evict_first_policy() : 0ull;
    auto copy = [&](uint32_t dst, const void *src, int bytes) {
      if (hint)
        bulk_g2s_hint(dst, src, static_cast<uint32_t>(bytes), fb, pol);
      else
        bulk_g2s(dst, src, static_cast<uint32_t>(bytes), fb);
    };
    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(NM * rv * (rowbytes + 8 * G)));
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const QMat &W = m == 0 ? a.w0 : a.w1;
      const int r0 = m * RT;
      copy(stage + r0 * rowbytes, W.codes + e * W.codes_stride + n0 * rowbytes, rv * rowbytes);
      copy(stage + NR * rowbytes + r0 * G * 4, W.scales + e * W.groups_stride + n0 * G, rv * G * 4);
      copy(stage + NR * rowbytes + NR * G * 4 + r0 * G * 4, W.zps + e * W.groups_stride + n0 * G,
           rv * G * 4);
    }
  };
  // Every thread tracks the producer's position (it is cheap and keeps the
  // issuing role free to rotate over the warps); thread 0 fills the ring.
  TileIt pit = it_begin();
  int64_t issued = 0;
  for (int st = 0; st < STAGES && pit.valid; ++st) {
    if (threadIdx.x == 0) issue(pit, st);
    it_next(pit);
    ++issued;
  }
  if constexpr (MODE != kGateUp) {
    if (!before_act() && threadIdx.x == 0) abort_s = 1;  // read after the next barrier
  }

  const int kslot = (warp % KW) * 32 + lane;  // this lane's slice of K
  const int col0 = kslot * XPL;               // its columns
  const int gi = col0 / a.group;
  const uint32_t lane_off = static_cast<uint32_t>(kslot * LB);
  const int row0 = (warp / KW) * NRG;         // first stage row of this warp's group
  // Activation slices: the balanced digits (one or two rows per pass) or
  // fp32 pairs (eight rows per pass).
  constexpr bool kD = TBMAX <= 2;
  f32x2_t xp[kD ? 1 : TBMAX][XPL / 2];
  uint32_t xl[kD ? TBMAX : 1][3][XPL / 4];  // the three top digits
  // this warp's area for the two low digits
  const uint32_t low = ring + C::kRingBytes + C::kRedBytes + warp * (C::kLowBytes / kCW);
  float xsc[kD ? TBMAX : 1];
  int32_t sld[kD ? TBMAX : 1][kDigits];
  bool wide = false;  // digit form: this warp's slices need all five digits
  int cur_s = -1, cur_b = -1;
  // The activations of pass b of segment s, in this lane's slice (every lane
  // of the CTA takes part: the digit form reduces over the warp).
  auto load_act = [&](int s, int b) {
    const int e = s_active[s];
    const int p0 = s_off[e];
    const int t0 = b * TBMAX;
    const int Tb = min(TBMAX, s_off[e + 1] - p0 - t0);
    const void *xr[TBMAX];
#pragma unroll
    for (int t = 0; t < TBMAX; ++t) {
      const int64_t tt = t0 + (t < Tb ? t : 0);
      if constexpr (MODE == kLinear) {
        xr[t] = XBF16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.x) + tt * a.K)
                      : static_cast<const void *>(static_cast<const float *>(a.x) + tt * a.K);
      } else if constexpr (MODE == kGateUp) {
        const int64_t tok = (idx ? s_asg[p0 + tt] : a.ws.assign[p0 + tt]) / a.k;
        xr[t] = XBF16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.x) + tok * a.K)
                      : static_cast<const void *>(static_cast<const float *>(a.x) + tok * a.K);
      } else {
        xr[t] = a.ws.h + (p0 + tt) * a.K;
      }
    }
    if constexpr (kD)
      wide = load_x_digits<BITS, XPL, (MODE != kDown) && XBF16, TBMAX>(xr, Tb, col0, xl, low, lane,
                                                                        sld, xsc);
    else
      load_x<BITS, XPL, (MODE != kDown) && XBF16, TBMAX>(xr, Tb, col0, xp);
    cur_s = s;
    cur_b = b;
  };
  int64_t i = 0, pending = 0;
  bool stop = false;
  for (TileIt it = it_begin(); it.valid && !stop; it_next(it), ++i) {
    pending = i;
    const int s = it.s, b = it.b;
    const int e = s_active[s];
    const int p0 = s_off[e];
    const int T = s_off[e + 1] - p0;
    const int st = static_cast<int>(i % STAGES);
    // A new (segment, pass) reads its activations before the stage is waited
    // for, so that their latency overlaps the stage's copy.
    if (s != cur_s || b != cur_b) load_act(s, b);
    // warp-uniform, so that every lane takes part in the warp's shuffles
    const bool ok = __all_sync(0xFFFFFFFFu,
                               wait_ok(smem_addr(&full_bar[st]),
                                       static_cast<uint32_t>((i / STAGES) & 1), a.status,
                                       abort_flag));
    const uint32_t stage = ring + st * kStageBytes;
    const int64_t n0 = it.j * RT;
    const int t0 = b * TBMAX;
    const int Tb = min(TBMAX, T - t0);
    const int TB = Tb <= 1 ? 1 : Tb <= 2 ? 2 : Tb <= 4 ? 4 : 8;
    float *red_w = red + (i & 1) * kCW * RED + warp * RED;
    if (ok) {
      if constexpr (kD) {
        if (TBMAX == 1 || TB == 1) {
          if (wide)
            tile_compute_digits<true, BITS, XPL, NR, NRG, 1, TBMAX>(stage, rowbytes, G, gi, lane_off,
                                                                    row0, xl, low, sld, xsc, red_w,
                                                                    lane);
          else
            tile_compute_digits<false, BITS, XPL, NR, NRG, 1, TBMAX>(stage, rowbytes, G, gi,
                                                                     lane_off, row0, xl, low, sld,
                                                                     xsc, red_w, lane);
        } else {
          if constexpr (TBMAX >= 2) {
            if (wide)
              tile_compute_digits<true, BITS, XPL, NR, NRG, 2, TBMAX>(stage, rowbytes, G, gi,
                                                                      lane_off, row0, xl, low, sld,
                                                                      xsc, red_w, lane);
            else
              tile_compute_digits<false, BITS, XPL, NR, NRG, 2, TBMAX>(stage, rowbytes, G, gi,
                                                                       lane_off, row0, xl, low,
                                                                       sld, xsc, red_w, lane);
          }
        }
      } else if (TBMAX == 1 || TB == 1) {
        tile_compute<BITS, XPL, NR, NRG, 1, TBMAX>(stage, rowbytes, G, gi, lane_off, row0, xp, red_w,
                                                   lane);
      } else {
        if constexpr (TBMAX >= 2) {
          if (TB == 2)
            tile_compute<BITS, XPL, NR, NRG, 2, TBMAX>(stage, rowbytes, G, gi, lane_off, row0, xp,
                                                       red_w, lane);
        }
        if constexpr (TBMAX >= 8) {
          if (TB == 4)
            tile_compute<BITS, XPL, NR, NRG, 4, TBMAX>(stage, rowbytes, G, gi, lane_off, row0, xp,
                                                       red_w, lane);
          else if (TB == 8)
            tile_compute<BITS, XPL, NR, NRG, 8, TBMAX>(stage, rowbytes, G, gi, lane_off, row0, xp,
                                                       red_w, lane);
        }
      }
    }
    // Every warp has written its partials and finished reading the stage;
    // the OR tells all threads whether any gave up.
    if (consumers_sync_or(!ok || *abort_flag != 0)) {
      stop = true;
      break;
    }
    if (pit.valid) {
      // The stage is free: lane 0 of warp i % 8 refills it with the work
      // item STAGES ahead (the role rotates so that no warp is always late).
      if (lane == 0 && warp == static_cast<int>(i % kCW)) {
        fence_proxy_async_smem();
        issue(pit, st);
      }
      it_next(pit);
      ++issued;
    }
    // Finalise: thread q sums the KW warp partials of one (row, token)
    // output in warp order (the warps of the row's group); q = 0 starts at
    // warp (i + 1) % 8, so the usually short list of outputs also rotates
    // over the warps.
    const float *rb = red + (i & 1) * kCW * RED;
    const int q = (threadIdx.x + kThreads - 32 * static_cast<int>((i + 1) % kCW)) % kThreads;
    if (q < RT * TB) {
      const int r = q / TB, t = q % TB;
      // stage row R: sum over the warps of its row group, in order
      auto row_sum = [&](int R) {
        const int g = R / NRG;
        const float *rr = rb + g * KW * RED + (R - g * NRG) * TB + t;
        float acc = 0.0f;
#pragma unroll
        for (int w = 0; w < KW; ++w) acc += rr[w * RED];
        return acc;
      };
      if (t < Tb && n0 + r < rows) {
        const float acc0 = row_sum(r);
        const int64_t pos = static_cast<int64_t>(p0) + t0 + t;
        if constexpr (MODE == kGateUp) {
          const float acc1 = row_sum(RT + r);
          a.ws.h[pos * rows + n0 + r] = silu(acc0) * acc1;
        } else if constexpr (MODE == kDown) {
          a.ws.out[pos * rows + n0 + r] = acc0;
        } else {
          store_y(a.y, pos * rows + n0 + r, acc0, a.y_bf16);
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    // After an abort, wait (bounded) for the copies that may still be landing
    // (tiles pending .. issued - 1); after a normal end they have all landed.
    for (int64_t u = pending; u < issued; ++u)
      mbar_wait_bounded(smem_addr(&full_bar[u % STAGES]), static_cast<uint32_t>((u / STAGES) & 1),
                        a.status);
  }
  __syncthreads();
}

template <int BITS, int XPL, int KW, int MODE, bool XBF16, int TBMAX>
__global__ void __launch_bounds__(kThreads, Cfg<TBMAX>::kCtas) smallm_kernel(const Args a) {
  smallm_body<BITS, XPL, KW, MODE, XBF16, TBMAX>(a, a.idx, []() {
    pdl_enter();
    return true;
  });
}

template <int BITS, int XPL, int KW, int MODE, bool XBF16, int TBMAX>
cudaError_t run(const Args &a, cudaStream_t s) {
  auto k = smallm_kernel<BITS, XPL, KW, MODE, XBF16, TBMAX>;
  const int smem = Cfg<TBMAX>::smem_bytes(a.E, a.idx ? a.MK : 0);
  cudaError_t e = ensure_smem(reinterpret_cast<const void *>(k), smem);
  if (e != cudaSuccess) return e;
  // A linear layer with fewer tiles than CTA slots gets one CTA per tile,
  // which leaves the other slots to the next launch's early prologue.
  int grid = Cfg<TBMAX>::kCtas * sm_count();
  if (MODE == kLinear && a.tiles < grid) grid = a.tiles;
  return launch_pdl(k, dim3(grid), dim3(kThreads), smem, s, a);
}

// K = 4096: eight warps of 16 columns per lane.  K = 2048: the digit form
// keeps 16 columns per lane (four warps per row, two row groups: half the
// per-row reduction and conversion work per code of eight columns); the
// eight-row fp32 form keeps eight warps of 8 columns (its activation rows
// would not fit in registers at 16).
template <int MODE, bool XBF16, int TBMAX>
cudaError_t run_shape(const Args &a, cudaStream_t s) {
  const bool wide = a.K == 4096;
  if constexpr (TBMAX == 1) {
    // routed experts, one token per pass: 32 columns per lane (K = 4096:
    // four warps per row, two row groups; K = 2048: two warps, four groups)
    if (a.w0.bits == 4)
      return wide ? run<4, 32, 4, MODE, XBF16, TBMAX>(a, s) : run<4, 32, 2, MODE, XBF16, TBMAX>(a, s);
    return wide ? run<8, 32, 4, MODE, XBF16, TBMAX>(a, s) : run<8, 32, 2, MODE, XBF16, TBMAX>(a, s);
  } else if constexpr (TBMAX == 2) {
    if (a.w0.bits == 4)
      return wide ? run<4, 16, 8, MODE, XBF16, TBMAX>(a, s) : run<4, 16, 4, MODE, XBF16, TBMAX>(a, s);
    return wide ? run<8, 16, 8, MODE, XBF16, TBMAX>(a, s) : run<8, 16, 4, MODE, XBF16, TBMAX>(a, s);
  } else {
    if (a.w0.bits == 4)
      return wide ? run<4, 16, 8, MODE, XBF16, TBMAX>(a, s) : run<4, 8, 8, MODE, XBF16, TBMAX>(a, s);
    return wide ? run<8, 16, 8, MODE, XBF16, TBMAX>(a, s) : run<8, 8, 8, MODE, XBF16, TBMAX>(a, s);
  }
}

// TBMAX 1: the routed experts (gate/up, down); TBMAX 2 and 8: the linear
// layer.
template <int TBMAX>
cudaError_t run_class(int mode, bool x_bf16, const Args &a, cudaStream_t s) {
  if constexpr (TBMAX == 1) {
    if (mode == kGateUp)
      return x_bf16 ? run_shape<kGateUp, true, 1>(a, s) : run_shape<kGateUp, false, 1>(a, s);
    if (mode == kDown) return run_shape<kDown, false, 1>(a, s);
    return cudaErrorInvalidValue;
  } else {
    if (mode == kLinear)
      return x_bf16 ? run_shape<kLinear, true, TBMAX>(a, s) : run_shape<kLinear, false, TBMAX>(a, s);
    return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace smallm
}  // namespace qmm
