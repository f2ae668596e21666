// attn.cu -- decode attention for one token with rotary positions and a KV
// cache ("Why I hand-wrote a DeepSeek inference engine in pure C", section
// 3.4): the kernels between the layer's quantised projections (qmm_linear).
//
//   rope_table_kernel  cos / sin of pos * base^(-2i/d), one thread per entry
//   rope_kv_kernel     rotates the query heads in place and the new key, and
//                      writes key and value into cache row pos
//   attn_part_kernel   one CTA per (query head, chunk of 64 cache rows):
//                      scores q.k / sqrt(d), their maximum, the exponentials
//                      and their sum, and the exponential-weighted sum of the
//                      value rows (a split of the softmax over the rows, so
//                      that long caches spread over the SMs)
//   attn_merge_kernel  one CTA per query head: the chunks' partial results
//                      rescaled to the overall maximum and summed in chunk
//                      order, divided by the overall sum
//
// GB300: the step is bound by reading the cache (2 n_kv T d fp32 values) and
// by launch latency; every kernel is launched with programmatic stream
// serialization so that its prologue overlaps the previous one.  The orders
// of all sums are fixed, so results are reproducible bit for bit.
#include <cstdint>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int kChunk = 64;      // cache rows per partial CTA
constexpr int kPartThreads = 128;

__global__ void __launch_bounds__(256) rope_table_kernel(int64_t max_seq, int head_dim,
                                                          double base, float *cos_t,
                                                          float *sin_t) {
  pdl_enter();
  const int hp = head_dim / 2;
  const int64_t n = max_seq * hp;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = u / hp;
    const int i = static_cast<int>(u - p * hp);
    const double theta = pow(base, -2.0 * static_cast<double>(i) / static_cast<double>(head_dim));
    const double ang = static_cast<double>(p) * theta;
    cos_t[u] = static_cast<float>(cos(ang));
    sin_t[u] = static_cast<float>(sin(ang));
  }
}

// Pairs (2i, 2i + 1) of every head vector rotate by the angle of position
// pos: (a, b) -> (a c - b s, a s + b c).  Threads [0, n_head hp) take the
// query pairs (in place), the next n_kv hp the key pairs (to cache row pos),
// the next n_kv d the value elements.
__global__ void __launch_bounds__(256) rope_kv_kernel(float *q, const float *k, const float *v,
                                                      int n_head, int n_kv, int head_dim,
                                                      int64_t max_seq, int64_t pos,
                                                      const float *cos_t, const float *sin_t,
                                                      float *cache) {
  pdl_enter();
  const int hp = head_dim / 2;
  const int nq = n_head * hp, nk = n_kv * hp, nv = n_kv * head_dim;
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u < nq + nk) {
    const bool isq = u < nq;
    const int w = isq ? u : u - nq;  // pair index within q or k
    const int h = w / hp, i = w - h * hp;
    const float c = cos_t[pos * hp + i], s = sin_t[pos * hp + i];
    const float *src = isq ? q : k;
    const float a = src[h * head_dim + 2 * i], b = src[h * head_dim + 2 * i + 1];
    const float r0 = fmaf(a, c, -b * s), r1 = fmaf(a, s, b * c);
    float *dst = isq ? q + h * head_dim : cache + (static_cast<int64_t>(h) * max_seq + pos) * head_dim;
    dst[2 * i] = r0;
    dst[2 * i + 1] = r1;
  } else if (u < nq + nk + nv) {
    const int w = u - nq - nk;
    const int h = w / head_dim, d = w - h * head_dim;
    cache[(static_cast<int64_t>(n_kv + h) * max_seq + pos) * head_dim + d] = v[w];
  }
}

// Partial softmax-weighted sum over cache rows [c * 64, min(T, c * 64 + 64))
// of query head blockIdx.x (key/value head blockIdx.x / (n_head / n_kv)):
// part = {max score, sum of exp(score - max), sum of exp(score - max) v}.
__global__ void __launch_bounds__(kPartThreads) attn_part_kernel(const float *q,
                                                                 const float *cache, int n_head,
                                                                 int n_kv, int head_dim,
                                                                 int64_t max_seq, int64_t T,
                                                                 float scale, float *part) {
  __shared__ __align__(16) float qs[512];
  __shared__ float ps[kChunk];
  __shared__ float red[kPartThreads / 32];
  pdl_enter();
  const int h = blockIdx.x, c = blockIdx.y;
  const int kvh = h / (n_head / n_kv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(c) * kChunk;
  const int nt = static_cast<int>(min64(kChunk, T - t0));
  for (int d = threadIdx.x; d < head_dim; d += kPartThreads) qs[d] = q[h * head_dim + d];
  __syncthreads();
  // scores: warp w takes rows w, w + 4, ...; lane l columns 4l + 128j
  const float *kb = cache + (static_cast<int64_t>(kvh) * max_seq + t0) * head_dim;
  const int d4 = head_dim / 4;
  for (int r = warp; r < nt; r += kPartThreads / 32) {
    const float4 *kr = reinterpret_cast<const float4 *>(kb + static_cast<int64_t>(r) * head_dim);
    float acc = 0.0f;
    for (int j = lane; j < d4; j += 32) {
      const float4 kv = kr[j];
      const float4 qv = *reinterpret_cast<const float4 *>(qs + 4 * j);
      acc = fmaf(qv.x, kv.x, acc);
      acc = fmaf(qv.y, kv.y, acc);
      acc = fmaf(qv.z, kv.z, acc);
      acc = fmaf(qv.w, kv.w, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) ps[r] = acc * scale;
  }
  __syncthreads();
  // maximum and exponentials (thread r < nt owns row r)
  float m = -3.402823466e38f;
  for (int r = 0; r < nt; ++r) m = fmaxf(m, ps[r]);
  float e = 0.0f;
  if (threadIdx.x < nt) e = expf(ps[threadIdx.x] - m);
  __syncthreads();
  if (threadIdx.x < nt) ps[threadIdx.x] = e;
  // sum of the exponentials: warp sums, then the warps in order
  const float ws = warp_sum(e);
  if (lane == 0) red[warp] = ws;
  __syncthreads();
  float l = 0.0f;
#pragma unroll
  for (int w = 0; w < kPartThreads / 32; ++w) l += red[w];
  // exponential-weighted sum of the value rows, rows in order
  const float *vb = cache + (static_cast<int64_t>(n_kv + kvh) * max_seq + t0) * head_dim;
  float *out = part + (static_cast<int64_t>(h) * gridDim.y + c) * (head_dim + 2);
  for (int d = threadIdx.x; d < head_dim; d += kPartThreads) {
    float acc = 0.0f;
    for (int r = 0; r < nt; ++r) acc = fmaf(ps[r], vb[static_cast<int64_t>(r) * head_dim + d], acc);
    out[2 + d] = acc;
  }
  if (threadIdx.x == 0) {
    out[0] = m;
    out[1] = l;
  }
}

// out[h, d] = sum_c exp(m_c - M) o_c[d] / sum_c exp(m_c - M) l_c, chunks in
// order (M = max_c m_c).
__global__ void __launch_bounds__(kPartThreads) attn_merge_kernel(const float *part, int nchunk,
                                                                  int head_dim, float *out) {
  pdl_enter();
  const int h = blockIdx.x;
  const float *ph = part + static_cast<int64_t>(h) * nchunk * (head_dim + 2);
  float M = -3.402823466e38f;
  for (int c = 0; c < nchunk; ++c) M = fmaxf(M, ph[c * (head_dim + 2)]);
  float L = 0.0f;
  for (int c = 0; c < nchunk; ++c)
    L = fmaf(expf(ph[c * (head_dim + 2)] - M), ph[c * (head_dim + 2) + 1], L);
  const float inv = 1.0f / L;
  for (int d = threadIdx.x; d < head_dim; d += kPartThreads) {
    float acc = 0.0f;
    for (int c = 0; c < nchunk; ++c) {
      const float *pc = ph + c * (head_dim + 2);
      acc = fmaf(expf(pc[0] - M), pc[2 + d], acc);
    }
    out[h * head_dim + d] = acc * inv;
  }
}

}  // namespace

int attn_chunks(int64_t T) { return static_cast<int>((T + kChunk - 1) / kChunk); }

cudaError_t launch_rope_table(int64_t max_seq, int head_dim, double base, float *cos_t,
                              float *sin_t, cudaStream_t s) {
  const int64_t n = max_seq * (head_dim / 2);
  const int64_t blocks = min64((n + 255) / 256, static_cast<int64_t>(sm_count()) * 8);
  return launch_pdl(rope_table_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    max_seq, head_dim, base, cos_t, sin_t);
}

cudaError_t launch_attn_decode_core(float *q, const float *k, const float *v, int n_head,
                                    int n_kv, int head_dim, int64_t max_seq, int64_t pos,
                                    const float *cos_t, const float *sin_t, float *cache,
                                    float *part, float *attn_out, cudaStream_t s) {
  const int nthreads = (n_head + n_kv) * (head_dim / 2) + n_kv * head_dim;
  cudaError_t e = launch_pdl(rope_kv_kernel, dim3((nthreads + 255) / 256), dim3(256), 0, s, q, k,
                             v, n_head, n_kv, head_dim, max_seq, pos, cos_t, sin_t, cache);
  if (e != cudaSuccess) return e;
  const int64_t T = pos + 1;
  const int nchunk = attn_chunks(T);
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(head_dim)));
  e = launch_pdl(attn_part_kernel, dim3(n_head, nchunk), dim3(kPartThreads), 0, s,
                 static_cast<const float *>(q), static_cast<const float *>(cache), n_head, n_kv,
                 head_dim, max_seq, T, scale, part);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_merge_kernel, dim3(n_head), dim3(kPartThreads), 0, s,
                    static_cast<const float *>(part), nchunk, head_dim, attn_out);
}

}  // namespace qmm
