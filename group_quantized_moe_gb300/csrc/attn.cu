// attn.cu -- decode attention for one token with rotary positions and a KV
// cache ("Why I hand-wrote a DeepSeek inference engine in pure C", section
// 3.4): the kernels between the layer's quantised projections (qmm_linear).
//
//   rope_table_kernel  cos / sin of pos * base^(-2i/d), one thread per entry
//   attn_part_kernel   one CTA per (query head, chunk of 64 cache rows):
//                      rotates the query (and, in the last chunk, this
//                      step's key, which it writes to cache row pos with the
//                      value), then the scores q.k / sqrt(d), their maximum,
//                      the exponentials and their sum, and the
//                      exponential-weighted sum of the value rows (a split of
//                      the softmax over the rows, so that long caches spread
//                      over the SMs)
//   attn_merge_kernel  one CTA per query head: the chunks' partial results
//                      rescaled to the overall maximum and summed in chunk
//                      order, divided by the overall sum (for up to eight
//                      chunks -- 512 cache rows -- the chunks of a head run
//                      as one cluster and merge in distributed shared memory
//                      instead, with no second launch)
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
constexpr int kPartThreads = 256;
constexpr int kMaxCluster = 8;  // chunks merged inside a cluster (portable cluster size)

// Distributed shared memory of the thread-block cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Every thread of every CTA of the cluster; shared-memory writes before it
// are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Requests `bytes` (a multiple of 16) at `src` into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

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

// Partial softmax-weighted sum over cache rows [c * 64, min(T, c * 64 + 64))
// of query head blockIdx.x (key/value head kvh = blockIdx.x / (n_head /
// n_kv)): part = {max score, sum of exp(score - max), sum of
// exp(score - max) v}.  The query arrives unrotated and is rotated here
// (pairs (2i, 2i + 1) by the angles of position pos: (a, b) ->
// (a c - b s, a s + b c)); the last chunk also takes this step's key (rotated
// here) and value from the projections for row pos, which the CTA of the
// group's first query head writes to the cache.
// 256 threads: warp w scores rows 8w .. 8w + 7 (lane l holds the 16-byte
// column units l, l + 32, ...; a batch of rows' loads is in flight before
// the sums); the value rows are summed by (row group, column unit) threads
// and the row groups combined in order.  The chunk's cache rows (written by
// earlier steps, complete before this launch may start) are requested into
// L2 before the wait for the projections.
// CLUSTER: the chunks of a head form one thread-block cluster (at most 8);
// each CTA leaves its partial result in shared memory and the cluster's
// first CTA merges them in chunk order (as attn_merge_kernel does) and
// writes the head's output, so no merge launch follows.
template <int NU, bool CLUSTER>  // NU: 16-byte column units per lane, ceil(head_dim / 128)
__global__ void __launch_bounds__(kPartThreads) attn_part_kernel(
    const float *q, const float *knew, const float *vnew, float *cache, int n_head, int n_kv,
    int head_dim, int64_t max_seq, int64_t pos, const float *cos_t, const float *sin_t,
    float scale, float *part, float *attn_out) {
  __shared__ __align__(16) float qs[512];
  __shared__ __align__(16) float kn[512];
  __shared__ __align__(16) float vn[512];
  __shared__ float ps[kChunk];
  __shared__ float red[kPartThreads / 32];
  __shared__ __align__(16) float4 vred[kPartThreads];
  __shared__ __align__(16) float cpart[CLUSTER ? 512 + 2 : 1];  // this chunk's result
  const int h = blockIdx.x, c = blockIdx.y;
  const int grp = n_head / n_kv, kvh = h / grp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t T = pos + 1;
  const int64_t t0 = static_cast<int64_t>(c) * kChunk;
  const int nt = static_cast<int>(min64(kChunk, T - t0));
  const bool last = t0 + nt == T;         // this chunk holds row pos ...
  const int nc = last ? nt - 1 : nt;      // ... which is not read from the cache
  if (threadIdx.x == 0 && nc > 0) {
    const uint32_t bytes = static_cast<uint32_t>(nc) * head_dim * 4;
    prefetch_l2_bulk(cache + (static_cast<int64_t>(kvh) * max_seq + t0) * head_dim, bytes);
    prefetch_l2_bulk(cache + (static_cast<int64_t>(n_kv + kvh) * max_seq + t0) * head_dim, bytes);
  }
  pdl_enter();
  const int hp = head_dim / 2, d4 = head_dim / 4;
  const float *cr = cos_t + pos * hp, *sr = sin_t + pos * hp;
  for (int i = threadIdx.x; i < hp; i += kPartThreads) {
    const float cc = cr[i], ss = sr[i];
    const float a = q[h * head_dim + 2 * i], b = q[h * head_dim + 2 * i + 1];
    qs[2 * i] = fmaf(a, cc, -b * ss);
    qs[2 * i + 1] = fmaf(a, ss, b * cc);
    if (last) {
      const float ka = knew[kvh * head_dim + 2 * i], kb = knew[kvh * head_dim + 2 * i + 1];
      kn[2 * i] = fmaf(ka, cc, -kb * ss);
      kn[2 * i + 1] = fmaf(ka, ss, kb * cc);
      vn[2 * i] = vnew[kvh * head_dim + 2 * i];
      vn[2 * i + 1] = vnew[kvh * head_dim + 2 * i + 1];
    }
  }
  __syncthreads();
  if (last && h % grp == 0) {  // this step's key and value into cache row pos
    float *kd = cache + (static_cast<int64_t>(kvh) * max_seq + pos) * head_dim;
    float *vd = cache + (static_cast<int64_t>(n_kv + kvh) * max_seq + pos) * head_dim;
    for (int d = threadIdx.x; d < head_dim; d += kPartThreads) {
      kd[d] = kn[d];
      vd[d] = vn[d];
    }
  }
  // value rows of this thread (row group g, column unit u: rows g, g + RG,
  // ...), requested now so that their latency overlaps the scores
  const float *vb = cache + (static_cast<int64_t>(n_kv + kvh) * max_seq + t0) * head_dim;
  const int RG = kPartThreads / d4;  // row groups (>= 2: head_dim <= 512)
  const int g = threadIdx.x / d4, u = threadIdx.x - g * d4;
  constexpr int VPF = NU == 1 ? 8 : 1;  // value rows held per thread (RG >= 8 when NU == 1)
  float4 vpre[VPF];
#pragma unroll
  for (int i = 0; i < VPF; ++i) {
    const int r = g + RG * i;
    vpre[i] = (g < RG && r < nc)
                  ? __ldg(reinterpret_cast<const float4 *>(vb + static_cast<int64_t>(r) * head_dim) + u)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // scores of the cache rows
  float4 qv[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const int j = lane + 32 * u;
    qv[u] = j < d4 ? reinterpret_cast<const float4 *>(qs)[j] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  constexpr int RPW = kChunk / (kPartThreads / 32);  // rows per warp
  constexpr int RB = NU == 1 ? 8 : NU == 2 ? 4 : 2;  // rows per batch of loads
  const float *kb = cache + (static_cast<int64_t>(kvh) * max_seq + t0) * head_dim;
#pragma unroll 1
  for (int rb = 0; rb < RPW; rb += RB) {
    float4 kv[RB][NU];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int row = warp * RPW + rb + r;
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const int j = lane + 32 * u;
        kv[r][u] = (row < nc && j < d4)
                       ? __ldg(reinterpret_cast<const float4 *>(kb + static_cast<int64_t>(row) *
                                                                         head_dim) + j)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      float acc = 0.0f;
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        acc = fmaf(qv[u].x, kv[r][u].x, acc);
        acc = fmaf(qv[u].y, kv[r][u].y, acc);
        acc = fmaf(qv[u].z, kv[r][u].z, acc);
        acc = fmaf(qv[u].w, kv[r][u].w, acc);
      }
      acc = warp_sum(acc);
      const int row = warp * RPW + rb + r;
      if (lane == 0 && row < nc) ps[row] = acc * scale;
    }
  }
  if (last && warp == 0) {  // the score of row pos, from the rotated new key
    float acc = 0.0f;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int j = lane + 32 * u;
      if (j < d4) {
        const float4 kk = reinterpret_cast<const float4 *>(kn)[j];
        acc = fmaf(qv[u].x, kk.x, acc);
        acc = fmaf(qv[u].y, kk.y, acc);
        acc = fmaf(qv[u].z, kk.z, acc);
        acc = fmaf(qv[u].w, kk.w, acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) ps[nt - 1] = acc * scale;
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
  const float wsum = warp_sum(e);
  if (lane == 0) red[warp] = wsum;
  __syncthreads();
  float l = 0.0f;
#pragma unroll
  for (int w = 0; w < kPartThreads / 32; ++w) l += red[w];
  // value rows: thread (g, u) sums rows g, g + RG, ... of column unit u
  // (the first VPF of them already in registers); row pos (the new value)
  // comes last, after the row groups are combined
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (g < RG) {
#pragma unroll
    for (int i = 0; i < VPF; ++i) {
      const int r = g + RG * i;
      if (r < nc) {
        const float p = ps[r];
        acc.x = fmaf(p, vpre[i].x, acc.x);
        acc.y = fmaf(p, vpre[i].y, acc.y);
        acc.z = fmaf(p, vpre[i].z, acc.z);
        acc.w = fmaf(p, vpre[i].w, acc.w);
      }
    }
#pragma unroll 4
    for (int r = g + RG * VPF; r < nc; r += RG) {
      const float p = ps[r];
      const float4 vv = __ldg(reinterpret_cast<const float4 *>(vb + static_cast<int64_t>(r) *
                                                                        head_dim) + u);
      acc.x = fmaf(p, vv.x, acc.x);
      acc.y = fmaf(p, vv.y, acc.y);
      acc.z = fmaf(p, vv.z, acc.z);
      acc.w = fmaf(p, vv.w, acc.w);
    }
  }
  vred[threadIdx.x] = acc;
  __syncthreads();
  float *out = CLUSTER ? cpart : part + (static_cast<int64_t>(h) * gridDim.y + c) * (head_dim + 2);
  if (threadIdx.x < d4) {
    float4 t = vred[threadIdx.x];
    for (int gg = 1; gg < RG; ++gg) {
      const float4 o = vred[gg * d4 + threadIdx.x];
      t.x += o.x;
      t.y += o.y;
      t.z += o.z;
      t.w += o.w;
    }
    if (last) {
      const float p = ps[nt - 1];
      const float4 vv = reinterpret_cast<const float4 *>(vn)[threadIdx.x];
      t.x = fmaf(p, vv.x, t.x);
      t.y = fmaf(p, vv.y, t.y);
      t.z = fmaf(p, vv.z, t.z);
      t.w = fmaf(p, vv.w, t.w);
    }
    out[2 + 4 * threadIdx.x] = t.x;
    out[3 + 4 * threadIdx.x] = t.y;
    out[4 + 4 * threadIdx.x] = t.z;
    out[5 + 4 * threadIdx.x] = t.w;
  }
  if (threadIdx.x == 0) {
    out[0] = m;
    out[1] = l;
  }
  if constexpr (CLUSTER) {
    // the cluster's first CTA merges the chunks' results in chunk order:
    // sum_c exp(m_c - M) o_c / sum_c exp(m_c - M) l_c, M = max_c m_c
    cluster_sync_all();
    if (cluster_rank() == 0) {
      const int nch = static_cast<int>(gridDim.y);
      const uint32_t base = smem_addr(cpart);
      float M = -3.402823466e38f;
      for (int r = 0; r < nch; ++r) M = fmaxf(M, ld_cluster_f32(map_to_rank(base, r)));
      float L = 0.0f;
      for (int r = 0; r < nch; ++r) {
        const uint32_t b = map_to_rank(base, r);
        L = fmaf(expf(ld_cluster_f32(b) - M), ld_cluster_f32(b + 4), L);
      }
      const float inv = 1.0f / L;
      for (int d = threadIdx.x; d < head_dim; d += kPartThreads) {
        float a = 0.0f;
        for (int r = 0; r < nch; ++r) {
          const uint32_t b = map_to_rank(base, r);
          a = fmaf(expf(ld_cluster_f32(b) - M), ld_cluster_f32(b + 4 * (2 + d)), a);
        }
        attn_out[h * head_dim + d] = a * inv;
      }
    }
    cluster_sync_all();  // the other CTAs' shared memory stays until it has been read
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

cudaError_t launch_attn_decode_core(const float *q, const float *k, const float *v, int n_head,
                                    int n_kv, int head_dim, int64_t max_seq, int64_t pos,
                                    const float *cos_t, const float *sin_t, float *cache,
                                    float *part, float *attn_out, cudaStream_t s) {
  const int nchunk = attn_chunks(pos + 1);
  const float scale = static_cast<float>(1.0 / sqrt(static_cast<double>(head_dim)));
  const dim3 grid(n_head, nchunk);
  const int nu = (head_dim + 127) / 128;
  if (nchunk <= kMaxCluster) {
    // one cluster per head: the merge happens in distributed shared memory
    auto kern = nu == 1 ? attn_part_kernel<1, true>
                        : (nu == 2 ? attn_part_kernel<2, true> : attn_part_kernel<4, true>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kPartThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = static_cast<unsigned>(nchunk);
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, q, k, v, cache, n_head, n_kv, head_dim,
                                             max_seq, pos, cos_t, sin_t, scale, part, attn_out);
    count_launch();
    return e;
  }
  cudaError_t e;
  if (nu == 1)
    e = launch_pdl(attn_part_kernel<1, false>, grid, dim3(kPartThreads), 0, s, q, k, v, cache,
                   n_head, n_kv, head_dim, max_seq, pos, cos_t, sin_t, scale, part, attn_out);
  else if (nu == 2)
    e = launch_pdl(attn_part_kernel<2, false>, grid, dim3(kPartThreads), 0, s, q, k, v, cache,
                   n_head, n_kv, head_dim, max_seq, pos, cos_t, sin_t, scale, part, attn_out);
  else
    e = launch_pdl(attn_part_kernel<4, false>, grid, dim3(kPartThreads), 0, s, q, k, v, cache,
                   n_head, n_kv, head_dim, max_seq, pos, cos_t, sin_t, scale, part, attn_out);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_merge_kernel, dim3(n_head), dim3(kPartThreads), 0, s,
                    static_cast<const float *>(part), nchunk, head_dim, attn_out);
}

}  // namespace qmm
