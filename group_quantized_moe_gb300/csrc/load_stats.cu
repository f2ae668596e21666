// load_stats.cu -- routing load statistics and the bounded-wait diagnostic.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.5 (last
// paragraph): the grouped expert computation degenerates towards serial work
// when many tokens pick the same expert, so the engine checks how often each
// expert was chosen and warns when one exceeds a threshold.  Here the check
// runs on the device over the router's histogram and raises a bit in the
// device status word instead of printing.
#include <cstdint>

#include "../../include/qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

// One block of 1024 threads; thread e reads expert e's count (E <= 1024).
// stats: [0] largest count, [1] its expert (the lowest index among equal
// counts), [2] experts with at least one token, [3] sum of the counts.
__global__ void __launch_bounds__(1024) load_stats_kernel(const int32_t *__restrict__ counts,
                                                          int E, int64_t threshold,
                                                          int64_t *__restrict__ stats,
                                                          uint32_t *status) {
  pdl_enter();
  __shared__ uint64_t part_key[32];
  __shared__ int64_t part_sum[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int32_t c = e < E ? counts[e] : 0;
  // key: the count in the high half (offset so that negative counts order
  // below zero), 1023 - e in the low half, so the largest key has the largest
  // count and, among equal counts, the lowest expert index
  uint64_t key = e < E ? (static_cast<uint64_t>(static_cast<uint32_t>(c) ^ 0x80000000u) << 32) |
                             static_cast<uint32_t>(1023 - e)
                       : 0ull;
  int64_t sum = c;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const uint64_t k2 = __shfl_xor_sync(0xFFFFFFFFu, key, o);
    key = k2 > key ? k2 : key;
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  }
  if (lane == 0) {
    part_key[warp] = key;
    part_sum[warp] = sum;
  }
  const int touched = __syncthreads_count(e < E && c > 0);
  if (e == 0) {
    uint64_t best = part_key[0];
    int64_t total = part_sum[0];
    for (int w = 1; w < 32; ++w) {
      best = part_key[w] > best ? part_key[w] : best;
      total += part_sum[w];
    }
    const int32_t mx = static_cast<int32_t>(static_cast<uint32_t>(best >> 32) ^ 0x80000000u);
    stats[0] = mx;
    stats[1] = 1023 - static_cast<int64_t>(best & 0xFFFFFFFFull);
    stats[2] = touched;
    stats[3] = total;
    if (mx > threshold) atomicOr(status, kDevExpertOverload);
  }
}

// A single thread waits on a barrier that expects one arrival and never
// gets it, with the library's bounded wait and the given limit.
__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    mbar_fence_init();
    mbar_wait_bounded(b, 0, status, limit_ns);
  }
}

}  // namespace

cudaError_t launch_load_stats(const int32_t *counts, int E, int64_t threshold, int64_t *stats,
                              cudaStream_t s) {
  return launch_pdl(load_stats_kernel, dim3(1), dim3(1024), 0, s, counts, E, threshold, stats,
                    device_status());
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, cudaStream_t s) {
  return launch_pdl(wait_timeout_kernel, dim3(1), dim3(32), 0, s, limit_ns, device_status());
}

}  // namespace qmm
