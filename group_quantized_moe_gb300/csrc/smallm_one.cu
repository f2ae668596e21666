// smallm_one.cu -- small-M kernels with one activation row per pass and 32
// columns per lane (two CTAs per SM): the routed experts of decode batches.
#include "smallm_kernel.cuh"

namespace qmm {
namespace smallm {

cudaError_t run_one(int mode, bool x_bf16, const Args &a, cudaStream_t s) {
  return run_class<1>(mode, x_bf16, a, s);
}

}  // namespace smallm
}  // namespace qmm
