// smallm_lo.cu -- small-M kernels with two activation rows per pass (two
// CTAs per SM): the linear layer with 1..2 rows.
#include "smallm_kernel.cuh"

namespace qmm {
namespace smallm {

cudaError_t run_lo(int mode, bool x_bf16, const Args &a, cudaStream_t s) {
  return run_class<2>(mode, x_bf16, a, s);
}

}  // namespace smallm
}  // namespace qmm
