// smallm_hi.cu -- small-M kernels with eight activation rows per pass (one
// CTA per SM): the linear layer with 3..8 rows.
#include "smallm_kernel.cuh"

namespace qmm {
namespace smallm {

cudaError_t run_hi(int mode, bool x_bf16, const Args &a, cudaStream_t s) {
  return run_class<8>(mode, x_bf16, a, s);
}

}  // namespace smallm
}  // namespace qmm
