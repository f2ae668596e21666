// smallm.cu -- host side of the small-M fused dequantise-matmul: argument
// set-up and the launchers used by qmm_linear and the MoE layer (kernel in
// smallm_kernel.cuh, design notes in smallm.cuh).
#include <cstdint>

#include "smallm.cuh"

namespace qmm {
namespace smallm {

Args base_args(const QMat &w, int nm) {
  Args a{};
  a.w0 = w;
  a.w1 = w;
  a.rows = w.rows;
  a.K = w.cols;
  a.rowbytes = static_cast<int>(w.cols * w.bits / 8);
  a.G = static_cast<int>(w.cols / w.group);
  a.group = w.group;
  const int nr = (w.bits == 4 ? 16 : 8) * 16 / static_cast<int>(w.cols / 256);
  const int rt = nr / nm;
  a.tiles = static_cast<int>((w.rows + rt - 1) / rt);
  a.status = device_status();
  return a;
}

}  // namespace smallm

bool smallm_supported(int bits, int group, int64_t K) {
  if (bits != 4 && bits != 8) return false;
  if (K != 2048 && K != 4096) return false;
  if (group < 64 || K % group != 0 || (K / group) % 4 != 0) return false;
  return group % 16 == 0;  // a lane's 16 (or 8) columns never straddle a group
}

cudaError_t launch_smallm_linear(const void *x, bool x_bf16, int64_t M, const QMat &w, void *y,
                                 bool y_bf16, cudaStream_t s) {
  smallm::Args a = smallm::base_args(w, 1);
  a.E = 1;
  a.k = 1;
  a.M = M;
  a.x = x;
  a.y = y;
  a.y_bf16 = y_bf16;
  // One segment of M rows.  One or two rows: the two-row digit kernel; but
  // a small INT4 matrix with one row takes the eight-row fp32 kernel, whose
  // activations need no conversion: such a launch is bound by its latency
  // chain (activation load and conversion, one or two tiles per CTA, the
  // output), not by its arithmetic (GB300: INT4 g128 4096x4096 + 2048x4096,
  // 12.4 us per pair against 13.1 with the digit kernel; INT8 4096x4096 pairs
  // are faster on the digit kernel, 14.6 against 15.5 us).
  if (M == 1 && w.bits == 4 && w.rows * w.cols <= (int64_t(1) << 25))
    return smallm::run_hi(smallm::kLinear, x_bf16, a, s);
  return M <= 2 ? smallm::run_lo(smallm::kLinear, x_bf16, a, s)
                : smallm::run_hi(smallm::kLinear, x_bf16, a, s);
}

cudaError_t launch_smallm_gateup(const void *x, bool x_bf16, int k, int E, const QMat &gate,
                                 const QMat &up, const MoeWork &ws, cudaStream_t s,
                                 const int32_t *idx, int64_t MK) {
  smallm::Args a = smallm::base_args(gate, 2);
  a.w1 = up;
  a.E = E;
  a.k = k;
  a.ws = ws;
  a.x = x;
  a.idx = idx;
  a.MK = MK;
  a.pos_out = idx ? ws.pos : nullptr;
  return smallm::run_one(smallm::kGateUp, x_bf16, a, s);
}

cudaError_t launch_smallm_down(int k, int E, const QMat &down, const MoeWork &ws, cudaStream_t s,
                               const int32_t *idx, int64_t MK) {
  smallm::Args a = smallm::base_args(down, 1);
  a.E = E;
  a.k = k;
  a.ws = ws;
  a.idx = idx;
  a.MK = MK;
  return smallm::run_one(smallm::kDown, false, a, s);
}

}  // namespace qmm
