// smallm.cu -- host side of the small-M fused dequantise-matmul: argument
// set-up and the launchers used by qmm_linear and the MoE layer (kernel in
// smallm_kernel.cuh, design notes in smallm.cuh).
#include <cstdint>

#include "smallm.cuh"

namespace qmm {
namespace smallm {
namespace {

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

}  // namespace
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
  // One segment of M rows: the class its token count selects (one row: 32
  // columns per lane, which spreads the per-row work over twice the codes).
  if (M == 1) return smallm::run_one(smallm::kLinear, x_bf16, a, s);
  return M <= 2 ? smallm::run_lo(smallm::kLinear, x_bf16, a, s)
                : smallm::run_hi(smallm::kLinear, x_bf16, a, s);
}

cudaError_t launch_smallm_gateup(const void *x, bool x_bf16, int k, int E, const QMat &gate,
                                 const QMat &up, const MoeWork &ws, cudaStream_t s,
                                 int rows_per_pass, const int32_t *idx, int64_t MK) {
  smallm::Args a = smallm::base_args(gate, 2);
  a.w1 = up;
  a.E = E;
  a.k = k;
  a.ws = ws;
  a.x = x;
  a.idx = idx;
  a.MK = MK;
  a.pos_out = idx ? ws.pos : nullptr;
  return rows_per_pass == 2 ? smallm::run_lo(smallm::kGateUp, x_bf16, a, s)
                            : smallm::run_one(smallm::kGateUp, x_bf16, a, s);
}

cudaError_t launch_smallm_down(int k, int E, const QMat &down, const MoeWork &ws, cudaStream_t s,
                               int rows_per_pass, const int32_t *idx, int64_t MK) {
  smallm::Args a = smallm::base_args(down, 1);
  a.E = E;
  a.k = k;
  a.ws = ws;
  a.idx = idx;
  a.MK = MK;
  return rows_per_pass == 2 ? smallm::run_lo(smallm::kDown, false, a, s)
                            : smallm::run_one(smallm::kDown, false, a, s);
}

}  // namespace qmm
