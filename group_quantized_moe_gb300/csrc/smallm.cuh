// smallm.cuh -- fused dequantise-matmul for a few activation rows per weight
// matrix on the CUDA cores: the routed experts of a decode batch and the
// one- or two-token experts of a prefill batch (gate + up with the SwiGLU
// epilogue, then down), and qmm_linear for 1..8 rows.
//
// "Why I hand-wrote a DeepSeek inference engine in pure C", section 3.2
// (the codes are dequantised inside the dot product, never written out as
// fp32 weights) and section 3.5 (the tokens routed to one expert share one
// pass over its weights).
//
// GB300 design (HBM-bound: each weight byte is used by 1..8 tokens):
//  * CTAs of eight warps, one or two per SM (see Cfg).  One thread streams
//    tiles of whole weight rows -- codes, fp32 scales and int32 zero points,
//    three 1-D bulk copies per matrix -- through a ring of 40 KB stages,
//    completion on one mbarrier per stage (every wait bounded).  A stage is
//    refilled right after the CTA barrier that ends its last use, so no
//    "empty" barrier is needed.
//  * KW warps split the K range of a row (K = 32 KW XPL; the 8 / KW row
//    groups of the CTA take disjoint rows of each stage): lane l of warp w
//    owns columns [(32 (w mod KW) + l) XPL, +XPL), XPL = 8, 16 or 32, and
//    keeps those columns of its activation rows in registers for as long as
//    the CTA stays on one expert.  The slice never straddles a quantisation
//    group, so it needs one scale and one zero point per row.
//  * Each lane dequantises its slice of a row once and applies it to every
//    token.  The per-lane partials of a block of rows are reduced across the
//    warp by a butterfly that halves the values a lane carries at every step
//    (about one shuffle per value instead of five), then across the KW
//    warps of the row group through shared memory in a fixed order.
//  * Each CTA takes one contiguous range of tiles, balanced by a per-tile
//    cost that grows with the expert's token count; it therefore reads one
//    contiguous stretch of HBM and reloads activations only when its range
//    crosses into the next expert.
#pragma once

#include <cstdint>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace smallm {

constexpr int kCW = 8;                       // warps; the K range is split 8 ways
constexpr int kThreads = kCW * 32;
constexpr int kStageBytes = 40960;

// Three configurations (TBMAX = activation rows per pass).  TBMAX 1 and 2
// use two CTAs per SM (128 registers) and integer byte dot products of the
// codes with the activations held as balanced digits (smallm_kernel.cuh).
// TBMAX 1 runs the routed experts of decode batches and the experts of a
// prefill batch that have one or two tokens: most of them have one token, and
// with one row per pass a lane can hold 32 columns, which halves the per-row
// work (scale, zero point, conversions, reduction) per code; an expert with T
// tokens is applied in T passes, each a sweep over the CTA's tiles of that
// expert (activations load once per pass, the tiles stream again, from L2
// after the first pass).  TBMAX 2 (16 columns per lane) runs the linear layer
// with one or two rows.  TBMAX 8 (one CTA per SM, eight fp32 rows per pass)
// runs the linear layer with 3..8 rows, where every tile serves all M rows,
// and small INT4 matrices with one row (no activation conversion).
template <int TBMAX>
struct Cfg {
  static constexpr int kCtas = TBMAX <= 2 ? 2 : 1;      // CTAs per SM
  static constexpr int kStages = TBMAX <= 2 ? 2 : 4;    // ring stages per CTA
  static constexpr int kRedMax = TBMAX * 32;            // rows x tokens per tile
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kRedBytes = 2 * kCW * kRedMax * 4;
  // the two low activation digits of the one- and two-row configurations
  // (TBMAX rows x 2 digits x XPL / 4 words per lane, XPL = 32 / TBMAX), read
  // only by warps that need all five digits
  static constexpr int kLowBytes = TBMAX <= 2 ? kCW * 32 * 2 * 8 * 4 : 0;
  // segments (3 E + 2 ints), and for the in-CTA grouping of a decode batch
  // the assignments' experts and sorted order (2 MK) and the counts (E)
  static int smem_bytes(int E, int64_t MK) {
    return kRingBytes + kRedBytes + kLowBytes + (3 * E + 2) * 4 +
           static_cast<int>(2 * MK + E) * 4;
  }
};

enum Mode { kLinear = 0, kGateUp = 1, kDown = 2 };

struct Args {
  QMat w0, w1;      // linear / down: w0; gate/up: w0 = gate, w1 = up
  int64_t rows;     // rows of each matrix (N, I or H)
  int64_t K;        // columns
  int rowbytes;     // code bytes per row
  int G;            // groups per row
  int group;
  int tiles;        // tiles per segment: ceil(rows / rows-per-matrix-per-tile)
  int E;            // experts (MoE); 1 for the linear layer
  int k;            // top-k: sorted position p holds token assign[p] / k
  int64_t M;        // linear: activation rows
  MoeWork ws;
  // Decode batches: the expert kernels group the M k assignments themselves
  // from the top-k indices (no dispatch kernel); gate/up's CTA 0 writes the
  // sorted position of every assignment to pos_out for the combine.
  const int32_t *idx;  // [M k] expert of each assignment, or NULL (use ws)
  int64_t MK;
  int32_t *pos_out;
  const void *x;    // linear and gate/up: activations [*, K]
  void *y;          // linear: output [M, rows], fp32 or (y_bf16) bf16
  bool y_bf16;
  uint32_t *status;
};

// Rows of all matrices per tile (one stage): the most whole rows, a power
// of two, whose codes, scales and zero points fit 40 KB for group >= 64
// (KB = K / 256).
template <int BITS, int KB>
__host__ __device__ constexpr int rows_per_tile() {
  return (BITS == 4 ? 16 : 8) * 16 / KB;
}

// Cost of one tile of a segment with T tokens applied in passes of TBMAX:
// every pass streams and dequantises the tile (~2 token units), then one
// unit per token.
__host__ __device__ __forceinline__ int tile_cost(int T, int TBMAX) {
  return 2 * ((T + TBMAX - 1) / TBMAX) + T;
}

// Arguments for nm matrices of w's shape sharing a tile (gate/up: 2), the
// rest zero (host).
Args base_args(const QMat &w, int nm);

// Launch with TBMAX 1 (the routed experts), 2 (any mode) or 8 (the linear
// layer only).
cudaError_t run_one(int mode, bool x_bf16, const Args &a, cudaStream_t s);
cudaError_t run_lo(int mode, bool x_bf16, const Args &a, cudaStream_t s);
cudaError_t run_hi(int mode, bool x_bf16, const Args &a, cudaStream_t s);

}  // namespace smallm
}  // namespace qmm
