"""Input recipes of the five workloads (shapes, seeds, streams, distributions).

Host-side generation only (numpy, via the counter-based generator in
``synth.c``); both the CUDA path and the oracle read these arrays.  Every
tensor has its own stream so that any row range can be regenerated alone:
a stacked expert tensor [E, rows, cols] is one stream indexed by
e * rows * cols + row * cols + col.

Streams: x 1; first weight 2, second weight 3 (outlier masks: stream + 100);
router weight 10; router bias 20; expert gate 11, up 12, down 13.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import normal, outliers, to_bf16, zipf_bias

S_X, S_W0, S_W1, S_WR, S_BIAS = 1, 2, 3, 10, 20
S_GATE, S_UP, S_DOWN = 11, 12, 13
OUTLIER_STREAM_OFFSET = 100


@dataclass(frozen=True)
class LinearRecipe:
    name: str
    N: int
    K: int
    M: int
    bits: int
    group: int
    stream: int
    sigma: float = 0.02
    outlier_p: float = 0.0
    outlier_factor: float = 20.0
    seed: int = 0


@dataclass(frozen=True)
class MoeRecipe:
    name: str
    M: int
    H: int
    I: int
    E: int
    k: int
    bits: int
    group: int
    x_bf16: bool
    zipf_s: float | None  # router bias strength (None: no bias)
    sigma_w: float = 0.02
    sigma_r: float = 0.02
    seed: int = 0


# Single INT8 group-64 linear (small correctness case).
CFG1 = LinearRecipe("int8_g64_k256_n128", N=128, K=256, M=1, bits=8, group=64, stream=S_W0)
# Decode GEMV, INT8 group 64, 1% outliers x20; trunk projection and vocab head.
CFG2_TRUNK = LinearRecipe("int8_g64_k4096_n4096", N=4096, K=4096, M=1, bits=8, group=64,
                          stream=S_W0, outlier_p=0.01)
CFG2_VOCAB = LinearRecipe("int8_g64_k4096_n129280", N=129280, K=4096, M=1, bits=8, group=64,
                          stream=S_W1, outlier_p=0.01)
# Decode GEMV, INT4 group 128.
CFG3_A = LinearRecipe("int4_g128_k4096_n4096", N=4096, K=4096, M=1, bits=4, group=128,
                      stream=S_W0)
CFG3_B = LinearRecipe("int4_g128_k4096_n2048", N=2048, K=4096, M=1, bits=4, group=128,
                      stream=S_W1)
# MoE decode layer (8 tokens).
CFG4 = MoeRecipe("moe_decode_m8_int4_g64", M=8, H=4096, I=2048, E=256, k=6, bits=4, group=64,
                 x_bf16=False, zipf_s=None)
# Batched-prefill MoE (512 bf16 tokens) with Zipf(1.1) expert popularity.
CFG5 = MoeRecipe("moe_prefill_m512_bf16_int8_g128", M=512, H=4096, I=2048, E=256, k=6, bits=8,
                 group=128, x_bf16=True, zipf_s=1.1)

LINEARS = {r.name: r for r in (CFG1, CFG2_TRUNK, CFG2_VOCAB, CFG3_A, CFG3_B)}
MOES = {r.name: r for r in (CFG4, CFG5)}


def linear_x(r: LinearRecipe, M: int | None = None) -> np.ndarray:
    """Activations [M, K] ~ N(0, 1), fp32."""
    M = r.M if M is None else M
    return normal(r.seed, S_X, M * r.K, 1.0).reshape(M, r.K)


def linear_weight_rows(r: LinearRecipe, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Rows [row0, row0 + nrows) of W ~ N(0, sigma^2) (+ outliers), fp32."""
    nrows = r.N - row0 if nrows is None else nrows
    off = row0 * r.K
    w = normal(r.seed, r.stream, nrows * r.K, r.sigma, offset=off)
    if r.outlier_p > 0:
        outliers(r.seed, r.stream + OUTLIER_STREAM_OFFSET, w, r.outlier_p, r.outlier_factor,
                 offset=off)
    return w.reshape(nrows, r.K)


def moe_x(r: MoeRecipe, rows: np.ndarray | None = None):
    """Token activations [M, H] ~ N(0, 1).  Returns (fp32 values the kernels
    see, bf16 bit patterns or None).  For bf16 workloads the fp32 values are
    the bf16 values widened exactly."""
    x = normal(r.seed, S_X, r.M * r.H, 1.0).reshape(r.M, r.H)
    if not r.x_bf16:
        return x, None
    bits = to_bf16(x)
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    return xf, bits


def moe_router(r: MoeRecipe):
    """Router weight [E, H] ~ N(0, sigma_r^2) and bias [E] (None or Zipf)."""
    wr = normal(r.seed, S_WR, r.E * r.H, r.sigma_r).reshape(r.E, r.H)
    bias = zipf_bias(r.seed, S_BIAS, r.E, r.zipf_s) if r.zipf_s is not None else None
    return wr, bias


def moe_expert_rows(r: MoeRecipe, which: str, e: int, row0: int = 0,
                    nrows: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Rows of expert e's fp32 matrix: gate/up [I, H], down [H, I]."""
    stream = {"gate": S_GATE, "up": S_UP, "down": S_DOWN}[which]
    rows, cols = (r.I, r.H) if which in ("gate", "up") else (r.H, r.I)
    nrows = rows - row0 if nrows is None else nrows
    off = (e * rows + row0) * cols
    flat = None if out is None else out.reshape(-1)
    w = normal(r.seed, stream, nrows * cols, r.sigma_w, offset=off, out=flat)
    return w.reshape(nrows, cols)
