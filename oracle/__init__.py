"""CPU oracle for the group-wise quantised linear layer, the routed MoE FFN and
the decode attention step that uses the same quantised projections.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The arithmetic lives in plain C
(``qmm_oracle.c``, single thread, -O2 -ffp-contract=off, no -ffast-math); this
module only marshals numpy arrays to it.  It shares no code with the CUDA
library and never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_HDR = os.path.join(_HERE, "qmm_oracle.h")
_LIB_PATH = os.path.join(_HERE, "libqmm_oracle.so")
# A prebuilt variant of the same source (the tests' sanitizer build) may be
# named in QMM_ORACLE_LIB; it is loaded as it is.
_LIB_OVERRIDE = os.environ.get("QMM_ORACLE_LIB")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``libqmm_oracle.so`` (gcc, single thread)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _QW(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zps", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            i32, i64, vp, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            pqw = ctypes.POINTER(_QW)
            lib.orc_quantize.argtypes = [vp, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp]
            lib.orc_quantize.restype = ctypes.c_int
            lib.orc_code_at.argtypes = [pqw, i64, i64]
            lib.orc_code_at.restype = i32
            lib.orc_dequantize.argtypes = [pqw, vp]
            lib.orc_dequantize.restype = None
            for name in ("orc_linear_fused", "orc_linear_two_step", "orc_linear_bound"):
                getattr(lib, name).argtypes = [vp, i64, pqw, vp]
                getattr(lib, name).restype = None
            lib.orc_router_logits.argtypes = [vp, i64, i64, vp, vp, i32, vp]
            lib.orc_router_logits.restype = None
            lib.orc_topk.argtypes = [vp, i64, i32, i32, vp, vp]
            lib.orc_topk.restype = None
            lib.orc_moe_ffn.argtypes = [vp, i64, i64, i64, vp, vp, i32, i32,
                                        pqw, pqw, pqw, dbl, vp, vp]
            lib.orc_moe_ffn.restype = ctypes.c_int
            lib.orc_load_stats.argtypes = [vp, i64, i32, i32, i64, vp]
            lib.orc_load_stats.restype = ctypes.c_int
            lib.orc_rope_table.argtypes = [i64, i32, dbl, vp, vp]
            lib.orc_rope_table.restype = None
            lib.orc_rope_apply.argtypes = [vp, i32, i32, i64, vp, vp, vp]
            lib.orc_rope_apply.restype = None
            lib.orc_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i64,
                                          i64, vp, vp]
            lib.orc_attention.restype = None
            lib.orc_attn_decode.argtypes = [vp, i64, i32, i32, i32, i64, pqw, pqw, pqw, pqw,
                                            vp, vp, vp, vp, vp, vp, vp]
            lib.orc_attn_decode.restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


@dataclass
class QWeight:
    """Quantised W[N,K] as the oracle stores it (numpy arrays)."""
    bits: int
    group: int
    N: int
    K: int
    codes: np.ndarray   # uint8 [N*K] (int8 bit patterns) or [N*K/2] packed
    scales: np.ndarray  # float32 [N, K/group]
    zps: np.ndarray     # int32 [N, K/group]

    def _struct(self) -> _QW:
        return _QW(self.bits, self.group, self.N, self.K, self.codes.ctypes.data,
                   self.scales.ctypes.data, self.zps.ctypes.data)


def quantize(w: np.ndarray, bits: int, group: int) -> QWeight:
    w = _c(w, np.float32)
    N, K = w.shape
    nbytes = N * K if bits == 8 else N * K // 2
    codes = np.zeros(nbytes, dtype=np.uint8)
    G = K // group if group > 0 else 0
    scales = np.zeros((N, G), dtype=np.float32)
    zps = np.zeros((N, G), dtype=np.int32)
    rc = _load().orc_quantize(w.ctypes.data, N, K, bits, group, codes.ctypes.data,
                              scales.ctypes.data, zps.ctypes.data)
    if rc != 0:
        raise ValueError(f"orc_quantize rejected N={N} K={K} bits={bits} group={group}")
    return QWeight(bits, group, N, K, codes, scales, zps)


def code_at(qw: QWeight, n: int, k: int) -> int:
    s = qw._struct()
    return int(_load().orc_code_at(ctypes.byref(s), n, k))


def dequantize(qw: QWeight) -> np.ndarray:
    out = np.empty((qw.N, qw.K), dtype=np.float32)
    s = qw._struct()
    _load().orc_dequantize(ctypes.byref(s), out.ctypes.data)
    return out


def _linear(name: str, x: np.ndarray, qw: QWeight) -> np.ndarray:
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M = x.shape[0]
    assert x.shape[1] == qw.K
    y = np.empty((M, qw.N), dtype=np.float64)
    s = qw._struct()
    getattr(_load(), name)(x.ctypes.data, M, ctypes.byref(s), y.ctypes.data)
    return y


def linear_fused(x, qw):
    """y[m,n] = sum_k x[m,k] (q-zp) s, dequantised inside the k loop (double)."""
    return _linear("orc_linear_fused", x, qw)


def linear_two_step(x, qw):
    """Dequantise the whole matrix, then multiply (double)."""
    return _linear("orc_linear_two_step", x, qw)


def linear_bound(x, qw):
    """1e-5 * sum_k |x_k w^_k| + 1e-6 per output."""
    return _linear("orc_linear_bound", x, qw)


def router_logits(x: np.ndarray, wr: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    x = _c(x, np.float32)
    wr = _c(wr, np.float32)
    M, H = x.shape
    E = wr.shape[0]
    assert wr.shape[1] == H
    out = np.empty((M, E), dtype=np.float32)
    bp = None
    if bias is not None:
        bias = _c(bias, np.float32)
        bp = bias.ctypes.data
    _load().orc_router_logits(x.ctypes.data, M, H, wr.ctypes.data, bp, E, out.ctypes.data)
    return out


def topk(logits: np.ndarray, k: int):
    logits = _c(logits, np.float32)
    M, E = logits.shape
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float32)
    _load().orc_topk(logits.ctypes.data, M, E, k, idx.ctypes.data, w.ctypes.data)
    return idx, w


def _qw_array(ws, E):
    arr = (_QW * E)()
    for e in range(E):
        if ws[e] is not None:
            arr[e] = ws[e]._struct()
    return arr


def moe_ffn(x: np.ndarray, idx: np.ndarray, w: np.ndarray, gate, up, down,
            dw: float = 0.0, with_bound: bool = True):
    """Routed SwiGLU MoE output y[M,H] (double) and its per-element bound.

    gate/up/down: lists of length E holding QWeight (or None for experts that
    no token selected)."""
    x = _c(x, np.float32)
    idx = _c(idx, np.int32)
    w = _c(w, np.float32)
    M, H = x.shape
    k = idx.shape[1]
    E = len(gate)
    I = next(g.N for g in gate if g is not None)
    y = np.empty((M, H), dtype=np.float64)
    bound = np.empty((M, H), dtype=np.float64) if with_bound else None
    ga, ua, da = _qw_array(gate, E), _qw_array(up, E), _qw_array(down, E)
    rc = _load().orc_moe_ffn(x.ctypes.data, M, H, I, idx.ctypes.data, w.ctypes.data, k, E,
                             ga, ua, da, dw, y.ctypes.data,
                             bound.ctypes.data if bound is not None else None)
    if rc != 0:
        raise ValueError(f"orc_moe_ffn failed ({rc})")
    return y, bound


def load_stats(idx: np.ndarray, E: int, threshold: int):
    """Routing load check: (stats int64 [4] = largest count, its expert, experts
    touched, total selections; flag = largest count > threshold)."""
    idx = _c(idx, np.int32)
    M, k = idx.shape
    stats = np.zeros(4, dtype=np.int64)
    flag = _load().orc_load_stats(idx.ctypes.data, M, k, E, threshold, stats.ctypes.data)
    if flag < 0:
        raise MemoryError("orc_load_stats")
    return stats, bool(flag)


# ------------------------------------------------------------ decode attention

def _ptr(a):
    return a.ctypes.data if a is not None else None


def rope_table(max_seq: int, head_dim: int, base: float = 10000.0):
    """cos, sin float32 [max_seq, head_dim/2] of pos * base^(-2i/head_dim)."""
    hp = head_dim // 2
    c = np.empty((max_seq, hp), dtype=np.float32)
    s = np.empty((max_seq, hp), dtype=np.float32)
    _load().orc_rope_table(max_seq, head_dim, float(base), c.ctypes.data, s.ctypes.data)
    return c, s


def rope_apply(x: np.ndarray, pos: int, cos_t: np.ndarray, sin_t: np.ndarray) -> np.ndarray:
    """Rotates each row of x [n_vec, head_dim] (pairs 2i, 2i+1) to position pos."""
    x = _c(x, np.float64)
    n_vec, hd = x.shape
    cos_t, sin_t = _c(cos_t, np.float32), _c(sin_t, np.float32)
    assert 0 <= pos < cos_t.shape[0] and cos_t.shape[1] == hd // 2
    out = np.empty_like(x)
    _load().orc_rope_apply(x.ctypes.data, n_vec, hd, pos, cos_t.ctypes.data, sin_t.ctypes.data,
                           out.ctypes.data)
    return out


def attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, T: int,
              dq: np.ndarray | None = None, k_last=None, v_last=None, dk_last=None,
              dv_last=None):
    """Decode attention: q [n_head, hd]; caches float32 [n_kv, max_seq, hd],
    rows t < T (row T-1 from k_last / v_last [n_kv, hd] when given).  Returns
    (out [n_head, hd] double, bound)."""
    q = _c(q, np.float64)
    n_head, hd = q.shape
    k_cache, v_cache = _c(k_cache, np.float32), _c(v_cache, np.float32)
    n_kv, max_seq, hd2 = k_cache.shape
    assert hd2 == hd and v_cache.shape == k_cache.shape and 1 <= T <= max_seq
    assert n_head % n_kv == 0
    conv = [None if a is None else _c(a, np.float64) for a in (dq, k_last, v_last, dk_last, dv_last)]
    out = np.empty((n_head, hd), dtype=np.float64)
    bound = np.empty((n_head, hd), dtype=np.float64)
    _load().orc_attention(q.ctypes.data, *[_ptr(a) for a in conv[:1]], k_cache.ctypes.data,
                          v_cache.ctypes.data, *[_ptr(a) for a in conv[1:]], n_head, n_kv, hd,
                          max_seq, T, out.ctypes.data, bound.ctypes.data)
    return out, bound


def attn_decode(x: np.ndarray, pos: int, n_head: int, n_kv: int, head_dim: int,
                wq: QWeight, wk: QWeight, wv: QWeight, wo: QWeight, cos_t, sin_t,
                cache_in: np.ndarray):
    """One decode token through the attention layer.  cache_in float32
    [2, n_kv, max_seq, head_dim] (rows < pos are read).  Returns (y [D_out]
    double, bound, kv_new [2, n_kv, head_dim] double, kv_bound)."""
    x = _c(x, np.float32).reshape(-1)
    cache_in = _c(cache_in, np.float32)
    two, nkv2, max_seq, hd2 = cache_in.shape
    assert two == 2 and nkv2 == n_kv and hd2 == head_dim and 0 <= pos < max_seq
    cos_t, sin_t = _c(cos_t, np.float32), _c(sin_t, np.float32)
    y = np.empty(wo.N, dtype=np.float64)
    bound = np.empty(wo.N, dtype=np.float64)
    kv_new = np.empty((2, n_kv, head_dim), dtype=np.float64)
    kv_bound = np.empty((2, n_kv, head_dim), dtype=np.float64)
    rc = _load().orc_attn_decode(x.ctypes.data, pos, n_head, n_kv, head_dim, max_seq,
                                 ctypes.byref(wq._struct()), ctypes.byref(wk._struct()),
                                 ctypes.byref(wv._struct()), ctypes.byref(wo._struct()),
                                 cos_t.ctypes.data, sin_t.ctypes.data, cache_in.ctypes.data,
                                 kv_new.ctypes.data, kv_bound.ctypes.data, y.ctypes.data,
                                 bound.ctypes.data)
    if rc != 0:
        raise ValueError(f"orc_attn_decode failed ({rc})")
    return y, bound, kv_new, kv_bound
