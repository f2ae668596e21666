"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This package holds random-number generation and input shaping only (Gaussian
draws, sparse outliers, a seeded permutation and Zipf-shaped bias, a bf16
cast).  It contains none of the quantisation, matmul or routing arithmetic, so
the CUDA path and the CPU oracle can both consume its output without sharing
any of the method's code.  The generator itself is defined in ``synth.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32, dbl = (ctypes.c_uint64, ctypes.c_int64,
                                  ctypes.c_int32, ctypes.c_double)
            vp = ctypes.c_void_p
            lib.synth_raw.argtypes = [u64, u64, u64]
            lib.synth_raw.restype = u64
            lib.synth_normal.argtypes = [u64, u64, u64, u64, dbl, vp]
            lib.synth_normal.restype = None
            lib.synth_outliers.argtypes = [u64, u64, u64, u64, dbl, dbl, vp]
            lib.synth_outliers.restype = i64
            lib.synth_to_bf16.argtypes = [vp, vp, u64]
            lib.synth_to_bf16.restype = None
            lib.synth_permutation.argtypes = [u64, u64, i32, vp]
            lib.synth_permutation.restype = None
            lib.synth_zipf_bias.argtypes = [u64, u64, i32, dbl, vp]
            lib.synth_zipf_bias.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("array must be C-contiguous")
    return a.ctypes.data


def raw(seed: int, stream: int, counter: int) -> int:
    """The 64-bit generator output at ``counter`` of (seed, stream)."""
    return int(_load().synth_raw(seed, stream, counter))


def normal(seed: int, stream: int, count: int, sigma: float = 1.0,
           offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """Elements [offset, offset+count) of the N(0, sigma^2) stream, fp32."""
    if out is None:
        out = np.empty(count, dtype=np.float32)
    if out.dtype != np.float32 or out.size != count:
        raise ValueError("out must be float32 with `count` elements")
    if count:
        _load().synth_normal(seed, stream, offset, count, sigma, _ptr(out))
    return out


def outliers(seed: int, stream: int, arr: np.ndarray, p: float,
             factor: float, offset: int = 0) -> int:
    """Scale elements of ``arr`` (in place) by ``factor`` with probability p."""
    if arr.dtype != np.float32:
        raise ValueError("arr must be float32")
    if arr.size == 0:
        return 0
    return int(_load().synth_outliers(seed, stream, offset, arr.size, p,
                                      factor, _ptr(arr)))


def to_bf16(arr: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even bf16 bit patterns (uint16) of a float32 array."""
    arr = np.ascontiguousarray(arr, dtype=np.float32)
    out = np.empty(arr.shape, dtype=np.uint16)
    if arr.size:
        _load().synth_to_bf16(_ptr(arr), _ptr(out), arr.size)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_permutation(seed, stream, n, _ptr(out))
    return out


def zipf_bias(seed: int, stream: int, n: int, s: float) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_zipf_bias(seed, stream, n, s, _ptr(out))
    return out
