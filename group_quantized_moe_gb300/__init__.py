"""Python binding of libqmm.so: group-wise INT8/INT4 quantised linear layer and
routed SwiGLU MoE layer on GB300 (sm_103a).

Thin layer over the C ABI declared in ``include/qmm.h``: every function here
has the name of the C entry point it calls, turns torch tensors into device
pointers and sizes, allocates outputs with torch when the caller passes none,
and raises ``QmmError`` on a non-zero status.  All arithmetic runs in the
library's CUDA kernels; there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import operator
import os
import threading
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")

QMM_OK = 0
QMM_ERR_INVALID_ARG = 1
QMM_ERR_SHAPE = 2
QMM_ERR_ALIGN = 3
QMM_ERR_WORKSPACE = 4
QMM_ERR_CUDA = 5
QMM_ERR_UNSUPPORTED = 6
QMM_F32 = 0
QMM_BF16 = 1
QMM_DEV_WAIT_TIMEOUT = 1
QMM_DEV_BAD_EXPERT = 2
QMM_DEV_EXPERT_OVERLOAD = 4

EXPORTED = ("qmm_quantize_groupwise", "qmm_linear", "moe_route_workspace_bytes", "moe_route_topk",
            "moe_ffn_workspace_bytes", "moe_ffn_forward", "qmm_last_error", "qmm_launch_count",
            "qmm_device_status", "moe_route_topk_noalloc", "moe_route_load_stats",
            "qmm_diag_wait_timeout", "qmm_linear_batched_workspace_bytes",
            "qmm_linear_batched", "qmm_rope_table", "qmm_attn_decode_workspace_bytes",
            "qmm_attn_decode", "moe_decode_workspace_bytes", "moe_decode_forward",
            "qmm_tc_timing", "qmm_tc_timing_ms")
QMM_NOALLOC_MAX_LOGITS = 262144


class QmmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[qmm status {code}] {msg}")
        self.code = code


class _Weight(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zps", ctypes.c_void_p)]


class _ExpertWeights(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("codes_stride", ctypes.c_int64),
                ("scales", ctypes.c_void_p), ("zps", ctypes.c_void_p),
                ("groups_stride", ctypes.c_int64)]


class _AttnLayer(ctypes.Structure):
    _fields_ = [("n_head", ctypes.c_int32), ("n_head_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("max_seq", ctypes.c_int64),
                ("wq", _Weight), ("wk", _Weight), ("wv", _Weight), ("wo", _Weight),
                ("rope_cos", ctypes.c_void_p), ("rope_sin", ctypes.c_void_p)]


class _Experts(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("gate", _ExpertWeights), ("up", _ExpertWeights), ("down", _ExpertWeights)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libqmm.so.  Raises if the library has not been built: there
    is deliberately no fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            i32, i64, u64, vp, sz = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                     ctypes.c_void_p, ctypes.c_size_t)
            L.qmm_quantize_groupwise.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, vp]
            L.qmm_quantize_groupwise.restype = ctypes.c_int
            L.qmm_linear.argtypes = [vp, i32, i64, ctypes.POINTER(_Weight), vp, i32, vp]
            L.qmm_linear.restype = ctypes.c_int
            L.moe_route_workspace_bytes.argtypes = [i64, i32]
            L.moe_route_workspace_bytes.restype = sz
            L.moe_route_topk.argtypes = [vp, i32, i64, i64, vp, vp, i32, i32, vp, vp, vp, vp,
                                         sz, vp]
            L.moe_route_topk.restype = ctypes.c_int
            L.moe_ffn_workspace_bytes.argtypes = [i64, i32, ctypes.POINTER(_Experts)]
            L.moe_ffn_workspace_bytes.restype = sz
            L.moe_ffn_forward.argtypes = [vp, i32, i64, vp, vp, i32, ctypes.POINTER(_Experts), vp,
                                          i32, vp, sz, vp]
            L.moe_ffn_forward.restype = ctypes.c_int
            L.qmm_last_error.argtypes = []
            L.qmm_last_error.restype = ctypes.c_char_p
            L.qmm_launch_count.argtypes = []
            L.qmm_launch_count.restype = u64
            L.qmm_tc_timing.argtypes = [i32]
            L.qmm_tc_timing.restype = ctypes.c_int
            L.qmm_tc_timing_ms.argtypes = [ctypes.POINTER(ctypes.c_float),
                                           ctypes.POINTER(ctypes.c_float)]
            L.qmm_tc_timing_ms.restype = ctypes.c_int
            L.qmm_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
            L.qmm_device_status.restype = ctypes.c_int
            L.moe_route_topk_noalloc.argtypes = [vp, i32, i64, i64, vp, vp, i32, i32, vp, vp, vp,
                                                 vp]
            L.moe_route_topk_noalloc.restype = ctypes.c_int
            L.moe_route_load_stats.argtypes = [vp, i32, i64, vp, vp]
            L.moe_route_load_stats.restype = ctypes.c_int
            L.qmm_diag_wait_timeout.argtypes = [u64, vp]
            L.qmm_diag_wait_timeout.restype = ctypes.c_int
            L.qmm_linear_batched_workspace_bytes.argtypes = [i64, ctypes.POINTER(_Weight)]
            L.qmm_linear_batched_workspace_bytes.restype = sz
            L.qmm_linear_batched.argtypes = [vp, i32, i64, ctypes.POINTER(_Weight), vp, i32, vp,
                                             sz, vp]
            L.qmm_linear_batched.restype = ctypes.c_int
            L.moe_decode_workspace_bytes.argtypes = [i64, i32, ctypes.POINTER(_Experts)]
            L.moe_decode_workspace_bytes.restype = sz
            L.moe_decode_forward.argtypes = [vp, i32, i64, vp, vp, i32, ctypes.POINTER(_Experts),
                                             vp, i32, vp, vp, vp, vp, sz, vp]
            L.moe_decode_forward.restype = ctypes.c_int
            L.qmm_rope_table.argtypes = [i64, i32, ctypes.c_double, vp, vp, vp]
            L.qmm_rope_table.restype = ctypes.c_int
            L.qmm_attn_decode_workspace_bytes.argtypes = [ctypes.POINTER(_AttnLayer)]
            L.qmm_attn_decode_workspace_bytes.restype = sz
            L.qmm_attn_decode.argtypes = [vp, i32, i64, ctypes.POINTER(_AttnLayer), vp, vp, i32,
                                          vp, sz, vp]
            L.qmm_attn_decode.restype = ctypes.c_int
            _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != QMM_OK:
        raise QmmError(rc, lib().qmm_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)
    return t.data_ptr() if t.numel() else None


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return QMM_F32
    if t.dtype == torch.bfloat16:
        return QMM_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and isinstance(t, torch.Tensor) and t.numel() and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if t is not None and isinstance(t, torch.Tensor) and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _need(t, numel: int, dtypes, name: str) -> None:
    """A buffer the kernels read or write must hold exactly the elements they
    touch, of a matching type: the library sees only its address, so a short
    buffer would be overrun and a buffer of another type misread.  (A raw
    integer address is the caller's responsibility.)"""
    if t is None or not isinstance(t, torch.Tensor):
        return
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected "
                        + " or ".join(str(d) for d in dtypes))
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


@dataclass
class QWeight:
    """A quantised W[N, K] on the device: codes (int8 [N, K] or uint8
    [N, K/2]), scales fp32 [N, K/group], zps int32 [N, K/group]."""
    bits: int
    group: int
    N: int
    K: int
    codes: torch.Tensor
    scales: torch.Tensor
    zps: torch.Tensor

    def _c(self) -> _Weight:
        return _Weight(self.bits, self.group, self.N, self.K, _ptr(self.codes), _ptr(self.scales),
                       _ptr(self.zps))

    def rows(self, r0: int, r1: int) -> "QWeight":
        """Rows [r0, r1) as a QWeight sharing this one's storage."""
        return QWeight(self.bits, self.group, r1 - r0, self.K, self.codes[r0:r1],
                       self.scales[r0:r1], self.zps[r0:r1])


def alloc_qweight(N: int, K: int, bits: int, group: int, device="cuda") -> QWeight:
    """Uninitialised output buffers for qmm_quantize_groupwise."""
    G = K // group
    if bits == 8:
        codes = torch.empty((N, K), dtype=torch.int8, device=device)
    else:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
    return QWeight(bits, group, N, K, codes,
                   torch.empty((N, G), dtype=torch.float32, device=device),
                   torch.empty((N, G), dtype=torch.int32, device=device))


def _qweight_tensors(w: QWeight):
    return (w.codes, w.scales, w.zps)


def _qweight_sizes(w: QWeight, name: str = "w") -> None:
    """codes int8 or uint8 [N K bits / 8], scales fp32 and zps int32 [N K / group]
    (a descriptor the library rejects anyway is left to its own check)."""
    if w.bits in (4, 8) and w.group > 0 and w.K % w.group == 0:
        G = w.K // w.group
        _need(w.codes, w.N * w.K * w.bits // 8, (torch.int8, torch.uint8), f"{name}.codes")
        _need(w.scales, w.N * G, (torch.float32,), f"{name}.scales")
        _need(w.zps, w.N * G, (torch.int32,), f"{name}.zps")


def qmm_quantize_groupwise(w: torch.Tensor, bits: int, group: int, out: QWeight | None = None,
                           stream=None) -> QWeight:
    """Group-wise quantisation of fp32 w[N, K] (see include/qmm.h)."""
    if w.dtype != torch.float32 or w.dim() != 2:
        raise TypeError("w must be a 2-D float32 tensor")
    N, K = w.shape
    if out is not None:
        if (out.N, out.K, out.bits, out.group) != (N, K, bits, group):
            raise ValueError(f"out describes N={out.N} K={out.K} bits={out.bits} "
                             f"group={out.group}, the call N={N} K={K} bits={bits} group={group}")
        _qweight_sizes(out, "out")
    _require_cuda(w)
    if out is not None:
        _require_cuda(*_qweight_tensors(out))
    if out is None:
        out = alloc_qweight(N, K, bits, group, device=w.device)
    _check(lib().qmm_quantize_groupwise(_ptr(w), N, K, bits, group, _ptr(out.codes),
                                        _ptr(out.scales), _ptr(out.zps), _stream(stream)))
    return out


def qmm_linear(x: torch.Tensor, w: QWeight, y: torch.Tensor | None = None,
               y_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """y[M, N] = x[M, K] . deq(W)^T (fp32 or bf16 output: the dtype of y when
    given, else y_dtype)."""
    if x.dim() == 0 or x.shape[-1] != w.K:
        raise ValueError(f"x has shape {tuple(x.shape)}: its last dimension must be K = {w.K}")
    x2 = x.reshape(-1, w.K) if x.dim() != 2 else x
    M = x2.shape[0]
    # A weight is checked once; its descriptor is kept with the check, keyed by
    # the tensor objects and their addresses (this runs on every call, and a
    # decode-size launch is only a few microseconds of GPU time).
    c = w.__dict__.get("_desc_for")
    codes, scales, zps = w.codes, w.scales, w.zps
    shape = (w.bits, w.group, w.N, w.K)
    known = (c is not None and c[0] is codes and c[1] is scales and c[2] is zps
             and c[3] == codes.data_ptr() and c[4] == scales.data_ptr() and c[5] == zps.data_ptr()
             and c[7] == shape)
    if not known:
        _qweight_sizes(w)
    _need(y, M * w.N, (torch.float32, torch.bfloat16), "y")
    _require_cuda(x, y)
    if known:
        desc = c[6]
    else:
        _require_cuda(codes, scales, zps)
        desc = w._c()
        w.__dict__["_desc_for"] = (codes, scales, zps, codes.data_ptr(), scales.data_ptr(),
                                   zps.data_ptr(), desc, shape)
    if y is None:
        y = torch.empty((M, w.N), dtype=y_dtype, device=x.device)
    _check(lib().qmm_linear(_ptr(x2), _dtype_code(x2), M, ctypes.byref(desc), _ptr(y),
                            _dtype_code(y), _stream(stream)))
    return y


def qmm_linear_batched_workspace_bytes(M: int, w: QWeight) -> int:
    desc = w._c()
    return int(lib().qmm_linear_batched_workspace_bytes(M, ctypes.byref(desc)))


def qmm_linear_batched(x: torch.Tensor, w: QWeight, y: torch.Tensor | None = None,
                       y_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """qmm_linear for batches of rows: bf16 rows (M >= 9, INT8, group >= 64)
    run on the tensor cores (see include/qmm.h); everything else is
    qmm_linear."""
    if x.dim() == 0 or x.shape[-1] != w.K:
        raise ValueError(f"x has shape {tuple(x.shape)}: its last dimension must be K = {w.K}")
    x2 = x.reshape(-1, w.K) if x.dim() != 2 else x
    M = x2.shape[0]
    _qweight_sizes(w)
    _need(y, M * w.N, (torch.float32, torch.bfloat16), "y")
    _require_cuda(x, y, workspace, *_qweight_tensors(w))
    desc = w._c()
    if y is None:
        y = torch.empty((M, w.N), dtype=y_dtype, device=x.device)
    if workspace is None:  # a caller's workspace is size-checked by the library
        nbytes = int(lib().qmm_linear_batched_workspace_bytes(M, ctypes.byref(desc)))
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=x.device)
    _check(lib().qmm_linear_batched(_ptr(x2), _dtype_code(x2), M, ctypes.byref(desc), _ptr(y),
                                    _dtype_code(y), _ptr(workspace), _nbytes(workspace),
                                    _stream(stream)))
    return y


def moe_route_workspace_bytes(M: int, E: int) -> int:
    return int(lib().moe_route_workspace_bytes(M, E))


def _check_route(x, w_router, bias, k, topk_idx, topk_w, expert_counts):
    """x [M, H] fp32 or bf16, w_router fp32 [E, H], bias fp32 [E], outputs
    topk_idx int32 and topk_w fp32 [M, k], expert_counts int32 [E]."""
    if x.dim() != 2 or w_router.dim() != 2:
        raise ValueError("x must be [M, H] and w_router [E, H]")
    M, H = x.shape
    E = w_router.shape[0]
    _dtype_code(x)
    _need(w_router, E * H, (torch.float32,), "w_router")
    _need(bias, E, (torch.float32,), "bias")
    _need(topk_idx, M * k, (torch.int32,), "topk_idx")
    _need(topk_w, M * k, (torch.float32,), "topk_w")
    _need(expert_counts, E, (torch.int32,), "expert_counts")
    _require_cuda(x, w_router, bias, topk_idx, topk_w, expert_counts)
    return M, H, E


def moe_route_topk(x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor | None, k: int,
                   topk_idx=None, topk_w=None, expert_counts=None, workspace=None,
                   with_counts: bool = True, stream=None):
    """Router: fixed-order fp32 logits, top-k (lower index wins ties) and
    renormalised softmax weights.  Returns (topk_idx, topk_w, expert_counts)."""
    M, H, E = _check_route(x, w_router, bias, k, topk_idx, topk_w, expert_counts)
    _require_cuda(workspace)
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((M, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((M, k), dtype=torch.float32, device=dev)
    if expert_counts is None and with_counts:
        expert_counts = torch.empty((E,), dtype=torch.int32, device=dev)
    if workspace is None:  # a caller's workspace is size-checked by the library
        workspace = torch.empty((moe_route_workspace_bytes(M, E),), dtype=torch.uint8, device=dev)
    _check(lib().moe_route_topk(_ptr(x), _dtype_code(x), M, H, _ptr(w_router), _ptr(bias), E, k,
                                _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts),
                                _ptr(workspace), _nbytes(workspace), _stream(stream)))
    return topk_idx, topk_w, expert_counts


@dataclass
class MoeExperts:
    """E routed experts stacked along dim 0: gate/up codes [E, I, H*bits/8],
    down codes [E, H, I*bits/8]; scales / zps [E, rows, cols/group]."""
    E: int
    H: int
    I: int
    bits: int
    group: int
    gate_codes: torch.Tensor
    gate_scales: torch.Tensor
    gate_zps: torch.Tensor
    up_codes: torch.Tensor
    up_scales: torch.Tensor
    up_zps: torch.Tensor
    down_codes: torch.Tensor
    down_scales: torch.Tensor
    down_zps: torch.Tensor

    def _mat(self, which: str) -> _ExpertWeights:
        codes = getattr(self, f"{which}_codes")
        scales = getattr(self, f"{which}_scales")
        zps = getattr(self, f"{which}_zps")
        rows, cols = (self.I, self.H) if which in ("gate", "up") else (self.H, self.I)
        return _ExpertWeights(self.bits, self.group, rows, cols, _ptr(codes),
                              codes.stride(0) * codes.element_size(), _ptr(scales), _ptr(zps),
                              scales.stride(0))

    def _c(self) -> _Experts:
        return _Experts(self.E, self.H, self.I, self._mat("gate"), self._mat("up"),
                        self._mat("down"))


def alloc_experts(E: int, H: int, I: int, bits: int, group: int, device="cuda") -> MoeExperts:
    """Uninitialised stacked expert buffers (filled by quantising each expert)."""
    def mat(rows, cols):
        cb = cols if bits == 8 else cols // 2
        dt = torch.int8 if bits == 8 else torch.uint8
        return (torch.empty((E, rows, cb), dtype=dt, device=device),
                torch.empty((E, rows, cols // group), dtype=torch.float32, device=device),
                torch.empty((E, rows, cols // group), dtype=torch.int32, device=device))
    g, u, d = mat(I, H), mat(I, H), mat(H, I)
    return MoeExperts(E, H, I, bits, group, *g, *u, *d)


def _experts_tensors(ex: MoeExperts):
    return tuple(getattr(ex, f"{w}_{p}") for w in ("gate", "up", "down")
                 for p in ("codes", "scales", "zps"))


def _experts_sizes(ex: MoeExperts) -> None:
    """Stacked expert buffers: codes int8 or uint8 [E, rows, cols bits / 8],
    scales fp32 and zps int32 [E, rows, cols / group], rows x cols = I x H for
    gate and up, H x I for down (what the library's checks cannot see)."""
    if ex.bits not in (4, 8) or ex.group <= 0 or ex.H % ex.group or ex.I % ex.group:
        return
    for which in ("gate", "up", "down"):
        rows, cols = (ex.I, ex.H) if which != "down" else (ex.H, ex.I)
        _need(getattr(ex, f"{which}_codes"), ex.E * rows * cols * ex.bits // 8,
              (torch.int8, torch.uint8), f"{which}_codes")
        _need(getattr(ex, f"{which}_scales"), ex.E * rows * (cols // ex.group), (torch.float32,),
              f"{which}_scales")
        _need(getattr(ex, f"{which}_zps"), ex.E * rows * (cols // ex.group), (torch.int32,),
              f"{which}_zps")


def moe_ffn_workspace_bytes(M: int, k: int, experts: MoeExperts) -> int:
    desc = experts._c()
    return int(lib().moe_ffn_workspace_bytes(M, k, ctypes.byref(desc)))


def moe_ffn_forward(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                    experts: MoeExperts, y: torch.Tensor | None = None,
                    y_dtype: torch.dtype = torch.float32, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Routed SwiGLU MoE layer: y[m] = sum_i w[m,i] FFN_{idx[m,i]}(x[m])."""
    if x.dim() != 2 or x.shape[1] != experts.H or topk_idx.dim() != 2:
        raise ValueError(f"x must be [M, H = {experts.H}] and topk_idx [M, k]")
    M, H = x.shape
    k = topk_idx.shape[1]
    _dtype_code(x)
    _need(topk_idx, M * k, (torch.int32,), "topk_idx")
    _need(topk_w, M * k, (torch.float32,), "topk_w")
    _need(y, M * H, (torch.float32, torch.bfloat16), "y")
    # The experts are checked once and their descriptor kept, keyed by the
    # tensor objects, their addresses and the shape fields (building it costs
    # more host time than the rest of the call).
    ts = _experts_tensors(experts)
    shape = (experts.E, experts.H, experts.I, experts.bits, experts.group)
    c = experts.__dict__.get("_desc_for")
    known = (c is not None and c[2] == shape and all(map(operator.is_, c[0], ts))
             and c[1] == tuple(t.data_ptr() for t in ts))
    if not known:
        _experts_sizes(experts)
    _require_cuda(x, topk_idx, topk_w, y, workspace)
    if known:
        desc = c[3]
    else:
        _require_cuda(*ts)
        desc = experts._c()
        experts.__dict__["_desc_for"] = (ts, tuple(t.data_ptr() for t in ts), shape, desc)
    if y is None:
        y = torch.empty((M, H), dtype=y_dtype, device=x.device)
    if workspace is None:  # a caller's workspace is size-checked by the library
        nbytes = int(lib().moe_ffn_workspace_bytes(M, k, ctypes.byref(desc)))
        workspace = torch.empty((nbytes,), dtype=torch.uint8, device=x.device)
    _check(lib().moe_ffn_forward(_ptr(x), _dtype_code(x), M, _ptr(topk_idx), _ptr(topk_w), k,
                                 ctypes.byref(desc), _ptr(y), _dtype_code(y), _ptr(workspace),
                                 _nbytes(workspace), _stream(stream)))
    return y


def _experts_desc(experts: MoeExperts):
    """The experts' descriptor, checked once and kept (see moe_ffn_forward)."""
    ts = _experts_tensors(experts)
    shape = (experts.E, experts.H, experts.I, experts.bits, experts.group)
    c = experts.__dict__.get("_desc_for")
    if (c is not None and c[2] == shape and all(map(operator.is_, c[0], ts))
            and c[1] == tuple(t.data_ptr() for t in ts)):
        return c[3]
    _experts_sizes(experts)
    _require_cuda(*ts)
    desc = experts._c()
    experts.__dict__["_desc_for"] = (ts, tuple(t.data_ptr() for t in ts), shape, desc)
    return desc


def moe_decode_workspace_bytes(M: int, k: int, experts: MoeExperts) -> int:
    return int(lib().moe_decode_workspace_bytes(M, k, ctypes.byref(_experts_desc(experts))))


def moe_decode_forward(x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor | None, k: int,
                       experts: MoeExperts, y: torch.Tensor | None = None,
                       y_dtype: torch.dtype = torch.float32, topk_idx=None, topk_w=None,
                       expert_counts=None, workspace: torch.Tensor | None = None, stream=None):
    """The routed MoE layer of a decode batch (1..8 tokens) in one launch:
    router, top-k, grouping, experts and combine (see include/qmm.h).
    Returns y; topk_idx / topk_w / expert_counts are filled when given."""
    M, H, E = _check_route(x, w_router, bias, k, topk_idx, topk_w, expert_counts)
    if H != experts.H or E != experts.E:
        raise ValueError(f"router is [{E}, {H}], experts have E = {experts.E}, H = {experts.H}")
    _need(y, M * H, (torch.float32, torch.bfloat16), "y")
    _require_cuda(y, workspace)
    desc = _experts_desc(experts)
    if y is None:
        y = torch.empty((M, H), dtype=y_dtype, device=x.device)
    if workspace is None:  # a caller's workspace is size-checked by the library
        nbytes = int(lib().moe_decode_workspace_bytes(M, k, ctypes.byref(desc)))
        workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=x.device)
    _check(lib().moe_decode_forward(_ptr(x), _dtype_code(x), M, _ptr(w_router), _ptr(bias), k,
                                    ctypes.byref(desc), _ptr(y), _dtype_code(y), _ptr(topk_idx),
                                    _ptr(topk_w), _ptr(expert_counts), _ptr(workspace),
                                    _nbytes(workspace), _stream(stream)))
    return y


def moe_route_topk_noalloc(x: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor | None,
                           k: int, topk_idx=None, topk_w=None, expert_counts=None,
                           with_counts: bool = True, stream=None):
    """The router without a workspace, for callers that cannot allocate device
    memory: its logits scratch is a fixed 1 MiB array inside the library
    (M * E <= QMM_NOALLOC_MAX_LOGITS).  Outputs are allocated here only when
    the caller passes none.  Returns (topk_idx, topk_w, expert_counts)."""
    M, H, E = _check_route(x, w_router, bias, k, topk_idx, topk_w, expert_counts)
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((M, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((M, k), dtype=torch.float32, device=dev)
    if expert_counts is None and with_counts:
        expert_counts = torch.empty((E,), dtype=torch.int32, device=dev)
    _check(lib().moe_route_topk_noalloc(_ptr(x), _dtype_code(x), M, H, _ptr(w_router), _ptr(bias),
                                        E, k, _ptr(topk_idx), _ptr(topk_w), _ptr(expert_counts),
                                        _stream(stream)))
    return topk_idx, topk_w, expert_counts


def moe_route_load_stats(expert_counts: torch.Tensor, threshold: int, stats=None,
                         stream=None) -> torch.Tensor:
    """Load statistics of a routing histogram (int32 [E]): int64 [4] = largest
    count, its expert, experts touched, total; sets QMM_DEV_EXPERT_OVERLOAD in
    the device status word when the largest count exceeds `threshold`."""
    if expert_counts.dim() != 1:
        raise ValueError("expert_counts must be 1-D [E]")
    E = expert_counts.shape[0]
    _need(expert_counts, E, (torch.int32,), "expert_counts")
    _need(stats, 4, (torch.int64,), "stats")
    _require_cuda(expert_counts, stats)
    if stats is None:
        stats = torch.empty((4,), dtype=torch.int64, device=expert_counts.device)
    _check(lib().moe_route_load_stats(_ptr(expert_counts), E, int(threshold), _ptr(stats),
                                      _stream(stream)))
    return stats


def qmm_diag_wait_timeout(limit_ns: int, stream=None) -> None:
    """Runs the bounded-wait diagnostic kernel (see include/qmm.h)."""
    _check(lib().qmm_diag_wait_timeout(int(limit_ns), _stream(stream)))


def qmm_last_error() -> str:
    return lib().qmm_last_error().decode(errors="replace")


def qmm_launch_count() -> int:
    return int(lib().qmm_launch_count())


def qmm_tc_timing(enable: bool) -> None:
    """Switch the timing of the tensor-core prefill GEMM launches on or off
    (see include/qmm.h)."""
    _check(lib().qmm_tc_timing(1 if enable else 0))


def qmm_tc_timing_ms() -> tuple[float, float]:
    """(gate/up ms, down ms) of the last tensor-core moe_ffn_forward since
    timing was switched on; waits for that call's events."""
    g, d = ctypes.c_float(), ctypes.c_float()
    _check(lib().qmm_tc_timing_ms(ctypes.byref(g), ctypes.byref(d)))
    return float(g.value), float(d.value)


def qmm_device_status(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().qmm_device_status(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def quantize_experts(E: int, H: int, I: int, bits: int, group: int, rows_fn, device="cuda",
                     stream=None) -> MoeExperts:
    """Quantises the fp32 matrices of E experts into stacked device buffers.

    ``rows_fn(which, e, out)`` fills ``out`` (a float32 numpy array of shape
    [I, H] for "gate"/"up", [H, I] for "down") with expert e's weights.  Each
    matrix is staged through pinned host memory to the device and quantised
    there by qmm_quantize_groupwise, so no fp32 copy of the experts stays
    resident."""
    ex = alloc_experts(E, H, I, bits, group, device=device)
    n = I * H
    pinned = [torch.empty((n,), dtype=torch.float32).pin_memory() for _ in range(2)]
    staging = [torch.empty((n,), dtype=torch.float32, device=device) for _ in range(2)]
    s = torch.cuda.current_stream(device) if stream is None else stream
    events = [None, None]
    j = 0
    for e in range(E):
        for which in ("gate", "up", "down"):
            rows, cols = (I, H) if which in ("gate", "up") else (H, I)
            b = j % 2
            if events[b] is not None:
                events[b].synchronize()  # the previous copy out of this pinned buffer is done
            host = pinned[b].numpy().reshape(rows, cols)
            rows_fn(which, e, host)
            with torch.cuda.stream(s):
                staging[b].copy_(pinned[b], non_blocking=True)
                out = QWeight(bits, group, rows, cols, getattr(ex, f"{which}_codes")[e],
                              getattr(ex, f"{which}_scales")[e], getattr(ex, f"{which}_zps")[e])
                qmm_quantize_groupwise(staging[b].view(rows, cols), bits, group, out=out, stream=s)
                ev = torch.cuda.Event()
                ev.record(s)
                events[b] = ev
            j += 1
    torch.cuda.synchronize(device)
    return ex


# ------------------------------------------------------------ decode attention

def rope_table(max_seq: int, head_dim: int, base: float = 10000.0, device="cuda", stream=None):
    """cos, sin fp32 [max_seq, head_dim / 2] of pos * base^(-2i / head_dim)
    (see include/qmm.h)."""
    hp = head_dim // 2
    c = torch.empty((max_seq, hp), dtype=torch.float32, device=device)
    s = torch.empty((max_seq, hp), dtype=torch.float32, device=device)
    _check(lib().qmm_rope_table(max_seq, head_dim, float(base), _ptr(c), _ptr(s),
                                _stream(stream)))
    return c, s


@dataclass
class AttnLayer:
    """One attention layer for decoding: quantised projections and the RoPE
    table (device tensors), shapes as in include/qmm.h."""
    n_head: int
    n_head_kv: int
    head_dim: int
    max_seq: int
    wq: QWeight
    wk: QWeight
    wv: QWeight
    wo: QWeight
    rope_cos: torch.Tensor
    rope_sin: torch.Tensor

    def _c(self) -> _AttnLayer:
        return _AttnLayer(self.n_head, self.n_head_kv, self.head_dim, self.max_seq,
                          self.wq._c(), self.wk._c(), self.wv._c(), self.wo._c(),
                          _ptr(self.rope_cos), _ptr(self.rope_sin))

    def kv_cache(self, device="cuda") -> torch.Tensor:
        """A zeroed cache [2, n_head_kv, max_seq, head_dim] fp32."""
        return torch.zeros((2, self.n_head_kv, self.max_seq, self.head_dim),
                           dtype=torch.float32, device=device)


def quantize_attn_layer(wq: torch.Tensor, wk: torch.Tensor, wv: torch.Tensor, wo: torch.Tensor,
                        n_head: int, n_head_kv: int, head_dim: int, max_seq: int, bits: int = 8,
                        group: int = 64, base: float = 10000.0, stream=None) -> AttnLayer:
    """An AttnLayer from fp32 weights: wq, wk, wv quantised as one stacked
    matrix (so that the decode step runs the three projections as one
    launch), wo on its own, and the RoPE table."""
    nq, nk = wq.shape[0], wk.shape[0]
    qkv = qmm_quantize_groupwise(torch.cat([wq, wk, wv], dim=0).contiguous(), bits, group,
                                 stream=stream)
    c, s = rope_table(max_seq, head_dim, base, device=wq.device, stream=stream)
    return AttnLayer(n_head, n_head_kv, head_dim, max_seq, qkv.rows(0, nq),
                     qkv.rows(nq, nq + nk), qkv.rows(nq + nk, nq + 2 * nk),
                     qmm_quantize_groupwise(wo, bits, group, stream=stream), c, s)


def qmm_attn_decode_workspace_bytes(layer: AttnLayer) -> int:
    return int(lib().qmm_attn_decode_workspace_bytes(ctypes.byref(layer._c())))


def attn_decode(x: torch.Tensor, pos: int, layer: AttnLayer, kv_cache: torch.Tensor,
                y: torch.Tensor | None = None, y_dtype: torch.dtype = torch.float32,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One decode step of the attention layer for the token x [D] at position
    pos: writes row pos of kv_cache and returns y [D_out] (see include/qmm.h)."""
    D = layer.wq.K
    if x.numel() != D:
        raise ValueError(f"x has {x.numel()} elements, expected D = {D}")
    _dtype_code(x)
    for name in ("wq", "wk", "wv", "wo"):
        _qweight_sizes(getattr(layer, name), name)
    hp = layer.head_dim // 2
    _need(layer.rope_cos, layer.max_seq * hp, (torch.float32,), "rope_cos")
    _need(layer.rope_sin, layer.max_seq * hp, (torch.float32,), "rope_sin")
    _need(kv_cache, 2 * layer.n_head_kv * layer.max_seq * layer.head_dim, (torch.float32,),
          "kv_cache")
    _need(y, layer.wo.N, (torch.float32, torch.bfloat16), "y")
    ts = [t for w in (layer.wq, layer.wk, layer.wv, layer.wo) for t in _qweight_tensors(w)]
    _require_cuda(x, kv_cache, y, workspace, layer.rope_cos, layer.rope_sin, *ts)
    desc = layer._c()
    if y is None:
        y = torch.empty((layer.wo.N,), dtype=y_dtype, device=x.device)
    if workspace is None:  # a caller's workspace is size-checked by the library
        nbytes = int(lib().qmm_attn_decode_workspace_bytes(ctypes.byref(desc)))
        workspace = torch.empty((max(nbytes, 1),), dtype=torch.uint8, device=x.device)
    _check(lib().qmm_attn_decode(_ptr(x), _dtype_code(x), pos, ctypes.byref(desc), _ptr(kv_cache),
                                 _ptr(y), _dtype_code(y), _ptr(workspace), _nbytes(workspace),
                                 _stream(stream)))
    return y
