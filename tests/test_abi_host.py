"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/qmm.h declares, and rejects bad arguments with the
documented status codes before touching the device."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import group_quantized_moe_gb300 as q
from group_quantized_moe_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")

# Fake, 256-byte aligned addresses: every call below must fail validation on
# the host, so these are never dereferenced.  As a second line of defence the
# fake-pointer tests run only where no CUDA device is visible: a case that
# wrongly passed validation must never reach a kernel launch on a real GPU.
P = 0x7F0000000000
P2 = P + 0x100000


def _gpu_visible() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return q.lib()


@pytest.fixture
def Lfake(L):
    if _gpu_visible():
        pytest.skip("fake device pointers are only passed where no GPU is visible")
    return L


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_entry_points_exported(L):
    names = _declared_functions()
    for n in ("qmm_quantize_groupwise", "qmm_linear", "moe_route_topk", "moe_ffn_forward"):
        assert n in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in qmm.h but not exported"
    assert set(names) == set(q.EXPORTED)


def test_launch_count_starts_readable(L):
    assert q.qmm_launch_count() >= 0


def _w(bits=8, group=64, N=128, K=256, codes=P, scales=P, zps=P):
    return q._Weight(bits, group, N, K, codes, scales, zps)


@pytest.mark.parametrize("kw,code", [
    (dict(bits=5), q.QMM_ERR_INVALID_ARG),
    (dict(group=48), q.QMM_ERR_UNSUPPORTED),
    (dict(group=16), q.QMM_ERR_UNSUPPORTED),
    (dict(K=200), q.QMM_ERR_SHAPE),
    (dict(K=0), q.QMM_ERR_SHAPE),
    (dict(N=-1), q.QMM_ERR_SHAPE),
    (dict(codes=None), q.QMM_ERR_INVALID_ARG),
    (dict(scales=P + 4), q.QMM_ERR_ALIGN),
    (dict(codes=P + 8), q.QMM_ERR_ALIGN),
    (dict(K=32768, group=256), q.QMM_ERR_UNSUPPORTED),
])
def test_linear_rejects(Lfake, kw, code):
    L = Lfake
    w = _w(**kw)
    rc = L.qmm_linear(P2, q.QMM_F32, 1, ctypes.byref(w), P2, q.QMM_F32, None)
    assert rc == code, q.qmm_last_error()
    assert q.qmm_last_error()


def test_linear_rejects_bad_dtype_and_x(Lfake):
    L = Lfake
    w = _w()
    assert L.qmm_linear(P2, 7, 1, ctypes.byref(w), P2, q.QMM_F32, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_linear(P2 + 4, q.QMM_F32, 1, ctypes.byref(w), P2, q.QMM_F32, None) == q.QMM_ERR_ALIGN
    assert L.qmm_linear(None, q.QMM_F32, 1, ctypes.byref(w), P2, q.QMM_F32, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_linear(P2, q.QMM_F32, 1, None, P2, q.QMM_F32, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_linear(P2, q.QMM_F32, -1, ctypes.byref(w), P2, q.QMM_F32, None) == q.QMM_ERR_SHAPE


def test_linear_empty_is_noop(Lfake):
    L = Lfake
    w = _w()
    assert L.qmm_linear(None, q.QMM_F32, 0, ctypes.byref(w), None, q.QMM_F32, None) == q.QMM_OK
    w0 = _w(N=0)
    assert L.qmm_linear(None, q.QMM_F32, 3, ctypes.byref(w0), None, q.QMM_F32, None) == q.QMM_OK


def test_quantize_rejects(Lfake):
    L = Lfake
    f = L.qmm_quantize_groupwise
    assert f(P, 4, 256, 3, 64, P, P, P, None) == q.QMM_ERR_INVALID_ARG
    assert f(P, 4, 250, 8, 64, P, P, P, None) == q.QMM_ERR_SHAPE
    assert f(P, 4, 256, 8, 96, P, P, P, None) == q.QMM_ERR_UNSUPPORTED
    assert f(None, 4, 256, 8, 64, P, P, P, None) == q.QMM_ERR_INVALID_ARG
    assert f(P + 4, 4, 256, 8, 64, P, P, P, None) == q.QMM_ERR_ALIGN
    assert f(P, 4, 256, 4, 64, P, P + 8, P, None) == q.QMM_ERR_ALIGN
    assert f(None, 0, 256, 8, 64, None, None, None, None) == q.QMM_OK  # N = 0: no-op


def test_router_rejects(Lfake):
    L = Lfake
    f = L.moe_route_topk
    ws = q.moe_route_workspace_bytes(8, 256)
    assert ws >= 8 * 256 * 4 and ws % 256 == 0
    ok = (P, q.QMM_F32, 8, 4096, P, None, 256, 6, P2, P2, None, P2, ws, None)

    def call(**kw):
        a = list(ok)
        names = ["x", "dt", "M", "H", "wr", "bias", "E", "k", "idx", "w", "cnt", "ws", "wsb", "s"]
        for k_, v in kw.items():
            a[names.index(k_)] = v
        return f(*a)

    assert call(k=7, E=6) == q.QMM_ERR_INVALID_ARG
    assert call(k=0) == q.QMM_ERR_INVALID_ARG
    assert call(k=17) == q.QMM_ERR_INVALID_ARG
    assert call(E=1025) == q.QMM_ERR_INVALID_ARG
    assert call(H=4094) == q.QMM_ERR_SHAPE
    assert call(dt=3) == q.QMM_ERR_INVALID_ARG
    assert call(x=None) == q.QMM_ERR_INVALID_ARG
    assert call(x=P + 8) == q.QMM_ERR_ALIGN
    assert call(wsb=ws - 1) == q.QMM_ERR_WORKSPACE
    assert call(ws=None) == q.QMM_ERR_WORKSPACE
    assert call(ws=P2 + 16) == q.QMM_ERR_ALIGN
    assert call(M=0, x=None, idx=None, w=None) == q.QMM_OK
    # sizes whose workspace or grid would not fit are refused before any
    # product of them is formed
    assert call(M=1 << 31) == q.QMM_ERR_UNSUPPORTED
    assert call(M=(1 << 62) + 1) == q.QMM_ERR_UNSUPPORTED
    assert call(H=(1 << 24) + 4) == q.QMM_ERR_UNSUPPORTED
    assert q.moe_route_workspace_bytes(1 << 31, 256) == 2 ** 64 - 1
    assert q.moe_route_workspace_bytes((1 << 62) + 1, 256) == 2 ** 64 - 1


def test_noalloc_router_rejects(Lfake):
    """The allocation-free router checks the built-in scratch size before it
    touches the device: M * E beyond it, including an M whose product with E
    would wrap around 64 bits, is refused."""
    L = Lfake
    f = L.moe_route_topk_noalloc
    lim = q.QMM_NOALLOC_MAX_LOGITS
    assert f(P, q.QMM_F32, lim // 256 + 1, 4096, P, None, 256, 6, P2, P2, None, None) == \
        q.QMM_ERR_WORKSPACE
    assert f(P, q.QMM_F32, (1 << 62) + 1, 4096, P, None, 256, 6, P2, P2, None, None) == \
        q.QMM_ERR_WORKSPACE
    assert f(P, q.QMM_F32, 2, 4096, P, None, 256, 17, P2, P2, None, None) == q.QMM_ERR_INVALID_ARG
    assert f(P, q.QMM_F32, 2, 4094, P, None, 256, 6, P2, P2, None, None) == q.QMM_ERR_SHAPE
    assert f(P + 8, q.QMM_F32, 2, 4096, P, None, 256, 6, P2, P2, None, None) == q.QMM_ERR_ALIGN


def _experts(E=8, H=256, I=256, bits=4, group=64, **over):
    def mat(nrows, ncols, **o):
        rows, cols = nrows, ncols
        d = dict(bits=bits, group=group, rows=rows, cols=cols, codes=P,
                 codes_stride=rows * cols * bits // 8, scales=P, zps=P,
                 groups_stride=rows * cols // group)
        d.update(o)
        return q._ExpertWeights(d["bits"], d["group"], d["rows"], d["cols"], d["codes"],
                                d["codes_stride"], d["scales"], d["zps"], d["groups_stride"])
    g = mat(I, H, **over.get("gate", {}))
    u = mat(I, H, **over.get("up", {}))
    dn = mat(H, I, **over.get("down", {}))
    return q._Experts(over.get("E", E), H, I, g, u, dn)


def test_moe_workspace_bytes(L):
    ex = _experts()
    a = L.moe_ffn_workspace_bytes(8, 6, ctypes.byref(ex))
    b = L.moe_ffn_workspace_bytes(16, 6, ctypes.byref(ex))
    assert a > 0 and b > a and a % 256 == 0
    # holds at least the per-assignment activations and outputs
    assert a >= 8 * 6 * (256 + 256) * 4


@pytest.mark.parametrize("over,code", [
    (dict(E=0), q.QMM_ERR_INVALID_ARG),
    (dict(gate=dict(rows=64)), q.QMM_ERR_SHAPE),
    (dict(gate=dict(cols=128), up=dict(cols=128), down=dict(rows=128)), q.QMM_ERR_SHAPE),
    (dict(down=dict(cols=512)), q.QMM_ERR_SHAPE),
    (dict(up=dict(bits=8)), q.QMM_ERR_UNSUPPORTED),
    (dict(down=dict(group=128)), q.QMM_ERR_UNSUPPORTED),
    (dict(gate=dict(codes=None)), q.QMM_ERR_INVALID_ARG),
    (dict(gate=dict(codes_stride=8)), q.QMM_ERR_ALIGN),
    (dict(up=dict(scales=P + 4)), q.QMM_ERR_ALIGN),
])
def test_moe_rejects_experts(Lfake, over, code):
    L = Lfake
    ex = _experts(**over)
    ws = 1 << 30
    rc = L.moe_ffn_forward(P, q.QMM_F32, 8, P, P, 6, ctypes.byref(ex), P2, q.QMM_F32, P2, ws, None)
    assert rc == code, q.qmm_last_error()


def test_moe_rejects_args(Lfake):
    L = Lfake
    ex = _experts()
    need = L.moe_ffn_workspace_bytes(8, 6, ctypes.byref(ex))
    f = L.moe_ffn_forward
    assert f(P, q.QMM_F32, 8, P, P, 6, ctypes.byref(ex), P2, q.QMM_F32, P2, need - 1, None) == q.QMM_ERR_WORKSPACE
    assert f(P, q.QMM_F32, 8, P, P, 6, ctypes.byref(ex), P2, q.QMM_F32, P2 + 128, need, None) == q.QMM_ERR_ALIGN
    assert f(P, q.QMM_F32, 8, P, P, 9, ctypes.byref(ex), P2, q.QMM_F32, P2, need, None) == q.QMM_ERR_INVALID_ARG
    assert f(P, 5, 8, P, P, 6, ctypes.byref(ex), P2, q.QMM_F32, P2, need, None) == q.QMM_ERR_INVALID_ARG
    assert f(P, q.QMM_F32, 8, P, P, 6, ctypes.byref(ex), P2, 9, P2, need, None) == q.QMM_ERR_INVALID_ARG
    assert f(None, q.QMM_F32, 8, P, P, 6, ctypes.byref(ex), P2, q.QMM_F32, P2, need, None) == q.QMM_ERR_INVALID_ARG
    assert f(P + 4, q.QMM_F32, 8, P, P, 6, ctypes.byref(ex), P2, q.QMM_F32, P2, need, None) == q.QMM_ERR_ALIGN
    assert f(None, q.QMM_F32, 0, None, None, 6, ctypes.byref(ex), None, q.QMM_F32, None, 0, None) == q.QMM_OK
    assert f(P, q.QMM_F32, 8, P, P, 6, None, P2, q.QMM_F32, P2, need, None) == q.QMM_ERR_INVALID_ARG
    # groups per row not a multiple of 4
    odd = _experts(H=256, I=128, bits=4, group=64)
    assert f(P, q.QMM_F32, 8, P, P, 6, ctypes.byref(odd), P2, q.QMM_F32, P2, 1 << 40, None) == q.QMM_ERR_UNSUPPORTED
    # rows longer than one copy slot holds
    big = _experts(H=8192, I=512, bits=8, group=128)
    assert f(P, q.QMM_F32, 8, P, P, 6, ctypes.byref(big), P2, q.QMM_F32, P2, 1 << 40, None) == q.QMM_ERR_UNSUPPORTED


def test_decode_one_launch_rejects(Lfake):
    """moe_decode_forward: argument errors, and shapes it does not take, return
    before anything is enqueued."""
    f = Lfake.moe_decode_forward
    ex = _experts(E=16, H=4096, I=2048, bits=4, group=64)
    need = Lfake.moe_decode_workspace_bytes(8, 6, ctypes.byref(ex))
    assert need > 0 and Lfake.moe_decode_workspace_bytes(9, 6, ctypes.byref(ex)) == 0

    def call(x=P, dt=q.QMM_F32, M=8, wr=P, k=6, e=ex, y=P2, ydt=q.QMM_F32, ws=P2 + (1 << 30),
             wsb=need):
        return f(x, dt, M, wr, None, k, ctypes.byref(e), y, ydt, None, None, None, ws, wsb, None)

    assert call(M=0) == q.QMM_OK  # a no-op
    assert call(M=9) == q.QMM_ERR_UNSUPPORTED
    assert call(k=0) == q.QMM_ERR_INVALID_ARG
    assert call(k=17) == q.QMM_ERR_INVALID_ARG
    assert call(dt=4) == q.QMM_ERR_INVALID_ARG
    assert call(ydt=4) == q.QMM_ERR_INVALID_ARG
    assert call(x=None) == q.QMM_ERR_INVALID_ARG
    assert call(wr=None) == q.QMM_ERR_INVALID_ARG
    assert call(x=P + 4) == q.QMM_ERR_ALIGN
    assert call(wsb=need - 1) == q.QMM_ERR_WORKSPACE
    assert call(ws=P2 + 16) == q.QMM_ERR_ALIGN
    # shapes outside the one-launch form: another width, more than 256 experts
    assert call(e=_experts(E=16, H=2048, I=2048, bits=4, group=64)) == q.QMM_ERR_UNSUPPORTED
    big = _experts(E=512, H=4096, I=2048, bits=4, group=64)
    assert call(e=big, wsb=1 << 40) == q.QMM_ERR_UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """No silent fallback: a missing library is an error, not a CPU path."""
    import importlib
    monkeypatch.setattr(q, "LIB_PATH", str(tmp_path / "libqmm.so"))
    monkeypatch.setattr(q, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        q.lib()
    monkeypatch.undo()
    importlib.reload(q)


def test_header_is_plain_c_and_a_c_program_links(tmp_path, L):
    """The boundary is a C ABI: include/qmm.h compiles as C99 with warnings as
    errors, and a C program linked against libqmm.so calls the entry points
    that need no GPU (no launch happens: M = 0 is a no-op by contract)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    src = tmp_path / "use_qmm.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "qmm.h"
int main(void) {
  qmm_weight w;
  memset(&w, 0, sizeof w);
  w.bits = 8; w.group = 64; w.N = 128; w.K = 256;
  if (qmm_linear(NULL, QMM_F32, 0, &w, NULL, QMM_F32, NULL) != QMM_OK) return 1;
  if (qmm_linear(NULL, 7, 1, &w, NULL, QMM_F32, NULL) != QMM_ERR_INVALID_ARG) return 2;
  if (strlen(qmm_last_error()) == 0) return 3;
  if (moe_route_workspace_bytes(8, 256) < (size_t)8 * 256 * 4) return 4;
  printf("ok %llu\n", (unsigned long long)qmm_launch_count());
  return 0;
}
''')
    exe = tmp_path / "use_qmm"
    libdir = os.path.dirname(build_lib.LIB)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-lqmm", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.returncode, r.stdout, r.stderr)


# ------------------------------------------------------------ decode attention

def _attn(L, n_head=4, n_kv=2, hd=32, max_seq=16, D=128, **over):
    # the structure types the loaded library was declared with (an earlier
    # test reloads the binding module, which makes new classes)
    AL = L.qmm_attn_decode_workspace_bytes.argtypes[0]._type_
    W = dict(AL._fields_)["wq"]

    def w(N, K):
        return W(8, 64, N, K, P, P, P)

    layer = AL(n_head, n_kv, hd, max_seq, w(n_head * hd, D), w(n_kv * hd, D), w(n_kv * hd, D),
               w(D, n_head * hd), P, P)
    for k, v in over.items():
        if k in ("wq", "wk", "wv", "wo"):
            v = w(*v)
        setattr(layer, k, v)
    return layer


def test_rope_table_rejects(Lfake):
    f = Lfake.qmm_rope_table
    assert f(0, 64, 10000.0, P, P2, None) == q.QMM_ERR_INVALID_ARG
    assert f(16, 63, 10000.0, P, P2, None) == q.QMM_ERR_INVALID_ARG
    assert f(16, 64, 0.0, P, P2, None) == q.QMM_ERR_INVALID_ARG
    assert f(16, 64, -1.0, P, P2, None) == q.QMM_ERR_INVALID_ARG
    assert f(16, 64, 10000.0, None, P2, None) == q.QMM_ERR_INVALID_ARG
    assert f(16, 64, 10000.0, P + 2, P2, None) == q.QMM_ERR_ALIGN


def test_attn_workspace_bytes(L):
    f = L.qmm_attn_decode_workspace_bytes
    assert f(None) == 0
    assert f(ctypes.byref(_attn(L, head_dim=3))) == 0
    assert f(ctypes.byref(_attn(L, max_seq=0))) == 0
    # q, k, v, output rows, and n_head x ceil(max_seq / 64) x (head_dim + 2) partials
    small = f(ctypes.byref(_attn(L, max_seq=64)))
    more = f(ctypes.byref(_attn(L, max_seq=65)))
    assert small > 0 and more - small == ((4 * 2 * 34 * 4 + 255) // 256 * 256
                                          - (4 * 1 * 34 * 4 + 255) // 256 * 256)


def test_attn_decode_rejects(Lfake):
    ws = Lfake.qmm_attn_decode_workspace_bytes(ctypes.byref(_attn(Lfake)))

    def call(layer=None, pos=3, dt=q.QMM_F32, ydt=q.QMM_F32, x=P, cache=P, y=P, w=P2, wsb=ws):
        layer = _attn(Lfake) if layer is None else layer
        return Lfake.qmm_attn_decode(x, dt, pos, ctypes.byref(layer), cache, y, ydt, w, wsb, None)

    assert call(pos=16) == q.QMM_ERR_INVALID_ARG
    assert call(pos=-1) == q.QMM_ERR_INVALID_ARG
    assert call(layer=_attn(Lfake, n_head=3)) == q.QMM_ERR_INVALID_ARG
    assert call(layer=_attn(Lfake, n_kv=0)) == q.QMM_ERR_INVALID_ARG
    assert call(layer=_attn(Lfake, hd=6)) == q.QMM_ERR_UNSUPPORTED
    assert call(layer=_attn(Lfake, hd=1024)) == q.QMM_ERR_UNSUPPORTED
    assert call(layer=_attn(Lfake, wk=(3 * 32, 128))) == q.QMM_ERR_SHAPE
    assert call(layer=_attn(Lfake, wo=(128, 64))) == q.QMM_ERR_SHAPE
    assert call(layer=_attn(Lfake, rope_cos=None)) == q.QMM_ERR_INVALID_ARG
    assert call(dt=2) == q.QMM_ERR_INVALID_ARG
    assert call(ydt=5) == q.QMM_ERR_INVALID_ARG
    assert call(x=None) == q.QMM_ERR_INVALID_ARG
    assert call(cache=P + 4) == q.QMM_ERR_ALIGN
    assert call(wsb=ws - 1) == q.QMM_ERR_WORKSPACE
    assert call(w=None) == q.QMM_ERR_WORKSPACE
    assert call(w=P2 + 16) == q.QMM_ERR_ALIGN
