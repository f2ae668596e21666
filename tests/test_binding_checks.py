"""The Python binding's buffer checks, on the CPU.

The C ABI sees only addresses, so the binding checks every buffer a kernel
will touch (element count and type) before the device check and before any
library call.  Host tensors therefore reach the device check only when their
shapes and types are right: the call patterns the GPU tests, the benchmark
and the smoke check use must get that far, and each unsafe variant (a short
output, indices of another integer type, a weight of the wrong size) must be
stopped by its own check first.
"""
import pytest
import torch

import group_quantized_moe_gb300 as q

DEVICE_MSG = "CUDA device"


def _qw(N=64, K=256, bits=8, group=64):
    return q.alloc_qweight(N, K, bits, group, device="cpu")


def _reaches_device_check(fn, *a, **kw):
    with pytest.raises(ValueError, match=DEVICE_MSG):
        fn(*a, **kw)


def test_linear_accepts_the_used_shapes():
    w = _qw()
    for x in (torch.zeros(256), torch.zeros(1, 256), torch.zeros(5, 256),
              torch.zeros(3, 256, dtype=torch.bfloat16)):
        _reaches_device_check(q.qmm_linear, x, w)
    _reaches_device_check(q.qmm_linear, torch.zeros(3, 256), w, y=torch.zeros(3, 64))
    _reaches_device_check(q.qmm_linear, torch.zeros(1, 4096), _qw(128, 4096, 4, 128),
                          y=torch.zeros(1, 128))


@pytest.mark.parametrize("bad", ["y_short", "y_dtype", "x_cols", "codes", "scales", "zps_dtype"])
def test_linear_rejects(bad):
    w, x, y = _qw(), torch.zeros(3, 256), torch.zeros(3, 64)
    exc = ValueError
    if bad == "y_short":
        y = torch.zeros(3, 63)
    elif bad == "y_dtype":
        y, exc = torch.zeros(3, 64, dtype=torch.float16), TypeError
    elif bad == "x_cols":
        x = torch.zeros(3, 257)
    elif bad == "codes":
        w.codes = torch.zeros(64, 128, dtype=torch.int8)
    elif bad == "scales":
        w.scales = torch.zeros(64, 3)
    else:
        w.zps, exc = torch.zeros(64, 4, dtype=torch.int64), TypeError
    with pytest.raises(exc) as e:
        q.qmm_linear(x, w, y=y)
    assert DEVICE_MSG not in str(e.value)


def test_quantize_out_must_match_the_call():
    w = torch.zeros(64, 256)
    _reaches_device_check(q.qmm_quantize_groupwise, w, 8, 64)
    _reaches_device_check(q.qmm_quantize_groupwise, w, 8, 64, out=_qw())
    for out in (_qw(N=32), _qw(bits=4), _qw(group=128)):
        with pytest.raises(ValueError, match="out describes"):
            q.qmm_quantize_groupwise(w, 8, 64, out=out)


def test_router_accepts_the_used_shapes():
    M, E, H, k = 8, 16, 512, 4
    x, wr = torch.zeros(M, H), torch.zeros(E, H)
    _reaches_device_check(q.moe_route_topk, x, wr, None, k)
    _reaches_device_check(q.moe_route_topk, x.bfloat16(), wr, torch.zeros(E), k,
                          topk_idx=torch.zeros(M, k, dtype=torch.int32), topk_w=torch.zeros(M, k),
                          expert_counts=torch.zeros(E, dtype=torch.int32))
    _reaches_device_check(q.moe_route_topk_noalloc, x, wr, None, k)


@pytest.mark.parametrize("bad", ["wr_dtype", "wr_cols", "bias", "idx_dtype", "w_short", "counts"])
def test_router_rejects(bad):
    M, E, H, k = 8, 16, 512, 4
    a = dict(x=torch.zeros(M, H), w_router=torch.zeros(E, H), bias=None, k=k)
    exc = ValueError
    if bad == "wr_dtype":
        a["w_router"], exc = torch.zeros(E, H, dtype=torch.float64), TypeError
    elif bad == "wr_cols":
        a["w_router"] = torch.zeros(E, H - 4)
    elif bad == "bias":
        a["bias"] = torch.zeros(E + 1)
    elif bad == "idx_dtype":
        a["topk_idx"], exc = torch.zeros(M, k, dtype=torch.int64), TypeError
    elif bad == "w_short":
        a["topk_w"] = torch.zeros(M, k - 1)
    else:
        a["expert_counts"] = torch.zeros(E - 1, dtype=torch.int32)
    for fn in (q.moe_route_topk, q.moe_route_topk_noalloc):
        with pytest.raises(exc) as e:
            fn(**a)
        assert DEVICE_MSG not in str(e.value)


def _experts():
    return q.alloc_experts(4, 256, 128, 4, 64, device="cpu")


def test_moe_accepts_the_used_shapes():
    ex, M, k = _experts(), 5, 2
    idx, w = torch.zeros(M, k, dtype=torch.int32), torch.zeros(M, k)
    for x, y in ((torch.zeros(M, 256), None), (torch.zeros(M, 256), torch.zeros(M, 256)),
                 (torch.zeros(M, 256, dtype=torch.bfloat16), torch.zeros(M, 256, dtype=torch.bfloat16))):
        _reaches_device_check(q.moe_ffn_forward, x, idx, w, ex, y=y)


@pytest.mark.parametrize("bad", ["idx_dtype", "idx_short", "w_dtype", "y_short", "x_cols",
                                 "down_codes", "gate_scales"])
def test_moe_rejects(bad):
    ex, M, k = _experts(), 5, 2
    x, idx, w, y = torch.zeros(M, 256), torch.zeros(M, k, dtype=torch.int32), torch.zeros(M, k), None
    exc = ValueError
    if bad == "idx_dtype":
        idx, exc = torch.zeros(M, k, dtype=torch.int64), TypeError
    elif bad == "idx_short":
        w = torch.zeros(M - 1, k)
    elif bad == "w_dtype":
        w, exc = torch.zeros(M, k, dtype=torch.float64), TypeError
    elif bad == "y_short":
        y = torch.zeros(M, 255)
    elif bad == "x_cols":
        x = torch.zeros(M, 512)
    elif bad == "down_codes":
        ex.down_codes = torch.zeros(4, 256, 32, dtype=torch.uint8)
    else:
        ex.gate_scales = torch.zeros(4, 128, 3)
    with pytest.raises(exc) as e:
        q.moe_ffn_forward(x, idx, w, ex, y=y)
    assert DEVICE_MSG not in str(e.value)


def test_linear_weight_check_is_cached_and_invalidated(monkeypatch):
    """A weight is checked once and its descriptor kept; swapping one of its
    tensors or changing its shape fields runs the check again (the library
    and the device check are stubbed: this is the binding's own logic)."""
    calls = []

    class FakeLib:
        def qmm_linear(self, *a):
            calls.append(a)
            return q.QMM_OK

    fake = FakeLib()
    monkeypatch.setattr(q, "lib", lambda: fake)
    monkeypatch.setattr(q, "_require_cuda", lambda *ts: None)
    monkeypatch.setattr(q, "_stream", lambda s: 0)
    sizes = []
    real_sizes = q._qweight_sizes
    monkeypatch.setattr(q, "_qweight_sizes", lambda w, name="w": (sizes.append(1), real_sizes(w, name)))
    w, x, y = _qw(), torch.zeros(2, 256), torch.zeros(2, 64)
    for _ in range(3):
        q.qmm_linear(x, w, y=y)
    assert len(calls) == 3 and len(sizes) == 1
    w.codes = torch.zeros(64, 255, dtype=torch.int8)  # another tensor, the wrong size
    with pytest.raises(ValueError, match="codes"):
        q.qmm_linear(x, w, y=y)
    w.codes = torch.zeros(64, 256, dtype=torch.int8)
    q.qmm_linear(x, w, y=y)
    assert len(sizes) == 3
    w.N = 65  # shape fields changed under the same tensors
    with pytest.raises(ValueError):
        q.qmm_linear(x, w, y=torch.zeros(2, 65))


def test_moe_experts_descriptor_is_cached_and_invalidated(monkeypatch):
    calls = []

    class FakeLib:
        def moe_ffn_workspace_bytes(self, *a):
            return 1 << 16

        def moe_ffn_forward(self, *a):
            calls.append(a)
            return q.QMM_OK

    fake = FakeLib()
    monkeypatch.setattr(q, "lib", lambda: fake)
    monkeypatch.setattr(q, "_require_cuda", lambda *ts: None)
    monkeypatch.setattr(q, "_stream", lambda s: 0)
    built = []
    real_c = q.MoeExperts._c
    monkeypatch.setattr(q.MoeExperts, "_c", lambda self: (built.append(1), real_c(self))[1])
    ex, M, k = _experts(), 5, 2
    x, idx, w = torch.zeros(M, 256), torch.zeros(M, k, dtype=torch.int32), torch.zeros(M, k)
    for _ in range(3):
        q.moe_ffn_forward(x, idx, w, ex)
    assert len(calls) == 3 and len(built) == 1
    ex.down_codes = torch.zeros(4, 256, 32, dtype=torch.uint8)  # another tensor, the wrong size
    with pytest.raises(ValueError, match="down_codes"):
        q.moe_ffn_forward(x, idx, w, ex)
    ex.down_codes = torch.zeros(4, 256, 64, dtype=torch.uint8)
    q.moe_ffn_forward(x, idx, w, ex)
    assert len(built) == 2
