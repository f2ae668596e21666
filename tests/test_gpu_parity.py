"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars: bit-exact quantised codes, scales, zero points, router logits and
top-k indices; routing weights within 2e-6; fp32 outputs within
|err| <= 1e-5 * sum_k |x_k w_k| + 1e-6 (propagated through SwiGLU for the MoE
layer); bf16 outputs within a 1e-2 relative L2 error per row with the same
arg-max.  Full-size workloads are checked on sampled rows / tokens that the
oracle computes one by one.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import recipes
import group_quantized_moe_gb300 as q
from group_quantized_moe_gb300 import build_lib
from parity_checks import assert_bf16_rows, assert_within
import oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.build()
    q.lib()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    q.qmm_device_status(clear=True)
    yield d
    assert q.qmm_device_status(clear=True) == 0


def T(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _codes_u8(qw):
    return qw.codes.cpu().numpy().view(np.uint8).reshape(-1)


def assert_quant_equal(gq, oq):
    np.testing.assert_array_equal(_codes_u8(gq), oq.codes.reshape(-1))
    np.testing.assert_array_equal(gq.scales.cpu().numpy().view(np.uint32),
                                  oq.scales.view(np.uint32))
    np.testing.assert_array_equal(gq.zps.cpu().numpy(), oq.zps)


def _weights(N, K, seed=0, stream=2, outl=False, sigma=0.02):
    w = synth.normal(seed, stream, N * K, sigma).reshape(N, K)
    if outl:
        synth.outliers(seed, stream + 100, w.reshape(-1), 0.01, 20.0)
    return w


# ------------------------------------------------------------- quantise (A1)

QSHAPES = [(8, 64, 128, 256, False), (8, 64, 4096, 4096, True), (4, 128, 4096, 4096, False),
           (4, 128, 2048, 4096, False), (8, 32, 37, 96, False), (4, 256, 3, 512, True),
           (8, 256, 1, 256, False), (4, 32, 5, 32, False), (4, 64, 64, 4096, False),
           (8, 128, 96, 2048, False)]


@pytest.mark.parametrize("bits,group,N,K,outl", QSHAPES)
def test_quantize_bit_exact(dev, bits, group, N, K, outl):
    w = _weights(N, K, outl=outl)
    g = q.qmm_quantize_groupwise(T(w, dev), bits, group)
    assert_quant_equal(g, oracle.quantize(w, bits, group))


@pytest.mark.parametrize("bits", [8, 4])
def test_quantize_degenerate_groups(dev, bits):
    """Constant groups (zero, positive, negative), a group whose range is one
    ulp (conversions saturate), a mix with ordinary groups, and exact half
    ties: codes and a zero point that round away from zero, and a maximum
    that reaches 2^bits after rounding and is clamped (the worked examples
    of the oracle's pins, padded with zeros inside their range)."""
    K, group = 256, 32
    rows = [np.zeros(K), np.full(K, 0.5), np.full(K, -3.0),
            np.where(np.arange(K) % 2 == 0, 100.0, np.nextafter(np.float32(100.0), np.float32(200))),
            _weights(1, K)[0]]
    mix = _weights(1, K, stream=5)[0].copy()
    mix[:32] = 7.25
    mix[64:96] = 0.0
    rows.append(mix)
    ties8 = np.zeros(K)
    ties8[:6] = [0, 255, 0.5, 2.5, 127.5, 254.5]
    ties8[32:36] = [-2.5, 252.5, 0.5, -0.5]
    ties4 = np.zeros(K)
    ties4[:4] = [-0.5, 14.5, 2.5, 6.5]
    rows += [ties8, ties4]
    w = np.stack(rows).astype(np.float32)
    g = q.qmm_quantize_groupwise(T(w, dev), bits, group)
    assert_quant_equal(g, oracle.quantize(w, bits, group))


@pytest.mark.slow
def test_quantize_vocab_head_sampled_rows(dev):
    """Full INT8 g64 vocab head W[129280, 4096] (with outliers) quantised on
    the GPU; 48 rows re-quantised by the oracle from regenerated rows."""
    r = recipes.CFG2_VOCAB
    w = recipes.linear_weight_rows(r)
    g = q.qmm_quantize_groupwise(T(w, dev), r.bits, r.group)
    del w
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 1, r.N - 1], rng.integers(0, r.N, 45)]))
    codes = g.codes.cpu().numpy().view(np.uint8)
    scales, zps = g.scales.cpu().numpy(), g.zps.cpu().numpy()
    for n in rows:
        oq = oracle.quantize(recipes.linear_weight_rows(r, int(n), 1), r.bits, r.group)
        np.testing.assert_array_equal(codes[n], oq.codes)
        np.testing.assert_array_equal(scales[n].view(np.uint32), oq.scales[0].view(np.uint32))
        np.testing.assert_array_equal(zps[n], oq.zps[0])


# -------------------------------------------------------------- linear (A2)

def _linear_case(dev, bits, group, N, K, M, bf16, outl=False, stream=2):
    w = _weights(N, K, outl=outl, stream=stream)
    x = synth.normal(3, 1, M * K).reshape(M, K)
    if bf16:
        xb = synth.to_bf16(x)
        x = synth.bf16_to_f32(xb)
        xd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        xd = T(x, dev)
    oq = oracle.quantize(w, bits, group)
    g = q.qmm_quantize_groupwise(T(w, dev), bits, group)
    y = q.qmm_linear(xd, g).cpu().numpy()
    assert_within(y, oracle.linear_fused(x, oq), oracle.linear_bound(x, oq),
                  f"linear b{bits} g{group} N{N} K{K} M{M} bf16={bf16}")


@pytest.mark.parametrize("bits,group,N,K,outl", [(8, 64, 128, 256, False),
                                                 (8, 64, 4096, 4096, True),
                                                 (4, 128, 4096, 4096, False),
                                                 (4, 128, 2048, 4096, False)])
def test_linear_configs(dev, bits, group, N, K, outl):
    _linear_case(dev, bits, group, N, K, 1, False, outl)


@pytest.mark.parametrize("bits,group,N,K", [(8, 64, 37, 256), (4, 32, 5, 64), (8, 256, 1, 512),
                                            (4, 64, 333, 1024), (8, 32, 19, 8192),
                                            (4, 128, 7, 16384)])
@pytest.mark.parametrize("M", [1, 2, 3, 5])
def test_linear_ragged(dev, bits, group, N, K, M):
    _linear_case(dev, bits, group, N, K, M, False)


@pytest.mark.parametrize("bits,group", [(8, 64), (4, 128)])
@pytest.mark.parametrize("M", [1, 4, 9])
def test_linear_bf16_activations(dev, bits, group, M):
    _linear_case(dev, bits, group, 256, 1024, M, True)


@pytest.mark.slow
def test_linear_vocab_head_sampled(dev):
    """Decode step of the INT8 g64 workload at full size: x[1, 4096] against
    the 129280-row vocab head; 64 sampled outputs computed by the oracle."""
    r = recipes.CFG2_VOCAB
    x = recipes.linear_x(r)
    w = recipes.linear_weight_rows(r)
    g = q.qmm_quantize_groupwise(T(w, dev), r.bits, r.group)
    del w
    y = q.qmm_linear(T(x, dev), g).cpu().numpy()[0]
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, r.N - 1], rng.integers(0, r.N, 62)]))
    for n in rows:
        oq = oracle.quantize(recipes.linear_weight_rows(r, int(n), 1), r.bits, r.group)
        assert_within(y[n:n + 1], oracle.linear_fused(x, oq)[0], oracle.linear_bound(x, oq)[0],
                      f"row {n}")


def test_linear_chain_on_one_stream(dev):
    """Kernels overlap their launches with the preceding kernel: a layer
    whose input is the previous layer's output must still see that output,
    and a linear layer launched right after re-quantising its weights in
    place must see the new codes.  Two layers back to back on one stream
    (M = 1 GEMV and M = 3 small-M path), then an in-place re-quantisation
    followed at once by a linear call, all without host synchronisation."""
    K1, N1, N2 = 2048, 2048, 1000
    w1 = _weights(N1, K1, seed=3, stream=2)
    w2 = _weights(N2, N1, seed=3, stream=3)
    w1b = _weights(N1, K1, seed=4, stream=2)
    o1, o2, o1b = oracle.quantize(w1, 8, 64), oracle.quantize(w2, 4, 128), oracle.quantize(w1b, 8, 64)
    g1 = q.qmm_quantize_groupwise(T(w1, dev), 8, 64)
    g2 = q.qmm_quantize_groupwise(T(w2, dev), 4, 128)
    w1b_d = T(w1b, dev)
    d2 = np.abs(oracle.dequantize(o2).astype(np.float64))
    for M in (1, 3):
        x = synth.normal(11 + M, 1, M * K1).reshape(M, K1)
        xd = T(x, dev)
        y1 = torch.empty((M, N1), dtype=torch.float32, device=dev)
        y2 = torch.empty((M, N2), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        q.qmm_linear(xd, g1, y=y1)
        q.qmm_linear(y1, g2, y=y2)
        y2 = y2.cpu().numpy()
        r1, b1 = oracle.linear_fused(x, o1), oracle.linear_bound(x, o1)
        r2 = oracle.linear_fused(r1.astype(np.float32), o2)
        # the first layer's error (within b1) propagates through |W2|
        b2 = oracle.linear_bound(r1.astype(np.float32), o2) + b1 @ d2.T + 1e-6 * np.abs(r2)
        assert_within(y2, r2, b2, f"chained layers M={M}")
    x = synth.normal(15, 1, K1).reshape(1, K1)
    xd = T(x, dev)
    y_new = torch.empty((1, N1), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    # three kernels back to back: linear, in-place quantise, linear
    y_old = q.qmm_linear(xd, g1)
    q.qmm_quantize_groupwise(w1b_d, 8, 64, out=g1)
    q.qmm_linear(xd, g1, y=y_new)
    y_new = y_new.cpu().numpy()
    assert_within(y_old.cpu().numpy(), oracle.linear_fused(x, o1), oracle.linear_bound(x, o1), "old")
    assert_within(y_new, oracle.linear_fused(x, o1b), oracle.linear_bound(x, o1b), "re-quantised")


# -------------------------------------------------------------- router (A3)

def _router_case(dev, M, E, H, k, bias_kind, bf16, wr=None, x=None):
    if x is None:
        x = synth.normal(4, 1, M * H).reshape(M, H)
    if bf16:
        xb = synth.to_bf16(x)
        x = synth.bf16_to_f32(xb)
        xd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        xd = T(x, dev)
    if wr is None:
        wr = synth.normal(4, 10, E * H, 0.02).reshape(E, H)
    bias = None
    if bias_kind == "zipf":
        bias = synth.zipf_bias(0, 20, E, 1.1)
    ws = torch.zeros(q.moe_route_workspace_bytes(M, E), dtype=torch.uint8, device=dev)
    idx, w, cnt = q.moe_route_topk(xd, T(wr, dev), None if bias is None else T(bias, dev), k,
                                   workspace=ws)
    torch.cuda.synchronize()
    logits = oracle.router_logits(x, wr, bias)
    glog = ws[: M * E * 4].view(torch.float32).cpu().numpy().reshape(M, E)
    np.testing.assert_array_equal(glog.view(np.uint32), logits.view(np.uint32))
    oidx, ow = oracle.topk(logits, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    assert np.abs(w.cpu().numpy() - ow).max() <= 2e-6
    np.testing.assert_array_equal(cnt.cpu().numpy(), np.bincount(oidx.reshape(-1), minlength=E))


@pytest.mark.parametrize("M,E,H,k,bias,bf16", [
    (8, 256, 4096, 6, None, False),     # MoE decode router
    (512, 256, 4096, 6, "zipf", True),  # batched prefill router, Zipf bias
    (1, 256, 4096, 6, None, False),
    (3, 100, 4096, 1, "zipf", False),
    (17, 64, 4100, 16, None, True),
    (5, 8, 64, 3, None, False),
    (70, 1024, 256, 8, "zipf", False),
    # tiles staged through shared memory (M > 64, H a multiple of 512):
    # ragged token and expert tiles, a single chunk, fp32 and bf16 tokens
    (100, 40, 1024, 6, None, False),
    (129, 256, 2048, 8, "zipf", True),
    (65, 16, 512, 4, None, True),
    (300, 1024, 4096, 16, "zipf", False),
])
def test_router(dev, M, E, H, k, bias, bf16):
    _router_case(dev, M, E, H, k, bias, bf16)


def test_router_exact_ties_lower_index_wins(dev):
    """Duplicated router rows give bit-identical logits; the lower expert
    index must be selected first."""
    E, H, M = 32, 512, 6
    wr = synth.normal(5, 10, E * H, 0.02).reshape(E, H)
    for a, b in ((3, 17), (17, 30), (5, 6), (0, 31)):
        wr[b] = wr[a]
    x = synth.normal(5, 1, M * H).reshape(M, H)
    x[:, :] = x[0]  # same token repeated
    _router_case(dev, M, E, H, 6, None, False, wr=wr, x=x)
    wr2 = np.tile(wr[:1], (E, 1))  # every logit equal -> experts 0..k-1
    _router_case(dev, 2, E, H, 4, None, False, wr=wr2)
    # the same ties through the shared-memory tiled path (M > 64)
    x80 = np.tile(x[:1], (80, 1))
    _router_case(dev, 80, E, H, 6, None, False, wr=wr, x=x80)


# ----------------------------------------------------------- MoE layer (A4-A6)

def _small_experts(dev, E, H, I, bits, group, seed=1):
    def fill(which, e, out):
        stream = {"gate": 11, "up": 12, "down": 13}[which] + 10 * e
        out[...] = synth.normal(seed, stream, out.size, 0.05).reshape(out.shape)
    ex = q.quantize_experts(E, H, I, bits, group, fill, device=dev)
    og, ou, od = [], [], []
    for e in range(E):
        for which, lst in (("gate", og), ("up", ou), ("down", od)):
            rows, cols = (I, H) if which != "down" else (H, I)
            buf = np.empty((rows, cols), np.float32)
            fill(which, e, buf)
            lst.append(oracle.quantize(buf, bits, group))
    return ex, og, ou, od


def _moe_check(dev, x, xd, idx, w, ex, og, ou, od, y_dtype=torch.float32, what=""):
    """fp32 activations run the fp32 CUDA-core path (strict bound); bf16
    activations may run the fp16 tensor-core path (bf16 bar)."""
    y = q.moe_ffn_forward(xd, T(idx, dev), T(w, dev), ex, y_dtype=y_dtype)
    y = y.float().cpu().numpy().astype(np.float64)
    yref, bound = oracle.moe_ffn(x, idx, w, og, ou, od)
    if y_dtype == torch.float32 and xd.dtype == torch.float32:
        assert_within(y, yref, bound, what)
    else:
        assert_bf16_rows(y, yref, what)
    return y


def _bf16_x(x, dev):
    xb = synth.to_bf16(x)
    return synth.bf16_to_f32(xb), torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)


@pytest.mark.parametrize("bits,group,H,I", [(4, 64, 256, 256), (8, 128, 512, 512),
                                            (4, 32, 512, 128), (8, 64, 256, 768)])
@pytest.mark.parametrize("bf16", [False, True])
def test_moe_small(dev, bits, group, H, I, bf16):
    E, k, M = 8, 2, 5
    ex, og, ou, od = _small_experts(dev, E, H, I, bits, group)
    x = synth.normal(6, 1, M * H).reshape(M, H)
    if bf16:
        xb = synth.to_bf16(x)
        x = synth.bf16_to_f32(xb)
        xd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        xd = T(x, dev)
    wr = synth.normal(6, 10, E * H, 0.05).reshape(E, H)
    idx, w = oracle.topk(oracle.router_logits(x, wr, None), k)
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what=f"b{bits} g{group} bf16={bf16}")
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, y_dtype=torch.bfloat16, what="bf16 out")


def test_moe_one_hot_expert_many_tokens(dev):
    """Every token on the same expert (a long token list, ragged last chunk),
    plus M = 1."""
    E, H, I = 4, 256, 256
    ex, og, ou, od = _small_experts(dev, E, H, I, 4, 64, seed=2)
    M = 37
    x = synth.normal(7, 1, M * H).reshape(M, H)
    idx = np.full((M, 1), 2, np.int32)
    w = np.ones((M, 1), np.float32)
    _moe_check(dev, x, T(x, dev), idx, w, ex, og, ou, od, what="one expert")
    idx2 = np.stack([np.full(M, 2), np.arange(M) % 4], axis=1).astype(np.int32)
    idx2[idx2[:, 1] == 2, 1] = 0
    w2 = np.full((M, 2), 0.5, np.float32)
    _moe_check(dev, x, T(x, dev), idx2, w2, ex, og, ou, od, what="two slots")
    _moe_check(dev, x[:1], T(x[:1], dev), idx2[:1], w2[:1], ex, og, ou, od, what="M=1")


@pytest.mark.parametrize("group,H,I", [(64, 512, 256), (128, 1024, 512), (256, 1024, 1024)])
def test_moe_tensor_core_tiles(dev, group, H, I):
    """bf16 tokens, INT8 experts: the tensor-core path.  One expert gets 160
    tokens (two 128-token tiles, ragged last tile), others 1-17 tokens, some
    none; H and I span several 128-feature tiles and 64-wide K stages."""
    E, k = 6, 2
    ex, og, ou, od = _small_experts(dev, E, H, I, 8, group, seed=9)
    M = 160
    x, xd = _bf16_x(synth.normal(9, 1, M * H).reshape(M, H), dev)
    idx = np.zeros((M, k), np.int32)
    idx[:, 0] = 3
    idx[:, 1] = np.where(np.arange(M) % 17 == 0, 1, np.where(np.arange(M) % 5 == 0, 5, 0))
    w = np.full((M, k), 0.5, np.float32)
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what=f"tc g{group}")
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, y_dtype=torch.bfloat16, what="tc bf16 out")
    # a single token, and a bad index (skipped, flagged)
    _moe_check(dev, x[:1], xd[:1], idx[:1], w[:1], ex, og, ou, od, what="tc M=1")
    bad = idx[:7].copy()
    bad[2, 1] = 77
    q.qmm_device_status(clear=True)
    y = q.moe_ffn_forward(xd[:7], T(bad, dev), T(w[:7], dev), ex).cpu().numpy()
    assert q.qmm_device_status(clear=True) & q.QMM_DEV_BAD_EXPERT
    w_ok = np.where(bad < E, w[:7], 0).astype(np.float32)
    yref, _ = oracle.moe_ffn(x[:7], np.where(bad < E, bad, 0).astype(np.int32), w_ok, og, ou, od)
    assert_bf16_rows(y, yref, "tc bad index")


def test_tc_timing_events(dev):
    """qmm_tc_timing: the tensor-core path records its two GEMM launches;
    the result is unchanged and the durations are positive."""
    E, H, I, k = 6, 512, 256, 2
    ex, og, ou, od = _small_experts(dev, E, H, I, 8, 64, seed=13)
    M = 96
    x, xd = _bf16_x(synth.normal(13, 1, M * H).reshape(M, H), dev)
    idx = np.stack([np.full(M, 3), np.where(np.arange(M) % 4 == 0, 1, 5)], axis=1).astype(np.int32)
    w = np.full((M, k), 0.5, np.float32)
    y0 = _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what="tc, timing off")
    q.qmm_tc_timing(True)
    try:
        with pytest.raises(q.QmmError):
            q.qmm_tc_timing_ms()  # nothing recorded yet
        y1 = _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what="tc, timing on")
        g_ms, d_ms = q.qmm_tc_timing_ms()
    finally:
        q.qmm_tc_timing(False)
    np.testing.assert_array_equal(y1, y0)
    assert 0.0 < g_ms < 1000.0 and 0.0 < d_ms < 1000.0, (g_ms, d_ms)


def test_moe_gate_up_layouts_differ(dev):
    """Gate and up whose scale and zero-point arrays have different strides
    between experts (up's inside padded buffers, described to the library
    through its C descriptor): the tensor-core path, whose dequantising
    threads share one scale offset between the two matrices, is not taken,
    and the CUDA-core kernels give the strict fp32 bound for bf16 tokens.
    The same experts in one layout take the tensor-core path."""
    E, H, I, group, k = 6, 512, 256, 64, 2
    ex, og, ou, od = _small_experts(dev, E, H, I, 8, group, seed=11)
    G = H // group
    pad = 128
    us = torch.zeros((E, I + pad, G), dtype=torch.float32, device=dev)
    uz = torch.zeros((E, I + pad, G), dtype=torch.int32, device=dev)
    us[:, :I] = ex.up_scales.view(E, I, G)
    uz[:, :I] = ex.up_zps.view(E, I, G)
    desc = ex._c()
    desc.up.scales = us.data_ptr()
    desc.up.zps = uz.data_ptr()
    desc.up.groups_stride = (I + pad) * G
    assert desc.up.groups_stride != desc.gate.groups_stride
    M = 40
    x, xd = _bf16_x(synth.normal(11, 1, M * H).reshape(M, H), dev)
    idx = np.stack([np.full(M, 2), np.where(np.arange(M) % 3 == 0, 4, 0)], axis=1).astype(np.int32)
    w = np.full((M, k), 0.5, np.float32)
    idx_d, w_d = T(idx, dev), T(w, dev)
    y = torch.empty((M, H), dtype=torch.float32, device=dev)
    L = q.lib()
    ws = torch.empty((int(L.moe_ffn_workspace_bytes(M, k, ctypes.byref(desc))),),
                     dtype=torch.uint8, device=dev)
    rc = L.moe_ffn_forward(xd.data_ptr(), q.QMM_BF16, M, idx_d.data_ptr(), w_d.data_ptr(), k,
                           ctypes.byref(desc), y.data_ptr(), q.QMM_F32, ws.data_ptr(),
                           ws.numel(), None)
    assert rc == 0, q.lib().qmm_last_error()
    torch.cuda.synchronize()
    yref, bound = oracle.moe_ffn(x, idx, w, og, ou, od)
    assert_within(y.cpu().numpy().astype(np.float64), yref, bound,
                  "gate and up in different layouts")
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what="gate and up in one layout")


def test_moe_bad_expert_index_flagged(dev):
    """An out-of-range index sets QMM_DEV_BAD_EXPERT and contributes nothing."""
    E, H, I = 4, 256, 256
    ex, og, ou, od = _small_experts(dev, E, H, I, 8, 64, seed=3)
    M = 3
    x = synth.normal(8, 1, M * H).reshape(M, H)
    idx = np.array([[0, 9], [1, 2], [-1, 3]], np.int32)
    w = np.array([[0.6, 0.4], [0.5, 0.5], [0.3, 0.7]], np.float32)
    q.qmm_device_status(clear=True)
    y = q.moe_ffn_forward(T(x, dev), T(idx, dev), T(w, dev), ex).cpu().numpy()
    assert q.qmm_device_status(clear=True) & q.QMM_DEV_BAD_EXPERT
    idx_ok = np.where((idx >= 0) & (idx < E), idx, 0).astype(np.int32)
    w_ok = np.where((idx >= 0) & (idx < E), w, 0).astype(np.float32)
    yref, bound = oracle.moe_ffn(x, idx_ok, w_ok, og, ou, od)
    assert_within(y, yref, bound, "bad index")


# ------------------------- small-M kernels (2..8 rows per matrix, K 2048 / 4096)

SMALLM_SHAPES = [(8, 64, 4096), (4, 64, 4096), (8, 128, 2048), (4, 128, 2048)]


@pytest.mark.parametrize("bits,group,K", SMALLM_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_linear_small_m(dev, bits, group, K, M):
    # N = 1000 is not a multiple of the rows per tile: ragged last tile
    _linear_case(dev, bits, group, 1000, K, M, False, outl=True)


@pytest.mark.parametrize("bits,group,K", [(8, 64, 4096), (4, 128, 2048)])
def test_linear_small_m_bf16(dev, bits, group, K):
    _linear_case(dev, bits, group, 777, K, 6, True)


@pytest.mark.parametrize("bits,group,H,I", [(4, 64, 2048, 2048), (8, 128, 4096, 2048),
                                            (4, 128, 2048, 4096), (8, 64, 2048, 2048)])
@pytest.mark.parametrize("bf16", [False, True])
def test_moe_small_m(dev, bits, group, H, I, bf16):
    """Decode-sized batches (M <= 8) on the small-M expert kernels."""
    E, k = 8, 3
    ex, og, ou, od = _small_experts(dev, E, H, I, bits, group, seed=4)
    wr = synth.normal(9, 10, E * H, 0.05).reshape(E, H)
    for M in (1, 3, 8):
        x = synth.normal(9 + M, 1, M * H).reshape(M, H)
        if bf16:
            x, xd = _bf16_x(x, dev)
        else:
            xd = T(x, dev)
        idx, w = oracle.topk(oracle.router_logits(x, wr, None), k)
        _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what=f"b{bits} g{group} M{M} bf16={bf16}")


def test_moe_tensor_core_few_token_experts(dev):
    """bf16 tokens with M > 8 on the tensor-core path, H = I = 2048: experts with one
    or two tokens run on the small-M kernels (two tokens per pass), the others on the
    tensor cores, in the same call."""
    E, k, H, I, M = 8, 2, 2048, 2048, 24
    ex, og, ou, od = _small_experts(dev, E, H, I, 8, 128, seed=13)
    x, xd = _bf16_x(synth.normal(13, 1, M * H).reshape(M, H), dev)
    idx = np.zeros((M, k), np.int32)
    idx[:, 0] = 0                  # 24 tokens: tensor cores
    idx[:, 1] = 4                  # 17 tokens: tensor cores
    idx[0, 1] = 1                  # one token
    idx[1:3, 1] = 2                # two tokens
    idx[3:6, 1] = 3                # three tokens: tensor cores
    idx[6, 1] = 7                  # one token
    w = np.tile(np.array([0.6, 0.4], np.float32), (M, 1))
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, what="split fp32 out")
    _moe_check(dev, x, xd, idx, w, ex, og, ou, od, y_dtype=torch.bfloat16, what="split bf16 out")
    # every expert light (k = 1: expert 0 gets two tokens, the others one), so
    # the tensor-core launches find no work items
    idx2 = (np.arange(9, dtype=np.int32) % E).reshape(9, 1)
    w2 = np.ones((9, 1), np.float32)
    _moe_check(dev, x[:9], xd[:9], idx2, w2, ex, og, ou, od, what="all light")


def test_moe_small_m_token_patterns(dev):
    """Every token on the same experts (8 tokens per expert), an expert
    repeated inside each token (16 assignments: two passes of 8), and one
    expert with 5 tokens beside single-token experts."""
    E, H, I = 8, 2048, 2048
    ex, og, ou, od = _small_experts(dev, E, H, I, 4, 64, seed=5)
    M = 8
    x = synth.normal(12, 1, M * H).reshape(M, H)
    w = np.tile(np.array([0.5, 0.3, 0.2], np.float32), (M, 1))
    idx = np.tile(np.array([1, 4, 6], np.int32), (M, 1))
    _moe_check(dev, x, T(x, dev), idx, w, ex, og, ou, od, what="8 tokens per expert")
    idx = np.tile(np.array([2, 2, 5], np.int32), (M, 1))
    _moe_check(dev, x, T(x, dev), idx, w, ex, og, ou, od, what="repeated expert")
    idx = np.array([[3, m % 3, 4 + m % 4] for m in range(M)], np.int32)
    idx[5:, 0] = 7
    _moe_check(dev, x, T(x, dev), idx, w, ex, og, ou, od, what="mixed")


def test_moe_decode_bad_expert_index_flagged(dev):
    """Decode batches group their assignments inside the expert kernels: an
    out-of-range index there is also skipped (its slot contributes nothing)
    and flagged as QMM_DEV_BAD_EXPERT."""
    E, H, I = 8, 2048, 2048
    ex, og, ou, od = _small_experts(dev, E, H, I, 4, 64, seed=6)
    M = 4
    x = synth.normal(13, 1, M * H).reshape(M, H)
    idx = np.array([[0, 5, 2], [8, 1, 2], [3, -1, 5], [7, 6, 1]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.4, 0.4, 0.2], [0.6, 0.3, 0.1], [0.2, 0.3, 0.5]], np.float32)
    q.qmm_device_status(clear=True)
    y = q.moe_ffn_forward(T(x, dev), T(idx, dev), T(w, dev), ex).cpu().numpy()
    assert q.qmm_device_status(clear=True) & q.QMM_DEV_BAD_EXPERT
    ok = (idx >= 0) & (idx < E)
    yref, bound = oracle.moe_ffn(x, np.where(ok, idx, 0).astype(np.int32),
                                 np.where(ok, w, 0).astype(np.float32), og, ou, od)
    assert_within(y, yref, bound, "decode bad index")


def test_moe_decode_combine_outputs(dev):
    """Decode batches (the in-kernel grouping): every output element is
    written (y starts as NaN), a token with no valid slot gets zeros, a
    workspace left dirty by an earlier call is reused, bf16 output rounds the
    fp32 sum, and repeated calls agree bit for bit."""
    E, H, I = 8, 2048, 2048
    ex, og, ou, od = _small_experts(dev, E, H, I, 8, 64, seed=21)
    M, k = 6, 3
    x = synth.normal(21, 1, M * H).reshape(M, H)
    idx = np.array([[0, 5, 2], [-1, 9, 100], [3, 3, 5], [7, 6, 1], [4, -2, 4], [1, 0, 2]],
                   np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.4, 0.4, 0.2], [0.6, 0.3, 0.1], [0.2, 0.3, 0.5],
                  [0.7, 0.2, 0.1], [0.25, 0.25, 0.5]], np.float32)
    ok = (idx >= 0) & (idx < E)
    yref, bound = oracle.moe_ffn(x, np.where(ok, idx, 0).astype(np.int32),
                                 np.where(ok, w, 0).astype(np.float32), og, ou, od)
    xd, idxd, wd = T(x, dev), T(idx, dev), T(w, dev)
    nbytes = q.moe_ffn_workspace_bytes(M, k, ex)
    ws = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device=dev)
    outs = []
    for rep in range(3):
        y = torch.full((M, H), float("nan"), dtype=torch.float32, device=dev)
        q.qmm_device_status(clear=True)
        q.moe_ffn_forward(xd, idxd, wd, ex, y=y, workspace=ws)
        assert q.qmm_device_status(clear=True) & q.QMM_DEV_BAD_EXPERT
        outs.append(y.cpu().numpy())
    yv = outs[0].astype(np.float64)
    assert np.isfinite(yv).all()
    assert (outs[0][1] == 0).all()
    assert_within(yv, yref, bound, "decode combine")
    for o in outs[1:]:
        np.testing.assert_array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    yb = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=dev)
    q.moe_ffn_forward(xd, idxd, wd, ex, y=yb, workspace=ws)
    q.qmm_device_status(clear=True)
    expect = torch.from_numpy(outs[0]).to(torch.bfloat16)
    np.testing.assert_array_equal(yb.cpu().view(torch.int16).numpy(),
                                  expect.view(torch.int16).numpy())


# ----------------------------------------------- full-size MoE workloads

def _full_moe(dev, r):
    def fill(which, e, out):
        recipes.moe_expert_rows(r, which, e, out=out)
    ex = q.quantize_experts(r.E, r.H, r.I, r.bits, r.group, fill, device=dev)
    return ex


def _oracle_experts(r, needed):
    og, ou, od = [None] * r.E, [None] * r.E, [None] * r.E
    for e in sorted(set(int(v) for v in needed)):
        og[e] = oracle.quantize(recipes.moe_expert_rows(r, "gate", e), r.bits, r.group)
        ou[e] = oracle.quantize(recipes.moe_expert_rows(r, "up", e), r.bits, r.group)
        od[e] = oracle.quantize(recipes.moe_expert_rows(r, "down", e), r.bits, r.group)
    return og, ou, od


@pytest.mark.slow
def test_moe_decode_full_size(dev):
    """MoE decode layer at full size: M=8, 256 experts INT4 g64, top-6."""
    r = recipes.CFG4
    x, _ = recipes.moe_x(r)
    wr, bias = recipes.moe_router(r)
    ex = _full_moe(dev, r)
    idx, w, cnt = q.moe_route_topk(T(x, dev), T(wr, dev), None, r.k)
    oidx, ow = oracle.topk(oracle.router_logits(x, wr, bias), r.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    assert np.abs(w.cpu().numpy() - ow).max() <= 2e-6
    og, ou, od = _oracle_experts(r, oidx.reshape(-1))
    # FFN from the oracle's routing, then the whole GPU pipeline with its own
    # routing weights (|dw| <= 2e-6 enters the bound).
    _moe_check(dev, x, T(x, dev), oidx, ow, ex, og, ou, od, what="decode ffn")
    y = q.moe_ffn_forward(T(x, dev), idx, w, ex).cpu().numpy()
    yref, bound = oracle.moe_ffn(x, oidx, ow, og, ou, od, dw=2e-6)
    assert_within(y, yref, bound, "decode pipeline")


# ------------------------------------------- one-launch decode layer (f)2

def _route_and_ffn(dev, x, xd, wr, bias, k, ex, y_dtype=torch.float32):
    """The two-call path (moe_route_topk, moe_ffn_forward) on the same inputs."""
    idx, w, cnt = q.moe_route_topk(xd, T(wr, dev), None if bias is None else T(bias, dev), k)
    y = q.moe_ffn_forward(xd, idx, w, ex, y_dtype=y_dtype)
    return idx, w, cnt, y


@pytest.mark.parametrize("bits,group", [(4, 64), (8, 128)])
@pytest.mark.parametrize("bf16", [False, True])
def test_moe_decode_one_launch(dev, bits, group, bf16):
    """The whole decode layer in one cooperative launch: the top-k indices and
    the histogram bit-exact against the oracle, weights within 2e-6, outputs
    within the fp32 bound (routing-weight difference included), and
    bit-identical to the two-call path (same logits order, same expert
    kernels, same combine order) for fp32 and bf16 outputs."""
    E, H, I = 16, 4096, 2048
    ex, og, ou, od = _small_experts(dev, E, H, I, bits, group, seed=31)
    wr = synth.normal(32, 10, E * H, 0.05).reshape(E, H)
    bias = synth.normal(33, 20, E, 0.5)
    for M, k, b in ((1, 6, None), (3, 1, bias), (8, 6, bias), (5, 16, None)):
        x = synth.normal(34 + M, 1, M * H).reshape(M, H)
        if bf16:
            x, xd = _bf16_x(x, dev)
        else:
            xd = T(x, dev)
        bd = None if b is None else T(b, dev)
        idx = torch.empty((M, k), dtype=torch.int32, device=dev)
        w = torch.empty((M, k), dtype=torch.float32, device=dev)
        cnt = torch.empty((E,), dtype=torch.int32, device=dev)
        y = q.moe_decode_forward(xd, T(wr, dev), bd, k, ex, topk_idx=idx, topk_w=w,
                                 expert_counts=cnt)
        oidx, ow = oracle.topk(oracle.router_logits(x, wr, b), k)
        np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
        assert np.abs(w.cpu().numpy() - ow).max() <= 2e-6
        np.testing.assert_array_equal(cnt.cpu().numpy(), np.bincount(oidx.reshape(-1), minlength=E))
        yref, bound = oracle.moe_ffn(x, oidx, ow, og, ou, od, dw=2e-6)
        assert_within(y.cpu().numpy().astype(np.float64), yref, bound, f"one launch M{M} k{k}")
        i2, w2, c2, y2 = _route_and_ffn(dev, x, xd, wr, b, k, ex)
        np.testing.assert_array_equal(idx.cpu().numpy(), i2.cpu().numpy())
        np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), w2.cpu().numpy().view(np.uint32))
        np.testing.assert_array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
        yb = q.moe_decode_forward(xd, T(wr, dev), bd, k, ex, y_dtype=torch.bfloat16)
        _, _, _, yb2 = _route_and_ffn(dev, x, xd, wr, b, k, ex, y_dtype=torch.bfloat16)
        np.testing.assert_array_equal(yb.cpu().view(torch.int16).numpy(),
                                      yb2.cpu().view(torch.int16).numpy())


def test_moe_decode_one_launch_repeatable_with_dirty_workspace(dev):
    E, H, I, M, k = 8, 4096, 2048, 8, 6
    ex, og, ou, od = _small_experts(dev, E, H, I, 4, 64, seed=41)
    wr = T(synth.normal(42, 10, E * H, 0.05).reshape(E, H), dev)
    x = T(synth.normal(43, 1, M * H).reshape(M, H), dev)
    ws = torch.full((q.moe_decode_workspace_bytes(M, k, ex),), 0x77, dtype=torch.uint8, device=dev)
    ys = [q.moe_decode_forward(x, wr, None, k, ex, workspace=ws).cpu().numpy() for _ in range(3)]
    for yy in ys[1:]:
        np.testing.assert_array_equal(yy.view(np.uint32), ys[0].view(np.uint32))
    with pytest.raises(q.QmmError):  # a shape it does not take
        ex2, *_ = _small_experts(dev, 4, 2048, 2048, 4, 64, seed=44)
        q.moe_decode_forward(T(synth.normal(45, 1, 2 * 2048).reshape(2, 2048), dev),
                             T(synth.normal(46, 10, 4 * 2048, 0.05).reshape(4, 2048), dev),
                             None, 2, ex2)


@pytest.mark.slow
def test_moe_decode_one_launch_full_size(dev):
    """The full decode layer (M = 8, 256 INT4 g64 experts, top-6) in one
    launch: indices exact, outputs of every token within the bound of the
    oracle, and bit-identical to the two-call path."""
    r = recipes.CFG4
    x, _ = recipes.moe_x(r)
    wr, bias = recipes.moe_router(r)
    ex = _full_moe(dev, r)
    idx = torch.empty((r.M, r.k), dtype=torch.int32, device=dev)
    w = torch.empty((r.M, r.k), dtype=torch.float32, device=dev)
    y = q.moe_decode_forward(T(x, dev), T(wr, dev), None if bias is None else T(bias, dev), r.k,
                             ex, topk_idx=idx, topk_w=w)
    oidx, ow = oracle.topk(oracle.router_logits(x, wr, bias), r.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    og, ou, od = _oracle_experts(r, oidx.reshape(-1))
    yref, bound = oracle.moe_ffn(x, oidx, ow, og, ou, od, dw=2e-6)
    assert_within(y.cpu().numpy().astype(np.float64), yref, bound, "one launch full size")
    _, _, _, y2 = _route_and_ffn(dev, x, T(x, dev), wr, bias, r.k, ex)
    np.testing.assert_array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))


@pytest.mark.slow
def test_moe_prefill_full_size_sampled(dev):
    """Batched-prefill MoE at full size: M=512 bf16 tokens, Zipf-biased
    routing, 256 experts INT8 g128; 64 or more tokens through the oracle,
    covering every tensor-bound expert's token tiles."""
    r = recipes.CFG5
    x, xb = recipes.moe_x(r)
    wr, bias = recipes.moe_router(r)
    ex = _full_moe(dev, r)
    xd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    idx, w, cnt = q.moe_route_topk(xd, T(wr, dev), T(bias, dev), r.k)
    oidx, ow = oracle.topk(oracle.router_logits(x, wr, bias), r.k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    assert np.abs(w.cpu().numpy() - ow).max() <= 2e-6
    # Tokens: for every expert with 64 or more tokens (the tensor-bound
    # ones), its first and last token -- the last one sits in the expert's
    # last, ragged 128-token tile -- and one from the middle of each further
    # tile; then tokens of the lightest experts; then random ones, 64 or more
    # in all.
    toks = set()
    for e in np.where(np.bincount(oidx.reshape(-1), minlength=r.E) >= 64)[0]:
        mine = np.where((oidx == e).any(axis=1))[0]
        toks.update(int(t) for t in mine[[0, -1]])
        toks.update(int(mine[min(len(mine) - 1, 128 * j + 64)]) for j in range((len(mine) + 127) // 128))
    counts = np.bincount(oidx.reshape(-1), minlength=r.E)
    for e in np.where((counts > 0) & (counts <= 2))[0][:8]:
        toks.add(int(np.where((oidx == e).any(axis=1))[0][0]))
    rng = np.random.default_rng(5)
    while len(toks) < 64:
        toks.add(int(rng.integers(0, r.M)))
    toks = np.array(sorted(toks))
    yref, bound = oracle_pool.moe_tokens(r.name, toks, x[toks], oidx[toks], ow[toks], dw=2e-6)
    for ydt in (torch.float32, torch.bfloat16):
        y = q.moe_ffn_forward(xd, idx, w, ex, y_dtype=ydt).float().cpu().numpy()
        assert_bf16_rows(y[toks], yref, f"prefill y={ydt} ({len(toks)} tokens)")


# ------------------------- activations with massive channels (wide slices)
#
# A few channels 1e3..1e5 times larger than the rest, and weight rows whose
# dequantised weight at those channels is exactly zero (a zero weight
# quantises to q = zp): those rows' outputs get nothing from the large
# channels, so their tolerance is set by the small activations alone, while
# the large ones share the kernels' per-lane activation slices with them.

def _massive_x(seed, M, K, sigma, chans, big):
    x = synth.normal(seed, 1, M * K, sigma).reshape(M, K)
    for j, c in enumerate(chans):
        x[:, c] = big * (1.0 if j % 2 == 0 else -1.0) * (1.0 + 0.1 * np.arange(M))
    return x.astype(np.float32)


def _zero_columns(w, chans, every=2):
    w = w.copy()
    for c in chans:
        w[::every, c] = 0.0
    return w


MASSIVE = [(1e-2, 1e3), (1e-2, 1e4), (1e-3, 1e3), (1e-3, 1e4), (1.0, 1e5)]


@pytest.mark.parametrize("sigma,big", MASSIVE)
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_linear_small_m_massive_activations(dev, sigma, big, M):
    """INT8 g64, K = 4096 (the vocab-head row length and kernel) and INT4
    g128 K = 2048, M = 1..8, fp32 activations with three massive channels."""
    for bits, group, K, N in ((8, 64, 4096, 1536), (4, 128, 2048, 1000)):
        chans = [5, 1000, K - 7]
        w = _zero_columns(_weights(N, K, outl=True), chans)
        x = _massive_x(40 + M, M, K, sigma, chans, big)
        oq = oracle.quantize(w, bits, group)
        assert all((oracle.dequantize(oq)[::2, c] == 0).all() for c in chans)
        g = q.qmm_quantize_groupwise(T(w, dev), bits, group)
        y = q.qmm_linear(T(x, dev), g).cpu().numpy()
        assert_within(y, oracle.linear_fused(x, oq), oracle.linear_bound(x, oq),
                      f"massive b{bits} K{K} M{M} sigma={sigma} big={big}")


@pytest.mark.parametrize("sigma,big", [(1e-2, 1e3), (1e-3, 1e4)])
def test_linear_small_m_massive_bf16_activations(dev, sigma, big):
    K, N, M = 4096, 1000, 2
    chans = [64, 2047, 3000]
    w = _zero_columns(_weights(N, K), chans)
    x, xd = _bf16_x(_massive_x(50, M, K, sigma, chans, big), dev)
    oq = oracle.quantize(w, 8, 64)
    g = q.qmm_quantize_groupwise(T(w, dev), 8, 64)
    y = q.qmm_linear(xd, g).cpu().numpy()
    assert_within(y, oracle.linear_fused(x, oq), oracle.linear_bound(x, oq), "massive bf16")


@pytest.mark.parametrize("sigma,big", [(1e-2, 1e3), (1e-3, 1e4), (1.0, 1e5)])
def test_moe_decode_massive_activations(dev, sigma, big):
    """Decode-sized MoE (INT4 g64, the one-token-per-pass expert kernels with
    32 columns per lane) on tokens with massive channels; the gate and up rows
    of every other intermediate feature hold a zero weight at those channels."""
    E, H, I, k, M = 8, 2048, 2048, 3, 6
    chans = [3, 777, 2040]

    def fill(which, e, out):
        stream = {"gate": 11, "up": 12, "down": 13}[which] + 10 * e
        out[...] = synth.normal(21, stream, out.size, 0.05).reshape(out.shape)
        if which != "down":
            out[...] = _zero_columns(out, chans)

    ex = q.quantize_experts(E, H, I, 4, 64, fill, device=dev)
    og, ou, od = [], [], []
    for e in range(E):
        for which, lst in (("gate", og), ("up", ou), ("down", od)):
            rows, cols = (I, H) if which != "down" else (H, I)
            buf = np.empty((rows, cols), np.float32)
            fill(which, e, buf)
            lst.append(oracle.quantize(buf, 4, 64))
    x = _massive_x(60, M, H, sigma, chans, big)
    idx = np.array([[m % E, (m + 3) % E, (m + 5) % E] for m in range(M)], np.int32)
    w = np.tile(np.array([0.5, 0.3, 0.2], np.float32), (M, 1))
    _moe_check(dev, x, T(x, dev), idx, w, ex, og, ou, od, what=f"massive sigma={sigma} big={big}")


# ------------- tensor-core path: weights and tokens outside fp16's easy range
#
# The fp16 operands of the tensor-core path are kept in range by power-of-two
# scalings (per weight row, per token row, per SwiGLU row) and groups whose
# zero point is outside the fast form's exact range are dequantised exactly.
# Weights of 1e-3 and 1e-4 (scales far below fp16's normal range),
# single-signed groups (zero points in the thousands and in the millions) and
# bf16 tokens at +-1e5 (beyond fp16's largest finite value) must all meet
# the bf16 bar.

def _domain_experts(dev, E, H, I, kind, seed):
    def fill(which, e, out):
        stream = {"gate": 11, "up": 12, "down": 13}[which] + 10 * e
        if kind in ("tiny3", "tiny4"):
            sigma = 1e-3 if kind == "tiny3" else 1e-4
            out[...] = synth.normal(seed, stream, out.size, sigma).reshape(out.shape)
        elif kind == "offset":
            # gate: all positive around 1 (zp near -4600); up: all negative
            # around -0.5 (zp near +2200); down: 100 + small noise (zp in the
            # millions)
            centre, sig = {"gate": (1.0, 0.01), "up": (-0.5, 0.01), "down": (100.0, 0.001)}[which]
            out[...] = centre + synth.normal(seed, stream, out.size, sig).reshape(out.shape)
        else:
            out[...] = synth.normal(seed, stream, out.size, 0.05).reshape(out.shape)
    ex = q.quantize_experts(E, H, I, 8, 128, fill, device=dev)
    og, ou, od = [], [], []
    for e in range(E):
        for which, lst in (("gate", og), ("up", ou), ("down", od)):
            rows, cols = (I, H) if which != "down" else (H, I)
            buf = np.empty((rows, cols), np.float32)
            fill(which, e, buf)
            lst.append(oracle.quantize(buf, 8, 128))
    return ex, og, ou, od


@pytest.mark.parametrize("kind", ["tiny3", "tiny4", "offset", "big_tokens"])
def test_moe_tensor_core_numeric_domain(dev, kind):
    E, k, H, I, M = 6, 2, 1024, 512, 160
    ex, og, ou, od = _domain_experts(dev, E, H, I, kind, seed=31)
    if kind == "offset":
        zg, zd = og[3].zps, od[3].zps
        assert zg.min() < -3000 and ou[3].zps.max() > 1100 and np.abs(zd).min() > 10 ** 5
    x = synth.normal(32, 1, M * H).reshape(M, H)
    if kind == "big_tokens":
        x[::3, ::97] = 1e5
        x[1::3, 5::101] = -1e5
    x, xd = _bf16_x(x, dev)
    if kind == "big_tokens":
        assert np.abs(x).max() > 65504
    idx = np.zeros((M, k), np.int32)
    idx[:, 0] = 3
    idx[:, 1] = np.where(np.arange(M) % 17 == 0, 1, np.where(np.arange(M) % 5 == 0, 5, 0))
    idx[7, 1] = 2  # one single-token expert (small-M kernels beside the tensor cores)
    w = np.full((M, k), 0.5, np.float32)
    for ydt in (torch.float32, torch.bfloat16):
        _moe_check(dev, x, xd, idx, w, ex, og, ou, od, y_dtype=ydt, what=f"tc {kind} y={ydt}")


# ----------------------------------------------------- routing load check

@pytest.mark.parametrize("M,E,k,zipf", [(512, 256, 6, True), (8, 256, 6, False), (37, 16, 3, True),
                                        (1000, 1024, 8, True)])
def test_route_load_stats(dev, M, E, k, zipf):
    """Load statistics of the router's own histogram, bit-exact against the
    oracle's count of its top-k indices; the overload bit is set exactly when
    the largest count exceeds the threshold."""
    H = 512
    x = synth.normal(70 + M, 1, M * H).reshape(M, H)
    wr = synth.normal(71, 10, E * H, 0.05).reshape(E, H)
    bias = synth.zipf_bias(0, 20, E, 1.1) * 4 if zipf else None
    idx, w, cnt = q.moe_route_topk(T(x, dev), T(wr, dev), None if bias is None else T(bias, dev), k)
    oidx, _ = oracle.topk(oracle.router_logits(x, wr, bias), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), oidx)
    ref, _ = oracle.load_stats(oidx, E, 0)
    for thr in (int(ref[0]) - 1, int(ref[0])):
        q.qmm_device_status(clear=True)
        st = q.moe_route_load_stats(cnt, thr).cpu().numpy()
        np.testing.assert_array_equal(st, ref)
        over = bool(q.qmm_device_status(clear=True) & q.QMM_DEV_EXPERT_OVERLOAD)
        assert over == (ref[0] > thr)


def test_route_load_stats_ties_and_empty(dev):
    """Equal largest counts report the lowest expert; a histogram of zeros
    reports nothing touched."""
    cnt = torch.tensor([0, 5, 2, 5, 0, 5], dtype=torch.int32, device=dev)
    np.testing.assert_array_equal(q.moe_route_load_stats(cnt, 100).cpu().numpy(), [5, 1, 4, 17])
    z = torch.zeros(7, dtype=torch.int32, device=dev)
    np.testing.assert_array_equal(q.moe_route_load_stats(z, 0).cpu().numpy(), [0, 0, 0, 0])
    assert q.qmm_device_status(clear=True) == 0


# ------------------------------------------------------------ bounded waits

def test_bounded_wait_expires_and_reports(dev):
    """A wait that nothing completes gives up after its limit: the kernel
    returns, QMM_DEV_WAIT_TIMEOUT is set, and the device keeps working."""
    import time
    q.qmm_device_status(clear=True)
    t0 = time.time()
    q.qmm_diag_wait_timeout(1_000_000)  # 1 ms
    status = q.qmm_device_status(clear=True)  # synchronises: the kernel returned
    assert status & q.QMM_DEV_WAIT_TIMEOUT
    assert time.time() - t0 < 30
    assert q.qmm_device_status(clear=True) == 0
    # the context is still usable: a linear call afterwards is correct
    w = _weights(64, 256)
    x = synth.normal(80, 1, 256).reshape(1, 256)
    oq = oracle.quantize(w, 8, 64)
    y = q.qmm_linear(T(x, dev), q.qmm_quantize_groupwise(T(w, dev), 8, 64)).cpu().numpy()
    assert_within(y, oracle.linear_fused(x, oq), oracle.linear_bound(x, oq), "after timeout")


# ------------------------------------- batched linear layer on the tensor cores

@pytest.mark.parametrize("M", [9, 16, 33, 64, 200])
@pytest.mark.parametrize("group,N,K", [(64, 1000, 4096), (128, 384, 2048)])
def test_linear_batched_tensor_cores(dev, M, group, N, K):
    """bf16 rows, INT8 codes: the tensor-core linear path (split K, ordered
    reduction of the splits, ragged N) against the oracle at the bf16 bar, for
    fp32 and bf16 outputs; two calls give identical bits."""
    w = _weights(N, K, outl=True, stream=7)
    x, xd = _bf16_x(synth.normal(90 + M, 1, M * K).reshape(M, K), dev)
    oq = oracle.quantize(w, 8, group)
    g = q.qmm_quantize_groupwise(T(w, dev), 8, group)
    assert q.qmm_linear_batched_workspace_bytes(M, g) > 256
    ref = oracle.linear_fused(x, oq)
    y1 = q.qmm_linear_batched(xd, g)
    y2 = q.qmm_linear_batched(xd, g)
    np.testing.assert_array_equal(y1.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert_bf16_rows(y1.cpu().numpy(), ref, f"batched M{M} g{group} N{N}")
    yb = q.qmm_linear_batched(xd, g, y_dtype=torch.bfloat16).float().cpu().numpy()
    assert_bf16_rows(yb, ref, f"batched bf16 out M{M}")


def test_linear_batched_numeric_domain(dev):
    """Tiny and single-signed weights and bf16 rows beyond fp16's range on the
    tensor-core linear path (the power-of-two row scalings and the exact
    dequantisation of far zero points)."""
    M, N, K = 24, 256, 1024
    rows = [synth.normal(95, 7, 64 * K, 1e-4).reshape(64, K),
            1.0 + synth.normal(95, 8, 64 * K, 0.01).reshape(64, K),
            100.0 + synth.normal(95, 9, 64 * K, 0.001).reshape(64, K),
            synth.normal(95, 10, 64 * K, 0.05).reshape(64, K)]
    w = np.concatenate(rows).astype(np.float32)
    xr = synth.normal(96, 1, M * K).reshape(M, K)
    xr[::5, ::61] = 1e5
    x, xd = _bf16_x(xr, dev)
    oq = oracle.quantize(w, 8, 128)
    assert oq.zps.min() < -10 ** 5
    g = q.qmm_quantize_groupwise(T(w, dev), 8, 128)
    y = q.qmm_linear_batched(xd, g).cpu().numpy()
    assert_bf16_rows(y, oracle.linear_fused(x, oq), "batched domain")


def test_linear_batched_falls_back(dev):
    """fp32 rows, or fewer than nine rows, take qmm_linear's CUDA-core paths
    (the fp32 bound) through the same entry point."""
    N, K = 300, 1024
    w = _weights(N, K, stream=9)
    oq = oracle.quantize(w, 8, 64)
    g = q.qmm_quantize_groupwise(T(w, dev), 8, 64)
    for M in (4, 12):
        x = synth.normal(97, 1, M * K).reshape(M, K)
        y = q.qmm_linear_batched(T(x, dev), g).cpu().numpy()
        assert_within(y, oracle.linear_fused(x, oq), oracle.linear_bound(x, oq), f"fallback M{M}")
