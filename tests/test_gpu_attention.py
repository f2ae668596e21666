"""GPU parity of the decode attention step ("Why I hand-wrote a DeepSeek
inference engine in pure C", section 3.4) against the CPU oracle, through the
C ABI: the RoPE table, the cache row the step writes, and the layer output.

Bars: the table within one fp32 ulp of the oracle's (both evaluate the angle
in double; the libraries' double sin/cos may differ in the last double bit);
cache rows and outputs within the oracle's propagated bound (each fp32 stage
held to 1e-5 * sum |terms| + 1e-6, as for the linear layer); rows the step
does not own left untouched bit for bit; repeated calls identical bit for
bit.  The weights are the oracle's quantised codes copied to the device, the
earlier cache rows seeded random values (the same bytes on both sides).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import group_quantized_moe_gb300 as q
from group_quantized_moe_gb300 import build_lib
from parity_checks import assert_within

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


def _to_device(ow, dev):
    """The oracle's quantised weight as a device QWeight (same bytes)."""
    codes = ow.codes.reshape(ow.N, -1)
    if ow.bits == 8:
        codes = codes.view(np.int8)
    return q.QWeight(ow.bits, ow.group, ow.N, ow.K, T(codes, dev), T(ow.scales, dev),
                     T(ow.zps, dev))


def _stacked(ows, dev):
    """The oracle's wq, wk, wv as one device matrix (row-wise quantisation:
    the same bytes as quantising the stacked matrix) and three row views."""
    cat = [np.concatenate([getattr(o, f).reshape(o.N, -1) for o in ows])
           for f in ("codes", "scales", "zps")]
    if ows[0].bits == 8:
        cat[0] = cat[0].view(np.int8)
    N = sum(o.N for o in ows)
    big = q.QWeight(ows[0].bits, ows[0].group, N, ows[0].K, *(T(a, dev) for a in cat))
    out, r = [], 0
    for o in ows:
        out.append(big.rows(r, r + o.N))
        r += o.N
    return out


def _build(dev, seed, D, n_head, n_kv, hd, max_seq, bits=8, group=64, D_out=None,
           base=10000.0, sigma=0.05, stacked=False):
    D_out = D if D_out is None else D_out
    r = synth.normal
    ow = {
        "wq": oracle.quantize(r(seed, 1, n_head * hd * D, sigma).reshape(n_head * hd, D), bits, group),
        "wk": oracle.quantize(r(seed, 2, n_kv * hd * D, sigma).reshape(n_kv * hd, D), bits, group),
        "wv": oracle.quantize(r(seed, 3, n_kv * hd * D, sigma).reshape(n_kv * hd, D), bits, group),
        "wo": oracle.quantize(r(seed, 4, D_out * n_head * hd, sigma).reshape(D_out, n_head * hd),
                              bits, group),
    }
    oc, os_ = oracle.rope_table(max_seq, hd, base)
    gc, gs = q.rope_table(max_seq, hd, base, device=dev)
    if stacked:
        wqkv = _stacked([ow["wq"], ow["wk"], ow["wv"]], dev)
    else:
        wqkv = [_to_device(ow[k], dev) for k in ("wq", "wk", "wv")]
    layer = q.AttnLayer(n_head, n_kv, hd, max_seq, *wqkv, _to_device(ow["wo"], dev), gc, gs)
    return layer, ow, oc, os_


def _cache(seed, n_kv, max_seq, hd):
    return synth.normal(seed, 77, 2 * n_kv * max_seq * hd).reshape(2, n_kv, max_seq, hd)


def _check_step(dev, layer, ow, oc, os_, x, pos, cache, x_bf16=False, y_bf16=False, what=""):
    n_head, n_kv, hd = layer.n_head, layer.n_head_kv, layer.head_dim
    if x_bf16:
        xb = synth.to_bf16(x)
        x = synth.bf16_to_f32(xb)
        xd = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        xd = T(x, dev)
    cd = T(cache, dev)
    y = q.attn_decode(xd, pos, layer, cd, y_dtype=torch.bfloat16 if y_bf16 else torch.float32)
    yref, bound, kv_new, kv_bound = oracle.attn_decode(x, pos, n_head, n_kv, hd, ow["wq"], ow["wk"],
                                                       ow["wv"], ow["wo"], oc, os_, cache)
    got = y.float().cpu().numpy().astype(np.float64)
    if y_bf16:
        bound = bound + np.abs(yref) * 2.0 ** -8
    assert_within(got, yref, bound, f"{what} y pos={pos}")
    c = cd.cpu().numpy()
    assert_within(c[:, :, pos, :].astype(np.float64), kv_new, kv_bound, f"{what} cache row {pos}")
    keep = np.ones(layer.max_seq, bool)
    keep[pos] = False
    np.testing.assert_array_equal(c[:, :, keep, :].view(np.uint32),
                                  cache.astype(np.float32)[:, :, keep, :].view(np.uint32))
    return got


def test_rope_table_matches_oracle(dev):
    for max_seq, hd, base in ((4096, 128, 10000.0), (1024, 512, 10000.0), (300, 6, 500000.0)):
        gc, gs = q.rope_table(max_seq, hd, base, device=dev)
        oc, os_ = oracle.rope_table(max_seq, hd, base)
        for g, o in ((gc, oc), (gs, os_)):
            g = g.cpu().numpy()
            ulp = np.spacing(np.maximum(np.abs(o), np.float32(1e-30)).astype(np.float32))
            assert (np.abs(g - o) <= ulp).all(), (max_seq, hd, base, float(np.abs(g - o).max()))


@pytest.mark.parametrize("n_head,n_kv,hd,bits,group,stacked",
                         [(4, 4, 64, 8, 64, False), (8, 2, 32, 4, 128, True),
                          (6, 1, 128, 8, 32, False), (2, 2, 512, 8, 64, True),
                          (4, 2, 256, 8, 64, True), (16, 16, 4, 8, 64, False)])
def test_attn_decode_positions(dev, n_head, n_kv, hd, bits, group, stacked):
    """Positions at chunk edges (one row, the last row of a chunk, the first
    of the next, a ragged last chunk, the last cache row); head sizes from 4
    to 512; q/k/v weights stored apart (three projection launches) or as one
    stacked matrix (one launch)."""
    D, max_seq = 256, 300
    layer, ow, oc, os_ = _build(dev, 5 + n_head, D, n_head, n_kv, hd, max_seq, bits, group,
                                stacked=stacked)
    cache = _cache(6 + hd, n_kv, max_seq, hd)
    for pos in (0, 1, 63, 64, 65, 130, max_seq - 1):
        x = synth.normal(7 + pos, 1, D)
        _check_step(dev, layer, ow, oc, os_, x, pos, cache, what=f"h{n_head}/{n_kv} d{hd}")


def test_attn_decode_dtypes_and_repeatability(dev):
    D, n_head, n_kv, hd, max_seq, pos = 512, 8, 4, 64, 200, 150
    layer, ow, oc, os_ = _build(dev, 21, D, n_head, n_kv, hd, max_seq, D_out=384)
    cache = _cache(22, n_kv, max_seq, hd)
    x = synth.normal(23, 1, D)
    a = _check_step(dev, layer, ow, oc, os_, x, pos, cache, what="f32")
    b = _check_step(dev, layer, ow, oc, os_, x, pos, cache, what="f32 again")
    np.testing.assert_array_equal(a.view(np.uint64), b.view(np.uint64))
    _check_step(dev, layer, ow, oc, os_, x, pos, cache, x_bf16=True, what="bf16 x")
    _check_step(dev, layer, ow, oc, os_, x, pos, cache, y_bf16=True, what="bf16 y")


def test_attn_decode_sequence_writes_each_row(dev):
    """Steps 0..N-1 in order on one cache: each step's row matches the
    oracle's key / value for that token and position (they depend on the
    token and position only), and no row beyond the last step is touched.
    (The outputs are checked step by step above, on caches whose earlier rows
    are oracle-side inputs, never values the GPU wrote.)"""
    D, n_head, n_kv, hd, max_seq, N = 256, 4, 2, 64, 160, 140
    layer, ow, oc, os_ = _build(dev, 31, D, n_head, n_kv, hd, max_seq)
    cd = layer.kv_cache(dev)
    xs = [synth.normal(32, t, D) for t in range(N)]
    ws = torch.empty((q.qmm_attn_decode_workspace_bytes(layer),), dtype=torch.uint8, device=dev)
    for t in range(N):
        q.attn_decode(T(xs[t], dev), t, layer, cd, workspace=ws)
    c = cd.cpu().numpy()
    for t in (0, 1, 63, 64, 100, N - 1):
        _, _, kv_new, kv_bound = oracle.attn_decode(xs[t], t, n_head, n_kv, hd, ow["wq"], ow["wk"],
                                                    ow["wv"], ow["wo"], oc, os_,
                                                    np.zeros((2, n_kv, max_seq, hd), np.float32))
        assert_within(c[:, :, t, :].astype(np.float64), kv_new, kv_bound, f"row {t}")
    assert (c[:, :, N:, :] == 0).all()


@pytest.mark.slow
def test_attn_decode_full_size(dev):
    """Width 4096, 32 heads of 128 (multi-head), INT8 g64 projections, a
    4096-row cache, the token at position 511 (a 512-token context)."""
    D, n_head, n_kv, hd, max_seq, pos = 4096, 32, 32, 128, 4096, 511
    layer, ow, oc, os_ = _build(dev, 41, D, n_head, n_kv, hd, max_seq, sigma=0.02, stacked=True)
    cache = _cache(42, n_kv, max_seq, hd)
    _check_step(dev, layer, ow, oc, os_, synth.normal(43, 1, D), pos, cache, what="full")


@pytest.mark.slow
def test_attn_decode_grouped_heads_full_width(dev):
    """Grouped heads (8 query heads over one key/value head of 512, as in the
    ds4 walkthrough's 64:1 grouping at a width qmm_linear takes), 2000 rows."""
    D, n_head, n_kv, hd, max_seq, pos = 4096, 8, 1, 512, 2048, 1999
    layer, ow, oc, os_ = _build(dev, 51, D, n_head, n_kv, hd, max_seq, sigma=0.02)
    cache = _cache(52, n_kv, max_seq, hd)
    _check_step(dev, layer, ow, oc, os_, synth.normal(53, 1, D), pos, cache, what="gqa")


def test_attn_decode_rejects_bad_arguments(dev):
    D, n_head, n_kv, hd, max_seq = 128, 4, 2, 32, 16
    layer, ow, oc, os_ = _build(dev, 61, D, n_head, n_kv, hd, max_seq)
    cd = layer.kv_cache(dev)
    x = T(synth.normal(62, 1, D), dev)
    with pytest.raises(q.QmmError):
        q.attn_decode(x, max_seq, layer, cd)          # pos beyond the cache
    with pytest.raises(q.QmmError):
        q.attn_decode(x, -1, layer, cd)
    bad = q.AttnLayer(3, 2, hd, max_seq, layer.wq, layer.wk, layer.wv, layer.wo,
                      layer.rope_cos, layer.rope_sin)
    with pytest.raises(q.QmmError):
        q.attn_decode(x, 0, bad, cd)                  # n_head not a multiple of n_kv
    assert (cd == 0).all()                            # nothing was enqueued


def test_attn_decode_long_cache(dev):
    """Up to 512 rows the chunks of a head merge inside one cluster; from 513
    rows (nine chunks) a merge kernel does it: both sides of that boundary,
    and a long cache."""
    D, n_head, n_kv, hd, max_seq = 256, 4, 2, 64, 1100
    layer, ow, oc, os_ = _build(dev, 81, D, n_head, n_kv, hd, max_seq, stacked=True)
    cache = _cache(82, n_kv, max_seq, hd)
    for pos in (511, 512, 513, 1099):
        _check_step(dev, layer, ow, oc, os_, synth.normal(83 + pos, 1, D), pos, cache,
                    what="long cache")


def test_attn_decode_launches(dev):
    """Stacked q/k/v weights: one projection launch, the attention kernel (its
    chunks merged inside a cluster up to 512 rows, by a second kernel beyond)
    and the output projection; apart: three projection launches.
    quantize_attn_layer builds the stacked form."""
    D, n_head, n_kv, hd, max_seq = 256, 4, 2, 64, 64
    for stacked, expect in ((True, 3), (False, 5)):
        layer, ow, oc, os_ = _build(dev, 71, D, n_head, n_kv, hd, max_seq, stacked=stacked)
        cd = layer.kv_cache(dev)
        x = T(synth.normal(72, 1, D), dev)
        q.attn_decode(x, 3, layer, cd)
        torch.cuda.synchronize()
        n0 = q.qmm_launch_count()
        q.attn_decode(x, 3, layer, cd)
        assert q.qmm_launch_count() - n0 == expect
    wq, wk, wv = (torch.from_numpy(synth.normal(73, i, n * D, 0.05).reshape(n, D)).to(dev)
                  for i, n in enumerate((n_head * hd, n_kv * hd, n_kv * hd)))
    wo = torch.from_numpy(synth.normal(74, 0, D * n_head * hd, 0.05).reshape(D, n_head * hd))
    layer = q.quantize_attn_layer(wq, wk, wv, wo.to(dev), n_head, n_kv, hd, max_seq)
    cd = layer.kv_cache(dev)
    x = T(synth.normal(75, 1, D), dev)
    q.attn_decode(x, 0, layer, cd)
    torch.cuda.synchronize()
    n0 = q.qmm_launch_count()
    q.attn_decode(x, 1, layer, cd)
    assert q.qmm_launch_count() - n0 == 3
