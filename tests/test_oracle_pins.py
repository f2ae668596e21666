"""Pins for the CPU oracle: worked examples, closed forms, invariants and
brute force on tiny inputs.  Nothing here touches a GPU.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a swapped nibble, a transposed operand, the wrong tie
rule) fails at least one of them.
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quantize_worked_examples.txt")


def _parse_examples(path):
    out, cur = [], None
    for line in open(path, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "example":
            cur = {"name": rest}
            out.append(cur)
        else:
            cur[key] = rest
    return out


EXAMPLES = _parse_examples(GOLDEN)


@pytest.mark.parametrize("ex", EXAMPLES, ids=[e["name"] for e in EXAMPLES])
def test_worked_example(ex):
    """Hand-worked fp32 examples of the group-wise scheme (the INT8/INT4
    quantisation section of the pure-C DeepSeek engine article)."""
    bits = int(ex["bits"])
    v = np.array([float(t) for t in ex["values"].split()], dtype=np.float32)
    qw = oracle.quantize(v[None, :], bits, v.size)
    assert qw.scales.view(np.uint32)[0, 0] == int(ex["scale_hex"], 16)
    assert qw.zps[0, 0] == int(ex["zp"])
    codes = [oracle.code_at(qw, 0, k) for k in range(v.size)]
    assert codes == [int(t) for t in ex["codes"].split()]
    assert list(qw.codes) == [int(t, 16) for t in ex["stored_hex"].split()]
    deq = oracle.dequantize(qw)[0]
    want = np.array([float(t) for t in ex["dequant"].split()], dtype=np.float32)
    np.testing.assert_allclose(deq, want, rtol=2e-7, atol=0)


def _weights(seed, stream, N, K, sigma=0.02, outliers=False):
    w = synth.normal(seed, stream, N * K, sigma).reshape(N, K)
    if outliers:
        synth.outliers(seed, stream + 100, w.reshape(-1), 0.01, 20.0)
    return w


@pytest.mark.parametrize("bits,group,N,K,outl", [
    (8, 64, 96, 256, False), (8, 64, 64, 512, True), (8, 128, 40, 512, False),
    (4, 128, 64, 512, False), (4, 64, 33, 256, True), (4, 32, 17, 96, False),
    (8, 2, 5, 8, False), (4, 2, 3, 6, False)])
def test_quantize_invariants(bits, group, N, K, outl):
    """Codes lie in 0..2^b-1; every group's minimum maps to code 0 (roundf is
    odd-symmetric, so round(min/s) + round(-min/s) = 0); the maximum maps to
    2^b-2 or 2^b-1; every element reconstructs within scale/2 (plus fp32
    rounding slack); scales are positive."""
    w = _weights(0, 2, N, K, outliers=outl)
    qw = oracle.quantize(w, bits, group)
    qmax = (1 << bits) - 1
    G = K // group
    q = np.array([[oracle.code_at(qw, n, k) for k in range(K)] for n in range(N)]) \
        if N * K <= 4096 else None
    deq = oracle.dequantize(qw)
    assert (qw.scales > 0).all()
    for n in range(N):
        for j in range(G):
            sl = slice(j * group, (j + 1) * group)
            grp = w[n, sl]
            s = float(qw.scales[n, j])
            err = np.abs(grp.astype(np.float64) - deq[n, sl].astype(np.float64))
            slack = s * (0.5 + 2.0 ** -16) + 2.0 ** -22 * (np.abs(grp) + np.abs(deq[n, sl]))
            assert (err <= slack).all(), (n, j, err.max(), s)
            if q is not None:
                gq = q[n, sl]
                assert gq.min() >= 0 and gq.max() <= qmax
                assert gq[np.argmin(grp)] == 0
                assert gq[np.argmax(grp)] in (qmax - 1, qmax)


def test_int8_storage_is_code_minus_128():
    w = _weights(0, 2, 4, 128)
    qw = oracle.quantize(w, 8, 64)
    stored = qw.codes.view(np.int8).reshape(4, 128).astype(np.int32)
    q = np.array([[oracle.code_at(qw, n, k) for k in range(128)] for n in range(4)])
    assert (q == stored + 128).all()


def test_int4_nibble_order_low_first():
    """Even column in the low nibble: a row whose even entries are the group
    minimum and odd entries the maximum packs to 0xF0 bytes."""
    row = np.array([-1.0, 0.875] * 8, dtype=np.float32)
    qw = oracle.quantize(row[None, :], 4, 16)
    # scale = 1.875 / 15 = 0.125 exactly, zp = round(8) = 8, codes 0 and 15
    assert qw.scales[0, 0] == 0.125 and qw.zps[0, 0] == 8
    assert (qw.codes == 0xF0).all()


def test_fused_equals_two_step():
    """Dequantising inside the k loop equals dequantising the whole matrix
    first and then multiplying (both double, same summation order)."""
    for bits, group in ((8, 64), (4, 128), (4, 32)):
        w = _weights(1, 2, 37, 256)
        x = synth.normal(1, 1, 3 * 256).reshape(3, 256)
        qw = oracle.quantize(w, bits, group)
        a = oracle.linear_fused(x, qw)
        b = oracle.linear_two_step(x, qw)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("bits", [8, 4])
def test_exact_grid_reduces_to_plain_gemv(bits):
    """Weights that lie exactly on a power-of-two grid with both ends present
    in every group quantise losslessly, so the quantised linear layer equals
    the plain matmul of the fp32 weights (computed in float64 by numpy)."""
    rng = np.random.default_rng(7)
    qmax = (1 << bits) - 1
    N, K, group = 12, 256, 64
    s = 2.0 ** -6
    w = np.empty((N, K), dtype=np.float32)
    for n in range(N):
        for j in range(K // group):
            zp = int(rng.integers(0, qmax + 1))
            q = rng.integers(0, qmax + 1, size=group)
            q[rng.integers(0, group)] = 0
            q[(rng.integers(1, group) + np.argmin(q)) % group] = qmax
            w[n, j * group:(j + 1) * group] = (q - zp) * s
    qw = oracle.quantize(w, bits, group)
    np.testing.assert_array_equal(oracle.dequantize(qw), w)
    x = synth.normal(3, 1, 2 * K).reshape(2, K)
    y = oracle.linear_fused(x, qw)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_linear_brute_force_tiny():
    """K=64, N=3: every product written out from the codes, scales and zero
    points read back by index."""
    w = _weights(4, 2, 3, 64)
    x = synth.normal(4, 1, 64)
    for bits in (8, 4):
        qw = oracle.quantize(w, bits, 32)
        y = oracle.linear_fused(x, qw)[0]
        for n in range(3):
            acc = 0.0
            for k in range(64):
                g = k // 32
                wh = np.float32(np.float32(oracle.code_at(qw, n, k) - int(qw.zps[n, g])) * qw.scales[n, g])
                acc += float(x[k]) * float(wh)
            assert y[n] == pytest.approx(acc, rel=1e-13, abs=1e-15)


# --------------------------- tolerance bounds ----------------------------
# The per-output fp32 tolerance of a linear output is 1e-5 * sum_k |x_k w^_k|
# + 1e-6; the MoE tolerance propagates it through SwiGLU and the down
# projection.  They decide every fp32 parity verdict, so they are pinned by
# special cases and properties, not by their formula.


@pytest.mark.parametrize("bits", [8, 4])
def test_linear_bound_one_hot_reads_one_weight(bits):
    """x = c e_k: the bound is 1e-5 |c w^[n,k]| + 1e-6 for every row n (a
    wrong index, a transposed operand or a wrong factor changes it)."""
    N, K = 5, 128
    qw = oracle.quantize(_weights(21, 1, N, K, outliers=True), bits, 32)
    wh = oracle.dequantize(qw).astype(np.float64)
    for k, c in ((0, 2.0), (77, -0.5), (127, 8.0)):
        x = np.zeros(K, np.float32)
        x[k] = c
        b = oracle.linear_bound(x, qw)[0]
        np.testing.assert_allclose(b, 1e-5 * np.abs(c * wh[:, k]) + 1e-6, rtol=1e-14, atol=0)


def test_linear_bound_sign_invariance_and_dominance():
    """Flipping the signs of x leaves the bound unchanged (it sums absolute
    products); it dominates 1e-5 |y| + 1e-6 (triangle inequality), with
    equality when every product x_k w^_k is non-negative."""
    N, K = 4, 256
    qw = oracle.quantize(_weights(22, 1, N, K), 8, 64)
    wh = oracle.dequantize(qw).astype(np.float64)
    x = synth.normal(22, 2, K)
    flip = np.where(synth.normal(22, 3, K) > 0, 1.0, -1.0).astype(np.float32)
    b = oracle.linear_bound(x, qw)[0]
    np.testing.assert_array_equal(oracle.linear_bound(x * flip, qw)[0], b)
    y = oracle.linear_fused(x, qw)[0]
    assert (b - 1e-6 >= 1e-5 * np.abs(y) * (1 - 1e-12)).all()
    assert (b - 1e-6 > 2 * 1e-5 * np.abs(y)).any()  # mixed signs: strictly looser
    for n in range(N):
        xs = (np.abs(x) * np.where(wh[n] >= 0, 1.0, -1.0)).astype(np.float32)
        bn = oracle.linear_bound(xs, qw)[0, n]
        yn = oracle.linear_fused(xs, qw)[0, n]
        assert bn - 1e-6 == pytest.approx(1e-5 * yn, rel=1e-12)


def test_linear_bound_covers_a_plain_fp32_gemv():
    """The tolerance exists for fp32 implementations: a plain fp32 GEMV of
    the dequantised weights (sequential fp32 accumulation, the worst common
    order) stays within it, and the bound is not orders of magnitude loose."""
    N, K = 16, 4096
    qw = oracle.quantize(_weights(23, 1, N, K, outliers=True), 8, 64)
    wh = oracle.dequantize(qw)
    x = synth.normal(23, 2, K)
    y = oracle.linear_fused(x, qw)[0]
    b = oracle.linear_bound(x, qw)[0]
    y32 = np.zeros(N, np.float32)
    for k in range(K):
        y32 = (y32 + x[k] * wh[:, k]).astype(np.float32)
    err = np.abs(y32.astype(np.float64) - y)
    assert (err <= b).all()
    sabs = (b - 1e-6) / 1e-5
    assert (b < 1e-3 * sabs + 1e-6).all()


def _moe_case(seed, k=2, M=3, E=4, H=64, I=32):
    gate, up, down = _experts(seed, E, H, I, 8, 32)
    x = synth.normal(seed, 1, M * H).reshape(M, H)
    idx = np.array([[(m + i) % E for i in range(k)] for m in range(M)], np.int32)
    return x, idx, gate, up, down


def test_moe_bound_homogeneous_and_additive_in_routing_weights():
    """With no routing-weight error (dw = 0) every slot adds |w_i| times its
    own propagated bound: scaling w by c scales the bound (less the 1e-6
    floor) by |c|, and the slots' contributions add."""
    x, idx, gate, up, down = _moe_case(31)
    w = np.array([[0.75, 0.25], [0.5, 0.5], [0.125, 0.875]], np.float32)
    _, b = oracle.moe_ffn(x, idx, w, gate, up, down)
    _, b2 = oracle.moe_ffn(x, idx, (-2 * w).astype(np.float32), gate, up, down)
    np.testing.assert_allclose(b2 - 1e-6, 2 * (b - 1e-6), rtol=1e-12)
    w0 = w.copy()
    w0[:, 1] = 0
    w1 = w.copy()
    w1[:, 0] = 0
    _, ba = oracle.moe_ffn(x, idx, w0, gate, up, down)
    _, bb = oracle.moe_ffn(x, idx, w1, gate, up, down)
    np.testing.assert_allclose(b - 1e-6, (ba - 1e-6) + (bb - 1e-6), rtol=1e-12)


def test_moe_bound_routing_weight_term():
    """The routing-weight error dw adds dw |o_i| per slot, o_i the slot's
    expert output (read off with one-hot weights), not dw |sum_i o_i|."""
    x, idx, gate, up, down = _moe_case(32)
    w = np.array([[0.6, 0.4], [0.3, 0.7], [0.9, 0.1]], np.float32)
    dw = 2e-6
    _, b0 = oracle.moe_ffn(x, idx, w, gate, up, down)
    _, b1 = oracle.moe_ffn(x, idx, w, gate, up, down, dw=dw)
    e0 = np.zeros_like(w)
    e0[:, 0] = 1
    e1 = np.zeros_like(w)
    e1[:, 1] = 1
    o0, _ = oracle.moe_ffn(x, idx, e0, gate, up, down)
    o1, _ = oracle.moe_ffn(x, idx, e1, gate, up, down)
    np.testing.assert_allclose(b1 - b0, dw * (np.abs(o0) + np.abs(o1)), rtol=1e-9, atol=1e-20)


def test_moe_bound_first_order_propagation_through_swiglu():
    """One expert, one slot, w = 1, and a diagonal down matrix (each group
    holds one nonzero and zeros, which the quantiser keeps exactly): output n
    depends on h_n = silu(g_n) u_n alone, so its bound is 1e-6 + 1e-5 |wd h_n|
    + |wd| dh_n + 1e-6, where dh_n, the first-order error of h_n, must equal
    the largest change of silu(g) u when g and u move by their own linear
    bounds (found here by perturbation, not by a derivative formula), plus
    the 1e-6 |h_n| of h's own rounding."""
    H = I = 64
    gate = [oracle.quantize(_weights(34, 1, I, H), 8, 32)]
    up = [oracle.quantize(_weights(34, 2, I, H), 8, 32)]
    v = np.array([0.02 * (1 + n % 5) * (-1) ** n for n in range(H)], np.float32)
    down = [oracle.quantize(np.diag(v).astype(np.float32), 8, 32)]
    wd = oracle.dequantize(down[0]).astype(np.float64)
    np.testing.assert_array_equal(wd - np.diag(np.diag(wd)), 0)
    assert (np.abs(np.diag(wd) - v) <= 1e-3 * np.abs(v)).all()
    x = synth.normal(34, 3, 2 * H).reshape(2, H)
    y, b = oracle.moe_ffn(x, np.zeros((2, 1), np.int32), np.ones((2, 1), np.float32),
                          gate, up, down)
    g, u = oracle.linear_fused(x, gate[0]), oracle.linear_fused(x, up[0])
    dg, du = oracle.linear_bound(x, gate[0]), oracle.linear_bound(x, up[0])
    h = _silu(g) * u
    moved = [np.abs(_silu(g + sg * dg) * (u + su * du) - h) for sg in (1, -1) for su in (1, -1)]
    dh = np.max(moved, axis=0) + 1e-6 * np.abs(h)
    d = np.abs(np.diag(wd))
    np.testing.assert_allclose(y, np.diag(wd)[None, :] * h, rtol=1e-12)
    expect = 1e-6 + 1e-5 * d[None, :] * np.abs(h) + d[None, :] * dh + 1e-6
    np.testing.assert_allclose(b, expect, rtol=1e-4)


def test_moe_bound_covers_an_fp32_layer():
    """An fp32 evaluation of the same layer (fp32 GEMVs of the dequantised
    weights, SwiGLU and the combine in fp32) stays within the MoE bound, and
    the bound is not orders of magnitude above the error scale it models."""
    E, H, I, k, M = 4, 1024, 512, 2, 3
    gate, up, down = _experts(33, E, H, I, 8, 64)
    x = synth.normal(33, 1, M * H).reshape(M, H)
    idx = np.array([[0, 1], [2, 3], [1, 3]], np.int32)
    w = np.array([[0.7, 0.3], [0.45, 0.55], [0.2, 0.8]], np.float32)
    y, b = oracle.moe_ffn(x, idx, w, gate, up, down)
    deq = lambda q: oracle.dequantize(q)
    for m in range(M):
        acc = np.zeros(H, np.float32)
        for i in range(k):
            e = idx[m, i]
            g = (deq(gate[e]) @ x[m]).astype(np.float32)
            u = (deq(up[e]) @ x[m]).astype(np.float32)
            h = (g / (np.float32(1) + np.exp(-g)) * u).astype(np.float32)
            acc = (acc + w[m, i] * (deq(down[e]) @ h)).astype(np.float32)
        err = np.abs(acc.astype(np.float64) - y[m])
        assert (err <= b[m]).all()
        assert (b[m] < 1e-2 * (np.abs(y[m]).max() + 1e-3)).all()


# --------------------------- router ------------------------------------


def _brute_topk(logits, k):
    """All k-subsets: the selected set is the one whose every member beats
    every non-member under (larger logit, then lower index)."""
    E = logits.size
    key = lambda e: (-float(logits[e]), e)
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if all(key(a) < key(b) for a in S for b in rest):
            return sorted(S, key=key)
    raise AssertionError("no dominating subset")


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(11)
    for trial in range(60):
        base = rng.normal(size=8).astype(np.float32)
        # plant exact ties
        dup = rng.integers(0, 8, size=3)
        base[dup[1]] = base[dup[0]]
        base[dup[2]] = base[dup[0]]
        if trial % 5 == 0:
            base[:] = 0.25  # all equal -> indices 0, 1, 2
        idx, w = oracle.topk(base[None, :], 3)
        assert list(idx[0]) == _brute_topk(base, 3)
    idx, _ = oracle.topk(np.full((1, 8), 0.25, np.float32), 3)
    assert list(idx[0]) == [0, 1, 2]


def test_topk_weights_closed_form():
    """Renormalised weights sum to 1 and equal a softmax over the k selected
    logits alone (the full-softmax denominator cancels)."""
    logits = synth.normal(5, 30, 16 * 256, 2.0).reshape(16, 256)
    idx, w = oracle.topk(logits, 6)
    sel = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), axis=1)
    ref = np.exp(sel - sel.max(axis=1, keepdims=True))
    ref /= ref.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, ref, rtol=2e-7, atol=1e-9)
    np.testing.assert_allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert (np.diff(sel, axis=1) <= 0).all()


def test_topk_softmax_survives_large_logits():
    """Maximum subtracted before exp (article section on attention softmax):
    logits near 1e4 still give finite weights."""
    l = np.array([[1e4, 1e4 - 1, 1e4 - 2, 0, 1, 2, 3, 4]], dtype=np.float32)
    idx, w = oracle.topk(l, 3)
    assert list(idx[0]) == [0, 1, 2]
    e = np.exp([0.0, -1.0, -2.0])
    np.testing.assert_allclose(w[0], e / e.sum(), rtol=1e-6)


def test_router_logits_match_float64_dot():
    """The fixed-order fp32 sum is a dot product: it lies within the fp32
    error bound of the float64 dot (gamma_n * sum |x w|), bias added last."""
    M, H, E = 5, 4096, 256
    x = synth.normal(6, 1, M * H).reshape(M, H)
    wr = synth.normal(6, 10, E * H, 0.02).reshape(E, H)
    bias = synth.zipf_bias(6, 20, E, 1.1)
    l = oracle.router_logits(x, wr, bias)
    exact = x.astype(np.float64) @ wr.astype(np.float64).T
    absd = np.abs(x.astype(np.float64)) @ np.abs(wr.astype(np.float64)).T
    gamma = (32 + 8) * 2.0 ** -24
    err = np.abs(l.astype(np.float64) - bias.astype(np.float64) - exact)
    assert (err <= gamma * absd + 4 * 2.0 ** -24 * np.abs(l)).all()


def test_router_one_hot_input_reads_one_weight():
    """x = e_j gives logit[e] = Wr[e, j] + bias[e] exactly (one nonzero
    product, every other partial is an exact zero)."""
    H, E = 512, 16
    wr = synth.normal(8, 10, E * H, 0.02).reshape(E, H)
    bias = synth.normal(8, 21, E)
    for j in (0, 1, 127, 128, 300, 511):
        x = np.zeros((1, H), np.float32)
        x[0, j] = 1.0
        l = oracle.router_logits(x, wr, bias)[0]
        np.testing.assert_array_equal(l, (wr[:, j] + bias).astype(np.float32))
        l0 = oracle.router_logits(x, wr, None)[0]
        np.testing.assert_array_equal(l0, wr[:, j])


def test_router_expert_permutation_equivariance():
    M, H, E = 4, 256, 32
    x = synth.normal(9, 1, M * H).reshape(M, H)
    wr = synth.normal(9, 10, E * H, 0.02).reshape(E, H)
    bias = synth.normal(9, 21, E, 0.5)
    perm = synth.permutation(9, 22, E)
    l = oracle.router_logits(x, wr, bias)
    lp = oracle.router_logits(x, wr[perm], bias[perm])
    np.testing.assert_array_equal(lp, l[:, perm])
    idx, w = oracle.topk(l, 6)
    idxp, wp = oracle.topk(lp, 6)
    np.testing.assert_array_equal(perm[idxp], idx)
    np.testing.assert_array_equal(wp, w)


def test_router_summation_order_worked_examples():
    """The logit's fixed fp32 order, worked by hand: partial p is one fma
    chain over h = p, p + 128, ...; level 1 sums (P0 + P1) + (P2 + P3) per four
    partials; then t_l += t_{l+o} for o = 16, 8, 4, 2, 1; the bias is added
    last.  Each row puts exact products where only that order gives the
    stated logit (2^24 + 1 rounds to 2^24: a tie, to even)."""
    H, big = 256, np.float32(2.0 ** 24)
    wr = np.ones((2, H), np.float32)
    a = np.float32(1 + 2.0 ** -12)
    wr[1, 128] = a
    x = np.zeros((5, H), np.float32)
    # A: x0 w0 = -1, x128 w128 = (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24.  One fma
    # on -1 keeps 2^-11 + 2^-24 exactly; a rounded product first gives 2^-11.
    x[0, 0], x[0, 128] = -1, a
    # B: 2^24 (h = 0), -2^24 (h = 1), 1 (h = 128).  With 128 partials h = 128
    # joins partial 0: 2^24 + 1 -> 2^24, then 2^24 - 2^24 = 0.  (127 partials
    # would put h = 128 with h = 1: -2^24 + 1 exactly, logit 1.)
    x[1, 0], x[1, 1], x[1, 128] = big, -big, 1
    # C: P0..P3 = 2^24, 1, 1, -2^24.  (P0 + P1) + (P2 + P3) = 2^24 + (1 - 2^24)
    # = 1; ((P0 + P1) + P2) + P3 = 0.
    x[2, 0:4] = [big, 1, 1, -big]
    # D: t0 = 2^24, t8 = -2^24, t16 = 1, t24 = 1 (partials 0, 32, 64, 96).  o =
    # 16: t0 = 2^24 + 1 -> 2^24, t8 = -2^24 + 1; o = 8: t0 = 1.  A sequential
    # or reversed (o = 1 first) tree gives 2.
    x[3, 0], x[3, 32], x[3, 64], x[3, 96] = big, -big, 1, 1
    # E: 2^24 - 2^24 = 0 in the tree; the bias (1) comes after it.  Added into
    # partial 0 instead it would vanish in 2^24 + 1.
    x[4, 0], x[4, 1] = big, -big
    lg = oracle.router_logits(x, wr, None)
    assert lg[0, 1] == np.float32(2.0 ** -11 + 2.0 ** -24)
    assert lg[0, 0] == np.float32(2.0 ** -12)
    assert lg[1:, 0].tolist() == [0.0, 1.0, 1.0, 0.0]
    lb = oracle.router_logits(x, wr, np.array([1.0, 0.0], np.float32))
    assert lb[1:, 0].tolist() == [1.0, 2.0, 2.0, 1.0]


def test_router_partial_order_is_fixed():
    """The summation order is part of the definition: reversing the columns
    generally changes low bits (shows the test above is not vacuous) but
    the result stays within the fp32 bound."""
    H = 4096
    x = synth.normal(10, 1, H)[None, :]
    wr = synth.normal(10, 10, 64 * H, 0.02).reshape(64, H)
    a = oracle.router_logits(x, wr, None)
    b = oracle.router_logits(x[:, ::-1], wr[:, ::-1], None)
    assert not np.array_equal(a, b)
    np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-5)


# ----------------------------- MoE FFN ---------------------------------


def _experts(seed, E, H, I, bits, group):
    gate = [oracle.quantize(_weights(seed, 11 + 10 * e, I, H), bits, group) for e in range(E)]
    up = [oracle.quantize(_weights(seed, 12 + 10 * e, I, H), bits, group) for e in range(E)]
    down = [oracle.quantize(_weights(seed, 13 + 10 * e, H, I), bits, group) for e in range(E)]
    return gate, up, down


def _silu(a):
    return a / (1.0 + np.exp(-a))


def test_moe_single_expert_reduces_to_swiglu_of_linears():
    H, I = 128, 64
    gate, up, down = _experts(12, 1, H, I, 8, 32)
    x = synth.normal(12, 1, 3 * H).reshape(3, H)
    idx = np.zeros((3, 1), np.int32)
    w = np.ones((3, 1), np.float32)
    y, _ = oracle.moe_ffn(x, idx, w, gate, up, down)
    g = oracle.linear_fused(x, gate[0])
    u = oracle.linear_fused(x, up[0])
    h = _silu(g) * u
    wd = oracle.dequantize(down[0]).astype(np.float64)
    np.testing.assert_allclose(y, h @ wd.T, rtol=1e-12, atol=1e-14)


def test_moe_dense_brute_force():
    """Tiny routed layer against a dense float64 computation from the
    dequantised matrices: y = sum_i w_i * (silu(x Wg^T) * (x Wu^T)) Wd^T."""
    E, H, I, k, M = 6, 64, 32, 3, 5
    gate, up, down = _experts(13, E, H, I, 4, 32)
    x = synth.normal(13, 1, M * H).reshape(M, H)
    wr = synth.normal(13, 10, E * H, 0.1).reshape(E, H)
    idx, w = oracle.topk(oracle.router_logits(x, wr, None), k)
    y, bound = oracle.moe_ffn(x, idx, w, gate, up, down)
    xd = x.astype(np.float64)
    for m in range(M):
        ref = np.zeros(H)
        for i in range(k):
            e = idx[m, i]
            g = oracle.dequantize(gate[e]).astype(np.float64) @ xd[m]
            u = oracle.dequantize(up[e]).astype(np.float64) @ xd[m]
            ref += float(w[m, i]) * (oracle.dequantize(down[e]).astype(np.float64) @ (_silu(g) * u))
        np.testing.assert_allclose(y[m], ref, rtol=1e-11, atol=1e-13)
    assert (bound > 1e-6).all()


def test_moe_linear_in_routing_weights_and_token_order():
    E, H, I, k, M = 4, 64, 32, 2, 4
    gate, up, down = _experts(14, E, H, I, 8, 32)
    x = synth.normal(14, 1, M * H).reshape(M, H)
    idx = np.array([[0, 1], [2, 3], [1, 2], [3, 0]], np.int32)
    w = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1], [0.2, 0.8]], np.float32)
    y, _ = oracle.moe_ffn(x, idx, w, gate, up, down)
    y2, _ = oracle.moe_ffn(x, idx, (w * 2).astype(np.float32), gate, up, down)
    np.testing.assert_allclose(y2, 2 * y, rtol=1e-12, atol=1e-15)
    p = np.array([2, 0, 3, 1])
    y3, _ = oracle.moe_ffn(x[p], idx[p], w[p], gate, up, down)
    np.testing.assert_array_equal(y3, y[p])


# ------------------------------------------------------- routing load check

def test_load_stats_worked_examples():
    """The load check of the engine's MoE layer (the warning when one expert
    is chosen more often than a threshold), worked by hand."""
    # 3 tokens, k = 2, E = 5: expert 2 three times, 1 twice, 3 once
    idx = np.array([[1, 2], [2, 3], [2, 1]], np.int32)
    st, flag = oracle.load_stats(idx, 5, 2)
    assert st.tolist() == [3, 2, 3, 6] and flag
    st, flag = oracle.load_stats(idx, 5, 3)
    assert st.tolist() == [3, 2, 3, 6] and not flag
    # equal largest counts: the lower expert index is reported
    st, _ = oracle.load_stats(np.array([[4, 1], [1, 4]], np.int32), 5, 10)
    assert st.tolist() == [2, 1, 2, 4]
    # an index outside [0, E) is not counted
    st, flag = oracle.load_stats(np.array([[0, 7], [-1, 0]], np.int32), 5, 1)
    assert st.tolist() == [2, 0, 1, 2] and flag
    # every token on one expert: the largest count is M
    st, _ = oracle.load_stats(np.full((9, 1), 3, np.int32), 8, 100)
    assert st.tolist() == [9, 3, 1, 9]
