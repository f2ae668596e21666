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
