"""Pins for the oracle's decode attention ("Why I hand-wrote a DeepSeek
inference engine in pure C", section 3.4: rotary positions from a
precomputed [max_seq, head_dim/2] cos/sin table, softmax(q k^T / sqrt(d))
with the maximum subtracted, the KV cache).  Closed forms, invariants and
brute force on tiny inputs; nothing here touches a GPU.

Each check is chosen so that a plausible slip (pairing i with i + d/2
instead of 2i + 1, a sign of the sine, the frequency exponent, a missing
1/sqrt(d), the wrong key/value head for grouped queries, reading one cache
row too many or too few, a wrong row for the step's own key) fails one.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ RoPE table

def test_rope_table_position_zero_is_identity():
    c, s = oracle.rope_table(4, 16)
    assert (c[0] == 1.0).all() and (s[0] == 0.0).all()


def test_rope_table_closed_forms():
    """head_dim 4, base 10000: theta_0 = 1 and theta_1 = 10000^(-1/2) = 0.01,
    so row p holds cos/sin of p and of p / 100 (rounded to fp32)."""
    c, s = oracle.rope_table(50, 4, 10000.0)
    for p in (1, 2, 7, 49):
        assert c[p, 0] == np.float32(math.cos(p)) and s[p, 0] == np.float32(math.sin(p))
        assert c[p, 1] == np.float32(math.cos(p / 100.0))
        assert s[p, 1] == np.float32(math.sin(p / 100.0))


def test_rope_table_frequencies_decrease_geometrically():
    """At a small position the angle of pair i is pos * base^(-2i/d): the ratio
    of consecutive angles is base^(-2/d) (sin ~ angle there)."""
    d, base = 64, 10000.0
    c, s = oracle.rope_table(2, d, base)
    ang = np.arctan2(s[1].astype(np.float64), c[1].astype(np.float64))
    ratio = ang[1:] / ang[:-1]
    np.testing.assert_allclose(ratio, base ** (-2.0 / d), rtol=1e-6)


# --------------------------------------------------------------- RoPE rotation

def test_rope_pairs_are_adjacent_and_rotate_counterclockwise():
    """(1, 0) in pair i goes to (cos, sin) of that pair's angle; (0, 1) to
    (-sin, cos); the other pairs are untouched."""
    c, s = oracle.rope_table(10, 8)
    for i in range(4):
        e = np.zeros((1, 8))
        e[0, 2 * i] = 1.0
        r = oracle.rope_apply(e, 5, c, s)
        exp = np.zeros(8)
        exp[2 * i], exp[2 * i + 1] = c[5, i], s[5, i]
        np.testing.assert_array_equal(r[0], exp)
        e = np.zeros((1, 8))
        e[0, 2 * i + 1] = 1.0
        r = oracle.rope_apply(e, 5, c, s)
        exp = np.zeros(8)
        exp[2 * i], exp[2 * i + 1] = -s[5, i], c[5, i]
        np.testing.assert_array_equal(r[0], exp)


def test_rope_preserves_pair_norms_and_composes():
    d, P = 32, 40
    c, s = oracle.rope_table(2 * P, d)
    x = _rng(1).normal(size=(3, d))
    for a, b in ((3, 5), (0, 17), (11, 28)):
        ra = oracle.rope_apply(x, a, c, s)
        n0 = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
        n1 = ra[:, 0::2] ** 2 + ra[:, 1::2] ** 2
        np.testing.assert_allclose(n1, n0, rtol=3e-7)
        # R_b R_a = R_{a+b} (the table's fp32 rounding leaves ~1e-7)
        rab = oracle.rope_apply(ra, b, c, s)
        np.testing.assert_allclose(rab, oracle.rope_apply(x, a + b, c, s), atol=2e-6)


def test_rope_dot_products_depend_on_relative_position_only():
    """<R_m q, R_n k> = <R_(m-n) q, k>: the property that makes RoPE encode
    relative positions."""
    d = 16
    c, s = oracle.rope_table(64, d)
    q, k = _rng(2).normal(size=(2, 1, d))
    for m, n in ((9, 4), (30, 30), (63, 1)):
        lhs = float(oracle.rope_apply(q, m, c, s)[0] @ oracle.rope_apply(k, n, c, s)[0])
        rhs = float(oracle.rope_apply(q, m - n, c, s)[0] @ k[0])
        assert abs(lhs - rhs) <= 1e-5 * (np.abs(q).sum() * np.abs(k).sum())


# ------------------------------------------------------------------- attention

def _softmax_attention_numpy(q, K, V):
    """Brute force for one head: library softmax over q.K^T / sqrt(d)."""
    from scipy.special import softmax
    sc = (K @ q) / math.sqrt(q.shape[0])
    return softmax(sc) @ V


@pytest.mark.parametrize("n_head,n_kv,T", [(1, 1, 1), (2, 2, 5), (4, 2, 7), (6, 1, 3)])
def test_attention_brute_force(n_head, n_kv, T):
    hd, max_seq = 8, 9
    r = _rng(10 + n_head + T)
    q = r.normal(size=(n_head, hd))
    kc = r.normal(size=(n_kv, max_seq, hd)).astype(np.float32)
    vc = r.normal(size=(n_kv, max_seq, hd)).astype(np.float32)
    out, bound = oracle.attention(q, kc, vc, T)
    grp = n_head // n_kv
    for h in range(n_head):
        ref = _softmax_attention_numpy(q[h], kc[h // grp, :T].astype(np.float64),
                                       vc[h // grp, :T].astype(np.float64))
        np.testing.assert_allclose(out[h], ref, rtol=1e-12, atol=1e-12)
    assert (bound > 0).all()


def test_attention_single_row_returns_its_value():
    hd = 16
    r = _rng(3)
    kc = r.normal(size=(1, 4, hd)).astype(np.float32)
    vc = r.normal(size=(1, 4, hd)).astype(np.float32)
    out, _ = oracle.attention(r.normal(size=(3, hd)), kc, vc, 1)
    for h in range(3):
        np.testing.assert_array_equal(out[h], vc[0, 0].astype(np.float64))


def test_attention_equal_keys_average_the_values():
    hd, T = 8, 6
    r = _rng(4)
    kc = np.tile(r.normal(size=(1, 1, hd)), (1, T, 1)).astype(np.float32)
    vc = r.normal(size=(1, T, hd)).astype(np.float32)
    out, _ = oracle.attention(r.normal(size=(1, hd)), kc, vc, T)
    np.testing.assert_allclose(out[0], vc[0].astype(np.float64).mean(axis=0), rtol=1e-12,
                               atol=1e-14)


def test_attention_large_scores_pick_the_best_row():
    """Scores of order 1e4: without the maximum subtracted exp overflows; with
    it the output is the best-matching row's value."""
    hd, T = 4, 5
    kc = np.zeros((1, T, hd), np.float32)
    for t in range(T):
        kc[0, t, 0] = float(t)
    vc = np.arange(T * hd, dtype=np.float32).reshape(1, T, hd)
    q = np.array([[2e4, 0, 0, 0]])
    out, _ = oracle.attention(q, kc, vc, T)
    np.testing.assert_allclose(out[0], vc[0, T - 1], rtol=0, atol=1e-9)


def test_attention_reads_rows_before_T_only_and_permutation_invariant():
    hd, T, max_seq = 8, 5, 8
    r = _rng(5)
    q = r.normal(size=(2, hd))
    kc = r.normal(size=(1, max_seq, hd)).astype(np.float32)
    vc = r.normal(size=(1, max_seq, hd)).astype(np.float32)
    out, _ = oracle.attention(q, kc, vc, T)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, T:] = 1e6
    vc2[:, T:] = np.nan
    out2, _ = oracle.attention(q, kc2, vc2, T)
    np.testing.assert_array_equal(out, out2)
    perm = np.array([3, 0, 4, 1, 2])
    kc3, vc3 = kc.copy(), vc.copy()
    kc3[:, :T] = kc[:, perm]
    vc3[:, :T] = vc[:, perm]
    out3, _ = oracle.attention(q, kc3, vc3, T)
    np.testing.assert_allclose(out3, out, rtol=1e-13, atol=1e-14)


def test_attention_last_row_override():
    """k_last / v_last replace row T-1 (the row the decode step writes)."""
    hd, T = 8, 4
    r = _rng(6)
    q = r.normal(size=(2, hd))
    kc = r.normal(size=(1, 6, hd)).astype(np.float32)
    vc = r.normal(size=(1, 6, hd)).astype(np.float32)
    kl, vl = r.normal(size=(1, hd)), r.normal(size=(1, hd))
    out, _ = oracle.attention(q, kc, vc, T, k_last=kl, v_last=vl)
    kc2, vc2 = kc.astype(np.float64), vc.astype(np.float64)
    kc2[0, T - 1], vc2[0, T - 1] = kl[0], vl[0]
    for h in range(2):
        np.testing.assert_allclose(out[h], _softmax_attention_numpy(q[h], kc2[0, :T], vc2[0, :T]),
                                   rtol=1e-12, atol=1e-13)


def test_attention_bound_grows_with_input_error():
    hd, T = 8, 5
    r = _rng(7)
    q = r.normal(size=(1, hd))
    kc = r.normal(size=(1, T, hd)).astype(np.float32)
    vc = r.normal(size=(1, T, hd)).astype(np.float32)
    _, b0 = oracle.attention(q, kc, vc, T)
    _, b1 = oracle.attention(q, kc, vc, T, dq=np.full((1, hd), 1e-3))
    assert (b1 > b0).all()
    # the bound covers a real perturbation of q of that size
    out, _ = oracle.attention(q, kc, vc, T)
    outp, _ = oracle.attention(q + 1e-3 * np.sign(r.normal(size=q.shape)), kc, vc, T)
    assert (np.abs(outp - out) <= b1).all()


# ------------------------------------------------------------- the decode step

def _layer(seed, D, n_head, n_kv, hd, bits=8, group=64):
    r = synth.normal
    wq = oracle.quantize(r(seed, 1, n_head * hd * D, 0.05).reshape(n_head * hd, D), bits, group)
    wk = oracle.quantize(r(seed, 2, n_kv * hd * D, 0.05).reshape(n_kv * hd, D), bits, group)
    wv = oracle.quantize(r(seed, 3, n_kv * hd * D, 0.05).reshape(n_kv * hd, D), bits, group)
    wo = oracle.quantize(r(seed, 4, D * n_head * hd, 0.05).reshape(D, n_head * hd), bits, group)
    return wq, wk, wv, wo


def test_attn_decode_position_zero_is_output_of_value():
    """At pos 0 the only cache row is the step's own: attention returns v and
    y = Wo (Wv x), whatever the query, key and rotation."""
    D, n_head, n_kv, hd = 128, 4, 2, 16
    wq, wk, wv, wo = _layer(11, D, n_head, n_kv, hd)
    x = synth.normal(12, 1, D)
    c, s = oracle.rope_table(8, hd)
    cache = np.full((2, n_kv, 8, hd), np.nan, np.float32)
    y, bound, kv_new, _ = oracle.attn_decode(x, 0, n_head, n_kv, hd, wq, wk, wv, wo, c, s, cache)
    v = oracle.linear_fused(x[None, :], wv)[0]
    attn = np.repeat(v.reshape(n_kv, hd), n_head // n_kv, axis=0).reshape(-1)
    ref = oracle.linear_fused(attn.astype(np.float32)[None, :], wo)[0]
    np.testing.assert_allclose(y, ref, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(kv_new[1].reshape(-1), v, rtol=1e-15)
    k = oracle.linear_fused(x[None, :], wk)[0].reshape(n_kv, hd)
    np.testing.assert_allclose(kv_new[0], k, rtol=1e-15)   # rotation by 0 is the identity
    assert (bound > 0).all()


def test_attn_decode_wiring_matches_the_steps():
    """pos > 0: the layer equals projections, rotation of q and the new k,
    attention over the cache with row pos replaced, output projection."""
    D, n_head, n_kv, hd, max_seq, pos = 128, 4, 2, 16, 12, 7
    wq, wk, wv, wo = _layer(13, D, n_head, n_kv, hd)
    x = synth.normal(14, 1, D)
    c, s = oracle.rope_table(max_seq, hd)
    cache = synth.normal(15, 1, 2 * n_kv * max_seq * hd).reshape(2, n_kv, max_seq, hd)
    y, bound, kv_new, _ = oracle.attn_decode(x, pos, n_head, n_kv, hd, wq, wk, wv, wo, c, s, cache)
    q = oracle.linear_fused(x[None, :], wq)[0].reshape(n_head, hd)
    k = oracle.linear_fused(x[None, :], wk)[0].reshape(n_kv, hd)
    v = oracle.linear_fused(x[None, :], wv)[0].reshape(n_kv, hd)
    qr, kr = oracle.rope_apply(q, pos, c, s), oracle.rope_apply(k, pos, c, s)
    a, _ = oracle.attention(qr, cache[0], cache[1], pos + 1, k_last=kr, v_last=v)
    ref = oracle.linear_fused(a.reshape(1, -1).astype(np.float32), wo)[0]
    # the oracle feeds the double attention output to Wo; the check rounds it
    # to fp32 first, so they agree to that rounding (relative 2^-24 of each term)
    sum_abs = np.abs(a.reshape(1, -1)) @ np.abs(oracle.dequantize(wo)).T
    assert (np.abs(y - ref) <= 1e-7 * sum_abs[0] + 1e-12).all()
    np.testing.assert_allclose(kv_new[0], kr, rtol=1e-15)
    np.testing.assert_allclose(kv_new[1], v, rtol=1e-15)
