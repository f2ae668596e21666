"""The seeded input generator shared by the oracle and the GPU tests.

It holds none of the method's arithmetic, but every parity case and every
sampled full-size check depends on it regenerating any element range on its
own: these tests pin it to its published definition (SplitMix64, the inverse
normal CDF of one uniform per element, an independent outlier stream) and to
the properties the tests rely on.
"""
import numpy as np
import pytest

import synth
from synth import recipes

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def _mix64(z):
    # SplitMix64 finaliser (Steele, Lea, Flood, OOPSLA 2014)
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_raw_is_splitmix64():
    # seed 0, stream 0 starts the sequence at state 0: the published first
    # outputs of SplitMix64 seeded with 0
    assert [synth.raw(0, 0, c) for c in range(3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    for seed, stream in ((3, 5), (0, 100), (12345, 1)):
        key = _mix64(seed ^ ((stream * GAMMA) & M64))
        for c in (0, 1, 7, 1 << 40):
            assert synth.raw(seed, stream, c) == _mix64((key + (c + 1) * GAMMA) & M64)


def test_normal_is_the_inverse_cdf_of_one_uniform_per_element():
    special = pytest.importorskip("scipy.special")
    seed, stream, sigma, n = 3, 5, 0.02, 200
    got = synth.normal(seed, stream, n, sigma)
    r = np.array([synth.raw(seed, stream, c) for c in range(n)], dtype=np.uint64)
    u = (2.0 * (r >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -54
    want = (sigma * special.ndtri(u)).astype(np.float32)
    # Acklam's approximation is within 1.15e-9 relative: at most one fp32 ulp
    np.testing.assert_array_max_ulp(got, want, maxulp=1)


def test_any_range_regenerates_on_its_own():
    full = synth.normal(7, 2, 10000, 1.0)
    for off, cnt in ((0, 1), (1, 99), (4095, 3000), (9999, 1)):
        np.testing.assert_array_equal(synth.normal(7, 2, cnt, 1.0, offset=off), full[off:off + cnt])
    # weights with outliers, by rows
    r = recipes.CFG2_TRUNK
    w = recipes.linear_weight_rows(r, 0, 64)
    np.testing.assert_array_equal(recipes.linear_weight_rows(r, 17, 5), w[17:22])
    # one expert's rows inside the stacked expert stream
    e = recipes.CFG4
    g = recipes.moe_expert_rows(e, "down", 3, 0, 8)
    np.testing.assert_array_equal(recipes.moe_expert_rows(e, "down", 3, 5, 2), g[5:7])
    assert not np.array_equal(recipes.moe_expert_rows(e, "down", 4, 0, 8), g)


def test_outliers_follow_their_own_uniform_stream():
    seed, stream, p, factor, n = 9, 102, 0.01, 20.0, 4000
    base = synth.normal(seed, 2, n, 0.02)
    w = base.copy()
    k = synth.outliers(seed, stream, w, p, factor)
    r = np.array([synth.raw(seed, stream, c) for c in range(n)], dtype=np.uint64)
    mask = (r >> np.uint64(11)).astype(np.float64) * 2.0 ** -53 < p
    assert k == int(mask.sum())
    np.testing.assert_array_equal(w[mask], (base[mask].astype(np.float64) * factor).astype(np.float32))
    np.testing.assert_array_equal(w[~mask], base[~mask])


def test_normal_moments_and_quantiles():
    x = synth.normal(11, 3, 1 << 20, 1.0).astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    for q, z in ((0.025, -1.959964), (0.5, 0.0), (0.975, 1.959964)):
        assert abs(np.mean(x < z) - q) < 2e-3


def test_zipf_bias_and_permutation():
    n, s = 256, 1.1
    perm = synth.permutation(0, 20, n)
    assert sorted(perm.tolist()) == list(range(n))
    b = synth.zipf_bias(0, 20, n, s)
    want = np.empty(n, np.float32)
    want[perm] = (-s * np.log(np.arange(1, n + 1, dtype=np.float64))).astype(np.float32)
    np.testing.assert_array_equal(b, want)


def test_bf16_rounds_to_nearest_even():
    bits = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001,
                     0xBF808000, 0x7F7FFFFF, 0x00000001], dtype=np.uint32)
    x = bits.view(np.float32)
    want = []
    for b in bits.tolist():
        hi, lo = b >> 16, b & 0xFFFF
        up = lo > 0x8000 or (lo == 0x8000 and (hi & 1))
        want.append((hi + up) & 0xFFFF)
    assert synth.to_bf16(x).tolist() == want
    np.testing.assert_array_equal(synth.bf16_to_f32(synth.to_bf16(x))[:1], x[:1])
