"""The two numeric bars of the GPU parity tests, kept free of GPU imports so
that the CPU suite can check them (tests/test_parity_checks.py).

fp32 paths: every element within its own bound, |y - y_ref| <= bound (the
bound from the oracle: 1e-5 * sum_k |x_k w^_k| + 1e-6 per linear output,
propagated through SwiGLU for the MoE layer).  bf16 tensor-core paths: per
row, relative L2 error <= 1e-2 and the same arg-max, except rows whose oracle
top-2 gap is below 1e-2 * max|y_ref| (a near tie that output rounding alone
can flip).  A NaN or infinity in the output, or a shape that differs from the
reference, fails either bar.
"""
import numpy as np


def assert_within(y, ref, bound, what=""):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    assert y.shape == ref.shape == bound.shape, (what, y.shape, ref.shape, bound.shape)
    err = np.abs(y - ref)
    bad = ~(err <= bound)  # NaN compares false: a NaN output is out of tolerance
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"err/bound {float(np.nanmax(err / bound)) if np.isfinite(err).any() else 'nan'}"
                           f", non-finite outputs {int((~np.isfinite(y)).sum())}")


def assert_bf16_rows(y, yref, what=""):
    y = np.asarray(y, dtype=np.float64)
    yref = np.asarray(yref, dtype=np.float64)
    assert y.shape == yref.shape and y.ndim == 2, (what, y.shape, yref.shape)
    assert np.isfinite(y).all(), (what, "non-finite outputs", int((~np.isfinite(y)).sum()))
    rel = np.linalg.norm(y - yref, axis=1) / np.linalg.norm(yref, axis=1)
    assert (rel <= 1e-2).all(), (what, float(rel.max()))
    top2 = np.sort(yref, axis=1)[:, -2:]
    near_tie = (top2[:, 1] - top2[:, 0]) < 1e-2 * np.abs(yref).max(axis=1)
    same = np.argmax(y, axis=1) == np.argmax(yref, axis=1)
    assert (same | near_tie).all(), (what, np.where(~(same | near_tie))[0])
