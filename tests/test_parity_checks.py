"""The GPU parity bars checked on the CPU: each accepts what it should and
rejects a result that is out of tolerance, non-finite or of the wrong shape
(so that a lax check cannot hide a kernel fault)."""
import numpy as np
import pytest

from parity_checks import assert_bf16_rows, assert_within


def test_within_accepts_up_to_the_bound():
    ref = np.array([[1.0, -2.0, 3.0]])
    bound = np.array([[1e-3, 2e-3, 1e-6]])
    assert_within(ref + 0.5 * bound, ref, bound)
    assert_within(ref - 0.99 * bound, ref, bound)


@pytest.mark.parametrize("bad", ["over", "nan", "inf", "shape"])
def test_within_rejects(bad):
    ref = np.array([[1.0, -2.0, 3.0]])
    bound = np.array([[1e-3, 2e-3, 1e-6]])
    y = ref.copy()
    if bad == "over":
        y[0, 2] += 2e-6
    elif bad == "nan":
        y[0, 1] = np.nan
    elif bad == "inf":
        y[0, 0] = np.inf
    else:
        y = ref[0]  # [3] against [1, 3] would broadcast
    with pytest.raises(AssertionError):
        assert_within(y, ref, bound)


def _rows():
    # long rows (1024) so that moving the winner by a little stays inside the
    # 1e-2 relative L2 bar and only the arg-max check can object
    rng = np.random.default_rng(0)
    yref = rng.normal(0.0, 3.0, size=(4, 1024))
    yref[:, 7] = 20.0   # the arg-max of every row
    yref[:, 3] = 19.7   # runner-up, 0.3 below: not a near tie (1e-2 * 20 = 0.2)
    return yref


def test_bf16_rows_accept_small_relative_error():
    yref = _rows()
    assert_bf16_rows(yref * (1 + 5e-3), yref)


@pytest.mark.parametrize("bad", ["rel", "argmax", "nan", "shape"])
def test_bf16_rows_reject(bad):
    yref = _rows()
    y = yref.copy()
    if bad == "rel":
        y[2] *= 1.03
    elif bad == "argmax":
        y[1, 3], y[1, 7] = 20.0, 19.7  # relative error 0.0045: only the arg-max moved
        assert np.linalg.norm(y[1] - yref[1]) / np.linalg.norm(yref[1]) < 1e-2
    elif bad == "nan":
        y[0, 0] = np.nan
    else:
        y = yref[:, :32]
    with pytest.raises(AssertionError):
        assert_bf16_rows(y, yref)


def test_bf16_rows_allow_a_flip_at_a_near_tie():
    yref = _rows()
    yref[3, 3] = 19.9  # top-2 gap 0.1 < 1e-2 * 20: a near tie
    y = yref.copy()
    y[3, 3], y[3, 7] = 20.0, 19.9
    assert_bf16_rows(y, yref)
