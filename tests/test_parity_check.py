"""The shared parity check itself (CPU): it must reject NaN, infinite and
unwritten outputs, not only outputs outside the tolerance."""
import numpy as np
import pytest
import torch

from parity import ATOL, RTOL, assert_close


def _case(rows=6, d=8, seed=0):
    rng = np.random.default_rng(seed)
    ref = rng.normal(size=(rows, d))
    ref_lse = rng.normal(size=(rows,))
    ref[2] = 0.0
    ref_lse[2] = -np.inf  # an empty row: o = 0, lse = -inf
    got = torch.tensor(ref, dtype=torch.float32)
    got_lse = torch.tensor(ref_lse, dtype=torch.float32)
    return got, got_lse, ref, ref_lse


def test_exact_and_within_tolerance_pass():
    got, got_lse, ref, ref_lse = _case()
    assert_close("exact", got, got_lse, ref, ref_lse)
    nudge = 0.9 * (ATOL + RTOL * np.abs(ref))
    nudge[2] = 0.0  # the empty row stays exactly 0
    nudged = got + torch.tensor(nudge, dtype=torch.float32)
    assert_close("nudged", nudged, got_lse, ref, ref_lse)


def test_outside_tolerance_fails():
    got, got_lse, ref, ref_lse = _case()
    got[0, 3] += 2 * (ATOL + RTOL * abs(ref[0, 3]))
    with pytest.raises(AssertionError, match="outside tolerance"):
        assert_close("off", got, got_lse, ref, ref_lse)


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), -float("inf")])
def test_nonfinite_output_with_finite_lse_fails(bad):
    """The pattern a 0 * NaN leak from stale cache bytes produces: one output
    element NaN (or inf) while the row's lse stays finite."""
    got, got_lse, ref, ref_lse = _case()
    got[1, 5] = bad
    with pytest.raises(AssertionError, match="NaN or infinite"):
        assert_close("leak", got, got_lse, ref, ref_lse)


def test_unwritten_row_fails():
    """A row the kernel never wrote keeps the NaN the tests pre-fill."""
    got, got_lse, ref, ref_lse = _case()
    got[4] = float("nan")
    got_lse[4] = float("nan")
    with pytest.raises(AssertionError):
        assert_close("unwritten", got, got_lse, ref, ref_lse)
    got, got_lse, ref, ref_lse = _case()
    got_lse[4] = float("nan")  # lse alone unwritten
    with pytest.raises(AssertionError, match="finiteness"):
        assert_close("unwritten lse", got, got_lse, ref, ref_lse)


def test_empty_row_must_be_zero_and_minus_inf():
    got, got_lse, ref, ref_lse = _case()
    got_lse[2] = float("nan")
    with pytest.raises(AssertionError):
        assert_close("empty lse nan", got, got_lse, ref, ref_lse)
    got, got_lse, ref, ref_lse = _case()
    got[2, 0] = 1e-30
    with pytest.raises(AssertionError, match="empty rows"):
        assert_close("empty row nonzero", got, got_lse, ref, ref_lse)


def test_lse_error_fails():
    got, got_lse, ref, ref_lse = _case()
    got_lse[0] += 1e-2
    with pytest.raises(AssertionError, match="lse max err"):
        assert_close("lse", got, got_lse, ref, ref_lse)
