"""The parity gate itself (tests/gpu_util.py check_close), on the CPU: an
element passes iff |got - ref| <= 2e-3 + 1e-2 |ref| (the "max abs error 2e-3
and max rel error 1e-2" bound in allclose form), NaN and infinities always
fail, the max rel error is taken over |ref| >= 0.2 only, and an element that
passes through the relative term alone while |ref| < 0.2 is flagged.  Each
case sits just inside or just outside a boundary, so a gate with a dropped
term, a swapped operand or a strict/loose comparison mixed up fails here."""
import copy

import numpy as np
import pytest
import torch

import gpu_util
from gpu_util import ATOL, RTOL, check_close


@pytest.fixture(autouse=True)
def _keep_session_totals():
    # these synthetic checks stay out of the run's reported tolerance totals
    saved = copy.deepcopy(gpu_util.STATS)
    yield
    gpu_util.STATS.clear()
    gpu_util.STATS.update(saved)


def _one(ref: float, diff: float):
    got = torch.tensor([ref + diff], dtype=torch.float64)
    return check_close(got, np.array([ref]), "synthetic")


def test_the_bounds_are_the_stated_ones():
    assert (ATOL, RTOL, gpu_util.REL_FLOOR) == (2e-3, 1e-2, 0.2)


def test_equal_outputs_pass_with_zero_errors():
    ref = np.linspace(-3.0, 3.0, 61)
    assert check_close(torch.tensor(ref), ref, "equal") == (0.0, 0.0, 0)


@pytest.mark.parametrize("ref", [0.0, 0.05, -0.15, 0.2, -1.0, 7.5, 300.0])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_pass_and_fail_on_either_side_of_the_bound(ref, sign):
    bound = ATOL + RTOL * abs(ref)
    _one(ref, sign * bound * (1 - 1e-6))
    with pytest.raises(AssertionError):
        _one(ref, sign * bound * (1 + 1e-6))


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
def test_non_finite_outputs_always_fail(bad):
    ref = np.array([0.0, 1.0, 1e4])
    got = torch.tensor([0.0, bad, 1e4], dtype=torch.float64)
    with pytest.raises(AssertionError):
        check_close(got, ref, "non-finite")


def test_a_non_finite_reference_is_never_matched():
    # the oracle never produces one; if it did, the gate must not pass it
    with pytest.raises(AssertionError):
        check_close(torch.tensor([1.0], dtype=torch.float64), np.array([float("nan")]), "nan ref")


def test_max_rel_counts_only_large_references_and_flags_small_ones():
    ref = np.array([0.1, 0.19, 0.2, 2.0, -4.0])
    diff = np.array([0.0025, 0.0001, 0.003, 0.019, -0.02])   # all inside the bound
    max_abs, max_rel, flagged = check_close(torch.tensor(ref + diff), ref, "mixed")
    assert max_abs == pytest.approx(0.02)
    # over |ref| >= 0.2: 0.003 / 0.2 = 0.015 is the largest relative error
    assert max_rel == pytest.approx(0.015)
    # only 0.1 (+0.0025) passes through the relative term with |ref| < 0.2
    assert flagged == 1


def test_the_session_totals_accumulate_the_worst_flagged_element():
    gpu_util.STATS.update(checks=0, elements=0, max_abs=0.0, max_rel=0.0, flagged=0, worst_flagged=None)
    check_close(torch.tensor([0.1 + 0.0026, 0.5], dtype=torch.float64), np.array([0.1, 0.5]), "first")
    check_close(torch.tensor([-0.05 - 0.0024], dtype=torch.float64), np.array([-0.05]), "second")
    st = gpu_util.STATS
    assert (st["checks"], st["elements"], st["flagged"]) == (2, 3, 2)
    assert st["worst_flagged"][1] == "first" and st["worst_flagged"][0] == pytest.approx(0.0026)


def test_the_first_failure_is_named_in_the_message():
    ref = np.zeros((2, 3))
    got = torch.zeros((2, 3), dtype=torch.float64)
    got[1, 2] = 0.01
    with pytest.raises(AssertionError, match=r"1 of 6 elements.*first bad at \(1, 2\)"):
        check_close(got, ref, "where")
