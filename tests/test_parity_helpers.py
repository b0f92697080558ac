"""The GPU parity tests' comparisons, checked on the CPU: each tolerance
accepts what it should and rejects a result just outside it, non-finite
values must match exactly, and the tiny-loss allowance of the mean stays
confined to the seeded random soak."""
import pathlib
import re

import numpy as np
import pytest

import parity as P

TESTS = pathlib.Path(__file__).resolve().parent


def test_loss_tolerance_is_2e_5_relative():
    ref = np.array([1.0, 10.0, 1e-30, 0.0])
    P.assert_loss(ref * (1 + 1.9e-5), ref)
    with pytest.raises(AssertionError):
        P.assert_loss(ref * (1 + 2.1e-5), ref)


def test_loss_non_finite_must_match():
    ref = np.array([np.nan, np.inf, 1.0])
    P.assert_loss(ref.copy(), ref)
    for bad in ([1.0, np.inf, 1.0], [np.nan, -np.inf, 1.0], [np.nan, 1e30, 1.0], [np.nan, np.inf, np.nan]):
        with pytest.raises(AssertionError):
            P.assert_loss(np.array(bad), ref)


def test_mean_tolerance_is_1e_6_relative():
    P.assert_mean(3.0 * (1 + 0.9e-6), 3.0)
    with pytest.raises(AssertionError):
        P.assert_mean(3.0 * (1 + 1.1e-6), 3.0)
    P.assert_mean(float("nan"), float("nan"))
    with pytest.raises(AssertionError):
        P.assert_mean(1.0, float("nan"))
    with pytest.raises(AssertionError):
        P.assert_mean(1e308, float("inf"))


def test_mean_allowance_only_for_tiny_rows():
    """The allowance adds 2e-5 of each row below 1e-4, weighted by its share:
    rows of ordinary losses get none."""
    big = np.full(8, 2.0)
    with pytest.raises(AssertionError):
        P.assert_mean(2.0 * (1 + 2e-6), 2.0, tiny_loss_rows=big)
    tiny = np.full(8, 1e-6)
    P.assert_mean(1e-6 * (1 + 1.5e-5), 1e-6, tiny_loss_rows=tiny)
    with pytest.raises(AssertionError):
        P.assert_mean(1e-6 * (1 + 2.5e-5), 1e-6, tiny_loss_rows=tiny)


def test_grad_tolerance_is_1e_6_absolute():
    ref = np.array([[0.5, -0.25], [1e-9, 0.0]])
    P.assert_grad(ref + 0.9e-6, ref)
    with pytest.raises(AssertionError):
        P.assert_grad(ref + np.array([[0.0, 0.0], [1.1e-6, 0.0]]), ref)


def test_tokens_exact_and_integral():
    P.assert_tokens(np.array([0.0, 5.0, 151935.0]), [0, 5, 151935])
    with pytest.raises(AssertionError):
        P.assert_tokens(np.array([0.0, 6.0, 151935.0]), [0, 5, 151935])
    with pytest.raises(AssertionError):
        P.assert_tokens(np.array([0.0, 5.5, 151935.0]), [0, 5, 151935])


def test_candidates_bit_for_bit():
    ref = np.array([[1.0, -0.0, np.nan, -np.inf]], dtype=np.float32)
    P.assert_candidates(ref.copy(), ref)
    with pytest.raises(AssertionError):
        P.assert_candidates(np.array([[1.0, 0.0, np.nan, -np.inf]], dtype=np.float32), ref)  # -0 vs +0


def test_split_sum_bound():
    parts = np.array([[1.0, 1e8], [2.0, -1e8]])
    ref = parts.sum(axis=0)
    P.assert_split_sum(ref + np.array([0.0, 5.0]), ref, None, parts, add=False)
    with pytest.raises(AssertionError):
        P.assert_split_sum(ref + np.array([0.0, 13.0]), ref, None, parts, add=False)


def test_tiny_loss_allowance_confined_to_the_random_soak():
    """Only the seeded random soak (rows drawn with nothing but tiny losses)
    may pass tiny_loss_rows: every fixed workload is held to 1e-6."""
    users = sorted(p.name for p in TESTS.glob("*.py")
                   if p.name not in ("parity.py", "test_parity_helpers.py") and re.search(r"tiny_loss_rows\s*=", p.read_text()))
    assert users == ["test_gpu_random_cases.py"], users
