"""The oracle's page-f32 diagnostic (the literal f32 form of
crossEntropyLoss's entry, "the sum in 16 lanes"): parity unpinned -- the
pages fix neither the lanes nor their join -- so nothing is graded against
it; these checks only keep it what it claims to be. CPU only."""
import math

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_close_to_the_f64_oracle_on_ordinary_rows(orc):
    rng = np.random.default_rng(0)
    for vocab in (1, 2, 15, 16, 17, 1000, 32001):
        x = (3.0 * rng.standard_normal((6, vocab))).astype(np.float32)
        y = rng.integers(0, vocab, 6)
        f64 = orc.ce_rows(x, vocab, y)
        f32 = orc.ce_rows_page_f32(x, vocab, y).astype(np.float64)
        ok = f64 > 0.5  # away from the cancellation the diagnostic is kept to show
        assert np.all(np.abs(f32[ok] - f64[ok]) <= 1e-5 * f64[ok] + 1e-5), (vocab, f32, f64)


def test_uniform_rows_give_log_v(orc):
    for vocab in (1, 2, 1000, 50257):
        x = np.full((1, vocab), 2.5, np.float32)
        got = float(orc.ce_rows_page_f32(x, vocab, np.array([vocab // 2]))[0])
        assert abs(got - math.log(vocab)) <= 2 * np.spacing(np.float32(max(math.log(vocab), 1e-30))), (vocab, got)


def test_the_literal_form_loses_a_dominant_label(orc):
    """Label at the max, the other column 30 below: the loss is log1p(e^-30)
    ~ 9.4e-14; m + logf(1 + 9.4e-14) rounds to m, so the f32 form gives 0."""
    x = np.array([[40.0, 10.0]], np.float32)
    y = np.array([0])
    want = math.log1p(math.exp(-30.0))
    assert abs(orc.ce_rows(x, 2, y)[0] - want) <= 1e-12 * want
    assert orc.ce_rows_page_f32(x, 2, y)[0] == 0.0


def test_nan_and_bad_labels(orc):
    x = np.zeros((3, 40), np.float32)
    x[0, 7] = np.nan
    got = orc.ce_rows_page_f32(x, 40, np.array([0, -1, 39]))
    assert np.isnan(got[0]) and np.isnan(got[1]) and abs(got[2] - math.log(40)) < 1e-6
