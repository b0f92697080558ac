"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (element by element, CUDA path vs the f64 CPU oracle):
  per-row loss   relative 2e-5 (absolute 2^-126 below the f32 normal range,
                 where f32 has no relative precision left)
  mean loss      relative 1e-6. Every workload and every fixed case meets it
                 as it stands. One documented deviation, used by the seeded
                 random soak alone (its drawn rows may be nothing but tiny
                 losses): assert_mean(..., tiny_loss_rows=l) adds, for each
                 row whose loss is below 1e-4, that row's own 2e-5 allowance
                 weighted by its share of the mean. Such a loss is a sum of
                 exponentials of logits far below a labelled max, each carrying
                 up to |x - m| 2^-23 relative error from f32 arguments, and the
                 mean of few such rows cannot be better than the rows themselves
  gradient       absolute 1e-6
  argmax token   exact
  softmax row    absolute 1e-6 (the gradient's: the same kernel and arithmetic)
  log-softmax    relative 2e-5 (the loss's: it shares one log1pf of the same
                 sum and one rounded subtraction per element)
  candidates     exact, bit for bit (values are copies of the logits)
  split sums     the f32 recursive-summation bound, per element:
                 (terms - 1) * 2^-24 * sum of |terms| (and 2^-149, one denormal)
A NaN must meet a NaN, and an infinity the same infinity.
"""
from __future__ import annotations

import numpy as np
import torch

LOSS_REL = 2e-5
MEAN_REL = 1e-6
GRAD_ABS = 1e-6
F32_TINY = 2.0 ** -126


def _np(x):
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _same_specials(got, ref, what):
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    if not (nan_g == nan_r).all():
        k = int(np.argmax(nan_g != nan_r))
        raise AssertionError(f"{what}: NaN mismatch at flat {k}: got {got.ravel()[k]}, ref {ref.ravel()[k]}")
    inf_g, inf_r = np.isinf(got), np.isinf(ref)
    if not ((inf_g == inf_r) & (~inf_r | (np.sign(got) == np.sign(ref)))).all():
        k = int(np.argmax((inf_g != inf_r) | (inf_r & (np.sign(got) != np.sign(ref)))))
        raise AssertionError(f"{what}: inf mismatch at flat {k}: got {got.ravel()[k]}, ref {ref.ravel()[k]}")
    return ~(nan_r | inf_r)


def assert_loss(got, ref, what="loss"):
    got, ref = _np(got), _np(ref)
    fin = _same_specials(got, ref, what)
    err = np.abs(got[fin] - ref[fin])
    tol = LOSS_REL * np.abs(ref[fin]) + F32_TINY
    if (err > tol).any():
        k = int(np.argmax(err / tol))
        raise AssertionError(f"{what}: rel err {err[k] / max(abs(ref[fin][k]), 1e-300):.3e} "
                             f"(got {got[fin][k]!r}, ref {ref[fin][k]!r})")


TINY_LOSS = 1e-4


def assert_mean(got, ref, what="mean", tiny_loss_rows=None):
    """The mean loss within 1e-6 relative. ``tiny_loss_rows`` (the oracle's
    row losses) adds the allowance of rows below TINY_LOSS -- the documented
    deviation of the random soak only (see the module docstring)."""
    got, ref = float(got), float(ref)
    if np.isnan(ref):
        assert np.isnan(got), f"{what}: {got} != NaN"
        return
    if np.isinf(ref):  # a row with loss +inf (its label at a -inf logit)
        assert got == ref, f"{what}: {got!r} vs {ref!r}"
        return
    tol = MEAN_REL * abs(ref)
    if tiny_loss_rows is not None:
        l = np.abs(np.asarray(tiny_loss_rows, dtype=np.float64))
        if l.size:
            tol += LOSS_REL * l[l < TINY_LOSS].sum() / l.size
    assert abs(got - ref) <= tol, f"{what}: {got!r} vs {ref!r} (tolerance {tol:.3e})"


def assert_grad(got, ref, what="grad"):
    got, ref = _np(got), _np(ref)
    fin = _same_specials(got, ref, what)
    err = np.abs(got - ref)
    err[~fin] = 0.0
    if (err > GRAD_ABS).any():
        k = int(np.argmax(err))
        raise AssertionError(f"{what}: abs err {err.ravel()[k]:.3e} at flat {k} "
                             f"(got {got.ravel()[k]!r}, ref {ref.ravel()[k]!r})")


def assert_tokens(got, ref, what="argmax"):
    got = _np(got)
    ref = np.asarray(ref, dtype=np.int64)
    assert got.shape == ref.shape, f"{what}: shape"
    assert (got == np.floor(got)).all(), f"{what}: tokens must be integral f32"
    bad = got.astype(np.int64) != ref
    if bad.any():
        k = int(np.argmax(bad))
        raise AssertionError(f"{what}: row {k}: got {int(got[k])}, ref {ref[k]} ({int(bad.sum())} rows differ)")


LOGP_REL = LOSS_REL
SOFTMAX_ABS = GRAD_ABS


def assert_softmax(got, ref, what="softmax"):
    """Softmax rows: the gradient's absolute tolerance."""
    assert_grad(got, ref, what)


def assert_log_softmax(got, ref, what="log-softmax"):
    """Log-softmax rows: the loss's relative tolerance."""
    assert_loss(got, ref, what)


def assert_candidates(got, ref, what="candidates"):
    """Candidate rows: equal bit for bit."""
    g = np.ascontiguousarray(got.detach().cpu().numpy() if isinstance(got, torch.Tensor) else got,
                             dtype=np.float32)
    r = np.ascontiguousarray(ref, dtype=np.float32)
    assert g.shape == r.shape, f"{what}: shape {g.shape} != {r.shape}"
    bad = g.view(np.int32) != r.view(np.int32)
    if bad.any():
        k = int(np.argmax(bad.ravel()))
        row, f = divmod(k, g.shape[-1])
        t, rest = divmod(f, 8)
        raise AssertionError(f"{what}: row {row} thread {t} float {rest}: got {g.ravel()[k]!r}, "
                             f"ref {r.ravel()[k]!r} ({int(bad.sum())} floats differ)")


def assert_split_sum(got, ref, y, parts, add, what="split_sum"):
    """Split sums against the f64 oracle, within the f32 summation bound."""
    got, ref = _np(got), _np(ref)
    p = np.asarray(parts, dtype=np.float64)
    mag = np.abs(p).sum(axis=0)
    terms = p.shape[0]
    if add:
        mag = mag + np.abs(np.asarray(y, dtype=np.float64))
        terms += 1
    fin = _same_specials(got, ref, what)
    tol = max(terms - 1, 1) * 2.0 ** -24 * mag + 2.0 ** -149
    err = np.abs(got - ref)
    if (err[fin] > tol[fin]).any():
        k = int(np.argmax(np.where(fin, err / tol, 0)))
        raise AssertionError(f"{what}: element {k}: got {got[k]!r}, ref {ref[k]!r}, bound {tol[k]:.3e}")
