"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (element by element, CUDA path vs the f64 CPU oracle):
  per-row loss   relative 2e-5 (absolute 2^-126 below the f32 normal range,
                 where f32 has no relative precision left)
  mean loss      relative 1e-6
  gradient       absolute 1e-6
  argmax token   exact
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


def assert_mean(got, ref, what="mean"):
    got, ref = float(got), float(ref)
    if np.isnan(ref):
        assert np.isnan(got), f"{what}: {got} != NaN"
        return
    assert abs(got - ref) <= MEAN_REL * abs(ref), f"{what}: {got!r} vs {ref!r}"


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
