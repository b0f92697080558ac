"""Seeded random cases through every entry point (C ABI) against the f64 CPU
oracle: random row counts, vocab sizes, row strides, base offsets (16-byte
misalignment), padding values, value scales, special values and forced launch
plans. Each case is drawn from a fixed seed, so a failure names a case that
reproduces."""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
from parity import (assert_candidates, assert_grad, assert_log_softmax, assert_loss, assert_mean,
                    assert_softmax, assert_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
THREADS = os.cpu_count() or 1
N_CASES = int(os.environ.get("CE_RANDOM_CASES", "48"))  # raise for a longer soak

FUSED_PLANS = [(0, 0, 0), (1, 0, 0), (1, 2, 128), (1, 5, 0), (2, 0, 0), (2, 3, 128), (4, 0, 0)]
ROW_PLANS = [(0, 0, 0), (2, 0, 0), (2, 4, 128), (6, 0, 0)]
CAND_PLANS = [(0, 0, 0), (0, 1, 0), (0, 3, 0), (0, 4, 0), (0, 8, 0)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)
    yield
    ce.debug_force(0, 0, 0)
    ce.debug_grid_cap(0)
    ce.device_error_reset()


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    rows = int(rng.choice([1, 2, 3, 7, 31, 64, 129, 300]))
    vocab = int(rng.choice([1, 2, 5, 17, 255, 1000, 4099, 16385, 32001, 70001]))
    stride = vocab + int(rng.choice([0, 0, 1, 3, 8]))
    offset = int(rng.integers(0, 4))
    sigma = float(rng.choice([0.5, 3.0, 30.0]))
    pad = float(rng.choice([np.nan, 1e30, -1e30]))
    x = np.full((rows, stride), pad, dtype=np.float32)
    x[:, :vocab] = (sigma * rng.standard_normal((rows, vocab))).astype(np.float32)
    if rng.random() < 0.5 and vocab > 4:                 # integer-valued rows: ties everywhere
        r = rng.integers(0, rows)
        x[r, :vocab] = rng.integers(0, 3, size=vocab).astype(np.float32)
    if rng.random() < 0.4 and rows > 1:                  # special values in one row
        r = rng.integers(0, rows)
        cols = rng.integers(0, vocab, size=3)
        x[r, cols] = rng.choice([np.nan, np.inf, -np.inf, -0.0], size=3).astype(np.float32)
    if rng.random() < 0.3 and rows > 2:                  # a masked row: few finite values
        r = rng.integers(0, rows)
        keep = rng.integers(0, vocab, size=2)
        vals = x[r, keep].copy()
        x[r, :vocab] = -np.inf
        x[r, keep] = vals
    labels = rng.integers(0, vocab, size=rows).astype(np.int64)
    plans = dict(fused=FUSED_PLANS[rng.integers(len(FUSED_PLANS))],
                 rows=ROW_PLANS[rng.integers(len(ROW_PLANS))],
                 cand=CAND_PLANS[rng.integers(len(CAND_PLANS))])
    scale = float(rng.choice([1.0, 1.0 / rows, 0.5]))
    # drawn last, so the earlier draws of a seed stay as they were
    plans["grid_cap"] = int(rng.choice([0, 0, 0, 1, 2, 5]))     # clusters looping over several rows
    plans["host_chunk"] = int(rng.choice([0, 1, 5, rows]))      # ce_grad_host's rows per copied chunk
    plans["ring"] = [(7, 0, 0), (7, 1, 0), (7, 3, 0), (7, 8, 0)][int(rng.integers(4))]  # the ring argmax
    return x, labels, vocab, offset, scale, plans


def on_device(x, offset):
    rows, stride = x.shape
    buf = torch.full((rows * stride + offset + 8,), 3.0, device=DEV)
    d = buf[offset: offset + rows * stride].view(rows, stride)
    d.copy_(torch.from_numpy(x).to(DEV))
    return d


def forced_call(plan, fn, *args, **kw):
    ce.debug_force(*plan)
    try:
        return fn(*args, **kw)
    finally:
        ce.debug_force(0, 0, 0)


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(orc, seed):
    x, labels, vocab, offset, scale, plans = draw_case(seed)
    what = f"case {seed}: {x.shape[0]}x{vocab} stride {x.shape[1]} offset {offset} plans {plans}"
    dx = on_device(x, offset)
    dy = torch.from_numpy(labels).to(DEV)
    def fused(fn, *args, **kw):
        try:
            return forced_call(plans["fused"], fn, *args, **kw)
        except ce.CeError:
            # a forced staged plan may not fit this shape; the automatic plan always does
            return fn(*args, **kw)

    xh = torch.from_numpy(x).pin_memory()
    yh = torch.from_numpy(labels).pin_memory()
    ce.debug_grid_cap(plans["grid_cap"])
    try:
        grad, lr, top = fused(ce.ce_grad, dx, dy, scale, vocab=vocab, loss_rows=True, top=True)
        # the whole step: the same fused kernel, then its mean as a programmatic dependent
        grad_s, lr_s, top_s, mean_s = fused(ce.ce_grad_step, dx, dy, scale, vocab=vocab)
        soft = fused(ce.softmax_rows, dx, vocab=vocab)
        logp = fused(ce.log_softmax_rows, dx, vocab=vocab)
        lr2 = forced_call(plans["rows"], ce.ce_rows, dx, dy, vocab=vocab)
        top2 = forced_call(plans["rows"], ce.argmax_rows, dx, vocab=vocab)
        mean = ce.ce_mean(lr2)
        cand = forced_call(plans["cand"], ce.candidates_rows, dx, vocab=vocab)
        top3 = forced_call(plans["ring"], ce.argmax_rows, dx, vocab=vocab)
        hs = ce.ce_grad_host(xh[:, :vocab], yh, scale, ce.HostStep(x.shape[0], vocab, DEV),
                             chunk_rows=plans["host_chunk"])
        torch.cuda.synchronize()
    finally:
        ce.debug_grid_cap(0)

    g_ref, l_ref = orc.ce_grad(x, vocab, labels, scale, threads=THREADS)
    a_ref = orc.argmax(x, vocab, threads=THREADS)
    assert_grad(grad, g_ref, f"{what}: ce_grad")
    assert_loss(lr, l_ref, f"{what}: ce_grad loss")
    assert_tokens(top, a_ref, f"{what}: ce_grad top")
    assert_loss(lr2, l_ref, f"{what}: ce_rows")
    assert_tokens(top2, a_ref, f"{what}: argmax_rows")
    assert_tokens(top3, a_ref, f"{what}: argmax_rows (ring)")
    # the documented tiny-loss deviation: drawn rows may hold nothing but tiny losses
    assert_mean(mean.item(), orc.ce_mean(l_ref), f"{what}: ce_mean", tiny_loss_rows=l_ref)
    assert_grad(grad_s, g_ref, f"{what}: ce_grad_step")
    assert_loss(lr_s, l_ref, f"{what}: ce_grad_step loss")
    assert_tokens(top_s, a_ref, f"{what}: ce_grad_step tokens")
    assert_mean(mean_s.item(), orc.ce_mean(l_ref), f"{what}: ce_grad_step mean", tiny_loss_rows=l_ref)
    assert_softmax(soft, orc.softmax(x, vocab, threads=THREADS), f"{what}: softmax_rows")
    assert_log_softmax(logp, orc.log_softmax(x, vocab, threads=THREADS), f"{what}: log_softmax_rows")
    assert_candidates(cand, orc.candidates(x, vocab, threads=THREADS), f"{what}: candidates_rows")
    assert_grad(hs.grad, g_ref, f"{what}: ce_grad_host grad")
    assert_tokens(hs.top_h, a_ref, f"{what}: ce_grad_host tokens")
    assert_mean(hs.mean_h.item(), orc.ce_mean(l_ref), f"{what}: ce_grad_host mean", tiny_loss_rows=l_ref)
