"""Parity of the vocab-sharded cross-entropy (ce_stats, ce_stats_combine,
ce_grad_from_stats, through the C ABI) with the f64 CPU oracle: each slice's
statistics against the slice oracle, and the combined loss, token and
gradient against the whole-row oracle (crossEntropyRows, Tensor.argmax,
crossEntropyGrad), for even, uneven and random splits of the columns.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_grad, assert_loss, assert_tokens

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)
    ce.device_error_reset()
    yield


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def sharded_step(x, y, cuts, scale):
    """Stats of each slice, their combination, and every slice's gradient."""
    V = cuts[-1]
    stats = torch.stack([ce.ce_stats(x, y, col0=a, vocab=b - a) for a, b in zip(cuts, cuts[1:])])
    loss, top, comb = ce.ce_stats_combine(stats, y, V)
    grads = [ce.ce_grad_from_stats(x[:, a:b], y, a, comb, scale) for a, b in zip(cuts, cuts[1:])]
    torch.cuda.synchronize()
    return stats, loss, top, comb, torch.cat(grads, dim=1)


def assert_stats(got, ref, what):
    """m, top and x[label] exactly; t (where m is finite) within the loss's
    relative tolerance, and 1e-30 absolute (exp terms below 2^-126 flush)."""
    g = got.detach().cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref[:, 0])
    assert np.array_equal(g[:, 0], ref[:, 0]), f"{what}: m"
    assert np.array_equal(g[:, 2], ref[:, 2]), f"{what}: top"
    assert np.array_equal(g[:, 3], ref[:, 3], equal_nan=True), f"{what}: x[label]"
    gt, rt = g[fin, 1], ref[fin, 1]
    assert np.array_equal(np.isnan(gt), np.isnan(rt)), f"{what}: t NaN pattern"
    ok = ~np.isnan(rt)
    err = np.abs(gt[ok] - rt[ok])
    assert (err <= 2e-5 * np.abs(rt[ok]) + 1e-30).all(), f"{what}: t, worst rel {np.max(err / (np.abs(rt[ok]) + 1e-30)):.3e}"


def check(orc, x, y, cuts, scale, res, what, rows=None):
    stats, loss, top, comb, grad = res
    xs = x.cpu().numpy() if rows is None else x[rows].cpu().numpy()
    ys = y.cpu().numpy() if rows is None else y[rows].cpu().numpy()
    pick = (lambda t: t) if rows is None else (lambda t: t[rows])
    V = cuts[-1]
    for k, (a, b) in enumerate(zip(cuts, cuts[1:])):
        assert_stats(pick(stats[k]), orc.ce_stats(xs, a, b - a, ys), f"{what}: slice {a}:{b} stats")
    g_ref, l_ref = orc.ce_grad(xs, V, ys, scale, threads=THREADS)
    assert_loss(pick(loss), l_ref, f"{what}: combined loss")
    assert_tokens(pick(top), orc.argmax(xs, V, threads=THREADS), f"{what}: combined token")
    assert_grad(pick(grad), g_ref, f"{what}: gradient from stats")


def _cuts(V, shards, seed):
    if shards == 1:
        return [0, V]
    rng = np.random.default_rng(seed)
    return [0] + sorted(rng.choice(np.arange(1, V), size=shards - 1, replace=False).tolist()) + [V]


@pytest.mark.parametrize("name", ["ce_64x1000", "ce_4096x32000"])
@pytest.mark.parametrize("shards", [1, 2, 3, 8])
def test_sharded_workloads_in_full(orc, name, shards):
    w = W.WORKLOADS[name]
    b = W.generate(w, device=DEV)
    for cuts in (list(range(0, w.vocab, -(-w.vocab // shards))) + [w.vocab], _cuts(w.vocab, shards, shards)):
        cuts = sorted(set(cuts))
        res = sharded_step(b.logits, b.labels, cuts, b.scale)
        check(orc, b.logits, b.labels, cuts, b.scale, res, f"{name} {cuts}")


def test_sharded_headline_sampled_rows(orc):
    """8192 x 128256 split 8 ways (16032 columns each, a tensor-parallel head)."""
    w = W.WORKLOADS[W.HEADLINE]
    b = W.generate(w, device=DEV)
    cuts = list(range(0, w.vocab, w.vocab // 8)) + [w.vocab]
    cuts = sorted(set(cuts))
    res = sharded_step(b.logits, b.labels, cuts, b.scale)
    rows = torch.unique(torch.cat([torch.randint(0, w.rows, (16,), generator=torch.Generator().manual_seed(2)),
                                   torch.tensor([0, w.rows - 1])])).to(DEV)
    check(orc, b.logits, b.labels, cuts, b.scale, res, "headline 8-way", rows=rows)


def test_sharded_nonfinite_and_masked_rows(orc):
    nan, inf = float("nan"), float("inf")
    V = 3001
    x, y = W.random_logits(10, V, sigma=3.0, seed=30)
    x[0, 5] = nan
    x[1, 2000] = inf
    x[2, :] = -inf
    x[3, :1500] = -inf              # a whole slice masked
    x[4, :1000] = nan               # a whole slice NaN
    y[4] = 2500
    x[5, :] = 1.0                   # ties across every slice
    x[6, 10] = x[6, 2900] = 40.0    # the max in two slices
    x[7, :] = -inf
    x[7, 2999] = 0.5
    x[8, 3] = 60.0
    y[8] = 3                        # a tiny loss
    for cuts in ([0, 1000, 1500, V], [0, 1, 2, 3, 4, V], [0, 1499, 1501, V]):
        res = sharded_step(x.to(DEV), y.to(DEV), cuts, 0.5)
        check(orc, x, y, cuts, 0.5, res, f"non-finite {cuts}")


def test_shards_held_apart_and_in_place(orc):
    """Each shard a tensor of its own (as on separate devices); the gradient
    written over the shard in place."""
    V, R = 50257, 6
    x, y = W.random_logits(R, V, sigma=4.0, seed=31)
    cuts = [0, 12565, 25130, 37695, V]
    shards = [x[:, a:b].contiguous().to(DEV) for a, b in zip(cuts, cuts[1:])]
    yd = y.to(DEV)
    stats = torch.stack([ce.ce_stats_shard(s, yd, a) for s, a in zip(shards, cuts)])
    loss, top, comb = ce.ce_stats_combine(stats, yd, V)
    for s, a in zip(shards, cuts):
        g = ce.ce_grad_from_stats(s, yd, a, comb, 0.25, grad=s)
        assert g.data_ptr() == s.data_ptr()
    torch.cuda.synchronize()
    g_ref, l_ref = orc.ce_grad(x.numpy(), V, y.numpy(), 0.25)
    assert_loss(loss, l_ref, "apart: loss")
    assert_tokens(top, orc.argmax(x.numpy(), V), "apart: token")
    assert_grad(torch.cat(shards, dim=1), g_ref, "apart: in-place gradient")


def test_sharded_bad_labels_counter(orc):
    V, R = 4000, 5
    x, y = W.random_logits(R, V, seed=32)
    y[1], y[3] = -1, V
    ce.device_error_reset()
    res = sharded_step(x.to(DEV), y.to(DEV), [0, 2000, V], 1.0)
    check(orc, x, y, [0, 2000, V], 1.0, res, "bad labels")
    assert ce.device_error_count() == (2, 0)
    ce.device_error_reset()


@pytest.mark.parametrize("plan", [(2, 0, 0), (6, 0, 0)], ids=["cta-per-row", "warp-per-row"])
def test_sharded_stats_on_each_row_kernel(orc, plan):
    V, R = 20000, 700
    x, y = W.random_logits(R, V, sigma=2.0, seed=33)
    x[5, :8000] = -float("inf")
    cuts = [0, 7001, 8000, 13333, V]
    ce.debug_force(*plan)
    try:
        res = sharded_step(x.to(DEV), y.to(DEV), cuts, 1.0 / R)
    finally:
        ce.debug_force(0, 0, 0)
    check(orc, x, y, cuts, 1.0 / R, res, f"stats via {plan}")
