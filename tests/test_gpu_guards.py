"""Guard bands around every input and output (C ABI): no entry point reads or
writes outside its buffers.

Inputs sit inside a larger buffer whose margins and row padding hold +1e30:
a read of any of them would become a row max (changing the loss, token,
softmax and candidates against the oracle, which reads only the valid
columns). Outputs sit inside a larger buffer whose margins hold a sentinel
bit pattern that must survive the call. Rows start at every 16-byte phase.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import (assert_candidates, assert_grad, assert_log_softmax, assert_loss, assert_softmax,
                    assert_split_sum, assert_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 1e30
MARGIN = 67           # floats of guard on each side (not a multiple of 4)
SENTINEL = 0x7FBADBAD  # a NaN bit pattern no result can take


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)
    yield
    ce.debug_force(0, 0, 0)
    ce.device_error_reset()


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def guarded_input(x_host, offset):
    """x_host [rows, stride] (padding already GUARD) inside a GUARD-filled buffer."""
    rows, stride = x_host.shape
    buf = torch.full((MARGIN + offset + rows * stride + MARGIN,), GUARD, device=DEV)
    v = buf[MARGIN + offset: MARGIN + offset + rows * stride].view(rows, stride)
    v.copy_(torch.from_numpy(x_host).to(DEV))
    return v


class GuardedOut:
    """An output tensor of `shape` inside a sentinel-filled buffer."""

    def __init__(self, shape, offset, dtype=torch.float32):
        n = int(np.prod(shape))
        self.buf = torch.empty(MARGIN + offset + n + MARGIN, dtype=torch.int32, device=DEV)
        self.buf.fill_(SENTINEL)
        self.lo, self.hi = MARGIN + offset, MARGIN + offset + n
        self.t = self.buf[self.lo: self.hi].view(torch.float32).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        b = self.buf.cpu().numpy()
        assert (b[: self.lo] == SENTINEL).all() and (b[self.hi:] == SENTINEL).all(), f"{what}: wrote outside"


def make_rows(rows, vocab, pad, seed):
    x, y = W.random_logits(rows, vocab, stride=vocab + pad, sigma=3.0, seed=seed, pad_value=GUARD)
    return x.numpy(), y


SHAPES = [(1, 1, 0), (3, 5, 3), (7, 1000, 1), (33, 4099, 0), (5, 20011, 5), (2, 200003, 2)]
PLANS = [(0, 0, 0), (2, 3, 128), (1, 2, 0)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}+{s[2]}")
@pytest.mark.parametrize("offset", [0, 1, 3])
@pytest.mark.parametrize("plan", PLANS, ids=lambda p: f"path{p[0]}-c{p[1]}")
def test_guard_bands(orc, shape, offset, plan):
    rows, vocab, pad = shape
    xh, y = make_rows(rows, vocab, pad, seed=rows * 31 + vocab + offset)
    x = guarded_input(xh, offset)
    yd = y.to(DEV)
    g_ref, l_ref = orc.ce_grad(xh, vocab, y.numpy(), 0.5)
    a_ref = orc.argmax(xh, vocab)

    def forced(fn, *args, **kw):
        # a forced staged plan may not fit this shape (refused before any
        # launch); the automatic plan always does
        ce.debug_force(*plan)
        try:
            return fn(*args, **kw)
        except ce.CeError:
            ce.debug_force(0, 0, 0)
            return fn(*args, **kw)
        finally:
            ce.debug_force(0, 0, 0)

    grad, loss, top = GuardedOut((rows, vocab), offset), GuardedOut((rows,), offset), GuardedOut((rows,), offset)
    forced(ce.ce_grad, x, yd, 0.5, vocab=vocab, grad=grad.t, loss_rows=loss.t, top=top.t)
    lr = GuardedOut((rows,), offset)
    forced(ce.ce_rows, x, yd, vocab=vocab, out=lr.t)
    am = GuardedOut((rows,), offset)
    forced(ce.argmax_rows, x, vocab=vocab, out=am.t)
    soft, logp = GuardedOut((rows, vocab), offset), GuardedOut((rows, vocab), offset)
    forced(ce.softmax_rows, x, vocab=vocab, out=soft.t)
    forced(ce.log_softmax_rows, x, vocab=vocab, out=logp.t)
    cand = GuardedOut((rows, ce.CANDIDATE_ROW), offset)
    ce.candidates_rows(x, vocab=vocab, out=cand.t)
    for o, what in ((grad, "ce_grad grad"), (loss, "ce_grad loss"), (top, "ce_grad top"), (lr, "ce_rows"),
                    (am, "argmax_rows"), (cand, "candidates_rows")):
        o.check(what)
    assert_grad(grad.t, g_ref, "ce_grad")
    assert_loss(loss.t, l_ref, "ce_grad loss")
    assert_tokens(top.t, a_ref, "ce_grad top")
    assert_loss(lr.t, l_ref, "ce_rows")
    assert_tokens(am.t, a_ref, "argmax_rows")
    assert_candidates(cand.t, orc.candidates(xh, vocab), "candidates_rows")
    soft.check("softmax_rows")
    logp.check("log_softmax_rows")
    assert_softmax(soft.t, orc.softmax(xh, vocab), "softmax_rows")
    assert_log_softmax(logp.t, orc.log_softmax(xh, vocab), "log_softmax_rows")


@pytest.mark.parametrize("offset", [0, 1, 2])
def test_guard_bands_sharded_and_split_sum(orc, offset):
    rows, vocab, pad = 9, 5003, 3
    xh, y = make_rows(rows, vocab, pad, seed=77 + offset)
    x = guarded_input(xh, offset)
    yd = y.to(DEV)
    cuts = [0, 1001, 2999, vocab]
    a16 = (4 - MARGIN % 4) % 4  # the float4 outputs start on a 16-byte boundary
    stats = [GuardedOut((rows, 4), a16 + 4 * ((offset + k) % 2)) for k in range(len(cuts) - 1)]
    for s, (a, b) in zip(stats, zip(cuts, cuts[1:])):
        ce.ce_stats(x, yd, col0=a, vocab=b - a, out=s.t)
    st = torch.stack([s.t for s in stats])
    loss, top, comb = GuardedOut((rows,), offset), GuardedOut((rows,), offset), GuardedOut((rows, 4), a16)
    ce.ce_stats_combine(st, yd, vocab, loss_rows=loss.t, top=top.t, combined=comb.t)
    grads = [GuardedOut((rows, b - a), offset) for a, b in zip(cuts, cuts[1:])]
    for gr, (a, b) in zip(grads, zip(cuts, cuts[1:])):
        ce.ce_grad_from_stats(x[:, a:b], yd, a, comb.t, 0.25, grad=gr.t)
    for o in stats + [loss, top, comb] + grads:
        o.check("sharded")
    g_ref, l_ref = orc.ce_grad(xh, vocab, y.numpy(), 0.25)
    assert_loss(loss.t, l_ref, "sharded loss")
    assert_tokens(top.t, orc.argmax(xh, vocab), "sharded token")
    assert_grad(torch.cat([g.t for g in grads], dim=1), g_ref, "sharded grad")

    parts_h = (np.random.default_rng(offset).standard_normal((5, 1001)) * 10).astype(np.float32)
    pbuf = torch.full((MARGIN + offset + parts_h.size + MARGIN,), GUARD, device=DEV)
    parts = pbuf[MARGIN + offset: MARGIN + offset + parts_h.size].view(5, 1001)
    parts.copy_(torch.from_numpy(parts_h).to(DEV))
    yo = GuardedOut((1001,), offset)
    yo.t.zero_()
    ce.split_sum(parts, yo.t, add=True)
    yo.check("split_sum")
    assert_split_sum(yo.t, orc.split_sum(np.zeros(1001, np.float32), parts_h, True), np.zeros(1001), parts_h, True,
                     "split_sum")
