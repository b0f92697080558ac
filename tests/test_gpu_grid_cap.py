"""Row loops carried across rows (C ABI): with the grid capped at a few
clusters, each cluster runs several rows back to back, so chunk rings,
prefetches of the next row and cluster barriers cross row boundaries on
small inputs. Parity with the f64 CPU oracle is unchanged."""
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import (assert_candidates, assert_grad, assert_loss, assert_softmax, assert_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROWS = 11
CAPS = [1, 2, 3, 7]
# a CTA's share of a row is 1, 2, 3 or many chunks of 15 blocks of 256 columns
VOCABS = [5, 1000, 3841, 7681, 20011]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)
    ce.debug_grid_cap(0)
    yield
    ce.debug_force(0, 0, 0)
    ce.debug_grid_cap(0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def capped(cap, plan, fn, *args, **kw):
    """fn under a grid cap and a forced plan; a forced plan that does not fit
    the shape is refused before any launch, and the automatic one is used."""
    ce.debug_grid_cap(cap)
    try:
        ce.debug_force(*plan)
        try:
            return fn(*args, **kw)
        except ce.CeError:
            ce.debug_force(0, 0, 0)
            return fn(*args, **kw)
    finally:
        ce.debug_force(0, 0, 0)
        ce.debug_grid_cap(0)


@pytest.mark.parametrize("vocab", VOCABS)
@pytest.mark.parametrize("cap", CAPS)
def test_candidates_rows_in_sequence(orc, cap, vocab):
    x, _ = W.random_logits(ROWS, vocab, stride=vocab + 3, sigma=2.0, seed=cap * 100 + vocab % 97)
    x[2, ::5] = float("nan")
    x[4] = torch.randint(0, 3, (vocab + 3,), generator=torch.Generator().manual_seed(4)).float()  # ties
    x[6, : vocab // 2] = -float("inf")
    xd = x.to(DEV)[:, :vocab]
    ref = orc.candidates(x.numpy(), vocab)
    for c in (1, 2, 3, 8):
        got = capped(cap, (0, c, 0), ce.candidates_rows, xd, vocab=vocab)
        torch.cuda.synchronize()
        assert_candidates(got, ref, f"cap {cap} cluster {c} V={vocab}")


@pytest.mark.parametrize("vocab", VOCABS)
@pytest.mark.parametrize("cap", CAPS)
def test_fused_and_row_kernels_in_sequence(orc, cap, vocab):
    x, y = W.random_logits(ROWS, vocab, stride=vocab + 1, sigma=3.0, seed=cap * 7 + vocab)
    xh = x.numpy()
    xd, yd = x.to(DEV)[:, :vocab], y.to(DEV)
    g_ref, l_ref = orc.ce_grad(xh, vocab, y.numpy(), 0.5)
    a_ref = orc.argmax(xh, vocab)
    s_ref = orc.softmax(xh, vocab)
    for plan in ((0, 0, 0), (1, 2, 0), (4, 2, 128), (2, 3, 0)):
        grad = torch.empty(ROWS, vocab, device=DEV)
        loss = torch.empty(ROWS, device=DEV)
        top = torch.empty(ROWS, device=DEV)
        capped(cap, plan, ce.ce_grad, xd, yd, 0.5, vocab=vocab, grad=grad, loss_rows=loss, top=top)
        soft = capped(cap, plan, ce.softmax_rows, xd, vocab=vocab)
        torch.cuda.synchronize()
        assert_grad(grad, g_ref, f"grad cap {cap} {plan} V={vocab}")
        assert_loss(loss, l_ref, f"grad loss cap {cap} {plan} V={vocab}")
        assert_tokens(top, a_ref, f"grad top cap {cap} {plan} V={vocab}")
        assert_softmax(soft, s_ref, f"softmax cap {cap} {plan} V={vocab}")
    for plan in ((0, 0, 0), (2, 1, 0), (2, 3, 128), (6, 0, 0), (7, 0, 0), (7, 3, 0)):
        lr = capped(cap, plan, ce.ce_rows, xd, yd, vocab=vocab)
        tk = capped(cap, plan, ce.argmax_rows, xd, vocab=vocab)
        torch.cuda.synchronize()
        assert_loss(lr, l_ref, f"rows cap {cap} {plan} V={vocab}")
        assert_tokens(tk, a_ref, f"argmax cap {cap} {plan} V={vocab}")


def test_grid_cap_shows_in_the_plan():
    ce.debug_grid_cap(3)
    try:
        p = ce.plan(ce.OP_CANDIDATES, 1000, 151936)
        assert p["ctas"] == 3 * p["cluster"], p
    finally:
        ce.debug_grid_cap(0)
    assert ce.plan(ce.OP_CANDIDATES, 1000, 151936)["ctas"] == 1000
