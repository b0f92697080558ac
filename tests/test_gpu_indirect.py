"""Parity of the indirect forms of argmaxInto and candidatesInto (rows read at
the addresses of a device table; C ABI) with the f64 CPU oracle applied to the
same rows gathered on the host."""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_candidates, assert_tokens

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)
    yield
    ce.debug_force(0, 0, 0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def pool_rows(n_rows, vocab, seed):
    """A flat device pool holding n_rows rows of `vocab` floats at random
    4-byte offsets (so rows start on every 16-byte phase), ties and NaN in
    some; returns the pool, each row's element offset, and the rows on the host."""
    g = torch.Generator().manual_seed(seed)
    offs, pos = [], 0
    for _ in range(n_rows):
        pos += int(torch.randint(0, 7, (1,), generator=g))
        offs.append(pos)
        pos += vocab
    host = torch.full((pos + 8,), 1e30)
    rows = (3.0 * torch.randn(n_rows, vocab, generator=g)).float()
    if n_rows > 2 and vocab > 4:
        rows[1] = torch.randint(0, 3, (vocab,), generator=g).float()   # ties
        rows[2, ::3] = float("nan")
    for r, o in enumerate(offs):
        host[o: o + vocab] = rows[r]
    return host.to(DEV), torch.tensor(offs, dtype=torch.int64), rows


def table_of(pool, offs, pick):
    return (pool.data_ptr() + offs[pick] * 4).to(DEV)


PLANS = [(0, 0, 0), (2, 1, 0), (2, 2, 0), (2, 4, 128), (6, 0, 0), (7, 0, 0), (7, 3, 0)]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: f"path{p[0]}-c{p[1]}-t{p[2]}")
@pytest.mark.parametrize("vocab", [1, 5, 1000, 4099, 20011])
def test_indirect_argmax_and_candidates(orc, plan, vocab):
    pool, offs, rows = pool_rows(40, vocab, seed=vocab)
    pick = torch.tensor([5, 0, 39, 5, 17, 2, 1, 2, 33, 8, 8, 21])   # any order, repeats
    table = table_of(pool, offs, pick)
    xs = rows[pick].numpy().copy()
    ce.debug_force(*plan)
    try:
        top = ce.argmax_rows_indirect(table, vocab)
    finally:
        ce.debug_force(0, 0, 0)
    cand_plan = (0, plan[1], 0) if plan[0] == 2 else (0, 0, 0)
    ce.debug_force(*cand_plan)
    try:
        cand = ce.candidates_rows_indirect(table, vocab)
    finally:
        ce.debug_force(0, 0, 0)
    torch.cuda.synchronize()
    assert_tokens(top, orc.argmax(xs, vocab), f"indirect argmax {plan} V={vocab}")
    assert_candidates(cand, orc.candidates(xs, vocab), f"indirect candidates {cand_plan} V={vocab}")


def test_indirect_bad_addresses_are_never_read(orc):
    vocab = 3000
    pool, offs, rows = pool_rows(6, vocab, seed=3)
    table = table_of(pool, offs, torch.arange(6))
    table[1] = 0                             # null
    table[4] = table[4] + 2                  # not 4-byte aligned
    top = ce.argmax_rows_indirect(table, vocab)
    cand = ce.candidates_rows_indirect(table, vocab)
    torch.cuda.synchronize()
    t = top.cpu().numpy()
    assert np.isnan(t[1]) and np.isnan(t[4])
    good = [0, 2, 3, 5]
    assert_tokens(t[good], orc.argmax(rows[good].numpy().copy(), vocab), "good rows beside bad ones")
    c = cand.cpu().numpy().reshape(6, -1, 2)
    for r in (1, 4):
        assert (c[r, :, 0] == -np.inf).all() and (c[r, :, 1] == -1).all()
    assert_candidates(cand[good], orc.candidates(rows[good].numpy().copy(), vocab), "good candidates")


def test_indirect_decode_batch(orc):
    """256 rows picked from a 1024 x 151936 (stride 152064) pool of decode logits."""
    w = W.WORKLOADS[W.DECODE].with_rows(1024)
    b = W.generate(w, device=DEV)
    pick = torch.randperm(1024, generator=torch.Generator().manual_seed(9))[:256]
    table = ce.row_addresses(b.logits, pick)
    top = ce.argmax_rows_indirect(table, w.vocab)
    cand = ce.candidates_rows_indirect(table, w.vocab)
    torch.cuda.synchronize()
    xs = b.logits[pick.to(DEV)].cpu().numpy()
    assert_tokens(top, orc.argmax(xs, w.vocab, threads=THREADS), "decode indirect argmax")
    assert_candidates(cand, orc.candidates(xs, w.vocab, threads=THREADS), "decode indirect candidates")
    # the same rows read in place through the direct call
    assert_tokens(ce.argmax_rows(b.logits[pick.to(DEV)], vocab=w.vocab), orc.argmax(xs, w.vocab), "direct")


def test_indirect_refuses_the_even_split():
    """Large enough for the even split (rows x vocab >= 2 x SMs x 8192), forced: refused."""
    pool, offs, _ = pool_rows(64, 100000, seed=4)
    table = table_of(pool, offs, torch.arange(64))
    ce.debug_force(5, 0, 0)
    try:
        with pytest.raises(ce.CeError):
            ce.argmax_rows_indirect(table, 100000)
    finally:
        ce.debug_force(0, 0, 0)
