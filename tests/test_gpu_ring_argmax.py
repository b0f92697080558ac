"""The ring argmax (path 7, C ABI): argmaxInto through a ring of bulk-copied
row chunks, against the f64 CPU oracle -- shapes that cross the chunk and
the 16-byte grid at both row ends, every row phase, non-finite rows, ties
across chunks, threads and CTAs, and the decode workload at full size."""
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CLUSTERS = [0, 1, 2, 3, 8]


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


def ring_argmax(x, vocab, cluster):
    ce.debug_force(ce.PATH_RING, cluster, 0)
    try:
        return ce.argmax_rows(x, vocab=vocab)
    finally:
        ce.debug_force(0, 0, 0)


@pytest.mark.parametrize("cluster", CLUSTERS)
@pytest.mark.parametrize("offset", [0, 1, 2, 3])
def test_shapes_and_phases(orc, cluster, offset):
    for rows, vocab, pad in ((1, 1, 0), (3, 5, 2), (33, 1025, 0), (7, 3841, 1), (9, 4099, 3), (5, 20011, 5),
                             (2, 65539, 0)):
        stride = vocab + pad
        x, _ = W.random_logits(rows, vocab, stride=stride, sigma=2.0, seed=rows * 13 + vocab + offset,
                               pad_value=1e30)  # padding that would win if it were read
        buf = torch.full((rows * stride + offset + 8,), 1e30, device=DEV)
        dx = buf[offset: offset + rows * stride].view(rows, stride)
        dx.copy_(x.to(DEV))
        top = ring_argmax(dx, vocab, cluster)
        torch.cuda.synchronize()
        assert_tokens(top, orc.argmax(x.numpy(), vocab), f"ring c{cluster} off{offset} {rows}x{vocab}+{pad}")


@pytest.mark.parametrize("cluster", CLUSTERS)
def test_nonfinite_rows_and_ties(orc, cluster):
    nan, inf = float("nan"), float("inf")
    V = 7681  # two chunks and a block: ties across chunks, threads and CTAs
    x = W.random_logits(14, V, seed=9)[0]
    x[0, 17] = nan
    x[1, 1500] = inf
    x[2, :] = -inf                      # all -inf: 0
    x[3, :] = nan                       # all NaN: 0
    x[4, ::2] = -inf
    x[5, :] = -inf
    x[5, 2000] = nan                    # -inf and NaN only: 0
    x[6, :] = 0.0
    x[6, 0] = -0.0                      # -0 == +0: the first wins
    x[7, :] = nan
    x[7, 700] = -inf
    x[8, 3] = inf
    x[8, 9] = inf                       # two +inf: 3
    x[9, :] = 1.0                       # all equal: 0
    x[10, [4000, 3841, 7680]] = 50.0    # tie across chunks: 3841
    x[11, [257, 1]] = 50.0              # tie across threads of one block: 1
    x[12, [6000, 3000]] = 50.0          # a tie whose columns sit in different CTAs of a cluster: 3000
    x[13, V - 1] = 99.0                 # the last column
    top = ring_argmax(x.to(DEV), V, cluster)
    torch.cuda.synchronize()
    assert_tokens(top, orc.argmax(x.numpy(), V), f"non-finite / ties c{cluster}")


def test_decode_workload_full_size(orc):
    w = W.WORKLOADS[W.DECODE]
    b = W.generate(w, device=DEV)
    ref = orc.argmax(b.logits.cpu().numpy(), w.vocab, threads=16)
    for cluster in (0, 1, 2):
        top = ring_argmax(b.logits[:, : w.vocab], w.vocab, cluster)
        torch.cuda.synchronize()
        assert_tokens(top, ref, f"decode ring c{cluster}")
        assert (top[b.tie_rows.to(DEV)].long() == b.tie_cols[:, 0].to(DEV)).all()


@pytest.mark.parametrize("extra", [0, 1], ids=["large-chunks", "small-chunks"])
def test_both_chunk_sizes(orc, extra):
    """Rows just at and just past two CTAs per SM: the ring's 32-block and
    15-block chunks on the same kind of rows (odd vocab: every row phase)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, V = 2 * sms + extra, 20011
    x, _ = W.random_logits(rows, V, stride=V + 2, sigma=2.0, seed=31 + extra, pad_value=1e30)
    x[1, 4000] = x[1, 12000] = 40.0            # a tie across chunks: the lower column
    x[2, :V] = float("nan")
    x[3, :V] = -float("inf")
    ce.debug_force(ce.PATH_RING, 1, 0)
    try:
        p = ce.plan(ce.OP_ARGMAX, rows, V, V + 2)
        assert p["smem"] == 48 + 3 * ((15 if extra else 32) * 256 + 4) * 4, p
    finally:
        ce.debug_force(0, 0, 0)
    top = ring_argmax(x.to(DEV), V, 1)
    assert_tokens(top, orc.argmax(x.numpy(), V), f"ring {rows} x {V}")


def test_other_operations_refuse_the_ring():
    x, y = W.random_logits(4, 1000, seed=1)
    xd, yd = x.to(DEV), y.to(DEV)
    ce.debug_force(ce.PATH_RING, 0, 0)
    try:
        for fn, args in ((ce.ce_rows, (xd, yd)), (ce.ce_grad, (xd, yd, 1.0)), (ce.softmax_rows, (xd,)),
                         (ce.log_softmax_rows, (xd,)), (ce.candidates_rows, (xd,))):
            with pytest.raises(ce.CeError):
                fn(*args)
    finally:
        ce.debug_force(0, 0, 0)


def test_automatic_plans():
    """The ring from four rows per SM up where one warp per row does not apply."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ce.plan(ce.OP_ARGMAX, 4 * sms, 151936)["path"] == ce.PATH_RING
    assert ce.plan(ce.OP_ARGMAX, 16384, 50257)["path"] == ce.PATH_RING
    assert ce.plan(ce.OP_ARGMAX, 8192, 128256)["path"] == ce.PATH_RING
    assert ce.plan(ce.OP_ARGMAX, 4 * sms - 1, 151936)["path"] == ce.PATH_STREAM
    assert ce.plan(ce.OP_ARGMAX, 256, 151936)["path"] == ce.PATH_STREAM
    assert ce.plan(ce.OP_ARGMAX, 4096, 32000)["path"] == ce.PATH_WARP
    assert ce.plan(ce.OP_ROWS, 8192, 128256)["path"] == ce.PATH_STREAM


@pytest.mark.parametrize("cluster", [1, 3])
def test_indirect_rows_and_bad_addresses(orc, cluster):
    """Rows read at the addresses of a table (any 4-byte phase, repeats);
    a null or misaligned address is never read: that row's token is NaN."""
    vocab, n = 7681, 12
    g = torch.Generator().manual_seed(cluster)
    rows = (3.0 * torch.randn(n, vocab, generator=g)).float()
    rows[2, ::3] = float("nan")
    pool = torch.full((n * (vocab + 7) + 8,), 1e30, device=DEV)
    offs = [r * (vocab + 7) + (r % 4) for r in range(n)]
    for r, o in enumerate(offs):
        pool[o: o + vocab] = rows[r].to(DEV)
    pick = torch.tensor([5, 0, 11, 5, 2, 9, 1, 3])
    table = (pool.data_ptr() + torch.tensor(offs)[pick] * 4).to(DEV)
    table[1] = 0                      # null
    table[6] = table[6] + 2           # not 4-byte aligned
    ce.debug_force(ce.PATH_RING, cluster, 0)
    try:
        top = ce.argmax_rows_indirect(table, vocab)
    finally:
        ce.debug_force(0, 0, 0)
    torch.cuda.synchronize()
    t = top.cpu().numpy()
    assert torch.isnan(top[1]) and torch.isnan(top[6])
    good = [0, 2, 3, 4, 5, 7]
    assert_tokens(t[good], orc.argmax(rows[pick[good]].numpy().copy(), vocab), f"ring indirect c{cluster}")
