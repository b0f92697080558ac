"""Parity of the CUDA path (through the C ABI) with the f64 CPU oracle.

Every workload is compared with the oracle on every row. The full-size ones
(8192 x 128256 and 16384 x 50257) run at full size through the entry point
and launch shape the bench times (ce_grad_step: gradient, row losses, tokens
and mean from one read), and are compared in chunks of rows: each row's
loss, token and gradient element, and the mean against the oracle's own f64
mean of its own row losses. The mean tolerance here is the plain 1e-6
relative, with no allowance for tiny losses.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_grad, assert_loss, assert_mean, assert_tokens

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
    ce.debug_force(0, 0, 0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def run_all(x, y, scale, vocab=None):
    """Every entry point on one batch; returns host numpy results."""
    grad, lr, top, mean_step = ce.ce_grad_step(x, y, scale, vocab=vocab)
    grad2, lr4, _ = ce.ce_grad(x, y, scale, vocab=vocab, loss_rows=True)
    mean, lr2 = ce.ce_loss(x, y, vocab=vocab)
    lr3 = ce.ce_rows(x, y, vocab=vocab)
    mean2 = ce.ce_mean(lr)
    top2 = ce.argmax_rows(x, vocab=vocab)
    torch.cuda.synchronize()
    # ce_grad is ce_grad_step's kernel without the tokens and the mean: the same bits
    assert torch.equal(grad2.view(torch.int32), grad.view(torch.int32)), "ce_grad vs ce_grad_step gradient"
    assert torch.equal(lr4.view(torch.int32), lr.view(torch.int32)), "ce_grad vs ce_grad_step row losses"
    return dict(grad=grad.cpu().numpy(), loss_grad=lr.cpu().numpy(), loss=lr2.cpu().numpy(),
                loss_rows=lr3.cpu().numpy(), mean=float(mean.item()), mean_of_grad_rows=float(mean2.item()),
                mean_step=float(mean_step.item()), top=top.cpu().numpy(), top_argmax=top2.cpu().numpy())


def check_all(res, orc, xs, vocab, ys, scale, what):
    g_ref, l_ref = orc.ce_grad(xs, vocab, ys, scale, threads=THREADS)
    a_ref = orc.argmax(xs, vocab, threads=THREADS)
    m_ref = orc.ce_mean(l_ref)
    assert_loss(res["loss_grad"], l_ref, f"{what}: ce_grad loss rows")
    assert_loss(res["loss"], l_ref, f"{what}: ce_loss rows")
    assert_loss(res["loss_rows"], l_ref, f"{what}: ce_rows")
    assert_mean(res["mean"], m_ref, f"{what}: ce_loss mean")
    assert_mean(res["mean_of_grad_rows"], m_ref, f"{what}: ce_mean")
    assert_mean(res["mean_step"], m_ref, f"{what}: ce_grad_step mean")
    assert_grad(res["grad"], g_ref, f"{what}: ce_grad")
    assert_tokens(res["top"], a_ref, f"{what}: ce_grad top")
    assert_tokens(res["top_argmax"], a_ref, f"{what}: argmax_rows")


# ---------------------------------------------------------------------------
# the workloads

@pytest.mark.parametrize("name", ["ce_64x1000", "ce_4096x32000"])
def test_small_workloads_in_full(orc, name):
    b = W.generate(W.WORKLOADS[name], device="cpu")
    res = run_all(b.logits.to(DEV), b.labels.to(DEV), b.scale)
    check_all(res, orc, b.logits.numpy(), b.workload.vocab, b.labels.numpy(), b.scale, name)


def test_decode_argmax_in_full(orc):
    w = W.WORKLOADS[W.DECODE]
    b = W.generate(w, device=DEV)
    top = ce.argmax_rows(b.logits, vocab=w.vocab)
    x_host = b.logits.cpu().numpy()
    ref = orc.argmax(x_host, w.vocab, threads=THREADS)
    assert_tokens(top, ref, "decode argmax")
    # the planted ties resolve to the lower column
    top_h = top.cpu().numpy().astype(np.int64)
    for r, (c1, _) in zip(b.tie_rows.tolist(), b.tie_cols.tolist()):
        assert top_h[r] == c1
    # the same through a [rows, vocab] view of the padded rows
    top_v = ce.argmax_rows(b.logits[:, : w.vocab])
    assert_tokens(top_v, ref, "decode argmax (view)")


CHUNK_ROWS = 512


@pytest.mark.parametrize("name", ["ce_8192x128256", "ce_16384x50257_x30"])
def test_full_size_every_row(orc, name):
    """The full-size workloads against the oracle on every row, through the
    bench's step (ce_grad_step) and the standalone ce_rows, ce_loss and
    argmax_rows; compared in chunks of rows so host memory stays bounded."""
    w = W.WORKLOADS[name]
    b = W.generate(w, device=DEV)
    x, y, V, scale = b.logits, b.labels, w.vocab, b.scale
    grad, lr, top, mean_step = ce.ce_grad_step(x, y, scale)
    lr2 = ce.ce_rows(x, y)
    mean_loss, lr3 = ce.ce_loss(x, y)
    top2 = ce.argmax_rows(x)
    torch.cuda.synchronize()

    l_all = np.empty(w.rows, dtype=np.float64)
    for a in range(0, w.rows, CHUNK_ROWS):
        c = min(w.rows, a + CHUNK_ROWS)
        xs = x[a:c].cpu().numpy()
        ys = y[a:c].cpu().numpy()
        g_ref, l_ref = orc.ce_grad(xs, V, ys, scale, threads=THREADS)
        a_ref = orc.argmax(xs, V, threads=THREADS)
        l_all[a:c] = l_ref
        what = f"{name} rows {a}..{c - 1}"
        assert_loss(lr[a:c], l_ref, f"{what}: ce_grad_step loss rows")
        assert_loss(lr2[a:c], l_ref, f"{what}: ce_rows")
        assert_loss(lr3[a:c], l_ref, f"{what}: ce_loss rows")
        assert_tokens(top[a:c], a_ref, f"{what}: ce_grad_step tokens")
        assert_tokens(top2[a:c], a_ref, f"{what}: argmax_rows")
        assert_grad(grad[a:c], g_ref, f"{what}: ce_grad_step gradient")
        del g_ref, xs

    # the mean: against the oracle's f64 mean of its own row losses, in row order
    m_ref = orc.ce_mean(l_all)
    assert_mean(mean_step.item(), m_ref, f"{name}: ce_grad_step mean")
    assert_mean(mean_loss.item(), m_ref, f"{name}: ce_loss mean")
    # the planted rows: constant rows lose log V and take token 0; a
    # label-at-max row's token is its label
    if b.const_rows.numel():
        c = b.const_rows.to(DEV)
        assert_loss(lr[c], np.full(c.numel(), np.log(V)), f"{name}: constant rows = log V")
        assert (top[c] == 0).all()
    if b.label_at_max_rows.numel():
        r = b.label_at_max_rows.to(DEV)
        assert (top[r].long() == y[r]).all()


def test_headline_plan_is_staged_cluster():
    """8192 x 128256: the persistent staged kernel with slices for four CTAs per SM."""
    p = ce.plan(ce.OP_GRAD, 8192, 128256)
    assert p["path"] == ce.PATH_STAGED and p["cluster"] == 10 and p["ctas"] < 8192, p


# ---------------------------------------------------------------------------
# edge cases

PLANS = [(0, 0, 0), (1, 1, 0), (1, 2, 128), (1, 3, 256), (1, 16, 0), (2, 1, 0), (2, 7, 128), (2, 16, 0),
         (4, 1, 0), (4, 2, 0), (4, 5, 0), (4, 16, 0)]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: f"path{p[0]}-c{p[1]}-t{p[2]}")
def test_shapes_and_paths(orc, plan):
    ce.debug_force(*plan)
    try:
        for rows in (1, 2, 3, 31, 33):
            for vocab in (1, 2, 3, 4, 5, 15, 16, 17, 1023, 1025):
                x, y = W.random_logits(rows, vocab, sigma=3.0, seed=rows * 7919 + vocab)
                res = run_all(x.to(DEV), y.to(DEV), 1.0 / rows)
                check_all(res, orc, x.numpy(), vocab, y.numpy(), 1.0 / rows, f"{plan} {rows}x{vocab}")
    finally:
        ce.debug_force(0, 0, 0)


@pytest.mark.parametrize("plan", [(0, 0, 0), (1, 4, 0), (2, 5, 0), (4, 3, 0)], ids=str)
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_base_and_odd_stride(orc, plan, offset):
    """Row starts off any 16-byte boundary; padding of NaN and +1e30 never read."""
    ce.debug_force(*plan)
    try:
        rows, vocab = 9, 4099
        for stride, pad in ((vocab, 0.0), (vocab + 1, float("nan")), (vocab + 3, 1e30), (vocab + 6, float("nan"))):
            x, y = W.random_logits(rows, vocab, stride=stride, sigma=2.0, seed=offset * 31 + stride,
                                   pad_value=pad)
            buf = torch.full((rows * stride + offset + 8,), 7.0, device=DEV)
            dev_x = buf[offset: offset + rows * stride].view(rows, stride)
            dev_x.copy_(x.to(DEV))
            res = run_all(dev_x, y.to(DEV), 0.5, vocab=vocab)
            check_all(res, orc, x.numpy(), vocab, y.numpy(), 0.5, f"off{offset} stride{stride}")
            # a misaligned gradient row start too
            gbuf = torch.empty(rows * vocab + 4, device=DEV)
            g = gbuf[offset: offset + rows * vocab].view(rows, vocab)
            ce.ce_grad(dev_x, y.to(DEV), 0.5, vocab=vocab, grad=g)
            g_ref, _ = orc.ce_grad(x.numpy(), vocab, y.numpy(), 0.5)
            assert_grad(g, g_ref, f"misaligned grad off{offset} stride{stride}")
    finally:
        ce.debug_force(0, 0, 0)


@pytest.mark.parametrize("plan", [(0, 0, 0), (1, 3, 0), (2, 3, 0), (4, 3, 0)], ids=str)
def test_nonfinite_rows(orc, plan):
    nan, inf = float("nan"), float("inf")
    V = 2053
    base = W.random_logits(12, V, seed=5)[0]
    x = base.clone()
    x[0, 17] = nan                      # NaN entry: NaN loss and grad; argmax skips it
    x[1, 1500] = inf                    # +inf entry
    x[2, :] = -inf                      # all -inf
    x[3, :] = nan                       # all NaN: argmax 0
    x[4, ::2] = -inf                    # -inf entries, finite max
    x[5, :] = -inf
    x[5, 2000] = nan                    # -inf and NaN only: argmax = first non-NaN
    x[6, :] = 0.0
    x[6, 0] = -0.0                      # -0 == +0: the first wins
    x[7, :] = nan
    x[7, 700] = -inf                    # all NaN but one -inf
    x[8, 3] = inf
    x[8, 9] = inf                       # two +inf: argmax 3
    y = torch.randint(0, V, (12,), generator=torch.Generator().manual_seed(1))
    y[4] = 0                            # label at a -inf entry: loss +inf
    ce.debug_force(*plan)
    try:
        res = run_all(x.to(DEV), y.to(DEV), 0.25)
    finally:
        ce.debug_force(0, 0, 0)
    check_all(res, orc, x.numpy(), V, y.numpy(), 0.25, f"non-finite {plan}")
    assert np.isinf(res["loss"][4]) and res["loss"][4] > 0


@pytest.mark.parametrize("cluster", [2, 4, 16])
def test_ties_at_slice_and_lane_boundaries(orc, cluster):
    """Equal maxima split across CTAs of a cluster, warps and threads: the lower column wins."""
    V = 4096
    plans = [(1, cluster, 128), (2, cluster, 128), (4, cluster, 0)]
    cols = -(-V // cluster)
    cols += (-cols) % 4
    pairs = [(cols - 1, cols), (cols, 2 * cols), (3, 4), (127, 128), (511, 512), (0, V - 1), (V - 2, V - 1)]
    x = torch.zeros(len(pairs), V)
    for i, (a, b) in enumerate(pairs):
        a, b = min(a, V - 1), min(b, V - 1)
        x[i, a] = x[i, b] = 5.0
    y = torch.zeros(len(pairs), dtype=torch.int64)
    for plan in plans + [(0, 0, 0)]:
        ce.debug_force(*plan)
        try:
            res = run_all(x.to(DEV), y.to(DEV), 1.0)
        finally:
            ce.debug_force(0, 0, 0)
        check_all(res, orc, x.numpy(), V, y.numpy(), 1.0, f"ties {plan}")


@pytest.mark.parametrize("threads", [256, 128])
@pytest.mark.parametrize("cluster", [2, 3, 4, 16])
@pytest.mark.parametrize("offset", [0, 1, 3])
def test_argmax_ties_across_interleaved_blocks(orc, cluster, threads, offset):
    """The streaming argmax's cluster CTAs take a row's blocks of T vectors (4T
    columns past the first 16-byte boundary) in turn: equal maxima on both
    sides of a block boundary, in blocks of one CTA two turns apart, in the
    unaligned head and the tail, and NaN runs beside them -- the lower column
    wins, bit-exact against the oracle, on rows starting at every 16-byte
    phase."""
    V = 4 * threads * (3 * cluster + 1) + 3
    B = 4 * threads
    h = (4 - offset) % 4  # columns before the first 16-byte boundary
    pairs = [(h + B - 1, h + B), (h + 2 * B - 1, h + 2 * B), (h + 5, h + cluster * B + 5),
             (h + B + 7, h + (cluster + 1) * B + 7), (0, V - 1), (max(h - 1, 0), V - 2), (V - 3, V - 1)]
    R = len(pairs) + 2
    S = V + 5
    buf = torch.full((R * S + offset + 8,), 1e30)
    x = buf[offset: offset + R * S].view(R, S)
    x[:, :V] = torch.randn((R, V), generator=torch.Generator().manual_seed(cluster * 7 + threads + offset))
    for i, (a, b) in enumerate(pairs):
        x[i, a] = x[i, b] = 40.0
    x[len(pairs), : V // 2] = float("nan")                  # NaN blocks ahead of the max
    x[len(pairs), V // 2 + 1] = x[len(pairs), V - 1] = 40.0
    x[len(pairs) + 1, :V] = float("nan")                    # all NaN: token 0
    want = orc.argmax(x.numpy(), V)
    dbuf = buf.to(DEV)
    dx = dbuf[offset: offset + R * S].view(R, S)
    ce.debug_force(2, cluster, threads)
    try:
        got = ce.argmax_rows(dx, vocab=V)
        torch.cuda.synchronize()
    finally:
        ce.debug_force(0, 0, 0)
    assert_tokens(got, want, f"interleaved argmax, cluster {cluster}, {threads} threads, offset {offset}")


def test_bad_labels_and_error_counter(orc):
    V, R = 3000, 6
    x, y = W.random_logits(R, V, seed=9)
    y[1] = -1
    y[4] = V
    ce.device_error_reset()
    res = run_all(x.to(DEV), y.to(DEV), 1.0)
    check_all(res, orc, x.numpy(), V, y.numpy(), 1.0, "bad labels")
    bad, waits = ce.device_error_count()
    # ce_grad_step, ce_grad, ce_loss and ce_rows each see the two bad rows once
    assert bad == 8 and waits == 0, (bad, waits)
    ce.device_error_reset()
    assert ce.device_error_count() == (0, 0)


@pytest.mark.parametrize("plan", [(0, 0, 0), (2, 2, 0), (4, 2, 0), (4, 1, 0)], ids=str)
def test_in_place_gradient(orc, plan):
    V, R = 50257, 5
    x, y = W.random_logits(R, V, sigma=4.0, seed=3)
    g_ref, l_ref = orc.ce_grad(x.numpy(), V, y.numpy(), 0.125)
    d = x.to(DEV)
    ce.debug_force(*plan)
    try:
        g, lr, top = ce.ce_grad(d, y.to(DEV), 0.125, grad=d, loss_rows=True, top=True)
    finally:
        ce.debug_force(0, 0, 0)
    assert g.data_ptr() == d.data_ptr()
    assert_grad(d, g_ref, "in-place grad")
    assert_loss(lr, l_ref, "in-place loss")
    assert_tokens(top, orc.argmax(x.numpy(), V), "in-place top")


def test_deterministic_bits():
    b = W.generate(W.WORKLOADS["ce_4096x32000"].with_rows(512), device=DEV)
    outs = []
    for _ in range(3):
        res = run_all(b.logits, b.labels, b.scale)
        outs.append(res)
    for k in ("grad", "loss_grad", "loss", "loss_rows", "top", "top_argmax"):
        assert np.array_equal(outs[0][k], outs[1][k], equal_nan=True), k
        assert np.array_equal(outs[0][k], outs[2][k], equal_nan=True), k
    assert outs[0]["mean"] == outs[1]["mean"] == outs[2]["mean"]


def test_zero_rows():
    x = torch.empty((0, 100), device=DEV)
    y = torch.empty((0,), dtype=torch.int64, device=DEV)
    mean, lr = ce.ce_loss(x, y)
    g = ce.ce_grad(x, y, 1.0)
    t = ce.argmax_rows(x)
    g2, lr2, t2, mean2 = ce.ce_grad_step(x, y, 1.0)
    torch.cuda.synchronize()
    assert np.isnan(mean.item()) and lr.numel() == 0 and g.shape == (0, 100) and t.numel() == 0
    assert np.isnan(mean2.item()) and lr2.numel() == 0 and g2.shape == (0, 100) and t2.numel() == 0


def test_max_vocab_and_beyond(orc):
    V = 1 << 24
    x, y = W.random_logits(2, V, seed=2)
    res = run_all(x.to(DEV), y.to(DEV), 0.5)
    check_all(res, orc, x.numpy(), V, y.numpy(), 0.5, "vocab 2^24")
    too = torch.zeros((1, V + 1), device=DEV)
    with pytest.raises(ce.CeError):
        ce.argmax_rows(too)


@pytest.mark.parametrize("plan", [(0, 0, 0), (1, 1, 0), (4, 1, 0)], ids=str)
def test_more_rows_than_clusters(orc, plan):
    """Rows beyond the grid's 2^20 clusters: each cluster loops over rows."""
    R, V = (1 << 20) + 37, 6
    x, y = W.random_logits(R, V, sigma=2.0, seed=4)
    ce.debug_force(*plan)
    try:
        res = run_all(x.to(DEV), y.to(DEV), 1.0 / R)
    finally:
        ce.debug_force(0, 0, 0)
    check_all(res, orc, x.numpy(), V, y.numpy(), 1.0 / R, f"{R} rows {plan}")


@pytest.mark.parametrize("cluster", [1, 2, 3, 8])
@pytest.mark.parametrize("vocab", [3001, 50257])
def test_staged_many_rows_per_cluster(orc, cluster, vocab):
    """The persistent staged kernel with many rows per cluster and an odd vocab:
    every row starts at a different 16-byte offset, so each prefetched chunk
    lands in a range that held a differently aligned row."""
    rows = 5000 if vocab < 10000 else 1200
    x, y = W.random_logits(rows, vocab, sigma=4.0, seed=cluster * 13 + vocab)
    y[7] = vocab                    # a bad label inside the pipeline
    x[11, 5] = float("nan")         # a NaN row inside the pipeline
    ce.debug_force(1, cluster, 0)
    try:
        p = ce.plan(ce.OP_GRAD, rows, vocab)
        assert p["path"] == ce.PATH_STAGED and p["cluster"] == cluster
        assert rows > 2 * p["ctas"] // cluster, "want several rows per cluster"
        res = run_all(x.to(DEV), y.to(DEV), 1.0 / rows)
    finally:
        ce.debug_force(0, 0, 0)
    check_all(res, orc, x.numpy(), vocab, y.numpy(), 1.0 / rows, f"staged c{cluster} {rows}x{vocab}")


def test_scales_and_side_stream(orc):
    V, R = 777, 10
    x, y = W.random_logits(R, V, seed=8)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xd, yd = x.to(DEV), y.to(DEV)
        outs = {sc: ce.ce_grad(xd, yd, sc) for sc in (0.0, -2.0, 1e3)}
    s.synchronize()
    for sc, g in outs.items():
        g_ref, _ = orc.ce_grad(x.numpy(), V, y.numpy(), sc)
        if sc == 1e3:   # 1e-6 absolute on a gradient scaled by 1e3 means 1e-9 relative: compare scaled back
            assert_grad(g / 1e3, g_ref / 1e3, "scale 1e3 (divided back)")
        else:
            assert_grad(g, g_ref, f"scale {sc}")


def test_argmax_rows_never_takes_the_even_split(orc):
    """The even split over the whole GPU needs scratch for its per-segment
    keys, which argmax_rows does not have: the automatic plan never picks it,
    and forcing it is refused before any launch (argmax_rows_noalloc, which
    owns a fixed array, runs it)."""
    rows, vocab = 256, 151936
    x, _ = W.random_logits(rows, vocab, seed=77)
    xd = x.to(DEV)
    top = torch.full((rows,), -1.0, device=DEV)
    L = ce.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert ce.plan(ce.OP_ARGMAX, rows, vocab)["path"] != ce.PATH_FLAT
    assert L.argmax_rows(xd.data_ptr(), rows, vocab, vocab, top.data_ptr(), stream) == ce.CE_OK
    torch.cuda.synchronize()
    assert_tokens(top, orc.argmax(x.numpy(), vocab, threads=THREADS), "automatic plan")
    ce.debug_force(5, 0, 0)
    try:
        top.fill_(-1.0)
        assert L.argmax_rows(xd.data_ptr(), rows, vocab, vocab, top.data_ptr(), stream) == ce.CE_EINVAL
        torch.cuda.synchronize()
        assert (top == -1.0).all()
        with pytest.raises(ce.CeError):
            ce.plan(ce.OP_ARGMAX, rows, vocab)
    finally:
        ce.debug_force(0, 0, 0)


@pytest.mark.parametrize("offset", [0, 1, 3])
def test_warp_per_row_path(orc, offset):
    """The warp-per-row kernel (path 6): ce_rows, ce_loss and argmax_rows on
    shapes that cross its vector loop, misaligned rows, padding never read,
    and non-finite rows; fused calls reject the path."""
    nan, inf = float("nan"), float("inf")
    ce.debug_force(6, 0, 0)
    try:
        for rows, vocab, stride in ((1, 1, 1), (3, 5, 7), (37, 1000, 1003), (300, 4099, 4099), (2000, 129, 130)):
            x, y = W.random_logits(rows, vocab, stride=stride, sigma=3.0, seed=rows + vocab, pad_value=nan)
            if rows >= 37:
                x[0, 3] = nan
                x[1, :vocab] = -inf
                x[2, 7] = inf
                x[3, :vocab] = 2.0
                y[4] = -1
            buf = torch.full((rows * stride + offset + 8,), 1e30, device=DEV)
            dx = buf[offset: offset + rows * stride].view(rows, stride)
            dx.copy_(x.to(DEV))
            yd = y.to(DEV)
            lr = ce.ce_rows(dx, yd, vocab=vocab)
            mean, lr2 = ce.ce_loss(dx, yd, vocab=vocab)
            top = ce.argmax_rows(dx, vocab=vocab)
            torch.cuda.synchronize()
            l_ref = orc.ce_rows(x.numpy(), vocab, y.numpy())
            assert_loss(lr, l_ref, f"warp ce_rows {rows}x{vocab}")
            assert_loss(lr2, l_ref, f"warp ce_loss rows {rows}x{vocab}")
            assert_mean(mean.item(), orc.ce_mean(l_ref), f"warp mean {rows}x{vocab}")
            assert_tokens(top, orc.argmax(x.numpy(), vocab), f"warp argmax {rows}x{vocab}")
        with pytest.raises(ce.CeError):
            ce.ce_grad(dx, yd, 1.0, vocab=vocab)
    finally:
        ce.debug_force(0, 0, 0)
        ce.device_error_reset()


@pytest.mark.parametrize("words", [4, 4096, (1 << 20) + 12, 38928384])
def test_read_probe_reads_every_word(words):
    """ce_debug_read, the bench's plain-read ceiling, reads every word once:
    its XOR of the words equals the host's."""
    g = torch.Generator().manual_seed(words)
    x = torch.randint(-(2 ** 31), 2 ** 31 - 1, (words,), dtype=torch.int32, generator=g)
    out = ce.debug_read(x.to(DEV))
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(x.numpy().view(np.uint32))
    assert int(out.item()) & 0xFFFFFFFF == int(want)
