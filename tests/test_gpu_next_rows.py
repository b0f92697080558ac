"""Parity of the rows beside the loss (through the C ABI) with the f64 CPU
oracle: softmax and log-softmax rows, sampling candidates (candidatesInto),
split sums (splitSumInto), and the device-resident mean of a step replayed
from a CUDA graph.

Small cases are compared in full; the full-size cases run in the launch shape
the bench times and are compared on every row in chunks of rows, plus properties over every
row.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import (assert_candidates, assert_grad, assert_log_softmax, assert_loss, assert_mean,
                    assert_softmax, assert_split_sum, assert_tokens)

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


def both_softmaxes(x, vocab=None, out=None, log_out=None):
    p = ce.softmax_rows(x, vocab=vocab, out=out)
    lp = ce.log_softmax_rows(x, vocab=vocab, out=log_out)
    torch.cuda.synchronize()
    return p, lp


def check_softmaxes(orc, p, lp, xs, vocab, what):
    assert_softmax(p, orc.softmax(xs, vocab, threads=THREADS), f"{what}: softmax")
    assert_log_softmax(lp, orc.log_softmax(xs, vocab, threads=THREADS), f"{what}: log-softmax")


class forced:
    def __init__(self, plan):
        self.plan = plan

    def __enter__(self):
        ce.debug_force(*self.plan)

    def __exit__(self, *exc):
        ce.debug_force(0, 0, 0)


# ---------------------------------------------------------------------------
# softmax and log-softmax rows

@pytest.mark.parametrize("name", ["ce_64x1000", "ce_4096x32000", W.DECODE])
def test_softmax_workloads_in_full(orc, name):
    w = W.WORKLOADS[name]
    b = W.generate(w, device=DEV)
    p, lp = both_softmaxes(b.logits, vocab=w.vocab)
    check_softmaxes(orc, p, lp, b.logits.cpu().numpy(), w.vocab, name)


SOFTMAX_PLANS = [(0, 0, 0), (1, 1, 0), (1, 2, 128), (1, 3, 256), (1, 16, 0), (2, 1, 0), (2, 7, 128),
                 (2, 16, 0), (4, 0, 0), (4, 5, 0)]


@pytest.mark.parametrize("plan", SOFTMAX_PLANS, ids=lambda p: f"path{p[0]}-c{p[1]}-t{p[2]}")
def test_softmax_shapes_and_paths(orc, plan):
    with forced(plan):
        for rows in (1, 2, 3, 33):
            for vocab in (1, 2, 3, 5, 16, 17, 1023, 1025, 4099):
                x, _ = W.random_logits(rows, vocab, sigma=3.0, seed=rows * 131 + vocab)
                p, lp = both_softmaxes(x.to(DEV))
                check_softmaxes(orc, p, lp, x.numpy(), vocab, f"{plan} {rows}x{vocab}")


def test_retired_path_3_is_refused():
    x = torch.zeros((2, 100), device=DEV)
    y = torch.zeros((2,), dtype=torch.int64, device=DEV)
    with forced((3, 1, 0)):
        for call in (lambda: ce.softmax_rows(x), lambda: ce.log_softmax_rows(x), lambda: ce.ce_grad(x, y, 1.0)):
            with pytest.raises(ce.CeError):
                call()


@pytest.mark.parametrize("plan", [(0, 0, 0), (1, 4, 0), (2, 5, 0)], ids=str)
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_softmax_misaligned_base_and_odd_stride(orc, plan, offset):
    rows, vocab = 9, 4099
    with forced(plan):
        for stride, pad in ((vocab, 0.0), (vocab + 1, float("nan")), (vocab + 3, 1e30)):
            x, _ = W.random_logits(rows, vocab, stride=stride, sigma=2.0, seed=offset * 17 + stride,
                                   pad_value=pad)
            buf = torch.full((rows * stride + offset + 8,), 7.0, device=DEV)
            dx = buf[offset: offset + rows * stride].view(rows, stride)
            dx.copy_(x.to(DEV))
            obuf = torch.empty(2, rows * vocab + 4, device=DEV)
            out = obuf[0, offset: offset + rows * vocab].view(rows, vocab)
            lout = obuf[1, offset: offset + rows * vocab].view(rows, vocab)
            p, lp = both_softmaxes(dx, vocab=vocab, out=out, log_out=lout)
            check_softmaxes(orc, p, lp, x.numpy(), vocab, f"off{offset} stride{stride} {plan}")


@pytest.mark.parametrize("plan", [(0, 0, 0), (1, 3, 0), (2, 3, 0)], ids=str)
def test_softmax_nonfinite_rows(orc, plan):
    nan, inf = float("nan"), float("inf")
    V = 2053
    x = W.random_logits(8, V, seed=6)[0]
    x[0, 17] = nan
    x[1, 1500] = inf
    x[2, :] = -inf
    x[3, :] = nan
    x[4, ::2] = -inf          # p = 0 and log p = -inf there
    x[5, :] = 0.0
    x[5, 0] = -0.0
    x[6, 3] = 80.0            # a dominant token: log p close to 0
    with forced(plan):
        p, lp = both_softmaxes(x.to(DEV))
    check_softmaxes(orc, p, lp, x.numpy(), V, f"non-finite {plan}")
    assert np.isneginf(lp[4, ::2].cpu().numpy()).all()


@pytest.mark.parametrize("plan", [(0, 0, 0), (2, 2, 0), (4, 0, 0)], ids=str)
def test_softmax_in_place(orc, plan):
    V, R = 50257, 5
    x, _ = W.random_logits(R, V, sigma=4.0, seed=8)
    ref_p, ref_lp = orc.softmax(x.numpy(), V), orc.log_softmax(x.numpy(), V)
    d1, d2 = x.to(DEV), x.to(DEV)
    with forced(plan):
        p = ce.softmax_rows(d1, out=d1)
        lp = ce.log_softmax_rows(d2, out=d2)
    torch.cuda.synchronize()
    assert p.data_ptr() == d1.data_ptr() and lp.data_ptr() == d2.data_ptr()
    assert_softmax(d1, ref_p, "in-place softmax")
    assert_log_softmax(d2, ref_lp, "in-place log-softmax")


def test_softmax_full_size_every_row(orc):
    """Softmax and log-softmax rows of the 8192 x 128256 workload against the
    oracle on every row, in chunks of rows."""
    w = W.WORKLOADS[W.HEADLINE]
    b = W.generate(w, device=DEV)
    V = w.vocab
    out = torch.empty((w.rows, V), device=DEV)
    ce.softmax_rows(b.logits, out=out)
    torch.cuda.synchronize()
    for a in range(0, w.rows, 512):
        c = min(w.rows, a + 512)
        assert_softmax(out[a:c], orc.softmax(b.logits[a:c].cpu().numpy(), V, threads=THREADS),
                       f"full-size softmax rows {a}..{c - 1}")
    ce.log_softmax_rows(b.logits, out=out)
    torch.cuda.synchronize()
    for a in range(0, w.rows, 512):
        c = min(w.rows, a + 512)
        assert_log_softmax(out[a:c], orc.log_softmax(b.logits[a:c].cpu().numpy(), V, threads=THREADS),
                           f"full-size log-softmax rows {a}..{c - 1}")


def test_softmax_max_vocab(orc):
    V = 1 << 24
    x, _ = W.random_logits(2, V, seed=12)
    p, lp = both_softmaxes(x.to(DEV))
    check_softmaxes(orc, p, lp, x.numpy(), V, "vocab 2^24")


def test_softmax_zero_rows():
    x = torch.empty((0, 100), device=DEV)
    p, lp = both_softmaxes(x)
    assert p.shape == (0, 100) and lp.shape == (0, 100)


# ---------------------------------------------------------------------------
# sampling candidates

def test_candidates_decode_in_full(orc):
    w = W.WORKLOADS[W.DECODE]
    b = W.generate(w, device=DEV)
    cand = ce.candidates_rows(b.logits, vocab=w.vocab)
    ref = orc.candidates(b.logits.cpu().numpy(), w.vocab, threads=THREADS)
    assert_candidates(cand, ref, "decode candidates")
    # the best candidate of each row is its argmax token
    c = cand.cpu().numpy().reshape(w.rows, -1, 2)
    best = [min(((-v, t) for v, t in r if t >= 0)) for r in c]
    assert_tokens(np.array([t for _, t in best], dtype=np.float32),
                  orc.argmax(b.logits.cpu().numpy(), w.vocab, threads=THREADS), "best candidate")


CAND_PLANS = [(0, 0, 0), (0, 1, 0), (0, 2, 0), (0, 3, 256), (2, 4, 0), (0, 5, 256), (0, 6, 0), (0, 8, 0)]


@pytest.mark.parametrize("plan", CAND_PLANS, ids=lambda p: f"path{p[0]}-c{p[1]}-t{p[2]}")
def test_candidates_shapes_ties_and_clusters(orc, plan):
    """Small integers (ties everywhere) and NaN; every vocab crosses the
    256-column blocks differently."""
    g = torch.Generator().manual_seed(plan[1] * 13 + 1)
    with forced(plan):
        for vocab in (1, 3, 255, 256, 257, 1000, 4099, 20011):
            for rows in (1, 5):
                x = torch.randint(0, 7, (rows, vocab), generator=g).float()
                if rows > 1:
                    x[1, torch.randint(0, vocab, (vocab // 3 + 1,), generator=g)] = float("nan")
                cand = ce.candidates_rows(x.to(DEV))
                assert_candidates(cand, orc.candidates(x.numpy(), vocab), f"{plan} {rows}x{vocab}")


@pytest.mark.parametrize("plan", [(0, 0, 0), (0, 1, 0), (0, 3, 0), (0, 4, 0)], ids=str)
@pytest.mark.parametrize("offset", [1, 2, 3])
def test_candidates_misaligned_base_and_odd_stride(orc, plan, offset):
    rows, vocab = 7, 5003
    with forced(plan):
        for stride, pad in ((vocab, 0.0), (vocab + 1, float("nan")), (vocab + 2, 1e30), (vocab + 5, float("inf"))):
            x, _ = W.random_logits(rows, vocab, stride=stride, sigma=2.0, seed=offset * 7 + stride, pad_value=pad)
            buf = torch.full((rows * stride + offset + 8,), 7.0, device=DEV)
            dx = buf[offset: offset + rows * stride].view(rows, stride)
            dx.copy_(x.to(DEV))
            obuf = torch.empty(rows * ce.CANDIDATE_ROW + 4, device=DEV)
            out = obuf[offset: offset + rows * ce.CANDIDATE_ROW].view(rows, ce.CANDIDATE_ROW)
            ce.candidates_rows(dx, vocab=vocab, out=out)
            assert_candidates(out, orc.candidates(x.numpy(), vocab), f"off{offset} stride{stride} {plan}")


@pytest.mark.parametrize("plan", [(0, 0, 0), (0, 1, 0), (0, 4, 0), (0, 7, 0)], ids=str)
def test_candidates_nonfinite_rows(orc, plan):
    nan, inf = float("nan"), float("inf")
    V = 3000
    x = W.random_logits(8, V, seed=10)[0]
    x[0, :] = nan                      # nothing kept anywhere
    x[1, :] = -inf                     # -inf values are kept (they rank above an empty slot)
    x[2, :] = 0.0
    x[2, ::3] = -0.0                   # -0 == +0: ranked by column
    x[3, 100] = inf
    x[3, 356] = inf                    # the same thread: +inf twice, lower column first
    x[4, ::2] = nan
    x[5, :] = nan
    x[5, 4] = -inf                     # one value in the whole row
    x[6, 256:] = nan                   # only the first 256 columns: one value per thread
    x[7, :] = -inf                     # a masked row (a grammar allows three tokens)
    x[7, 5], x[7, 300], x[7, 2999] = 1.5, -2.0, 0.25
    with forced(plan):
        cand = ce.candidates_rows(x.to(DEV))
    assert_candidates(cand, orc.candidates(x.numpy(), V), f"non-finite {plan}")


def test_candidates_many_rows(orc):
    x, _ = W.random_logits(3000, 5003, sigma=3.0, seed=14)
    cand = ce.candidates_rows(x.to(DEV))
    assert_candidates(cand, orc.candidates(x.numpy(), 5003, threads=THREADS), "3000 x 5003")


@pytest.mark.parametrize("plan", [(0, 0, 0), (0, 8, 0)], ids=str)
def test_candidates_max_vocab(orc, plan):
    V = 1 << 24
    x, _ = W.random_logits(1, V, seed=15)
    with forced(plan):
        cand = ce.candidates_rows(x.to(DEV))
    assert_candidates(cand, orc.candidates(x.numpy(), V), f"vocab 2^24 {plan}")


def test_candidates_more_rows_than_clusters(orc):
    """Rows beyond the grid's 2^20 clusters: each cluster loops over rows."""
    R, V = (1 << 20) + 37, 5
    x, _ = W.random_logits(R, V, sigma=2.0, seed=16)
    cand = ce.candidates_rows(x.to(DEV))
    pick = torch.tensor([0, 1, 2, (1 << 20) - 1] + list(range(1 << 20, R)))
    xs = x[pick].numpy()
    assert_candidates(cand[pick.to(DEV)], orc.candidates(xs, V), "rows past the grid")


def test_candidates_full_size_every_row(orc):
    """8192 x 128256 against the oracle on every row, in chunks of rows."""
    w = W.WORKLOADS[W.HEADLINE]
    b = W.generate(w, device=DEV)
    cand = ce.candidates_rows(b.logits)
    torch.cuda.synchronize()
    for a in range(0, w.rows, 1024):
        c = min(w.rows, a + 1024)
        ref = orc.candidates(b.logits[a:c].cpu().numpy(), w.vocab, threads=THREADS)
        assert_candidates(cand[a:c], ref, f"full-size candidates rows {a}..{c - 1}")


# the ring's two chunk sizes (blocks of 256 columns per bulk copy): 32 where
# the grid has at most two CTAs per SM, else 15
def _ring_smem(chunk_blocks, split):
    return 48 + 3 * (chunk_blocks * 256 + 4) * 4 + ((256 * 4 * 8) if split else 0)


@pytest.mark.parametrize("extra", [0, 1], ids=["large-chunks", "small-chunks"])
def test_candidates_both_chunk_sizes(orc, extra):
    """Rows just at and just past two CTAs per SM: the same rows' candidates
    through each chunk size, exact against the oracle (odd vocab: every row
    at another 16-byte phase, ties, NaN and -inf runs inside the chunks)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, V = 2 * sms + extra, 20011
    p = ce.plan(ce.OP_CANDIDATES, rows, V, V + 2)
    assert p["cluster"] == 1 and p["smem"] == _ring_smem(15 if extra else 32, False), p
    x, _ = W.random_logits(rows, V, stride=V + 2, sigma=2.0, seed=17 + extra, pad_value=1e30)
    x[1, ::7] = float("nan")
    x[2, 100:9000] = -float("inf")
    x[3] = torch.randint(0, 3, (V + 2,), generator=torch.Generator().manual_seed(3)).float()
    cand = ce.candidates_rows(x.to(DEV), vocab=V)
    assert_candidates(cand, orc.candidates(x.numpy(), V, threads=THREADS), f"{rows} x {V}")


def test_candidates_zero_rows():
    x = torch.empty((0, 100), device=DEV)
    assert ce.candidates_rows(x).shape == (0, ce.CANDIDATE_ROW)


# ---------------------------------------------------------------------------
# split sums

@pytest.mark.parametrize("add", [False, True])
def test_split_sum_shapes(orc, add):
    g = torch.Generator().manual_seed(21)
    for splits in (1, 2, 3, 4, 5, 8, 17):
        for total in (1, 3, 4, 5, 1000, 1027, 65536):
            parts = (100 * torch.randn(splits, total, generator=g)).float()
            y0 = torch.randn(total, generator=g).float()
            ref = orc.split_sum(y0.numpy(), parts.numpy(), add)
            y = y0.to(DEV)
            ce.split_sum(parts.to(DEV), y, add=add)
            assert_split_sum(y, ref, y0.numpy(), parts.numpy(), add, f"{splits}x{total} add={add}")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_split_sum_misaligned(orc, offset):
    g = torch.Generator().manual_seed(offset)
    splits, total = 6, 4096
    parts = torch.randn(splits, total, generator=g).float()
    y0 = torch.randn(total, generator=g).float()
    pb = torch.empty(splits * total + 4, device=DEV)
    dp = pb[offset: offset + splits * total].view(splits, total)
    dp.copy_(parts.to(DEV))
    yb = torch.empty(total + 4, device=DEV)
    dy = yb[offset: offset + total]
    dy.copy_(y0.to(DEV))
    ce.split_sum(dp, dy, add=True)
    assert_split_sum(dy, orc.split_sum(y0.numpy(), parts.numpy(), True), y0.numpy(), parts.numpy(), True,
                     f"misaligned by {offset}")


def test_split_sum_into_part_zero(orc):
    g = torch.Generator().manual_seed(4)
    parts = torch.randn(5, 3001, generator=g).float()
    d = parts.to(DEV)
    y = d[0]
    ce.split_sum(d, y, add=False)
    assert_split_sum(y, orc.split_sum(np.zeros(3001, np.float32), parts.numpy(), False), None, parts.numpy(),
                     False, "y = part 0")


def test_split_sum_nonfinite_and_large(orc):
    splits, total = 4, 1 << 25
    g = torch.Generator(device=DEV).manual_seed(9)
    parts = torch.randn(splits, total, generator=g, device=DEV)
    parts[1, 5] = float("inf")
    parts[2, 6] = float("nan")
    parts[0, 7], parts[3, 7] = float("inf"), float("-inf")
    y = torch.full((total,), float("nan"), device=DEV)    # add=False never reads it
    ce.split_sum(parts, y, add=False)
    pick = torch.cat([torch.arange(0, 16), torch.randint(0, total, (4096,), generator=torch.Generator().manual_seed(1)),
                      torch.tensor([total - 1])]).to(DEV)
    ps = parts[:, pick].cpu().numpy()
    ref = orc.split_sum(np.zeros(pick.numel(), np.float32), ps, False)
    assert_split_sum(y[pick], ref, None, ps, False, "large split sum (sampled)")
    assert np.isinf(y[5].item()) and np.isnan(y[6].item()) and np.isnan(y[7].item())


# ---------------------------------------------------------------------------
# a training and a decode step replayed from one CUDA graph: the mean stays on
# the device, and nothing waits between replays

def test_step_replayed_from_a_cuda_graph(orc):
    R, V = 64, 5003
    sx = torch.zeros((R, V), device=DEV)
    sy = torch.zeros((R,), dtype=torch.int64, device=DEV)
    grad = torch.empty((R, V), device=DEV)
    lr = torch.empty((R,), device=DEV)
    top = torch.empty((R,), device=DEV)
    mean = torch.empty((), dtype=torch.float64, device=DEV)
    cand = torch.empty((R, ce.CANDIDATE_ROW), device=DEV)
    logp = torch.empty((R, V), device=DEV)

    def step():
        ce.ce_grad(sx, sy, 1.0 / R, grad=grad, loss_rows=lr, top=top)
        ce.ce_mean(lr, out=mean)
        ce.candidates_rows(sx, out=cand)
        ce.log_softmax_rows(sx, out=logp)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up: the library reads the device's properties once, outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    batches = [W.random_logits(R, V, sigma=s_, seed=100 + i) for i, s_ in enumerate((1.0, 3.0, 8.0))]
    means = []
    for x, y in batches:
        sx.copy_(x.to(DEV))
        sy.copy_(y.to(DEV))
        graph.replay()
        means.append(mean.clone())  # stays on the device: no host wait per step
    torch.cuda.synchronize()
    x, y = batches[-1]
    g_ref, l_ref = orc.ce_grad(x.numpy(), V, y.numpy(), 1.0 / R)
    assert_grad(grad, g_ref, "graph grad")
    assert_loss(lr, l_ref, "graph loss rows")
    assert_tokens(top, orc.argmax(x.numpy(), V), "graph top")
    assert_candidates(cand, orc.candidates(x.numpy(), V), "graph candidates")
    assert_log_softmax(logp, orc.log_softmax(x.numpy(), V), "graph log-softmax")
    for m, (x, y) in zip(means, batches):
        assert_mean(m.item(), orc.ce_mean(orc.ce_rows(x.numpy(), V, y.numpy())), "graph mean")


@pytest.mark.parametrize("shape", [(64, 5003), (8192, 2000)], ids=["64x5003", "8192x2000"])
def test_grad_step_replayed_from_a_cuda_graph(orc, shape):
    """ce_grad_step (the fused kernel and its mean as a programmatic dependent)
    and ce_loss captured in one CUDA graph: the dependent launches become graph
    edges; replays on new batches give the oracle's results, and the means stay
    on the device."""
    R, V = shape
    sx = torch.zeros((R, V), device=DEV)
    sy = torch.zeros((R,), dtype=torch.int64, device=DEV)
    grad = torch.empty((R, V), device=DEV)
    lr, top, lr2 = (torch.empty((R,), device=DEV) for _ in range(3))
    mean, mean2 = (torch.empty((), dtype=torch.float64, device=DEV) for _ in range(2))

    def step():
        ce.ce_grad_step(sx, sy, 1.0 / R, grad=grad, loss_rows=lr, top=top, mean=mean)
        ce.ce_loss(sx, sy, loss_rows=lr2, out=mean2)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    batches = [W.random_logits(R, V, sigma=s_, seed=200 + i) for i, s_ in enumerate((1.0, 4.0))]
    means = []
    for x, y in batches:
        sx.copy_(x.to(DEV))
        sy.copy_(y.to(DEV))
        graph.replay()
        means.append((mean.clone(), mean2.clone()))
    torch.cuda.synchronize()
    x, y = batches[-1]
    g_ref, l_ref = orc.ce_grad(x.numpy(), V, y.numpy(), 1.0 / R, threads=THREADS)
    assert_grad(grad, g_ref, "graph step grad")
    assert_loss(lr, l_ref, "graph step loss rows")
    assert_loss(lr2, l_ref, "graph ce_loss rows")
    assert_tokens(top, orc.argmax(x.numpy(), V, threads=THREADS), "graph step tokens")
    for (m, m2), (x, y) in zip(means, batches):
        m_ref = orc.ce_mean(orc.ce_rows(x.numpy(), V, y.numpy(), threads=THREADS))
        assert_mean(m.item(), m_ref, "graph step mean")
        assert_mean(m2.item(), m_ref, "graph ce_loss mean")


@pytest.mark.parametrize("rows", [256, 1024], ids=["decode-256", "decode-1024"])
def test_decode_step_replayed_from_a_cuda_graph(orc, rows):
    """A decode step's row calls -- argmax_rows, candidates_rows, softmax_rows
    and log_softmax_rows on the logits of a 151936 vocabulary with a 152064
    stride -- captured once in a CUDA graph and replayed on new logits: every
    replay gives the oracle's tokens, candidates and rows (the kernels keep no
    state between launches that a replay could see)."""
    V, S = 151936, 152064
    sx = torch.zeros((rows, S), device=DEV)
    top = torch.empty((rows,), device=DEV)
    cand = torch.empty((rows, ce.CANDIDATE_ROW), device=DEV)
    soft = torch.empty((rows, V), device=DEV)
    logp = torch.empty((rows, V), device=DEV)

    def step():
        ce.argmax_rows(sx, vocab=V, out=top)
        ce.candidates_rows(sx, vocab=V, out=cand)
        ce.softmax_rows(sx, vocab=V, out=soft)
        ce.log_softmax_rows(sx, vocab=V, out=logp)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for i, sigma in enumerate((1.0, 5.0)):
        x, _ = W.random_logits(rows, V, stride=S, sigma=sigma, seed=300 + rows + i, pad_value=-1e30)
        x[5, 17] = x[5, 90001] = 50.0              # a tie: the lower column
        x[6, :V] = float("nan")
        sx.copy_(x.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        xn = x.numpy()
        what = f"graph replay {i}, {rows} rows"
        assert_tokens(top, orc.argmax(xn, V, threads=THREADS), f"{what}: tokens")
        assert_candidates(cand, orc.candidates(xn, V, threads=THREADS), f"{what}: candidates")
        sample = list(range(0, rows, max(1, rows // 16))) + [5, 6]
        assert_softmax(soft[sample], orc.softmax(xn[sample], V, threads=THREADS), f"{what}: softmax")
        assert_log_softmax(logp[sample], orc.log_softmax(xn[sample], V, threads=THREADS), f"{what}: log-softmax")


def test_every_row_family_gives_the_same_bits_every_run():
    """Fixed-shape reductions and merges: five runs, identical bits (a race in a
    split-row combine or an exchange would show as a difference)."""
    x, y = W.random_logits(300, 20011, sigma=3.0, seed=44)
    xd, yd = x.to(DEV), y.to(DEV)
    cuts = [0, 7001, 13000, 20011]
    parts = xd[:4].contiguous()
    runs = []
    for _ in range(5):
        out = {
            "softmax": ce.softmax_rows(xd), "log_softmax": ce.log_softmax_rows(xd),
            "candidates": ce.candidates_rows(xd), "split_sum": ce.split_sum(parts),
        }
        stats = torch.stack([ce.ce_stats(xd, yd, col0=a, vocab=b - a) for a, b in zip(cuts, cuts[1:])])
        loss, top, comb = ce.ce_stats_combine(stats, yd, cuts[-1])
        out.update(stats=stats, sharded_loss=loss, sharded_top=top, combined=comb)
        torch.cuda.synchronize()
        runs.append({k: v.cpu().numpy().copy() for k, v in out.items()})
    for k in runs[0]:
        for r in runs[1:]:
            assert np.array_equal(runs[0][k].view(np.int32), r[k].view(np.int32)), k
