"""ce_grad_host (C ABI): the training step fed from host memory, the
logits copied in chunks of rows with each chunk's fused kernel running as
soon as it has landed. Checked against the f64 CPU oracle, and against
ce_grad + ce_mean on the same batch already on the device."""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_grad, assert_loss, assert_mean, assert_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def batch(rows, vocab, stride, seed):
    x, y = W.random_logits(rows, vocab, stride=stride, sigma=3.0, seed=seed)  # NaN padding, never read
    return x, y


def check(orc, step, x, y, vocab, scale, what):
    xh = x.numpy()
    g_ref, l_ref = orc.ce_grad(xh, vocab, y.numpy(), scale)
    a_ref = orc.argmax(xh, vocab)
    assert_grad(step.grad, g_ref, f"{what} grad")
    assert_loss(step.loss_rows, l_ref, f"{what} loss")
    assert_tokens(step.top, a_ref, f"{what} top")
    assert_tokens(step.top_h, a_ref, f"{what} top back on the host")
    assert_mean(step.mean_h, orc.ce_mean(l_ref), f"{what} mean back on the host")
    assert step.mean_h.item() == step.mean.item() or (np.isnan(step.mean_h.item()) and np.isnan(step.mean.item()))


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("chunk", [0, 1, 7, 64, 299, 1000])
def test_host_step_against_the_oracle(orc, chunk, pinned):
    rows, vocab, stride = 300, 5003, 5011
    x, y = batch(rows, vocab, stride, seed=chunk + 11)
    xh, yh = (x.pin_memory(), y.pin_memory()) if pinned else (x, y)
    step = ce.HostStep(rows, vocab, DEV)
    ce.ce_grad_host(xh[:, :vocab], yh, 0.25, step, chunk_rows=chunk)
    torch.cuda.synchronize()
    check(orc, step, x, y, vocab, 0.25, f"chunk {chunk}")
    # the same batch resident on the device through ce_grad + ce_mean
    g, l, t = ce.ce_grad(x.to(DEV)[:, :vocab], y.to(DEV), 0.25, loss_rows=True, top=True)
    torch.cuda.synchronize()
    assert torch.equal(step.top, t)
    if chunk >= rows:
        # one chunk: the same plan as the device call, so the same bits (other
        # chunkings may plan the rows differently: equal within tolerance)
        assert torch.equal(step.grad, g) and torch.equal(step.loss_rows, l)


def test_host_step_in_place_and_back_to_back(orc):
    """Gradient over the staged copy itself; three steps enqueued without a
    sync on the same buffers: each step's copies wait for the previous
    step's kernels, and the host outputs are the last step's."""
    rows, vocab = 257, 20011
    step = ce.HostStep(rows, vocab, DEV, in_place=True)
    assert step.grad.data_ptr() == step.logits.data_ptr()
    batches = [batch(rows, vocab, vocab, seed=s) for s in (1, 2, 3)]
    pinned = [(x.pin_memory(), y.pin_memory()) for x, y in batches]
    for xh, yh in pinned:
        ce.ce_grad_host(xh, yh, 1.0 / rows, step, chunk_rows=40)
    torch.cuda.synchronize()
    x, y = batches[-1]
    check(orc, step, x, y, vocab, 1.0 / rows, "third of three")


def test_host_step_on_a_side_stream(orc):
    rows, vocab = 96, 4099
    x, y = batch(rows, vocab, vocab + 5, seed=5)
    step = ce.HostStep(rows, vocab, DEV)
    xh, yh = x.pin_memory(), y.pin_memory()  # held until the stream is done with them
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ce.ce_grad_host(xh[:, :vocab], yh, -2.0, step)
    s.synchronize()
    check(orc, step, x, y, vocab, -2.0, "side stream")


def test_host_step_zero_rows():
    step = ce.HostStep(0, 7, DEV)
    ce.ce_grad_host(torch.empty(0, 7), torch.empty(0, dtype=torch.int64), 1.0, step)
    torch.cuda.synchronize()
    assert np.isnan(step.mean_h.item())


def test_host_step_shape_mismatch_refused():
    step = ce.HostStep(4, 10, DEV)
    with pytest.raises(ValueError):
        ce.ce_grad_host(torch.zeros(5, 10), torch.zeros(5, dtype=torch.int64), 1.0, step)


def test_host_step_replayed_from_a_cuda_graph(orc):
    """The host-fed step captured once (the copy stream forks from the
    captured stream and joins it again inside the graph); each replay copies
    what the pinned inputs hold at that moment."""
    rows, vocab = 64, 5003
    xh = torch.zeros((rows, vocab)).pin_memory()
    yh = torch.zeros(rows, dtype=torch.int64).pin_memory()
    step = ce.HostStep(rows, vocab, DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ce.ce_grad_host(xh, yh, 1.0 / rows, step, chunk_rows=16)  # warm-up: streams and events made outside
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ce.ce_grad_host(xh, yh, 1.0 / rows, step, chunk_rows=16)
    for seed in (1, 2):
        x, y = W.random_logits(rows, vocab, sigma=3.0, seed=seed)
        xh.copy_(x)
        yh.copy_(y)
        graph.replay()
        torch.cuda.synchronize()
        check(orc, step, x, y, vocab, 1.0 / rows, f"graph replay {seed}")


@pytest.mark.parametrize("name", ["ce_8192x128256", "ce_16384x50257_x30"])
def test_host_step_full_size_every_row(orc, name):
    """The bench's end-to-end step at full size (16 chunks, from pinned host
    memory) against the oracle on every row, in chunks of rows: each row's
    loss, token and gradient, and the mean against the oracle's mean."""
    w = W.WORKLOADS[name]
    b = W.generate(w, device=DEV)
    V = w.vocab
    xh = b.logits.cpu().pin_memory()
    yh = b.labels.cpu().pin_memory()
    step = ce.ce_grad_host(xh[:, :V], yh, b.scale, ce.HostStep(w.rows, V, DEV))
    torch.cuda.synchronize()
    threads = os.cpu_count() or 1
    xn, yn = xh.numpy(), yh.numpy()
    l_all = np.empty(w.rows, dtype=np.float64)
    for a in range(0, w.rows, 512):
        c = min(w.rows, a + 512)
        g_ref, l_ref = orc.ce_grad(xn[a:c], V, yn[a:c], b.scale, threads=threads)
        l_all[a:c] = l_ref
        what = f"{name} rows {a}..{c - 1}"
        assert_grad(step.grad[a:c], g_ref, f"{what}: host step grad")
        assert_loss(step.loss_rows[a:c], l_ref, f"{what}: host step loss")
        assert_tokens(step.top_h[a:c], orc.argmax(xn[a:c], V, threads=threads), f"{what}: host step tokens")
        del g_ref
    assert torch.equal(step.top.cpu(), step.top_h)
    assert_mean(step.mean_h.item(), orc.ce_mean(l_all), f"{name}: host step mean")
