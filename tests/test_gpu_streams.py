"""Every entry point at once on four CUDA streams (through the C ABI): the
calls share no scratch, so work enqueued on several streams and run
concurrently gives each its own results -- the f64 CPU oracle's, within the
tolerances, and the same bits in every pass."""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import (assert_candidates, assert_grad, assert_log_softmax, assert_loss, assert_mean,
                    assert_softmax, assert_tokens)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
THREADS = os.cpu_count() or 1
PASSES = 3


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_entry_points_concurrent_on_four_streams(orc):
    # four batches of different shapes, so the calls take different kernels:
    # the fused step (staged, odd vocab), the row losses and their mean (one
    # warp per row), argmax and candidates (decode, cluster-split streaming
    # and the chunk ring), softmax / log-softmax / row losses (few rows)
    xa, ya = W.random_logits(1024, 50257, sigma=4.0, seed=21)
    xb, yb = W.random_logits(4096, 32000, sigma=2.0, seed=22)
    bc = W.generate(W.WORKLOADS[W.DECODE], device=DEV)
    xd, yd = W.random_logits(300, 16385, stride=16392, sigma=3.0, seed=24, pad_value=1e30)
    da, dya = xa.to(DEV), ya.to(DEV)
    db, dyb = xb.to(DEV), yb.to(DEV)
    dd, dyd = xd.to(DEV), yd.to(DEV)
    Vc = bc.workload.vocab
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream() for _ in range(4)]
    passes = []
    for _ in range(PASSES):
        out = {}
        # enqueue round-robin, one call per stream at a time, so the streams' work interleaves
        with torch.cuda.stream(streams[0]):
            out["step"] = ce.ce_grad_step(da, dya, 1.0 / 1024)
        with torch.cuda.stream(streams[1]):
            out["loss"] = ce.ce_loss(db, dyb)
        with torch.cuda.stream(streams[2]):
            out["top"] = ce.argmax_rows(bc.logits, vocab=Vc)
        with torch.cuda.stream(streams[3]):
            out["soft"] = ce.softmax_rows(dd, vocab=16385)
        with torch.cuda.stream(streams[2]):
            out["cand"] = ce.candidates_rows(bc.logits, vocab=Vc)
        with torch.cuda.stream(streams[3]):
            out["logp"] = ce.log_softmax_rows(dd, vocab=16385)
            out["rows"] = ce.ce_rows(dd, dyd, vocab=16385)
        passes.append(out)
    torch.cuda.synchronize()

    first = passes[0]
    g_ref, l_ref = orc.ce_grad(xa.numpy(), 50257, ya.numpy(), 1.0 / 1024, threads=THREADS)
    grad, lr, top, mean = first["step"]
    assert_grad(grad, g_ref, "ce_grad_step grad")
    assert_loss(lr, l_ref, "ce_grad_step loss rows")
    assert_tokens(top, orc.argmax(xa.numpy(), 50257, threads=THREADS), "ce_grad_step tokens")
    assert_mean(mean.item(), orc.ce_mean(l_ref), "ce_grad_step mean")

    m_ref, lb_ref = orc.ce_loss(xb.numpy(), 32000, yb.numpy(), threads=THREADS)
    assert_mean(first["loss"][0].item(), m_ref, "ce_loss mean")
    assert_loss(first["loss"][1], lb_ref, "ce_loss rows")

    xc = bc.logits.cpu().numpy()
    assert_tokens(first["top"], orc.argmax(xc, Vc, threads=THREADS), "argmax_rows decode")
    assert_candidates(first["cand"], orc.candidates(xc, Vc, threads=THREADS), "candidates_rows decode")

    xdn = xd.numpy()
    assert_softmax(first["soft"], orc.softmax(xdn, 16385, threads=THREADS), "softmax_rows")
    assert_log_softmax(first["logp"], orc.log_softmax(xdn, 16385, threads=THREADS), "log_softmax_rows")
    assert_loss(first["rows"], orc.ce_rows(xdn, 16385, yd.numpy(), threads=THREADS), "ce_rows")

    def flat(o):
        ts = o if isinstance(o, tuple) else (o,)
        return [t.cpu().numpy().reshape(-1).view(np.uint8) for t in ts]

    for k, later in enumerate(passes[1:], 1):
        for name in first:
            for a, b in zip(flat(first[name]), flat(later[name])):
                assert np.array_equal(a, b), f"{name}: pass {k} differs from pass 0"


def test_entry_points_from_four_host_threads(orc):
    """The C ABI called from four host threads at once (ctypes releases the
    interpreter lock during each call), each on its own stream and its own
    batch: the library's host state -- device table, forced-plan settings,
    the host pipe -- is shared under a lock, and every thread gets the
    oracle's results."""
    import threading
    shapes = [(300, 50257), (64, 151936), (1024, 32000), (37, 100003)]
    batches = [W.random_logits(R, V, sigma=3.0, seed=40 + i) for i, (R, V) in enumerate(shapes)]
    results = [None] * len(shapes)
    errors = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            x, y = batches[i]
            dx, dy = x.to(DEV), y.to(DEV)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                outs = []
                for _ in range(3):
                    grad, lr, top, mean = ce.ce_grad_step(dx, dy, 0.5)
                    outs.append((grad, lr, top, mean, ce.argmax_rows(dx), ce.candidates_rows(dx)))
            st.synchronize()
            results[i] = [tuple(t.cpu() for t in o) for o in outs]
        except Exception as e:  # reported by the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for i, ((x, y), (R, V)) in enumerate(zip(batches, shapes)):
        xn, yn = x.numpy(), y.numpy()
        g_ref, l_ref = orc.ce_grad(xn, V, yn, 0.5, threads=THREADS)
        a_ref = orc.argmax(xn, V, threads=THREADS)
        c_ref = orc.candidates(xn, V, threads=THREADS)
        first = results[i][0]
        assert_grad(first[0], g_ref, f"thread {i}: gradient")
        assert_loss(first[1], l_ref, f"thread {i}: loss rows")
        assert_tokens(first[2], a_ref, f"thread {i}: step tokens")
        assert_mean(first[3].item(), orc.ce_mean(l_ref), f"thread {i}: mean")
        assert_tokens(first[4], a_ref, f"thread {i}: argmax_rows")
        assert_candidates(first[5], c_ref, f"thread {i}: candidates")
        for k, later in enumerate(results[i][1:], 1):
            for a, b in zip(first, later):
                assert torch.equal(a.reshape(-1).view(torch.uint8), b.reshape(-1).view(torch.uint8)), \
                    f"thread {i}: call {k} differs from call 0"
