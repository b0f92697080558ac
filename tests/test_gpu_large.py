"""More than 2^31 elements (through the C ABI): 16448 rows x 131073 columns
of a 131080 stride, 8.6 GB of logits. Row 16383 crosses the 2^31st element of
the logits (and, at column 114689 of the dense output, of the gradient); the
last 64 rows lie wholly past it. Every row's loss and token is compared with
the f64 CPU oracle, and the mean with the oracle's own mean; the gradient,
softmax rows and sampling candidates on the crossing row, the rows past it
and a seeded sample."""
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_candidates, assert_grad, assert_loss, assert_mean, assert_softmax, assert_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
THREADS = os.cpu_count() or 1
BIG = W.Workload("ce_16448x131073_s131080", 16448, 131073, 131080, 2.0, seed=9, scale=1.0 / 16448,
                 pad_value=1e30, tie_frac=0.05)
CHUNK_ROWS = 1024


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def test_more_than_2_31_elements(orc):
    R, V, S = BIG.rows, BIG.vocab, BIG.stride
    assert (R - 65) * S < 2 ** 31 <= (R - 64) * S and R * V > 2 ** 31
    free, _ = torch.cuda.mem_get_info()
    if free < 20 * 2 ** 30:
        pytest.skip(f"needs 20 GB of free device memory, {free / 2 ** 30:.1f} GB free")
    b = W.generate(BIG, device=DEV)
    grad, lr, top, mean = ce.ce_grad_step(b.logits, b.labels, BIG.scale, vocab=V)
    rows2 = ce.ce_rows(b.logits, b.labels, vocab=V)
    top2 = ce.argmax_rows(b.logits, vocab=V)
    cand = ce.candidates_rows(b.logits, vocab=V)
    torch.cuda.synchronize()

    labels = b.labels.cpu().numpy()
    l_ref = np.empty(R)
    a_ref = np.empty(R, dtype=np.int64)
    for r0 in range(0, R, CHUNK_ROWS):
        r1 = min(R, r0 + CHUNK_ROWS)
        xs = b.logits[r0:r1].cpu().numpy()
        l_ref[r0:r1] = orc.ce_rows(xs, V, labels[r0:r1], threads=THREADS)
        a_ref[r0:r1] = orc.argmax(xs, V, threads=THREADS)
    assert_loss(lr, l_ref, "ce_grad_step loss rows")
    assert_loss(rows2, l_ref, "ce_rows")
    assert_tokens(top, a_ref, "ce_grad_step tokens")
    assert_tokens(top2, a_ref, "argmax_rows")
    assert_mean(mean.item(), orc.ce_mean(l_ref), "ce_grad_step mean")

    rng = np.random.default_rng(9)
    sample = sorted(set(range(R - 65, R)) | set(int(r) for r in rng.choice(R - 65, 63, replace=False)))
    idx = torch.tensor(sample, device=DEV)
    xs = b.logits[idx].cpu().numpy()
    g_ref, _ = orc.ce_grad(xs, V, labels[sample], BIG.scale, threads=THREADS)
    assert_grad(grad[idx], g_ref, "ce_grad_step gradient (sampled rows)")
    assert_candidates(cand[idx], orc.candidates(xs, V, threads=THREADS), "candidates_rows (sampled rows)")
    soft = ce.softmax_rows(b.logits, vocab=V, out=grad)
    torch.cuda.synchronize()
    assert_softmax(soft[idx], orc.softmax(xs, V, threads=THREADS), "softmax_rows (sampled rows)")
