"""argmax_rows_noalloc: argmaxInto's tokens without any device allocation by
the library.

Some callers cannot let a library allocate device memory: a runtime that
plans every byte of device memory itself, or a decode loop that cannot afford
the device-wide synchronisation a cudaMalloc may cause. For them the entry
point works out of a fixed 64 KiB array inside the library: it splits the
rows' elements evenly over P = min(2 x SMs, rows x vocab / 8192) CTAs (at
least one), and each CTA leaves one key per row it meets in the array.

These tests call it through the C ABI and check its tokens bit for bit
against the CPU oracle and against argmax_rows on the same inputs, on calls
in a row (a later call finds the earlier call's keys still in the array).
Exact ties are planted across its own split points, beside NaN runs, rows of
NaN or -inf only, and +1e30 padding that must never be read. They pass in a
fresh process -- the first call sets up the array's address -- and after
every other test. This file is collected last.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
THREADS = os.cpu_count() or 1
SCRATCH_KEYS = 8192  # the array's size in keys: rows + P must not exceed it


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def ctas(rows: int, vocab: int) -> int:
    """The CTA count of the entry point's even split."""
    return max(1, min(2 * sms(), rows * vocab // 8192))


def noalloc(x: torch.Tensor, rows: int, vocab: int, stride: int, top: torch.Tensor) -> int:
    """One call through the C ABI on the current stream; returns the status."""
    return ce.lib().argmax_rows_noalloc(ctypes.c_void_p(x.data_ptr()), rows, vocab, stride,
                                        ctypes.c_void_p(top.data_ptr()),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def tokens(x: torch.Tensor, vocab: int) -> np.ndarray:
    rows = x.shape[0]
    top = torch.full((rows,), -1.0, device=DEV)
    st = noalloc(x, rows, vocab, x.stride(0), top)
    torch.cuda.synchronize()
    assert st == ce.CE_OK, ce.status_string(st)
    return top.cpu().numpy()


def case_logits(case: str):
    if case == "decode":
        b = W.generate(W.WORKLOADS[W.DECODE], device=DEV)
        return b.logits, b.workload.vocab
    if case == "odd":
        x, _ = W.random_logits(37, 200003, stride=200007, seed=5, pad_value=1e30)
        return x.to(DEV), 200003
    if case == "one_cta":
        x, _ = W.random_logits(5, 1000, stride=1001, seed=6, pad_value=1e30)
        return x.to(DEV), 1000
    if case == "mid":
        x, _ = W.random_logits(40, 20000, stride=20003, seed=8, pad_value=1e30)
        return x.to(DEV), 20000
    x, _ = W.random_logits(4000, 3001, seed=7)
    return x.to(DEV), 3001


@pytest.mark.parametrize("case", ["decode", "odd", "one_cta", "mid", "many_rows"])
def test_noalloc_matches_the_oracle_and_argmax_rows_twice(orc, case):
    x, vocab = case_logits(case)
    x[0, 3] = x[0, 7] = 1e9               # an exact tie: the lower column wins
    want = orc.argmax(x.cpu().numpy(), vocab, threads=THREADS)
    direct = ce.argmax_rows(x, vocab=vocab).cpu().numpy()
    assert_tokens(direct, want, f"argmax_rows {case}")
    for k in range(2):
        got = tokens(x, vocab)
        assert_tokens(got, want, f"noalloc {case}, call {k} vs the oracle")
        assert np.array_equal(got, direct), f"noalloc {case}, call {k} vs argmax_rows"


def plant_at_splits(x: torch.Tensor, vocab: int, equal: bool):
    """Exact ties straddling every split point e_j = floor(j E / P) of the
    entry point's even split (E = rows x vocab): columns c - 1 and c of the
    row holding element e_j get the same value, so CTA j - 1 holds the lower
    column and CTA j the higher. With `equal`, every tie has one value (the
    first split of a row decides its token); otherwise values rise with j (the
    last split of a row decides)."""
    rows = x.shape[0]
    P = ctas(rows, vocab)
    E = rows * vocab
    for j in range(1, P):
        r, c = divmod(E * j // P, vocab)
        if c >= 1:
            x[r, c - 1] = x[r, c] = 50.0 if equal else 50.0 + j
    return P


@pytest.mark.parametrize("equal", [False, True], ids=["rising", "equal"])
@pytest.mark.parametrize("shape", [(256, 151936, 152064), (3, 1 << 20, 1 << 20), (300, 16384, 16384),
                                   (17, 200003, 200007), (40, 20000, 20003), (5, 1000, 1001)], ids=str)
def test_noalloc_ties_and_specials_at_its_split_points(orc, shape, equal):
    """Ties across the CTAs of its own split, NaN never winning, rows of NaN or
    -inf only giving 0, and +1e30 padding never read -- bit-exact against the
    oracle."""
    rows, vocab, stride = shape
    x, _ = W.random_logits(rows, vocab, stride=stride, sigma=1.0, seed=rows + vocab, pad_value=1e30)
    P = plant_at_splits(x, vocab, equal)
    assert P == ctas(rows, vocab)
    nan, inf = float("nan"), float("inf")
    if rows >= 3:
        x[1, : vocab // 2] = nan               # a long NaN run, several whole CTA segments
        x[2, :vocab] = nan                     # all NaN: token 0
        x[rows - 1, :vocab] = -inf             # all -inf: token 0
    if rows >= 5:
        x[3, :vocab] = nan
        x[3, vocab - 1] = -inf                 # NaN but for one -inf at the end: that column
        x[4, :] = x[4, :].clamp(max=1.0)
        x[4, vocab // 3] = nan                 # a NaN beside the row's max
        x[4, vocab // 3 + 1] = 2.0
    want = orc.argmax(x.numpy(), vocab, threads=THREADS)
    xd = x.to(DEV)
    for k in range(2):
        assert_tokens(tokens(xd, vocab), want, f"noalloc {shape} (P = {P}), call {k}")


def test_noalloc_at_its_row_limit(orc):
    """rows + P = 8192 fits the array and is exact; one row more is refused
    before any launch (CE_ERANGE)."""
    vocab = 512
    rows = SCRATCH_KEYS - 2 * sms()
    assert ctas(rows, vocab) == 2 * sms()
    x, _ = W.random_logits(rows + 1, vocab, seed=11)
    x[rows // 2, 100] = x[rows // 2, 300] = 40.0
    want = orc.argmax(x[:rows].numpy(), vocab, threads=THREADS)
    xd = x.to(DEV)
    assert_tokens(tokens(xd[:rows], vocab), want, f"noalloc at its limit ({rows} rows)")
    top = torch.full((rows + 1,), -1.0, device=DEV)
    st = noalloc(xd, rows + 1, vocab, vocab, top)
    torch.cuda.synchronize()
    assert st == ce.CE_ERANGE, ce.status_string(st)
    assert (top == -1.0).all(), "a rejected call must launch nothing"


def test_noalloc_leaves_device_memory_as_it_was(orc):
    """After a first call, later calls leave the device's free memory exactly
    where it was: nothing is allocated, not even lazily."""
    x, vocab = case_logits("decode")
    rows = x.shape[0]
    top = torch.full((rows,), -1.0, device=DEV)
    assert noalloc(x, rows, vocab, x.stride(0), top) == ce.CE_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert noalloc(x, rows, vocab, x.stride(0), top) == ce.CE_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
    assert_tokens(top, orc.argmax(x.cpu().numpy(), vocab, threads=THREADS), "noalloc after the memory check")


def test_noalloc_rejects_rows_beyond_its_scratch():
    x = torch.zeros((8200, 4), device=DEV)
    top = torch.full((8200,), -1.0, device=DEV)
    st = ce.lib().argmax_rows_noalloc(ctypes.c_void_p(x.data_ptr()), 8200, 4, 4,
                                      ctypes.c_void_p(top.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == ce.CE_ERANGE
    assert "argmax_rows_noalloc" in ce.status_string(st)
    assert (top == -1.0).all(), "a rejected call must launch nothing"
