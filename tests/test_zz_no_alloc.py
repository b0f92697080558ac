"""argmax_rows_noalloc: the tokens of argmax_rows without any device
allocation by the library.

Some callers cannot let a library allocate device memory: a runtime that
plans every byte of device memory itself, or a decode loop that cannot afford
the device-wide synchronisation a cudaMalloc may cause. For them the entry
point works out of a fixed 64 KiB array inside the library. These tests call
it through the C ABI and check its tokens against argmax_rows on the same
inputs, twice in a row (the second call finds the first call's keys still in
the array). They pass in a fresh process -- the first call sets up the array's
address -- and after every other test. This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import row_wise_softmax_ce_gb300 as ce
import workloads as W
from parity import assert_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    ce.debug_force(0, 0, 0)


def _noalloc(x, vocab, stride):
    """One call through the C ABI; returns the tokens (host) and the status."""
    rows = x.shape[0]
    top = torch.full((rows,), -1.0, device=DEV)
    st = ce.lib().argmax_rows_noalloc(ctypes.c_void_p(x.data_ptr()), rows, vocab, stride,
                                      ctypes.c_void_p(top.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return top.cpu().numpy(), st


@pytest.mark.parametrize("case", ["decode", "odd", "small", "many_rows"])
def test_noalloc_matches_argmax_rows_twice(case):
    if case == "decode":
        b = W.generate(W.WORKLOADS[W.DECODE], device=DEV)
        x, vocab = b.logits, b.workload.vocab
    elif case == "odd":
        x, _ = W.random_logits(37, 200003, stride=200007, seed=5, device=DEV)
        vocab = 200003
    elif case == "small":
        x, _ = W.random_logits(5, 1000, seed=6, device=DEV)
        vocab = 1000
    else:
        x, _ = W.random_logits(4000, 3001, seed=7, device=DEV)
        vocab = 3001
    x[0, 3] = x[0, 7] = 1e9               # an exact tie: the lower column wins
    stride = x.stride(0)
    want = ce.argmax_rows(x, vocab=vocab).cpu().numpy()
    for _ in range(2):
        got, st = _noalloc(x, vocab, stride)
        assert st == ce.CE_OK, ce.status_string(st)
        assert_tokens(got, want.astype(np.int64), f"noalloc {case}")


def test_noalloc_rejects_rows_beyond_its_scratch():
    x = torch.zeros((8200, 4), device=DEV)
    top = torch.full((8200,), -1.0, device=DEV)
    st = ce.lib().argmax_rows_noalloc(ctypes.c_void_p(x.data_ptr()), 8200, 4, 4,
                                      ctypes.c_void_p(top.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == ce.CE_ERANGE
    assert "argmax_rows_noalloc" in ce.status_string(st)
    assert (top == -1.0).all(), "a rejected call must launch nothing"
