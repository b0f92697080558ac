"""CPU oracle of the row-wise softmax cross-entropy path (f64, plain C).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library
never does, and this package imports nothing from it.

What each function computes follows the API reference page "gizml:netops"
(gizstack.com/docs/reference/gizml/netops.md), section Functions:
``crossEntropyRows`` (per-row loss), ``crossEntropyLoss`` (mean in f64 in row
order), ``crossEntropyGrad`` ((softmax - onehot) * scale), ``argmaxInto``,
``candidatesInto`` and ``splitSumInto``; section Methods: ``Tensor.argmax``
(first of equals, NaN never wins); section Constants: ``TOP_EACH``,
``CANDIDATE_ROW``. Softmax and log-softmax rows follow the same row statistics
(the gpukit API page's ``gkd_softmax_rows``; a request's ``logprobs`` in the
guide "Tensors, GPU kernels and AI models", Step 5). The C source
``ce_oracle.c`` states each definition, and each reading the pages leave
open, beside its code.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
closed forms, brute force, library routines and invariants; no function is
parity-unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ce_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libceoracle.so")

# Plain gcc; no fast-math, no FMA contraction, so each f64 operation rounds
# once as written in the source.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_default = None


def build(source: str = SOURCE, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile the oracle's C source into a shared library (gcc)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(source)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, source, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


class Oracle:
    """ctypes view of one compiled copy of the oracle.

    Logits are a 2-D float32 array ``[rows, stride]`` (C order); only the
    first ``vocab`` columns of each row are read. Labels are int64 ``[rows]``.
    ``threads`` splits rows across host threads (rows are independent; each
    row is still computed exactly as the C source says).
    """

    def __init__(self, lib_path: str):
        self.path = lib_path
        lib = ctypes.CDLL(lib_path)
        lib.oracle_version.restype = ctypes.c_int
        lib.oracle_ce_rows.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]
        lib.oracle_ce_rows.restype = ctypes.c_int
        lib.oracle_ce_rows_page_f32.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp]
        lib.oracle_ce_rows_page_f32.restype = ctypes.c_int
        lib.oracle_ce_grad.argtypes = [_vp, _i64, _i64, _i64, _vp, ctypes.c_double, _vp, _vp]
        lib.oracle_ce_grad.restype = ctypes.c_int
        lib.oracle_ce_mean.argtypes = [_vp, _i64]
        lib.oracle_ce_mean.restype = ctypes.c_double
        lib.oracle_argmax.argtypes = [_vp, _i64, _i64, _i64, _vp]
        lib.oracle_argmax.restype = ctypes.c_int
        for name in ("oracle_softmax", "oracle_log_softmax", "oracle_candidates"):
            getattr(lib, name).argtypes = [_vp, _i64, _i64, _i64, _vp]
            getattr(lib, name).restype = ctypes.c_int
        lib.oracle_split_sum.argtypes = [_vp, _vp, _i64, _i64, ctypes.c_int, _vp]
        lib.oracle_split_sum.restype = ctypes.c_int
        lib.oracle_ce_stats.argtypes = [_vp, _i64, _i64, _i64, _i64, _vp, _vp]
        lib.oracle_ce_stats.restype = ctypes.c_int
        lib.oracle_ce_stats_combine.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]
        lib.oracle_ce_stats_combine.restype = ctypes.c_int
        self.lib = lib

    # -- helpers ---------------------------------------------------------
    @staticmethod
    def _check(logits: np.ndarray, vocab: int):
        if logits.dtype != np.float32 or logits.ndim != 2:
            raise TypeError("logits must be a 2-D float32 array [rows, stride]")
        if not logits.flags["C_CONTIGUOUS"]:
            raise ValueError("logits must be C-contiguous")
        rows, stride = logits.shape
        if vocab < 1 or vocab > stride:
            raise ValueError(f"need 1 <= vocab <= stride (vocab={vocab}, stride={stride})")
        return rows, stride

    @staticmethod
    def _chunks(rows: int, threads: int):
        threads = max(1, min(threads, rows))
        step = -(-rows // threads) if rows else 0
        return [(a, min(rows, a + step)) for a in range(0, rows, step)] if rows else []

    def _run(self, fn, rows: int, threads: int):
        parts = self._chunks(rows, threads)
        if len(parts) <= 1:
            for a, b in parts:
                fn(a, b)
            return
        with ThreadPoolExecutor(len(parts)) as ex:
            for f in [ex.submit(fn, a, b) for a, b in parts]:
                f.result()

    # -- the four operations --------------------------------------------
    def ce_rows(self, logits: np.ndarray, vocab: int, labels: np.ndarray, threads: int = 1):
        """Per-row loss (crossEntropyRows), f64 [rows]."""
        rows, stride = self._check(logits, vocab)
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        out = np.empty(rows, dtype=np.float64)

        def fn(a, b):
            rc = self.lib.oracle_ce_rows(logits[a:b].ctypes.data, b - a, vocab, stride,
                                         labels[a:b].ctypes.data, out[a:b].ctypes.data)
            if rc:
                raise ValueError("oracle_ce_rows rejected its arguments")

        self._run(fn, rows, threads)
        return out

    def ce_rows_page_f32(self, logits: np.ndarray, vocab: int, labels: np.ndarray, threads: int = 1):
        """Diagnostic, not a reference: the row loss in the literal f32 form
        (16 lanes joined pairwise, m + logf(s) - x[label]), f32 [rows]."""
        rows, stride = self._check(logits, vocab)
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        out = np.empty(rows, dtype=np.float32)

        def fn(a, b):
            rc = self.lib.oracle_ce_rows_page_f32(logits[a:b].ctypes.data, b - a, vocab, stride,
                                                  labels[a:b].ctypes.data, out[a:b].ctypes.data)
            if rc:
                raise ValueError("oracle_ce_rows_page_f32 rejected its arguments")

        self._run(fn, rows, threads)
        return out

    def ce_grad(self, logits: np.ndarray, vocab: int, labels: np.ndarray, scale: float,
                threads: int = 1):
        """Gradient (crossEntropyGrad) f64 [rows, vocab] and the row losses f64 [rows]."""
        rows, stride = self._check(logits, vocab)
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        grad = np.empty((rows, vocab), dtype=np.float64)
        loss = np.empty(rows, dtype=np.float64)

        def fn(a, b):
            rc = self.lib.oracle_ce_grad(logits[a:b].ctypes.data, b - a, vocab, stride,
                                         labels[a:b].ctypes.data, float(scale),
                                         grad[a:b].ctypes.data, loss[a:b].ctypes.data)
            if rc:
                raise ValueError("oracle_ce_grad rejected its arguments")

        self._run(fn, rows, threads)
        return grad, loss

    def ce_mean(self, loss_rows: np.ndarray) -> float:
        """Mean of the row losses in f64 in row order (crossEntropyLoss)."""
        loss_rows = np.ascontiguousarray(loss_rows, dtype=np.float64)
        return float(self.lib.oracle_ce_mean(loss_rows.ctypes.data, loss_rows.shape[0]))

    def ce_loss(self, logits: np.ndarray, vocab: int, labels: np.ndarray, threads: int = 1):
        """crossEntropyLoss: the row losses' mean (f64) and the row losses."""
        rows = self.ce_rows(logits, vocab, labels, threads)
        return self.ce_mean(rows), rows

    def argmax(self, logits: np.ndarray, vocab: int, threads: int = 1):
        """Row argmax (argmaxInto / Tensor.argmax), int64 [rows]."""
        rows, stride = self._check(logits, vocab)
        out = np.empty(rows, dtype=np.int64)

        def fn(a, b):
            rc = self.lib.oracle_argmax(logits[a:b].ctypes.data, b - a, vocab, stride,
                                        out[a:b].ctypes.data)
            if rc:
                raise ValueError("oracle_argmax rejected its arguments")

        self._run(fn, rows, threads)
        return out

    # -- rows beside the loss -------------------------------------------
    def _rows_op(self, name, logits, vocab, width, dtype, threads):
        rows, stride = self._check(logits, vocab)
        out = np.empty((rows, width), dtype=dtype)
        fn_c = getattr(self.lib, name)

        def fn(a, b):
            if fn_c(logits[a:b].ctypes.data, b - a, vocab, stride, out[a:b].ctypes.data):
                raise ValueError(f"{name} rejected its arguments")

        self._run(fn, rows, threads)
        return out

    def softmax(self, logits: np.ndarray, vocab: int, threads: int = 1):
        """Softmax rows exp(x - m) / sum, f64 [rows, vocab]."""
        return self._rows_op("oracle_softmax", logits, vocab, vocab, np.float64, threads)

    def log_softmax(self, logits: np.ndarray, vocab: int, threads: int = 1):
        """Log-softmax rows (x - m) - log1p(t), f64 [rows, vocab]."""
        return self._rows_op("oracle_log_softmax", logits, vocab, vocab, np.float64, threads)

    def candidates(self, logits: np.ndarray, vocab: int, threads: int = 1):
        """Sampling candidates (candidatesInto), f32 [rows, 2048]: pair 4t + k is
        (value, column) of thread t's rank-k value; (-inf, -1) when empty."""
        return self._rows_op("oracle_candidates", logits, vocab, CANDIDATE_ROW, np.float32, threads)

    def split_sum(self, y: np.ndarray, parts: np.ndarray, add: bool):
        """splitSumInto: (add ? y : 0) + the sum of the parts in split order, f64
        [total]. ``parts`` is float32 [splits, total]; ``y`` float32 [total]."""
        parts = np.ascontiguousarray(parts, dtype=np.float32)
        if parts.ndim != 2 or parts.shape[0] < 1:
            raise ValueError("parts must be [splits >= 1, total]")
        splits, total = parts.shape
        y = np.ascontiguousarray(y, dtype=np.float32)
        if y.shape != (total,):
            raise ValueError("y must be [total]")
        out = np.empty(total, dtype=np.float64)
        if self.lib.oracle_split_sum(y.ctypes.data, parts.ctypes.data, total, splits,
                                     1 if add else 0, out.ctypes.data):
            raise ValueError("oracle_split_sum rejected its arguments")
        return out

    # -- vocab-sharded rows ----------------------------------------------
    def ce_stats(self, logits: np.ndarray, col0: int, vocab: int, labels: np.ndarray):
        """Row statistics (m, t, top, x[label] or 0) of the column slice
        [col0, col0 + vocab) of ``logits`` [rows, stride], f64 [rows, 4]."""
        rows, stride = self._check(logits, 1)
        if col0 < 0 or vocab < 1 or col0 + vocab > stride:
            raise ValueError("need 0 <= col0 and col0 + vocab <= stride")
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        out = np.empty((rows, 4), dtype=np.float64)
        if self.lib.oracle_ce_stats(logits.ctypes.data + 4 * col0, rows, vocab, stride, col0,
                                    labels.ctypes.data, out.ctypes.data):
            raise ValueError("oracle_ce_stats rejected its arguments")
        return out

    def ce_stats_combine(self, stats: np.ndarray, vocab_total: int, labels: np.ndarray):
        """Whole-row loss, token, max M and T from slice statistics
        ``stats`` f64 [shards, rows, 4]."""
        stats = np.ascontiguousarray(stats, dtype=np.float64)
        if stats.ndim != 3 or stats.shape[2] != 4 or stats.shape[0] < 1:
            raise ValueError("stats must be [shards >= 1, rows, 4]")
        shards, rows, _ = stats.shape
        labels = np.ascontiguousarray(labels, dtype=np.int64)
        loss = np.empty(rows, np.float64)
        top = np.empty(rows, np.int64)
        m = np.empty(rows, np.float64)
        t = np.empty(rows, np.float64)
        if self.lib.oracle_ce_stats_combine(stats.ctypes.data, shards, rows, vocab_total, labels.ctypes.data,
                                            loss.ctypes.data, top.ctypes.data, m.ctypes.data, t.ctypes.data):
            raise ValueError("oracle_ce_stats_combine rejected its arguments")
        return dict(loss=loss, top=top, m=m, t=t)


# candidatesInto's row: 256 threads x TOP_EACH = 4 (value, token) pairs.
CANDIDATE_THREADS = 256
TOP_EACH = 4
CANDIDATE_ROW = 2 * CANDIDATE_THREADS * TOP_EACH


def load(lib_path: str | None = None) -> Oracle:
    """The oracle built from ``ce_oracle.c`` (compiled on first use), or the
    library at ``lib_path``."""
    global _default
    if lib_path is not None:
        return Oracle(lib_path)
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default
