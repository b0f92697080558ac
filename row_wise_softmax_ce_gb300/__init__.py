"""Row-wise softmax cross-entropy, its gradient, and the row argmax on NVIDIA
GB300 (sm_103a).

A thin binding over the C ABI of ``libcerows.so`` (declared in
``include/ce_rows.h``): each function checks the tensors it is given,
passes their device pointers and the current CUDA stream to the entry point
of the same name, and returns. Every step of the computation runs in the
library's CUDA kernels; there is no other implementation to fall back to, so
a missing library is an error.

What the operations compute (API reference page "gizml:netops", section
Functions, and section Methods for the argmax rule):

- ``ce_rows``      crossEntropyRows: each row's loss m + log(sum exp(x - m)) - x[label]
- ``ce_mean``      the f64 mean of row losses (the last step of crossEntropyLoss)
- ``ce_loss``      crossEntropyLoss: ``ce_rows`` then ``ce_mean``
- ``ce_grad``      crossEntropyGrad: (softmax - onehot) * scale, optionally with
                   the row losses (and, through ``ce_grad_step``, the argmax
                   tokens) from the same read
- ``ce_grad_step`` the whole step from one read of the logits: gradient, row
                   losses, argmax tokens and the f64 mean loss
- ``argmax_rows``  argmaxInto: each row's token (first of equals, NaN never wins) as f32
- ``candidates_rows``  candidatesInto: each row's 2048-float sampling candidates
                   (256 threads x TOP_EACH = 4 (value, token) pairs)
- ``argmax_rows_indirect`` / ``candidates_rows_indirect``  the same over rows
                   given by a device table of addresses (the indirect form)
- ``softmax_rows`` / ``log_softmax_rows``  the softmax and the log probabilities
                   of each row, from the same row statistics as the loss
- ``split_sum``    splitSumInto: y (+)= the sum of split partial results
- ``ce_stats`` / ``ce_stats_combine`` / ``ce_grad_from_stats``  the loss, token
                   and gradient of rows whose vocabulary is split over slices,
                   from one exchange of 16 bytes per row and slice

Logits are a CUDA float32 tensor ``[rows, cols]`` whose rows are contiguous
(``stride(1) == 1``); its row stride ``stride(0)`` may exceed ``vocab``
(padded rows), and ``vocab`` defaults to ``cols``. Labels are int64 ``[rows]``.
Calls are asynchronous on ``torch.cuda.current_stream()``.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcerows.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "ce_rows.h")

CE_OK, CE_EINVAL, CE_EALIGN, CE_ECUDA, CE_EDEVICE, CE_ERANGE = 0, -1, -2, -3, -4, -5
PATH_AUTO, PATH_STAGED, PATH_STREAM, PATH_STAGED_PER_ROW, PATH_FLAT, PATH_WARP, PATH_RING = 0, 1, 2, 4, 5, 6, 7
OP_ROWS, OP_GRAD, OP_ARGMAX, OP_SOFTMAX, OP_LOG_SOFTMAX, OP_CANDIDATES = 0, 1, 2, 3, 4, 5
# candidatesInto's workgroup, TOP_EACH and CANDIDATE_ROW (gizml:netops, Constants)
CANDIDATE_THREADS, TOP_EACH, CANDIDATE_ROW = 256, 4, 2048

_lock = threading.Lock()
_lib = None


class CeError(RuntimeError):
    """A call of the C ABI returned a non-zero status."""

    def __init__(self, fn: str, status: int, text: str, cuda_error: int = 0):
        msg = f"{fn}: {text} (status {status})"
        if status == CE_ECUDA:
            msg += f", cudaError {cuda_error}"
        super().__init__(msg)
        self.status = status


def _bind(lib):
    i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    sig = {
        "ce_rows": [vp, i64, i64, i64, vp, vp, vp],
        "ce_mean": [vp, i64, vp, vp],
        "ce_loss": [vp, i64, i64, i64, vp, vp, vp, vp],
        "ce_grad": [vp, i64, i64, i64, vp, ctypes.c_double, vp, vp, vp],
        "ce_grad_step": [vp, i64, i64, i64, vp, ctypes.c_double, vp, vp, vp, vp, vp],
        "argmax_rows": [vp, i64, i64, i64, vp, vp],
        "argmax_rows_noalloc": [vp, i64, i64, i64, vp, vp],
        "softmax_rows": [vp, i64, i64, i64, vp, vp],
        "log_softmax_rows": [vp, i64, i64, i64, vp, vp],
        "candidates_rows": [vp, i64, i64, i64, vp, vp],
        "split_sum": [vp, vp, i64, i64, i32, vp],
        "argmax_rows_indirect": [vp, i64, i64, vp, vp],
        "candidates_rows_indirect": [vp, i64, i64, vp, vp],
        "ce_stats": [vp, i64, i64, i64, i64, vp, vp, vp],
        "ce_stats_combine": [vp, i64, i64, i64, vp, vp, vp, vp, vp],
        "ce_grad_from_stats": [vp, i64, i64, i64, i64, vp, vp, ctypes.c_double, vp, vp],
        "ce_version": [],
        "ce_last_cuda_error": [],
        "ce_device_error_count": [vp, ctypes.POINTER(ctypes.c_int64)],
        "ce_device_wait_timeouts": [vp, ctypes.POINTER(ctypes.c_int64)],
        "ce_device_error_reset": [vp],
        "ce_debug_force": [i32, i32, i32],
        "ce_debug_grid_cap": [i64],
        "ce_grad_host": [vp, i64, i64, i64, vp, ctypes.c_double, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp],
        "ce_plan": [i32, i64, i64, i64, ctypes.POINTER(ctypes.c_int64)],
        "ce_debug_read": [vp, i64, vp, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    lib.ce_status_string.argtypes = [i32]
    lib.ce_status_string.restype = ctypes.c_char_p
    return lib


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {LIB_PATH} is missing: build it with "
                    "`python -m row_wise_softmax_ce_gb300.build` (or __graft_entry__.build())")
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


def declared_functions(header: str = HEADER) -> list[str]:
    """Names of the functions that include/ce_rows.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*CE_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def _check(fn: str, status: int):
    if status != CE_OK:
        L = lib()
        raise CeError(fn, status, L.ce_status_string(status).decode(), L.ce_last_cuda_error())


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _logits_view(logits: torch.Tensor, vocab: int | None):
    if not isinstance(logits, torch.Tensor) or logits.dtype != torch.float32:
        raise TypeError("logits must be a float32 torch.Tensor")
    if not logits.is_cuda:
        raise ValueError("logits must be on a CUDA device")
    if logits.dim() != 2:
        raise ValueError("logits must be 2-D [rows, cols]")
    rows, cols = logits.shape
    if rows > 0 and cols > 1 and logits.stride(1) != 1:
        raise ValueError("each row of logits must be contiguous (stride(1) == 1)")
    stride = logits.stride(0) if rows > 1 else max(cols, 1)
    vocab = cols if vocab is None else int(vocab)
    if not 1 <= vocab <= cols:
        raise ValueError(f"need 1 <= vocab <= logits.shape[1] (vocab={vocab}, cols={cols})")
    if rows > 1 and stride < vocab:
        raise ValueError("rows of logits overlap (stride(0) < vocab)")
    return rows, vocab, max(stride, vocab)


def _labels(labels: torch.Tensor, rows: int, device):
    if labels.dtype != torch.int64 or labels.dim() != 1 or labels.shape[0] != rows:
        raise ValueError(f"labels must be int64 [rows={rows}]")
    if labels.device != device or not labels.is_contiguous():
        raise ValueError("labels must be contiguous and on the logits' device")
    return labels


def _out(t, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")
    return t


def ce_rows(logits: torch.Tensor, labels: torch.Tensor, vocab: int | None = None,
            out: torch.Tensor | None = None) -> torch.Tensor:
    """crossEntropyRows: each row's loss, f32 ``[rows]``."""
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    labels = _labels(labels, rows, dev)
    out = _out(out, (rows,), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check("ce_rows", lib().ce_rows(logits.data_ptr(), rows, vocab, stride, labels.data_ptr(),
                                         out.data_ptr(), _stream(dev)))
    return out


def ce_mean(loss_rows: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Mean of f32 row losses in f64, as a 0-d float64 tensor on the device."""
    if loss_rows.dtype != torch.float32 or loss_rows.dim() != 1 or not loss_rows.is_contiguous():
        raise ValueError("loss_rows must be a contiguous float32 [rows] tensor")
    dev = loss_rows.device
    out = _out(out, (), torch.float64, dev, "out")
    with torch.cuda.device(dev):
        _check("ce_mean", lib().ce_mean(loss_rows.data_ptr(), loss_rows.shape[0], out.data_ptr(),
                                         _stream(dev)))
    return out


def ce_loss(logits: torch.Tensor, labels: torch.Tensor, vocab: int | None = None,
            loss_rows: torch.Tensor | None = None, out: torch.Tensor | None = None):
    """crossEntropyLoss: the mean loss (0-d float64 on the device) and the row losses."""
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    labels = _labels(labels, rows, dev)
    loss_rows = _out(loss_rows, (rows,), torch.float32, dev, "loss_rows")
    out = _out(out, (), torch.float64, dev, "out")
    with torch.cuda.device(dev):
        _check("ce_loss", lib().ce_loss(logits.data_ptr(), rows, vocab, stride, labels.data_ptr(),
                                         loss_rows.data_ptr(), out.data_ptr(), _stream(dev)))
    return out, loss_rows


def ce_grad(logits: torch.Tensor, labels: torch.Tensor, scale: float, vocab: int | None = None,
            grad: torch.Tensor | None = None, loss_rows: bool | torch.Tensor = False,
            top: bool | torch.Tensor = False):
    """crossEntropyGrad: ``(softmax - onehot) * scale``, dense f32 ``[rows, vocab]``.

    ``grad`` may be ``logits`` itself (in place) when the logits are dense.
    With ``loss_rows`` / ``top`` (True or a tensor) the same kernel also
    writes each row's loss and argmax token (``top`` goes through the C entry
    point ``ce_grad_step``, without its mean); the result is then a tuple
    ``(grad, loss_rows, top)`` with None for what was not asked.
    """
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    labels = _labels(labels, rows, dev)
    grad = _out(grad, (rows, vocab), torch.float32, dev, "grad")
    lr = None if loss_rows is False else _out(None if loss_rows is True else loss_rows,
                                              (rows,), torch.float32, dev, "loss_rows")
    tp = None if top is False else _out(None if top is True else top, (rows,), torch.float32, dev, "top")
    ptr = lambda t: t.data_ptr() if t is not None else None
    with torch.cuda.device(dev):
        if tp is None:
            _check("ce_grad", lib().ce_grad(logits.data_ptr(), rows, vocab, stride, labels.data_ptr(),
                                             float(scale), grad.data_ptr(), ptr(lr), _stream(dev)))
        else:
            _check("ce_grad_step", lib().ce_grad_step(logits.data_ptr(), rows, vocab, stride, labels.data_ptr(),
                                                       float(scale), grad.data_ptr(), ptr(lr), ptr(tp), None,
                                                       _stream(dev)))
    if loss_rows is False and top is False:
        return grad
    return grad, lr, tp


def ce_grad_step(logits: torch.Tensor, labels: torch.Tensor, scale: float, vocab: int | None = None,
                 grad: torch.Tensor | None = None, loss_rows: torch.Tensor | None = None,
                 top: torch.Tensor | None = None, mean: torch.Tensor | None = None):
    """The training step's whole path from one read of the logits: returns
    ``(grad, loss_rows, top, mean)`` -- the gradient (dense f32 ``[rows,
    vocab]``), each row's loss and argmax token (f32 ``[rows]``) and the mean
    loss (0-d float64 on the device). Outputs not given are allocated."""
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    labels = _labels(labels, rows, dev)
    grad = _out(grad, (rows, vocab), torch.float32, dev, "grad")
    loss_rows = _out(loss_rows, (rows,), torch.float32, dev, "loss_rows")
    top = _out(top, (rows,), torch.float32, dev, "top")
    mean = _out(mean, (), torch.float64, dev, "mean")
    with torch.cuda.device(dev):
        _check("ce_grad_step", lib().ce_grad_step(logits.data_ptr(), rows, vocab, stride, labels.data_ptr(),
                                                   float(scale), grad.data_ptr(), loss_rows.data_ptr(),
                                                   top.data_ptr(), mean.data_ptr(), _stream(dev)))
    return grad, loss_rows, top, mean


class HostStep:
    """Device buffers of ``ce_grad_host`` for batches of one shape, kept and
    reused across steps, and the page-locked host outputs it copies back."""

    def __init__(self, rows: int, vocab: int, device, in_place: bool = False):
        dev = torch.device(device)
        self.rows, self.vocab, self.device = rows, vocab, dev
        self.logits = torch.empty((rows, vocab), dtype=torch.float32, device=dev)
        self.labels = torch.empty(rows, dtype=torch.int64, device=dev)
        self.grad = self.logits if in_place else torch.empty((rows, vocab), dtype=torch.float32, device=dev)
        self.loss_rows = torch.empty(rows, dtype=torch.float32, device=dev)
        self.top = torch.empty(rows, dtype=torch.float32, device=dev)
        self.mean = torch.empty((), dtype=torch.float64, device=dev)
        self.mean_h = torch.empty((), dtype=torch.float64, pin_memory=True)
        self.top_h = torch.empty(rows, dtype=torch.float32, pin_memory=True)


def ce_grad_host(logits_h: torch.Tensor, labels_h: torch.Tensor, scale: float, step: HostStep,
                 vocab: int | None = None, chunk_rows: int = 0) -> HostStep:
    """crossEntropyGrad + crossEntropyLoss of a batch in host memory: the
    logits and labels are copied into ``step``'s device buffers chunk by
    chunk, each chunk's gradient, row losses and tokens computed as soon as
    it has landed, then the mean; the mean and tokens come back into
    ``step.mean_h`` / ``step.top_h``. Enqueued on the current stream: read the
    host outputs after synchronising it."""
    if not isinstance(logits_h, torch.Tensor) or logits_h.dtype != torch.float32 or logits_h.is_cuda:
        raise TypeError("logits_h must be a float32 CPU tensor")
    if logits_h.dim() != 2 or (logits_h.shape[1] > 1 and logits_h.stride(1) != 1):
        raise ValueError("logits_h must be 2-D with contiguous rows")
    rows, cols = logits_h.shape
    vocab = cols if vocab is None else int(vocab)
    if not 1 <= vocab <= cols:
        raise ValueError(f"need 1 <= vocab <= logits_h.shape[1] (vocab={vocab}, cols={cols})")
    stride = max(logits_h.stride(0) if rows > 1 else cols, vocab)
    if labels_h.dtype != torch.int64 or labels_h.is_cuda or tuple(labels_h.shape) != (rows,) or \
            not labels_h.is_contiguous():
        raise ValueError(f"labels_h must be a contiguous int64 CPU tensor [rows={rows}]")
    if (step.rows, step.vocab) != (rows, vocab):
        raise ValueError(f"step buffers are for {step.rows} x {step.vocab}, not {rows} x {vocab}")
    dev = step.device
    with torch.cuda.device(dev):
        _check("ce_grad_host", lib().ce_grad_host(
            logits_h.data_ptr(), rows, vocab, stride, labels_h.data_ptr(), float(scale), step.logits.data_ptr(),
            step.labels.data_ptr(), step.grad.data_ptr(), step.loss_rows.data_ptr(), step.top.data_ptr(),
            step.mean.data_ptr(), step.mean_h.data_ptr(), step.top_h.data_ptr(), int(chunk_rows), _stream(dev)))
    return step


def argmax_rows(logits: torch.Tensor, vocab: int | None = None,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """argmaxInto: each row's token as f32 ``[rows]`` (first of equals; NaN never wins)."""
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    out = _out(out, (rows,), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check("argmax_rows", lib().argmax_rows(logits.data_ptr(), rows, vocab, stride, out.data_ptr(),
                                                _stream(dev)))
    return out


def argmax_rows_noalloc(logits: torch.Tensor, vocab: int | None = None,
                        out: torch.Tensor | None = None) -> torch.Tensor:
    """argmaxInto's tokens without any device allocation by the library: for
    callers whose device memory is planned by someone else, or who cannot
    afford an allocation's possible device-wide synchronisation. Uses the
    library's fixed 64 KiB scratch; calls running at the same time on the GPU
    race on it. ``out`` may be given to avoid this wrapper's own allocation."""
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    out = _out(out, (rows,), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check("argmax_rows_noalloc", lib().argmax_rows_noalloc(logits.data_ptr(), rows, vocab, stride,
                                                                out.data_ptr(), _stream(dev)))
    return out


def _rows_out(fn: str, logits, vocab, out, width=None):
    rows, vocab, stride = _logits_view(logits, vocab)
    dev = logits.device
    out = _out(out, (rows, vocab if width is None else width), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check(fn, getattr(lib(), fn)(logits.data_ptr(), rows, vocab, stride, out.data_ptr(), _stream(dev)))
    return out


def softmax_rows(logits: torch.Tensor, vocab: int | None = None,
                 out: torch.Tensor | None = None) -> torch.Tensor:
    """Each row's softmax exp(x - m) * f32(1/sum), dense f32 ``[rows, vocab]``
    (``out`` may be ``logits`` itself when the logits are dense)."""
    return _rows_out("softmax_rows", logits, vocab, out)


def log_softmax_rows(logits: torch.Tensor, vocab: int | None = None,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """Each row's log probabilities (x - m) - log(sum), dense f32 ``[rows, vocab]``."""
    return _rows_out("log_softmax_rows", logits, vocab, out)


def candidates_rows(logits: torch.Tensor, vocab: int | None = None,
                    out: torch.Tensor | None = None) -> torch.Tensor:
    """candidatesInto: f32 ``[rows, 2048]``; pair 4t + k (floats 2(4t+k), +1) is
    thread t's rank-k (value, token) of the columns t, t + 256, ...; (-inf, -1)
    where thread t read fewer than 4 values."""
    return _rows_out("candidates_rows", logits, vocab, out, CANDIDATE_ROW)


def row_addresses(logits: torch.Tensor, index: torch.Tensor) -> torch.Tensor:
    """Device addresses (int64) of the rows ``logits[index]``, for the indirect calls."""
    if not logits.is_cuda or logits.dim() != 2 or logits.dtype != torch.float32:
        raise ValueError("logits must be a 2-D float32 CUDA tensor")
    index = index.to(device=logits.device, dtype=torch.int64)
    return logits.data_ptr() + index * (logits.stride(0) * 4)


def _row_table(row_addrs: torch.Tensor):
    if row_addrs.dtype not in (torch.int64, torch.uint64) or row_addrs.dim() != 1 or not row_addrs.is_cuda \
            or not row_addrs.is_contiguous():
        raise ValueError("row_addrs must be a contiguous 1-D int64 CUDA tensor of row addresses")
    return row_addrs


def argmax_rows_indirect(row_addrs: torch.Tensor, vocab: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """argmaxInto, indirect form: the token (f32) of each row read at the device
    address ``row_addrs[i]`` (``vocab`` floats each); NaN for a null or
    misaligned address."""
    row_addrs = _row_table(row_addrs)
    rows, dev = row_addrs.shape[0], row_addrs.device
    out = _out(out, (rows,), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check("argmax_rows_indirect", lib().argmax_rows_indirect(row_addrs.data_ptr(), rows, int(vocab),
                                                                  out.data_ptr(), _stream(dev)))
    return out


def candidates_rows_indirect(row_addrs: torch.Tensor, vocab: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """candidatesInto, indirect form: ``[rows, 2048]`` candidates of the rows at
    the addresses ``row_addrs``."""
    row_addrs = _row_table(row_addrs)
    rows, dev = row_addrs.shape[0], row_addrs.device
    out = _out(out, (rows, CANDIDATE_ROW), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check("candidates_rows_indirect", lib().candidates_rows_indirect(row_addrs.data_ptr(), rows, int(vocab),
                                                                          out.data_ptr(), _stream(dev)))
    return out


def split_sum(parts: torch.Tensor, y: torch.Tensor | None = None, add: bool = False) -> torch.Tensor:
    """splitSumInto: ``y = (y if add else 0) + parts[0] + ... + parts[-1]`` in f32
    in split order. ``parts`` is a contiguous f32 ``[splits, total]`` tensor;
    ``y`` f32 ``[total]`` (allocated when None; then ``add`` must be False)."""
    if parts.dtype != torch.float32 or parts.dim() != 2 or not parts.is_contiguous() or not parts.is_cuda:
        raise ValueError("parts must be a contiguous float32 CUDA tensor [splits, total]")
    splits, total = parts.shape
    dev = parts.device
    if y is None and add:
        raise ValueError("add=True needs y")
    y = _out(y, (total,), torch.float32, dev, "y")
    with torch.cuda.device(dev):
        _check("split_sum", lib().split_sum(y.data_ptr(), parts.data_ptr(), total, splits, 1 if add else 0,
                                            _stream(dev)))
    return y


# -- vocab-sharded cross-entropy ------------------------------------------------

def _slice_view(logits: torch.Tensor, col0: int, vocab: int | None):
    rows, cols = logits.shape
    vocab = cols - col0 if vocab is None else int(vocab)
    if col0 < 0 or vocab < 1 or col0 + vocab > cols:
        raise ValueError(f"need 0 <= col0 and col0 + vocab <= logits.shape[1] (col0={col0}, vocab={vocab})")
    view = logits[:, col0: col0 + vocab]
    r, v, stride = _logits_view(view, vocab)
    return view, r, v, stride


def ce_stats(logits: torch.Tensor, labels: torch.Tensor, col0: int = 0, vocab: int | None = None,
             out: torch.Tensor | None = None) -> torch.Tensor:
    """Row statistics (m, t, top, x[label] or 0) of the column slice
    ``logits[:, col0:col0 + vocab]`` of whole rows, f32 ``[rows, 4]``;
    ``labels`` are the rows' global columns. For a shard held on its own (its
    first column being global column col0) use ``ce_stats_shard``."""
    view, rows, vocab, stride = _slice_view(logits, col0, vocab)
    return ce_stats_shard(view, labels, col0, out=out)


def ce_stats_shard(shard: torch.Tensor, labels: torch.Tensor, col0: int,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """Row statistics of a shard ``[rows, width]`` (row-contiguous, any row
    stride) whose first column is global column ``col0``; f32 ``[rows, 4]``."""
    rows, vocab, stride = _logits_view(shard, None)
    dev = shard.device
    labels = _labels(labels, rows, dev)
    out = _out(out, (rows, 4), torch.float32, dev, "out")
    with torch.cuda.device(dev):
        _check("ce_stats", lib().ce_stats(shard.data_ptr(), rows, vocab, stride, int(col0), labels.data_ptr(),
                                           out.data_ptr(), _stream(dev)))
    return out


def ce_stats_combine(stats: torch.Tensor, labels: torch.Tensor, vocab_total: int,
                     loss_rows: bool | torch.Tensor = True, top: bool | torch.Tensor = True,
                     combined: bool | torch.Tensor = True):
    """Merge slices' statistics ``stats`` f32 ``[shards, rows, 4]`` (slices in
    column order) into the whole rows' loss, token and combined (M, T, top,
    x[label]); returns ``(loss_rows, top, combined)`` with None for what was
    not asked."""
    if stats.dtype != torch.float32 or stats.dim() != 3 or stats.shape[2] != 4 or not stats.is_contiguous():
        raise ValueError("stats must be a contiguous float32 [shards, rows, 4] tensor")
    shards, rows, _ = stats.shape
    dev = stats.device
    labels = _labels(labels, rows, dev)
    lr = None if loss_rows is False else _out(None if loss_rows is True else loss_rows, (rows,), torch.float32,
                                              dev, "loss_rows")
    tp = None if top is False else _out(None if top is True else top, (rows,), torch.float32, dev, "top")
    cb = None if combined is False else _out(None if combined is True else combined, (rows, 4), torch.float32,
                                             dev, "combined")
    ptr = lambda t: t.data_ptr() if t is not None else None
    with torch.cuda.device(dev):
        _check("ce_stats_combine", lib().ce_stats_combine(stats.data_ptr(), shards, rows, int(vocab_total),
                                                           labels.data_ptr(), ptr(lr), ptr(tp), ptr(cb),
                                                           _stream(dev)))
    return lr, tp, cb


def ce_grad_from_stats(shard: torch.Tensor, labels: torch.Tensor, col0: int, combined: torch.Tensor,
                       scale: float, grad: torch.Tensor | None = None) -> torch.Tensor:
    """The shard's slice of crossEntropyGrad from the combined row state,
    dense f32 ``[rows, width]`` (``grad`` may be ``shard`` itself when dense)."""
    rows, vocab, stride = _logits_view(shard, None)
    dev = shard.device
    labels = _labels(labels, rows, dev)
    if combined.dtype != torch.float32 or tuple(combined.shape) != (rows, 4) or not combined.is_contiguous():
        raise ValueError(f"combined must be a contiguous float32 [{rows}, 4] tensor")
    grad = _out(grad, (rows, vocab), torch.float32, dev, "grad")
    with torch.cuda.device(dev):
        _check("ce_grad_from_stats", lib().ce_grad_from_stats(shard.data_ptr(), rows, vocab, stride, int(col0),
                                                               labels.data_ptr(), combined.data_ptr(),
                                                               float(scale), grad.data_ptr(), _stream(dev)))
    return grad


# -- diagnostics and tuning ---------------------------------------------------

def version() -> int:
    return lib().ce_version()


def status_string(status: int) -> str:
    return lib().ce_status_string(status).decode()


def device_error_count(device=None) -> tuple[int, int]:
    """(rows seen with a bad label, waits that gave up) on the device, from
    ce_device_error_count and ce_device_wait_timeouts; waits for its stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    bad, waits = ctypes.c_int64(0), ctypes.c_int64(0)
    with torch.cuda.device(dev):
        L = lib()
        _check("ce_device_error_count", L.ce_device_error_count(_stream(dev), ctypes.byref(bad)))
        _check("ce_device_wait_timeouts", L.ce_device_wait_timeouts(_stream(dev), ctypes.byref(waits)))
    return int(bad.value), int(waits.value)


def device_error_reset(device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check("ce_device_error_reset", lib().ce_device_error_reset(_stream(dev)))


def debug_force(path: int = 0, cluster: int = 0, threads: int = 0) -> None:
    """Force the launch plan of later calls (0 = automatic); see ce_debug_force."""
    _check("ce_debug_force", lib().ce_debug_force(path, cluster, threads))


def debug_grid_cap(clusters: int = 0) -> None:
    """Cap the grid of later row-kernel launches at `clusters` clusters (0 = no cap); see ce_debug_grid_cap."""
    _check("ce_debug_grid_cap", lib().ce_debug_grid_cap(clusters))


def debug_read(t: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """Read probe (ce_debug_read): one plain read of the whole of the
    contiguous CUDA tensor ``t``, its words XORed into ``out`` (a uint32-sized
    int32 tensor on the device, zeroed when allocated here)."""
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("t must be a contiguous CUDA tensor")
    nbytes = t.numel() * t.element_size()
    dev = t.device
    if out is None:
        out = torch.zeros((), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check("ce_debug_read", lib().ce_debug_read(t.data_ptr(), nbytes, out.data_ptr(), _stream(dev)))
    return out


def plan(op: int, rows: int, vocab: int, stride: int | None = None) -> dict:
    """The launch plan the library would pick for op (OP_ROWS ... OP_CANDIDATES)."""
    out = (ctypes.c_int64 * 6)()
    _check("ce_plan", lib().ce_plan(op, rows, vocab, vocab if stride is None else stride, out))
    keys = ("path", "cluster", "threads", "smem", "cols", "ctas")
    return dict(zip(keys, (int(v) for v in out)))
