"""The C-ABI library loads and exports every function include/ce_rows.h
declares; host-side argument checks reject bad calls before any launch.
CPU only: no call here reaches a kernel."""
import ctypes

import pytest

import row_wise_softmax_ce_gb300 as ce
from row_wise_softmax_ce_gb300 import build as cuda_build


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return ce.lib()


def test_exports_every_declared_function(lib):
    names = ce.declared_functions()
    assert set(names) >= {"ce_rows", "ce_mean", "ce_loss", "ce_grad", "ce_grad_step", "argmax_rows",
                          "ce_status_string",
                          "ce_version", "ce_last_cuda_error", "ce_device_error_count", "ce_device_wait_timeouts",
                          "ce_device_error_reset", "ce_debug_force", "ce_debug_grid_cap", "ce_plan", "ce_debug_read", "softmax_rows",
                          "log_softmax_rows", "candidates_rows", "split_sum", "argmax_rows_noalloc",
                          "argmax_rows_indirect", "candidates_rows_indirect"}
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_only_declared_functions_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", ce.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == set(ce.declared_functions()), exported ^ set(ce.declared_functions())


def test_version_and_status_strings(lib):
    assert ce.version() == 10000
    for st in (ce.CE_OK, ce.CE_EINVAL, ce.CE_EALIGN, ce.CE_ECUDA, ce.CE_EDEVICE, 12345):
        assert isinstance(ce.status_string(st), str) and ce.status_string(st)


V = ctypes.c_void_p


@pytest.mark.parametrize("args", [
    (V(256), -1, 10, 10),        # rows < 0
    (V(256), 4, 0, 10),          # vocab < 1
    (V(256), 4, 10, 9),          # stride < vocab
    (V(256), 4, (1 << 24) + 1, (1 << 24) + 1),  # token not exact in f32
    (None, 4, 10, 10),           # null logits
])
def test_bad_sizes_rejected_before_launch(lib, args):
    logits, rows, vocab, stride = args
    assert lib.ce_rows(logits, rows, vocab, stride, V(512), V(1024), None) == ce.CE_EINVAL
    assert lib.argmax_rows(logits, rows, vocab, stride, V(1024), None) == ce.CE_EINVAL
    assert lib.ce_grad(logits, rows, vocab, stride, V(512), 1.0, V(4096), None, None) == ce.CE_EINVAL
    assert lib.ce_grad_step(logits, rows, vocab, stride, V(512), 1.0, V(4096), V(1 << 20), None, V(1 << 21),
                            None) == ce.CE_EINVAL
    for fn in (lib.softmax_rows, lib.log_softmax_rows, lib.candidates_rows):
        assert fn(logits, rows, vocab, stride, V(1 << 20), None) == ce.CE_EINVAL


def test_misaligned_pointers_rejected(lib):
    assert lib.ce_rows(V(258), 4, 10, 10, V(512), V(1024), None) == ce.CE_EALIGN
    assert lib.ce_rows(V(256), 4, 10, 10, V(516), V(1024), None) == ce.CE_EALIGN     # labels need 8 B
    assert lib.argmax_rows(V(256), 4, 10, 10, V(1026), None) == ce.CE_EALIGN
    assert lib.ce_grad_step(V(256), 4, 10, 10, V(512), 1.0, V(4096), V(1 << 20), V((1 << 21) + 2), None,
                            None) == ce.CE_EALIGN                                     # tokens 4 B
    assert lib.ce_grad_step(V(256), 4, 10, 10, V(512), 1.0, V(4096), V(1 << 20), None, V((1 << 21) + 4),
                            None) == ce.CE_EALIGN                                     # double mean
    assert lib.ce_mean(V(256), 4, V(260), None) == ce.CE_EALIGN                       # double out


def test_null_outputs_and_bad_scale_rejected(lib):
    assert lib.ce_rows(V(256), 4, 10, 10, None, V(1024), None) == ce.CE_EINVAL
    assert lib.ce_rows(V(256), 4, 10, 10, V(512), None, None) == ce.CE_EINVAL
    assert lib.argmax_rows(V(256), 4, 10, 10, None, None) == ce.CE_EINVAL
    assert lib.ce_mean(V(256), 4, None, None) == ce.CE_EINVAL
    assert lib.ce_loss(V(256), 4, 10, 10, V(512), V(1024), None, None) == ce.CE_EINVAL
    for s in (float("nan"), float("inf")):
        assert lib.ce_grad(V(256), 4, 10, 10, V(512), s, V(4096), None, None) == ce.CE_EINVAL
        assert lib.ce_grad_step(V(256), 4, 10, 10, V(512), s, V(4096), None, None, None, None) == ce.CE_EINVAL
    assert lib.ce_grad(V(256), 4, 10, 10, V(512), 1.0, None, None, None) == ce.CE_EINVAL
    # the step's mean reads the row losses: a mean without them is refused
    assert lib.ce_grad_step(V(256), 4, 10, 10, V(512), 1.0, V(4096), None, None, V(1 << 21), None) == ce.CE_EINVAL
    # the debug counters need somewhere to write
    assert lib.ce_device_error_count(None, None) == ce.CE_EINVAL
    assert lib.ce_device_wait_timeouts(None, None) == ce.CE_EINVAL


def test_grad_overlap_rules(lib):
    # in place needs stride == vocab; a partial overlap is rejected
    assert lib.ce_grad(V(4096), 4, 10, 12, V(512), 1.0, V(4096), None, None) == ce.CE_EINVAL
    assert lib.ce_grad(V(4096), 4, 10, 10, V(512), 1.0, V(4100), None, None) == ce.CE_EINVAL
    assert lib.ce_grad_step(V(4096), 4, 10, 10, V(512), 1.0, V(4100), None, None, None, None) == ce.CE_EINVAL


def test_rows_beside_the_loss_validation(lib):
    for fn in (lib.softmax_rows, lib.log_softmax_rows, lib.candidates_rows):
        assert fn(V(256), 4, 10, 10, None, None) == ce.CE_EINVAL          # no output
        assert fn(V(256), 4, 10, 10, V(1 << 20 | 2), None) == ce.CE_EALIGN
        assert fn(None, 0, 10, 10, None, None) == ce.CE_OK                # nothing launched
    # in place needs stride == vocab; any partial overlap is rejected
    assert lib.softmax_rows(V(4096), 4, 10, 12, V(4096), None) == ce.CE_EINVAL
    assert lib.log_softmax_rows(V(4096), 4, 10, 10, V(4100), None) == ce.CE_EINVAL
    # candidates never alias the logits
    assert lib.candidates_rows(V(4096), 4, 10, 10, V(4096), None) == ce.CE_EINVAL
    assert lib.candidates_rows(V(1 << 20), 2, 10, 10, V((1 << 20) - 2 * 8192 + 16), None) == ce.CE_EINVAL


def test_split_sum_validation(lib):
    assert lib.split_sum(V(256), V(1 << 20), 10, 0, 0, None) == ce.CE_EINVAL     # splits < 1
    assert lib.split_sum(V(256), V(1 << 20), -1, 2, 0, None) == ce.CE_EINVAL     # total < 0
    assert lib.split_sum(None, V(1 << 20), 10, 2, 0, None) == ce.CE_EINVAL
    assert lib.split_sum(V(256), None, 10, 2, 1, None) == ce.CE_EINVAL
    assert lib.split_sum(V(258), V(1 << 20), 10, 2, 0, None) == ce.CE_EALIGN
    assert lib.split_sum(V(256), V(1 << 20), (1 << 62), 4, 0, None) == ce.CE_EINVAL  # bytes overflow
    # y inside the parts but not part 0 itself
    assert lib.split_sum(V(4096 + 40), V(4096), 10, 2, 0, None) == ce.CE_EINVAL
    assert lib.split_sum(None, None, 0, 3, 1, None) == ce.CE_OK                    # nothing launched


def test_vocab_sharded_validation(lib):
    # ce_stats: slice bounds, 16-byte stats, no overlap with the logits
    assert lib.ce_stats(V(256), 4, 10, 10, -1, V(512), V(4096), None) == ce.CE_EINVAL
    assert lib.ce_stats(V(256), 4, 10, 10, (1 << 24) - 5, V(512), V(4096), None) == ce.CE_EINVAL
    assert lib.ce_stats(V(256), 4, 10, 10, 0, None, V(4096), None) == ce.CE_EINVAL
    assert lib.ce_stats(V(256), 4, 10, 10, 0, V(512), V(4100), None) == ce.CE_EALIGN
    assert lib.ce_stats(V(4096), 4, 10, 10, 0, V(512), V(4096 + 16), None) == ce.CE_EINVAL
    assert lib.ce_stats(None, 0, 10, 10, 0, None, None, None) == ce.CE_OK
    # ce_stats_combine
    assert lib.ce_stats_combine(V(4096), 0, 4, 100, V(512), None, None, None, None) == ce.CE_EINVAL
    assert lib.ce_stats_combine(V(4096), 2, 4, (1 << 24) + 1, V(512), None, None, None, None) == ce.CE_EINVAL
    assert lib.ce_stats_combine(V(4104), 2, 4, 100, V(512), None, None, None, None) == ce.CE_EALIGN
    assert lib.ce_stats_combine(V(4096), 2, 4, 100, V(512), None, None, V(4096 + 64), None) == ce.CE_EINVAL
    assert lib.ce_stats_combine(None, 2, 0, 100, None, None, None, None, None) == ce.CE_OK
    # ce_grad_from_stats
    assert lib.ce_grad_from_stats(V(256), 4, 10, 10, 0, V(512), V(1024), float("nan"), V(8192), None) == ce.CE_EINVAL
    assert lib.ce_grad_from_stats(V(256), 4, 10, 10, 0, V(512), V(1032), 1.0, V(8192), None) == ce.CE_EALIGN
    assert lib.ce_grad_from_stats(V(4096), 4, 10, 12, 0, V(512), V(1024), 1.0, V(4096), None) == ce.CE_EINVAL
    assert lib.ce_grad_from_stats(V(256), 4, 10, 10, 0, V(512), None, 1.0, V(8192), None) == ce.CE_EINVAL


def test_indirect_validation(lib):
    for fn in (lib.argmax_rows_indirect, lib.candidates_rows_indirect):
        assert fn(None, 4, 10, V(4096), None) == ce.CE_EINVAL                 # no table
        assert fn(V(4100), 4, 10, V(4096), None) == ce.CE_EALIGN              # table not 8-byte aligned
        assert fn(V(4096), 4, 0, V(8192), None) == ce.CE_EINVAL               # vocab < 1
        assert fn(V(4096), 4, (1 << 24) + 1, V(8192), None) == ce.CE_EINVAL   # token not exact in f32
        assert fn(V(4096), -1, 10, V(8192), None) == ce.CE_EINVAL
        assert fn(V(4096), 4, 10, None, None) == ce.CE_EINVAL                 # no output
        assert fn(V(4096), 4, 10, V(8194), None) == ce.CE_EALIGN
        assert fn(None, 0, 10, None, None) == ce.CE_OK                        # nothing launched


def test_zero_rows_is_a_no_op_without_device(lib):
    # nothing is launched, so no device is needed
    assert lib.ce_rows(None, 0, 10, 10, None, None, None) == ce.CE_OK
    assert lib.argmax_rows(None, 0, 10, 10, None, None) == ce.CE_OK
    assert lib.ce_grad(None, 0, 10, 10, None, 1.0, None, None, None) == ce.CE_OK
    assert lib.ce_grad_step(None, 0, 10, 10, None, 1.0, None, None, None, None, None) == ce.CE_OK


def test_read_probe_validation(lib):
    assert lib.ce_debug_read(V(256), 32, None, None) == ce.CE_EINVAL        # no output
    assert lib.ce_debug_read(V(256), 30, V(4096), None) == ce.CE_EINVAL     # not whole 16-byte vectors
    assert lib.ce_debug_read(V(256), -16, V(4096), None) == ce.CE_EINVAL
    assert lib.ce_debug_read(None, 32, V(4096), None) == ce.CE_EINVAL
    assert lib.ce_debug_read(V(264), 32, V(4096), None) == ce.CE_EALIGN     # 16-byte aligned reads
    assert lib.ce_debug_read(V(256), 32, V(4098), None) == ce.CE_EALIGN


def test_debug_force_validation(lib):
    assert lib.ce_debug_force(8, 0, 0) == ce.CE_EINVAL
    assert lib.ce_debug_force(7, 0, 0) == ce.CE_OK
    assert lib.ce_debug_force(6, 0, 0) == ce.CE_OK
    assert lib.ce_debug_force(0, 17, 0) == ce.CE_EINVAL
    assert lib.ce_debug_force(0, 0, 1024) == ce.CE_EINVAL
    assert lib.ce_debug_force(0, 0, 96) == ce.CE_EINVAL
    assert lib.ce_debug_force(0, 0, 0) == ce.CE_OK
    assert lib.ce_debug_grid_cap(-1) == ce.CE_EINVAL
    assert lib.ce_debug_grid_cap(3) == ce.CE_OK
    assert lib.ce_debug_grid_cap(0) == ce.CE_OK


def test_no_device_here_reports_edevice(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    assert lib.ce_rows(V(256), 4, 10, 10, V(512), V(1024), None) == ce.CE_EDEVICE
    out = (ctypes.c_int64 * 6)()
    assert lib.ce_plan(1, 8192, 128256, 128256, out) == ce.CE_EDEVICE


def test_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(4, 10)
    with pytest.raises(ValueError):
        ce.argmax_rows(x)
    with pytest.raises(TypeError):
        ce.argmax_rows(x.double())


def test_grad_host_validation(lib):
    """ce_grad_host: every argument check answers before any device call."""
    def call(logits_h=V(256), rows=4, vocab=10, stride=10, labels_h=V(512), scale=1.0, logits_d=V(1 << 16),
             labels_d=V(1 << 17), grad=V(1 << 18), loss_rows=V(1 << 19), top=V(1 << 20), mean=V(1 << 21),
             mean_h=V(1 << 22), top_h=V(1 << 23), chunk=0):
        return lib.ce_grad_host(logits_h, rows, vocab, stride, labels_h, scale, logits_d, labels_d, grad,
                                loss_rows, top, mean, mean_h, top_h, chunk, None)
    assert call(logits_h=None) == ce.CE_EINVAL
    assert call(stride=9) == ce.CE_EINVAL
    assert call(vocab=(1 << 24) + 1, stride=(1 << 24) + 1) == ce.CE_EINVAL
    assert call(scale=float("nan")) == ce.CE_EINVAL
    assert call(chunk=-1) == ce.CE_EINVAL
    assert call(mean=None) == ce.CE_EINVAL
    for k in ("labels_h", "logits_d", "labels_d", "grad", "loss_rows"):
        assert call(**{k: None}) == ce.CE_EINVAL, k
    assert call(top=None) == ce.CE_EINVAL                        # tokens back need the device tokens
    assert call(labels_h=V(516)) == ce.CE_EALIGN                 # int64 on 8 bytes
    assert call(mean_h=V((1 << 22) + 4)) == ce.CE_EALIGN         # double on 8 bytes
    assert call(top_h=V((1 << 23) + 2)) == ce.CE_EALIGN
    assert call(grad=V((1 << 16) + 40)) == ce.CE_EINVAL          # grad overlaps the staged logits
