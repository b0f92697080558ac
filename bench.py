"""Benchmark of the row-wise softmax cross-entropy path on GB300.

One step is one pass of the whole path over one batch of the training
workload ce_8192x128256 (8192 rows x 128256 vocab, f32 logits N(0, 3^2),
4.2 GB): one ce_grad_step call, whose fused kernel writes the gradient, each
row's loss and each row's argmax token from one read of the logits, and whose
mean kernel (a programmatic dependent launch) writes the f64 mean loss.

Printed (one JSON line, rank 0):
  value       fused loss + grad GB/s of the step: algorithmic bytes
              (8 * rows * vocab + 16 * rows + 8) / device time per step
  roofline    the dominant kernel (the fused one) against measured HBM
              bandwidth: the same launch timed alone, K times, with events
              around each launch, right after the steps
  argmax      rows/s of argmax_rows on the decode workload (256 x 151936,
              row stride 152064), L2 flushed before every timed launch, with
              a plain read of the same buffer beside it (the library's read
              probe, same run, same flush) as the ceiling of a read of that size
  candidates  rows/s of candidates_rows on the same decode batch, likewise
  e2e         the same metric through ce_grad_host: the inputs copied from
              pinned host memory (in chunks, overlapped with the kernels) and
              the mean loss and tokens copied back inside the timed region;
              the median of back-to-back steps (the mean beside it); beside it
              a plain pinned host-to-device copy of the same logits (same run),
              the host link's ceiling
  d2d_copy    a plain device copy of the same bytes, for comparison
  cpu_baseline the CPU oracle (f64) timed on the host cores on a row sample,
              and on one core

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --case grad|rows|loss|argmax|softmax|log_softmax|candidates|split_sum|sharded
                    [--workload W] [--rows R] [--force "path,cluster,threads;..."] [--flush]
    python bench.py --report     every operation on every workload

With N > 1 (launched by torch.distributed.run) every rank runs its own batch
on its own GPU (rows are independent: weak scaling, no collective on the
data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "fused CE loss+grad GB/s (% of HBM peak); argmax rows/s at 1 GB300"
FALLBACK_HBM_GBS = 6800.0
PROFILE = os.path.join(ROOT, "profiles", "k_grad_staged__ce_8192x128256.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "row_wise_softmax_ce_gb300", "csrc", f)
                  for f in ("ce_kernels.cu", "ce_device.cuh", "ce_internal.h", "ce_api.cu")]


# GB300's nominal HBM3e bandwidth, the ~8 TB/s a roofline fraction is often
# quoted against; reported beside the measured peak, which is the denominator
NOMINAL_HBM_GBS = 8000.0


def step_bytes(rows: int, vocab: int) -> int:
    """Algorithmic bytes of one step: logits read + gradient written (4 B each
    per element), labels read (8 B/row), loss rows and tokens written (4 B/row
    each), mean written (8 B)."""
    return 8 * rows * vocab + 16 * rows + 8


def argmax_bytes(rows: int, vocab: int) -> int:
    """Algorithmic bytes of argmax_rows: the first vocab columns read, one token written."""
    return 4 * rows * vocab + 4 * rows


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the fused kernel from the committed ncu
    summary, or None if absent or taken on different kernel sources."""
    if not os.path.exists(PROFILE):
        return None
    vals = {}
    with open(PROFILE) as f:
        for line in f:
            if ":" in line and not line.startswith(("#", " ")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(float(vals["dram_bytes_per_full_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[3:7]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def l2_flush(buf: torch.Tensor) -> None:
    """Evict L2 by reading a buffer of twice its size (a read leaves clean
    lines, so the timed kernel pays no write-back of the flush)."""
    torch.sum(buf)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    """The largest of the ranks' values (the slowest rank's time): a host
    tensor over gloo, a device tensor over NCCL."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(w, rank: int):
    """Rank r's batch: the same shape, its own seed (replicas of independent rows)."""
    import dataclasses
    return w if rank == 0 else dataclasses.replace(w, seed=w.seed + 1000 * rank)


def aggregate_gbs(ws: int, bytes_per_rank_step: int, step_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank moved in a step over the slowest rank's step time."""
    return ws * bytes_per_rank_step / (step_ms * 1e-3) / 1e9


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing


def time_oracle(batch, sample_rows: int, threads: int, chunk: int = 1024):
    """Wall time of the oracle's loss rows + gradient + argmax + mean over the
    first sample_rows rows, taken in chunks of rows (bounded host memory)."""
    import numpy as np
    import oracle
    orc = oracle.load()
    w = batch.workload
    total = 0.0
    losses = []
    for a in range(0, sample_rows, chunk):
        b = min(sample_rows, a + chunk)
        xs = batch.logits[a:b].cpu().numpy()
        ys = batch.labels[a:b].cpu().numpy()
        t0 = time.perf_counter()
        g, l = orc.ce_grad(xs, w.vocab, ys, batch.scale, threads=threads)
        orc.argmax(xs, w.vocab, threads=threads)
        total += time.perf_counter() - t0
        losses.append(l)
        del g
    t0 = time.perf_counter()
    orc.ce_mean(np.concatenate(losses))
    return total + time.perf_counter() - t0


def time_oracle_argmax(batch, sample_rows: int, threads: int, chunk: int = 1024):
    """Wall time of the oracle's argmax over the first sample_rows rows."""
    import oracle
    orc = oracle.load()
    total = 0.0
    for a in range(0, sample_rows, chunk):
        xs = batch.logits[a:min(sample_rows, a + chunk)].cpu().numpy()
        t0 = time.perf_counter()
        orc.argmax(xs, batch.workload.vocab, threads=threads)
        total += time.perf_counter() - t0
    return total


def report_oracle(w, cores: int):
    """The oracle on one core and on all cores for one workload: the whole
    workload where it is small, else a 256-row sample scaled to the
    workload's rows ("sampled"). One JSON line per thread count."""
    sampled = w.rows * w.vocab > 2e8
    n = 256 if sampled else w.rows
    b = W.generate(w.with_rows(n), device="cuda")
    grad_ops = "grad" in w.ops
    nbytes = step_bytes(w.rows, w.vocab) if grad_ops else argmax_bytes(w.rows, w.vocab)
    for threads in (1, cores):
        dt = time_oracle(b, n, threads) if grad_ops else time_oracle_argmax(b, n, threads)
        full = dt * w.rows / n
        print(json.dumps({"oracle": w.name, "step": "loss rows + gradient + argmax + mean" if grad_ops else "argmax",
                          "threads": threads, "rows_timed": n, "seconds": round(dt, 4),
                          "seconds_full": round(full, 4), "sampled": sampled,
                          "GB/s": round(nbytes / full / 1e9, 3)}), flush=True)


def report_page_f32(w):
    """The oracle's page-f32 diagnostic (the literal f32 form of the loss,
    16 lanes) beside the f64 oracle and the GPU's row losses, on up to 256
    rows of a loss workload: reported, not graded -- the pages fix neither
    the lanes nor their join."""
    import numpy as np
    import oracle
    import row_wise_softmax_ce_gb300 as ce
    n = min(w.rows, 256)
    b = W.generate(w.with_rows(n), device="cuda")
    gpu = ce.ce_rows(b.logits[:, : w.vocab], b.labels).double().cpu().numpy()
    xs, ys = b.logits.cpu().numpy(), b.labels.cpu().numpy()
    orc = oracle.load()
    ref = orc.ce_rows(xs, w.vocab, ys, threads=cpu_cores())
    page = orc.ce_rows_page_f32(xs, w.vocab, ys, threads=cpu_cores()).astype(np.float64)
    ok = np.isfinite(ref) & (ref > 0)
    rel_gpu = np.abs(gpu[ok] - ref[ok]) / ref[ok]
    rel_page = np.abs(page[ok] - ref[ok]) / ref[ok]
    print(json.dumps({"page_f32": w.name, "rows": n, "graded": False,
                      "gpu_max_rel": float(rel_gpu.max()), "page_f32_max_rel": float(rel_page.max()),
                      "gpu_rows_over_2e-5": int((rel_gpu > 2e-5).sum()),
                      "page_f32_rows_over_2e-5": int((rel_page > 2e-5).sum())}), flush=True)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    w = W.WORKLOADS[W.HEADLINE]
    sample = args.ref_rows
    cores = cpu_cores()
    b = W.generate(w.with_rows(sample), device="cpu")
    for _ in range(args.warmup):
        time_oracle(b, sample, cores)
    times = [time_oracle(b, sample, cores) for _ in range(args.steps)]
    total = sum(times)
    value = step_bytes(sample, w.vocab) * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "rows_per_step": sample, "vocab": w.vocab,
                   "step": "oracle ce_grad + argmax + mean over the first rows of the workload"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} of {w.rows} rows per step"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import row_wise_softmax_ce_gb300 as ce

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    # ---- the training step on the headline workload
    w = replica_workload(W.WORKLOADS[W.HEADLINE], rank)
    b = W.generate(w, device=dev)
    x, y, scale = b.logits, b.labels, b.scale
    R, V = w.rows, w.vocab
    grad = torch.empty((R, V), dtype=torch.float32, device=dev)
    loss_rows = torch.empty(R, dtype=torch.float32, device=dev)
    top = torch.empty(R, dtype=torch.float32, device=dev)
    mean = torch.empty((), dtype=torch.float64, device=dev)

    def step():
        # the fused kernel, then the mean as its programmatic dependent
        ce.ce_grad_step(x, y, scale, grad=grad, loss_rows=loss_rows, top=top, mean=mean)

    def fused_only():
        # the same fused launch without the mean
        ce.ce_grad(x, y, scale, grad=grad, loss_rows=loss_rows, top=top)

    for _ in range(max(3, args.warmup)):
        step()
        fused_only()
    torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # the steps: nothing between the fused kernel and its mean
        t_start.record(stream)
        for _ in range(K):
            step()
        t_end.record(stream)
        # the dominant kernel alone, events around each launch
        for i in range(K):
            ev[i][0].record(stream)
            fused_only()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    step_ms_local = t_start.elapsed_time(t_end) / K
    step_ms = max_over_ranks(step_ms_local, ws)
    fused_all = [a.elapsed_time(c) for a, c in ev]
    fused_ms = statistics.mean(fused_all)
    bytes_step = step_bytes(R, V)
    value = aggregate_gbs(ws, bytes_step, step_ms)
    peak, peak_kind = peaks()
    fused_bytes = 8 * R * V + 16 * R   # what one ce_grad launch moves
    achieved = fused_bytes / (fused_ms * 1e-3) / 1e9
    traffic = profiled_traffic()
    clk = clocks.summary()

    # ---- a plain device-to-device copy of the same logits into the same
    # gradient buffer (the bytes one fused launch moves), printed beside
    for _ in range(2):
        grad.copy_(x)
    copy_ms = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        grad.copy_(x)
        e1.record(stream)
        e1.synchronize()
        copy_ms.append(e0.elapsed_time(e1))
    copy_best = min(copy_ms)
    copy_bytes = 2 * x.numel() * 4

    # ---- decode argmax (rows/s), L2 flushed before every timed launch
    wd = W.WORKLOADS[W.DECODE]
    bd = W.generate(wd, device=dev)
    topd = torch.empty(wd.rows, dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    for _ in range(5):
        ce.argmax_rows(bd.logits, vocab=wd.vocab, out=topd)
    n_arg = max(20, min(200, K))
    times = []
    for _ in range(n_arg):
        l2_flush(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ce.argmax_rows(bd.logits, vocab=wd.vocab, out=topd)
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    arg_all = [a.elapsed_time(c) for a, c in times]
    arg_ms = max_over_ranks(statistics.median(arg_all), ws)
    # the ceiling of a read of this size on this machine, same run, same flush: the
    # library's read probe over the same buffer (its padding included, +0.08%),
    # and torch.sum of it beside
    def timed_reads(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(n_arg):
            l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(c) for a, c in ts]

    probe_out = torch.zeros((), dtype=torch.int32, device=dev)
    read_all = timed_reads(lambda: ce.debug_read(bd.logits, out=probe_out))
    read_ms = statistics.median(read_all)
    sum_all = timed_reads(lambda: torch.sum(bd.logits))
    read_bytes = bd.logits.numel() * 4
    # sampling candidates (candidatesInto) of the same decode batch, L2 flushed too
    cand = torch.empty((wd.rows, ce.CANDIDATE_ROW), dtype=torch.float32, device=dev)
    for _ in range(3):
        ce.candidates_rows(bd.logits, vocab=wd.vocab, out=cand)
    times = []
    for _ in range(n_arg):
        l2_flush(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ce.candidates_rows(bd.logits, vocab=wd.vocab, out=cand)
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    cand_all = [a.elapsed_time(c) for a, c in times]
    cand_ms = max_over_ranks(statistics.median(cand_all), ws)
    cand_bytes = 4 * wd.rows * wd.vocab + 4 * ce.CANDIDATE_ROW * wd.rows
    del flush, bd, cand

    # ---- end to end through ce_grad_host: logits and labels from pinned host
    # memory (copied in chunks of rows, each chunk's kernel running as soon as
    # it has landed), the mean and the tokens back into pinned host memory
    xh = torch.empty((R, V), dtype=torch.float32, pin_memory=True)
    xh.copy_(x)
    xh_bytes = xh.numel() * 4
    yh = y.cpu().pin_memory()
    hs = ce.HostStep(R, V, dev)

    def e2e_step():
        ce.ce_grad_host(xh, yh, scale, hs)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    # the steps back to back, each between its own events: the host link is
    # shared with the rest of the machine, and a plain copy of the same bytes
    # stalls now and then as a step does (8-140 ms beside 20 ms), so the
    # median step is reported, with the mean and the stalled steps beside it
    K2 = max(5, min(K, 20))
    barrier(ws)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(K2 + 1)]
    marks[0].record(stream)
    for i in range(K2):
        e2e_step()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    e2e_all = [marks[i].elapsed_time(marks[i + 1]) for i in range(K2)]
    e2e_ms = max_over_ranks(statistics.median(e2e_all), ws)
    e2e_mean = max_over_ranks(marks[0].elapsed_time(marks[K2]) / K2, ws)
    e2e_value = aggregate_gbs(ws, bytes_step, e2e_ms)
    h2d = xh.numel() * 4 + yh.numel() * 8
    d2h = 8 + hs.top_h.numel() * 4
    # the host link's ceiling, same run: a plain pinned copy of the same logits
    link_ms = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        hs.logits.copy_(xh, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        link_ms.append(e0.elapsed_time(e1))
    link_med = statistics.median(link_ms)
    link_gbs = xh.numel() * 4 / (link_med * 1e-3) / 1e9
    del xh, hs

    # ---- the CPU oracle on a row sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cores = cpu_cores()
        sample = args.cpu_rows
        dt = time_oracle(b, sample, cores)
        one = max(1, min(sample, 128))
        dt1 = time_oracle(b, one, 1)
        cpu = {"value": round(step_bytes(sample, V) / dt / 1e9, 3), "unit": "GB/s", "cores": cores,
               "kind": "oracle", "sample": f"first {sample} of {R} rows of {w.name} "
                                           f"(loss rows + gradient + argmax + mean, f64), {dt:.2f} s wall",
               "single_thread": {"value": round(step_bytes(one, V) / dt1 / 1e9, 3), "unit": "GB/s",
                                 "sample": f"first {one} rows, {dt1:.2f} s wall"}}

    plan = ce.plan(ce.OP_GRAD, R, V)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(step_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "rows": R, "vocab": V, "stride": V, "logits": "N(0, 3^2) f32",
                       "scale": scale,
                       "step": "ce_grad_step: the fused kernel (gradient + loss rows + argmax) and the "
                               "f64 mean as its programmatic dependent",
                       "l2": "no flush: inputs (4.2 GB) larger than L2", "parallelism": f"replicas x{ws}",
                       "plan": plan},
            "percent_of_hbm_peak": round(100 * value / ws / peak, 2),
            "roofline": {"bound": "hbm", "kernel": "k_grad_staged", "achieved": round(achieved, 1),
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4), "traffic": traffic,
                         "algorithmic_bytes": fused_bytes, "ms_per_launch": round(fused_ms, 4),
                         "ms_per_launch_min": round(min(fused_all), 4)},
            "d2d_copy": {"what": "grad.copy_(logits): the same 4.2 GB read and written", "bytes": copy_bytes,
                         "ms_best_of_5": round(copy_best, 4),
                         "GB/s": round(copy_bytes / (copy_best * 1e-3) / 1e9, 1)},
            "argmax": {"workload": wd.name, "rows_per_s": round(ws * wd.rows / (arg_ms * 1e-3), 1),
                       "ms": round(arg_ms, 5), "ms_min": round(min(arg_all), 5),
                       "GB/s": round(argmax_bytes(wd.rows, wd.vocab) / (arg_ms * 1e-3) / 1e9, 1),
                       "frac": round(argmax_bytes(wd.rows, wd.vocab) / (arg_ms * 1e-3) / 1e9 / peak, 4),
                       "l2": "flushed before each launch",
                       "plain_read": {"what": "ce_debug_read (one CTA per SM, 32 KB bulk copies through four "
                                              "shared-memory stages) of the same padded buffer, same flush",
                                      "bytes": read_bytes, "ms": round(read_ms, 5),
                                      "ms_min": round(min(read_all), 5),
                                      "GB/s": round(read_bytes / (read_ms * 1e-3) / 1e9, 1),
                                      "argmax_over_read": round(arg_ms / read_ms, 4),
                                      "torch_sum_ms": round(statistics.median(sum_all), 5)}},
            "candidates": {"workload": wd.name, "rows_per_s": round(ws * wd.rows / (cand_ms * 1e-3), 1),
                           "ms": round(cand_ms, 5), "ms_min": round(min(cand_all), 5),
                           "GB/s": round(cand_bytes / (cand_ms * 1e-3) / 1e9, 1),
                           "frac": round(cand_bytes / (cand_ms * 1e-3) / 1e9 / peak, 4),
                           "l2": "flushed before each launch"},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                    "statistic": f"median of {K2} steps, each between its own events",
                    "ms_per_step_mean": round(e2e_mean, 3),
                    "steps_over_1.2x_median": sum(t > 1.2 * e2e_ms for t in e2e_all),
                    "ms_steps": [round(t, 2) for t in e2e_all],
                    "host_link": {"what": "a plain pinned host-to-device copy of the logits, median of 5",
                                  "bytes": xh_bytes, "ms": round(link_med, 3), "ms_min": round(min(link_ms), 3),
                                  "GB/s": round(link_gbs, 1), "e2e_step_over_copy": round(e2e_ms / link_med, 4)}},
            "gpu_launches": 2 * K,
            "gpu_launches_note": "the steps' region: k_grad_staged + k_mean per step; the fused "
                                 "kernel's own loop adds K more launches of k_grad_staged",
            "cpu_baseline": cpu,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_case(args):
    """One operation on a chosen number of rows of a workload, with an optional
    forced launch plan: for launch-shape sweeps and small profiler captures."""
    import row_wise_softmax_ce_gb300 as ce

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    name = args.workload or (W.DECODE if args.case in ("argmax", "candidates") else W.HEADLINE)
    w = W.WORKLOADS[name]
    if args.rows:
        w = w.with_rows(args.rows)
    b = W.generate(w, device=dev)
    R, V = w.rows, w.vocab
    out = torch.empty(R, dtype=torch.float32, device=dev)
    if args.case == "grad":
        grad = torch.empty((R, V), dtype=torch.float32, device=dev)
        op = lambda: ce.ce_grad(b.logits, b.labels, b.scale, vocab=V, grad=grad, loss_rows=out)
        nbytes, opn = 8 * R * V + 12 * R, ce.OP_GRAD
    elif args.case == "rows":
        op = lambda: ce.ce_rows(b.logits, b.labels, vocab=V, out=out)
        nbytes, opn = 4 * R * V + 12 * R, ce.OP_ROWS
    elif args.case == "loss":
        # crossEntropyLoss: the row losses, then their f64 mean on the device
        mean = torch.empty((), dtype=torch.float64, device=dev)
        op = lambda: ce.ce_loss(b.logits, b.labels, vocab=V, loss_rows=out, out=mean)
        nbytes, opn = 4 * R * V + 16 * R + 8, ce.OP_ROWS
    elif args.case in ("softmax", "log_softmax"):
        dense = torch.empty((R, V), dtype=torch.float32, device=dev)
        fn = ce.softmax_rows if args.case == "softmax" else ce.log_softmax_rows
        op = lambda: fn(b.logits, vocab=V, out=dense)
        nbytes, opn = 8 * R * V, ce.OP_SOFTMAX if args.case == "softmax" else ce.OP_LOG_SOFTMAX
    elif args.case == "candidates":
        cand = torch.empty((R, ce.CANDIDATE_ROW), dtype=torch.float32, device=dev)
        op = lambda: ce.candidates_rows(b.logits, vocab=V, out=cand)
        nbytes, opn = 4 * R * V + 4 * ce.CANDIDATE_ROW * R, ce.OP_CANDIDATES
    elif args.case == "sharded":
        # the vocab split into `splits` slices: stats of each, combine, each slice's gradient
        shards = max(1, args.splits)
        cuts = sorted(set([min(V, k * -(-V // shards)) for k in range(shards + 1)]))
        stats = torch.empty((len(cuts) - 1, R, 4), dtype=torch.float32, device=dev)
        grads = [torch.empty((R, c - a), dtype=torch.float32, device=dev) for a, c in zip(cuts, cuts[1:])]
        lr = torch.empty(R, dtype=torch.float32, device=dev)
        comb = torch.empty((R, 4), dtype=torch.float32, device=dev)

        def op():
            for k, (a, c) in enumerate(zip(cuts, cuts[1:])):
                ce.ce_stats(b.logits, b.labels, col0=a, vocab=c - a, out=stats[k])
            ce.ce_stats_combine(stats, b.labels, V, loss_rows=lr, top=out, combined=comb)
            for (a, c), g in zip(zip(cuts, cuts[1:]), grads):
                ce.ce_grad_from_stats(b.logits[:, a:c], b.labels, a, comb, b.scale, grad=g)
        # what this split moves: each slice read twice (stats, gradient), the gradient written once
        nbytes, opn = 12 * R * V + 32 * R * (len(cuts) - 1), None
    elif args.case == "split_sum":
        # the workload's logits as `splits` parts of R * V / splits values
        splits = max(1, args.splits)
        total = (R * V) // splits
        parts = b.logits[:, :V].reshape(-1)[: splits * total].view(splits, total)
        if not parts.is_contiguous():
            parts = parts.contiguous()
        y = torch.empty(total, dtype=torch.float32, device=dev)
        op = lambda: ce.split_sum(parts, y, add=False)
        nbytes, opn = 4 * (splits + 1) * total, None
    else:
        op = lambda: ce.argmax_rows(b.logits, vocab=V, out=out)
        nbytes, opn = argmax_bytes(R, V), ce.OP_ARGMAX
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev) if args.flush else None
    peak, kind = peaks()
    for force in (args.force.split(";") if args.force else ["0,0,0"]):
        ce.debug_force(*[int(v) for v in force.split(",")])
        try:
            for _ in range(max(1, args.warmup)):
                op()
            torch.cuda.synchronize()
            evs = []
            for _ in range(args.steps):
                if flush is not None:
                    l2_flush(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                op()
                e1.record(stream)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            plan = ce.plan(opn, R, V, w.stride) if opn is not None else None
        except ce.CeError as e:
            print(json.dumps({"case": args.case, "workload": w.name, "force": force, "error": str(e)}), flush=True)
            continue
        finally:
            ce.debug_force(0, 0, 0)
        ms = [a.elapsed_time(c) for a, c in evs]
        med = statistics.median(ms)
        print(json.dumps({"case": args.case, "workload": w.name, "rows": R, "vocab": V, "force": force,
                          "plan": plan, "ms_median": round(med, 5), "ms_min": round(min(ms), 5),
                          "GB/s": round(nbytes / (med * 1e-3) / 1e9, 1), "rows/s": round(R / (med * 1e-3), 1),
                          "frac": round(nbytes / (med * 1e-3) / 1e9 / peak, 4), "peak_kind": kind,
                          "flush": bool(args.flush)}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=8192, help="rows of the CPU-oracle sample")
    ap.add_argument("--ref-rows", type=int, default=256, help="rows per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["grad", "rows", "loss", "argmax", "softmax", "log_softmax", "candidates",
                                       "split_sum", "sharded"],
                    help="time one operation only (sweeps, profiler captures)")
    ap.add_argument("--report", action="store_true",
                    help="time every operation on every workload (one JSON line each)")
    ap.add_argument("--splits", type=int, default=4,
                    help="with --case split_sum: parts to join; with --case sharded: vocab slices")
    ap.add_argument("--workload", choices=sorted(W.WORKLOADS), help="with --case: the workload")
    ap.add_argument("--rows", type=int, default=0, help="with --case: rows of the workload to use")
    ap.add_argument("--force", default="", help="with --case: path,cluster,threads (see ce_debug_force)")
    ap.add_argument("--flush", action="store_true", help="with --case: flush L2 before each launch")
    args = ap.parse_args()
    if args.report:
        # every workload x operation, one JSON line each (L2 flushed for the
        # workloads smaller than a few L2 sizes)
        import copy
        for name, w in W.WORKLOADS.items():
            small = 4 * w.rows * w.stride < 4 * torch.cuda.get_device_properties(0).L2_cache_size
            for case in ("rows", "loss", "grad", "argmax", "softmax", "candidates"):
                a = copy.copy(args)
                a.case, a.workload, a.rows, a.force, a.flush = case, name, 0, "", small
                a.steps = min(args.steps, 50)
                run_case(a)
        # the oracle beside, single-threaded and on every host core
        for w in W.WORKLOADS.values():
            report_oracle(w, cpu_cores())
        # the literal f32 form of the loss beside (a diagnostic, not graded)
        for w in W.WORKLOADS.values():
            if "loss" in w.ops or "rows" in w.ops:
                report_page_f32(w)
        return 0
    if args.case:
        return run_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
