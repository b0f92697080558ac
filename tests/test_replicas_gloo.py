"""The multi-process (replica) path of bench.py on CPU: two ranks over gloo.
Rows are independent, so N GPUs run N replicas; the only collectives are the
timing barrier and the max of the step time over ranks. Nothing here uses a
GPU."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import bench
    import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        local_ms = [1.25, 2.5][rank]              # the slower rank sets the step time
        step_ms = bench.max_over_ranks(local_ms, ws)
        w = bench.replica_workload(W.WORKLOADS["ce_64x1000"], rank)
        b = W.generate(w, device="cpu")
        firsts = [torch.zeros(1) for _ in range(ws)]
        dist.all_gather(firsts, b.logits[0, :1].clone())
        out.put((rank, step_ms, w.seed, [float(f) for f in firsts]))
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_replicas_over_gloo():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5], "max over ranks"
    assert res[0][2] != res[1][2], "each replica draws its own batch"
    assert res[0][3][0] != res[0][3][1], "the two ranks' batches differ"
    sys.path.insert(0, ROOT)
    import bench
    # whole-job GB/s = the bytes of both ranks over the slowest rank's time
    assert bench.aggregate_gbs(2, 10 ** 9, 2.5) == pytest.approx(2 * 10 ** 9 / 2.5e-3 / 1e9)


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 times the oracle; the other ranks print nothing and exit 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
