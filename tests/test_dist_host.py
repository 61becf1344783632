"""The multi-GPU path is replicas only: every rank streams its own copy of the
workload, ranks meet only at the barriers around the timed region, and rank 0
reports the aggregate over the slowest rank's time.  Its host logic runs here
as two gloo ranks on the CPU (no GPU), plus the reference arm under torchrun
with two ranks (rank 0 alone prints)."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    d = bench.dist_init("gloo")
    assert d is not None and d.get_world_size() == world
    d.barrier()
    # each rank "timed" a different duration; the job time is the slowest rank's
    t = bench.max_over_ranks(d, 0.010 * (rank + 1), "cpu")
    value = bench.aggregate_gbps(world, 20, 209111040, t)
    out[rank] = (t, value)
    d.barrier()
    d.destroy_process_group()


def test_two_gloo_ranks_max_time_and_aggregate():
    world = 2
    port = free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == pytest.approx(0.020)
    # two replicas of 20 steps of 209,111,040 bytes in 20 ms
    assert res[0][1] == res[1][1] == pytest.approx(2 * 20 * 209111040 / 0.020 / 1e9)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(None, 0.5, "cpu") == 0.5
    assert bench.aggregate_gbps(1, 10, 1e9, 2.0) == pytest.approx(5.0)


def test_reference_arm_under_torchrun_rank0_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
