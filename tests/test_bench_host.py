"""Host-side logic of the multi-GPU bench path, on CPU with gloo ranks.

The hot path does not shard across GPUs (each rank runs an independent
replica of the verify step), so the only multi-rank logic is the timing
reduction (max over ranks), the whole-job throughput, and the reference arm
running on rank 0 only.  These run here as world-size-2 gloo process groups.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r "measured" (step ms, e2e ms, split us) = (1 + r, 10 - r, 5 + 2 r)
    got = bench.reduce_max([1.0 + rank, 10.0 - rank, 5.0 + 2 * rank], "cpu")
    value = bench.aggregate_gbs(world, 1e9, got[0])
    out_q.put((rank, got, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 10.0, 7.0]          # the slowest rank's numbers on every rank
        assert value == pytest.approx(2 * 1e9 / 2e-3 / 1e9)  # both replicas' bytes / slowest time


def test_single_rank_reduce_is_identity():
    import bench
    assert bench.reduce_max([3.0, 4.5], "cpu") == [3.0, 4.5]
    assert bench.aggregate_gbs(1, 134217728, 0.04) == pytest.approx(3355.44320)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched the way the multi-GPU run launches
    it: rank 0 times the oracle and prints one JSON line, rank 1 exits 0."""
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "2", "--warmup", "1", "--gpus", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
