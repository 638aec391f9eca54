"""The multi-replica path of bench.py on CPU: two gloo ranks (127.0.0.1).
The decode step does not shard (one independent replica per GPU, no
collective on the data path); what runs across ranks is the timing
reduction (max over ranks) and the whole-job aggregation, checked here, and
the launch contract of the reference arm under torchrun."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports step time 1 + r, e2e 10 - r, kernel 0.5 * (r + 1)
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * (rank + 1)], world, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r] == [2.0, 10.0, 1.0]  # every rank sees the slowest replica


def test_whole_job_value_and_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    # 2 replicas x 1 GB in the slowest replica's 0.5 s -> 4 GB/s for the job
    assert bench.whole_job_gbs(1e9, 0.5, 2) == pytest.approx(4.0)


def test_reference_arm_two_ranks_prints_once():
    """Under torchrun with two ranks the oracle arm runs on rank 0 only and
    prints one JSON line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(30500 + os.getpid() % 1000),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "1", "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle"
