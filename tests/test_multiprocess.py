"""The N > 1 host logic of bench.py on CPU, world size 2 over gloo: the
barrier, the max-over-ranks timing reduction and the whole-job rate of
replicas, and the reference arm launched under torchrun (rank 0 alone runs
and prints; the other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port,
                            rank=rank, world_size=world)
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks(1.5 * (rank + 1), world, torch.device("cpu"))
        rate = bench.whole_job_rate(1000, slowest, 2, world)
        bench.barrier(world)
        out_q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_barrier_max_over_ranks_and_rate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    for _, slowest, rate in res:
        assert slowest == 3.0                       # the max of 1.5 and 3.0
        # two replicas of 1000 tokens per step, 1.5 ms per step on the slowest
        assert rate == pytest.approx(2 * 1000 / 1.5e-3)


def test_whole_job_rate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(16384, 2.0, 20, 1) == pytest.approx(16384 / 1e-4)


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny_fp32_B1_H2_T256_d64", "--steps", "1", "--warmup", "0",
           "--gpus", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
