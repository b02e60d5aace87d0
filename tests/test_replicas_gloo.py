"""The multi-GPU path is replicas only: every rank runs the same workload with no
exchange, the job's time is the slowest rank's and its rate counts every rank's
work.  These CPU tests run that host logic with two gloo ranks (no GPU)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    ws, r, _ = bench.dist_setup()
    t_ms = [2.0, 3.0][r]                     # this rank's step time
    bench.barrier(ws)
    t_max = bench.reduce_max(t_ms, ws)
    q.put((r, ws, dist.get_backend(), t_max, bench.job_rate(ws, 1.5e12, t_max, 1e12)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, ws, backend, t_max, rate in got:
        assert ws == 2 and backend == "gloo"
        assert t_max == 3.0                   # the max over ranks, seen by both
        assert abs(rate - 2 * 1.5e12 / 3e-3 / 1e12) < 1e-6   # both ranks' work over the slowest time


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1"]
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
