"""bench.py's multi-process path on CPU: two ranks joined over gloo (127.0.0.1), as torchrun
would start them. The layer itself shards nothing (replicas only), so what is tested is the
host logic every replica runs: the rendezvous, the barrier, the max-over-ranks step time, the
weak-scaling aggregate and that the reference arm prints one line on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(code: str, world: int = 2, timeout: float = 240.0):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   WORLD_SIZE=str(world), RANK=str(r), LOCAL_RANK=str(r),
                   MOE_DIST_BACKEND="gloo", CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    out = []
    try:
        for p in procs:
            o, e = p.communicate(timeout=timeout)
            out.append((p.returncode, o, e))
    finally:
        for p in procs:  # only the processes started here
            if p.poll() is None:
                p.kill()
                p.wait()
    return out


def test_barrier_and_max_over_ranks():
    code = (
        "import json, bench\n"
        "ws, rank, _ = bench.dist_setup()\n"
        "bench.barrier(ws)\n"
        "ms = bench.allreduce_max(10.0 + 5.0 * rank, ws)\n"
        "v = bench.job_throughput(3.0e12, ms, ws)\n"
        "print(json.dumps({'rank': rank, 'ws': ws, 'ms': ms, 'v': v}))\n"
        "import torch.distributed as dist; dist.destroy_process_group()\n")
    res = _run_ranks(code)
    for rc, o, e in res:
        assert rc == 0, e[-2000:]
    lines = [json.loads(o.strip().splitlines()[-1]) for _, o, _ in res]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    for d in lines:
        assert d["ws"] == 2
        assert d["ms"] == 15.0  # the slower rank's time on both ranks
        assert d["v"] == pytest.approx(2 * 3.0e12 / 15e-3)


def test_reference_arm_runs_on_rank0_only():
    code = (
        "import sys, bench\n"
        "sys.argv = ['bench.py', '--impl', 'reference', '--config', 'tiny', '--steps', '1',\n"
        "            '--warmup', '0', '--gpus', '2']\n"
        "bench.main()\n")
    res = _run_ranks(code)
    for rc, o, e in res:
        assert rc == 0, e[-2000:]
    rank0 = [l for l in res[0][1].splitlines() if l.startswith("{")]
    rank1 = [l for l in res[1][1].splitlines() if l.startswith("{")]
    assert len(rank0) == 1 and rank1 == []
    line = json.loads(rank0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_throughput(1e12, 10.0, 1) == pytest.approx(1e14)
    assert bench.job_throughput(1e12, 10.0, 8) == pytest.approx(8e14)
