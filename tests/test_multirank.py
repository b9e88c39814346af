"""The multi-process path of bench.py on CPU (gloo, world size 2): decode
shards by sequence with no exchange, so N GPUs run N replicas; what crosses
ranks is the timing (the slowest rank sets the job's time) and the launch
contract (under torchrun only rank 0 prints the reference line)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r measured (step, decode) = (1 + r, 10 - r) ms: the job takes the max of each
    ms, dms = bench.max_over_ranks(dist, [1.0 + rank, 10.0 - rank], "cpu")
    dist.barrier()
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump({"ms": ms, "dms": dms,
                       "rate": bench.job_throughput(world, 1000.0, ms)}, f)
    dist.destroy_process_group()


def test_timings_reduce_to_the_slowest_rank(tmp_path):
    torch = pytest.importorskip("torch")
    out = tmp_path / "r.json"
    torch.multiprocessing.start_processes(_rank_main, args=(2, _free_port(), str(out)), nprocs=2,
                                          join=True, start_method="spawn")
    r = json.loads(out.read_text())
    assert r["ms"] == 2.0 and r["dms"] == 10.0
    assert r["rate"] == pytest.approx(2 * 1000.0 / 2e-3)      # both replicas' units / slowest time


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(None, [3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.job_throughput(1, 500.0, 2.0) == pytest.approx(250000.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-seconds", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=240, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["e2e"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
