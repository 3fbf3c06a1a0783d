"""Multi-process paths on CPU (gloo, world size 2): the benchmark's whole-job
aggregation takes the slowest rank's time and every rank's units, and the
reference arm under torchrun prints exactly one line from rank 0 while the
other rank exits cleanly.  (Every GPU run here has one device, so the
multi-rank native arm is replicas only; its host logic is what is tested.)"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _aggregate_worker(rank: int, ws: int, port: int, out_dir: str):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        seconds = [0.5, 2.0][rank]
        t = bench.max_over_ranks(seconds, ws)
        value, tmax = bench.aggregate(100.0, seconds, ws)
        bench.barrier(ws)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"t": t, "value": value, "tmax": tmax}, f)
    finally:
        dist.destroy_process_group()


def test_aggregate_uses_slowest_rank_and_all_units(tmp_path):
    ws, port = 2, _free_port()
    mp.start_processes(_aggregate_worker, args=(ws, port, str(tmp_path)), nprocs=ws, join=True, start_method="spawn")
    for r in range(ws):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["t"] == 2.0 and d["tmax"] == 2.0
        assert d["value"] == pytest.approx(100.0 * ws / 2.0)


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--workload", "llama8b-20k"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
