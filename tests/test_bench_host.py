"""Host-side logic of bench.py, on CPU: the multi-rank reduction with two gloo
ranks, and the reference arm (the CPU oracle) end to end."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # Rank r "took" r + 1 ms; every rank must see the slowest, 2 ms.
    ms = bench.max_over_ranks(rank + 1.0, dist, device="cpu")
    value = bench.job_value(units_per_rank=1000.0, world=world, max_seconds=ms * 1e-3)
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"ms": ms, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    got = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    assert all(g["ms"] == 2.0 for g in got)
    assert all(g["value"] == pytest.approx(2 * 1000.0 / 2e-3) for g in got)


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(10.0, 1, 2.0) == 5.0


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--ref-seconds", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["metric"] == bench.METRIC


def test_reference_arm_under_two_ranks_prints_once():
    """Launched the way a multi-GPU run is (torch.distributed.run, 2 ranks):
    rank 0 alone times the oracle and prints; rank 1 exits 0 without work."""
    pytest.importorskip("torch")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-seconds", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
