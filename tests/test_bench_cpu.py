"""bench.py's host-side paths on the CPU: the reference arm (the oracle timed on
the host), its JSON line, and the multi-rank launch (torchrun, gloo, two ranks:
replicas only, rank 0 prints one line, the others exit 0), plus the
max-over-ranks reduction the timed arm uses."""

import json
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


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--workload", "tiny-fp32"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "TFLOPS" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny-fp32"


def test_reference_arm_two_ranks_gloo():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
                        "--workload", "tiny-fp32"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    q.put((rank, bench.max_over_ranks(float(rank + 1) * 1.5, world)))
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 3.0), (1, 3.0)]


def test_routing_summary_hand_worked():
    """The routing histogram the bench line reports, on a hand-worked count vector."""
    sys.path.insert(0, ROOT)
    import bench
    counts = [0, 1, 127, 128, 129, 300, 0, 5, 1000, 2, 50, 60]
    r = bench.routing_summary(counts)
    # 1802 rows; nonempty sorted 1 2 5 50 60 127 128 129 300 1000; busiest eight hold 1799;
    # 128-row tiles: 2560 rows computed
    assert r == {"max_count": 1000, "empty_experts": 2, "median_nonempty": 93.5, "experts_below_128_rows": 6,
                 "top8_share": 0.9983, "tile128_padding": 0.2961}
    assert bench.routing_summary([0, 0])["tile128_padding"] == 0.0


def test_gpus_flag_spawns_ranks_without_torchrun():
    """--gpus 2 in a plain launch starts the two ranks itself (gloo on the CPU):
    rank 0 prints the one line with n_gpus 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny-fp32"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def test_gpus_flag_mismatch_fails_loudly():
    """Under a launcher whose WORLD_SIZE differs from --gpus the bench stops with an
    error instead of timing the wrong number of replicas."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "3", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny-fp32"], cwd=ROOT, capture_output=True, text=True,
                       timeout=120, env=env)
    assert r.returncode != 0
    assert "does not match WORLD_SIZE" in r.stderr
    assert not _json_lines(r.stdout)
