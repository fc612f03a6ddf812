"""Host-side logic of bench.py on the CPU: the replicas' max-over-ranks timing
with two gloo ranks, the whole-job throughput, and the reference arm's line."""
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    try:
        # rank 0 is slower in the first region, rank 1 in the second
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(port, out), nprocs=2, join=True)
        assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]


def test_single_process_is_identity():
    assert bench.max_over_ranks([3.5, 4.5], "cpu") == [3.5, 4.5]


def test_job_throughput_sums_the_replicas():
    one = bench.job_gbs(100, 1, 0.01)
    assert one == pytest.approx(100 * len(bench.MS) * bench.W_BYTES / 0.01 / 1e9)
    assert bench.job_gbs(100, 4, 0.01) == pytest.approx(4 * one)


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
