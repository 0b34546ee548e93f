"""Host logic of bench.py (no GPU): the reference arm's JSON line, the
whole-job aggregation, and the rank plumbing under a 2-process gloo group."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_aggregate_is_units_over_slowest_rank():
    assert bench.aggregate(10.0, 4, 2.0) == 20.0
    assert bench.aggregate(3.0, 1, 1.5) == 2.0


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_3x8x8_h2", "--steps", "2", "--warmup", "1", "--ref-rows", "16"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["workload"] == "tiny_3x8x8_h2"


def test_conv_reference_arm_and_cpu_baseline():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "wan_vae_conv3d_360x640_192", "--steps", "1", "--warmup", "1", "--ref-rows", "8"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["metric"] == bench.CONV_METRIC and rec["value"] > 0
    assert rec["config"]["kind"] == "conv3d" and rec["config"]["c_out"] == 192
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    cb = bench.cpu_baseline(CONV_WORKLOADS["wan_vae_conv3d_720p_384"], 16)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and "output positions" in cb["sample"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), WAN_BENCH_BACKEND="gloo")
    r, w, _ = bench.dist_setup(world)
    bench.barrier(w)
    m = bench.max_over_ranks(1.0 + r, w)
    q.put((r, w, m))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_gloo_max_over_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
    assert res == [(0, 2, 2.0), (1, 2, 2.0)]
