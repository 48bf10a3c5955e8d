"""Host logic of bench.py: multi-rank aggregation (gloo, world size 2, CPU),
clock-sample parsing and the CPU reference arm's JSON line."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r pretends its timed region took (r + 1) seconds for 10 units
        t = bench.reduce_max(float(rank + 1), dist)
        q.put((rank, t, bench.aggregate(10.0, t, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [2.0, 2.0]          # slowest rank's time on every rank
    assert [g[2] for g in got] == [10.0, 10.0]         # 2 ranks x 10 units / 2 s


def test_single_process_aggregate():
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.aggregate(100.0, 2.0, 1) == 50.0


def test_clock_rows_parsing():
    rows = [
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active".split(","),
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active".split(","),
        "0, 2000, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active".split(","),
    ]
    s = bench.parse_clock_rows(rows, bench.ClockSampler.REASONS)
    assert s["sm_mhz"] == 2000 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_reference_arm_line_on_cpu():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny", "--steps", "3", "--warmup", "1"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["higher_is_better"] is True


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched the way the multi-GPU bench is (torchrun, 2 ranks; gloo on a
    CPU-only host): rank 0 alone runs the reference arm and prints one line,
    the other rank exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1", "--gpus", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_form_flags_and_traffic_lookup():
    """--one-launch / --tc parse; the committed ncu traffic figures are found
    for the workloads they were taken on only while the kernel sources match
    the hash they were taken with."""
    a = bench.parse_args(["--one-launch", "--tc", "--workload", "d256_b8"])
    assert a.one_launch and a.tc and a.workload == "d256_b8"
    d = bench.parse_args([])
    assert not d.one_launch and not d.tc and d.workload == "serving"
    with open(bench.TRAFFIC_FILE) as f:
        t = json.load(f)
    if t.get("kernel_source_sha256") == bench.kernel_source_hash():
        for w, e in t["workloads"].items():
            assert bench.traffic_per_launch(w) == e["dram_bytes_per_launch"]
    else:
        assert bench.traffic_per_launch("serving") is None
