"""Host-side logic of bench.py that needs no GPU: the multi-rank reductions (run as two gloo ranks
on CPU) and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mx = bench.max_over_ranks(10.0 + rank)
        sm = bench.sum_over_ranks(1.5 * (rank + 1))
        q.put((rank, mx, sm))
    finally:
        dist.destroy_process_group()


def test_rank_reductions_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0, 4.5), (1, 11.0, 4.5)]


def test_reductions_are_identity_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25 and bench.sum_over_ranks(2.0) == 2.0


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_summary_keeps_only_samples_inside_the_timed_region():
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.lines = ["2026/12/02 06:00:00.000, 0, 1000, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "2026/12/02 06:00:01.000, 0, 1900, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
               "2026/12/02 06:00:01.100, 0, 1950, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "2026/12/02 06:00:01.200, 0, 2000, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "2026/12/02 06:00:09.000, 0, 300, 2070, 90.0, 0x8, Active, Not Active, Not Active, Not Active",
               "garbled"]
    c.t_start = datetime.datetime(2026, 12, 2, 6, 0, 0, 500000)
    c.t_stop = datetime.datetime(2026, 12, 2, 6, 0, 2)
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1950 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["window"] == "timed region"
    c.t_start = datetime.datetime(2026, 12, 2, 7)
    c.t_stop = datetime.datetime(2026, 12, 2, 8)
    s = c.summary()
    assert s["samples"] == 5 and "hw_slowdown" in s["reasons"]


def test_profiled_traffic_is_null_once_the_kernel_changed(tmp_path):
    sys.path.insert(0, ROOT)
    import hashlib
    import bench
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    prof = tmp_path / "p.md"
    h = hashlib.sha256(b"kernel v1").hexdigest()
    prof.write_text(f"kernel_source_sha256 = {h}\ntraffic_per_step_bytes = 1234\n")
    assert bench.profiled_traffic(str(prof), [str(src)]) == 1234
    src.write_text("kernel v2")
    assert bench.profiled_traffic(str(prof), [str(src)]) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md"), [str(src)]) is None


def test_copy_and_anchor_byte_counts():
    """The per-sequence byte figures the secondary sections sum: the decode workload's 64 heads x 64
    rows of 128 values; NVFP4 = half a byte per value + one e4m3 byte per 16 values + a 4-byte row
    scale; FP8 = a byte per value + the row scale; the shared NVFP4 state has no separate anchor."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    d = synth.workload("decode_b256_h64").dims
    rows = 64 * 64
    assert bench._copy_bytes(d, "bf16") == rows * 128 * 2
    assert bench._copy_bytes(d, "fp8") == rows * (128 + 4)
    assert bench._copy_bytes(d, "nvfp4") == rows * (64 + 8 + 4) == 311296
    assert bench._anchor_bytes(d, "fp32") == rows * 128 * 4 == 2 * 1024 * 1024
    assert bench._anchor_bytes(d, "fp16_sr") == rows * 128 * 2
    assert bench._anchor_bytes(d, "nvfp4_sr_shared") == 0
