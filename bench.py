"""Benchmark of the exact-replay SSD hot path on GB300.

Headline: replay-decode seq-steps/s per layer at B=256 (256 sequences x 64 heads / 8 groups,
headdim 64, dstate 128, chunk = refresh period 16, each sequence starting at a uniform-random
position in its partial chunk).  One step = one ers_replay_decode call over the batch, including
the fused checkpoint refresh of the sequences whose chunk fills.  The same line reports SSD
prefill tok/s (2048 tokens x 32 heads; varlen {2048, 777, 513, 1} x 64 heads), speculative
verify + commit (512 sequences, 4 drafts, L = 16) and the per-token-writeback SSU comparison
kernel, each against its HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own 256-sequence batch on its own GPU (weak scaling, no
collective on the data path); the timed region is bracketed by a barrier and a device sync on
both sides and the slowest rank's time is reported.  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

# Algorithmic HBM bytes per sequence-step of the decode workload (64 heads x 64 x 128):
#   fp32 checkpoint read 2,097,152 + E[p] = 7.5 buffered rows x 10,496 (x 8,192 + dt 256 + B 2,048)
#   + new-token read 12,544 + buffer append 12,544 + y 8,192 + refresh write 2,097,152 / 16
DECODE_BYTES_PER_SEQ_STEP = 2_340_224
SSU_BYTES_PER_SEQ_STEP = 4_215_040       # state read + write 4,194,304 + token in 12,544 + y 8,192
PREFILL_BYTES = {"prefill_2048_h32": 19_136_896, "varlen_4seq_h64": 77_626_880}
PREFILL_FLOPS = {"prefill_2048_h32": 3.29e9, "varlen_4seq_h64": 11.38e9}
L2_FLUSH_BYTES = 256 << 20


DECODE_PROFILE = os.path.join(ROOT, "profiles", "k_decode_heads.decode_b256_h64.md")
DECODE_SOURCES = [os.path.join(ROOT, "exact_replay_decode_gb300", "csrc", f)
                  for f in ("ers_decode.cu", "warp_heads.cuh", "ers_common.cuh")]


def profiled_traffic(profile: str = DECODE_PROFILE, sources=None):
    """DRAM bytes per step (dram__bytes_read.sum + dram__bytes_write.sum of the step's launches) from the
    committed ncu summary, or None when the kernel's sources have changed since the capture (sha256 over the
    concatenated files) or no record exists."""
    import hashlib
    import re
    sources = DECODE_SOURCES if sources is None else sources
    try:
        text = open(profile).read()
        want = re.search(r"kernel_source_sha256 = ([0-9a-f]{64})", text).group(1)
        traffic = int(re.search(r"traffic_per_step_bytes = (\d+)", text).group(1))
        hsh = hashlib.sha256()
        for f in sources:
            hsh.update(open(f, "rb").read())
    except (OSError, AttributeError):
        return None
    return traffic if hsh.hexdigest() == want else None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------------------------
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 100 ms while running.

    Each sample carries nvidia-smi's own timestamp, so the summary can keep only the samples
    taken inside the timed region (``mark_start``/``mark_stop`` bracket it on the host)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark_start(self):
        self.t_start = datetime.datetime.now()

    def mark_stop(self):
        self.t_stop = datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)          # let the last sample of the window arrive
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def _parse(self):
        out = []
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                out.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        return out

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = self._parse()
        window = "timed region"
        sel = [r for r in rows if self.t_start and self.t_stop and self.t_start <= r[0] <= self.t_stop]
        if not sel:
            sel, window = rows, "warm-up soak + timed region (no sample fell inside the timed region)"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({n for r in sel for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel), "window": window}


# ---------------------------------------------------------------------------------------------
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank float over the default process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def _barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------------------------
TOKEN_RING = 64          # distinct token sets cycled through by the decode steps
SOAK_S = 0.5             # untimed decode steps before the timed region (clocks settle, samples exist)


class DecodeBench:
    """The B=256 replay-decode workload, prefilled to its random starting positions.

    Step k feeds token set k mod TOKEN_RING (fresh N(0,1) bf16 x/B/C and dt for every sequence);
    the ring keeps host-side generation bounded while every step still does the full work."""

    def __init__(self, dev, seed: int, batch: int = None):
        import torch
        import exact_replay_decode_gb300 as ers
        from synth import torch_io
        self.ers, self.torch = ers, torch
        w = synth.workload("decode_b256_h64")
        d = w.dims
        self.w = w
        self.S = batch or w.batch
        params, hist, p0, stream = synth.decode_inputs(w, seed=seed, batch=self.S, steps=TOKEN_RING)
        A, D, dtb = torch_io.params_to(params, dev)
        self.prm = ers.LayerParams(A, D, dtb)
        self.cache = ers.ReplayCache(self.S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.bfloat16)
        ht = synth.Tokens.concat(hist)
        cu = torch.tensor(np.concatenate([[0], np.cumsum([h.ntokens for h in hist])]), dtype=torch.int32, device=dev)
        ers.chunked_prefill(self.cache, self.prm, *torch_io.tokens_to(ht, dev), cu)
        self.tok = torch_io.tokens_to(stream, dev, lead=(TOKEN_RING, self.S))
        self.y = torch.empty(self.S, d.nheads, d.headdim, dtype=torch.bfloat16, device=dev)
        self.status = ers.Status(dev)
        # k_decode_heads twice: the slots whose step fills the chunk, then the others as its
        # programmatic dependent (the kernel advances the positions itself)
        self.launches_per_step = 2

    def step(self, k: int):
        x, dt, B, C = (t[k % TOKEN_RING] for t in self.tok)
        self.ers.replay_decode(self.cache, self.prm, x, dt, B, C, status=self.status, check=False, out=self.y)


def _soak(step, seconds: float, k0: int = 0):
    import torch
    t0 = time.perf_counter()
    k = k0
    while time.perf_counter() - t0 < seconds:
        for _ in range(32):
            step(k)
            k += 1
        torch.cuda.synchronize()
    return k


def time_decode(dev, steps: int, warmup: int, seed: int, batch=None):
    import torch
    b = DecodeBench(dev, seed, batch)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        for k in range(warmup):
            b.step(k)
        k = _soak(b.step, SOAK_S, warmup)
        torch.cuda.synchronize()
        _barrier()
        torch.cuda.synchronize()
        clk.mark_start()
        e0.record(s)
        for i in range(steps):
            b.step(k + i)
        e1.record(s)
        torch.cuda.synchronize()
        clk.mark_stop()
        _barrier()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    b.status.raise_if_error("bench decode")
    return b, ms, clk.summary()


def time_decode_e2e(dev, steps: int, warmup: int, seed: int, batch=None):
    """Same workload through the public API with host buffers.  Every step copies its tokens from
    pinned host memory and reads its outputs back into pinned host memory, inside the timed region.
    The copies are pipelined the way a serving loop would: step k+1's inputs upload on one copy
    stream and step k-1's outputs download on another while step k computes (double-buffered device
    tensors; events order every reuse).  A step's inputs are one packed pinned block, so each step
    makes one upload and one download call."""
    import torch
    b = DecodeBench(dev, seed, batch)
    # one step's x, dt, B and C travel as one packed pinned block and one copy (each part starts on a
    # 16-byte boundary); the decode call gets views of the device block
    parts = [t[0] for t in b.tok]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = np.concatenate([[0], np.cumsum([(n + 15) // 16 * 16 for n in sizes])]).astype(int)
    host = torch.empty(TOKEN_RING, int(offs[-1]), dtype=torch.uint8).pin_memory()
    for k in range(TOKEN_RING):
        for q, t in enumerate(b.tok):
            host[k, offs[q]:offs[q] + sizes[q]].copy_(t[k].reshape(-1).view(torch.uint8).cpu())
    dev_blk = [torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = [[blk[offs[q]:offs[q] + sizes[q]].view(parts[q].dtype).view(parts[q].shape) for q in range(4)]
              for blk in dev_blk]
    y_dev = [torch.empty_like(b.y) for _ in range(2)]
    y_host = [torch.empty(b.y.shape, dtype=b.y.dtype).pin_memory() for _ in range(2)]
    h2d = sum(sizes)
    d2h = y_host[0].numel() * y_host[0].element_size()
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, y_ready, y_free = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in in_free + y_free:
        e.record(comp)

    def upload(k):
        j = k % 2
        up.wait_event(in_free[j])
        with torch.cuda.stream(up):
            dev_blk[j].copy_(host[k % TOKEN_RING], non_blocking=True)
        in_ready[j].record(up)

    def run(k0, n):
        upload(k0)
        for k in range(k0, k0 + n):
            j = k % 2
            if k + 1 < k0 + n:
                upload(k + 1)
            comp.wait_event(in_ready[j])
            comp.wait_event(y_free[j])
            b.ers.replay_decode(b.cache, b.prm, *dev_in[j], status=b.status, check=False, out=y_dev[j])
            in_free[j].record(comp)
            y_ready[j].record(comp)
            down.wait_event(y_ready[j])
            with torch.cuda.stream(down):
                y_host[j].copy_(y_dev[j], non_blocking=True)
            y_free[j].record(down)

    run(0, warmup)
    torch.cuda.synchronize()
    _barrier()
    t0 = time.perf_counter()
    run(warmup, steps)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    _barrier()
    b.status.raise_if_error("bench decode e2e")
    return el * 1e3, h2d, d2h


def _flush_buf(dev):
    import torch
    return torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)


def _l2_flush(fb):
    """Evict L2 by READING a buffer larger than it: the lines it leaves are clean, so the timed
    kernel's misses cost no write-backs of the flush itself (a write-based flush would leave ~129 MB
    of dirty lines for the timed kernel to write back)."""
    fb.sum()


def time_per_iter(fn, iters: int, warmup: int, dev, flush: bool = True, graph: bool = False):
    """Median device time of fn() over iters, L2 flushed before each timed call (events per call).
    With graph=True, fn is captured once in a CUDA graph and each timed call replays it, so that the
    host-side work of a call (argument checks, marshalling, launch) cannot leave the device idle
    between the events: the replay is enqueued while the preceding flush still runs."""
    import torch
    fb = _flush_buf(dev) if flush else None
    for _ in range(warmup):
        fn()
    run = fn
    if graph:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        run = g.replay
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(iters):
        if fb is not None:
            _l2_flush(fb)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        run()
        e1.record(s)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median([a.elapsed_time(b) for a, b in evs])


def bench_prefill(dev, name: str, iters: int, warmup: int, hbm: float, tc: float):
    import torch
    import exact_replay_decode_gb300 as ers
    from synth import torch_io
    w = synth.workload(name)
    params, toks, cu = synth.prefill_inputs(w, seed=0)
    A, D, dtb = torch_io.params_to(params, dev)
    prm = ers.LayerParams(A, D, dtb)
    x, dt, B, C = torch_io.tokens_to(toks, dev)
    cu_t = torch.from_numpy(cu).to(dev)
    S = len(cu) - 1
    ms_len = int(np.diff(cu).max())
    y = torch.empty_like(x)
    fin = torch.empty(S, w.dims.nheads, w.dims.headdim, w.dims.dstate, dtype=torch.float32, device=dev)
    ws = torch.empty(1 << 28, dtype=torch.uint8, device=dev)
    st = ers.Status(dev)
    fn = lambda: ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=w.dims.chunk, cu_seqlens=cu_t, max_seqlen=ms_len,
                                  status=st, check=False, out=(y, fin), workspace=ws)
    ms = time_per_iter(fn, iters, warmup, dev, graph=True)
    st.raise_if_error("bench prefill")
    T = toks.ntokens
    ach = PREFILL_BYTES[name] / (ms * 1e-3) / 1e9
    return {"tok_per_s": T / (ms * 1e-3), "us_per_call": ms * 1e3, "achieved_gbs": ach,
            "hbm_frac": ach / hbm, "roofline_us": PREFILL_BYTES[name] / (hbm * 1e9) * 1e6,
            "tflops": PREFILL_FLOPS[name] / (ms * 1e-3) / 1e12,
            "l2": "flushed before each call (one CUDA-graph replay of the call per timed iteration)"}


def flat_prefill(pf: dict, cpu: dict = None) -> dict:
    """The SSD prefill figures as one flat object of scalars (the 2048-token workload's keys bare,
    the varlen workload's prefixed), with the oracle's prefill tokens/s beside them when measured."""
    a, v = pf["prefill_2048_h32"], pf["varlen_4seq_h64"]
    out = {"workload": "prefill_2048_h32 (1 x 2048 tok, 32 heads / 1 group) and varlen_4seq_h64 "
                       "({2048, 777, 513, 1}, 64 heads / 8 groups); headdim 64, dstate 128, chunk 256, bf16"}
    for pre, r in (("", a), ("varlen_", v)):
        for k in ("tok_per_s", "us_per_call", "achieved_gbs", "hbm_frac", "roofline_us", "tflops"):
            out[pre + k] = r[k]
        out[pre + "algorithmic_bytes"] = PREFILL_BYTES["prefill_2048_h32" if pre == "" else "varlen_4seq_h64"]
    out["l2"] = a["l2"]
    if cpu is not None:
        out["cpu_tok_per_s"] = cpu.get("prefill_tok_per_s")
        out["cpu_cores"] = cpu.get("cores")
        out["cpu_tok_per_s_one_core"] = cpu.get("prefill_tok_per_s_one_core")
    return out


def _copy_bytes(d, read_dtype: str) -> int:
    """Bytes of one sequence's read copy: bf16 values; FP8 codes + an fp32 scale per row; NVFP4
    codes (half a byte per value) + an e4m3 scale per 16 values + an fp32 scale per row."""
    rows = d.nheads * d.headdim
    if read_dtype == "bf16":
        return rows * d.dstate * 2
    if read_dtype == "fp8":
        return rows * (d.dstate + 4)
    return rows * (d.dstate // 2 + d.dstate // 16 + 4)


VERIFY_WARMUP = 3   # untimed verify + commit steps before the timed ones


def bench_verify(dev, steps: int, hbm: float, read_dtype: str = "bf16", anchor: str = "fp32"):
    import torch
    import exact_replay_decode_gb300 as ers
    from synth import torch_io
    w = synth.workload("verify_b512_t4")
    d = w.dims
    S, T, L = w.batch, w.drafts, d.chunk
    params, hist, drafts, acc = synth.verify_inputs(w, seed=0, steps=steps)
    A, D, dtb = torch_io.params_to(params, dev)
    prm = ers.LayerParams(A, D, dtb)
    hx, hdt, hB, hC = torch_io.tokens_to(hist, dev)
    cu = torch.arange(0, S * 32 + 1, 32, dtype=torch.int32, device=dev)
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=L, cu_seqlens=cu)
    cache = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                            read_dtype=read_dtype, anchor=anchor, sr_key=(0x5EED, 0xF00D))
    _seed_cache(ers, cache, prm, fin, L)
    anchor_bytes = _anchor_bytes(d, anchor)
    # read copy per sequence: bf16 values, or FP8 codes + one fp32 scale per state row
    copy_bytes = _copy_bytes(d, read_dtype)
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev, lead=(steps, S, T))
    acc_t = torch.from_numpy(acc).to(dev)
    y = torch.empty(S, T, d.nheads, d.headdim, dtype=torch.bfloat16, device=dev)
    st = ers.Status(dev)
    # algorithmic bytes from the actual committed pointers and flush decisions
    hs = np.zeros(S, dtype=np.int64)
    total_bytes = 0
    warm = VERIFY_WARMUP   # untimed steps first: module loading and first-launch setup stay outside
    for k in range(steps):
        flush = hs + T > L
        base = np.where(flush, 0, hs)
        b = S * (copy_bytes + 50_176 + 50_176 + 32_768) + int(base.sum()) * 10_496
        # a flushing slot reads and writes its anchor and writes its copy instead of reading it (a
        # shared NVFP4 state: reads the copy as the anchor and writes it)
        flush_extra = copy_bytes if anchor == "nvfp4_sr_shared" else 2 * anchor_bytes
        b += int(flush.sum()) * flush_extra + int(hs[flush].sum()) * 10_496
        if k >= warm:
            total_bytes += b
        hs = base + acc[k]

    def step(k):
        cache.sr_nonce = k + 1
        ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k], status=st, check=False, out=y)
        ers.commit(cache, acc_t[k], T, status=st, check=False)

    for k in range(warm):
        step(k)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for k in range(warm, steps):
        step(k)
    e1.record(s)
    torch.cuda.synchronize()
    st.raise_if_error("bench verify")
    ms = e0.elapsed_time(e1)
    timed = steps - warm
    ach = total_bytes / (ms * 1e-3) / 1e9
    return {"read_copy": read_dtype, "anchor": anchor, "seq_verify_steps_per_s": S * timed / (ms * 1e-3),
            "committed_tok_per_s": float(acc[warm:].sum()) / (ms * 1e-3), "us_per_step": ms * 1e3 / timed,
            "achieved_gbs": ach, "hbm_frac": ach / hbm, "algorithmic_bytes": total_bytes, "steps": timed,
            "warmup_steps": warm}


def bench_verify_exact(dev, steps: int, hbm: float, T: int = 4):
    """Exact-mode speculative verify + commit that keep the chunk grid (ers_spec_verify_exact /
    ers_commit_exact) on the decode workload: 256 sequences with fp32 checkpoints, chunk 16, T
    drafts per step, accepted ~ U{0..T}; 3 untimed steps, then `steps` timed ones.  Bytes: the
    single-pass minimum of the method (each sequence's checkpoint read once, its buffered rows, the
    drafts in and their outputs, the accepted drafts appended, a chunk fold's checkpoint write);
    the kernels make about T + 1 passes (a shadow snapshot, T decode steps), so the fraction is low
    by construction."""
    import ctypes
    import torch
    import exact_replay_decode_gb300 as ers
    from exact_replay_decode_gb300 import _abi
    from synth import torch_io
    w = synth.workload("decode_b256_h64")
    d = w.dims
    S, Q = w.batch, d.chunk
    warm = VERIFY_WARMUP
    K = steps + warm
    params, hist, p0, stream = synth.decode_inputs(w, seed=5, batch=S, steps=K * T)
    A, D, dtb = torch_io.params_to(params, dev)
    prm = ers.LayerParams(A, D, dtb)
    cu = torch.tensor(np.concatenate([[0], np.cumsum([h.ntokens for h in hist])]), dtype=torch.int32, device=dev)
    hx, hdt, hB, hC = torch_io.tokens_to(synth.Tokens.concat(hist), dev)
    cache = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, Q, torch.bfloat16)
    ers.chunked_prefill(cache, prm, hx, hdt, hB, hC, cu)
    del hx, hdt, hB, hC
    drafts = [t.transpose(1, 2).contiguous() for t in torch_io.tokens_to(stream, dev, lead=(K, T, S))]
    acc = np.random.Generator(np.random.PCG64(6)).integers(0, T + 1, size=(K, S)).astype(np.int32)
    acc_t = torch.from_numpy(acc).to(dev)
    ws = torch.empty(_abi.lib().ers_spec_verify_exact_workspace_size(ctypes.byref(cache.dims), S), dtype=torch.uint8,
                     device=dev)
    y = torch.empty(S, T, d.nheads, d.headdim, dtype=torch.bfloat16, device=dev)
    st = ers.Status(dev)
    state_bytes = d.nheads * d.headdim * d.dstate * 4
    hs = p0.astype(np.int64)
    total = 0
    for k in range(K):
        b = S * (state_bytes + T * (12_544 + 8_192)) + int(hs.sum()) * 10_496 + int(acc[k].sum()) * 12_544
        b += int(((hs + acc[k]) >= Q).sum()) * state_bytes          # a filled chunk's checkpoint write
        if k >= warm:
            total += b
        hs = (hs + acc[k]) % Q

    def step(k, mid=None):
        dx, ddt, dB, dC = (t[k] for t in drafts)
        ers.spec_verify_exact(cache, prm, dx, ddt, dB, dC, status=st, check=False, out=y, workspace=ws)
        if mid is not None:
            mid.record(torch.cuda.current_stream())
        ers.commit_exact(cache, prm, acc_t[k], dx, ddt, dB, dC, status=st, check=False, workspace=ws)

    for k in range(warm):
        step(k)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    # events at every step's start and after its verify: the step and its verify share
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for n, k in enumerate(range(warm, K)):
        ev[n][0].record(s)
        step(k, ev[n][1])
    e1.record(s)
    torch.cuda.synchronize()
    st.raise_if_error("bench exact verify")
    verify_ms = sum(a.elapsed_time(b) for a, b in ev)
    if not np.array_equal(cache.pos.cpu().numpy(), hs.astype(np.int32)):
        raise AssertionError("exact verify bench: positions differ from the byte model")
    ms = e0.elapsed_time(e1)
    ach = total / (ms * 1e-3) / 1e9
    return {"drafts": T, "seq_verify_steps_per_s": S * steps / (ms * 1e-3),
            "committed_tok_per_s": float(acc[warm:].sum()) / (ms * 1e-3), "us_per_step": ms * 1e3 / steps,
            "verify_us_per_step": verify_ms * 1e3 / steps, "achieved_gbs": ach, "hbm_frac": ach / hbm,
            "single_pass_bytes": total, "steps": steps, "warmup_steps": warm}


def _anchor_bytes(d, anchor: str) -> int:
    """Bytes of one sequence's separate anchor: fp32 or fp16 (none for the shared NVFP4 state)."""
    if anchor == "nvfp4_sr_shared":
        return 0
    return d.nheads * d.headdim * d.dstate * (2 if anchor == "fp16_sr" else 4)


def _seed_cache(ers, cache, prm, fin, L: int) -> None:
    """Put the fp32 state fin into the cache with every position 0: anchor copied and read copy cast,
    or (shared NVFP4 state) the round-to-nearest cast."""
    if cache.anchor == "nvfp4_sr_shared":
        cache.seed(fin, prm)
        return
    cache.state.copy_(fin)
    ers.refresh(cache, prm, replayssm=True, drafts_T=L + 1)


def bench_rssm_decode(dev, cycles: int, hbm: float, read_dtype: str, anchor: str = "fp32"):
    """Non-speculative ReplaySSM decode of the B=256 decode workload: each step is one fused decode
    call, which applies the flush rule for one token (h + 1 > L: fold the anchor, recast the read
    copy) and decodes from the read copy.  One ring cycle of steps (TOKEN_RING) is captured as a
    CUDA graph and replayed, so the host's per-call overhead does not pace the GPU.  Start positions
    h0 ~ U{0..L-1} per sequence (untimed decodes of slot subsets).  anchor "fp16_sr": fp16 anchors
    written by stochastic rounding (nonce = the ring step; the graph replays the same nonces)."""
    import torch
    import exact_replay_decode_gb300 as ers
    from synth import torch_io
    w = synth.workload("decode_b256_h64")
    d = w.dims
    S, L = w.batch, d.chunk
    params, hist, h0, stream = synth.decode_inputs(w, seed=3, batch=S, steps=TOKEN_RING)
    A, D, dtb = torch_io.params_to(params, dev)
    prm = ers.LayerParams(A, D, dtb)
    ht = synth.Tokens.concat(hist)
    cu = torch.tensor(np.concatenate([[0], np.cumsum([h.ntokens for h in hist])]), dtype=torch.int32, device=dev)
    hx, hdt, hB, hC = torch_io.tokens_to(ht, dev)
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=L, cu_seqlens=cu)
    del hx, hdt, hB, hC
    cache = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                            read_dtype=read_dtype, anchor=anchor, sr_key=(0x5EED, 0xF00D))
    _seed_cache(ers, cache, prm, fin, L)                                # h = 0: cast the read copy
    tok = torch_io.tokens_to(stream, dev, lead=(TOKEN_RING, S))
    y = torch.empty(S, d.nheads, d.headdim, dtype=torch.bfloat16, device=dev)
    st = ers.Status(dev)
    for r in range(L - 1):                                              # advance slot i to h0[i]
        sel = torch.from_numpy(np.nonzero(h0 > r)[0].astype(np.int32)).to(dev)
        if sel.numel():
            sl = sel.long()
            ers.replay_decode(cache, prm, *(t[TOKEN_RING - 1][sl] for t in tok), slot=sel, replayssm=True,
                              fuse_refresh=False)

    def step(k):
        cache.sr_nonce = k
        ers.replay_decode(cache, prm, *(t[k] for t in tok), replayssm=True, fuse_refresh=True, status=st,
                          check=False, out=y)

    # algorithmic bytes from the run's own pointers: a flush reads and writes the anchor (a shared
    # NVFP4 state: reads and writes the copy), reads the h buffered rows and writes the copy, and its
    # output comes from the new values; a decode without a flush reads the copy; every step reads
    # its h rows and the new token and writes the token to the buffer and y
    copy_bytes = _copy_bytes(d, read_dtype)
    anchor_bytes = _anchor_bytes(d, anchor)
    shared = anchor == "nvfp4_sr_shared"
    hs = h0.astype(np.int64)

    def cycle_bytes():
        nonlocal hs
        b = 0
        for _ in range(TOKEN_RING):
            fl = hs + 1 > L
            nfl = int(fl.sum())
            b += nfl * (2 * anchor_bytes + copy_bytes + (copy_bytes if shared else 0)) + int(hs[fl].sum()) * 10_496
            hs = np.where(fl, 0, hs)
            b += (S - nfl) * copy_bytes + S * (12_544 + 12_544 + 8_192) + int(hs.sum()) * 10_496
            hs = hs + 1
        return b

    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):            # captured, not run
        for k in range(TOKEN_RING):
            step(k)
    g.replay()                                                          # untimed cycle
    cycle_bytes()
    total = sum(cycle_bytes() for _ in range(cycles))
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(cycles):
        g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    st.raise_if_error("bench replayssm decode")
    if not np.array_equal(cache.pos.cpu().numpy(), hs.astype(np.int32)):
        raise AssertionError("ReplaySSM decode bench: positions differ from the byte model")
    nsteps = cycles * TOKEN_RING
    ms = e0.elapsed_time(e1) / nsteps
    ach = total / nsteps / (ms * 1e-3) / 1e9
    return {"read_copy": read_dtype, "anchor": anchor, "seq_steps_per_s": S / (ms * 1e-3), "us_per_step": ms * 1e3,
            "achieved_gbs": ach, "hbm_frac": ach / hbm, "bytes_per_step": total / nsteps, "steps": nsteps,
            # two launches per fused call whatever the copy (the tensor-core kernel for bf16, the
            # warp-per-head kernel otherwise): the flushing slots, then the others as its dependent
            "launches_per_step": 2}


def bench_conv(dev, hbm: float, reps: int = 50):
    """The causal conv1d upstream of the SSM on the decode workload's channels (x, B and C: 64 x 64 +
    2 x 8 x 128 = 6144), width 4, bf16: one update step for 256 sequences (bytes: state read and
    write 2 x 3 rows, x and y rows, per sequence) and a 2048-token prefill (x read, y written).  L2 is
    flushed (a 256 MB read) before each timed call."""
    import torch
    import exact_replay_decode_gb300 as ers
    rng = np.random.Generator(np.random.PCG64(12))
    C, W, S, T = 6144, 4, 256, 2048
    cast = lambda a: torch.from_numpy(a.astype(np.float32)).to(dev).to(torch.bfloat16)
    w = cast(rng.standard_normal((C, W)) * 0.5)
    b = cast(rng.standard_normal(C) * 0.1)
    xs = cast(rng.standard_normal((S, C)))
    xp = cast(rng.standard_normal((T, C)))
    state = cast(rng.standard_normal((S, W - 1, C)))
    y = torch.empty_like(xs)
    yp = torch.empty_like(xp)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    flush = _flush_buf(dev)
    st = ers.Status(dev)

    def timed(fn):
        s = torch.cuda.current_stream()
        ts = []
        for _ in range(reps):
            _l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))
    upd = lambda: ers.conv1d_update(xs, w, b, state, status=st, check=False, out=y)
    pre = lambda: ers.conv1d_fwd(xp, w, b, cu, max_seqlen=T, status=st, check=False, out=yp)
    for _ in range(3):
        upd(); pre()
    ms_u, ms_p = timed(upd), timed(pre)
    st.raise_if_error("bench conv")
    bytes_u = S * C * 2 * (2 * (W - 1) + 2) + C * W * 2 + C * 2
    bytes_p = 2 * T * C * 2 + C * W * 2 + C * 2
    return {"update_b256": {"us": ms_u * 1e3, "seq_steps_per_s": S / (ms_u * 1e-3), "bytes": bytes_u,
                            "hbm_frac": bytes_u / (ms_u * 1e-3) / 1e9 / hbm},
            "prefill_2048": {"us": ms_p * 1e3, "tok_per_s": T / (ms_p * 1e-3), "bytes": bytes_p,
                             "hbm_frac": bytes_p / (ms_p * 1e-3) / 1e9 / hbm},
            "l2": "flushed before each call"}


def bench_gdn_verify(dev, steps: int, hbm: float, batch: Optional[int] = None):
    """Output-only verify of a gated-delta-rule layer: 512 sequences x 4 drafts, 32 value heads / 16
    key groups, dk = dv = 128, window 16, bf16 io, 3 warm-up steps (then the cache goes back to its
    start), 32 timed verify + commit steps; the 512 MiB read copy exceeds L2.  Bytes from the run's own
    pointers and flushes: per sequence-step the read copy (32 x 128 x 128 bf16), the drafts' q, k, v,
    g, beta in and o out, the committed records' k and cached residuals (and g, beta) read, and the
    drafts' k, v, residuals, g, beta written to the buffer; per flush the anchor read and written, the
    copy written instead of read, and the records' k and v read."""
    import torch
    import exact_replay_decode_gb300 as ers
    d = synth.GDN_VERIFY["dims"]
    S, T = batch or synth.GDN_VERIFY["batch"], synth.GDN_VERIFY["drafts"]
    anchor, toks, acc = synth.gdn_verify_inputs(0, S, steps, d, T)
    cache = ers.GdnCache(S, d.nheads, d.ngroups, d.dk, d.dv, d.window, torch.bfloat16)
    cache.anchor.copy_(torch.from_numpy(anchor))
    cache.read_copy.copy_(cache.anchor)
    to = lambda a, dt: torch.from_numpy(a).to(dev).to(dt)
    q = to(toks.q, torch.bfloat16).view(steps, S, T, d.ngroups, d.dk)
    k = to(toks.k, torch.bfloat16).view(steps, S, T, d.ngroups, d.dk)
    v = to(toks.v, torch.bfloat16).view(steps, S, T, d.nheads, d.dv)
    g = to(toks.g, torch.float32).view(steps, S, T, d.nheads)
    beta = to(toks.beta, torch.float32).view(steps, S, T, d.nheads)
    acc_t = torch.from_numpy(acc).to(dev)
    o = torch.empty(S, T, d.nheads, d.dv, dtype=torch.bfloat16, device=dev)
    st = ers.Status(dev)
    H, G, D = d.nheads, d.ngroups, d.dk
    copy = H * D * D * 2
    row_read = G * D * 2 + H * D * 4 + H * 8                 # committed k, residual u, g and beta
    row_write = G * D * 2 + H * D * 2 + H * D * 4 + H * 8    # a draft's k, v, u, g, beta
    io = T * (2 * G * D * 2 + H * D * 2 + H * 8) + T * H * D * 2
    for kk in range(min(3, steps)):                              # warm-up, then back to the start
        ers.gdn_verify(cache, q[kk], k[kk], v[kk], g[kk], beta[kk], status=st, check=False, out=o)
        ers.gdn_commit(cache, acc_t[kk], T, status=st, check=False)
    cache.anchor.copy_(torch.from_numpy(anchor))
    cache.read_copy.copy_(cache.anchor)
    cache.pos.zero_()
    hs = np.zeros(S, dtype=np.int64)
    total = 0
    for kk in range(steps):
        fl = hs + T > d.window
        base = np.where(fl, 0, hs)
        total += S * (copy + io + T * row_write) + int(base.sum()) * row_read
        total += int(fl.sum()) * (2 * H * D * D * 4) + int(hs[fl].sum()) * (G * D * 2 + H * D * 2 + H * 8)
        hs = base + acc[kk]
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for kk in range(steps):
        ers.gdn_verify(cache, q[kk], k[kk], v[kk], g[kk], beta[kk], status=st, check=False, out=o)
        ers.gdn_commit(cache, acc_t[kk], T, status=st, check=False)
    e1.record(s)
    torch.cuda.synchronize()
    st.raise_if_error("bench gdn verify")
    ms = e0.elapsed_time(e1)
    ach = total / (ms * 1e-3) / 1e9
    return {"seq_verify_steps_per_s": S * steps / (ms * 1e-3), "committed_tok_per_s": float(acc.sum()) / (ms * 1e-3),
            "us_per_step": ms * 1e3 / steps, "achieved_gbs": ach, "hbm_frac": ach / hbm, "algorithmic_bytes": total,
            "steps": steps}


def bench_ssu(dev, steps: int, hbm: float):
    import torch
    import exact_replay_decode_gb300 as ers
    from synth import torch_io
    w = synth.workload("decode_b256_h64")
    d = w.dims
    S = w.batch
    rng = np.random.Generator(np.random.PCG64(5))
    params = synth.make_params(rng, d.nheads)
    toks = synth.make_tokens(rng, (steps + 3) * S, d, True)
    A, D, dtb = torch_io.params_to(params, dev)
    prm = ers.LayerParams(A, D, dtb)
    x, dt, B, C = torch_io.tokens_to(toks, dev, lead=(steps + 3, S))
    state = torch.randn(S, d.nheads, d.headdim, d.dstate, device=dev)
    y = torch.empty(S, d.nheads, d.headdim, dtype=torch.bfloat16, device=dev)
    st = ers.Status(dev)
    for k in range(3):
        ers.ssu_update(state, prm, x[k], dt[k], B[k], C[k], status=st, check=False, out=y)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for k in range(3, steps + 3):
        ers.ssu_update(state, prm, x[k], dt[k], B[k], C[k], status=st, check=False, out=y)
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ach = SSU_BYTES_PER_SEQ_STEP * S / (ms * 1e-3) / 1e9
    return {"seq_steps_per_s": S / (ms * 1e-3), "us_per_step": ms * 1e3, "achieved_gbs": ach, "hbm_frac": ach / hbm}


# ---------------------------------------------------------------------------------------------
class _OracleDecode:
    """The fp64 oracle advancing a sample of the B=256 decode workload token by token.

    Tokens come from a small pre-generated ring (sequence-major, ready for the oracle's varlen
    call) so that only the recurrence itself is timed; the state is carried from call to call."""

    def __init__(self, seed: int, S: int, K: int, ring: int = 4, threads: Optional[int] = None):
        import oracle
        self.oracle = oracle
        w = synth.workload("decode_b256_h64")
        self.d = d = w.dims
        self.threads = threads or oracle.default_threads()
        rng = np.random.Generator(np.random.PCG64(seed))
        self.params = synth.make_params(rng, d.nheads)
        self.S, self.K = S, K
        order = np.arange(S * K).reshape(K, S).T.reshape(-1)
        self.ring = []
        for _ in range(ring):
            t = synth.make_tokens(rng, S * K, d, True)
            self.ring.append(tuple(np.ascontiguousarray(a[order]) for a in (t.x, t.dt, t.B, t.C)))
        self.cu = np.arange(0, S * K + 1, K)
        self.state = rng.standard_normal((S, d.nheads, d.headdim, d.dstate))
        self.i = 0

    def call(self):
        x, dt, B, C = self.ring[self.i % len(self.ring)]
        self.i += 1
        p = self.params
        _, self.state = self.oracle.recurrence(x, dt, p.A, B, C, p.D, p.dt_bias, self.cu, self.state,
                                               nthreads=self.threads)
        return self.S * self.K


def _timed(fn, budget_s: float):
    """Calls fn() (returning units done) until budget_s has passed; returns (units, seconds)."""
    done, t0 = 0, time.perf_counter()
    while True:
        done += fn()
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done, el


def _oracle_prefill(threads: int, budget_s: float):
    """The oracle's prefill of prefill_2048_h32 (one call = all 2048 tokens): tokens/s."""
    import oracle
    w = synth.workload("prefill_2048_h32")
    params, toks, cu = synth.prefill_inputs(w, seed=0)
    def run():
        oracle.recurrence(toks.x, toks.dt, params.A, toks.B, toks.C, params.D, params.dt_bias, cu, nthreads=threads)
        return toks.ntokens
    done, el = _timed(run, budget_s)
    return {"value": done / el, "unit": "tok/s", "cores": threads,
            "sample": f"prefill_2048_h32 whole calls, {done // toks.ntokens} in {el:.1f} s"}


def _oracle_verify(threads: int, budget_s: float):
    """The oracle's ReplaySSM protocol model on 16 sequences of verify_b512_t4 (verify + commit per
    step, flushes included): sequence-verify-steps/s."""
    import oracle
    w = synth.workload("verify_b512_t4")
    S, K, T, L = 16, 8, w.drafts, w.dims.chunk
    params, hist, drafts, acc = synth.verify_inputs(w, seed=0, batch=S, steps=K)
    _, anchor = oracle.recurrence(hist.x, hist.dt, params.A, hist.B, hist.C, params.D, params.dt_bias,
                                  np.arange(0, S * 32 + 1, 32), nthreads=threads)
    sh = lambda a: a.reshape(K, S, T, *a.shape[1:])
    dr = [[tuple(sh(a)[k, i] for a in (drafts.x, drafts.dt, drafts.B, drafts.C)) for i in range(S)] for k in range(K)]
    state = {"m": None, "k": K}

    def step():
        if state["k"] == K:
            state["m"], state["k"] = oracle.ReplaySSMModel(params, anchor, L, nthreads=threads), 0
        k = state["k"]
        state["m"].verify(dr[k])
        state["m"].commit(acc[k])
        state["k"] += 1
        return S
    done, el = _timed(step, budget_s)
    return {"value": done / el, "unit": "seq-verify-steps/s", "cores": threads,
            "sample": f"{S} of the 512 sequences x {done // S} verify + commit steps (bf16 read copy, L 16, "
                      f"4 drafts), {el:.1f} s"}


def cpu_baseline(seed: int, budget_s: float = 10.0):
    """fp64 oracle on this host's cores: decode seq-steps/s on a bounded sample of the B=256
    workload (32 of the sequences advanced 16 steps per call, state carried, for ~budget_s), plus
    the same on one core and, on all cores and on one, prefill_2048_h32 tokens/s and
    verify_b512_t4 sequence-verify-steps/s (bounded samples of ~2 s each)."""
    o = _OracleDecode(seed, S=32, K=16)
    o.call()
    done, el = _timed(o.call, budget_s)
    d = o.d
    out = {"value": done / el, "unit": "seq-steps/s", "cores": o.threads, "kind": "oracle",
           "sample": f"{o.S} of the 256 sequences x {done // o.S} decode steps, state carried (fp64 recurrence, "
                     f"{d.nheads} heads, headdim {d.headdim}, dstate {d.dstate}), {el:.1f} s"}
    o1 = _OracleDecode(seed, S=8, K=4, threads=1)
    done1, el1 = _timed(o1.call, 2.0)
    # the other samples as flat scalars (value, then its sample text)
    out["decode_one_core"] = done1 / el1
    out["decode_one_core_sample"] = f"8 sequences x {done1 // 8} decode steps, 1 core, {el1:.1f} s"
    for key, fn, unit in (("prefill", _oracle_prefill, "tok_per_s"), ("verify", _oracle_verify, "seq_verify_steps_per_s")):
        for suffix, th in (("", o.threads), ("_one_core", 1)):
            r = fn(th, 2.0)
            out[f"{key}_{unit}{suffix}"] = r["value"]
            out[f"{key}_sample{suffix}"] = f"{r['sample']}, {th} core(s)"
    return out


def reference_arm(args):
    """The fp64 oracle as the reference implementation, timed on host cores.  One step advances a
    16-sequence sample of the B=256 workload by 4 tokens."""
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    o = _OracleDecode(1, S=16, K=4)
    for _ in range(args.warmup):
        o.call()
    t0 = time.perf_counter()
    done = 0
    for _ in range(args.steps):
        done += o.call()
    el = time.perf_counter() - t0
    v = done / el
    line = {"impl": "reference", "metric": "replay-decode seq-steps/s per layer @B=256", "value": v,
            "unit": "seq-steps/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode_b256_h64 (sampled)", "batch": 256,
                       "sample_per_step": f"{o.S} seqs x {o.K} steps"},
            "cpu_baseline": {"value": v, "unit": "seq-steps/s", "cores": o.threads, "kind": "oracle",
                             "sample": f"{o.S} sequences x {o.K} decode steps per step, state carried, "
                                       f"fp64 recurrence"},
            "e2e": {"value": v, "unit": "seq-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-only", action="store_true", help="only the headline decode measurement")
    ap.add_argument("--batch", type=int, default=None,
                    help="decode (or, with --section gdn, GDN) sequences per GPU (profiling runs only)")
    ap.add_argument("--section", choices=["prefill", "verify", "rssm", "ssu", "conv", "gdn", "exact"], default=None,
                    help="run only this secondary workload and print its JSON (profiling aid, no headline)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist
    ws, rank, local = _dist()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm, tc, peak_kind = _peaks()
    if args.section is not None:
        if args.section == "prefill":
            out = {n: bench_prefill(dev, n, 20, args.warmup, hbm, tc) for n in ("prefill_2048_h32", "varlen_4seq_h64")}
        elif args.section == "conv":
            out = bench_conv(dev, hbm)
        elif args.section == "gdn":
            out = bench_gdn_verify(dev, 32, hbm, args.batch)
        elif args.section == "exact":
            out = bench_verify_exact(dev, 32, hbm)
        elif args.section == "rssm":
            out = {r: bench_rssm_decode(dev, 4, hbm, r) for r in ("bf16", "fp8", "nvfp4")}
            out["nvfp4_fp16sr"] = bench_rssm_decode(dev, 4, hbm, "nvfp4", "fp16_sr")
            out["nvfp4_shared_sr"] = bench_rssm_decode(dev, 4, hbm, "nvfp4", "nvfp4_sr_shared")
        elif args.section == "verify":
            out = bench_verify(dev, 32 + VERIFY_WARMUP, hbm)
            fp8 = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "fp8")
            nv4 = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "nvfp4")
            nv4sr = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "nvfp4", "fp16_sr")
            nv4sh = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "nvfp4", "nvfp4_sr_shared")
            if rank == 0:
                print(json.dumps({"verify_fp8": fp8, "verify_nvfp4": nv4, "verify_nvfp4_fp16sr": nv4sr,
                                  "verify_nvfp4_shared_sr": nv4sh}))
        else:
            out = bench_ssu(dev, 16, hbm)
        if rank == 0:
            print(json.dumps({args.section: out}))
        return 0

    b, ms, clocks = time_decode(dev, args.steps, args.warmup, seed=1000 + rank, batch=args.batch)
    ms = max_over_ranks(ms, dev)
    S = b.S
    value = S * args.steps * ws / (ms * 1e-3)
    ms_step = ms / args.steps
    ach = DECODE_BYTES_PER_SEQ_STEP * S / (ms_step * 1e-3) / 1e9
    e2e_ms, h2d, d2h = time_decode_e2e(dev, args.steps, args.warmup, seed=2000 + rank, batch=args.batch)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    launches_per_step = b.launches_per_step
    del b
    torch.cuda.empty_cache()

    extra = {}
    pf = None
    if not args.decode_only:
        pf = {n: bench_prefill(dev, n, 20, 3, hbm, tc) for n in ("prefill_2048_h32", "varlen_4seq_h64")}
        extra["prefill"] = flat_prefill(pf)
        extra["verify"] = bench_verify(dev, 32 + VERIFY_WARMUP, hbm)
        extra["verify_fp8"] = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "fp8")
        extra["verify_nvfp4"] = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "nvfp4")
        extra["verify_nvfp4_fp16sr"] = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "nvfp4", "fp16_sr")
        extra["verify_nvfp4_shared_sr"] = bench_verify(dev, 32 + VERIFY_WARMUP, hbm, "nvfp4", "nvfp4_sr_shared")
        extra["replayssm_decode"] = {r: bench_rssm_decode(dev, 4, hbm, r) for r in ("bf16", "fp8", "nvfp4")}
        extra["replayssm_decode"]["nvfp4_fp16sr"] = bench_rssm_decode(dev, 4, hbm, "nvfp4", "fp16_sr")
        extra["replayssm_decode"]["nvfp4_shared_sr"] = bench_rssm_decode(dev, 4, hbm, "nvfp4", "nvfp4_sr_shared")
        extra["ssu"] = bench_ssu(dev, 16, hbm)
        extra["conv1d"] = bench_conv(dev, hbm)
        extra["gdn_verify"] = bench_gdn_verify(dev, 32, hbm)
        extra["verify_exact"] = bench_verify_exact(dev, 32, hbm)
    line = {
        "metric": "replay-decode seq-steps/s per layer @B=256",
        "value": value,
        "unit": "seq-steps/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "decode_b256_h64: 256 seqs x 64 heads / 8 groups, headdim 64, dstate 128, "
                               "chunk = refresh period 16, start position ~U{0..15}, bf16 x/B/C, fp32 checkpoint",
                   "batch_per_gpu": S, "global_batch": S * ws, "parallelism": f"replicas x{ws} (independent sequences)",
                   "l2": "inputs larger than L2 (512 MiB fp32 checkpoints per step)"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                     "traffic": profiled_traffic(), "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "kernel": "k_decode_heads (one replay-decode step; time is the whole step)",
                     "algorithmic_bytes_per_launch": DECODE_BYTES_PER_SEQ_STEP * S},
        "e2e": {"value": S * args.steps * ws / (e2e_ms * 1e-3), "unit": "seq-steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    line.update(extra)
    if pf is not None:   # the SSD scan's own roofline fractions beside the decode kernel's
        for pre, n in (("ssd_prefill_", "prefill_2048_h32"), ("ssd_prefill_varlen_", "varlen_4seq_h64")):
            line["roofline"][pre + "us"] = pf[n]["us_per_call"]
            line["roofline"][pre + "hbm_frac"] = pf[n]["hbm_frac"]
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(seed=7)
        if pf is not None:
            line["prefill"] = flat_prefill(pf, line["cpu_baseline"])
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0



if __name__ == "__main__":
    sys.exit(main())
