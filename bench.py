"""Benchmark of the exact attention forward on GB300.

One step = one pass of the whole hot path on resident synthetic inputs:
  1. causal bf16 prefill  B=1 H=32 N=16384 D=128, Q,K ~ N(0, 3^2), V ~ N(0, 1)
     (fa_fwd, the tensor-core kernel) - the headline workload;
  2. split-KV decode      B=64 H=32 D=128, KV lengths U[1024, 32768], 16 chunks
     (fa_decode_splitkv + fa_combine_states).
`value` is the prefill throughput in TFLOP/s (4 B H N^2 D, halved for causal)
over the prefill launches of the timed steps; the decode bandwidth is reported
in the `decode` object.  Inputs (537 MB prefill, ~17.7 GB decode) are larger
than the 129 MB L2, so no flush is needed between iterations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) each rank runs the same workload on its own GPU (weak
scaling, no collective on the data path); the time is the max over ranks.
`--impl reference` times the float64 CPU oracle instead, on a bounded sample
of the prefill workload per step (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import fa_inputs as inp  # noqa: E402

PREFILL = dict(B=1, H=32, N=16384, D=128)
DECODE = dict(B=64, H=32, D=128, S=16)
ROWSTATS = dict(R=65536, C=4096)  # LayerNorm statistics of 4 x 16384 tokens, hidden 4096
METRIC = "attention fwd TFLOP/s (bf16, causal) and % of GB300 BF16 peak; decode GB/s"
WORKLOAD = ("prefill B=1 H=32 N=16384 D=128 causal bf16, Q,K~N(0,9) V~N(0,1); "
            "decode B=64 H=32 D=128 L~U[1024,32768] 16 KV chunks")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def prefill_flops(B, H, N, D, causal=True) -> float:
    f = 4.0 * B * H * N * N * D
    return f / 2 if causal else f


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def load_traffic(kernel: str, source: str):
    """DRAM bytes per launch from a committed ncu capture, or None when the
    kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d:
        return None
    with open(os.path.join(ROOT, source), "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    return d["bytes_per_launch"] if d.get("source_sha256") == h else None


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed
    region runs.  Reads NVML through ctypes every 20 ms in a background thread
    (read-only queries), keeping the samples taken between mark_start() and
    mark_end(); without NVML it falls back to `nvidia-smi -lms 50`."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, index: int, uuid: Optional[str] = None):
        self.index = index
        self.uuid = uuid
        self.samples = []  # (time, sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.t0 = self.t1 = None
        self.proc = None
        self.thread = None
        self.stop = threading.Event()

    def _nvml(self):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index),
                                                   ctypes.byref(h)) == 0
        if not ok:
            return None
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = SM clock
            self.max_mhz = float(mx.value)
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons

    def _poll(self, lib, h, reasons):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if reasons(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((time.perf_counter(), float(clk.value), int(r)))
            self.stop.wait(0.02)

    def __enter__(self):
        try:
            nv = self._nvml()
        except OSError:
            nv = None
        if nv is not None:
            self.thread = threading.Thread(target=self._poll, args=nv, daemon=True)
            self.thread.start()
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
        time.sleep(0.1)  # let the first samples arrive before the timed region
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        self.stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            bits = [0x8, 0x40, 0x20, 0x4]
            for line in (out or "").strip().splitlines():
                parts = [x.strip() for x in line.split(",")]
                try:
                    sm = float(parts[0])
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    continue
                r = sum(b for b, v in zip(bits, parts[2:6]) if v.lower() == "active")
                self.samples.append((None, sm, r))

    def summary(self):
        inside = [x for x in self.samples
                  if x[0] is None or self.t0 is None or self.t0 <= x[0] <= (self.t1 or x[0])]
        sm = [x[1] for x in inside]
        reasons = set()
        for x in inside:
            for bit, name in self.REASONS.items():
                if x[2] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(dev) -> Optional[str]:
    """NVML's name of the CUDA device ("GPU-<uuid>"), when torch knows it."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle arm

def oracle_sample_step(q, k, v, scale, head: int, rows):
    """The float64 oracle on query rows `rows` of one head; returns the
    algorithmic causal FLOPs of that sample."""
    from oracle import attention as ora
    ora.attention_head_ref(q[head], k[head], v[head], scale, True, rows)
    D = q.shape[-1]
    return float(sum(4.0 * D * (int(r) + 1) for r in rows))


def cpu_sample_inputs(heads: int = 2):
    """The first `heads` heads of the prefill workload, drawn on the CPU
    generator with the prefill seed, as float64 (rows sampled per step)."""
    import numpy as np
    c = inp.dense(1, heads, PREFILL["N"], PREFILL["D"], seed=3, causal=True, qk_std=3.0)
    f = lambda t: t[0].to(torch.float64).numpy()
    return f(c.q), f(c.k), f(c.v), c.scale, np


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    q, k, v, scale, np = cpu_sample_inputs()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    N = PREFILL["N"]
    rows = np.arange(N - 384, N)  # the last 384 rows: each sees ~16K keys
    for _ in range(args.warmup):
        oracle_sample_step(q, k, v, scale, 0, rows[:64])
    t0 = time.perf_counter()
    flops = 0.0
    for s in range(args.steps):
        flops += oracle_sample_step(q, k, v, scale, s % 2, rows)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"float64 NumPy oracle, per step the last {len(rows)} query rows of one "
              f"head (of {PREFILL['H']}) against all visible keys, N={N} D={PREFILL['D']} causal")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def cpu_baseline_leg():
    """The oracle as it stands on this host's cores, on a bounded sample
    (about 10 s): full causal attention of 10 of the prefill workload's 32
    heads, every query row, in chunks of 2048 rows."""
    heads = 10
    q, k, v, scale, np = cpu_sample_inputs(heads)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    N = PREFILL["N"]
    oracle_sample_step(q, k, v, scale, 0, np.arange(N - 32, N))
    t0 = time.perf_counter()
    flops = 0.0
    for h in range(heads):
        for r0 in range(0, N, 2048):
            flops += oracle_sample_step(q, k, v, scale, h, np.arange(r0, min(N, r0 + 2048)))
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"all {N} query rows of {heads} of the 32 heads, N={N} D=128 causal, "
                      f"float64 NumPy ({dt:.1f} s)"}


# ------------------------------------------------------------------ GPU arm

def _time_launches(fn, iters: int, warmup: int = 2) -> float:
    """Mean device milliseconds of fn() over `iters` back-to-back calls
    (CUDA events on the current stream, after warm-up)."""
    for _ in range(warmup):
        fn()
    st = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(st)
    for _ in range(iters):
        fn()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def other_configs(fa):
    """The remaining workloads, each timed on its own after the main timed
    region (not part of `value`): dense causal B=4 H=16 N=2048 D=128, the
    ragged varlen prefill (65536 tokens, H=16, D=64 and 128), the causal
    sliding window, the backward, the Welford row statistics, prefix
    attention, paged GQA decode and the fp32 path (B=H=1, N=256, D=64)."""
    out = {}
    c2 = inp.config2(device="cuda")
    ms = _time_launches(lambda: fa.fa_fwd(c2.q, c2.k, c2.v, c2.scale, True), 20)
    out["dense_B4_H16_N2048_D128_causal"] = {
        "tflops": prefill_flops(4, 16, 2048, 128) / (ms * 1e-3) / 1e12, "ms": ms,
        "l2": "hot (inputs of 134 MB stay in the 129 MB L2 between launches)"}
    # the same with L2 flushed before every launch: a 512 MB write between
    # launches, each launch timed alone
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    times = []
    for it in range(23):
        flush.fill_(float(it))
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fa.fa_fwd(c2.q, c2.k, c2.v, c2.scale, True)
        b.record(st)
        b.synchronize()
        if it >= 3:
            times.append(a.elapsed_time(b))
    ms_cold = sum(times) / len(times)
    out["dense_B4_H16_N2048_D128_causal_cold_l2"] = {
        "tflops": prefill_flops(4, 16, 2048, 128) / (ms_cold * 1e-3) / 1e12, "ms": ms_cold,
        "l2": "flushed by a 512 MB write before each launch"}
    del flush
    for D in (64, 128):
        c5 = inp.config5(D, device="cuda")
        cu = c5.cu_seqlens.cuda()
        flops = sum(2.0 * 16 * L * L * D for L in c5.meta["lens"])  # causal: 4 H L^2 D / 2
        ms = _time_launches(lambda: fa.fa_fwd_varlen(c5.q, c5.k, c5.v, cu, c5.max_seqlen,
                                                     c5.scale, True), 20)
        out[f"varlen_T65536_H16_D{D}_causal"] = {
            "tflops": flops / (ms * 1e-3) / 1e12, "ms": ms, "seqs": len(c5.meta["lens"])}
    # causal sliding window, B=1 H=32 N=16384 D=128, window 4096
    cw = inp.dense(1, 32, 16384, 128, seed=3, causal=True, qk_std=3.0, device="cuda")
    ms = _time_launches(lambda: fa.fa_fwd_window(cw.q, cw.k, cw.v, 4096, cw.scale), 10)
    wf = 32 * 4.0 * 128 * sum(min(i + 1, 4096) for i in range(16384))
    out["window4096_B1_H32_N16384_D128"] = {"tflops": wf / (ms * 1e-3) / 1e12, "ms": ms}
    del cw
    # backward by recomputation of the causal prefill workload (B=1 H=32
    # N=16384 D=128): five N x N x D products per head, half of them under
    # the causal mask = 2.5x the forward's FLOPs
    cb = inp.dense(1, 32, 16384, 128, seed=5, causal=True, device="cuda")
    dout = inp.output_grad((1, 32, 16384, 128), seed=6, device="cuda")
    ob, lb = fa.fa_fwd(cb.q, cb.k, cb.v, cb.scale, True)
    gq, gk, gv = (torch.empty_like(cb.q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 32, 16384) // 4, dtype=torch.float32,
                     device="cuda")
    ms = _time_launches(lambda: fa.fa_bwd(cb.q, cb.k, cb.v, ob, dout, lb, cb.scale, True,
                                          gq, gk, gv, ws), 10)
    out["bwd_B1_H32_N16384_D128_causal"] = {
        "tflops": 2.5 * prefill_flops(1, 32, 16384, 128) / (ms * 1e-3) / 1e12, "ms": ms}
    # backward of the causal sliding window 4096 on the same tensors
    ow, lw = fa.fa_fwd_window(cb.q, cb.k, cb.v, 4096, cb.scale)
    ms = _time_launches(lambda: fa.fa_bwd_window(cb.q, cb.k, cb.v, ow, dout, lw, 4096, cb.scale,
                                                 gq, gk, gv, ws), 10)
    wf = 32 * 4.0 * 128 * sum(min(i + 1, 4096) for i in range(16384))
    out["bwd_window4096_B1_H32_N16384_D128"] = {"tflops": 2.5 * wf / (ms * 1e-3) / 1e12,
                                                "ms": ms}
    del cb, dout, ob, lb, gq, gk, gv, ws, ow, lw
    # backward over the packed varlen workload (65536 tokens, H=16, D=128)
    c5 = inp.config5(128, device="cuda")
    cu = c5.cu_seqlens.cuda()
    o5, l5 = fa.fa_fwd_varlen(c5.q, c5.k, c5.v, cu, c5.max_seqlen, c5.scale, True)
    d5 = inp.output_grad(tuple(c5.q.shape), seed=7, device="cuda")
    g5 = [torch.empty_like(c5.q) for _ in range(3)]
    w5 = torch.empty(fa.fa_bwd_workspace_bytes(1, 16, c5.q.shape[0]) // 4, dtype=torch.float32,
                     device="cuda")
    ms = _time_launches(lambda: fa.fa_bwd_varlen(c5.q, c5.k, c5.v, o5, d5, l5, cu, c5.max_seqlen,
                                                 c5.scale, True, *g5, w5), 10)
    vf = sum(2.0 * 16 * L * L * 128 for L in c5.meta["lens"])
    out["bwd_varlen_T65536_H16_D128_causal"] = {"tflops": 2.5 * vf / (ms * 1e-3) / 1e12,
                                                "ms": ms}
    del c5, o5, l5, d5, g5, w5
    # Welford row statistics: LayerNorm statistics of 4 x 16384 tokens at
    # hidden size 4096 (bf16, 512 MiB, larger than L2), and the split-K pair
    # on 64 rows of 2^22 fp32 values in 128 chunks
    R, C = ROWSTATS["R"], ROWSTATS["C"]
    xs = inp.stats_rows(R, C, seed=11, loc=0.5, std=1.0, row_spread=1.0, device="cuda")
    outs = [torch.empty(R, dtype=torch.float32, device="cuda") for _ in range(3)]
    ms = _time_launches(lambda: fa.fa_row_stats(xs, 1e-5, *outs), 20)
    out[f"rowstats_R{R}_C{C}_bf16"] = {"gbs": R * C * 2 / (ms * 1e-3) / 1e9, "ms": ms}
    del xs, outs
    ys = inp.stats_rows(64, 1 << 22, seed=12, loc=2.0, std=1.0, dtype=torch.float32,
                        device="cuda")

    def split():
        fa.fa_row_stats_combine(*fa.fa_row_stats_partials(ys, 128))
    ms = _time_launches(split, 20)
    out["rowstats_split_R64_C4194304_f32_S128"] = {
        "gbs": 64 * (1 << 22) * 4 / (ms * 1e-3) / 1e9, "ms": ms}
    del ys
    # prefix attention over the decode workload's caches: every prefix of
    # every sequence (K, V read once, O and LSE written for every key)
    pc = inp.decode(DECODE["B"], DECODE["H"], DECODE["D"], seed=4, num_splits=DECODE["S"],
                    device="cuda")
    cu = pc.cu_seqlens_k.cuda()
    T = pc.meta["T"]
    po = torch.empty_like(pc.k_cache)
    pl = torch.empty((DECODE["H"], T), dtype=torch.float32, device="cuda")
    ms = _time_launches(lambda: fa.fa_prefix_attention(pc.q, pc.k_cache, pc.v_cache, cu,
                                                       pc.scale, po, pl), 10)
    sb = float(T) * DECODE["H"] * DECODE["D"] * 2 * 3 + float(T) * DECODE["H"] * 4
    out["prefix_scan_B64_H32_D128_L1024-32768"] = {"gbs": sb / (ms * 1e-3) / 1e9, "ms": ms,
                                                   "bytes": sb}
    del pc, po, pl
    # few long rows (B=2, H=4, 262144 keys each): every row cut into 64
    # chunks scanned at once
    lc = inp.decode(2, 4, 128, seed=5, num_splits=64, lens=[262144, 262144], device="cuda")
    lcu = lc.cu_seqlens_k.cuda()
    ms = _time_launches(lambda: fa.fa_prefix_attention_chunked(lc.q, lc.k_cache, lc.v_cache, lcu,
                                                               64, lc.scale), 5)
    T = lc.meta["T"]
    lb = float(T) * 4 * 128 * 2 * 3 + float(T) * 4 * 4
    out["prefix_scan_chunked_B2_H4_L262144_S64"] = {"gbs": lb / (ms * 1e-3) / 1e9, "ms": ms,
                                                    "bytes": lb}
    del lc
    # paged KV decode with grouped query heads: the decode lengths, H=32 over
    # H_kv=8, pages of 64 keys
    # (4 KV chunks per sequence: B * H_kv * 4 = 2048 CTAs of 128-key tiles)
    pc = inp.paged_decode(64, 32, 8, 128, 64, seed=4, num_splits=4, device="cuda")
    tab, sl = pc.block_table.cuda(), pc.seqlens.cuda()

    def paged():
        pm, pd, po = fa.fa_decode_paged_splitkv(pc.q, pc.k_pages, pc.v_pages, tab, sl, 4,
                                                pc.scale)
        fa.fa_combine_states(pm, pd, po)
    ms = _time_launches(paged, 10)
    kvb = float(sum(pc.meta["lens"])) * 8 * 128 * 2 * 2
    out["paged_gqa_decode_B64_H32_Hkv8_page64"] = {"gbs": kvb / (ms * 1e-3) / 1e9, "ms": ms,
                                                  "kv_bytes": kvb}

    def paged16():
        pm, pd, po = fa.fa_decode_paged_splitkv(pc.q, pc.k_pages, pc.v_pages, tab, sl, 16,
                                                pc.scale)
        fa.fa_combine_states(pm, pd, po)
    ms = _time_launches(paged16, 10)
    out["paged_gqa_decode_B64_H32_Hkv8_page64_S16"] = {"gbs": kvb / (ms * 1e-3) / 1e9, "ms": ms,
                                                      "kv_bytes": kvb}
    del pc
    # the split-KV decode and its combine back to back, nothing between the
    # two launches (the combine's launch then overlaps the decode's tail)
    dc = inp.config4(device="cuda")
    dcu = dc.cu_seqlens_k.cuda()
    Dd = DECODE
    pm = torch.empty((Dd["B"], Dd["H"], Dd["S"]), dtype=torch.float32, device="cuda")
    pd = torch.empty_like(pm)
    po = torch.empty((Dd["B"], Dd["H"], Dd["S"], Dd["D"]), dtype=torch.float32, device="cuda")
    od = torch.empty((Dd["B"], Dd["H"], Dd["D"]), dtype=torch.bfloat16, device="cuda")
    lsed = torch.empty((Dd["B"], Dd["H"]), dtype=torch.float32, device="cuda")

    def dec_pair():
        fa.fa_decode_splitkv(dc.q, dc.k_cache, dc.v_cache, dcu, Dd["S"], dc.scale, pm, pd, po)
        fa.fa_combine_states(pm, pd, po, o=od, lse=lsed)
    ms = _time_launches(dec_pair, 10)
    alg = float(sum(dc.meta["lens"])) * Dd["H"] * Dd["D"] * 4 + \
        Dd["B"] * Dd["H"] * (Dd["D"] * 4 + 4)
    out["splitkv_decode_and_combine_B64_H32_D128_S16"] = {
        "ms": ms, "gbs": alg / (ms * 1e-3) / 1e9,
        "bytes": alg, "note": "K, V, q read; O, LSE written; no event between the launches"}
    del dc, pm, pd, po, od, lsed
    # A launch of this size takes less device time than a Python call, so
    # 100 launches are captured in a CUDA graph and the replays timed: the
    # device time per launch, not the host's call rate.
    c1 = inp.config1(device="cuda")
    o1 = torch.empty_like(c1.q)
    l1 = torch.empty((1, 1, 256), dtype=torch.float32, device="cuda")
    f1 = lambda: fa.fa_fwd_f32(c1.q, c1.k, c1.v, c1.scale, False, o=o1, lse=l1)
    s1 = torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        f1()
    torch.cuda.current_stream().wait_stream(s1)
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1):
        for _ in range(100):
            f1()
    ms = _time_launches(g1.replay, 10) / 100
    out["fp32_B1_H1_N256_D64"] = {"us": ms * 1e3, "timing": "CUDA graph of 100 launches",
                                  "gflops": 4.0 * 256 * 256 * 64 / (ms * 1e-3) / 1e9}
    return out


def run_gpu(args, rank, world, dist):
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()

    P = PREFILL
    pc = inp.dense(P["B"], P["H"], P["N"], P["D"], seed=3, causal=True, qk_std=3.0,
                   device="cuda")
    o = torch.empty_like(pc.q)
    lse = torch.empty((P["B"], P["H"], P["N"]), dtype=torch.float32, device=dev)
    dc = inp.config4(device="cuda")
    cu = dc.cu_seqlens_k.to(dev)
    Dd = DECODE
    pm = torch.empty((Dd["B"], Dd["H"], Dd["S"]), dtype=torch.float32, device=dev)
    pd = torch.empty_like(pm)
    po = torch.empty((Dd["B"], Dd["H"], Dd["S"], Dd["D"]), dtype=torch.float32, device=dev)
    od = torch.empty((Dd["B"], Dd["H"], Dd["D"]), dtype=torch.bfloat16, device=dev)
    lsed = torch.empty((Dd["B"], Dd["H"]), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(pc.q, pc.k, pc.v, pc.scale, True, o=o, lse=lse)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_decode_splitkv(dc.q, dc.k_cache, dc.v_cache, cu, Dd["S"], dc.scale, pm, pd, po)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_combine_states(pm, pd, po, o=od, lse=lsed)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = fa.fa_check_device_status()
    if status != fa.FA_OK:
        raise RuntimeError(f"device status after warm-up: {fa.fa_status_string(status)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(dev.index, gpu_uuid(dev)) as clk:
        clk.mark_start()
        start.record(stream)
        for s in range(args.steps):
            step(evs[s])
        end.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
    barrier(dist)
    total_ms = start.elapsed_time(end)
    t_pre = [e[0].elapsed_time(e[1]) for e in evs]
    t_dec = [e[1].elapsed_time(e[2]) for e in evs]
    t_cmb = [e[2].elapsed_time(e[3]) for e in evs]
    status = fa.fa_check_device_status()
    if status != fa.FA_OK:
        raise RuntimeError(f"device status after timing: {fa.fa_status_string(status)}")

    flops = prefill_flops(P["B"], P["H"], P["N"], P["D"])
    pre_ms = max_over_ranks(sum(t_pre), dist)
    dec_ms = max_over_ranks(sum(t_dec), dist)
    cmb_ms = max_over_ranks(sum(t_cmb), dist)
    total_ms = max_over_ranks(total_ms, dist)
    K = args.steps
    value = world * flops * K / (pre_ms * 1e-3) / 1e12

    lens = dc.meta["lens"]
    kv_bytes = float(sum(lens)) * Dd["H"] * Dd["D"] * 2 * 2
    dec_bytes = kv_bytes + Dd["B"] * Dd["H"] * Dd["D"] * 2 + \
        Dd["B"] * Dd["H"] * Dd["S"] * (Dd["D"] + 2) * 4        # q + partial states written
    cmb_bytes = Dd["B"] * Dd["H"] * (Dd["S"] * (Dd["D"] + 2) * 4 + Dd["D"] * 2 + 4)
    dec_alg = kv_bytes + Dd["B"] * Dd["H"] * (Dd["D"] * 2 * 2 + 4)  # K,V,q,O,LSE
    peaks, kind = load_peaks()
    pk_tf = float(peaks["bf16_tflops"])
    pk_bw = float(peaks["hbm_gbs"])
    achieved = flops / (pre_ms / K * 1e-3) / 1e12
    dec_gbs = dec_bytes / (dec_ms / K * 1e-3) / 1e9
    e2e_dec_gbs = world * dec_alg * K / ((dec_ms + cmb_ms) * 1e-3) / 1e9

    # End to end through the C ABI with host buffers (pinned): every step
    # copies its Q, K, V in and its O, LSE out.  Two device buffer sets let
    # step i+1's host-to-device copy (copy stream) overlap step i's kernel
    # (compute stream) and step i-1's device-to-host copy (third stream).
    e2e = None
    hq, hk, hv = (t.cpu().pin_memory() for t in (pc.q, pc.k, pc.v))
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    din = [[torch.empty_like(pc.q) for _ in range(3)] for _ in range(2)]
    dout = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    torch.cuda.synchronize()
    n_e2e = max(1, min(K, 20))
    ev_in = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_done = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_out = [torch.cuda.Event() for _ in range(n_e2e)]
    # two untimed passes of the same loop first (copy engines, pinned pages)
    for i in range(2):
        for dst, src in zip(din[i], (hq, hk, hv)):
            dst.copy_(src, non_blocking=True)
        fa.fa_fwd(*din[i], pc.scale, True, o=dout[i][0], lse=dout[i][1])
        ho[i].copy_(dout[i][0], non_blocking=True)
        hl[i].copy_(dout[i][1], non_blocking=True)
    torch.cuda.synchronize()
    barrier(dist)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])  # set b's inputs are free again
            for dst, src in zip(din[b], (hq, hk, hv)):
                dst.copy_(src, non_blocking=True)
            ev_in[i].record(s_in)
        comp.wait_event(ev_in[i])
        if i >= 2:
            comp.wait_event(ev_out[i - 2])  # set b's outputs were read back
        fa.fa_fwd(*din[b], pc.scale, True, o=dout[b][0], lse=dout[b][1])
        ev_done[i].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[i])
            ho[b].copy_(dout[b][0], non_blocking=True)
            hl[b].copy_(dout[b][1], non_blocking=True)
            ev_out[i].record(s_out)
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, dist)
    # The host link alone, for context: one step's input copy and output
    # copy, each timed by itself (after the timed region).
    h2d_b = 3 * pc.q.numel() * 2
    d2h_b = o.numel() * 2 + lse.numel() * 4

    def _copy_ms(fn, n=5):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def _h2d():
        for dst, src in zip(din[0], (hq, hk, hv)):
            dst.copy_(src, non_blocking=True)

    def _d2h():
        ho[0].copy_(dout[0][0], non_blocking=True)
        hl[0].copy_(dout[0][1], non_blocking=True)

    h2d_gbs = h2d_b / (_copy_ms(_h2d) * 1e-3) / 1e9
    d2h_gbs = d2h_b / (_copy_ms(_d2h) * 1e-3) / 1e9
    del din, dout
    e2e = {"value": world * flops * n_e2e / dt / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d_b,
           "d2h_bytes_per_step": d2h_b,
           "steps": n_e2e, "pipelined": "2 buffer sets, copies on their own streams",
           "h2d_gbs_alone": h2d_gbs, "d2h_gbs_alone": d2h_gbs}

    if rank != 0:
        return 0
    others = None if args.no_other_configs else other_configs(fa)
    cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline_leg()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (no flush)",
                   "prefill_ms": pre_ms / K, "decode_ms": dec_ms / K, "combine_ms": cmb_ms / K,
                   "parallelism": f"replicas x{world} (independent heads per GPU)"},
        "roofline": {"kernel": "fa_fwd_tc_kernel<128>", "bound": "tensor",
                     "achieved": achieved, "peak": pk_tf, "unit": "TFLOP/s",
                     "frac": achieved / pk_tf, "peak_kind": f"{kind} bf16 burst",
                     "traffic": load_traffic("fa_fwd_tc_kernel<128>",
                                             "exact_io_aware_15_gb300/csrc/fwd_tc.cu")},
        "decode": {"metric": "split-KV decode GB/s", "value": dec_gbs, "unit": "GB/s",
                   "frac": dec_gbs / pk_bw, "peak": pk_bw, "peak_kind": f"{kind} hbm copy",
                   "frac_of_nominal_8tbs": dec_gbs / 8000.0,
                   "bytes_per_launch": dec_bytes, "kv_tokens": int(sum(lens)),
                   "combine_us": cmb_ms / K * 1e3,
                   "combine_gbs": cmb_bytes / (cmb_ms / K * 1e-3) / 1e9,
                   "combine_bytes": cmb_bytes,
                   "end_to_end_gbs": e2e_dec_gbs,
                   "traffic": load_traffic("fa_decode_splitkv_kernel<128>",
                                           "exact_io_aware_15_gb300/csrc/decode.cu")},
        "cpu_baseline": cpu,
        "other_configs": others,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clk.summary(),
    }
    print(json.dumps(line))
    return 0


def run_profile_case(args):
    """Only one workload, W + K launches, nothing else: the command the ncu
    captures run.  prefill = the full causal N=16384 prefill (537 MB of
    inputs); bwd = its backward (Delta, dK/dV, dQ kernels); rowstats = the
    LayerNorm statistics of 65536 x 4096 bf16; paged = the paged GQA decode
    (B=64, H=32 over H_kv=8, pages of 64, 4.7 GB of KV); scan = prefix
    attention over the decode workload's caches; scan_small = the same on
    its first 8 sequences with every row cut into 4 chunks (about 2.2 GB of
    caches and 1.1 GB of output, 1024 CTAs); varlen64 = the packed causal
    prefill of 65536 tokens, H=16, D=64 (201 MB of inputs); decode = split-KV decode on the
    first 8 sequences of the decode workload (about 2.2 GB of KV cache, larger than L2, small enough for a
    multi-pass capture)."""
    import exact_io_aware_15_gb300 as fa
    fa.load_library()
    if args.profile_case == "prefill":
        P = PREFILL
        c = inp.dense(P["B"], P["H"], P["N"], P["D"], seed=3, causal=True, qk_std=3.0,
                      device="cuda")
        o = torch.empty_like(c.q)
        lse = torch.empty((P["B"], P["H"], P["N"]), dtype=torch.float32, device="cuda")
        run = lambda: fa.fa_fwd(c.q, c.k, c.v, c.scale, True, o=o, lse=lse)
    elif args.profile_case == "varlen64":
        c5 = inp.config5(64, device="cuda")
        cu = c5.cu_seqlens.cuda()
        run = lambda: fa.fa_fwd_varlen(c5.q, c5.k, c5.v, cu, c5.max_seqlen, c5.scale, True)
    elif args.profile_case == "bwd":
        P = PREFILL
        c = inp.dense(P["B"], P["H"], P["N"], P["D"], seed=5, causal=True, device="cuda")
        dout = inp.output_grad((P["B"], P["H"], P["N"], P["D"]), seed=6, device="cuda")
        o, lse = fa.fa_fwd(c.q, c.k, c.v, c.scale, True)
        grads = [torch.empty_like(c.q) for _ in range(3)]
        ws = torch.empty(P["B"] * P["H"] * P["N"], dtype=torch.float32, device="cuda")
        run = lambda: fa.fa_bwd(c.q, c.k, c.v, o, dout, lse, c.scale, True, *grads, ws)
    elif args.profile_case == "paged":
        pc = inp.paged_decode(64, 32, 8, 128, 64, seed=4, num_splits=4, device="cuda")
        tab, sl = pc.block_table.cuda(), pc.seqlens.cuda()
        run = lambda: fa.fa_combine_states(*fa.fa_decode_paged_splitkv(
            pc.q, pc.k_pages, pc.v_pages, tab, sl, 4, pc.scale))
    elif args.profile_case == "scan":
        pc = inp.decode(DECODE["B"], DECODE["H"], DECODE["D"], seed=4, num_splits=DECODE["S"],
                        device="cuda")
        cu = pc.cu_seqlens_k.cuda()
        po = torch.empty_like(pc.k_cache)
        pl = torch.empty((DECODE["H"], pc.meta["T"]), dtype=torch.float32, device="cuda")
        run = lambda: fa.fa_prefix_attention(pc.q, pc.k_cache, pc.v_cache, cu, pc.scale, po, pl)
    elif args.profile_case == "scan_small":
        g = torch.Generator().manual_seed(4)
        lens = torch.randint(1024, 32769, (64,), generator=g).tolist()[:8]
        pc = inp.decode(8, DECODE["H"], DECODE["D"], seed=4, num_splits=4, lens=lens,
                        device="cuda")
        cu = pc.cu_seqlens_k.cuda()
        po = torch.empty_like(pc.k_cache)
        pl = torch.empty((DECODE["H"], pc.meta["T"]), dtype=torch.float32, device="cuda")
        run = lambda: fa.fa_prefix_attention_chunked(pc.q, pc.k_cache, pc.v_cache, cu, 4,
                                                     pc.scale, po, pl)
    elif args.profile_case == "combine":
        # the state combine alone on states of the decode workload's shape
        # (B=64 x H=32 rows, 16 chunks: 17 MB), seeded, with no KV cache
        B, H, S, D = DECODE["B"], DECODE["H"], DECODE["S"], DECODE["D"]
        g = torch.Generator(device="cuda").manual_seed(13)
        pm = torch.randn((B, H, S), generator=g, device="cuda") * 20.0
        pd = torch.rand((B, H, S), generator=g, device="cuda") * 500.0 + 1.0
        po = torch.randn((B, H, S, D), generator=g, device="cuda") * 50.0
        od = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
        lsed = torch.empty((B, H), dtype=torch.float32, device="cuda")
        run = lambda: fa.fa_combine_states(pm, pd, po, o=od, lse=lsed)
    elif args.profile_case == "rowstats":
        x = inp.stats_rows(ROWSTATS["R"], ROWSTATS["C"], seed=11, loc=0.5, std=1.0,
                           row_spread=1.0, device="cuda")
        outs = [torch.empty(ROWSTATS["R"], dtype=torch.float32, device="cuda") for _ in range(3)]
        run = lambda: fa.fa_row_stats(x, 1e-5, *outs)
    else:
        g = torch.Generator().manual_seed(4)
        lens = torch.randint(1024, 32769, (64,), generator=g).tolist()[:8]
        c = inp.decode(8, DECODE["H"], DECODE["D"], seed=4, num_splits=DECODE["S"],
                       lens=lens, device="cuda")
        cu = c.cu_seqlens_k.cuda()
        run = lambda: fa.decode(c.q, c.k_cache, c.v_cache, cu, DECODE["S"], c.scale)
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize()
    rc = fa.fa_check_device_status()
    print(json.dumps({"profile_case": args.profile_case, "status": fa.fa_status_string(rc)}))
    return 0 if rc == fa.FA_OK else 1


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true")
    ap.add_argument("--profile-case", choices=["prefill", "decode", "bwd", "rowstats", "paged",
                                                "scan", "scan_small", "combine", "varlen64"],
                    default=None)
    args = ap.parse_args(argv)
    if args.profile_case:
        return run_profile_case(args)
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    rank, world, local, dist = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_gpu(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
