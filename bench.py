"""Benchmark of the TurboQuant KV-cache hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

A step is one fused decode-attention pass (tq_decode_attn) over the packed
turbo3 cache of a Qwen3-8B-shaped decode batch: B=8, 32 q-heads / 8 KV heads,
head_dim 128, context 32768, 3-bit codes + one fp16 norm per 32 values.  The
cache is built once by tq_quantize_kv from seeded N(0,1) fp16 K/V and is
resident in HBM when timing starts.  `value` is compressed-cache GB/s
(algorithmic bytes: every packed K/V byte of the context read once).  The
quantize kernel is timed in the same run on the Llama-3.2-1B-shaped KV
(16 layers x 8 heads x 2048 tokens x d=64, 4 outlier channels per head),
4-bit, per-vector and block-32, reported as Gvectors/s.

With --impl reference the float64 CPU oracle is timed instead, on a bounded
sample of the same workload, on this host's cores.

Multi-GPU: decode shards by (batch, KV head) with no exchange, so N ranks run
N independent replicas of the workload (weak scaling, no collective on the
data path; a barrier brackets the timed region).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused turbo3 decode-attn HBM GB/s (% of peak); KV quantize Gvectors/s"
WORKLOAD = "Qwen3-8B-shaped decode: B=8, Hq=32, Hkv=8, d=128, ctx=32768, turbo3 K/V (3-bit + fp16 norm per 32)"
DEC = dict(B=8, Hq=32, Hkv=8, d=128, ctx=32768)
TURBO3 = dict(block=32, bits=3)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM bytes (read + write) of one launch of the headline decode kernel,
# dram__bytes_read.sum + dram__bytes_write.sum from an ncu capture of the
# kernel as it is now (None once the kernel changes); not measured by this run.
DECODE_TRAFFIC_BYTES = (235.013888 + 3.719424) * 1e6


def decode_bytes(B, Hkv, ctx, d, k_bits, v_bits, k_block, v_block):
    """Algorithmic bytes of one decode pass: packed codes + fp16 scales of
    every K and V token of the context, each read once."""
    per_k = d * k_bits // 8 + 2 * (d // k_block)
    per_v = d * v_bits // 8 + 2 * (d // v_block)
    return B * Hkv * ctx * (per_k + per_v)


# ---------------------------------------------------------------- clocks
class _Nvml:
    """Just enough of NVML through ctypes to read the SM clock and the clock
    event reasons of one GPU (read-only queries)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")

    def sm_mhz(self):
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(v))   # NVML_CLOCK_SM
        return v.value

    def sm_max_mhz(self):
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(v))
        return v.value

    def reasons(self):
        v = self.ct.c_ulonglong()
        self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, self.ct.byref(v))
        return [n for bit, n in self.REASONS.items() if v.value & bit]


class ClockSampler:
    """Samples the SM clock and the clock event reasons while the timed
    region runs: NVML every ~0.2 ms from a thread (the timed region of a
    short run lasts milliseconds), and nvidia-smi every 20 ms as a second
    record.  Enter it before the warm-up; ``wait_ready`` blocks until both
    samplers have produced a first sample."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.fast = []          # (time, sm MHz, reasons)
        self.window = None
        self._stop = threading.Event()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        try:
            self.nvml = _Nvml(self.index)
            self.max_mhz = self.nvml.sm_max_mhz()
            self.fthread = threading.Thread(target=self._poll, daemon=True)
            self.fthread.start()
        except Exception:
            self.nvml = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def _poll(self):
        while not self._stop.is_set():
            self.fast.append((time.perf_counter(), self.nvml.sm_mhz(), tuple(self.nvml.reasons())))
            time.sleep(0.0002)

    def wait_ready(self, timeout=10.0):
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < timeout:
            if (self.proc is None or self.lines) and (self.nvml is None or self.fast):
                return
            time.sleep(0.01)

    def mark(self, t0, t1):
        """The timed region, in perf_counter seconds."""
        self.window = (t0, t1)

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def _in(self, t):
        return self.window is None or self.window[0] <= t <= self.window[1]

    def summary(self):
        sm, mx, reasons = [], [], set()
        src = None
        fast = [(m, r) for t, m, r in self.fast if self._in(t)]
        if fast:
            src = "nvml, ~0.2 ms period, timed region only"
            sm = [m for m, _ in fast]
            mx = [self.max_mhz]
            for _, r in fast:
                reasons.update(r)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        smi = [ln for t, ln in self.lines if self._in(t)]
        for ln in smi:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                if not fast:
                    sm.append(float(f[1]))
                    mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if smi and not fast:
            src = "nvidia-smi, 20 ms period, timed region only"
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "nvidia_smi_samples": len(smi), "source": src}


# ---------------------------------------------------------------- GPU arm
def headline_cache(tb, torch, inputs, dev):
    """The packed turbo3 cache of the Qwen3-8B-shaped decode batch, built on
    the device from the seeded fp16 K/V, and its query batch."""
    B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
    L = tb.make_layout(d, TURBO3["block"], TURBO3["bits"], 0, 0, 1)
    K = tb.PackedKV(L, (B, Hkv, ctx), device=dev)
    V = tb.PackedKV(L, (B, Hkv, ctx), device=dev)
    for b in range(B):                       # one batch row at a time bounds host memory
        kb = inputs.gaussian((Hkv, ctx, d), 1000 * 11 + b)
        vb = inputs.gaussian((Hkv, ctx, d), 1000 * 12 + b)
        for src, dst in ((kb, K), (vb, V)):
            part = tb.tq_quantize_kv(L, torch.from_numpy(src).to(dev))
            dst.codes[b].copy_(part.codes)
            dst.scales[b].copy_(part.scales)
    q = torch.from_numpy(inputs.gaussian((B, Hq, d), 10)).to(dev)
    return L, K, V, q


def _prefix(tb, C, ctx):
    """A contiguous copy of the first ctx tokens of a [B, H, S] cache."""
    B, H, _ = C.lead_shape
    P = tb.PackedKV(C.layout, (B, H, ctx), device=C.codes.device)
    P.codes.copy_(C.codes[:, :, :ctx])
    P.scales.copy_(C.scales[:, :, :ctx])
    return P


def bench_depth(tb, torch, dev, L, K, V, q, steps, warm):
    """The headline decode at growing context depth (same batch, heads and
    layout), L2 flushed before each call.  Depths up to the headline's 32768
    read prefixes of its cache; 65536 and 131072 read a cache of that length
    made by repeating it along the context (the kernel reads every byte
    either way).

    Two arms per depth: the fused decode (one tq_decode_attn call), and the
    bulk path the pages describe for the llama.cpp fork - tq_dequantize_kv
    of the whole K and V context to fp16, then dense fp16 attention (PyTorch's
    scaled_dot_product_attention, a library call used as the comparison only).
    Both report GB/s of the same compressed bytes, so the curves compare
    directly; the bulk arm also gives the dequantise kernel's own HBM
    fraction (packed bytes in + fp16 bytes out)."""
    import torch.nn.functional as F
    B, Hq, Hkv, d = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"]
    G = Hq // Hkv
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    hbm, _ = _peaks()
    res = {}
    S0 = K.lead_shape[2]
    for ctx in (2048, 8192, 32768, 65536, 131072):
        if ctx == S0:
            Kc, Vc = K, V
        elif ctx < S0:
            Kc, Vc = _prefix(tb, K, ctx), _prefix(tb, V, ctx)
        else:
            rep_n = ctx // S0
            Kc = tb.PackedKV(L, (B, Hkv, ctx), device=dev)
            Vc = tb.PackedKV(L, (B, Hkv, ctx), device=dev)
            for src, dst in ((K, Kc), (V, Vc)):
                for r in range(rep_n):
                    dst.codes[:, :, r * S0:(r + 1) * S0].copy_(src.codes)
                    dst.scales[:, :, r * S0:(r + 1) * S0].copy_(src.scales)
        ws_bytes, n_split = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        ms = _time(torch, lambda: tb.tq_decode_attn(Kc, Vc, q, ctx=ctx, workspace=ws, out=out),
                   flush, steps, warm)
        nbytes = decode_bytes(B, Hkv, ctx, d, 3, 3, 32, 32)
        # bulk arm: dequantise everything, then dense attention over fp16
        Kd = torch.empty((B, Hkv, ctx, d), dtype=torch.float16, device=dev)
        Vd = torch.empty_like(Kd)
        q4 = q.view(B, Hkv, G, d)

        def deq():
            tb.tq_dequantize_kv(Kc, torch.float16, out=Kd)
            tb.tq_dequantize_kv(Vc, torch.float16, out=Vd)

        def bulk():
            deq()
            return F.scaled_dot_product_attention(q4, Kd, Vd)

        ms_bulk = _time(torch, bulk, flush, steps, warm)
        ms_deq = _time(torch, deq, flush, steps, warm)
        deq_bytes = nbytes + 2 * Kd.numel() * 2          # packed in, fp16 K and V out
        o_bulk = bulk().reshape(B, Hq, d)
        tb.tq_decode_attn(Kc, Vc, q, ctx=ctx, workspace=ws, out=out)
        torch.cuda.synchronize()
        res[str(ctx)] = {"us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                         "n_split": n_split,
                         "bulk": {"us": round(ms_bulk * 1e3, 2), "GB/s": round(nbytes / (ms_bulk * 1e-3) / 1e9, 1),
                                  "dequantize_us": round(ms_deq * 1e3, 2),
                                  "dequantize_roofline": {"bound": "hbm",
                                                          "achieved": round(deq_bytes / (ms_deq * 1e-3) / 1e9, 1),
                                                          "peak": hbm, "unit": "GB/s",
                                                          "frac": round(deq_bytes / (ms_deq * 1e-3) / 1e9 / hbm, 4),
                                                          "bytes_per_step": deq_bytes},
                                  "max_abs_diff_vs_fused": round(float((o_bulk.float() - out.float()).abs().max()), 5)}}
        del Kd, Vd
        if Kc is not K:
            del Kc, Vc
        torch.cuda.empty_cache()
    return {"workload": "the headline decode (B=8, Hq=32, Hkv=8, d=128, turbo3) at context depth 2K-128K; "
                        "fused decode vs bulk dequantise + dense fp16 attention",
            "by_ctx": res}


def bench_window(tb, torch, inputs, dev, K, V, q, steps, warm, W=128):
    """The headline decode with an fp16 residual window of the last W tokens
    of every (batch, KV head) (tq_decode_attn_window): the packed cache plus
    W unquantised keys and values, one call per step, L2 flushed before each;
    the plain decode is timed beside it for the window's cost."""
    B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    kw = torch.from_numpy(inputs.gaussian((B, Hkv, W, d), 13)).to(dev)
    vw = torch.from_numpy(inputs.gaussian((B, Hkv, W, d), 14)).to(dev)
    ws = torch.empty(tb.tq_decode_window_workspace_bytes(B, Hq, Hkv, d, ctx, 0), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    ms_w = _time(torch, lambda: tb.tq_decode_attn_window(K, V, q, kw, vw, ctx=ctx, workspace=ws, out=out),
                 flush, steps, warm)
    ms_0 = _time(torch, lambda: tb.tq_decode_attn(K, V, q, ctx=ctx, workspace=ws, out=out), flush, steps, warm)
    nbytes = decode_bytes(B, Hkv, ctx, d, 3, 3, 32, 32) + 2 * B * Hkv * W * d * 2
    return {"workload": f"the headline decode plus an fp16 window of {W} tokens per (batch, KV head)",
            "us": round(ms_w * 1e3, 2), "GB/s": round(nbytes / (ms_w * 1e-3) / 1e9, 1),
            "bytes_per_step": nbytes, "plain_decode_us": round(ms_0 * 1e3, 2)}


def bench_k8v4(tb, torch, inputs, dev, steps, warm):
    """The headline decode batch (B=8, Hq=32, Hkv=8, d=128, ctx=32768) with
    8-bit keys and 4-bit values, block 32 ("TurboQuant From Scratch": the
    k8v4 setting), the same seeded K/V as the headline; one tq_decode_attn
    call per step (the CUDA-core split kernel), L2 flushed before each."""
    B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
    Lk = tb.make_layout(d, 32, 8, 0, 0, 1)
    Lv = tb.make_layout(d, 32, 4, 0, 0, 1)
    K = tb.PackedKV(Lk, (B, Hkv, ctx), device=dev)
    V = tb.PackedKV(Lv, (B, Hkv, ctx), device=dev)
    for b in range(B):
        kb = inputs.gaussian((Hkv, ctx, d), 1000 * 11 + b)
        vb = inputs.gaussian((Hkv, ctx, d), 1000 * 12 + b)
        for src, dst, L in ((kb, K, Lk), (vb, V, Lv)):
            part = tb.tq_quantize_kv(L, torch.from_numpy(src).to(dev))
            dst.codes[b].copy_(part.codes)
            dst.scales[b].copy_(part.scales)
    q = torch.from_numpy(inputs.gaussian((B, Hq, d), 10)).to(dev)
    ws_bytes, n_split = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    ms = _time(torch, lambda: tb.tq_decode_attn(K, V, q, ctx=ctx, workspace=ws, out=out),
               flush, steps, warm)
    nbytes = decode_bytes(B, Hkv, ctx, d, 8, 4, 32, 32)
    del K, V
    torch.cuda.empty_cache()
    return {"workload": "B=8, Hq=32, Hkv=8, d=128, ctx=32768; K 8-bit, V 4-bit, block 32 (k8v4)",
            "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes_per_step": nbytes}


def run_only(args, tb, torch, inputs, dev):
    """One workload on its own (for profiler runs): the same inputs and calls
    as the full run, `--warmup` untimed then `--steps` timed passes, one JSON
    line with the result and no contract keys."""
    res = {"only": args.only}
    if args.only == "decode":
        B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
        L, K, V, q = headline_cache(tb, torch, inputs, dev)
        ws_bytes, n_split = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, 0)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
        ms = _time(torch, lambda: tb.tq_decode_attn(K, V, q, ctx=ctx, workspace=ws, out=out),
                   flush, args.steps, args.warmup)
        nbytes = decode_bytes(B, Hkv, ctx, d, 3, 3, 32, 32)
        res.update(workload=WORKLOAD, ms=round(ms, 5), GBps=round(nbytes / (ms * 1e-3) / 1e9, 1))
    elif args.only == "quantize":
        res.update(bench_quantize(tb, torch, inputs, dev, args))
    elif args.only == "c1":
        res.update(bench_c1(tb, torch, inputs, dev, args.steps, args.warmup))
    elif args.only == "decode_depth":
        L, K, V, q = headline_cache(tb, torch, inputs, dev)
        res.update(bench_depth(tb, torch, dev, L, K, V, q, args.steps, args.warmup))
    elif args.only == "blocks":
        L, K, V, q = headline_cache(tb, torch, inputs, dev)
        res.update(bench_blocks(tb, torch, dev, K, args.steps, args.warmup))
    elif args.only == "decode_blocks":
        L, K, V, q = headline_cache(tb, torch, inputs, dev)
        res.update(bench_decode_blocks(tb, torch, dev, K, V, q, args.steps, args.warmup))
    elif args.only == "polar":
        res.update(bench_polar(tb, torch, inputs, dev, args.steps, args.warmup))
    elif args.only == "decode_k8v4":
        res.update(bench_k8v4(tb, torch, inputs, dev, args.steps, args.warmup))
    elif args.only == "decode_window":
        L, K, V, q = headline_cache(tb, torch, inputs, dev)
        res.update(bench_window(tb, torch, inputs, dev, K, V, q, args.steps, args.warmup))
    else:
        res.update(bench_extra(tb, torch, inputs, dev, args, which=args.only))
    print(json.dumps(res), flush=True)


def max_over_ranks(ms, dist=None, device="cpu"):
    """The slowest rank's mean step time: every rank passes its own and gets
    the maximum back (an all-reduce of one float; `dist` None = one rank).
    NCCL wants `device` to be the rank's GPU, gloo takes the CPU."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, nbytes_per_rank, ms_max):
    """Whole-job GB/s of `world` replicas that each read `nbytes_per_rank`
    per step, clocked by the slowest rank's step time."""
    return world * nbytes_per_rank / (ms_max * 1e-3) / 1e9


def run_gpu(args, rank, world):
    import torch
    from turboquant_kv_cache_gb300 import binding as tb
    from turboquant_kv_cache_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    if args.only:
        return run_only(args, tb, torch, inputs, dev)
    B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
    L, K, V, q = headline_cache(tb, torch, inputs, dev)
    ws_bytes, n_split = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    nbytes = decode_bytes(B, Hkv, ctx, d, 3, 3, 32, 32)
    stream = torch.cuda.current_stream()

    def step():
        # the library's own split count for this layout (the workspace is
        # sized for the largest any decode kernel picks)
        tb.tq_decode_attn(K, V, q, ctx=ctx, workspace=ws, out=out)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clocks:
        clocks.wait_ready()
        for _ in range(args.warmup):
            flush.zero_()
            step()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()                     # L2 flush between steps, outside the events
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        wall = t1 - t0
        clocks.mark(t0, t1)
    if dist:
        dist.barrier()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_max = max_over_ranks(statistics.mean(times), dist, dev)
    value = job_gbs(world, nbytes, ms_max)
    peak, peak_kind = _peaks()

    # end to end through the public API: per step, H2D of the new query and
    # the new K/V token, append-quantise, decode, D2H of the output
    e2e = e2e_decode(tb, torch, inputs, dev, K, V, L, ws, n_split, args)

    quant = bench_quantize(tb, torch, inputs, dev, args)
    c1 = bench_c1(tb, torch, inputs, dev, max(3, min(args.steps, 20)), 3)
    depth = None if args.no_extra else bench_depth(tb, torch, dev, L, K, V, q, max(3, min(args.steps, 20)), 3)
    window = None if args.no_extra else bench_window(tb, torch, inputs, dev, K, V, q, max(3, min(args.steps, 20)), 3)
    polar = None if args.no_extra else bench_polar(tb, torch, inputs, dev, max(3, min(args.steps, 20)), 3)
    blocks = None if args.no_extra else bench_blocks(tb, torch, dev, K, max(3, min(args.steps, 20)), 3)
    dblocks = None if args.no_extra else bench_decode_blocks(tb, torch, dev, K, V, q, max(3, min(args.steps, 20)), 3)
    k8v4 = None if args.no_extra else bench_k8v4(tb, torch, inputs, dev, max(3, min(args.steps, 20)), 3)
    extra = {} if args.no_extra else bench_extra(tb, torch, inputs, dev, args)
    clk = clocks.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16 x f16 -> f32",
            "data": "synthetic (seeded N(0,1) fp16 K/V/q, quantised on device)",
            "config": {"workload": WORKLOAD, "n_split": "library's choice", "algorithmic_bytes_per_step": nbytes,
                       "l2": "cache 235 MB > L2 and a 512 MB write flushes L2 between steps (outside events)",
                       "parallelism": f"replicas x{world}"},
            "percent_of_peak": round(100 * value / world / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(value / world, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(value / world / peak, 4),
                         "traffic": DECODE_TRAFFIC_BYTES,
                         "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                         "kernel": "decode_tc_kernel + decode_combine_kernel (one tq_decode_attn call, events around both)"},
            "e2e": e2e,
            "quantize": quant,
            "c1_roundtrip": c1,
            "decode_vs_depth": depth,
            "decode_with_fp16_window": window,
            "polar_codec": polar,
            "ggml_blocks": blocks,
            "decode_k8v4": k8v4,
            "decode_over_blocks": dblocks,
            "other_workloads": extra,
            "gpu_launches": args.steps * 2,
            "clocks": clk,
            "cycles_per_step_at_median_clock": (round(ms_max * 1e-3 * clk["sm_mhz"] * 1e6) if clk["sm_mhz"] else None),
            "wall_s_timed": round(wall, 4),
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def e2e_decode(tb, torch, inputs, dev, K, V, L, ws, n_split, args):
    B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
    q_h = torch.from_numpy(inputs.gaussian((B, Hq, d), 10)).pin_memory()
    kv_h = torch.from_numpy(inputs.gaussian((2, B, Hkv, d), 13)).pin_memory()
    out_h = torch.empty((B, Hq, d), dtype=torch.float16).pin_memory()
    q_d = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    kv_d = torch.empty((2, B, Hkv, d), dtype=torch.float16, device=dev)
    out_d = torch.empty_like(q_d)
    # the new token of every (b, head) is quantised straight into cache slot ctx-1
    pos = torch.full((B,), ctx - 1, dtype=torch.int32, device=dev)
    nbytes = decode_bytes(B, Hkv, ctx, d, 3, 3, 32, 32)

    def step():
        q_d.copy_(q_h, non_blocking=True)
        kv_d.copy_(kv_h, non_blocking=True)
        for i, cache in enumerate((K, V)):
            tb.tq_append_kv(cache, kv_d[i].unsqueeze(2), pos)
        tb.tq_decode_attn(K, V, q_d, ctx=ctx, workspace=ws, out=out_d)
        out_h.copy_(out_d, non_blocking=True)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    n_e2e = min(args.steps, 200)

    def timed(fn):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n_e2e

    dt_eager = timed(step)
    # the same step captured once as a CUDA graph (the library calls launch,
    # copy and allocate nothing that capture forbids) and replayed: the host
    # launch overhead of the 7 operations per step goes away
    graph_note = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
        torch.cuda.synchronize()
        dt_graph = timed(g.replay)
    except Exception as e:   # capture unsupported here: report the eager number only
        dt_graph, graph_note = None, f"graph capture failed: {type(e).__name__}"
    dt = dt_graph if dt_graph is not None else dt_eager
    res = {"value": round(nbytes / dt / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": q_h.numel() * 2 + kv_h.numel() * 2,
           "d2h_bytes_per_step": out_h.numel() * 2,
           "us_per_step": round(dt * 1e6, 2),
           "eager_value": round(nbytes / dt_eager / 1e9, 2),
           "cuda_graph": dt_graph is not None,
           "note": "per step: H2D query + new K/V token, tq_append_kv of K and V, decode, D2H output; "
                   "host clock; value = the step replayed as a CUDA graph, eager_value = issued call by call"}
    if graph_note:
        res["graph_note"] = graph_note
    return res


def bench_quantize(tb, torch, inputs, dev, args):
    """Quantise the K and V caches of a Llama-3.2-1B-shaped model step.
    Main figure: K and V stacked in one [2 x 16 layers x 8 heads x 2048, 64]
    input, one call (one launch) per step, as a fused K/V projection hands
    them over; `two_calls` is the same work as separate K and V calls (two
    launches, each paying the fixed launch cost).  Both are timed as CUDA
    graph replays (device time without the per-call host overhead, which at
    this size is as long as a kernel); *_eager is call by call."""
    w = inputs.llama1b_kv_workload()
    k = torch.from_numpy(w["k"]).to(dev)
    v = torch.from_numpy(w["v"]).to(dev)
    kv = torch.cat([k, v])
    n_vec = kv.numel() // 64
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    res = {"workload": "Llama-3.2-1B-shaped K and V: 16 layers x 8 heads x 2048 x d=64 fp16, 4 outlier channels x8",
           "vectors_per_step": n_vec, "unit": "Gvectors/s"}
    peak, _ = _peaks()

    def timed(fn):
        for _ in range(args.warmup if args.only else max(3, args.warmup)):
            flush.zero_()
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(min(args.steps, 100)):
            flush.zero_()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            times.append((s, e))
        torch.cuda.synchronize()
        return statistics.mean(s.elapsed_time(e) for s, e in times)

    def graph_ms(fn):
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            return timed(g.replay), True
        except Exception:
            return timed(fn), False

    for name, block in (("per_vector", 64), ("block32", 32)):
        L = tb.make_layout(64, block, 4, 0, 0, 1)
        okv = tb.tq_quantize_kv(L, kv)
        ok = tb.tq_quantize_kv(L, k)
        ov = tb.tq_quantize_kv(L, v)

        def stacked():
            tb.tq_quantize_kv(L, kv, out=okv)

        def two():
            tb.tq_quantize_kv(L, k, out=ok)
            tb.tq_quantize_kv(L, v, out=ov)

        ms, graphed = graph_ms(stacked)
        ms_eager = timed(stacked)
        ms2, _ = graph_ms(two)
        ms2_eager = timed(two)
        bytes_per_vec = 64 * 2 + 64 * 4 // 8 + 2 * (64 // block)
        gbs = n_vec * bytes_per_vec / (ms * 1e-3) / 1e9
        gbs2 = n_vec * bytes_per_vec / (ms2 * 1e-3) / 1e9
        # relative reconstruction error sum ||x - x~||^2 / sum ||x||^2 over K and V
        xr = tb.tq_dequantize_kv(okv, torch.float32)
        xf = kv.float()
        rel = float(((xr - xf) ** 2).sum()) / float((xf ** 2).sum())
        del xr, xf
        res[name] = {"gvec_per_s": round(n_vec / (ms * 1e-3) / 1e9, 3), "ms": round(ms, 5),
                     "ms_eager": round(ms_eager, 5), "cuda_graph": graphed, "launches_per_step": 1,
                     "relative_sq_error": round(rel, 5),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(gbs / peak, 4), "bytes_per_vector": bytes_per_vec},
                     "two_calls": {"ms": round(ms2, 5), "ms_eager": round(ms2_eager, 5), "launches_per_step": 2,
                                   "achieved_gbs": round(gbs2, 1), "frac": round(gbs2 / peak, 4)}}
    return res


def bench_c1(tb, torch, inputs, dev, steps, warm):
    """4096 random unit vectors of d=128 in fp32, 3-bit Lloyd-Max codes,
    one norm per vector (sign seed 1): quantise -> dequantise round trip
    on the GPU, its time and its mean squared error next to the pages'
    0.034 ("turboquant-pytorch" MSE table, 3 bits) and the Lloyd-Max
    distortion of N(0, 1/d) at 3 bits.  2.1 MB in: a launch-bound size."""
    from oracle import tq_oracle as O
    w = inputs.unit_roundtrip_workload()
    x = torch.from_numpy(w["x"]).to(dev)
    L = tb.make_layout(128, 128, 3, 0, 0, 1)
    pk = tb.tq_quantize_kv(L, x)
    xr = torch.empty_like(x)

    def rt():
        tb.tq_quantize_kv(L, x, out=pk)
        tb.tq_dequantize_kv(pk, torch.float32, out=xr)

    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    ms = _time(torch, rt, flush, steps, warm)
    rt()
    mse = float(((xr - x) ** 2).sum(dim=1).mean())
    return {"workload": "4096 unit vectors, d=128, fp32, 3-bit, one norm per vector (quantise + dequantise)",
            "us": round(ms * 1e3, 2), "mse": round(mse, 5), "pages_mse_3bit": 0.034,
            "lloyd_max_distortion_3bit": round(O.relative_distortion(3), 5),
            "bound": "launch (2.1 MB in, 0.2 MB packed)"}


def bench_blocks(tb, torch, dev, K, steps, warm):
    """GGML-style blocks of the headline K cache (turbo3: 14-byte blocks of
    32 values): tq_to_blocks and back, L2 flushed before each."""
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    peak, _ = _peaks()
    blocks = tb.tq_to_blocks(K)
    nbytes = 2 * K.nbytes()                     # read the packed cache, write the same bytes as blocks
    ms_to = _time(torch, lambda: tb.tq_to_blocks(K), flush, steps, warm)
    ms_from = _time(torch, lambda: tb.tq_from_blocks(K.layout, blocks), flush, steps, warm)
    res = {"workload": "the headline K cache (8 x 8 x 32768 turbo3 vectors of d=128) to 14-byte blocks and back"}
    for name, ms in (("to_blocks", ms_to), ("from_blocks", ms_from)):
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak,
                                                      "unit": "GB/s", "frac": round(gbs / peak, 4)}}
    return res


def bench_decode_blocks(tb, torch, dev, K, V, q, steps, warm):
    """The headline decode read straight from the block form of its K and V
    caches (14-byte turbo3 blocks, tq_decode_attn_blocks), L2 flushed before
    each call; the packed-layout call is timed beside it."""
    B, Hq, Hkv, d, ctx = DEC["B"], DEC["Hq"], DEC["Hkv"], DEC["d"], DEC["ctx"]
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    kb, vb = tb.tq_to_blocks(K), tb.tq_to_blocks(V)
    ws_bytes, n_split = tb.tq_decode_workspace_bytes(B, Hq, Hkv, d, ctx, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    ms = _time(torch, lambda: tb.tq_decode_attn_blocks(K.layout, kb, V.layout, vb, q, ctx=ctx, workspace=ws,
                                                       out=out), flush, steps, warm)
    ms_packed = _time(torch, lambda: tb.tq_decode_attn(K, V, q, ctx=ctx, workspace=ws, out=out),
                      flush, steps, warm)
    nbytes = kb.numel() + vb.numel()
    del kb, vb
    return {"workload": "the headline decode (B=8, Hq=32, Hkv=8, d=128, ctx=32768, turbo3) over 14-byte blocks",
            "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes_per_step": nbytes,
            "packed_layout_us": round(ms_packed * 1e3, 2)}


def bench_polar(tb, torch, inputs, dev, steps, warm):
    """The recursive polar-angle quantizer on the Llama-3.2-1B-shaped K and V
    (d = 64, 3-bit angles): quantise and dequantise (fp16 out) of all
    vectors per step, L2 flushed before each."""
    w = inputs.llama1b_kv_workload()
    x = torch.cat([torch.from_numpy(w["k"]).reshape(-1, 64), torch.from_numpy(w["v"]).reshape(-1, 64)]).to(dev)
    n = x.shape[0]
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    peak, _ = _peaks()
    bits = 3
    codes, radius = tb.tq_polar_quantize(x, bits)
    out = torch.empty_like(x)
    ms_q = _time(torch, lambda: tb.tq_polar_quantize(x, bits), flush, steps, warm)
    ms_d = _time(torch, lambda: tb.tq_polar_dequantize(codes, radius, 64, bits, out=out), flush, steps, warm)
    bq = 64 * 2 + 64 * bits // 8 + 2        # fp16 in; angle codes and fp16 radius out
    res = {"workload": "Llama-3.2-1B-shaped K and V (524,288 vectors of d=64), 3-bit angles", "vectors": n}
    for name, ms in (("quantize", ms_q), ("dequantize", ms_d)):
        gbs = n * bq / (ms * 1e-3) / 1e9
        res[name] = {"ms": round(ms, 4), "gvec_per_s": round(n / (ms * 1e-3) / 1e9, 3),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(gbs / peak, 4), "bytes_per_vector": bq}}
    return res


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured bf16_tflops (burst, cuBLAS); fp16 dense rate taken equal"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s"


def _time(torch, fn, flush, steps, warmup):
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        ts.append((s, e))
    torch.cuda.synchronize()
    return statistics.mean(s.elapsed_time(e) for s, e in ts)


def _cache_from(tb, torch, L, x_np, dev, S=None):
    """Packed cache of x [B, H, T, d] (numpy fp16), quantised on the device
    one (batch, head) at a time."""
    B, H, T, d = x_np.shape
    pk = tb.PackedKV(L, (B, H, T), device=dev, S=S)
    for b in range(B):
        for h in range(H):
            part = tb.tq_quantize_kv(L, torch.from_numpy(x_np[b, h]).to(dev), S=S)
            pk.codes[b, h].copy_(part.codes)
            pk.scales[b, h].copy_(part.scales)
            if pk.qjl is not None:
                pk.qjl[b, h].copy_(part.qjl)
                pk.rnorm[b, h].copy_(part.rnorm)
    return pk


def bench_extra(tb, torch, inputs, dev, args, which=None):
    """The other workloads of the path, each timed on its own (CUDA events,
    L2 flushed before every step): head_dim 256 / 131072-context decode and
    512-query causal prefill (turbo4 K, turbo3 V, Student-t keys), and the
    QJL-key decode (2-bit + 1-bit QJL keys, 3-bit values, 16384 context)."""
    out = {}
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    hbm, _ = _peaks()
    tflops, tsrc = _peak_tflops()
    steps = max(2, min(args.steps, 5))
    warm = 2
    if which:
        steps, warm = args.steps, args.warmup
    if which in (None, "decode_d256", "prefill"):
        out.update(_extra_d256(tb, torch, inputs, dev, flush, hbm, tflops, tsrc, steps, warm, which))
    if which in (None, "decode_qjl"):
        out.update(_extra_qjl(tb, torch, inputs, dev, flush, hbm, steps, warm))
    if which in (None, "quantize_qjl"):
        out.update(_extra_qjl_quantize(tb, torch, inputs, dev, flush, hbm, steps, warm))
    return out


def _extra_qjl_quantize(tb, torch, inputs, dev, flush, hbm, steps, warm):
    """Quantise the QJL-key workload's keys (B=4 x 8 KV heads x 16384 tokens,
    d=128, 2-bit + QJL m=128): one call over all 524,288 vectors."""
    w = inputs.qjl_decode_workload()
    S = torch.from_numpy(w["S"]).to(dev)
    L = tb.make_layout(128, 128, 2, 128, 0, 1)
    k = torch.from_numpy(w["k"]).to(dev).reshape(-1, 128)
    n = k.shape[0]
    o = tb.tq_quantize_kv(L, k, S=S)
    ms = _time(torch, lambda: tb.tq_quantize_kv(L, k, S=S, out=o), flush, steps, warm)
    nbytes = n * (128 * 2 + 128 * 2 // 8 + 2 + 128 // 8 + 2)   # fp16 in; codes, norm, bits, rho out
    gfma = n * 128 * 128 / 1e9
    return {"quantize_qjl_keys_524288": {
        "workload": "524,288 keys of d=128 (4 x 8 heads x 16384 tokens), 2-bit + QJL m=128, one norm per vector",
        "ms": round(ms, 4), "Gvec/s": round(n / (ms * 1e-3) / 1e9, 3),
        "projection_GFMA_per_s": round(gfma / (ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                     "bytes_per_vector": nbytes // n}}}


def _extra_d256(tb, torch, inputs, dev, flush, hbm, tflops, tsrc, steps, warm, which):
    out = {}
    # head_dim 256, 131072 context
    w = inputs.d256_longctx_workload()
    Lk = tb.make_layout(256, 32, 4, 0, 0, 1)
    Lv = tb.make_layout(256, 32, 3, 0, 0, 1)
    K = _cache_from(tb, torch, Lk, w["k"], dev)
    V = _cache_from(tb, torch, Lv, w["v"], dev)
    del w["k"], w["v"]
    q = torch.from_numpy(w["q"]).to(dev)
    ctx = 131072
    if which != "prefill":
        ms = _time(torch, lambda: tb.tq_decode_attn(K, V, q, ctx=ctx), flush, steps, warm)
        nbytes = K.nbytes() + V.nbytes()
        out["decode_d256_ctx131072"] = {
            "workload": "B=1, Hq=16, Hkv=4, d=256, ctx=131072, turbo4 K (Student-t nu=4) / turbo3 V",
            "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "roofline": {"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4)}}
    if which == "decode_d256":
        return out
    qp = torch.from_numpy(w["q_prefill"]).to(dev)
    Tq = qp.shape[2]
    ms = _time(torch, lambda: tb.tq_prefill_attn(K, V, qp, ctx, causal=True), flush,
               steps if which else 2, warm if which else 1)
    pairs = Tq * (ctx - Tq) + Tq * (Tq + 1) // 2       # causal (query, key) pairs per q-head
    flop = 4.0 * 256 * pairs * 16                       # QK^T + PV, 16 q-heads
    tf = flop / (ms * 1e-3) / 1e12
    out["prefill_d256_q512_ctx131072"] = {
        "workload": "B=1, Hq=16, Hkv=4, d=256, 512 causal queries at 130560..131071 over 131072 context",
        "ms": round(ms, 3), "TFLOP/s": round(tf, 1),
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": tflops, "unit": "TFLOP/s",
                     "frac": round(tf / tflops, 4), "peak_source": tsrc, "flop_per_step": flop}}
    del K, V
    torch.cuda.empty_cache()
    return out


def _extra_qjl(tb, torch, inputs, dev, flush, hbm, steps, warm):
    out = {}
    # QJL keys
    w = inputs.qjl_decode_workload()
    S = torch.from_numpy(w["S"]).to(dev)
    Lk = tb.make_layout(128, 128, 2, 128, 0, 1)
    Lv = tb.make_layout(128, 128, 3, 0, 0, 1)
    K = _cache_from(tb, torch, Lk, w["k"], dev, S=S)
    V = _cache_from(tb, torch, Lv, w["v"], dev)
    q = torch.from_numpy(w["q"]).to(dev)
    ms = _time(torch, lambda: tb.tq_decode_attn(K, V, q, ctx=16384), flush, steps, warm)
    nbytes = K.nbytes() + V.nbytes()
    out["decode_qjl_keys_ctx16384"] = {
        "workload": "B=4, Hq=32, Hkv=8, d=128, ctx=16384; K 2-bit + QJL m=128, V 3-bit, one norm per vector",
        "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4)}}
    # QJL on the values too (2-bit + QJL m=128 for K and V, each its own S)
    del V
    Sv = torch.from_numpy(inputs.qjl_matrix(128, 128, 8)).to(dev)
    V2 = _cache_from(tb, torch, Lk, w["v"], dev, S=Sv)
    ms = _time(torch, lambda: tb.tq_decode_attn(K, V2, q, ctx=16384), flush, steps, warm)
    nbytes = K.nbytes() + V2.nbytes()
    out["decode_qjl_keys_values_ctx16384"] = {
        "workload": "B=4, Hq=32, Hkv=8, d=128, ctx=16384; K and V 2-bit + QJL m=128, one norm per vector",
        "ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(nbytes / (ms * 1e-3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4)}}
    return out


# ---------------------------------------------------------------- CPU oracle
def _oracle_slice_inputs(b, kvh):
    """Oracle-encoded packed K/V of one (batch, KV head) of the decode
    workload (untimed) and its query group."""
    from oracle import tq_oracle as O
    from turboquant_kv_cache_gb300 import inputs
    d, ctx, Hq, Hkv = DEC["d"], DEC["ctx"], DEC["Hq"], DEC["Hkv"]
    L = O.Layout(d, TURBO3["block"], TURBO3["bits"], 0, 0, 1)
    k = inputs.gaussian((Hkv, ctx, d), 1000 * 11 + b)[kvh]
    v = inputs.gaussian((Hkv, ctx, d), 1000 * 12 + b)[kvh]
    q = inputs.gaussian((DEC["B"], Hq, d), 10)[b]
    g = Hq // Hkv
    return L, O.encode(k, L), O.encode(v, L), q[kvh * g:(kvh + 1) * g]


def oracle_decode_slice(L, kenc, venc, qg):
    from oracle import tq_oracle as O
    kd = O.dequantize(kenc[0], kenc[1], L)
    vd = O.dequantize(venc[0], venc[1], L)
    return O.decode_attention(qg[None], kd[None, None], vd[None, None])


def _threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def cpu_baseline(budget_s=12.0):
    """Times the oracle (as it stands) on this host: dequantise + attend the
    (batch 0, KV head 0) slice of the decode workload repeatedly until the
    budget is spent (the slice is encoded once, untimed)."""
    per_slice = decode_bytes(1, 1, DEC["ctx"], DEC["d"], 3, 3, 32, 32)
    L, ke, ve, qg = _oracle_slice_inputs(0, 0)
    done, elapsed = 0, 0.0
    while elapsed < budget_s or done == 0:
        t0 = time.perf_counter()
        oracle_decode_slice(L, ke, ve, qg)
        elapsed += time.perf_counter() - t0
        done += 1
    return {"value": round(done * per_slice / elapsed / 1e9, 5), "unit": "GB/s", "cores": _threads(),
            "kind": "oracle",
            "sample": f"{done} passes over one (batch, KV head) slice of the decode workload (32768 tokens: "
                      f"float64 dequantise of K and V + attention of its 4 q-heads), {elapsed:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    steps = []
    line_cpu = None
    per_slice = decode_bytes(1, 1, DEC["ctx"], DEC["d"], 3, 3, 32, 32)
    L, ke, ve, qg = _oracle_slice_inputs(0, 0)
    for _ in range(args.warmup):
        oracle_decode_slice(L, ke, ve, qg)
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_decode_slice(L, ke, ve, qg)
        steps.append(time.perf_counter() - t0)
    sec = statistics.mean(steps)
    value = per_slice / sec / 1e9
    line_cpu = {"value": round(value, 5), "unit": "GB/s", "cores": _threads(), "kind": "oracle",
                "sample": "one (batch, KV head) slice per step: 32768 tokens, float64 dequantise of K and V + "
                          "attention of its 4 q-heads"}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) fp16 K/V/q)",
        "config": {"workload": WORKLOAD, "sample": line_cpu["sample"]},
        "cpu_baseline": line_cpu,
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads (headline only)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--only", default=None,
                    choices=["decode", "quantize", "c1", "prefill", "decode_d256", "decode_qjl", "quantize_qjl", "decode_depth",
                             "decode_window", "polar", "blocks", "decode_k8v4",
                             "decode_blocks"],
                    help="time one workload alone and print its result only (profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world)


if __name__ == "__main__":
    main()
