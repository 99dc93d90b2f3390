#!/usr/bin/env python
"""Benchmark of the AttnRes mixture on GB300 (one JSON line on stdout).

A step is one attn_res call over the whole workload (every step of the path
runs in it).  Default workload: long prefill, T=8192 tokens, 8 valid blocks
in a 9-slot bank with padded slot stride 7232, delta and output norm on,
write-back into slot 8.  Its inputs (1.53 GB touched per step) are larger
than L2, so no flush is needed between steps.

  value      tokens/s, device time (CUDA events on the launching stream),
             inputs resident in HBM, max over ranks, summed over ranks
  e2e        the same metric through the public call with pinned HOST
             buffers: every step copies its inputs host->device and reads
             out, the updated prefix and the written bank slot back; steps
             pipelined over copy-in / compute / copy-out streams
  roofline   algorithmic bytes per launch / mean launch time vs the measured
             HBM copy bandwidth
  latency_us T=1 latency (single-token and 8-block cases): per call with an
             L2 flush in between (and the floor that timing has: a
             one-element add measured the same way), back-to-back in a CUDA
             graph on one input set, and back-to-back with every call's
             rows in a different slot of a pool larger than 3x L2 (rows
             from DRAM)
  pdl_chain  graph-replayed chains of calls with and without programmatic
             dependent launch (T=1 and T=1024)
  prefill_cells  T=1024/2048 prefill cells: µs per call from CUDA-graph
             replay, cycling through input copies larger than 3x L2
  width_cells  other model widths (H = 4096, 8192) through attn_res_h and
             the general kernel, graph replay over rotating input sets
  tp_cells   one rank's kernels of the hidden-sharded (TP8) mixture, both
             exchange forms, all-reduces excluded
  cpu_baseline  the CPU oracle on a bounded sample of the same workload, on
             all host cores (and on one core: cpu_baseline_one_core)

``--impl reference`` times the CPU oracle on the same workload and metric.
Multi-GPU (torchrun): every rank runs its own copy of the workload on its own
GPU (independent token rows, no collective on the data path: weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = ("AttnRes µs/call at T=1 and tokens/s + achieved HBM GB/s "
          "(% of peak) at T=1024–8192")
FALLBACK_HBM_GBS = 6800.0


# ---- workloads ----------------------------------------------------------------

def make(name: str):
    from attention_residual_fusion_gb300 import workloads as W
    if name == "long_prefill":
        return W.long_prefill(), "long prefill T=8192, S=8, bank [8192,9,7232] padded, delta, output norm, write-back slot 8, per-block scales U(1,30)"
    if name.startswith("long_prefill:"):   # same layout, fewer tokens (profiling)
        T = int(name.split(":")[1])
        return W.long_prefill(T), f"long prefill layout at T={T}, S=8, bank [T,9,7232] padded, delta, output norm, write-back slot 8"
    if name == "single_token":
        return W.single_token(), "single token T=1, S=4, bank [1,8,7168], delta, output norm, no write-back"
    kind, *a = name.split(":")
    if kind == "prefill":          # prefill:T:S:o:w
        T, S, o, w = (int(x) for x in a)
        return W.prefill(T, S, bool(o), w), f"prefill T={T}, S={S}, delta, output norm {bool(o)}, write_idx {w}, 1% outliers x50"
    if kind == "decode":           # decode:T
        T = int(a[0])
        return W.decode_batch(T), f"decode batch T={T}, S=8, delta, output norm, per-block scales U(0.5,20)"
    if kind == "width":            # width:H:T:S -- another model width (attn_res_h)
        H, T, S = (int(x) for x in a)
        return (W.make_workload(T, S, capacity=8, has_delta=True, has_out_norm=True,
                                block_write_idx=7, seed=0, outliers=True, H=H,
                                name=f"width_H{H}_T{T}_S{S}"),
                f"hidden size H={H}, T={T}, S={S}, delta, output norm, write_idx 7, 1% outliers x50")
    if kind == "variant":          # variant:T:S:d:o:w
        T, S, d, o, w = (int(x) for x in a)
        return W.variant_cell(T, S, bool(d), bool(o), w), f"variant T={T}, S={S}, delta {bool(d)}, output norm {bool(o)}, write_idx {w}"
    raise SystemExit(f"unknown workload {name}")


# Sources the timed kernel (the stream kernel) is built from: a recorded
# DRAM-traffic figure is used only while these are unchanged and for the same
# kernel variant (template arguments).
STREAM_SOURCES = ("attn_res_common.cuh", "attn_res_token.cuh", "attn_res_stream.cuh",
                  "attn_res_row.cuh")


def source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_residual_fusion_gb300", "csrc")
    for f in STREAM_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_label(wl, shape) -> str:
    """The timed kernel with its template arguments (S, delta, norm, split,
    vectors per thread, ring depth, shared bank rows, staged)."""
    d, o = int(wl.delta is not None), int(wl.out_norm_w is not None)
    if shape["kernel"] in ("stream", "staged"):
        vpc = 896 // shape["split"]
        v = -(-vpc // shape["threads"])  # vectors per thread
        return (f"attn_res_stream_kernel<{wl.num_blocks},{d},{o},{shape['split']},{v},"
                f"{shape['stages']},{int(wl.group > 1)},{int(shape['kernel'] == 'staged')}>")
    if shape["kernel"] in ("row", "row_smem"):
        return f"attn_res_{shape['kernel']}_kernel<{wl.num_blocks},{d},{o},{896 // shape['threads']}>"
    if shape["kernel"] == "split":
        return f"attn_res_split_kernel<{wl.num_blocks},{d},{o},{shape['split']}>"
    return f"attn_res_{shape['kernel']}_kernel<{wl.num_blocks},{d},{o}>"


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source, this workload and this kernel variant."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    e = d.get(workload)
    if not e or e.get("source_digest") != source_digest() or e.get("kernel") != kernel:
        return None
    return e.get("dram_bytes_per_launch")


# ---- clocks -------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock and throttle reasons.
    `mark()` brackets the timed region; the summary uses the samples taken
    inside it, or the two nearest ones when the region is shorter than the
    sampling period."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []  # (host time, fields)
        self.window = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)  # let nvidia-smi start sampling
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        if self.proc is None:
            return None
        good = [(t, f) for t, f in self.samples if len(f) >= 10]
        if self.window is not None and good:
            t0, t1 = self.window
            inside = [(t, f) for t, f in good if t0 <= t <= t1]
            if not inside:
                mid = (t0 + t1) / 2
                inside = sorted(good, key=lambda s: abs(s[0] - mid))[:2]
            good = inside
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, f in good:
            try:
                sm.append(float(f[2]))
                mx = float(f[3])
            except ValueError:
                continue
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- CPU oracle -----------------------------------------------------------------

def oracle_rate(wl, budget_s: float, threads: int):
    """Tokens/s of the oracle on a bounded sample of the workload: the first
    n token rows, repeated passes until about budget_s of CPU time.  Also
    returns the oracle's results for those rows (the first pass)."""
    import oracle
    n = min(wl.T, max(threads, 16))
    t0 = time.perf_counter()
    oracle.run_workload(wl, n_threads=threads, tokens=np.arange(n))
    dt = time.perf_counter() - t0
    n = int(min(wl.T, max(n, n * budget_s / max(dt, 1e-6))))
    toks = np.arange(n)
    passes, t0, first = 0, time.perf_counter(), None
    while True:
        r = oracle.run_workload(wl, n_threads=threads, tokens=toks)
        first = first or r
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or passes >= 1000:
            break
    return n * passes / dt, n, passes, dt, first


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns as float64 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def compare_with_oracle(wl, gpu: dict, ref: dict) -> dict:
    """The GPU's results for the oracle's token rows against the oracle: out
    within max(2 bf16 ulp of the oracle value, 1e-2) per element, the
    updated prefix and every bank slot of those rows bit-exact."""
    idx = ref["tokens"]
    g, r = widen(gpu["out"][idx]), widen(ref["out"])
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
    tol = np.maximum(2 * ulp, 1e-2)
    ratio = np.abs(g - r) / tol
    worst = float(np.max(ratio)) if ratio.size else 0.0
    res = {"checked": True, "tokens": int(len(idx)), "max_err_over_tol": round(worst, 4),
           "out_within_tol": bool(np.all(np.isfinite(g)) and worst <= 1.0),
           "prefix_bitexact": bool(np.array_equal(gpu["prefix"][idx], ref["prefix"][:, :wl.H])),
           "bank_bitexact": bool(np.array_equal(gpu["bank"][idx], ref["bank"]))}
    res["ok"] = res["out_within_tol"] and res["prefix_bitexact"] and res["bank_bitexact"]
    return res


# ---- ranks --------------------------------------------------------------------

def combine_ranks(dist, total_ms: float, tokens_per_rank: int, device=None):
    """Whole-job throughput: the slowest rank's time, tokens summed over
    ranks (each rank runs its own replica of the workload)."""
    if dist is None:
        return total_ms, tokens_per_rank / (total_ms / 1e3)
    import torch
    x = torch.tensor([total_ms], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    tmax = float(x.item())
    return tmax, tokens_per_rank * dist.get_world_size() / (tmax / 1e3)


# ---- GPU arm ------------------------------------------------------------------

def device_tensors(wl, torch, dev):
    def up(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return dict(prefix=up(wl.prefix), delta=None if wl.delta is None else up(wl.delta),
                bank=up(wl.bank), rms=up(wl.rms_w), res=up(wl.res_w),
                onw=None if wl.out_norm_w is None else up(wl.out_norm_w),
                out=torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev))


TUNE = dict(split=0, kernel=0, stages=0, vpt=0)  # launch overrides from the command line


def call(ar, wl, t, stream, pdl=False):
    ar.attn_res(t["prefix"], t["delta"], t["bank"][:, :, : wl.H], wl.num_blocks,
                wl.block_write_idx, t["res"], t["rms"], t["onw"], wl.eps, wl.out_eps,
                t["out"], pdl=pdl, stream=stream, **TUNE)


def warm_up(ar, wl, t, torch, stream, calls, min_seconds):
    """At least `calls` calls and at least `min_seconds` of them, so the GPU
    reaches its steady clocks and memory state whatever --warmup says."""
    n, t0 = 0, time.perf_counter()
    while n < calls or time.perf_counter() - t0 < min_seconds:
        for _ in range(max(1, calls if n == 0 else 16)):
            call(ar, wl, t, stream)
            n += 1
        torch.cuda.synchronize()
    return n


def time_device(ar, wl, t, torch, stream, steps, warmup, ev=None):
    """Device time of `steps` back-to-back calls (CUDA events on the launching
    stream).  `ev`: the steps + 1 events, created beforehand so that nothing
    slow runs between the synchronize before the region and its first call."""
    ev = ev or [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    for _ in range(warmup):
        call(ar, wl, t, stream)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        # a ~0.1 ms device-side pause ahead of the region, so the host has
        # queued the first calls when it starts: the first timed call then
        # measures the device, not the host's launch latency (untimed)
        torch.cuda._sleep(200_000)
        ev[0].record(stream)
        for i in range(steps):
            call(ar, wl, t, stream)
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[steps]), per


def input_sets(wl, t, torch, dev, at_least=1):
    """The device inputs plus extra copies, so that cycling through them
    touches at least 3x the L2 size: every launch then reads from HBM (and
    at least `at_least` sets)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n = min(16, max(at_least, -(-3 * l2 // wl.algorithmic_bytes())))
    sets = [t]
    for _ in range(n - 1):
        sets.append({k: (v.clone() if v is not None and k in ("prefix", "delta", "bank", "out") else v)
                     for k, v in t.items()})
    return sets


def replay_us(g, torch, stream, calls, warm_s=0.02, replays=5):
    """µs per call of a captured graph of `calls` calls: replays for at least
    `warm_s` seconds first (an idle GPU needs a moment to reach its steady
    clocks), then the median of `replays` timed replays."""
    t0 = time.perf_counter()
    while True:
        g.replay()
        torch.cuda.synchronize()
        if time.perf_counter() - t0 >= warm_s:
            break
    per = []
    for _ in range(replays):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        per.append(a.elapsed_time(b) * 1e3 / calls)
    return statistics.median(per)


def time_graph(ar, wl, sets, torch, stream, calls=64, pdl=False):
    """Mean µs per call of `calls` back-to-back launches replayed from a CUDA
    graph (no host launch overhead), cycling through the input sets; with
    `pdl` each launch may start while the previous one finishes."""
    for st in sets:
        call(ar, wl, st, stream, pdl=pdl)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(calls):
            call(ar, wl, sets[i % len(sets)], stream, pdl=pdl)
    us = replay_us(g, torch, stream, calls)
    del g
    return us


# every prefill case of the benchmark set: T x num_blocks x output norm x write-back
SWEEP = [f"prefill:{T}:{S}:{o}:{w}" for T in (1024, 2048) for S in (0, 4, 8) for o in (1, 0)
         for w in (7, -1)]


def sweep_prefill(ar, torch, dev, stream, peak):
    """The other T >= 1024 cells (every prefill case: T, num_blocks, output
    norm, write-back): µs per call from graph replay over rotating input sets
    larger than 3x L2, without and with programmatic dependent launch
    (`pdl_*`: each call may start while the previous one drains; the input
    sets rotate, so no call reads rows the previous one writes)."""
    rows = []
    for name in SWEEP:
        wl, _ = make(name)
        t = device_tensors(wl, torch, dev)
        sets = input_sets(wl, t, torch, dev, at_least=2)
        us = time_graph(ar, wl, sets, torch, stream)
        us_pdl = time_graph(ar, wl, sets, torch, stream, pdl=True)
        gbs = wl.algorithmic_bytes() / (us * 1e-6) / 1e9
        rows.append({"workload": name, "us_per_call": round(us, 2),
                     "tokens_per_s": round(wl.T / (us * 1e-6), 1),
                     "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "pdl_us_per_call": round(us_pdl, 2),
                     "pdl_frac": round(wl.algorithmic_bytes() / (us_pdl * 1e-6) / 1e9 / peak, 4),
                     "input_sets": len(sets)})
        del t, sets
        torch.cuda.empty_cache()
    return rows


WIDTHS = ["width:4096:2048:8", "width:8192:2048:8", "width:3000:2048:8"]


def width_kernel(wl) -> str:
    """Kernel attn_res_h runs for the workload's width (the routing its
    header documents): widths up to 16384 with a row exchange take the
    any-width split (T < 80, up to 8 CTAs) or stream form with ceil(H / 1024)
    CTAs per row, every other row the general kernel."""
    exchange = wl.num_blocks > 0 or wl.out_norm_w is not None
    kc = -(-wl.H // 1024)
    if exchange and kc <= 16:
        return "any-width split" if wl.T < 80 and kc <= 8 else "any-width stream"
    return "general"


def width_cells(ar, torch, dev, stream, peak):
    """Other model widths through attn_res_h: µs per call from graph replay
    over rotating input sets larger than 3x L2."""
    rows = []
    for name in WIDTHS:
        wl, _ = make(name)
        t = device_tensors(wl, torch, dev)
        sets = input_sets(wl, t, torch, dev)
        us = time_graph(ar, wl, sets, torch, stream)
        gbs = wl.algorithmic_bytes() / (us * 1e-6) / 1e9
        rows.append({"workload": name, "kernel": width_kernel(wl), "us_per_call": round(us, 2),
                     "tokens_per_s": round(wl.T / (us * 1e-6), 1), "gbs": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "input_sets": len(sets)})
        del t, sets
        torch.cuda.empty_cache()
    return rows


def tp_cells(ar, torch, dev, stream, peak, ranks=8):
    """One rank's kernels of the hidden-sharded mixture (shard width H/8, the
    TP8 layout): µs per step from CUDA-graph replay, contiguous [T, H/8]
    shard tensors, input copies rotated over more than 3x L2.  The
    all-reduces between the kernels are not part of the number (one GPU:
    there is nothing to exchange with); `kernels` says how many launches a
    step makes.  `frac` = single-pass algorithmic bytes of the shard per
    step / time, against the measured copy bandwidth; `frac_all_passes` the
    same with the bytes of every pass (each re-reads the rows)."""
    from attention_residual_fusion_gb300 import tp
    rows = []
    for name in ("long_prefill", "single_token"):
        wl, _ = make(name)
        Hs = wl.H // ranks
        full = device_tensors(wl, torch, dev)
        shard = {k: (None if v is None else
                     (v[:, :, :Hs] if k == "bank" else v[..., :Hs]).contiguous())
                 for k, v in full.items()}
        del full
        alg = wl.algorithmic_bytes() * Hs // wl.H
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n = min(16, max(1, -(-3 * l2 // alg)))
        sets = [shard] + [{k: (v.clone() if v is not None and k in ("prefix", "delta", "bank", "out")
                               else v) for k, v in shard.items()} for _ in range(n - 1)]
        for gram, chunk in ((False, None), (True, None)):
            def step(st):
                tp.attn_res_tp(st["prefix"], st["delta"], st["bank"], wl.num_blocks,
                               wl.block_write_idx, st["res"], st["rms"], st["onw"], wl.eps,
                               wl.out_eps, st["out"], H=wl.H, all_reduce=lambda x: None,
                               gram=gram, chunk_tokens=chunk, stream=stream)
            calls = 16 if wl.T > 1 else 64
            with torch.cuda.stream(stream):
                for st in sets:
                    step(st)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(calls):
                    step(sets[i % len(sets)])
            us = replay_us(g, torch, stream, calls)
            del g
            gbs = alg / (us * 1e-6) / 1e9
            nch = -(-wl.T // chunk) if chunk else 1
            form = "single exchange (Gram)" if gram else "two exchanges"
            if chunk:
                form += f", pipelined chunks of {chunk} rows"
            # every pass reads the token's rows again; the last also writes
            passes = 2 if gram else 3
            row_reads = wl.T * (wl.num_blocks + 1 + int(wl.delta is not None)) * Hs * 2
            moved = alg + (passes - 1) * row_reads
            rows.append({"workload": f"{name} shard 1/{ranks} (H_s={Hs})", "form": form,
                         "kernels": (2 if gram else 3) * nch,
                         "all_reduces": (1 if gram else 2) * nch,
                         "us_per_step": round(us, 3), "tokens_per_s": round(wl.T / (us * 1e-6), 1),
                         "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                         "passes": passes, "bytes_all_passes": moved,
                         "frac_all_passes": round(moved / (us * 1e-6) / 1e9 / peak, 4),
                         "input_sets": len(sets)})
        del sets, shard
        torch.cuda.empty_cache()
    return rows


DECODE = ["decode:64", "decode:256"]


def decode_cells(ar, torch, dev, stream, peak):
    """The decode-batch cells (T = 64 and 256, 8 bank rows, delta, output
    norm): µs per call from graph replay over rotating input sets larger than
    3x L2, without and with programmatic dependent launch."""
    rows = []
    for name in DECODE:
        wl, _ = make(name)
        t = device_tensors(wl, torch, dev)
        sets = input_sets(wl, t, torch, dev, at_least=2)
        us = time_graph(ar, wl, sets, torch, stream)
        us_pdl = time_graph(ar, wl, sets, torch, stream, pdl=True)
        gbs = wl.algorithmic_bytes() / (us * 1e-6) / 1e9
        rows.append({"workload": name, "us_per_call": round(us, 2),
                     "tokens_per_s": round(wl.T / (us * 1e-6), 1), "gbs": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "pdl_us_per_call": round(us_pdl, 2),
                     "input_sets": len(sets)})
        del t, sets
        torch.cuda.empty_cache()
    return rows


def pdl_chain(ar, torch, dev, stream):
    """Back-to-back calls replayed from a CUDA graph, with and without
    programmatic dependent launch (each call's bank-row and weight loads may
    then overlap the previous call's tail).  Workloads without a bank
    write-back, so a call never reads, before its grid-dependency wait, data
    the previous call writes."""
    out = {}
    for name in ("single_token", "prefill:1024:8:1:-1"):
        wl, _ = make(name)
        t = device_tensors(wl, torch, dev)
        sets = input_sets(wl, t, torch, dev)
        row = {}
        for pdl in (False, True):
            for st in sets:
                call(ar, wl, st, stream, pdl=pdl)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            n = 64
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    call(ar, wl, sets[i % len(sets)], stream, pdl=pdl)
            row["pdl_us_per_call" if pdl else "us_per_call"] = round(replay_us(g, torch, stream, n), 3)
            del g
        row["input_sets"] = len(sets)
        out[name] = row
        del t, sets
        torch.cuda.empty_cache()
    return out


def latency_t1(ar, torch, dev, stream, reps=200):
    """T=1 latency: per call with L2 flushed between calls (events around each
    call); back-to-back inside a captured CUDA graph on one input set (warm
    L2); and back-to-back in a graph whose calls each take their rows from a
    different slot of a pool larger than 3x L2 (each call's rows come from
    DRAM).  `flush_floor_us` is a one-element add timed like the flushed
    calls: the floor that timing puts under any kernel that follows the
    flush (an add, not a fill: a kernel other than the flush's own measured
    ~2 µs more than a second fill)."""
    from attention_residual_fusion_gb300 import workloads as W
    res = {}
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    one = torch.zeros(1, device=dev)
    floor = []
    for _ in range(reps):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            one.add_(1.0)
            b.record(stream)
        b.synchronize()
        floor.append(a.elapsed_time(b) * 1e3)
    res["flush_floor_us"] = round(statistics.median(floor), 3)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for name, wl in (("single_token_T1_S4", W.single_token()),
                     ("T1_S8_delta_norm", W.variant_cell(1, 8, True, True, -1))):
        t = device_tensors(wl, torch, dev)
        for _ in range(10):
            call(ar, wl, t, stream)
        times = []
        for _ in range(reps):
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call(ar, wl, t, stream)
                b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
        g = torch.cuda.CUDAGraph()
        n = 100
        with torch.cuda.graph(g, stream=stream):
            for _ in range(n):
                call(ar, wl, t, stream)
        graph_us = replay_us(g, torch, stream, n)
        del g
        # a pool of P single-token slots (bank rows, prefix, delta, out), each
        # call of the graph on the next slot
        per_call = wl.algorithmic_bytes()
        P = int(-(-3 * l2 // per_call))
        pool = dict(prefix=t["prefix"].repeat(P, 1),
                    delta=None if t["delta"] is None else t["delta"].repeat(P, 1),
                    bank=t["bank"].repeat(P, 1, 1),
                    out=torch.empty((P, wl.H), dtype=torch.bfloat16, device=dev))
        slot = lambda i: dict(t, prefix=pool["prefix"][i:i + 1], bank=pool["bank"][i:i + 1],
                              delta=None if pool["delta"] is None else pool["delta"][i:i + 1],
                              out=pool["out"][i:i + 1])
        for i in range(P):
            call(ar, wl, slot(i), stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(P):
                call(ar, wl, slot(i), stream)
        cold_us = replay_us(g, torch, stream, P)
        res[name] = {"flushed_p50": round(statistics.median(times), 3),
                     "flushed_p20": round(float(np.percentile(times, 20)), 3),
                     "flushed_p80": round(float(np.percentile(times, 80)), 3),
                     "graph_per_call": round(graph_us, 3),
                     "graph_dram_per_call": round(cold_us, 3), "graph_dram_slots": P}
        del t, g, pool
    del flush
    return res


def e2e(ar, wl, torch, dev, stream, steps):
    """Through the public call with pinned host buffers: every step copies all
    of its inputs host->device, makes the call and reads out, the updated
    prefix and the written bank slot back.  Steps are pipelined over a
    copy-in stream, the compute stream and a copy-out stream with two device
    input sets, so step k+1's inputs go up while step k's results come down
    (the host link carries both directions at once)."""
    pin = lambda a: torch.from_numpy(a.view(np.int16)).pin_memory().view(torch.bfloat16)
    hp = dict(prefix=pin(wl.prefix), delta=None if wl.delta is None else pin(wl.delta),
              bank=pin(wl.bank), rms=pin(wl.rms_w), res=pin(wl.res_w),
              onw=None if wl.out_norm_w is None else pin(wl.out_norm_w))
    sets = [device_tensors(wl, torch, dev) for _ in range(2)]
    h_out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    h_pre = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    h_slot = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory() \
        if wl.block_write_idx >= 0 else None
    h2d = sum(v.numel() * 2 for v in hp.values() if v is not None)
    d2h = h_out.numel() * 2 + (h_pre.numel() * 2 if wl.delta is not None else 0) + \
        (h_slot.numel() * 2 if h_slot is not None else 0)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_call = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_in + ev_call + ev_out:
        e.record(stream)

    def step(k):
        i = k % 2
        d = sets[i]
        s_in.wait_event(ev_out[i])        # set i is free once step k-2 is read back
        with torch.cuda.stream(s_in):
            for key, v in hp.items():
                if v is not None:
                    d[key].copy_(v, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        call(ar, wl, d, stream)
        ev_call[i].record(stream)
        s_out.wait_event(ev_call[i])
        with torch.cuda.stream(s_out):
            h_out.copy_(d["out"], non_blocking=True)
            if wl.delta is not None:
                h_pre.copy_(d["prefix"], non_blocking=True)
            if h_slot is not None:
                h_slot.copy_(d["bank"][:, wl.block_write_idx, : wl.H], non_blocking=True)
            ev_out[i].record(s_out)

    step(0)
    step(1)
    torch.cuda.synchronize()
    # three windows of `steps` steps; the median window is reported (the host
    # link's rate varies from window to window on a shared machine)
    windows = []
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        w0 = time.perf_counter()
        for k in range(steps):
            step(k)
        b.record(s_out)
        torch.cuda.synchronize()
        windows.append((a.elapsed_time(b), time.perf_counter() - w0))
    ms, wall = sorted(windows)[1]
    del sets, hp
    return {"value": wl.T * steps / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": ms / steps,
            "host_wall_ms_per_step": wall * 1e3 / steps,
            "window_ms_per_step": [round(w[0] / steps, 3) for w in windows],
            "pipeline": "copy-in / compute / copy-out streams, two device input sets; "
                        "median of three windows"}


def device_info(torch, dev) -> dict:
    """Device metadata for the JSON line."""
    pr = torch.cuda.get_device_properties(dev)
    return {"name": pr.name, "cc": f"{pr.major}.{pr.minor}", "sms": pr.multi_processor_count,
            "l2_bytes": getattr(pr, "L2_cache_size", None),
            "hbm_bytes": pr.total_memory, "torch": torch.__version__,
            "cuda_runtime": torch.version.cuda}


def run_ours(args, rank, world, local_rank, dist):
    import torch
    import attention_residual_fusion_gb300 as ar
    from attention_residual_fusion_gb300 import _build

    _build.build()
    ar.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl, desc = make(args.workload)
    stream = torch.cuda.Stream(dev)
    TUNE.update(split=args.split, kernel=args.kernel, stages=args.stages, vpt=args.vpt)
    shape = ar.launch_shape(wl.T, wl.num_blocks, wl.out_norm_w is not None,
                            ar.FLAG_SPLIT(args.split) | ar.FLAG_KERNEL(args.kernel) |
                            ar.FLAG_STAGES(args.stages) | ar.FLAG_VPT(args.vpt),
                            has_delta=wl.delta is not None)

    # The CPU-baseline leg (rank 0 of a one-GPU run), before the timed region:
    # one call on fresh device buffers in the launch configuration that is
    # timed, whose results for the oracle's sample rows must match the oracle
    # (the run stops otherwise), and the oracle's own rate on that sample.
    parity, cpu, cpu1 = None, None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t = device_tensors(wl, torch, dev)
        call(ar, wl, t, stream)
        torch.cuda.synchronize()
        down = lambda x: x.cpu().view(torch.int16).numpy().view(np.uint16)
        gpu = {"out": down(t["out"]), "prefix": down(t["prefix"]), "bank": down(t["bank"])}
        del t
        torch.cuda.empty_cache()
        threads = os.cpu_count() or 1
        rate, n, passes, dt, ref = oracle_rate(wl, args.cpu_budget, threads)
        parity = compare_with_oracle(wl, gpu, ref)
        parity["sample"] = f"first {n} token rows, one call on fresh buffers before timing"
        del gpu, ref
        cpu = {"value": round(rate, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"first {n} token rows of the same workload, {passes} pass(es), {dt:.1f} s"}
        rate1, n1, passes1, dt1, _ = oracle_rate(wl, args.cpu_budget / 2, 1)
        cpu1 = {"value": round(rate1, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"first {n1} token rows of the same workload, {passes1} pass(es), {dt1:.1f} s"}
        if not parity["ok"]:
            print(json.dumps({"metric": METRIC, "error": "GPU results differ from the oracle",
                              "parity": parity}), flush=True)
            sys.exit(3)

    t = device_tensors(wl, torch, dev)
    # the clock sampler starts first: its start-up pause must not fall between
    # the warm-up and the timed region (an idle GPU drops its clocks, and the
    # first timed launch then ran at 1.7x its steady time)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local_rank) as clk:
        w0 = time.perf_counter()
        warm_calls = warm_up(ar, wl, t, torch, stream, max(args.warmup, 3), args.warmup_seconds)
        warm_s = time.perf_counter() - w0
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        w0 = time.time()
        total_ms, per = time_device(ar, wl, t, torch, stream, args.steps, 0, ev)
        clk.mark(w0, time.time())
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    tmax, value = combine_ranks(dist, total_ms, wl.T * args.steps, dev)
    mean_launch_ms = statistics.mean(per)
    alg_bytes = wl.algorithmic_bytes()
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (mean_launch_ms / 1e3) / 1e9

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "warmup_calls": warm_calls, "warmup_s": round(warm_s, 3),
        "ms_per_step": round(tmax / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic (seeded numpy, distributions of the pages' workloads)",
        "config": {"workload": desc, "T": wl.T, "num_blocks": wl.num_blocks,
                   "capacity": wl.capacity, "slot_stride": wl.slot_stride,
                   "delta": wl.delta is not None, "output_norm": wl.out_norm_w is not None,
                   "block_write_idx": wl.block_write_idx, "H": wl.H,
                   "launch": shape, "pdl": False,
                   "l2": f"inputs larger than L2 ({alg_bytes / 1e9:.2f} GB touched per step); no flush",
                   "parallelism": f"replicas x{world} (token rows independent, no collective)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)",
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "mean_launch_us": round(mean_launch_ms * 1e3, 3),
                     "launch_us_p20_p50_p80": [round(float(np.percentile(per, q)) * 1e3, 3)
                                               for q in (20, 50, 80)],
                     "first_launches_us": [round(x * 1e3, 3) for x in per[:5]],
                     "traffic": recorded_traffic(args.workload, kernel_label(wl, shape)),
                     "kernel": kernel_label(wl, shape)},
        "parity": parity if parity is not None else {"checked": False,
                                                     "why": "one-GPU rank 0 with the CPU leg only"},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "device": device_info(torch, dev),
    }
    if rank == 0 and not args.no_latency:
        line["latency_us"] = latency_t1(ar, torch, dev, stream)
    if rank == 0 and not args.no_latency:
        line["pdl_chain"] = pdl_chain(ar, torch, dev, stream)
    del t
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_sweep:
        line["prefill_cells"] = sweep_prefill(ar, torch, dev, stream, peak)
        line["decode_cells"] = decode_cells(ar, torch, dev, stream, peak)
        line["width_cells"] = width_cells(ar, torch, dev, stream, peak)
    if rank == 0 and not args.no_tp:
        line["tp_cells"] = tp_cells(ar, torch, dev, stream, peak)
    if not args.no_e2e:
        torch.cuda.empty_cache()
        e = e2e(ar, wl, torch, dev, stream, max(3, min(args.steps, args.e2e_steps)))
        if dist is not None:
            e["ms_per_step"], e["value"] = combine_ranks(dist, e["ms_per_step"], wl.T, dev)
        e["value"] = round(e["value"], 1)
        line["e2e"] = e
    if cpu is not None:
        line["cpu_baseline"] = cpu
        line["cpu_baseline_one_core"] = cpu1
    line["summary"] = summary(line, parity)
    return line


def summary(line: dict, parity) -> dict:
    """The figures the target is read from, last on the line: the parity
    check, the timed kernel's fraction of the copy peak, the T = 1 latencies
    (4 and 8 bank rows; L2 flushed before each call, p50, and back to back in
    a graph), the worst prefill cell and the decode cells."""
    out = {"parity_ok": None if parity is None else parity["ok"],
           "parity_max_err_over_tol": None if parity is None else parity["max_err_over_tol"],
           "parity_tokens": None if parity is None else parity["tokens"],
           "headline_frac": line["roofline"]["frac"]}
    lat = line.get("latency_us")
    if lat:
        out["t1_us"] = {k: {"flushed_p50": v["flushed_p50"], "graph": v["graph_per_call"],
                            "graph_dram": v["graph_dram_per_call"]}
                        for k, v in lat.items() if isinstance(v, dict)}
        out["t1_us"]["flush_floor_us"] = lat.get("flush_floor_us")
    cells = line.get("prefill_cells")
    if cells:
        worst = min(cells, key=lambda c: c["frac"])
        out["prefill_min_frac"] = worst["frac"]
        out["prefill_min_cell"] = worst["workload"]
        out["prefill_cells_below_0.75"] = sum(c["frac"] < 0.75 for c in cells)
    dec = line.get("decode_cells")
    if dec:
        out["decode_us"] = {c["workload"]: c["us_per_call"] for c in dec}
    return out


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on rank 0 only."""
    if rank != 0:
        return None
    import oracle
    wl, desc = make(args.workload)
    threads = os.cpu_count() or 1
    # one step = a bounded sample of the workload, sized so that the whole run
    # stays within a few minutes
    n = min(wl.T, max(threads, 16))
    t0 = time.perf_counter()
    oracle.run_workload(wl, n_threads=threads, tokens=np.arange(n))
    per_tok = (time.perf_counter() - t0) / n
    steps_total = args.steps + args.warmup
    n = int(min(wl.T, max(threads, args.ref_budget / max(steps_total, 1) / per_tok)))
    toks = np.arange(n)
    for _ in range(args.warmup):
        oracle.run_workload(wl, n_threads=threads, tokens=toks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run_workload(wl, n_threads=threads, tokens=toks)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "io_dtype": "bf16",
            "data": "synthetic (seeded numpy)",
            "config": {"workload": desc, "T": wl.T, "sample_tokens_per_step": n},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"first {n} token rows of the workload per step"},
            "e2e": {"value": round(value, 2), "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--warmup-seconds", type=float, default=0.3,
                    help="warm up for at least this long, whatever --warmup says")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_prefill")
    ap.add_argument("--split", type=int, default=0, help="CTAs per token row (0 = automatic)")
    ap.add_argument("--kernel", type=int, default=0, help="1 split, 2 stream (0 = automatic)")
    ap.add_argument("--stages", type=int, default=0, help="stream kernel ring depth (0 = automatic)")
    ap.add_argument("--vpt", type=int, default=0, help="16-byte vectors per thread (0 = automatic)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=60.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-latency", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the prefill T=1024/2048 cells")
    ap.add_argument("--no-tp", action="store_true", help="skip the hidden-sharded cells")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
        dist = tdist
    line = run_ours(args, rank, world, local_rank, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
