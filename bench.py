"""Benchmark of the OSCAR mixed-precision INT2 KV-cache decode step on GB300.

A step is one decode token for every layer of the workload: for each layer,
append the new K/V (demoting the oldest recent token into the INT2 history)
and run decode attention over the BF16 sink | INT2 history | BF16 recent pool.
The metric is KV tokens/s = sum over layers of the sequence lengths attended,
divided by the step time, plus achieved HBM GB/s of the dominant kernel (the
INT2 history kernel) against the measured peak.

Workloads (synthetic, seeded; Qwen3-shaped random data, no model weights):
  qwen3_8b_36l  (default) 36 layers x (32 q / 8 kv heads, d=128), batch 1,
                102,400-token context (64 sink + 102,080 history + 256 recent)
  qwen3_4b_b32  36 layers, batch 32 x 102,400 tokens sharing a 92,160-token prefix
  qwen3_4b_b32_l1   1 layer of qwen3_4b_b32, for profiler captures
  qwen3_4b_b32_l4   4 layers of qwen3_4b_b32: the default run's bounded config-4 leg (key "config4")
  qwen3_8b_l1   1 layer, batch 1, 32,768 tokens
  qwen3_8b_100k_l1  1 layer of qwen3_8b_36l (the same decode launch), for profiler captures
  qwen3_32b_mixed   1 layer x (64 q / 8 kv heads), batch 8, lengths ~ U[98,304, 131,072]: one timed bulk
                    prefill of all requests, then decode steps (append + demotion + decode)
  qwen3_32b_mixed_b2  the same shapes, batch 2, lengths ~ U[30,000, 34,000], for profiler captures

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica (weak scaling).
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
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV tokens/s and achieved HBM GB/s vs GB300 peak, 100K ctx"
ALGO_NAMES = {0: "simt", 1: "mma", 2: "tc"}
DECODE_KERNEL_NAMES = {0: "k_int2_simt (INT2 history)", 1: "k_decode_mma (fused INT2 history + BF16 pages, mma.sync)",
                       2: "k_decode_tc (INT2 history on tcgen05 + BF16 pages)"}
UNIT = "KV tokens/s"
HIST_BYTES = 80          # per history token per kv head: 32 B K codes + 32 B V codes + 16 B fp16 scale/zero
HIST_BYTES_BY_META = {"f16": 80, "u8": 72, "cb": 80}   # the compact format stores 8 B of (mn8, mx8) per token
STORAGE = {"f16": "int2 history (fp16 scale/zero per 64-group) + bf16 sink/recent",
           "u8": "int2 history (8-bit min/max grid indices per 64-group, 2.25 bits per element) + bf16 sink/recent",
           "cb": "int2 history (Lloyd-Max 4-level codebook per kv head, fp16 range/zero per 64-group) + bf16 "
                 "sink/recent"}
META_FORMATS = {"f16": 0, "u8": 1, "cb": 2}
PREFILL_REPS = 3       # timed bulk prefill calls per layer (averaged)
BF16_BYTES = 512         # per BF16 token per kv head: K and V, 128 x 2 B each

WORKLOADS = {
    "qwen3_8b_36l": dict(layers=36, hq=32, hkv=8, batch=1, ctx=102400, shared=0),
    "qwen3_4b_b32": dict(layers=36, hq=32, hkv=8, batch=32, ctx=102400, shared=92160),
    "qwen3_4b_b32_l1": dict(layers=1, hq=32, hkv=8, batch=32, ctx=102400, shared=92160),
    "qwen3_4b_b32_l4": dict(layers=4, hq=32, hkv=8, batch=32, ctx=102400, shared=92160),
    "qwen3_8b_l1": dict(layers=1, hq=32, hkv=8, batch=1, ctx=32768, shared=0),
    "qwen3_8b_100k_l1": dict(layers=1, hq=32, hkv=8, batch=1, ctx=102400, shared=0),
    # ctx as (lo, hi): per-request lengths drawn uniformly, all requests prefilled by one bulk call
    "qwen3_32b_mixed": dict(layers=1, hq=64, hkv=8, batch=8, ctx=(98304, 131072), shared=0, d_model=5120),
    # the same shapes at a size an ncu capture of the prefill handles (about 0.3 GB of bf16 K and V)
    "qwen3_32b_mixed_b2": dict(layers=1, hq=64, hkv=8, batch=2, ctx=(30000, 34000), shared=0),
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor throughput (TFLOP/s): the measured burst figure, else the recipe's fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running (the first sample is taken
    before the block starts)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu, self.proc, self.lines = gpu, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t_end = time.time() + 3.0
            while not self.lines and time.time() < t_end and self.proc.poll() is None:
                time.sleep(0.01)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def mark(self):
        """Samples from here on describe the timed region (earlier ones only prove the sampler runs)."""
        self.start = len(self.lines)

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        lines = self.lines[getattr(self, "start", 0):] or self.lines[-1:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# workload construction


def build_workload(name: str, seed: int, device, with_bf16: bool = True, steps_capacity: int = 64, algo: int = 1,
                   meta: str = "f16", v_explicit: bool = False):
    import torch
    import bit_kv_cache_decode_gb300 as osc
    import synth

    w = WORKLOADS[name]
    B, H, hq, nl, shared = w["batch"], w["hkv"], w["hq"], w["layers"], w["shared"]
    mixed = isinstance(w["ctx"], tuple)
    lens = (synth.seq_lens_uniform(seed, B, *w["ctx"]) if mixed else np.full(B, w["ctx"])).astype(np.int64)
    L = int(lens.max())
    Lmax = L + steps_capacity
    n_hist_max = (Lmax - 320 + 63) // 64
    # page tables: shared prefix pages first (sink page + history pages covering the prefix), then private pages
    shp = (shared - 64) // 64 if shared else 0
    priv = n_hist_max - shp
    n_int2 = shp + B * priv
    n_bf16 = (1 + 4 * B) if shared else 5 * B
    hist_pt = np.zeros((B, n_hist_max), np.int32)
    bf16_pt = np.zeros((B, 5), np.int32)
    for r in range(B):
        hist_pt[r, :shp] = np.arange(shp)
        hist_pt[r, shp:] = shp + r * priv + np.arange(priv)
        if shared:
            bf16_pt[r, 0] = 0
            bf16_pt[r, 1:] = 1 + 4 * r + np.arange(4)
        else:
            bf16_pt[r] = 5 * r + np.arange(5)
    cfg = osc.CacheConfig(num_layers=nl, num_kv_heads=H, num_q_heads=hq, num_int2_pages=n_int2,
                          num_bf16_pages=n_bf16, max_batch=B, max_splits=512,
                          v_mode=osc.V_EXPLICIT if v_explicit else osc.V_ABSORBED,
                          meta_format=META_FORMATS[meta])
    cache = osc.OscarCache(cfg, device=device)
    cache.set_decode_algo(algo)
    # offline calibration on the host (library routine), one per (layer, kv head)
    sm = synth.sm_scale()

    def cal(lh):
        layer, h = lh
        qc, kc, vc = synth.calibration(seed, layer, h)
        c = osc.calibrate(qc, kc, vc, sm)
        if meta == "cb":
            c["kc"], c["vc"] = kc, vc
        return c

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 8) as ex:
        cals = list(ex.map(cal, [(l, h) for l in range(nl) for h in range(H)]))
    gen = torch.Generator(device=device)
    bf16_pages = None
    if with_bf16:
        npg = (Lmax + 63) // 64
        bf16_pages = torch.empty((nl, B * npg if not shared else (shared // 64 + B * (npg - shared // 64)), H, 2, 64,
                                  128), dtype=torch.bfloat16, device=device)
        bpt = np.zeros((B, npg), np.int32)
        sp = shared // 64
        for r in range(B):
            bpt[r, :sp] = np.arange(sp)
            bpt[r, sp:] = sp + r * (npg - sp) + np.arange(npg - sp)
    hp_d = torch.from_numpy(hist_pt).to(device)
    bp_d = torch.from_numpy(bf16_pt).to(device)
    prefill = {"ms": 0.0, "tokens": 0}
    fused = {"ms": 0.0, "tokens": 0, "d_model": w.get("d_model", 0)}
    for layer in range(nl):
        cs = cals[layer * H:(layer + 1) * H]
        cache.set_rotation(layer, np.stack([c["U_K"] for c in cs]), np.stack([c["U_V"] for c in cs]),
                           np.stack([c["tau_K"] for c in cs]), np.stack([c["tau_V"] for c in cs]))
        if meta == "cb":
            # Lloyd-Max codebooks from the calibration rows: keys rotated by the library, V as stored
            # (V-absorbed layout)
            kcal = torch.from_numpy(np.stack([c["kc"] for c in cs], axis=1)).to(device).to(torch.bfloat16)
            krot = cache.rotate(layer, osc.KIND_K, kcal).cpu().numpy()
            for h in range(H):
                cs[h]["cb_k"] = osc.calibrate_codebook(krot[:, h], cs[h]["tau_K"])
                cs[h]["cb_v"] = osc.calibrate_codebook(cs[h]["vc"], cs[h]["tau_V"])
            cache.set_codebook(layer, np.stack([c["cb_k"] for c in cs]), np.stack([c["cb_v"] for c in cs]))
        outl = np.stack([synth.head_stats(seed, layer, h).outliers for h in range(H)])
        gen.manual_seed(seed * 1000003 + layer)
        if mixed and fused["d_model"]:
            # the fused projection + write path from synthetic hidden states (timed like the bulk prefill;
            # the bulk prefill below then rewrites the pool with the workload's own K and V)
            tot, dm = int(lens.sum()), fused["d_model"]
            cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(device)
            x = torch.randn(tot, dm, generator=gen, device=device).to(torch.bfloat16)
            wk = (torch.randn(H * 128, dm, generator=gen, device=device) * dm ** -0.5).to(torch.bfloat16)
            wv = (torch.randn(H * 128, dm, generator=gen, device=device) * dm ** -0.5).to(torch.bfloat16)
            cache.project_quantize_prefill(layer, x, wk, wv, cu, hp_d, bp_d, total_tokens=tot)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(PREFILL_REPS):
                cache.project_quantize_prefill(layer, x, wk, wv, cu, hp_d, bp_d, total_tokens=tot)
            e1.record()
            torch.cuda.synchronize()
            fused["ms"] += e0.elapsed_time(e1) / PREFILL_REPS
            fused["tokens"] += tot
            del x, wk, wv
            gen.manual_seed(seed * 1000003 + layer)
        if mixed:
            # all requests in one bulk prefill call, timed: its throughput is this workload's write-path figure
            tot = int(lens.sum())
            k, v = synth.torch_kv_tokens(tot, H, outl, gen, device)
            cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(device)
            # one untimed call (module loading, first touch of the pool), then PREFILL_REPS timed calls
            # that rewrite the same pool bytes; the inputs (bf16 K and V) are far larger than L2
            cache.quantize_prefill(layer, k, v, cu, hp_d, bp_d, total_tokens=tot)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(PREFILL_REPS):
                cache.quantize_prefill(layer, k, v, cu, hp_d, bp_d, total_tokens=tot)
            e1.record()
            torch.cuda.synchronize()
            prefill["ms"] += e0.elapsed_time(e1) / PREFILL_REPS
            prefill["tokens"] += tot
            del k, v
            continue
        if shared:
            kp, vp = synth.torch_kv_tokens(shared, H, outl, gen, device)
        for r in range(B):
            n_priv = L - shared
            k, v = synth.torch_kv_tokens(n_priv, H, outl, gen, device)
            if shared:
                k, v = torch.cat([kp, k]), torch.cat([vp, v])
            cu = torch.tensor([0, L], dtype=torch.int32, device=device)
            cache.quantize_prefill(layer, k, v, cu, hp_d[r:r + 1], bp_d[r:r + 1], total_tokens=L)
            if with_bf16:
                pages = torch.from_numpy(bpt[r, :(L + 63) // 64]).to(device).long()
                kk = torch.zeros(((L + 63) // 64) * 64, H, 128, dtype=torch.bfloat16, device=device)
                vv = torch.zeros_like(kk)
                kk[:L], vv[:L] = k, v
                bf16_pages[layer, pages, :, 0] = kk.view(-1, 64, H, 128).transpose(1, 2)
                bf16_pages[layer, pages, :, 1] = vv.view(-1, 64, H, 128).transpose(1, 2)
            del k, v
        torch.cuda.synchronize()
    if cache.get_status() != 0:
        raise RuntimeError("device status error while building the workload")
    return dict(cache=cache, cfg=cfg, hist_pt=hp_d, bf16_pt=bp_d, L=L, lens=lens, prefill=prefill, fused=fused, B=B,
                H=H, hq=hq,
                layers=nl,
                bf16_pages=bf16_pages, base_pt=(torch.from_numpy(bpt).to(device) if with_bf16 else None),
                hist_np=hist_pt, bf16_np=bf16_pt, cals=cals, shared=shared, shp=shp)


def step_inputs(wl, steps: int, device, seed: int):
    """New-token K/V and queries for `steps` steps x layers, drawn on the device."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed + 7)
    nl, B, H, hq = wl["layers"], wl["B"], wl["H"], wl["hq"]
    kv = torch.randn(steps, nl, 2, B, H, 128, generator=g, device=device).to(torch.bfloat16)
    q = torch.randn(steps, nl, B, hq, 128, generator=g, device=device).to(torch.bfloat16)
    return kv, q


def history_bytes(L: int, B: int, H: int) -> int:
    return B * max(0, L - 320) * H * HIST_BYTES


def layer_bytes(lens, H: int, hq: int) -> int:
    """Algorithmic bytes of one layer's decode over requests of lengths `lens` (logical: a page that several
    requests share counts once per request): INT2 history, BF16 sink + recent, q and o."""
    return sum(history_bytes(int(L), 1, H) + min(int(L), 320) * H * BF16_BYTES + 2 * hq * 128 * 2 for L in lens)


def shared_unique_bytes(lens, shared: int, H: int, hq: int) -> int:
    """As layer_bytes with the shared prefix's history and sink pages counted once."""
    if not shared:
        return layer_bytes(lens, H, hq)
    shared_hist = (shared - 64) * H * HIST_BYTES
    return layer_bytes(lens, H, hq) - (len(lens) - 1) * (shared_hist + 64 * H * BF16_BYTES)


# ---------------------------------------------------------------------------------------------


def run_ours(args, rank: int, world: int, device):
    import torch
    import synth

    seed = replica_seed(rank)
    total_steps = args.warmup + args.steps
    mixed = isinstance(WORKLOADS[args.workload]["ctx"], tuple)
    # every leg appends one token per step: the eager step before capture, the graph's warm-up and timed
    # steps, the profiled eager steps (and the one that sizes their delay), and the warm-up and timed
    # steps of the two end-to-end legs
    appends = 1 + (args.warmup - 1 + args.steps) + 1 + args.steps + 2 * (args.warmup + args.steps)
    wl = build_workload(args.workload, seed, device, with_bf16=not (args.no_bf16 or mixed),
                        steps_capacity=appends + 16, algo=args.algo, meta=args.meta_format)
    cache, nl, B, H, hq = wl["cache"], wl["layers"], wl["B"], wl["H"], wl["hq"]
    stream = torch.cuda.current_stream()
    sm = synth.sm_scale()
    kv_new, q_all = step_inputs(wl, total_steps, device, seed)
    kv_cur = torch.empty_like(kv_new[0])          # the step's new K/V, [layers, 2, B, H, 128]
    q_cur = torch.empty_like(q_all[0])            # the step's queries, [layers, B, Hq, 128]
    out = torch.empty(nl, B, hq, 128, dtype=torch.bfloat16, device=device)
    seq = torch.from_numpy(wl["lens"].astype(np.int32)).to(device)
    # per layer, oscar_decode_step launches the step prologue (append with demotion, query rotation), then
    # the fused decode and the merge (mma), or the history kernel, the BF16 segment and the merge (simt)
    launches_per_layer = (4 if wl["shp"] else 3) if args.algo >= 1 else 4   # + the shared-prefix kernel

    def layers():
        for layer in range(nl):
            cache.decode_step(layer, q_cur[layer], kv_cur[layer, 0], kv_cur[layer, 1], seq, wl["hist_pt"],
                              wl["bf16_pt"], sm, out=out[layer], shared_hist_pages=wl["shp"])
        seq.add_(1)

    # capture one step (all layers) into a CUDA graph
    torch.cuda.synchronize()
    kv_cur.copy_(kv_new[0])
    q_cur.copy_(q_all[0])
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        layers()                                   # one eager step on the capture stream first
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            layers()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    if cache.get_status() != 0:
        raise RuntimeError("device status error during capture")

    def step(i):
        kv_cur.copy_(kv_new[i], non_blocking=True)
        q_cur.copy_(q_all[i], non_blocking=True)
        graph.replay()

    for i in range(1, args.warmup):
        step(i)
    torch.cuda.synchronize()
    lens_start = seq.cpu().numpy().astype(np.int64)
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        torch.cuda.synchronize()
        nvtx_id = torch.cuda.nvtx.range_start("timed_steps")     # profiler filter for the launch list
        clk.mark()
        ev0.record(stream)
        for i in range(args.warmup, total_steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_end(nvtx_id)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world, device)
    if cache.get_status() != 0:
        raise RuntimeError("device status error during the timed steps")
    # units: KV tokens attended per step (the appended token included), all layers
    kv_tokens = sum(int(lens_start.sum() + B * (1 + s)) * nl for s in range(args.steps))
    value = whole_job_rate(kv_tokens, ms, world)
    ms_step = ms / args.steps
    step_bytes = sum(layer_bytes(lens_start + 1 + s, H, hq) * nl for s in range(args.steps)) / args.steps
    step_unique = sum(shared_unique_bytes(lens_start + 1 + s, wl["shared"], H, hq) * nl
                      for s in range(args.steps)) / args.steps
    peak, peak_src = peaks()
    # dominant kernel: the fused decode kernel, timed per launch with the library's CUDA events in a second
    # timed region that issues the same steps without the graph
    dec_ms, dec_n, lens_prof, span_us = profile_decode_calls(wl, args, kv_new, q_all, seq, out)
    # algorithmic bytes of one layer's decode: with a shared prefix read once for the batch, its pages count once
    hb = shared_unique_bytes(lens_prof, wl["shared"], H, hq) if wl["shp"] else layer_bytes(lens_prof, H, hq)
    dec_avg_ms = dec_ms / max(dec_n, 1)
    achieved = hb / (dec_avg_ms / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (bf16 I/O)" if args.algo == 0 else "fp16 MMA operands, f32 accumulate (bf16 I/O)",
        "data": "synthetic",
        "config": {"workload": args.workload, **{k: v for k, v in WORKLOADS[args.workload].items()},
                   "head_dim": 128, "sink": 64, "recent": 256, "group": 64, "page": 64, "v_mode": "absorbed",
                   "storage": STORAGE[args.meta_format], "meta_format": args.meta_format,
                   "l2": "inputs larger than L2 (%.2f GB of pool streamed per step)" % (step_bytes / 1e9),
                   "parallelism": f"replicas x{world}", "decode_algo": ALGO_NAMES[args.algo],
                   "launch": "one CUDA graph per step (oscar_decode_step%s per layer), new tokens copied in"
                             % ("_shared, %d shared history pages" % wl["shp"] if wl["shp"] else "")},
        "hbm": {"step_algorithmic_bytes": step_bytes, "step_gbs": step_bytes / (ms_step / 1e3) / 1e9,
                "step_frac_of_peak": step_bytes / (ms_step / 1e3) / 1e9 / peak,
                "step_unique_bytes": step_unique, "step_unique_gbs": step_unique / (ms_step / 1e3) / 1e9},
        "roofline": {"bound": "hbm", "kernel": ("k_decode_shared (shared-prefix pages, all requests) + "
                                                if args.algo >= 1 and wl["shp"] else "") +
                     DECODE_KERNEL_NAMES[args.algo] +
                     ", CUDA events around each launch in an eager copy of the timed steps (enqueued ahead of the GPU)",
                     "achieved": achieved, "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_nominal_7900_gbs": achieved / 7900.0, "traffic": decode_traffic(args), "algorithmic_bytes_per_launch": hb,
                     "avg_launch_us": dec_avg_ms * 1e3, "launches": dec_n,
                     # one profiled launch's CTAs, first start to last end (device timestamps): the
                     # launch time above also holds the GPU's gap between an event and a kernel's first CTA
                     "cta_span_us": span_us,
                     "achieved_over_cta_span": hb / (span_us / 1e6) / 1e9 if span_us else None},
        "gpu_launches": launches_per_layer * nl * args.steps,
        "clocks": clk.summary(),
    }
    if wl["bf16_pages"] is not None:
        res["bf16_baseline"] = run_bf16(wl, args, q_all, device)
        res["bf16_baseline"]["speedup_of_int2_step"] = res["bf16_baseline"]["ms_per_step"] / ms_step
    if wl["prefill"]["tokens"]:
        pf, lens0 = wl["prefill"], wl["lens"]
        moved = pf["tokens"] * H * BF16_BYTES + layer_bytes(lens0, H, 0) * nl     # bf16 K/V read + pool written
        res["prefill"] = {"call": "oscar_quantize_prefill, all requests in one call per layer",
                          "tokens": pf["tokens"], "ms": pf["ms"],
                          "tokens_per_s": pf["tokens"] / (pf["ms"] / 1e3),
                          "algorithmic_bytes": moved, "gbs": moved / (pf["ms"] / 1e3) / 1e9,
                          "frac_of_peak": moved / (pf["ms"] / 1e3) / 1e9 / peak}
    if wl["fused"]["tokens"]:
        fz = wl["fused"]
        flops = 2.0 * fz["tokens"] * fz["d_model"] * 2 * H * 128 * nl          # x W_k^T and x W_v^T
        tpeak, tkind = bf16_peak()
        moved = fz["tokens"] * fz["d_model"] * 2 + layer_bytes(wl["lens"], H, 0) * nl   # x read + pool written
        res["fused_prefill"] = {"call": "oscar_project_quantize_prefill (x W^T, rotate, quantise, pack), one call per "
                                        "layer", "d_model": fz["d_model"], "tokens": fz["tokens"], "ms": fz["ms"],
                                "tokens_per_s": fz["tokens"] / (fz["ms"] / 1e3),
                                "tflops": flops / (fz["ms"] / 1e3) / 1e12, "bound": "tensor",
                                "frac_of_bf16_peak": flops / (fz["ms"] / 1e3) / 1e12 / tpeak, "peak_kind": tkind,
                                "algorithmic_bytes": moved, "gbs": moved / (fz["ms"] / 1e3) / 1e9}
    res["e2e"] = run_e2e(wl, args, device, graph, kv_cur, q_cur, out, seq)
    if cache.get_status() != 0:
        raise RuntimeError("device status error during the end-to-end steps")
    res["e2e_eager"] = run_e2e_eager(wl, args, device, start_lens=seq.cpu().numpy())
    if cache.get_status() != 0:
        raise RuntimeError("device status error during the eager end-to-end steps")
    if rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(wl, seed, device, budget_s=args.cpu_budget)
    return res


def profile_decode_calls(wl, args, kv_new, q_all, seq, out):
    """Eager steps with the library's CUDA events around the history (fused decode) kernel of every
    oscar_decode_step: returns (summed ms, launches, mean context, CTA span in us or None). The CTA
    span is the first profiled step's middle-layer decode kernel from its first CTA's start to its last
    CTA's end (%globaltimer stamps of oscar_trace_ctas; fused decode without a shared prefix only)."""
    import torch
    import synth
    cache, nl = wl["cache"], wl["layers"]
    sm = synth.sm_scale()

    def enqueue(i, trace_layer=-1, tbuf=None):
        for layer in range(nl):
            if layer == trace_layer:
                cache.trace_ctas(tbuf)
            cache.decode_step(layer, q_all[i, layer], kv_new[i, layer, 0], kv_new[i, layer, 1], seq, wl["hist_pt"],
                              wl["bf16_pt"], sm, out=out[layer], shared_hist_pages=wl["shp"])
            if layer == trace_layer:
                cache.trace_ctas(None)           # the launch above keeps the buffer it was given
        seq.add_(1)

    # Each step starts behind a GPU-side delay longer than the host needs to enqueue it, so the GPU runs the
    # step's launches back to back: the events then time the kernel, not the gaps in which the GPU waits
    # for the Python loop to submit the next launch.
    torch.cuda.synchronize()
    t = time.perf_counter()
    enqueue(0)
    host_s = time.perf_counter() - t
    torch.cuda.synchronize()
    delay_cycles = int(max(2.0 * host_s, 1e-3) * 2.2e9)
    lens0 = seq.cpu().numpy().astype(np.int64) + 1
    tbuf = None
    if args.algo == 1 and not wl["shp"]:
        tbuf = torch.zeros(8 * 16384, dtype=torch.int64, device=out.device)
    cache.profile_begin(nl * args.steps)
    for i in range(args.steps):
        torch.cuda._sleep(delay_cycles)
        enqueue(i, nl // 2 if i == 0 else -1, tbuf)
    ms, n = cache.profile_read()
    span_us = None
    if tbuf is not None:
        tr = tbuf.view(-1, 8).cpu().numpy()
        tr = tr[tr[:, 2] > 0]
        if 0 < len(tr) < 16384 and (tr[:, 5] > 0).all():     # every CTA of the launch recorded
            span_us = float(tr[:, 5].max() - tr[:, 2].min()) / 1e3
    return ms, n, lens0 + (args.steps - 1) // 2, span_us


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode launch of the 102,400-token
# Qwen3-8B layer, per decode kernel, from the ncu captures summarised under profiles/, with the digest of the
# CUDA sources each was taken on: a kernel changed since reports null until it is captured again.
NCU_DECODE_TRAFFIC = {
    1: {"bytes_per_launch": 66788864 + 142848, "kernel": "k_decode_mma<1, 3, 0>",
        "command": "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum "
                   "--clock-control none -k regex:k_decode_mma -s 3 -c 1 python bench.py --workload "
                   "qwen3_8b_100k_l1 --steps 3 --warmup 3 --no-bf16 --no-cpu",
        "sources_sha256": "264da5c45f7e2ffbc9061a25edb1f11e6bcdb5dd2881ec6ff728db679f4dfb3d"},
}

# the sources each decode kernel is compiled from (its file and the headers it includes)
DECODE_KERNEL_SOURCES = {
    1: ("decode_mma.cu", "bf16_page.cuh", "kernels.cuh", "common.cuh", "rotate.cuh", "tma.cuh", "timeline.cuh"),
    2: ("decode_tc.cu", "bf16_page.cuh", "tcgen05.cuh", "kernels.cuh", "common.cuh", "tma.cuh", "timeline.cuh"),
}


def sources_digest(algo: int) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_kv_cache_decode_gb300", "csrc")
    for f in DECODE_KERNEL_SOURCES[algo]:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "oscar.h"), "rb").read())
    return h.hexdigest()


def decode_traffic(args):
    rec = NCU_DECODE_TRAFFIC.get(args.algo)
    if rec is None or args.workload not in ("qwen3_8b_36l", "qwen3_8b_100k_l1") or args.meta_format != "f16":
        return None
    if rec["sources_sha256"] != sources_digest(args.algo):
        return None
    return rec["bytes_per_launch"]


def run_bf16(wl, args, q_all, device):
    """The all-BF16 paged decode kernel on the same K/V, all layers, timed like the INT2 step."""
    import torch
    import bit_kv_cache_decode_gb300 as osc
    import synth
    nl, B, H, hq, L = wl["layers"], wl["B"], wl["H"], wl["hq"], wl["L"]
    ws = torch.zeros(osc.bf16_decode_workspace_bytes(B, hq, 512), dtype=torch.uint8, device=device)
    out = torch.empty(B, hq, 128, dtype=torch.bfloat16, device=device)
    seq = torch.full((B,), L, dtype=torch.int32, device=device)
    pages, pt = wl["bf16_pages"], wl["base_pt"]
    sm = synth.sm_scale()

    def step(i):
        for layer in range(nl):
            osc.bf16_decode(pages[layer], q_all[i, layer], seq, pt, sm, H, ws, 512, out=out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        step(args.warmup + i)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    by = B * L * H * BF16_BYTES * nl
    return {"kernel": "BF16 paged decode (same build)", "ms_per_step": ms, "kv_tokens_per_s": B * L * nl / (ms / 1e3),
            "gbs": by / (ms / 1e3) / 1e9, "algorithmic_bytes_per_step": by}


def run_e2e(wl, args, device, graph, kv_cur, q_cur, out, seq):
    """The step end to end from host buffers: each step copies its new K/V and queries from pinned host
    memory into the captured step's input buffers, replays the step, and copies every layer's output back."""
    import torch
    nl, B, H, hq = wl["layers"], wl["B"], wl["H"], wl["hq"]
    host_kv = torch.randn(kv_cur.shape, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    host_q = torch.randn(q_cur.shape, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    host_out = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()

    def step():
        kv_cur.copy_(host_kv, non_blocking=True)
        q_cur.copy_(host_q, non_blocking=True)
        graph.replay()
        host_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    Ls = int(seq.sum().item())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    kv_tokens = sum((Ls + B * (1 + s)) * nl for s in range(args.steps)) / args.steps
    return {"value": kv_tokens / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": (host_kv.numel() + host_q.numel()) * 2, "d2h_bytes_per_step": host_out.numel() * 2,
            "path": "pinned host -> device copy, graph replay of the C-ABI calls, device -> host copy"}


def run_e2e_eager(wl, args, device, start_lens):
    """As run_e2e but issuing oscar_decode_step directly from Python every step (no graph)."""
    import torch
    import synth
    cache, nl, B, H, hq = wl["cache"], wl["layers"], wl["B"], wl["H"], wl["hq"]
    sm = synth.sm_scale()
    n_in = nl * (2 * B * H + B * hq) * 128
    host_in = torch.randn(n_in, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    host_out = torch.empty(nl * B * hq * 128, dtype=torch.bfloat16).pin_memory()
    dev_in = torch.empty_like(host_in, device=device)
    dev_out = torch.empty(nl, B, hq, 128, dtype=torch.bfloat16, device=device)
    torch.cuda.synchronize()
    seq = torch.as_tensor(start_lens, dtype=torch.int32).to(device)   # the cache's current lengths
    kvn = dev_in[:nl * 2 * B * H * 128].view(nl, 2, B, H, 128)
    qn = dev_in[nl * 2 * B * H * 128:].view(nl, B, hq, 128)

    def step():
        dev_in.copy_(host_in, non_blocking=True)
        for layer in range(nl):
            cache.decode_step(layer, qn[layer], kvn[layer, 0], kvn[layer, 1], seq, wl["hist_pt"], wl["bf16_pt"], sm,
                              out=dev_out[layer], shared_hist_pages=wl["shp"])
        host_out.copy_(dev_out.view(-1), non_blocking=True)
        seq.add_(1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    Ls = int(seq.sum().item())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    kv_tokens = sum((Ls + B * (1 + s)) * nl for s in range(args.steps)) / args.steps
    return {"value": kv_tokens / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": host_in.numel() * 2, "d2h_bytes_per_step": host_out.numel() * 2,
            "path": "pinned host -> device copy, direct C-ABI calls from Python, device -> host copy"}


def oracle_threads() -> int:
    """Threads the oracle's numpy can use: its BLAS pool (matrix products) as the environment sets it,
    else one per core this process may run on; the elementwise steps run on one of them."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, seed, device, min_s: float = 10.0, budget_s: float = 20.0):
    """The CPU oracle's decode of layer 0 of the workload (unpack, dequantise, fp64 exact softmax), from
    the pool bytes the GPU wrote, on the host cores: its kv heads in turn until about min_s seconds of
    work are done."""
    from oracle import attention as A
    from oracle import pool as P
    cache, H, hq, L = wl["cache"], wl["H"], wl["hq"], int(wl["lens"][0])
    import torch
    torch.cuda.synchronize()
    cfg = wl["cfg"]
    import bit_kv_cache_decode_gb300 as osc
    geo = P.PoolGeometry(hkv=H, meta_format={v: k for k, v in META_FORMATS.items()}[cfg.meta_format])
    pm = P.PoolModel(geo, cfg.num_int2_pages, cfg.num_bf16_pages)
    pm.int2[:] = cache.int2_pages(0).cpu().numpy()
    pm.bf16[:] = cache.bf16_pages(0).cpu().numpy().view(np.uint16).reshape(pm.bf16.shape)
    prm = [P.HeadParams(c["U_K"], c["U_V"], c["tau_K"], c["tau_V"], c.get("cb_k"), c.get("cb_v"))
           for c in wl["cals"][:H]]
    q = np.random.default_rng(seed).standard_normal((hq, 128)).astype(np.float32)
    Lnow = int(L)
    # best of three samples, each about a third of the time
    samples = []
    for _ in range(3):
        heads, dt, busy = time_head_decodes(
            lambda hd: A.decode_request(q, Lnow, pm, wl["hist_np"][0], wl["bf16_np"][0], prm, True,
                                        1 / math.sqrt(128), kv_heads=[hd]), H, min_s / 3, budget_s / 3)
        samples.append((Lnow * heads / H / dt, heads, dt, busy))   # KV tokens of one layer-step per H decodes
    rate, heads, dt, busy = max(samples)
    return {"value": rate, "unit": UNIT, "cores": oracle_threads(), "cpu_s_per_wall_s": busy, "kind": "oracle",
            "samples": [round(x[0], 1) for x in samples],
            "sample": f"layer 0, best of 3 samples (this one: {heads} kv-head decodes, its {H} kv heads in turn, "
                      f"{hq // H} q heads each, {dt:.1f} s), context {Lnow}; numpy fp64 unpack + dequantise + "
                      f"exact softmax"}


def time_head_decodes(decode_head, H: int, min_s: float, budget_s: float):
    """Run decode_head(0), decode_head(1), ..., cycling over the H kv heads, until at least min_s seconds
    have passed (and at least one decode ran), stopping early once budget_s is used. Returns (decodes,
    wall seconds, process CPU seconds per wall second: an upper bound on the busy cores, since BLAS
    threads spinning between products count too)."""
    t0, c0 = time.perf_counter(), time.process_time()
    n = 0
    while True:
        decode_head(n % H)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_s or el > budget_s:
            break
    dt = time.perf_counter() - t0
    return n, dt, (time.process_time() - c0) / dt


REFERENCE_SAMPLE_TOKENS = 32768


def run_reference(args, rank, world):
    """The oracle as the reference arm: one step = the oracle's decode of a bounded sample of the workload
    on the host cores: one kv head of layer 0 over at most the first 32,768 tokens of the context (a request
    of that length), so that a run of --steps K stays within minutes."""
    if rank != 0:
        return None
    from oracle import attention as A
    from oracle import pool as P
    from oracle import rotation
    import synth
    w = WORKLOADS[args.workload]
    ctx = w["ctx"][1] if isinstance(w["ctx"], tuple) else w["ctx"]
    L, H, hq = min(ctx, REFERENCE_SAMPLE_TOKENS), w["hkv"], w["hq"]
    seed = 1234
    # build layer 0 of the workload with the oracle itself (one kv head per step sample)
    geo = P.PoolGeometry(hkv=1, meta_format=args.meta_format)
    nh = (L - 320 + 63) // 64
    pm = P.PoolModel(geo, nh, 5)
    qc, kc, vc = synth.calibration(seed, 0, 0)
    cal = rotation.calibrate(qc, kc, vc, synth.sm_scale())
    prm = [P.HeadParams(cal["U_K"].astype(np.float32), cal["U_V"].astype(np.float32),
                        cal["tau_K"].astype(np.float32), cal["tau_V"].astype(np.float32))]
    if args.meta_format == "cb":
        from oracle import codebook as CB
        prm[0].cb_k = CB.calibrate_codebook(P.rotated_f32(kc, prm[0].u_k), prm[0].tau_k)
        prm[0].cb_v = CB.calibrate_codebook(vc.astype(np.float32), prm[0].tau_v)
    k, v = synth.kv_tokens(seed, 0, 0, L)
    P.prefill(pm, k[:, None], v[:, None], np.arange(nh), np.arange(5), prm, True)
    q = synth.queries(seed, 0, 0, hq // H)
    for _ in range(args.warmup):
        A.decode_request(q, L, pm, np.arange(nh), np.arange(5), prm, True, synth.sm_scale())
    t0, c0 = time.perf_counter(), time.process_time()
    for _ in range(args.steps):
        A.decode_request(q, L, pm, np.arange(nh), np.arange(5), prm, True, synth.sm_scale())
    busy = (time.process_time() - c0) / (time.perf_counter() - t0)
    dt = (time.perf_counter() - t0) / args.steps
    value = L / H / dt        # one kv head of one layer per step: L/H of the layer's KV tokens
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, **w},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "cpu_s_per_wall_s": busy,
                             "kind": "oracle",
                             "sample": f"layer 0, 1 of {H} kv heads ({hq // H} q heads), the first {L} tokens of "
                                       f"the {ctx}-token context as one request, per step; numpy fp64 unpack + "
                                       f"dequantise + exact softmax"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------------------------


def replica_seed(rank: int) -> int:
    """Each rank runs an independent replica of the workload (weak scaling) from its own seed."""
    return 1234 + rank


def whole_job_rate(units_per_rank: float, ms_max: float, world: int) -> float:
    """Units per second of the whole job: every rank processed units_per_rank within the slowest
    rank's time ms_max."""
    return units_per_rank * world / (ms_max / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config4_leg(args):
    """Config 4 (batch 32 x 102,400 tokens sharing a 92,160-token prefix) on its first 4 of 36 layers, as a
    bounded extra leg of the default run: the same bench in a child process (its own timed graph steps,
    10 of them), its line summarised. Every layer is the same launch chain, so 36 / 4 of its step time is
    the 36-layer step it stands for."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "qwen3_4b_b32_l4", "--steps", "10",
           "--warmup", "3", "--no-bf16", "--no-cpu", "--no-config4", "--algo", str(args.algo),
           "--meta-format", args.meta_format]
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    if p.returncode != 0 or not lines:
        return {"error": (p.stderr or p.stdout)[-400:], "command": " ".join(cmd[1:])}
    d = json.loads(lines[-1])
    return {"workload": "qwen3_4b_b32, first 4 of 36 layers", "command": " ".join(cmd[1:]),
            "ms_per_step_4_layers": d["ms_per_step"], "ms_per_layer": d["ms_per_step"] / 4,
            "ms_per_36_layer_step": d["ms_per_step"] * 9, "kv_tokens_per_s": d["value"],
            "step_unique_gbs": d["hbm"]["step_unique_gbs"], "step_unique_frac": d["hbm"]["step_unique_gbs"] /
            d["roofline"]["peak"], "decode_launch_us": d["roofline"]["avg_launch_us"], "clocks": d["clocks"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="qwen3_8b_36l")
    ap.add_argument("--algo", type=int, default=None, choices=(0, 1, 2),
                    help="INT2 decode kernel: 0 simt, 1 mma.sync (default), 2 tcgen05")
    ap.add_argument("--no-bf16", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-config4", action="store_true", help="skip the default run's 4-layer config-4 leg")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--meta-format", choices=["f16", "u8", "cb"], default="f16",
                    help="INT2 group metadata: fp16 scale/zero (default), the compact 16-bit format, or the "
                         "Lloyd-Max codebook format")
    args = ap.parse_args()
    global HIST_BYTES
    HIST_BYTES = HIST_BYTES_BY_META[args.meta_format]
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import __graft_entry__
    __graft_entry__.build()
    if args.algo is None:
        args.algo = 1
    res = run_ours(args, rank, world, device)
    if rank == 0 and world == 1 and args.workload == "qwen3_8b_36l" and not args.no_config4:
        res["config4"] = config4_leg(args)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
