#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = the whole hot path over one batch of synthetic input, run as the
layer stack of a model forward:
  * causal prefill at the Llama-3-8B attention shape at long context (batch 1,
    32 query / 8 key-value heads, head_dim 128, N = 32768, 1% of the keys
    scaled by 8), once per layer of that model (32 launches): attn_prefill;
  * single-token split-KV decode + LSE combine at the Qwen2.5-7B attention
    shape (28 / 4 heads) over a 30720-token contiguous cache, once per layer
    of that model (28 layers, each its own cache, launched back to back):
    attn_decode_splitkv + attn_combine.
The headline value is causal-prefill attention TFLOP/s (4 N^2 d heads, halved
for causal); the decode's HBM GB/s per layer is reported beside it.  Inputs
are resident in HBM when the timed region starts and exceed L2.  After the
timed region every other workload is measured once and reported under
"workloads" (Qwen prefill at N = 2048 and 8192, Llama prefill at N = 30720, the
decode split sweep single and chained, the paged batch decode), followed by
the next rows (append, packed, FP8, head_dim 256, variants).

`--impl reference` times the float64 CPU oracle (the only other place this file
runs anything under oracle/) on a bounded sample of the same workload.

N > 1 GPUs (torchrun): one independent replica per GPU ("replicas only": the
path needs no exchange between GPUs), barrier + max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal prefill attention TFLOP/s (% BF16 peak); split-KV decode HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal GB300 figures, for the fractions quoted beside the measured ones.
NOMINAL = {"bf16_tflops": 2250.0, "hbm_gbs": 7900.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "prefill_sm103_llama_n32768.txt")
PREFILL_SRC = os.path.join(ROOT, "exact_io_aware_order_gb300", "csrc", "prefill_sm103.cu")

HEADLINE = {
    "prefill": dict(n_q=32, n_kv=8, seqlen=32768, d=128, layers=32),
    "decode": dict(n_q=28, n_kv=4, kv_len=30720, layers=28),
    "desc": "Llama-3-8B attention, causal prefill N=32768 (32/8 heads, d=128, 1% keys x8) "
            "x 32 layers + Qwen2.5-7B attention, split-KV decode + combine over a "
            "30720-token cache (28/4 heads) x 28 layers",
}


def rank_env() -> tuple:
    """(rank, world size) from the launcher's environment; (0, 1) without one."""
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def rank_max(dist, vals, device=None) -> list:
    """Max over ranks of each timed quantity (identity in a single process).
    Every rank gets the same list back."""
    if dist is None:
        return [float(v) for v in vals]
    import torch

    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rate(units_per_step: float, steps: int, world: int, slowest_ms: float) -> float:
    """Whole-job throughput of replicas: every rank processes units_per_step
    each step (weak scaling), over the slowest rank's time."""
    return world * units_per_step * steps / (slowest_ms * 1e-3)


def prefill_flops(n_q: int, seqlen: int, d: int, batch: int = 1) -> float:
    return 4.0 * batch * n_q * float(seqlen) ** 2 * d / 2.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def code_hash(path: str) -> str:
    """First 16 hex digits of the SHA-256 of a C/CUDA source with its //
    comments, surrounding whitespace and blank lines removed: a comment edit
    keeps the hash, any change to the code changes it."""
    lines = []
    for line in open(path, encoding="utf-8").read().splitlines():
        code = line.split("//", 1)[0].strip()
        if code:
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the prefill kernel from the committed ncu
    summary, or None when the kernel's code changed since the capture."""
    try:
        text = open(PROFILE_SUMMARY).read()
        sha = code_hash(PREFILL_SRC)
        vals = dict(line.split(":", 1) for line in text.splitlines() if ":" in line)
        if vals.get("code_sha256_16", "").strip() != sha:
            return None
        return float(vals["dram_bytes_per_launch"].strip())
    except Exception:
        return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------------------
# The GB300 arm.
# ---------------------------------------------------------------------------
def _ev():
    import torch

    return torch.cuda.Event(enable_timing=True)


def _host_ahead():
    """Keeps the GPU busy for ~1 ms so that the launches queued next are
    already waiting when it gets to them (launch latency off the clock)."""
    import torch

    torch.cuda._sleep(2_000_000)


def _rooflines(achieved, peak, nominal, unit, bound, **extra):
    d = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "frac_of_nominal": round(achieved / nominal, 4)}
    d.update(extra)
    return d


def run_gb300(args, rank: int, world: int, dist):
    import torch

    import exact_io_aware_order_gb300 as attn
    from exact_io_aware_order_gb300 import workloads as W

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    attn.lib()  # fail loudly if the library is missing
    peaks, peak_src = load_peaks()
    P = HEADLINE["prefill"]
    Dc = HEADLINE["decode"]
    LP, LD = P["layers"], Dc["layers"]

    # ---- inputs (seeded, synthetic), resident in HBM ----
    x = W.llama_long_prefill(P["seqlen"])
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o = [torch.empty(tuple(x.q.shape), dtype=torch.float32, device=dev) for _ in range(2)]
    lse = [torch.empty(tuple(x.q.shape[:3]), dtype=torch.float32, device=dev) for _ in range(2)]
    flops = prefill_flops(P["n_q"], P["seqlen"], P["d"])
    dec = W.qwen_decode(Dc["kv_len"])
    dq, dlens = dec.q.to(dev), dec.kv_lens.to(dev)
    kc0, vc0 = dec.k_cache.to(dev), dec.v_cache.to(dev)
    caches = [(kc0, vc0)] + [(kc0.clone(), vc0.clone()) for _ in range(LD - 1)]  # one per layer
    B, Hq, D = dq.shape
    S = attn.decode_num_splits(B, dec.n_kv, dec.max_kv_len)
    op = torch.empty((S, B, Hq, D), dtype=torch.float32, device=dev)
    lp = torch.empty((S, B, Hq), dtype=torch.float32, device=dev)
    do = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    dl = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    dec_bytes = decode_bytes(dec)

    # A read-only sweep over twice the L2 between the prefill chain and the
    # decode chain: the prefill leaves much of its output dirty in L2, and
    # without the sweep the first decodes would pay for those write-backs.
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size) or (128 << 20)
    sweep = torch.ones((2 * l2) // 4, dtype=torch.float32, device=dev)
    sweep_out = torch.empty((), dtype=torch.float32, device=dev)

    def decode_layer(l):
        # Early cache streaming: each layer has its own cache, so the kernel
        # before a decode (the previous layer's combine, or the L2 sweep)
        # writes none of what the decode reads before its wait.
        kc, vc = caches[l]
        attn.decode_splitkv(dq, kc, vc, dlens, None, num_splits=S, max_kv_len=dec.max_kv_len,
                            scale=dec.scale, o_partial=op, lse_partial=lp, early_cache=True)
        attn.combine(op, lp, out=do, lse=dl)

    def step(ev=None):
        if ev is not None:
            ev[0].record()
        for l in range(LP):
            attn.prefill(q, k, v, x.scale, True, out=o[l & 1], lse=lse[l & 1])
        if ev is not None:
            ev[1].record()
        torch.sum(sweep, dim=0, out=sweep_out)
        _host_ahead()
        if ev is not None:
            ev[2].record()
        # decode + combine of every layer, back to back; no event between a
        # decode and its combine (it would stop the combine's early launch)
        for l in range(LD):
            decode_layer(l)
        if ev is not None:
            ev[3].record()

    for i in range(args.warmup):
        step()
    attn.check_device_status()
    evs = [[_ev() for _ in range(4)] for _ in range(args.steps)]
    gpu_uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + gpu_uuid) if gpu_uuid and not gpu_uuid.startswith("GPU-")
                           else (gpu_uuid or str(dev.index)))
    time.sleep(0.15)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start, t_end = _ev(), _ev()
    t_start.record()
    for i in range(args.steps):
        step(evs[i])
    t_end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    attn.check_device_status()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms, pre_total, dec_total = rank_max(dist, [total_ms, sum(pre_ms), sum(dec_ms)], dev)
    prefill_tflops = job_rate(flops * LP, args.steps, world, pre_total) / 1e12
    decode_gbs = job_rate(dec_bytes * LD, args.steps, world, dec_total) / 1e9
    avg_pre = statistics.mean(pre_ms) / LP
    achieved = flops / (avg_pre * 1e-3) / 1e12
    traffic = profiled_traffic()

    result = {
        "metric": METRIC, "value": round(prefill_tflops, 2), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(world),
        "roofline": _rooflines(achieved, peaks["bf16_tflops_sustained"], NOMINAL["bf16_tflops"],
                               "TFLOP/s", "tensor", traffic=traffic,
                               kernel="prefill_kernel<128, 0, 0>",
                               peak_source=peak_src + " bf16 sustained (the prefill runs "
                               "back to back for seconds inside the timed region)",
                               frac_of_burst_peak=round(achieved / peaks["bf16_tflops"], 4),
                               flops_per_launch=flops, avg_launch_ms=round(avg_pre, 4),
                               launches=LP * args.steps),
        "decode": {"value": round(decode_gbs, 1), "unit": "GB/s",
                   "what": f"decode + combine per layer, {LD} layers back to back (each its "
                           f"own {Dc['kv_len']}-token cache), chained by programmatic "
                           "dependent launch: steady state",
                   "frac": round(decode_gbs / peaks["hbm_gbs"], 4),
                   "frac_of_nominal": round(decode_gbs / NOMINAL["hbm_gbs"], 4),
                   "peak": peaks["hbm_gbs"], "peak_source": peak_src + " hbm copy",
                   "bytes_per_layer": dec_bytes, "num_splits": S,
                   "avg_layer_us": round(statistics.mean(dec_ms) / LD * 1e3, 2)},
        "gpu_launches": (LP + 2 * LD) * args.steps,
        "clocks": clocks,
    }
    del caches
    if args.no_extras:
        return result
    workloads = {}
    del q, k, v, o, lse
    torch.cuda.empty_cache()
    legs = set(("workloads,append,varlen,fp8,d256,variants" if args.legs == "all" else args.legs)
               .split(","))
    if "workloads" in legs:
        workloads["llama_prefill_long"] = time_prefill_lengths(
            attn, dev, dist, peaks, [(30720, W.llama_long_prefill)],
            extra={32768: (achieved, avg_pre)})
        workloads["qwen_prefill"] = time_prefill_lengths(
            attn, dev, dist, peaks, [(2048, W.qwen_prefill), (8192, W.qwen_prefill)])
        workloads["qwen_decode_30720"] = time_decode_sweep(
            args, attn, W, dev, dist, peaks, sweep, sweep_out, chain_two=dec_total / args.steps)
        workloads["paged_decode_batch16"] = time_paged_batch(args, attn, W, dev, dist, peaks, sweep,
                                                      sweep_out)
        result["workloads"] = workloads

    # ---- the next rows, on the Qwen2.5-7B layer at N = 8192 ----
    xq = W.qwen_prefill(8192)
    qq, kq, vq = xq.q.to(dev), xq.k.to(dev), xq.v.to(dev)
    oq = torch.empty(tuple(xq.q.shape), dtype=torch.float32, device=dev)
    lq = torch.empty(tuple(xq.q.shape[:3]), dtype=torch.float32, device=dev)
    dec_caches = [(kc0, vc0)] + [(kc0.clone(), vc0.clone()) for _ in range(3)]
    bf = peaks["bf16_tflops"]
    if "append" in legs:
        app = time_decode_append(args, attn, dq, dec_caches, dec, S, op, lp, sweep, sweep_out,
                                 dist, dev)
        if app is not None:
            app["roofline"]["peak"] = peaks["hbm_gbs"]
            app["roofline"]["frac"] = round(app["roofline"]["achieved"] / peaks["hbm_gbs"], 4)
            app["roofline"]["peak_source"] = peak_src + " hbm copy"
            result["decode_append"] = app
    if "varlen" in legs:
        vl = time_prefill_varlen(args, attn, W, dist, dev)
        vl["roofline"]["peak"] = bf
        vl["roofline"]["frac"] = round(vl["roofline"]["achieved"] / bf, 4)
        vl["roofline"]["peak_source"] = peak_src + " bf16 burst"
        result["prefill_varlen"] = vl
    if "fp8" in legs:
        f8 = time_fp8(args, attn, xq, qq, kq, vq, oq, lq, dist, dev)
        f8_meas = measure_fp8_gemm_peak(dev)
        if f8_meas is not None:
            f8_peak, f8_src = f8_meas, "measured e4m3 GEMM (torch._scaled_mm, 8192^3, best of 10)"
        else:
            f8_peak = bf * 2.0   # nominal dense fp8 / bf16 ratio (4.5 / 2.25)
            f8_src = peak_src + " bf16 burst x 2 (nominal fp8 / bf16)"
        f8["roofline"]["peak"] = round(f8_peak, 1)
        f8["roofline"]["frac"] = round(f8["roofline"]["achieved"] / f8_peak, 4)
        f8["roofline"]["frac_of_bf16_peak"] = round(f8["roofline"]["achieved"] / bf, 4)
        f8["roofline"]["peak_source"] = f8_src
        if "qwen_prefill" in workloads:
            f8["speedup_over_bf16_prefill"] = round(
                f8["roofline"]["achieved"] / workloads["qwen_prefill"]["N=8192"]["value"], 3)
        f8["quantize_frac_of_hbm"] = round(f8["quantize_gbs"] / peaks["hbm_gbs"], 4)
        result["prefill_fp8"] = f8
    if "d256" in legs:
        d256 = time_d256(args, attn, W, dist, dev)
        d256["roofline"]["peak"] = bf
        d256["roofline"]["frac"] = round(d256["roofline"]["achieved"] / bf, 4)
        d256["decode"]["roofline"]["peak"] = peaks["hbm_gbs"]
        d256["decode"]["roofline"]["frac"] = round(
            d256["decode"]["roofline"]["achieved"] / peaks["hbm_gbs"], 4)
        result["prefill_d256"] = d256
        d64 = time_d64(args, attn, W, dist, dev)
        d64["roofline"]["peak"] = bf
        d64["roofline"]["frac"] = round(d64["roofline"]["achieved"] / bf, 4)
        result["prefill_d64"] = d64
    if "variants" in legs:
        var = time_variants(args, attn, qq, kq, vq, xq.scale, oq, lq, dq, dec_caches, dec, S, op,
                            lp, sweep, sweep_out, dist, dev)
        for v_ in var["prefill"].values():
            v_["frac"] = round(v_["value"] / bf, 4)
        var["decode"]["frac"] = round(var["decode"]["value"] / peaks["hbm_gbs"], 4)
        result["variants"] = var
    del qq, kq, vq, oq, lq, dec_caches
    torch.cuda.empty_cache()
    if not args.no_e2e:
        result["e2e"] = run_e2e(args, x, dec, dev, world, dist)
    return result


def measure_fp8_gemm_peak(dev):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of the vendor library on this
    GPU (8192^3, best of 10 CUDA-event timings): the denominator of the FP8
    prefill's roofline.  None when the library call is unavailable."""
    import torch

    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()   # column-major operand
        one = torch.tensor(1.0, device=dev)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16,
                                      use_fast_accum=True)
        for _ in range(3):
            mm()
        best = float("inf")
        for _ in range(10):
            e0, e1 = _ev(), _ev()
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def decode_bytes(dec) -> int:
    """Algorithmic bytes of one decode: the K and V rows attended, q, and the
    final O and LSE (the split partials are overhead, not credited)."""
    B, Hq, D = dec.q.shape
    tokens = int(dec.kv_lens.sum())
    return tokens * dec.n_kv * D * 2 * 2 + B * Hq * D * 2 + B * Hq * (D + 1) * 4


def headline_config(world: int) -> dict:
    P, Dc = HEADLINE["prefill"], HEADLINE["decode"]
    return {"workload": HEADLINE["desc"], "batch": 1, "n_q_heads": P["n_q"],
            "n_kv_heads": P["n_kv"], "seqlen": P["seqlen"], "head_dim": P["d"],
            "prefill_layers_per_step": P["layers"], "spiked_keys": "1% of keys x8 per kv head",
            "decode": {"n_q_heads": Dc["n_q"], "n_kv_heads": Dc["n_kv"], "head_dim": 128,
                       "kv_len": Dc["kv_len"], "layers_per_step": Dc["layers"],
                       "num_splits": "the library's policy (attn_decode_num_splits)",
                       "cache": "contiguous, one per layer",
                       "launch": "decode with ATTN_DECODE_EARLY_CACHE, then attn_combine, "
                                 "layer after layer on one stream"},
            "l2": "inputs larger than L2 (prefill Q+K+V 403 MB, each launch writes a 537 MB "
                  "output; 28 decode caches of 63 MB); a read-only sweep of 2x L2 between "
                  "the prefill chain and the decode chain",
            "parallelism": f"replicas x{world}"}


def _timed(fn, n, dist, dev, before=None):
    """Sum over n launches of fn's CUDA-event time (max over ranks); `before`
    runs outside the events (an L2 sweep), then the host is put ahead."""
    import torch

    for i in range(3):
        fn(i)
    evs = [(_ev(), _ev()) for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        if before is not None:
            before()
        _host_ahead()
        evs[i][0].record()
        fn(i)
        evs[i][1].record()
    torch.cuda.synchronize()
    (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    return tot


def time_prefill_lengths(attn, dev, dist, peaks, cases, extra=None):
    """Causal prefill TFLOP/s per (sequence length, input maker); each launch
    writes a fresh output larger than L2 (two output buffers alternate)."""
    import torch

    out = {}
    for N, make in cases:
        x = make(N)
        q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
        o = [torch.empty(tuple(x.q.shape), dtype=torch.float32, device=dev) for _ in range(2)]
        l = [torch.empty(tuple(x.q.shape[:3]), dtype=torch.float32, device=dev) for _ in range(2)]
        Hq = x.q.shape[1]
        fl = prefill_flops(Hq, N, x.q.shape[3])
        n = 20 if N <= 8192 else 6
        t = _timed(lambda i: attn.prefill(q, k, v, x.scale, True, out=o[i & 1], lse=l[i & 1]), n,
                   dist, dev)
        attn.check_device_status()
        ach = fl / (t / n * 1e-3) / 1e12
        out[f"N={N}"] = {"value": round(ach, 2), "unit": "TFLOP/s",
                         "frac": round(ach / peaks["bf16_tflops"], 4),
                         "frac_of_nominal": round(ach / NOMINAL["bf16_tflops"], 4),
                         "peak": peaks["bf16_tflops"], "peak_source": "bf16 burst",
                         "avg_launch_ms": round(t / n, 4), "flops_per_launch": fl,
                         "heads": f"{Hq}/{x.k.shape[1]}", "launches": n}
        del q, k, v, o, l
    for N, (ach, ms) in (extra or {}).items():
        out[f"N={N}"] = {"value": round(ach, 2), "unit": "TFLOP/s",
                         "frac": round(ach / peaks["bf16_tflops_sustained"], 4),
                         "frac_of_burst_peak": round(ach / peaks["bf16_tflops"], 4),
                         "frac_of_nominal": round(ach / NOMINAL["bf16_tflops"], 4),
                         "peak": peaks["bf16_tflops_sustained"],
                         "peak_source": "bf16 sustained (the headline's timed region)",
                         "avg_launch_ms": round(ms, 4), "heads": "32/8"}
    torch.cuda.empty_cache()
    return out


def time_decode_sweep(args, attn, W, dev, dist, peaks, sweep, sweep_out, chain_two):
    """Single-token decode over the 30720-token Qwen2.5-7B-layer cache, for the
    split counts {1, 16, 64, 148} and the policy's: the decode kernel alone and
    decode + combine, each single (an L2 sweep before,
    outside the events) and, for the policy's count, chained over four caches."""
    import torch

    dec = W.qwen_decode(30720)
    dq, dlens = dec.q.to(dev), dec.kv_lens.to(dev)
    kc0, vc0 = dec.k_cache.to(dev), dec.v_cache.to(dev)
    caches = [(kc0, vc0)] + [(kc0.clone(), vc0.clone()) for _ in range(3)]
    B, Hq, D = dq.shape
    nbytes = decode_bytes(dec)
    hbm = peaks["hbm_gbs"]
    auto = attn.decode_num_splits(B, dec.n_kv, dec.max_kv_len)
    n = 20
    flush = lambda: torch.sum(sweep, dim=0, out=sweep_out)
    res = {"bytes_per_launch": nbytes, "policy_splits": auto, "peak": hbm,
           "peak_source": "measured hbm copy",
           "timing": "CUDA events around each launch group; single = one launch after an L2 "
                     "sweep with the host ahead; chain = back to back over distinct caches"}
    for S in (1, 16, 64, 148, auto):
        op = torch.empty((S, B, Hq, D), dtype=torch.float32, device=dev)
        lp = torch.empty((S, B, Hq), dtype=torch.float32, device=dev)
        o = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
        l = torch.empty((B, Hq), dtype=torch.float32, device=dev)

        def alone(i):
            kc, vc = caches[i % 4]
            attn.decode_splitkv(dq, kc, vc, dlens, None, num_splits=S, max_kv_len=30720,
                                scale=dec.scale, o_partial=op, lse_partial=lp)

        def two(i):
            alone(i)
            attn.combine(op, lp, out=o, lse=l)

        def alone_early(i):
            kc, vc = caches[i % 4]
            attn.decode_splitkv(dq, kc, vc, dlens, None, num_splits=S, max_kv_len=30720,
                                scale=dec.scale, o_partial=op, lse_partial=lp, early_cache=True)

        def two_early(i):
            alone_early(i)
            attn.combine(op, lp, out=o, lse=l)

        entry = {}
        for name, fn in (("decode", alone), ("decode+combine", two)):
            t = _timed(fn, n, dist, dev, before=flush)
            gbs = nbytes / (t / n * 1e-3) / 1e9
            entry[name] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                           "us": round(t / n * 1e3, 2)}
        attn.check_device_status()
        res[f"S={S}" + (" (policy)" if S == auto else "")] = entry
        if S == auto:
            chain = {}
            for name, fn in (("decode", alone), ("decode+combine", two),
                             ("decode, early cache streaming", alone_early),
                             ("decode+combine, early cache streaming", two_early)):
                L = 28
                t = _timed(lambda i: [fn(j) for j in range(L)], 5, dist, dev, before=flush)
                gbs = nbytes * L / (t / 5 * 1e-3) / 1e9
                chain[name] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                               "us_per_layer": round(t / 5 / L * 1e3, 2)}
            attn.check_device_status()
            step_gbs = nbytes * HEADLINE["decode"]["layers"] / (chain_two * 1e-3) / 1e9
            chain["decode+combine (headline step, 28 distinct caches)"] = {
                "GB/s": round(step_gbs, 1), "frac": round(step_gbs / hbm, 4)}
            res["chain (4 caches in rotation, 28 layers)"] = chain
    del caches
    torch.cuda.empty_cache()
    return res


def time_paged_batch(args, attn, W, dev, dist, peaks, sweep, sweep_out):
    """Paged decode of 16 sequences (lengths uniform in [1024, 32768]), 32 / 8
    heads, 16-token blocks, the policy's split count: decode alone and decode +
    combine, single launches over two device copies of the cache
    (2.4 GB, each launch reads HBM)."""
    import torch

    dec = W.llama_paged_decode()
    dq, dlens, dbt = dec.q.to(dev), dec.kv_lens.to(dev), dec.block_table.to(dev)
    caches = [(dec.k_cache.to(dev), dec.v_cache.to(dev))]
    caches.append((caches[0][0].clone(), caches[0][1].clone()))
    B, Hq, D = dq.shape
    S = attn.decode_num_splits(B, dec.n_kv, dec.max_kv_len)
    op = torch.empty((S, B, Hq, D), dtype=torch.float32, device=dev)
    lp = torch.empty((S, B, Hq), dtype=torch.float32, device=dev)
    o = torch.empty((B, Hq, D), dtype=torch.float32, device=dev)
    l = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    nbytes = decode_bytes(dec)
    hbm = peaks["hbm_gbs"]

    def alone(i):
        kc, vc = caches[i % 2]
        attn.decode_splitkv(dq, kc, vc, dlens, dbt, num_splits=S, max_kv_len=dec.max_kv_len,
                            scale=dec.scale, o_partial=op, lse_partial=lp)

    def two(i):
        alone(i)
        attn.combine(op, lp, out=o, lse=l)

    res = {"bytes_per_launch": nbytes, "num_splits": S, "tokens": int(dec.kv_lens.sum()),
           "peak": hbm, "peak_source": "measured hbm copy"}
    for name, fn in (("decode", alone), ("decode+combine", two)):
        t = _timed(fn, 10, dist, dev)
        gbs = nbytes / (t / 10 * 1e-3) / 1e9
        res[name] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                     "us": round(t / 10 * 1e3, 2)}
    attn.check_device_status()
    del caches
    torch.cuda.empty_cache()
    return res


def time_variants(args, attn, q, k, v, scale, o, lse, dq, caches, dec, S, op, lp, sweep, sweep_out,
                  dist, dev):
    """The attention variants on the step's shapes: prefill with a 4096-token
    sliding window and a soft cap of 50, and the decode with the same window.
    FLOPs count the keys each row actually sees (4 d per query-key pair and
    head); decode bytes count the K/V rows inside the window."""
    import torch

    Wl, cap = 4095, 50.0
    B, Hq, N, D = q.shape
    keys = sum(min(i + 1, Wl + 1) for i in range(N))
    flops = 4.0 * D * Hq * B * keys
    n = max(3, min(args.steps, 100))
    world = dist.get_world_size() if dist is not None else 1

    def timed(fn, before=None):
        for i in range(3):
            fn(i)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        for i in range(n):
            if before is not None:
                before()
            evs[i][0].record()
            fn(i)
            evs[i][1].record()
        torch.cuda.synchronize()
        attn.check_device_status()
        (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
        return tot

    full = 4.0 * D * Hq * B * sum(i + 1 for i in range(N))
    pre = {}
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32,
                          device=dev)
    for name, (w_, c_, al, fl) in {"window": (Wl, 0.0, None, flops),
                                   "softcap": (-1, cap, None, full),
                                   "window+softcap": (Wl, cap, None, flops),
                                   "alibi": (-1, 0.0, slopes, full)}.items():
        t = timed(lambda i: attn.prefill(q, k, v, scale, True, out=o, lse=lse, window_left=w_,
                                         softcap=c_, alibi_slopes=al))
        pre[name] = {"value": round(job_rate(fl, n, world, t) / 1e12, 2), "unit": "TFLOP/s",
                     "window_left": w_, "softcap": c_, "alibi": al is not None,
                     "flops_per_launch": fl,
                     "avg_launch_ms": round(t / n, 4)}
    Bd, Hqd, Dd = dq.shape
    lens = dec.kv_lens.to(dev)
    att = sum(min(int(n_), Wl + 1) for n_ in dec.kv_lens.tolist())
    dbytes = att * dec.n_kv * Dd * 2 * 2 + dq.numel() * 2 + Bd * Hqd * (Dd + 1) * 4
    # The split count for the tokens the window keeps (the policy on the
    # attended length), not for the whole cache.
    Sw = attn.decode_num_splits(Bd, dec.n_kv, min(int(dec.kv_lens.max()), Wl + 1))
    opw = torch.empty((Sw, Bd, Hqd, Dd), dtype=torch.float32, device=dev)
    lpw = torch.empty((Sw, Bd, Hqd), dtype=torch.float32, device=dev)
    t_dec = timed(lambda i: attn.decode_splitkv(dq, caches[i % len(caches)][0],
                                                caches[i % len(caches)][1], lens, None,
                                                num_splits=Sw, scale=dec.scale, o_partial=opw,
                                                lse_partial=lpw, window_left=Wl),
                  before=lambda: torch.sum(sweep, dim=0, out=sweep_out))
    return {"prefill": pre,
            "decode": {"value": round(job_rate(dbytes, n, world, t_dec) / 1e9, 1), "unit": "GB/s",
                       "window_left": Wl, "bytes_per_launch": dbytes, "num_splits": Sw,
                       "avg_launch_us": round(t_dec / n * 1e3, 2)}}


def time_d256(args, attn, W, dist, dev):
    """Causal prefill with head_dim 256 at a Gemma-2-9B-like attention shape
    (N = 8192, 16 query / 8 kv heads); inputs and output exceed L2."""
    import torch

    Hq, Hkv, N, D = 16, 8, 8192, 256
    x = W.make_prefill(1, Hq, Hkv, N, D, seed=0)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o = torch.empty((1, Hq, N, D), dtype=torch.float32, device=dev)
    lse = torch.empty((1, Hq, N), dtype=torch.float32, device=dev)
    flops = prefill_flops(Hq, N, D)
    n = max(3, min(args.steps, 100))
    for _ in range(3):
        attn.prefill(q, k, v, x.scale, True, out=o, lse=lse)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        evs[i][0].record()
        attn.prefill(q, k, v, x.scale, True, out=o, lse=lse)
        evs[i][1].record()
    torch.cuda.synchronize()
    attn.check_device_status()
    (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    world = dist.get_world_size() if dist is not None else 1
    avg_ms = tot / n
    res = {"value": round(job_rate(flops, n, world, tot) / 1e12, 2), "unit": "TFLOP/s",
           "shape": "N=8192, 16/8 heads, head_dim 256, causal",
           "roofline": {"bound": "tensor", "achieved": round(flops / (avg_ms * 1e-3) / 1e12, 2),
                        "unit": "TFLOP/s", "kernel": "prefill_kernel<256>",
                        "flops_per_launch": flops, "avg_launch_ms": round(avg_ms, 4)}}
    del q, k, v, o, lse, x

    # Split-KV decode at the same head shape over a contiguous 30720-token
    # cache (251 MB of K and V, two copies in rotation: every launch reads HBM).
    L = 30720
    dd = W.make_decode_contiguous(1, Hq, Hkv, D, L, seed=1, max_kv_len=L)
    dq, dlens = dd.q.to(dev), dd.kv_lens.to(dev)
    caches = [(dd.k_cache.to(dev), dd.v_cache.to(dev)) for _ in range(2)]
    S = attn.decode_num_splits(1, Hkv, L)
    op = torch.empty((S, 1, Hq, D), dtype=torch.float32, device=dev)
    lp = torch.empty((S, 1, Hq), dtype=torch.float32, device=dev)
    do = torch.empty((1, Hq, D), dtype=torch.float32, device=dev)
    dl = torch.empty((1, Hq), dtype=torch.float32, device=dev)
    dbytes = L * Hkv * D * 2 * 2 + dq.numel() * 2 + do.numel() * 4 + dl.numel() * 4

    def dec(i, ev=None, with_combine=True):
        # events around decode + combine, or around the decode alone: never
        # between the two (it would stop the combine's early launch)
        kc, vc = caches[i % 2]
        if ev is not None:
            ev[0].record()
        attn.decode_splitkv(dq, kc, vc, dlens, None, num_splits=S, max_kv_len=L, scale=dd.scale,
                            o_partial=op, lse_partial=lp)
        if with_combine:
            attn.combine(op, lp, out=do, lse=dl)
        if ev is not None:
            ev[1].record()

    for i in range(3):
        dec(i)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    evd = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        dec(i, evs[i])
    for i in range(n):
        dec(i, evd[i], with_combine=False)
    torch.cuda.synchronize()
    attn.check_device_status()
    dec_ms = [e[0].elapsed_time(e[1]) for e in evd]
    both_ms = [e[0].elapsed_time(e[1]) for e in evs]
    (tot_d,) = rank_max(dist, [sum(both_ms)], dev)
    avg_d = statistics.mean(dec_ms)
    res["decode"] = {"value": round(job_rate(dbytes, n, world, tot_d) / 1e9, 1), "unit": "GB/s",
                     "shape": f"1 x 30720 tokens, 16/8 heads, head_dim 256, {S} splits",
                     "roofline": {"bound": "hbm", "achieved": round(dbytes / (avg_d * 1e-3) / 1e9, 1),
                                  "unit": "GB/s", "kernel": "decode_splitkv_kernel<256>",
                                  "bytes_per_launch": dbytes,
                                  "avg_launch_us": round(avg_d * 1e3, 2),
                                  "decode_plus_combine_avg_us": round(statistics.mean(both_ms) * 1e3, 2)}}
    return res


def time_d64(args, attn, W, dist, dev):
    """Causal prefill with head_dim 64 (N = 8192, 32 query / 8 kv heads).
    Against head_dim 128 the products per key tile halve while the softmax's
    cost per score stays, so the softmax sets the rate."""
    import torch

    Hq, Hkv, N, D = 32, 8, 8192, 64
    x = W.make_prefill(1, Hq, Hkv, N, D, seed=0)
    q, k, v = x.q.to(dev), x.k.to(dev), x.v.to(dev)
    o = torch.empty((1, Hq, N, D), dtype=torch.float32, device=dev)
    lse = torch.empty((1, Hq, N), dtype=torch.float32, device=dev)
    flops = prefill_flops(Hq, N, D)
    n = max(3, min(args.steps, 100))
    for _ in range(3):
        attn.prefill(q, k, v, x.scale, True, out=o, lse=lse)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        evs[i][0].record()
        attn.prefill(q, k, v, x.scale, True, out=o, lse=lse)
        evs[i][1].record()
    torch.cuda.synchronize()
    attn.check_device_status()
    (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    world = dist.get_world_size() if dist is not None else 1
    avg_ms = tot / n
    res = {"value": round(job_rate(flops, n, world, tot) / 1e12, 2), "unit": "TFLOP/s",
           "shape": "N=8192, 32/8 heads, head_dim 64, causal",
           "roofline": {"bound": "tensor", "achieved": round(flops / (avg_ms * 1e-3) / 1e12, 2),
                        "unit": "TFLOP/s", "kernel": "prefill_kernel<64>",
                        "flops_per_launch": flops, "avg_launch_ms": round(avg_ms, 4)}}
    # The same shape in FP8 (block scales, rotation): the 128-column FP8
    # kernel, its copies reading zeros past column 64.
    g = torch.Generator().manual_seed(1)
    signs = torch.where(torch.rand(D, generator=g) < 0.5, -1.0, 1.0).to(torch.float32).to(dev)
    q8, qs = attn.quantize_fp8(q, signs, block_rows=128)
    k8, ks = attn.quantize_fp8(k, signs, block_rows=128)
    v8t, vs = attn.quantize_fp8(v, None, block_rows=0, transpose=True)
    for _ in range(3):
        attn.prefill_fp8(q8, k8, v8t, qs, ks, vs, x.scale, True, out=o, lse=lse)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        evs[i][0].record()
        attn.prefill_fp8(q8, k8, v8t, qs, ks, vs, x.scale, True, out=o, lse=lse)
        evs[i][1].record()
    torch.cuda.synchronize()
    attn.check_device_status()
    (tot8,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    res["fp8"] = {"value": round(job_rate(flops, n, world, tot8) / 1e12, 2), "unit": "TFLOP/s",
                  "kernel": "prefill_kernel<128, fp8> over 64 columns",
                  "avg_launch_ms": round(tot8 / n, 4),
                  "vs_bf16": round(tot / tot8, 3)}
    return res


def time_fp8(args, attn, x, q, k, v, o, lse, dist, dev):
    """FP8 prefill on the step's shape: the quantiser (rotation + block scales
    for Q and K, per-head scale for V, transposed) runs once outside the
    prefill's events and is timed on its own.  Accuracy: rms of O against the
    bf16 path's O, for naive FP8 (one scale per head, no rotation) and for
    block scales with the rotation."""
    import torch

    B, Hq, N, D = q.shape
    flops = prefill_flops(Hq, N, D, B)
    n = max(3, min(args.steps, 100))
    world = dist.get_world_size() if dist is not None else 1
    g = torch.Generator().manual_seed(11)
    signs = torch.where(torch.rand(D, generator=g) < 0.5, -1.0, 1.0).to(torch.float32).to(dev)

    def quantize(qq, kk, sg, block):
        q8, qs = attn.quantize_fp8(qq, sg, block_rows=block)
        k8, ks = attn.quantize_fp8(kk, sg, block_rows=block)
        v8t, vs = attn.quantize_fp8(v, None, block_rows=0, transpose=True)
        if block == 0:
            nb = -(-N // 128)
            qs = qs.unsqueeze(-1).expand(*qs.shape, nb).contiguous()
            ks = ks.unsqueeze(-1).expand(*ks.shape, nb).contiguous()
        return q8, k8, v8t, qs, ks, vs

    qin = quantize(q, k, signs, 128)
    o8 = torch.empty_like(o)
    l8 = torch.empty_like(lse)
    for _ in range(3):
        attn.prefill_fp8(*qin, x.scale, True, out=o8, lse=l8)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        evs[i][0].record()
        attn.prefill_fp8(*qin, x.scale, True, out=o8, lse=l8)
        evs[i][1].record()
    torch.cuda.synchronize()
    (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    # The quantiser on its own, into preallocated outputs, captured in a CUDA
    # graph so that the events time the kernels rather than the Python calls;
    # L2 is flushed (a write of 2x L2) outside the events before every replay.
    # Two forms: the fused call for Q, K and V (attn_quantize_fp8_qkv: three
    # launches), and the three separate calls (six launches).
    flush = torch.empty(2 * (int(torch.cuda.get_device_properties(dev).L2_cache_size) or (128 << 20)),
                        dtype=torch.uint8, device=dev)

    def graph_us(fn):
        fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(10)]
        for qa, qb in qev:
            flush.zero_()
            qa.record()
            graph.replay()
            qb.record()
        torch.cuda.synchronize()
        return statistics.median(qa.elapsed_time(qb) for qa, qb in qev) * 1e3

    outs = [torch.empty_like(t) for t in qin]
    fused = tuple(torch.empty_like(t) for t in qin)

    def quantize_into():
        attn.quantize_fp8(q, signs, 128, codes=outs[0], scales=outs[3])
        attn.quantize_fp8(k, signs, 128, codes=outs[1], scales=outs[4])
        attn.quantize_fp8(v, None, 0, True, codes=outs[2], scales=outs[5])

    quant_sep_us = graph_us(quantize_into)
    quant_us = graph_us(lambda: attn.quantize_fp8_qkv(q, k, v, signs, out=fused))
    assert all(torch.equal(a_, b_) for a_, b_ in zip(outs, qin)), "graph replay differs"
    assert all(torch.equal(a_, b_) for a_, b_ in zip(fused, qin)), "fused quantiser differs"
    del flush
    # algorithmic bytes: every element read once (bf16) and written once (e4m3)
    quant_bytes = (q.numel() + k.numel() + v.numel()) * 3
    # accuracy against the bf16 path, on queries and keys with four outlier
    # channels (x20): the structure the rotation is for (iid Gaussian inputs
    # have none, and there both schemes err alike)
    q_o, k_o = q.clone(), k.clone()
    q_o[..., :4] *= 20.0
    k_o[..., :4] *= 20.0
    attn.prefill(q_o, k_o, v, x.scale, True, out=o, lse=lse)
    ref = o.clone()
    rms = {}
    for name, sg, block in (("naive", None, 0), ("block+rotation", signs, 128)):
        attn.prefill_fp8(*quantize(q_o, k_o, sg, block), x.scale, True, out=o8, lse=l8)
        rms[name] = float(torch.sqrt(torch.mean((o8 - ref) ** 2)))
    attn.check_device_status()
    avg_ms = tot / n
    return {"value": round(job_rate(flops, n, world, tot) / 1e12, 2), "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": round(flops / (avg_ms * 1e-3) / 1e12, 2),
                         "unit": "TFLOP/s", "kernel": "prefill_kernel<128, fp8>",
                         "flops_per_launch": flops, "avg_launch_ms": round(avg_ms, 4)},
            "quantize_us": round(quant_us, 1),
            "quantize_gbs": round(quant_bytes / (quant_us * 1e-6) / 1e9, 1),
            "quantize_bytes": quant_bytes,
            "quantize_form": "attn_quantize_fp8_qkv (Q, K and V's amax in one launch; then V's "
                             "codes and scales)",
            "quantize_separate_calls_us": round(quant_sep_us, 1),
            "rms_vs_bf16": {k_: round(v_, 6) for k_, v_ in rms.items()},
            "error_ratio_naive_over_block_rotation": round(rms["naive"] / rms["block+rotation"], 2)}


def time_prefill_varlen(args, attn, W, dist, dev):
    """Packed variable-length prefill of 16 prompts (lengths uniform in
    [256, 4096], 28 / 4 heads, head_dim 128): inputs (262 MB of Q) and the
    output exceed L2, so consecutive launches do not reuse cached data."""
    import torch

    x = W.qwen_varlen_prefill()
    q, k, v, cu = x.q.to(dev), x.k.to(dev), x.v.to(dev), x.cu_seqlens.to(dev)
    n_q, T, d = x.q.shape
    o = torch.empty((n_q, T, d), dtype=torch.float32, device=dev)
    lse = torch.empty((n_q, T), dtype=torch.float32, device=dev)
    lens = (x.cu_seqlens[1:] - x.cu_seqlens[:-1]).tolist()
    flops = sum(prefill_flops(n_q, n, d) for n in lens)
    n = max(3, min(args.steps, 100))
    for _ in range(3):
        attn.prefill_varlen(q, k, v, cu, x.scale, True, out=o, lse=lse)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        evs[i][0].record()
        attn.prefill_varlen(q, k, v, cu, x.scale, True, out=o, lse=lse)
        evs[i][1].record()
    torch.cuda.synchronize()
    attn.check_device_status()
    (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    world = dist.get_world_size() if dist is not None else 1
    avg_ms = tot / n
    res = {"value": round(job_rate(flops, n, world, tot) / 1e12, 2), "unit": "TFLOP/s",
           "roofline": {"bound": "tensor", "achieved": round(flops / (avg_ms * 1e-3) / 1e12, 2),
                        "unit": "TFLOP/s", "kernel": "prefill_kernel<128, packed>",
                        "flops_per_launch": flops, "avg_launch_ms": round(avg_ms, 4)},
           "num_seqs": len(lens), "total_tokens": T, "launches": n}
    del q, k, v, o, lse
    # Packed FP8 on the same prompts with their lengths rounded up to 16 rows
    # (the FP8 path needs every sequence to start at a multiple of 16), beside
    # the bf16 packed kernel on those lengths; the quantiser runs outside the
    # events.
    lens16 = [-(-n_ // 16) * 16 for n_ in lens]
    x16 = W.make_prefill_varlen(lens16, n_q, x.k.shape[0], d, seed=0)
    q, k, v, cu = x16.q.to(dev), x16.k.to(dev), x16.v.to(dev), x16.cu_seqlens.to(dev)
    T16 = x16.q.shape[1]
    o = torch.empty((n_q, T16, d), dtype=torch.float32, device=dev)
    lse = torch.empty((n_q, T16), dtype=torch.float32, device=dev)
    g = torch.Generator().manual_seed(11)
    signs = torch.where(torch.rand(d, generator=g) < 0.5, -1.0, 1.0).to(torch.float32).to(dev)
    q8, qs = attn.quantize_fp8_varlen(q, cu, signs)
    k8, ks = attn.quantize_fp8_varlen(k, cu, signs)
    v8t, vs = attn.quantize_fp8(v, None, block_rows=0, transpose=True)
    flops16 = sum(prefill_flops(n_q, n_, d) for n_ in lens16)
    t16 = {}
    for name, fn in (("bf16", lambda: attn.prefill_varlen(q, k, v, cu, x16.scale, True, out=o,
                                                           lse=lse)),
                     ("fp8", lambda: attn.prefill_fp8_varlen(q8, k8, v8t, qs, ks, vs, cu,
                                                              x16.scale, True, out=o, lse=lse))):
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        torch.cuda.synchronize()
        for i in range(n):
            evs[i][0].record()
            fn()
            evs[i][1].record()
        torch.cuda.synchronize()
        (t16[name],) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    attn.check_device_status()
    res["fp8_packed"] = {
        "value": round(job_rate(flops16, n, world, t16["fp8"]) / 1e12, 2), "unit": "TFLOP/s",
        "bf16_same_lengths": round(job_rate(flops16, n, world, t16["bf16"]) / 1e12, 2),
        "speedup_over_bf16": round(t16["bf16"] / t16["fp8"], 3),
        "lengths": "the packed prompts' lengths rounded up to multiples of 16",
        "kernel": "prefill_kernel<128, packed, fp8>", "flops_per_launch": flops16,
        "avg_launch_ms": round(t16["fp8"] / n, 4)}
    return res


def time_decode_append(args, attn, dq, caches, dec, S, op, lp, sweep, sweep_out, dist, dev):
    """Decode with in-place append on the decode workload's shape: kv_len - 1
    cached tokens plus the appended one, so the same number of tokens is
    attended.  Timed like the step's decode (a read-only L2 sweep before each
    launch, outside its events; the cache copies rotate)."""
    import torch

    if dec.block_table is not None:
        return None  # measured on the contiguous single-sequence workload only
    n = max(3, min(args.steps, 200))
    B, Hq, D = dq.shape
    lens = (dec.kv_lens - 1).clamp(min=0).to(dev)
    g = torch.Generator().manual_seed(1)
    kn = torch.randn(B, dec.n_kv, D, generator=g).to(torch.bfloat16).to(dev)
    vn = torch.randn(B, dec.n_kv, D, generator=g).to(torch.bfloat16).to(dev)

    def launch(i):
        kc, vc = caches[i % len(caches)]
        attn.decode_append_splitkv(dq, kn, vn, kc, vc, lens, None, num_splits=S,
                                   scale=dec.scale, o_partial=op, lse_partial=lp)

    for i in range(3):
        launch(i)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    for i in range(n):
        torch.sum(sweep, dim=0, out=sweep_out)
        evs[i][0].record()
        launch(i)
        evs[i][1].record()
    torch.cuda.synchronize()
    attn.check_device_status()
    (tot,) = rank_max(dist, [sum(a.elapsed_time(b) for a, b in evs)], dev)
    tokens = int(dec.kv_lens.sum())
    # K and V of every attended token (the appended one is read back from the
    # cache), q, the new rows read and written, the final O and LSE.
    nbytes = tokens * dec.n_kv * D * 2 * 2 + dq.numel() * 2 + 2 * 2 * kn.numel() * 2 + \
        B * Hq * (D + 1) * 4
    avg_us = tot / n * 1e3
    world = dist.get_world_size() if dist is not None else 1
    return {"value": round(job_rate(nbytes, n, world, tot) / 1e9, 1), "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": round(nbytes / (avg_us * 1e-6) / 1e9, 1),
                         "unit": "GB/s", "kernel": "decode_splitkv_kernel<128> (append)",
                         "bytes_per_launch": nbytes, "avg_launch_us": round(avg_us, 2)},
            "tokens_attended": tokens, "launches": n}


def run_e2e(args, x, dec, dev, world, dist):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device and its results device->host.  Steps are
    pipelined as a serving loop runs them: three streams (input copies, the
    library's kernels, result copies) and two device buffer sets, so step
    i+1's inputs travel while step i computes and step i-1's results return.
    The timed region runs from before the first input copy to after the last
    result copy, so every step's copies are inside it.  Prefill steps (one
    Llama-3-8B layer at N = 32768 each) and decode steps (one Qwen2.5-7B layer
    over its 30720-token cache, copied from the host each step) are timed as
    two separate loops."""
    import torch

    import exact_io_aware_order_gb300 as attn

    pin = lambda t: t.contiguous().pin_memory()
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def pipelined(n, inputs, results, compute):
        """inputs: [(host, (dev0, dev1))]; results: [((dev0, dev1), (host0, host1))];
        compute(b) launches step's kernels on the current stream for buffer b."""
        in_done = [torch.cuda.Event() for _ in range(2)]
        c_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = _ev(), _ev()
        torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(c_done[b])    # step i-2's kernels have read buffer b
                for h, d in inputs:
                    d[b].copy_(h, non_blocking=True)
                in_done[b].record(s_in)
            with torch.cuda.stream(s_c):
                s_c.wait_event(in_done[b])
                if i >= 2:
                    s_c.wait_event(out_done[b])   # step i-2's results have left buffer b
                compute(b)
                c_done[b].record(s_c)
            with torch.cuda.stream(s_out):
                s_out.wait_event(c_done[b])
                for d, h in results:
                    h[b].copy_(d[b], non_blocking=True)
                out_done[b].record(s_out)
        s_out.wait_event(in_done[(n - 1) & 1])
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    two = lambda t: (torch.empty_like(t, device=dev), torch.empty_like(t, device=dev))
    flops = prefill_flops(x.q.shape[1], x.q.shape[2], x.q.shape[3])
    # ---- prefill ----
    hq, hk, hv = pin(x.q), pin(x.k), pin(x.v)
    ho = [torch.empty(tuple(x.q.shape), dtype=torch.float32).pin_memory() for _ in range(2)]
    hl = [torch.empty(tuple(x.q.shape[:3]), dtype=torch.float32).pin_memory() for _ in range(2)]
    q, k, v = two(hq), two(hk), two(hv)
    o = tuple(torch.empty(ho[0].shape, dtype=torch.float32, device=dev) for _ in range(2))
    lse = tuple(torch.empty(hl[0].shape, dtype=torch.float32, device=dev) for _ in range(2))
    pf = lambda b: attn.prefill(q[b], k[b], v[b], x.scale, True, out=o[b], lse=lse[b])
    p_in = [(hq, q), (hk, k), (hv, v)]
    p_out = [(o, ho), (lse, hl)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * 4 + hl[0].numel() * 4
    n = max(3, min(args.steps, args.e2e_steps))
    pipelined(2, p_in, p_out, pf)            # warm-up

    def copy_gbs(pairs, to_dev):
        """This box's copy rate for one step's inputs (to_dev) or results, alone."""
        e0, e1 = _ev(), _ev()
        torch.cuda.synchronize()
        e0.record()
        for h, d in pairs:
            (d[0].copy_(h, non_blocking=True) if to_dev else h[0].copy_(d[0], non_blocking=True))
        e1.record()
        torch.cuda.synchronize()
        return round((h2d if to_dev else d2h) / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)

    copy_rates = {"h2d_gbs": copy_gbs(p_in, True), "d2h_gbs": copy_gbs(p_out, False)}
    if dist is not None:
        dist.barrier()
    pre = pipelined(n, p_in, p_out, pf)
    attn.check_device_status()
    # The same loop with the kernels alone and with the copies alone: whether
    # this box overlapped the copies with the kernels (their sum against the
    # whole) is part of the end-to-end number.
    parts = {"kernels_only": pipelined(n, [], [], pf) / n,
             "copies_only": pipelined(n, p_in, p_out, lambda b: None) / n,
             "whole": pre / n}
    parts = {k_: round(v_, 3) for k_, v_ in parts.items()}
    # the results are the library's: the last step's output equals a direct call
    ref_o, _ = attn.prefill(q[0], k[0], v[0], x.scale, True)
    assert torch.equal(ho[(n - 1) & 1], ref_o.cpu()), "pipelined e2e result differs"
    del q, k, v, o, lse, ref_o, hq, hk, hv, ho, hl
    torch.cuda.empty_cache()
    # ---- decode ----
    hdq, hkc, hvc, hlen = pin(dec.q), pin(dec.k_cache), pin(dec.v_cache), pin(dec.kv_lens)
    B, Hq, D = dec.q.shape
    S = attn.decode_num_splits(B, dec.n_kv, dec.max_kv_len)
    hdo = [torch.empty((B, Hq, D), dtype=torch.float32).pin_memory() for _ in range(2)]
    hdl = [torch.empty((B, Hq), dtype=torch.float32).pin_memory() for _ in range(2)]
    dq, kc, vc, dlen = two(hdq), two(hkc), two(hvc), two(hlen)
    op = tuple(torch.empty((S, B, Hq, D), dtype=torch.float32, device=dev) for _ in range(2))
    lp = tuple(torch.empty((S, B, Hq), dtype=torch.float32, device=dev) for _ in range(2))
    do = tuple(torch.empty((B, Hq, D), dtype=torch.float32, device=dev) for _ in range(2))
    dlo = tuple(torch.empty((B, Hq), dtype=torch.float32, device=dev) for _ in range(2))

    def dc(b):
        attn.decode_splitkv(dq[b], kc[b], vc[b], dlen[b], None, num_splits=S,
                            max_kv_len=dec.max_kv_len, scale=dec.scale, o_partial=op[b],
                            lse_partial=lp[b])
        attn.combine(op[b], lp[b], out=do[b], lse=dlo[b])

    d_in = [(hdq, dq), (hkc, kc), (hvc, vc), (hlen, dlen)]
    d_out = [(do, hdo), (dlo, hdl)]
    h2d_dec = sum(h.numel() * h.element_size() for h, _ in d_in)
    d2h_dec = hdo[0].numel() * 4 + hdl[0].numel() * 4
    pipelined(2, d_in, d_out, dc)
    if dist is not None:
        dist.barrier()
    dcd = pipelined(n, d_in, d_out, dc)
    attn.check_device_status()
    pre, dcd = rank_max(dist, [pre, dcd], dev)
    return {"value": round(job_rate(flops, n, world, pre) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "what": "one Llama-3-8B-layer causal prefill at N = 32768 per step, Q/K/V copied "
                    "in and O/LSE copied out every step",
            "pipelining": "3 streams (H2D / kernels / D2H), 2 buffer sets",
            "copy_rates_alone": copy_rates,
            "ms_per_step_parts": parts,
            # settings that decide whether streams can overlap (unset: the defaults)
            "stream_env": {k_: os.environ.get(k_) for k_ in ("CUDA_DEVICE_MAX_CONNECTIONS",
                                                              "CUDA_LAUNCH_BLOCKING")},
            "decode_value": round(job_rate(decode_bytes(dec), n, world, dcd) / 1e9, 1),
            "decode_unit": "GB/s (end to end, cache copied from host each step)",
            "decode_h2d_bytes_per_step": h2d_dec, "decode_d2h_bytes_per_step": d2h_dec}


# ---------------------------------------------------------------------------
# The float64 CPU oracle (cpu_baseline leg and --impl reference).
# ---------------------------------------------------------------------------
def _cpu_worker(spec: dict) -> dict:
    """Runs inside a fresh interpreter with BLAS threads pinned: times the
    oracle on the requested sample of the headline workload and returns
    throughput figures."""
    import numpy as np

    from exact_io_aware_order_gb300 import workloads as W
    import oracle

    P = HEADLINE["prefill"]
    x = W.llama_long_prefill(P["seqlen"])
    out = {}
    if spec["kind"] == "heads":
        h = spec["heads"]
        g = P["n_q"] // P["n_kv"]
        nkv = -(-h // g)
        t0 = time.perf_counter()
        oracle.prefill(x.q[:, :h], x.k[:, :nkv], x.v[:, :nkv], x.scale, True)
        dt = time.perf_counter() - t0
        fl = prefill_flops(h, P["seqlen"], P["d"])
        out["prefill_tflops"] = fl / dt / 1e12
        out["prefill_s"] = dt
        out["sample"] = f"all {P['seqlen']} rows of {h} of {P['n_q']} query heads"
    else:  # per-step sampled rows, repeated
        N = P["seqlen"]
        rows = [(0, 0, int(i)) for i in np.linspace(0, N - 1, spec["rows"]).round()]
        fl = sum(4.0 * (i + 1) * P["d"] for _, _, i in rows)
        times = []
        for _ in range(spec["repeats"]):
            t0 = time.perf_counter()
            oracle.prefill_rows(x.q, x.k, x.v, x.scale, True, rows)
            times.append(time.perf_counter() - t0)
        out["prefill_tflops"] = fl * len(times) / sum(times) / 1e12
        out["prefill_s"] = sum(times)
        out["step_times"] = times
        out["sample"] = f"{spec['rows']} evenly spaced rows of query head 0 per step"
    if spec.get("decode", True):
        dec = W.qwen_decode(HEADLINE["decode"]["kv_len"])
        lens = dec.kv_lens.tolist()
        t0 = time.perf_counter()
        oracle.decode(dec.q, dec.k_cache, dec.v_cache, None, lens, dec.scale)
        dt = time.perf_counter() - t0
        out["decode_gbs"] = decode_bytes(dec) / dt / 1e9
        out["decode_s"] = dt
    return out


def run_cpu(spec: dict) -> dict:
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(cores), OMP_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", json.dumps(spec)],
                       env=env, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle worker failed:\n" + r.stderr[-2000:])
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = cores
    return out


def run_reference(args, rank: int, world: int):
    """Times the float64 oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return None
    import numpy as np

    P = HEADLINE["prefill"]
    rows = 32
    spec = {"kind": "rows", "rows": rows, "repeats": args.warmup + args.steps, "decode": False}
    r = run_cpu(spec)
    times = r["step_times"][args.warmup:]
    fl = sum(4.0 * (i + 1) * P["d"] for i in np.linspace(0, P["seqlen"] - 1, rows).round())
    value = fl * len(times) / sum(times) / 1e12
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": headline_config(world),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": r["cores"],
                             "kind": "oracle", "sample": r["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the timed headline steps (for profiling runs)")
    ap.add_argument("--legs", type=str, default="all",
                    help="comma list of the legs after the timed steps to run: workloads, append, "
                         "varlen, fp8, d256 (head_dims 256 and 64), variants (for profiling "
                         "runs); default all")
    ap.add_argument("--seqlen", type=int, default=HEADLINE["prefill"]["seqlen"],
                    help="prefill length of the timed step (profiling runs use a smaller one)")
    ap.add_argument("--layers", type=int, default=HEADLINE["prefill"]["layers"],
                    help="prefill launches per timed step")
    ap.add_argument("--cpu-heads", type=int, default=2,
                    help="query heads in the cpu_baseline sample (whole rows, N tokens)")
    ap.add_argument("--cpu-worker", type=str, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()

    if args.cpu_worker is not None:
        print(json.dumps(_cpu_worker(json.loads(args.cpu_worker))))
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    HEADLINE["prefill"]["seqlen"] = args.seqlen
    HEADLINE["prefill"]["layers"] = args.layers
    if (args.seqlen, args.layers) != (32768, 32):
        HEADLINE["desc"] = (f"profiling case: Llama-3-8B attention, causal prefill N={args.seqlen} "
                            f"x {args.layers} layers + the decode chain of the headline")
    rank, world = rank_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    # The CPU baseline runs before the first GPU call (its worker is a fresh
    # interpreter either way), on rank 0 at N = 1 only.
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        spec = {"kind": "heads", "heads": args.cpu_heads}
        r = run_cpu(spec)
        cpu = {"value": round(r["prefill_tflops"], 6), "unit": "TFLOP/s", "cores": r["cores"],
               "kind": "oracle", "sample": r["sample"] + "; float64 numpy, BLAS threads = cores",
               "seconds": round(r["prefill_s"], 2),
               "decode_value": round(r["decode_gbs"], 3), "decode_unit": "GB/s",
               "decode_seconds": round(r["decode_s"], 2)}

    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist_mod.init_process_group("nccl")
        dist = dist_mod
    res = run_gb300(args, rank, world, dist)
    if cpu is not None:
        res["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
