"""Benchmark: one step of the KIVI hot path on the Llama-3-8B attention-layer
workload (batch 8, 32 query / 8 KV heads, d = 128, 32768 context, 2-bit,
G = 32, R = 128).

A step is the whole path through the C ABI, inputs resident in HBM:
  1. kivi_quantize_prefill of the 32768 fp16 tokens into a fresh cache
     (keys per channel / values per token, packing, residual window),
  2. kivi_append_token of one new token (the residual is full, so this
     flushes 128 tokens into the quantised history first),
  3. kivi_decode_attention (one kernel: history splits, residual, merge).
`value` is the decode attention's effective GB/s: algorithmic bytes the
decode reads and writes (packed codes, scales/zero points, fp16 residual,
q and o) divided by its CUDA-event time.  Before each decode, untimed, a
256 MiB write flushes L2 and a 512 MiB read evicts the dirty lines the write
left, so the decode starts on a cold, clean L2; the prefill reads 1 GiB of
fp16 input, far above the 129 MB L2.

--impl reference times the CPU oracle (the plain C restatement of the
pages' method used by the tests) on a bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "quant-KV decode attn effective GB/s (% HBM peak), µs/step; quantize GB/s"
WORKLOAD = "llama3-8b-layer-32k-2bit"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_split_llama3-8b-layer-32k-2bit.txt")


def bytes_per_quant_token(bits, G, d=128, meta=0):
    """Algorithmic bytes of one quantised token of one (batch, kv-head) pair:
    key and value codes plus scale/zero metadata (fp32, or fp16 with meta=1);
    FP8 KV (bits 8): one byte per element, per-tensor scales."""
    if bits == 8:
        return 2 * d
    mw = 2 if meta else 4
    codes = 2 * d * bits // 8
    kmeta = 2 * d * mw / G         # per-channel (s, z) shared by G tokens
    vmeta = 2 * (d // G) * mw      # per-token (s, z) per channel group
    return codes + kmeta + vmeta


def decode_bytes(w, n_quant, n_resid, meta=0, n_sink=0):
    """Algorithmic bytes of one decode: packed codes and metadata of every
    quantised token, the fp16 rows (residual and sink), q read and o written."""
    per_pair = n_quant * bytes_per_quant_token(w.bits, w.G, w.d, meta) \
        + (n_resid + n_sink) * 2 * w.d * 2
    qo = 2 * w.B * w.Hq * w.d * 2
    return w.pairs * per_pair + qo


def prefill_bytes(w, T, nq_new, r_new, meta=0, n_sink=0):
    per_pair = T * 2 * w.d * 2 + nq_new * bytes_per_quant_token(w.bits, w.G, w.d, meta) \
        + (r_new + n_sink) * 2 * w.d * 2
    return w.pairs * per_pair


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def source_digest():
    """Digest of the sources of the decode kernel the roofline line times."""
    import hashlib
    h = hashlib.sha256()
    for f in ("kivi_decode_kernels.cuh", "kivi_decode.cu", "kivi_internal.cuh"):
        with open(os.path.join(ROOT, "bit_kv_cache_06_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic():
    """DRAM bytes per decode-split launch from the committed ncu summary, or
    None when the summary is missing or was taken on a different source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    vals = {}
    with open(PROFILE_TRAFFIC) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_digest") != source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(vals, world, device):
    """Element-wise maximum of per-rank timings over all ranks: the slowest
    rank sets the job's time (weak scaling, no data exchange between ranks)."""
    if world <= 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def whole_job_gbs(world, bytes_per_rank, ms):
    """Whole-job throughput: every rank moved bytes_per_rank in at most ms."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ our arm ----

def run_ours(args, rank, world, local_rank):
    import numpy as np  # noqa: F401

    from bit_kv_cache_06_gb300 import build as kbuild
    from bit_kv_cache_06_gb300 import kivi, synth

    kbuild.build()
    kivi.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = synth.CONFIGS[args.config]
    stream = torch.cuda.current_stream()

    # per-rank shard: an independent batch of the same shape (weak scaling)
    K, V = synth.make_kv(w, layer=rank, device=dev)
    q = synth.make_q(w, layer=rank, device=dev)
    k_new, v_new = synth.make_token(w, 0, layer=rank, device=dev)
    out = torch.empty_like(q)
    cache = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                           w.capacity()), device=dev)
    # L2 flush before each decode (untimed): a 256 MiB write pushes out every
    # line of the cache, a 512 MiB read then evicts the dirty lines that write
    # left, so the decode starts on a cold L2 without paying for their
    # write-back inside its own timed region
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_evict = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)

    def flush_l2():
        l2_flush.zero_()
        l2_evict.amax()

    def step(ev):
        # the flush also keeps the device busy while the host enqueues the
        # prefill, so its events bracket device work only
        flush_l2()
        ev[0].record(stream)
        cache.reset()
        cache.quantize_prefill(K, V)
        ev[1].record(stream)
        cache.append_token(k_new, v_new)
        ev[2].record(stream)
        flush_l2()
        ev[3].record(stream)
        cache.decode_attention(q, out)       # one fused kernel: splits + merge
        ev[4].record(stream)

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(5)]

    for _ in range(args.warmup):
        step(new_events())
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(1.0)                  # nvidia-smi needs a moment to start sampling
    launches0 = cache.kernel_launches
    evs = [new_events() for _ in range(args.steps)]
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    launches = cache.kernel_launches - launches0

    pre = [e[0].elapsed_time(e[1]) for e in evs]
    app = [e[1].elapsed_time(e[2]) for e in evs]
    dec = [e[3].elapsed_time(e[4]) for e in evs]
    step_ms = statistics.mean(a + b + c for a, b, c in zip(pre, app, dec))
    dec_ms = statistics.mean(dec)
    pre_ms = statistics.mean(pre)

    n_quant, n_resid = cache.n_quant, cache.n_resid
    T = w.T
    r_new = ((T - 1) % w.R) + 1
    dbytes = decode_bytes(w, n_quant, n_resid)
    pbytes = prefill_bytes(w, T, T - r_new, r_new)

    # max over ranks of the per-step times
    step_ms, dec_ms, pre_ms, wall = max_over_ranks([step_ms, dec_ms, pre_ms, wall], world, dev)

    value = whole_job_gbs(world, dbytes, dec_ms)
    kernel_gbs = whole_job_gbs(1, dbytes, dec_ms)      # one rank's decode kernel
    quant_gbs = whole_job_gbs(world, pbytes, pre_ms)
    peak, peak_kind = load_peaks()

    # the decode in the other steady state: right after the prefill, with the
    # residual window full (n_resid = R, 128 more fp16 tokens per pair)
    cache.reset()
    cache.quantize_prefill(K, V)
    full_state = {"n_quant": cache.n_quant, "n_resid": cache.n_resid}
    full_ms = statistics.mean(time_calls(lambda: cache.decode_attention(q, out), 20, stream,
                                         before=flush_l2))
    full_bytes = decode_bytes(w, cache.n_quant, cache.n_resid)
    full_ms = max_over_ranks([full_ms], world, dev)[0]
    full_gbs = full_bytes / (full_ms * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: H2D of the step's inputs
    # from pinned memory, the same calls, D2H of the output
    e2e = run_e2e(cache, w, K, V, q, k_new, v_new, out, stream, dbytes, args, world)

    splits = cache.num_splits(0)
    per_config = None
    if world == 1 and args.config == "c2" and not args.headline_only:
        del K, V, cache, l2_flush, l2_evict
        torch.cuda.empty_cache()
        sampler2 = ClockSampler(local_rank)
        sampler2.start()
        per_config = run_all_configs(dev, load_peaks()[0])
        per_config["clocks"] = sampler2.stop()

    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8 codes, fp32 accumulate",
        "data": "synthetic (seeded N(0,1) fp16 with key-channel and value-token outliers)",
        "config": {
            "workload": w.name, "batch_per_gpu": w.B, "global_batch": w.B * world,
            "num_q_heads": w.Hq, "num_kv_heads": w.Hkv, "head_dim": w.d, "seq_len": T,
            "bits": w.bits, "group": w.G, "residual": w.R,
            "decode_state": {"n_quant": n_quant, "n_resid": n_resid},
            "splits": splits,
            "l2": "before each prefill and each decode (untimed): 256 MiB write, then "
                  "512 MiB read (cold, clean L2); prefill input 1 GiB > L2",
            "parallelism": f"independent batch per GPU x{world}",
        },
        "decode_us": round(dec_ms * 1e3, 2),
        "decode_hbm_frac": round(value / world / peak, 4),
        "quantize_gbs": round(quant_gbs, 2),
        "quantize_us": round(pre_ms * 1e3, 2),
        "append_us": round(statistics.mean(app) * 1e3, 2),
        "decode_full_window": {"decode_state": full_state, "decode_us": round(full_ms * 1e3, 2),
                               "decode_gbs": round(full_gbs, 1),
                               "frac": round(full_gbs / load_peaks()[0], 4),
                               "algorithmic_bytes": int(full_bytes)},
        "wall_ms_per_step": round(wall / args.steps * 1e3, 4),
        "roofline": {
            "kernel": "decode_split_mma (history splits, residual and merge in one launch)",
            "bound": "hbm", "achieved": round(kernel_gbs, 2), "peak": peak, "unit": "GB/s",
            "frac": round(kernel_gbs / peak, 4), "peak_source": peak_kind,
            "traffic": profile_traffic(),
            "algorithmic_bytes_per_launch": dbytes,
            "us_per_launch": round(dec_ms * 1e3, 2),
        },
        "quantize_roofline": {
            "kernel": "quantize_kv_kernel + residual_copy_kernel (prefill)",
            "bound": "hbm", "achieved": round(quant_gbs / world, 2), "peak": peak, "unit": "GB/s",
            "frac": round(quant_gbs / world / peak, 4), "peak_source": peak_kind,
            "algorithmic_bytes_per_launch": pbytes, "us_per_launch": round(pre_ms * 1e3, 2),
        },
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    return line


# ------------------------------------------------- every workload config ----

def make_flusher(dev):
    """Untimed L2 flush: a 256 MiB write pushes every cache line out, a 512 MiB
    read then evicts the dirty lines the write left (cold, clean L2)."""
    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_evict = torch.zeros(512 << 20, dtype=torch.uint8, device=dev)

    def flush():
        l2_flush.zero_()
        l2_evict.amax()
    return flush


def time_calls(fn, n, stream, before=None):
    """Device time (ms) of each of n calls of fn, CUDA events on the stream;
    `before` (untimed) runs ahead of each call."""
    evs = []
    for _ in range(n):
        if before is not None:
            before()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def decode_line(name, w, cache, dbytes, dec_ms, peak, extra=None):
    gbs = dbytes / (dec_ms * 1e-3) / 1e9
    d = {"workload": name, "bits": w.bits, "group": w.G, "residual": w.R, "batch": w.B,
         "num_q_heads": w.Hq, "num_kv_heads": w.Hkv,
         "decode_state": {"n_quant": cache.n_quant, "n_resid": cache.n_resid},
         "splits": cache.num_splits(0), "decode_us": round(dec_ms * 1e3, 2),
         "decode_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
         "algorithmic_bytes": int(dbytes)}
    if extra:
        d.update(extra)
    return d


def bench_prefill_decode(w, dev, flush, peak, name, T=None, reps=3, dec_reps=20, layer=0,
                         variant=None):
    """Prefill T tokens into a fresh cache (timed reps times), append one token
    (a flush of the full residual), then decode (timed dec_reps times, cold L2).
    variant: extra cache fields (sink_tokens, meta, flush, fp8_format, ...)."""
    from bit_kv_cache_06_gb300 import kivi, synth
    stream = torch.cuda.current_stream()
    T = w.T if T is None else T
    variant = dict(variant or {})
    meta = variant.get("meta", 0)
    K, V = synth.make_kv(w, layer=layer, device=dev, T=T)
    q = synth.make_q(w, layer=layer, device=dev)
    k_new, v_new = synth.make_token(w, 0, layer=layer, device=dev)
    out = torch.empty_like(q)
    cache = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                           ((T + 1 + w.R - 1) // w.R) * w.R, **variant),
                           device=dev)

    def prefill():
        cache.reset()
        cache.quantize_prefill(K, V)
    pre = time_calls(prefill, reps, stream, before=flush)
    pbytes = prefill_bytes(w, T, cache.n_quant, cache.n_resid, meta, cache.n_sink)
    cache.append_token(k_new, v_new)
    torch.cuda.synchronize()
    del K, V
    dec = time_calls(lambda: cache.decode_attention(q, out), dec_reps, stream, before=flush)
    dec_ms = statistics.mean(dec[1:]) if len(dec) > 1 else dec[0]
    pre_ms = statistics.mean(pre[1:]) if len(pre) > 1 else pre[0]
    dbytes = decode_bytes(w, cache.n_quant, cache.n_resid, meta, cache.n_sink)
    extra = {"seq_len": T, "quantize_us": round(pre_ms * 1e3, 2),
             "quantize_gbs": round(pbytes / (pre_ms * 1e-3) / 1e9, 1),
             "quantize_frac": round(pbytes / (pre_ms * 1e-3) / 1e9 / peak, 4)}
    if variant:
        extra["variant"] = variant
        extra["decode_state"] = {"n_quant": cache.n_quant, "n_resid": cache.n_resid,
                                 "n_sink": cache.n_sink}
    line = decode_line(name, w, cache, dbytes, dec_ms, peak, extra)
    del cache
    torch.cuda.empty_cache()
    return line


def bench_streaming(w, dev, flush, peak):
    """The streaming workload: prefill, then w.steps x (append one token, decode);
    each append and each decode timed after an untimed L2 flush (a cold L2,
    and a busy device while the host enqueues the timed call, so that its
    events bracket device work only)."""
    from bit_kv_cache_06_gb300 import kivi, synth
    stream = torch.cuda.current_stream()
    K, V = synth.make_kv(w, device=dev)
    cache = kivi.KiviCache(kivi.CacheShape(w.bits, w.G, w.R, w.B, w.Hq, w.Hkv, w.d,
                                           w.capacity()), device=dev)
    cache.quantize_prefill(K, V)
    torch.cuda.synchronize()
    del K, V
    toks = [synth.make_token(w, s, device=dev) for s in range(w.steps)]
    qs = [synth.make_q(w, s, device=dev) for s in range(w.steps)]
    out = torch.empty_like(qs[0])
    app_ms, dec_ms, dec_gbs, flushes = [], [], [], 0
    for s in range(w.steps):
        k, v = toks[s]
        app_ms += time_calls(lambda: cache.append_token(k, v), 1, stream, before=flush)
        flushes += cache.n_resid == 1
        d = time_calls(lambda: cache.decode_attention(qs[s], out), 1, stream, before=flush)[0]
        dec_ms.append(d)
        dec_gbs.append(decode_bytes(w, cache.n_quant, cache.n_resid) / (d * 1e-3) / 1e9)
    gbs = statistics.mean(dec_gbs)
    line = decode_line(w.name, w, cache, decode_bytes(w, cache.n_quant, cache.n_resid),
                       statistics.mean(dec_ms), peak, {
                           "steps": w.steps, "residual_flushes": flushes,
                           "decode_gbs_mean_over_steps": round(gbs, 1),
                           "frac_mean_over_steps": round(gbs / peak, 4),
                           "append_us_mean": round(statistics.mean(app_ms) * 1e3, 2),
                           "step_us_mean": round(statistics.mean(
                               a + b for a, b in zip(app_ms, dec_ms)) * 1e3, 2)})
    del cache
    torch.cuda.empty_cache()
    return line


def bench_sweep(w, dev, flush, peak):
    """The 32-layer sweep: every (bits, batch, context) cell, one layer's cache
    at a time (32 layers of the largest cells do not fit in HBM together; the
    layers have one shape, so a 32-layer decode step is 32 layer decodes)."""
    from bit_kv_cache_06_gb300 import synth
    cells = []
    for bits in synth.C5_BITS:
        for B in synth.C5_BATCHES:
            for T in synth.C5_CONTEXTS:
                wc = w.with_(bits=bits, B=B, T=T)
                c = bench_prefill_decode(wc, dev, flush, peak, f"{w.name}/b{bits}-B{B}-T{T}",
                                         reps=2, dec_reps=6)
                c["decode_us_32_layers"] = round(c["decode_us"] * w.layers, 1)
                cells.append(c)
    return {"workload": w.name, "layers": w.layers, "cells": cells}


def run_all_configs(dev, peak):
    """One line per named workload besides the headline (each with its own
    decode roofline against the same measured peak)."""
    from bit_kv_cache_06_gb300 import synth
    flush = make_flusher(dev)
    res = {}
    res["c1"] = bench_prefill_decode(synth.C1, dev, flush, peak, synth.C1.name, reps=5,
                                     dec_reps=50)
    res["c3"] = bench_streaming(synth.C3, dev, flush, peak)
    res["c4"] = bench_prefill_decode(synth.C4, dev, flush, peak, synth.C4.name, reps=2,
                                     dec_reps=10)
    res["c5"] = bench_sweep(synth.C5, dev, flush, peak)
    ext = {}
    for name in EXTENSIONS:
        wv, var = extension_case(synth.C2, name)
        ext[name] = bench_prefill_decode(wv, dev, flush, peak, f"{synth.C2.name}/{name}",
                                         reps=3, dec_reps=20, variant=var)
    res["extensions"] = ext
    return res


# the extensions, each timed on the 8B-layer shape: fp16 scale / zero
# metadata, four fp16 sink tokens, the per-key-group flush, FP8 (E4M3) KV
EXTENSIONS = {
    "fp16-metadata": ({"meta": 1}, None),
    "sink-4": ({"sink_tokens": 4}, None),
    "group-flush": ({"flush": 1}, None),
    "fp8-e4m3": ({"fp8_format": 1, "fp8_k_scale": 1.0, "fp8_v_scale": 1.0}, 8),
}


def extension_case(w, name):
    """(workload, cache fields) of extension `name` on the shape of w."""
    var, bits = EXTENSIONS[name]
    return (w.with_(bits=bits) if bits else w), dict(var)


def run_case(args):
    """One workload (optionally shortened to --seq-len tokens, optionally with
    an extension) through bench_prefill_decode: prefill, one flushing append,
    cold-L2 decodes.  A small, single-kernel-shape run for profiling."""
    from bit_kv_cache_06_gb300 import build as kbuild, kivi, synth
    kbuild.build()
    kivi.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfg, _, ext = args.case.partition("/")
    w = synth.CONFIGS[cfg]
    if args.seq_len:
        w = w.with_(T=args.seq_len)
    var = None
    if ext:
        w, var = extension_case(w, ext)
    peak = load_peaks()[0]
    line = bench_prefill_decode(w, dev, make_flusher(dev), peak, args.case, reps=3,
                                dec_reps=max(args.steps, 3), variant=var)
    line["data"] = "synthetic"
    return line



def run_e2e(cache, w, K, V, q, k_new, v_new, out, stream, dbytes, args, world):
    hK = torch.empty(K.shape, dtype=K.dtype, pin_memory=True)
    hV = torch.empty(V.shape, dtype=V.dtype, pin_memory=True)
    hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hk = torch.empty(k_new.shape, dtype=k_new.dtype, pin_memory=True)
    hv = torch.empty(v_new.shape, dtype=v_new.dtype, pin_memory=True)
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hK.copy_(K)
    hV.copy_(V)
    hq.copy_(q)
    hk.copy_(k_new)
    hv.copy_(v_new)
    dK, dV, dq = torch.empty_like(K), torch.empty_like(V), torch.empty_like(q)
    dk, dv = torch.empty_like(k_new), torch.empty_like(v_new)

    def step():
        dK.copy_(hK, non_blocking=True)
        dV.copy_(hV, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        cache.reset()
        cache.quantize_prefill(dK, dV)
        cache.append_token(dk, dv)
        cache.decode_attention(dq, out)
        hout.copy_(out, non_blocking=True)

    n = max(3, min(args.steps, 10))
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks([e0.elapsed_time(e1) / n], world, q.device)[0]
    h2d = sum(t.numel() * t.element_size() for t in (hK, hV, hq, hk, hv))
    return {"value": round(whole_job_gbs(world, dbytes, ms), 3), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": hout.numel() * hout.element_size(),
            "what": "decode bytes / (H2D of K, V, q, new token + prefill + append + decode "
                    "+ D2H of o), per step"}


# -------------------------------------------------------- oracle (CPU) ----

def oracle_sample(w, nthreads, pairs=8):
    """One bounded sample of the workload on the CPU oracle: the first batch
    element (pairs kv heads): prefill of all T tokens, one append, fp64
    attention of its query heads.  Returns timings and byte counts."""
    import numpy as np

    import oracle
    from bit_kv_cache_06_gb300 import synth
    ws = w.with_(B=pairs // w.Hkv)
    K, V = synth.make_kv(ws)
    k, v = synth.make_token(ws, 0)
    q = synth.make_q(ws).numpy().reshape(-1, w.d)
    oc = oracle.OracleCache(ws.pairs, w.d, w.bits, w.G, w.R, w.capacity())
    t0 = time.perf_counter()
    oc.prefill(K.reshape(ws.pairs, w.T, w.d).numpy(), V.reshape(ws.pairs, w.T, w.d).numpy(),
               nthreads=nthreads)
    t1 = time.perf_counter()
    oc.append(k.reshape(ws.pairs, w.d).numpy(), v.reshape(ws.pairs, w.d).numpy())
    t2 = time.perf_counter()
    oc.attention(q, ws.g, nthreads=nthreads)
    t3 = time.perf_counter()
    dbytes = decode_bytes(ws, oc.n_quant, oc.n_resid)
    r_new = ((w.T - 1) % w.R) + 1
    pbytes = prefill_bytes(ws, w.T, w.T - r_new, r_new)
    del np
    return {"prefill_s": t1 - t0, "append_s": t2 - t1, "attn_s": t3 - t2,
            "decode_bytes": dbytes, "prefill_bytes": pbytes, "pairs": ws.pairs}


def cpu_baseline(w):
    nthreads = os.cpu_count() or 1
    s = oracle_sample(w, nthreads)
    return {"value": round(s["decode_bytes"] / s["attn_s"] / 1e9, 4), "unit": "GB/s",
            "cores": nthreads, "kind": "oracle",
            "sample": f"batch element 0 ({s['pairs']} of {w.pairs} kv-head pairs): oracle "
                      f"prefill of {w.T} tokens + 1 append + fp64 attention of its query "
                      f"heads; value = that attention's algorithmic bytes / its time",
            "attention_s": round(s["attn_s"], 3),
            "quantize_gbs": round(s["prefill_bytes"] / s["prefill_s"] / 1e9, 4),
            "single_core": single_core_baseline(w)}


def single_core_baseline(w):
    """The same oracle sample (batch element 0) on one host core."""
    s = oracle_sample(w, 1)
    return {"value": round(s["decode_bytes"] / s["attn_s"] / 1e9, 4), "unit": "GB/s",
            "cores": 1, "quantize_gbs": round(s["prefill_bytes"] / s["prefill_s"] / 1e9, 4),
            "attention_s": round(s["attn_s"], 3)}


def run_reference(args):
    from bit_kv_cache_06_gb300 import synth
    w = synth.CONFIGS[args.config]
    nthreads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_sample(w, nthreads, pairs=w.Hkv)
    samples = [oracle_sample(w, nthreads, pairs=w.Hkv) for _ in range(args.steps)]
    attn = statistics.mean(s["attn_s"] for s in samples)
    step = statistics.mean(s["prefill_s"] + s["append_s"] + s["attn_s"] for s in samples)
    value = samples[0]["decode_bytes"] / attn / 1e9
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32 quantiser, fp64 attention", "data": "synthetic",
        "config": {"workload": w.name, "batch_per_gpu": w.B, "num_q_heads": w.Hq,
                   "num_kv_heads": w.Hkv, "head_dim": w.d, "seq_len": w.T, "bits": w.bits,
                   "group": w.G, "residual": w.R},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                         "kind": "oracle",
                         "sample": f"each step: batch element 0 ({w.Hkv} of {w.pairs} pairs): "
                                   f"prefill {w.T} tokens + 1 append + fp64 attention"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c2", choices=["c2", "c4", "c1", "c3"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the per-config lines (tiny, streaming, 1M-context, sweep)")
    ap.add_argument("--case", default=None,
                    help="time one workload alone and print its decode line: c1, c2 or c4, "
                         "or c2/<extension> with extension fp16-metadata, sink-4, "
                         "group-flush or fp8-e4m3 (one GPU)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="with --case: the context length, in place of the workload's own")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N > 1 GPUs "
                 "with torch.distributed.run --nproc-per-node N (one rank per GPU)")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.case:
        if world != 1:
            sys.exit("bench.py: --case runs on one GPU")
        print(json.dumps(run_case(args)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
