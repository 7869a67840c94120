"""Benchmark: bifocal prefill TFLOP/s at 128K and decode us/token at 128K on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole hot path over one batch of synthetic input:
a bifocal prefill of the Qwen3-8B-shaped attention layer (B=1, Hq=32, Hkv=8,
D=128, S=131072, L_pre=32768, w=4096, theta=1e6; g=4) followed by a bifocal
decode of the last token over the same exact-RoPE K/V (n=131072).  Inputs
are seeded bf16 N(0,1) (counter-based generator) and are larger than L2.
``value`` is the prefill throughput (FA causal FLOP convention 2*B*Hq*D*S^2)
over the K timed steps; decode, the bifocal-off prefill, the roofline, the
end-to-end number (host buffers, copies inside the timed region) and the CPU
oracle baseline ride along in the same JSON line.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); time is the max over ranks and ``value`` the
sum of all ranks' work over that time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bifocal prefill attn TFLOP/s @128K (% of BF16 peak); decode µs/token @128K"
WORKLOAD = dict(B=1, Hq=32, Hkv=8, D=128, S=131072, L_pre=32768, w=4096, theta=1e6, seed=2)
DECODE_NS = (8192, 32768, 131072)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# DRAM bytes (read + write) of one 128K bifocal prefill launch, from the ncu
# counters of a one-launch capture, valid only for the prefill sources they
# were measured on (first 16 hex digits of the sha256 of their concatenation).
PREFILL_TRAFFIC = {"sha256_16": "28f23a7603d4d8e8", "bytes": 3.5630e9 + 1.0578e9}
PREFILL_SOURCES = ("prefill.cu", "corrector.cuh", "sm100_ptx.cuh", "jl_common.cuh", "tile_class.cuh")


def prefill_sources_sha16():
    import hashlib

    h = hashlib.sha256()
    for name in PREFILL_SOURCES:
        with open(os.path.join(ROOT, "zero_shot_rope_02_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def prefill_traffic():
    return PREFILL_TRAFFIC["bytes"] if prefill_sources_sha16() == PREFILL_TRAFFIC["sha256_16"] else None


def prefill_kernel_name(grp, D, remote=True):
    """The tile kernel libjetlong dispatches a launch to by default: the two-SM
    kernel at D = 128 with a multiple of four heads per kv head when the launch
    has remote keys, else one CTA per query tile of two heads of a GQA group
    (one when the group size is odd)."""
    if remote and D == 128 and grp % 4 == 0:
        return "prefill_pair_kernel"
    return f"prefill_kernel<{D},{2 if grp % 2 == 0 else 1}>"


def prefill_flops(B, Hq, D, S):
    return 2.0 * B * Hq * D * S * S


def chunk_prefill_flops(B, Hq, D, S_new, n_past):
    """Same convention as prefill_flops (4*D FLOP per (query, key) pair, the
    causal half of the new tokens' own block): S_new*n_past + S_new^2/2 pairs."""
    return 2.0 * B * Hq * D * (2.0 * S_new * n_past + S_new * S_new)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        peaks = {k: float(d[k]) for k in FALLBACK_PEAKS}
        # SM clock the sustained (power-capped, back-to-back) GEMM loop settled at
        mhz = (d.get("clocks_under_load") or {}).get("sm_mhz_median")
        peaks["sustained_sm_mhz"] = float(mhz) if mhz else None
        return peaks, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, sustained_sm_mhz=None), "fallback"


def sustained_frac_at_clock(achieved, peaks, kernel_mhz):
    """achieved / (the sustained GEMM rate per MHz x the kernel's own median SM
    clock): the sustained peak was taken at the clock a power-capped cuBLAS loop
    settles to, so it is rescaled to the clock this kernel actually ran at."""
    mhz0 = peaks.get("sustained_sm_mhz")
    if not mhz0 or not kernel_mhz:
        return None
    return achieved / (peaks["bf16_tflops_sustained"] / mhz0 * kernel_mhz)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ inputs
def make_inputs(dev, cfg, pinned=False):
    import torch

    from zero_shot_rope_02_b300 import inputs

    B, Hq, Hkv, D, S, seed = (cfg[k] for k in ("B", "Hq", "Hkv", "D", "S", "seed"))
    host = []
    for shape, tid in (((B, S, Hq, D), 0), ((B, S, Hkv, D), 1), ((B, S, Hkv, D), 2)):
        t = inputs.to_torch_bf16(inputs.normal_bf16_bits(shape, seed, tid))
        host.append(t.pin_memory() if pinned else t)
    if dev is None:
        return host
    return [t.to(dev) for t in host]


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, dev):
    import torch

    import zero_shot_rope_02_b300 as jl

    cfg = WORKLOAD
    B, Hq, Hkv, D, S, L, w, theta = (cfg[k] for k in ("B", "Hq", "Hkv", "D", "S", "L_pre", "w", "theta"))
    peaks, peaks_src = load_peaks()
    stream = torch.cuda.current_stream(dev)
    q, k, v = make_inputs(dev, cfg)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    qd = q[:, S - 1].contiguous()
    dout = torch.empty_like(qd)
    dlse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = torch.zeros(max(16, jl.jl_bifocal_decode_workspace_size(B, Hq, Hkv, S, D)), dtype=torch.uint8,
                     device=dev)

    def step(L_pre=L):
        jl.jl_bifocal_prefill(q, k, v, L_pre, w, theta, out=out, lse=lse, stream=stream)
        jl.jl_bifocal_decode(qd, k, v, S, L_pre, w, theta, workspace=ws, out=dout, lse=dlse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if jl.jl_debug_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for e in ev:
            e[0].record(stream)
            jl.jl_bifocal_prefill(q, k, v, L, w, theta, out=out, lse=lse, stream=stream)
            e[1].record(stream)
            jl.jl_bifocal_decode(qd, k, v, S, L, w, theta, workspace=ws, out=dout, lse=dlse, stream=stream)
            e[2].record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    flops = prefill_flops(B, Hq, D, S)
    value, total_ms = replica_value(flops * args.steps, t0.elapsed_time(t1), world)
    value /= 1e12
    prefill_ms = [a.elapsed_time(b) for a, b, _ in ev]
    decode_ms = [b.elapsed_time(c) for _, b, c in ev]
    ms_per_step = total_ms / args.steps
    avg_prefill_ms = sum(prefill_ms) / len(prefill_ms)
    achieved = flops / (avg_prefill_ms * 1e-3) / 1e12
    if jl.jl_debug_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    # bifocal off: L_pre >= S (g = 1), as the library runs it by default, and
    # on the same tile kernel as the bifocal run
    plain_ms = time_calls(lambda: jl.jl_bifocal_prefill(q, k, v, S, w, theta, out=out, lse=lse,
                                                        stream=stream), stream, dev, reps=max(3, args.steps))
    same_flags = jl.JL_PREFILL_CTA_PAIR if prefill_kernel_name(Hq // Hkv, D) == "prefill_pair_kernel" else \
        jl.JL_PREFILL_ONE_CTA
    plain_same_ms = time_calls(lambda: jl.jl_bifocal_prefill_ex(q, k, v, 0, S, w, theta, same_flags, out=out,
                                                                lse=lse, stream=stream), stream, dev, reps=3)
    decode = decode_sweep(jl, dev, stream, peaks)
    # the method's optional forms on the same 128K layer (same FLOP convention)
    variants = {}
    for name, flags in (("per_query_g", jl.JL_VARIANT_PER_QUERY_G), ("sliding_window", jl.JL_VARIANT_SLIDING),
                        ("query_shift", jl.JL_VARIANT_QUERY_SHIFT)):
        v_ms = time_calls(lambda f=flags: jl.jl_bifocal_prefill_ex(q, k, v, 0, L, w, theta, f, out=out, lse=lse,
                                                                   stream=stream), stream, dev, reps=3)
        variants[name] = {"ms": round(v_ms, 3), "tflops_causal_convention": round(flops / (v_ms * 1e-3) / 1e12, 2),
                          "g": jl.jl_group_factor_ex(S, L, w, flags)}
    variants["sliding_window"]["note"] = "attends only the last w keys: FLOPs counted on the full causal convention"
    # the other tile kernel on the same layer (JL_PREFILL_ONE_CTA: one CTA per
    # query tile of two heads), bifocal and plain
    one_cta = {}
    for tag, L_pre in (("bifocal", L), ("plain", S)):
        one_cta[tag + "_ms"] = round(time_calls(lambda Lp=L_pre: jl.jl_bifocal_prefill_ex(
            q, k, v, 0, Lp, w, theta, jl.JL_PREFILL_ONE_CTA, out=out, lse=lse, stream=stream), stream, dev, reps=3), 3)
    one_cta["bifocal_overhead"] = round(one_cta["bifocal_ms"] / one_cta["plain_ms"] - 1.0, 4)
    one_cta["tflops"] = round(flops / (one_cta["bifocal_ms"] * 1e-3) / 1e12, 2)
    if jl.jl_debug_status() != 0:
        raise RuntimeError("device status word set by the variant runs")
    # chunked prefill: the last 8K tokens of the same context over the cache of
    # the first 120K (same k / v buffers as the cache), s = S as above
    S_new = 8192
    n_past = S - S_new
    qc = q[:, n_past:].contiguous()
    outc = torch.empty_like(qc)
    lsec = torch.empty((B, Hq, S_new), dtype=torch.float32, device=dev)
    chunk_ms = time_calls(lambda: jl.jl_bifocal_prefill_chunk(qc, k, v, n_past, L, w, theta, out=outc,
                                                              lse=lsec, stream=stream),
                          stream, dev, reps=max(3, args.steps))
    chunk_flops = chunk_prefill_flops(B, Hq, D, S_new, n_past)
    paged = paged_decode(jl, dev, stream, peaks, args)
    # RoPE fused into the cache write: the whole context's raw k and v into a cache
    kc_dst = torch.empty_like(k)
    vc_dst = torch.empty_like(v)
    cw_ms = time_calls(lambda: jl.jl_rope_cache_write(k, v, kc_dst, vc_dst, 0, theta, stream=stream),
                       stream, dev, reps=max(3, args.steps))
    cw_bytes = 4 * k.numel() * k.element_size()  # read k and v, write both
    del kc_dst, vc_dst
    if jl.jl_debug_status() != 0:
        raise RuntimeError("device status word set by the chunk run")

    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded bf16 N(0,1) q/k/v treated as exact-RoPE; no weights)",
        "config": {"workload": "Qwen3-8B-shaped bifocal prefill at 128K + decode of the last token",
                   **{k_: cfg[k_] for k_ in ("B", "Hq", "Hkv", "D", "S", "L_pre", "w", "theta")},
                   "g": jl.jl_group_factor(S, L),
                   "l2": "inputs larger than L2 (q 1 GiB, k and v 256 MiB each)"},
        "prefill": {"tflops": round(achieved, 2), "ms": round(avg_prefill_ms, 3),
                    "frac_of_bf16_peak": round(achieved / peaks["bf16_tflops"], 4)},
        "plain_rope": {"tflops": round(flops / (plain_ms * 1e-3) / 1e12, 2), "ms": round(plain_ms, 3),
                       "kernel": prefill_kernel_name(Hq // Hkv, D, remote=False),
                       "bifocal_overhead": round(avg_prefill_ms / plain_ms - 1.0, 4),
                       "same_kernel_ms": round(plain_same_ms, 3),
                       "same_kernel_overhead": round(avg_prefill_ms / plain_same_ms - 1.0, 4)},
        "decode": decode,
        "variants": variants,
        "prefill_one_cta": one_cta,
        "paged_decode": paged,
        "rope_cache_write": {"rows": S, "us": round(1e3 * cw_ms, 2),
                             "gbs": round(cw_bytes / (cw_ms * 1e-3) / 1e9, 1),
                             "frac_of_hbm": round(cw_bytes / (cw_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
        "chunk": {"S_new": S_new, "n_past": n_past, "ms": round(chunk_ms, 3),
                  "tflops": round(chunk_flops / (chunk_ms * 1e-3) / 1e12, 2),
                  "frac_of_bf16_peak": round(chunk_flops / (chunk_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)},
        "decode_in_step_us": round(1e3 * sum(decode_ms) / len(decode_ms), 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "traffic": prefill_traffic(), "kernel": prefill_kernel_name(Hq // Hkv, D),
                     "peak_source": f"{peaks_src} bf16 burst",
                     # also reported: the back-to-back cuBLAS figure rescaled from
                     # the clock its power-capped loop settled at to this kernel's
                     # median clock over the timed steps (same work per cycle)
                     "sustained_peak": peaks["bf16_tflops_sustained"],
                     "sustained_peak_sm_mhz": peaks.get("sustained_sm_mhz"),
                     "frac_of_sustained_at_kernel_clock": None},
        # per step: the prefill tile kernel, its fp32 pass over the rows below
        # position 256, and the decode kernel
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    f_s = sustained_frac_at_clock(achieved, peaks, res["clocks"].get("sm_mhz"))
    res["roofline"]["frac_of_sustained_at_kernel_clock"] = None if f_s is None else round(f_s, 4)
    if not args.no_e2e:
        res["e2e"] = e2e(jl, args, dev, stream)
    if rank == 0 and not args.no_cpu:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return res


def paged_decode(jl, dev, stream, peaks, args):
    """One call decoding four sequences of their own lengths (and own g) over
    a paged cache: 64-key pages of one pool, in shuffled order."""
    import numpy as np
    import torch

    from zero_shot_rope_02_b300 import inputs

    lens = [131072, 65536, 32768, 8192]
    Hq, Hkv, D, P, L, w = 32, 8, 128, 64, 32768, 4096
    B = len(lens)
    pages_per = [n // P for n in lens]
    num_pages = sum(pages_per)
    perm = np.random.default_rng(7).permutation(num_pages).astype(np.int32)
    table = np.zeros((B, max(pages_per)), dtype=np.int32)
    o = 0
    for b, k in enumerate(pages_per):
        table[b, :k] = perm[o:o + k]
        o += k
    kp = inputs.to_torch_bf16(inputs.normal_bf16_bits((num_pages, P, Hkv, D), 8, 4)).to(dev)
    vp = inputs.to_torch_bf16(inputs.normal_bf16_bits((num_pages, P, Hkv, D), 8, 5)).to(dev)
    q = inputs.to_torch_bf16(inputs.normal_bf16_bits((B, Hq, D), 8, 3)).to(dev)
    table_d = torch.from_numpy(table).to(dev)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    ws = torch.zeros(max(16, jl.jl_bifocal_decode_paged_workspace_size(B, Hq, Hkv, max(lens), D)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    us = 1e3 * time_calls(lambda: jl.jl_bifocal_decode_paged(q, kp, vp, table_d, lens_d, max(lens), L, w,
                                                             1e6, workspace=ws, out=out, lse=lse,
                                                             stream=stream),
                          stream, dev, reps=20)
    if jl.jl_debug_status() != 0:
        raise RuntimeError("device status word set by the paged decode")
    nbytes = sum(lens) * Hkv * D * 2 * 2  # K and V rows of every sequence
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"lens": lens, "page_size": P, "g": [jl.jl_group_factor(n, L) for n in lens],
            "us_per_call": round(us, 2), "gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "timing": "eager; K and V pools 486 MB each, > 2x L2"}


def time_calls(fn, stream, dev, reps):
    import torch

    fn()
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / reps


def decode_sweep(jl, dev, stream, peaks):
    """us per decode call at n = 8K/32K/128K, Hq=32, Hkv=8, D=128, L=32768,
    w=4096 (g = 1, 1, 4).  The caches are rotated over copies totalling more
    than 2x L2 so every call reads K/V from HBM.  The calls are captured in a
    CUDA graph and the graph is replayed, so the number is device time per
    call, as in a serving loop; the eager per-call time (host enqueue
    included) rides along."""
    import torch

    from zero_shot_rope_02_b300 import inputs

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for n in DECODE_NS:
        nbytes = 2 * n * 8 * 128 * 2
        copies = max(1, math.ceil(2 * l2 / nbytes) + 1)
        q = inputs.to_torch_bf16(inputs.normal_bf16_bits((1, 32, 128), 3, 3)).to(dev)
        k0 = inputs.to_torch_bf16(inputs.normal_bf16_bits((1, n, 8, 128), 3, 4)).to(dev)
        v0 = inputs.to_torch_bf16(inputs.normal_bf16_bits((1, n, 8, 128), 3, 5)).to(dev)
        ks = [k0] + [k0.clone() for _ in range(copies - 1)]
        vs = [v0] + [v0.clone() for _ in range(copies - 1)]
        ws = torch.zeros(jl.jl_bifocal_decode_workspace_size(1, 32, 8, n, 128), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((1, 32), dtype=torch.float32, device=dev)
        it = [0]

        def call(st=None):
            c = it[0] % copies
            it[0] += 1
            jl.jl_bifocal_decode(q, ks[c], vs[c], n, 32768, 4096, 1e6, workspace=ws, out=o, lse=lse, stream=st)

        for _ in range(5):
            call(stream)
        eager_us = 1e3 * time_calls(lambda: call(stream), stream, dev, 50)
        per_graph = copies * max(1, 64 // copies)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                call()  # the capture stream is current
        graph.replay()
        torch.cuda.synchronize(dev)
        reps = 10 if n < 100000 else 4
        us = 1e3 * time_calls(graph.replay, stream, dev, reps) / per_graph
        gbs = nbytes / (us * 1e-6) / 1e9
        out[str(n)] = {"us_per_token": round(us, 2), "gbs": round(gbs, 1),
                       "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "g": jl.jl_group_factor(n, 32768),
                       "eager_us_per_call": round(eager_us, 2), "timing": "cuda graph replay"}
        del ks, vs, graph
    return out


def e2e(jl, args, dev, stream):
    """The same step through the public API from pinned HOST buffers: q/k/v
    host->device, prefill + decode, out/lse/decode-out device->host, every
    step's copies inside the timed region.  Steps are pipelined as a serving
    loop would run them: two device buffer sets, the upload of step i+1 and
    the download of step i-1 on their own streams while step i computes, the
    kernels of a step waiting (events) for its upload and for the download
    that last read its buffers.  The timed region runs from the first upload
    to the last download."""
    import torch

    cfg = WORKLOAD
    B, Hq, Hkv, D, S, L, w, theta = (cfg[k] for k in ("B", "Hq", "Hkv", "D", "S", "L_pre", "w", "theta"))
    hq, hk, hv = make_inputs(None, cfg, pinned=True)
    sets = []
    for _ in range(2):
        q = torch.empty(hq.shape, dtype=hq.dtype, device=dev)
        k = torch.empty(hk.shape, dtype=hk.dtype, device=dev)
        v = torch.empty(hv.shape, dtype=hv.dtype, device=dev)
        sets.append({"q": q, "k": k, "v": v, "out": torch.empty_like(q),
                     "lse": torch.empty((B, Hq, S), dtype=torch.float32, device=dev),
                     "dq": torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev),
                     "dout": torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev),
                     "dlse": torch.empty((B, Hq), dtype=torch.float32, device=dev),
                     "ws": torch.zeros(max(16, jl.jl_bifocal_decode_workspace_size(B, Hq, Hkv, S, D)),
                                       dtype=torch.uint8, device=dev)})
    h_out = torch.empty(sets[0]["out"].shape, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(sets[0]["lse"].shape, dtype=torch.float32).pin_memory()
    h_dout = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    h_dlse = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)

    def run(n_steps, timed):
        uploaded = [torch.cuda.Event() for _ in range(n_steps)]
        computed = [torch.cuda.Event() for _ in range(n_steps)]
        downloaded = [torch.cuda.Event() for _ in range(n_steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        if timed:
            t0.record(up)

        def upload(i):
            st = sets[i % 2]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[i - 2])  # step i-2's kernels have read this set
                st["q"].copy_(hq, non_blocking=True)
                st["k"].copy_(hk, non_blocking=True)
                st["v"].copy_(hv, non_blocking=True)
                uploaded[i].record(up)

        upload(0)
        for i in range(n_steps):
            if i + 1 < n_steps:
                upload(i + 1)
            st = sets[i % 2]
            with torch.cuda.stream(stream):
                stream.wait_event(uploaded[i])
                if i >= 2:
                    stream.wait_event(downloaded[i - 2])  # step i-2's results are on the host
                jl.jl_bifocal_prefill(st["q"], st["k"], st["v"], L, w, theta, out=st["out"], lse=st["lse"],
                                      stream=stream)
                st["dq"].copy_(st["q"][:, S - 1], non_blocking=True)
                jl.jl_bifocal_decode(st["dq"], st["k"], st["v"], S, L, w, theta, workspace=st["ws"],
                                     out=st["dout"], lse=st["dlse"], stream=stream)
                computed[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[i])
                h_out.copy_(st["out"], non_blocking=True)
                h_lse.copy_(st["lse"], non_blocking=True)
                h_dout.copy_(st["dout"], non_blocking=True)
                h_dlse.copy_(st["dlse"], non_blocking=True)
                downloaded[i].record(down)
        if timed:
            t1.record(down)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / n_steps if timed else None

    run(2, False)
    steps = max(2, min(args.steps, 8))
    ms = run(steps, True)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_lse, h_dout, h_dlse))
    return {"value": round(prefill_flops(B, Hq, D, S) / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 3), "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "uploads of step i+1 and downloads of step i-1 overlap step i's kernels; "
                         "first upload to last download timed"}


# ------------------------------------------------------------------ oracle arm
def oracle_sample(seconds_budget):
    """The fp64 oracle on a bounded sample of the 128K workload: full rows of
    query positions near the end of the sequence, all 32 heads.  Returns
    (TFLOP/s on the FA convention for the rows done, threads, description)."""
    import numpy as np

    import oracle
    from zero_shot_rope_02_b300 import inputs

    cfg = WORKLOAD
    B, Hq, Hkv, D, S, L, w, theta, seed = (cfg[k] for k in ("B", "Hq", "Hkv", "D", "S", "L_pre", "w",
                                                            "theta", "seed"))
    orc = oracle.default()
    kf = inputs.bf16_bits_to_f64(inputs.normal_bf16_bits((B, S, Hkv, D), seed, 1))
    vf = inputs.bf16_bits_to_f64(inputs.normal_bf16_bits((B, S, Hkv, D), seed, 2))
    rows_done, flops, elapsed = 0, 0.0, 0.0
    nrows = 2
    while elapsed < seconds_budget:
        rows = np.arange(S - rows_done - nrows, S - rows_done, dtype=np.int64)
        q = inputs.bf16_bits_to_f64(_q_rows_bits(seed, B, S, Hq, D, rows))
        t = time.perf_counter()
        orc.bifocal_rows(q, kf, vf, rows, S, L, w, theta)
        elapsed += time.perf_counter() - t
        flops += float(sum(4.0 * B * Hq * D * (int(r) + 1) for r in rows))
        rows_done += nrows
        nrows = min(2 * nrows, 64)
    desc = (f"fp64 oracle, {rows_done} full query rows (positions {S - rows_done}..{S - 1}) x {Hq} heads "
            f"of the 128K workload, incl. the per-call key correction; FLOPs on the same causal convention")
    return flops / elapsed / 1e12, orc.num_threads(), desc, elapsed


def _q_rows_bits(seed, B, S, Hq, D, rows):
    """Rows of the seeded q tensor without drawing the whole 1 GiB tensor:
    element e of the tensor uses counter e, so a row is a contiguous range."""
    import numpy as np

    from zero_shot_rope_02_b300 import inputs

    key = inputs._key(seed, 0)
    out = np.empty((B, len(rows), Hq, D), dtype=np.uint16)
    row_elems = Hq * D
    for b in range(B):
        for n, r in enumerate(rows):
            start = (b * S + int(r)) * row_elems
            vals = inputs._normal_chunk(key, start, row_elems).astype(np.float32)
            out[b, n] = inputs.fp32_to_bf16_bits(vals).reshape(Hq, D)
    return out


def cpu_baseline(seconds):
    v, cores, desc, el = oracle_sample(seconds)
    return {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
            "seconds": round(el, 2)}


def run_reference(args):
    per = max(2.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per / 4)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, cores, desc, _ = oracle_sample(per)
        vals.append(v)
    total = time.perf_counter() - t0
    value = sum(vals) / len(vals)
    return {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": "Qwen3-8B-shaped bifocal prefill at 128K + decode of the last token",
                       **{k_: WORKLOAD[k_] for k_ in ("B", "Hq", "Hkv", "D", "S", "L_pre", "w", "theta")},
                       "g": max(1, -(-WORKLOAD["S"] // WORKLOAD["L_pre"])),
                       "l2": "inputs larger than L2 (q 1 GiB, k and v 256 MiB each)"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ distributed glue
def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    """Max of a per-rank float over all ranks (the job's time is the slowest
    rank's); works on the nccl and gloo backends."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(units_per_rank, ms_per_rank, world):
    """Whole-job throughput of N independent replicas: every rank's units over
    the slowest rank's time (weak scaling; no exchange on the data path)."""
    total_ms = max_over_ranks(ms_per_rank, world)
    return world * units_per_rank / (total_ms * 1e-3), total_ms


def run_case(args):
    """Kernel-only runs for profiling (no JSON line): ``--case prefill`` launches
    the prefill ``--reps`` times at S=``--S`` (Qwen3-8B head shapes), ``--case
    decode`` the decode at n=``--n``; prints device time per launch and the
    host time to enqueue one call."""
    import torch

    import zero_shot_rope_02_b300 as jl
    from zero_shot_rope_02_b300 import inputs

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    if args.case == "prefill":
        cfg = dict(WORKLOAD, S=args.S)
        q, k, v = make_inputs(dev, cfg)
        out = torch.empty_like(q)
        lse = torch.empty((1, cfg["Hq"], args.S), dtype=torch.float32, device=dev)
        L = args.L if args.L > 0 else cfg["L_pre"]

        flags = jl.JL_PREFILL_CTA_PAIR if args.pair else (jl.JL_PREFILL_ONE_CTA if args.one_cta else 0)

        def call():
            jl.jl_bifocal_prefill_ex(q, k, v, 0, L, cfg["w"], cfg["theta"], flags, out=out, lse=lse, stream=stream)
        flops = prefill_flops(1, cfg["Hq"], cfg["D"], args.S)
    else:
        n = args.n
        q = inputs.to_torch_bf16(inputs.normal_bf16_bits((1, 32, 128), 3, 3)).to(dev)
        k = inputs.to_torch_bf16(inputs.normal_bf16_bits((1, n, 8, 128), 3, 4)).to(dev)
        v = inputs.to_torch_bf16(inputs.normal_bf16_bits((1, n, 8, 128), 3, 5)).to(dev)
        ws = torch.zeros(jl.jl_bifocal_decode_workspace_size(1, 32, 8, n, 128), dtype=torch.uint8, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((1, 32), dtype=torch.float32, device=dev)
        L = args.L if args.L > 0 else 32768

        def call():
            jl.jl_bifocal_decode(q, k, v, n, L, 4096, 1e6, workspace=ws, out=o, lse=lse, stream=stream)
        flops = 0.0
    call()
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    for _ in range(args.reps):
        call()
    host_us = 1e6 * (time.perf_counter() - t) / args.reps
    torch.cuda.synchronize(dev)
    ms = time_calls(call, stream, dev, args.reps)
    line = {"case": args.case, "ms_per_launch": round(ms, 4), "host_enqueue_us": round(host_us, 2),
            "status": jl.jl_debug_status()}
    if flops:
        line["tflops"] = round(flops / (ms * 1e-3) / 1e12, 2)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=("prefill", "decode"), default=None,
                    help="kernel-only run for profiling instead of the benchmark")
    ap.add_argument("--S", type=int, default=16384)
    ap.add_argument("--n", type=int, default=8192)
    ap.add_argument("--L", type=int, default=0)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--pair", action="store_true",
                    help="--case prefill: force the two-SM tile kernel (JL_PREFILL_CTA_PAIR)")
    ap.add_argument("--one-cta", action="store_true",
                    help="--case prefill: force the one-CTA tile kernel (JL_PREFILL_ONE_CTA)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch

    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    res = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
