#!/usr/bin/env python3
"""Benchmark: fp8-latent absorbed MLA decode on GB300.

By default one line per decode workload: tiny, single, batched, append, then the
headline, long: B=2 sequences x T=262144 cached tokens, H=128 heads, kv_lora 512 +
qk_rope 64 stored as e4m3 + two f32 scales per row (584 B/token, 306 MB of KV per
step, over twice L2, so no flush is needed between steps; workloads under twice
L2 are flushed by writing and then reading 256 MB).  One step = one decode query per sequence over
its whole cache (the "append" workload also quantizes 65536 fresh rows into the
cache inside the step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|produce|wuv|prefill|persist]
                    [--variant auto|simt|tcgen05] [--impl ours|reference]

Prints one JSON line per workload (rank 0), the headline last.  `value` = KV GB/s
over all ranks (KV bytes the step attends over / device time of the step);
token*heads/s rides along.
Under torchrun (N > 1) every rank runs an independent replica (the decode of
independent sequences needs no exchange): value = all ranks' bytes / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fp8-latent MLA decode: KV GB/s & token·heads/s, % of roofline (1 GB300)"
ROW_BYTES = 576 + 8                 # e4m3 row + two f32 scales
FLOP_PER_TOKEN_HEAD = 2 * (576 + 512)  # score dot over 576 + context over 512
FP32_LANES_PER_SM = 128
NUM_SMS = 152
SM_MAX_MHZ_NOMINAL = 2070.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL)), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": SM_MAX_MHZ_NOMINAL, "src": "fallback"}


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "decode_tc": ["fp8_mla_latent_gb300/csrc/decode_tc.cu", "fp8_mla_latent_gb300/csrc/kv8_common.cuh",
                  "fp8_mla_latent_gb300/csrc/tc_ptx.cuh"],
    "decode_pair": ["fp8_mla_latent_gb300/csrc/decode_pair.cu", "fp8_mla_latent_gb300/csrc/kv8_common.cuh",
                    "fp8_mla_latent_gb300/csrc/tc_ptx.cuh"],
    "produce_rows": ["fp8_mla_latent_gb300/csrc/quantize.cu", "fp8_mla_latent_gb300/csrc/kv8_common.cuh"],
    "wuv": ["fp8_mla_latent_gb300/csrc/wuv.cu", "fp8_mla_latent_gb300/csrc/kv8_common.cuh",
            "fp8_mla_latent_gb300/csrc/tc_ptx.cuh"],
    "prefill": ["fp8_mla_latent_gb300/csrc/prefill.cu", "fp8_mla_latent_gb300/csrc/tc_ptx.cuh",
                "fp8_mla_latent_gb300/csrc/kv8_common.cuh"],
    "decode_simt": ["fp8_mla_latent_gb300/csrc/decode_simt.cu",
                    "fp8_mla_latent_gb300/csrc/kv8_common.cuh"],
}


def traffic_for(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(f"{kernel}/{workload}")
    except Exception:
        return None
    if not d or d.get("source_sha") != source_hash(KERNEL_SOURCES[kernel]):
        return None
    return float(d["bytes_per_launch"])


def flush_l2(buf):
    """Evict L2: write a buffer larger than L2, then read it back, so that the lines
    left in L2 are clean and the timed kernel's loads write nothing back."""
    buf.zero_()
    buf.amax()


def rank_sync():
    """Barrier across the ranks of a torchrun launch (no-op in a single process)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def slowest_rank(values, device):
    """Each timing's maximum over the ranks (the values themselves in a single
    process): replicas report the whole job's throughput at the slowest rank's pace."""
    import torch
    import torch.distributed as dist
    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kv8_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swpc=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 0.3 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in loaded:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("swpc", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r["sm"] for r in loaded])),
                "sm_max_mhz": float(max(r["smax"] for r in rows)),
                "reasons": sorted(reasons), "samples": len(loaded)}


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import fp8_mla_latent_gb300 as pkg
    from fp8_mla_latent_gb300 import workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    variant = {"auto": pkg.KV8_DECODE_AUTO, "simt": pkg.KV8_DECODE_SIMT,
               "tcgen05": pkg.KV8_DECODE_TCGEN05, "tc_cta": pkg.KV8_DECODE_TCGEN05_CTA,
               "tc_pair": pkg.KV8_DECODE_TCGEN05_PAIR}[args.variant]

    w = workloads.make(args.workload, scale=args.scale)
    codes = torch.zeros((w.n_slots, 576), dtype=torch.uint8, device=dev)
    scales = torch.zeros((w.n_slots, 2), dtype=torch.float32, device=dev)
    pkg.kv8_quantize_rows(torch.from_numpy(w.cache_rows).to(dev), codes, scales,
                          dst_slot=torch.from_numpy(w.cache_slots).to(dev))
    fresh = fresh_slots = None
    if w.fresh_rows is not None:
        fresh = torch.from_numpy(w.fresh_rows).to(dev)
        fresh_slots = torch.from_numpy(w.fresh_slots).to(dev)
    ql = torch.from_numpy(w.q_lat).to(dev)
    qr = torch.from_numpy(w.q_rope).to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty((w.B, w.H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    ws_bytes = pkg.mla_absorb_decode_fp8_batch_workspace_size(w.B, w.H, w.max_blocks,
                                                              variant=variant)
    ws = pkg.alloc_workspace(ws_bytes, dev)
    # Between timed steps L2 must hold nothing the step reads: a workload whose
    # inputs are over twice L2 (129 MB) streams past anything left there, so it
    # runs without a flush (a flush would only leave dirty lines for the step to
    # write back); a smaller one is flushed by a 256 MB write.
    L2_BYTES = 129 << 20
    in_bytes = w.kv_bytes() + ql.numel() * 4 + qr.numel() * 4
    do_flush = in_bytes <= 2 * L2_BYTES
    flush = torch.empty(256 << 20 if do_flush else 1, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    plan_variant = variant
    if variant == pkg.KV8_DECODE_AUTO:
        plan_variant = pkg.KV8_DECODE_TCGEN05 if (w.H >= 16 and tc_built(pkg, dev)) \
            else pkg.KV8_DECODE_SIMT
    if plan_variant == pkg.KV8_DECODE_TCGEN05:
        plan_variant = pkg.KV8_DECODE_TCGEN05_PAIR if w.H > 64 else pkg.KV8_DECODE_TCGEN05_CTA

    def step(evs=None):
        if evs is not None:
            evs[0].record(stream)
        if fresh is not None:
            pkg.kv8_quantize_rows(fresh, codes, scales, dst_slot=fresh_slots)
        if evs is not None:
            evs[1].record(stream)
        pkg.mla_absorb_decode_fp8_batch_partials(ql, qr, codes, scales, bt, sl, w.sm_scale, ws,
                                                 variant=variant)
        if evs is not None:
            evs[2].record(stream)
        pkg.mla_absorb_decode_fp8_batch_combine(sl, w.H, w.max_blocks, out, lse, ws,
                                                variant=variant)
        if evs is not None:
            evs[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pkg.kv8_workspace_error(ws) == 0

    # The timed steps replay CUDA graphs of the three phases (captured from the same
    # calls), so the device-timed value is kernel time, not host launch latency; the
    # e2e number below goes through the public call as a user makes it.
    graphs = []
    for phase in range(3):
        if phase == 0 and fresh is None:
            graphs.append(None)
            continue
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if phase == 0:
                pkg.kv8_quantize_rows(fresh, codes, scales, dst_slot=fresh_slots)
            elif phase == 1:
                pkg.mla_absorb_decode_fp8_batch_partials(ql, qr, codes, scales, bt, sl, w.sm_scale,
                                                         ws, variant=variant)
            else:
                pkg.mla_absorb_decode_fp8_batch_combine(sl, w.H, w.max_blocks, out, lse, ws,
                                                        variant=variant)
        graphs.append(g)
    stream = torch.cuda.current_stream()

    def step(evs=None):  # noqa: F811 -- the graphed step replaces the direct one
        for phase in range(3):
            if evs is not None:
                evs[phase].record(stream)
            if graphs[phase] is not None:
                graphs[phase].replay()
        if evs is not None:
            evs[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert pkg.kv8_workspace_error(ws) == 0

    sampler = ClockSampler(local_rank) if rank == 0 else None
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    # keep the GPU busy for the sampler's first samples, then time exactly K steps
    t_wall = time.perf_counter()
    for k in range(args.steps):
        if do_flush:
            flush_l2(flush)  # evict L2 between timed steps (outside the step's events)
        step(evs[k])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None

    step_ms = np.array([e[0].elapsed_time(e[3]) for e in evs])
    dec_ms = np.array([e[1].elapsed_time(e[2]) for e in evs])
    q_ms = np.array([e[0].elapsed_time(e[1]) for e in evs])
    comb_ms = np.array([e[2].elapsed_time(e[3]) for e in evs])
    ms_step = float(step_ms.mean())
    ms_dec = float(dec_ms.mean())

    # ---- e2e through the public fused call, host buffers in the timed region
    q_host = torch.cat([ql, qr], dim=2).cpu().pin_memory()
    ql_h = q_host[..., :512].contiguous().pin_memory()
    qr_h = q_host[..., 512:].contiguous().pin_memory()
    fr_h = w.fresh_rows
    fresh_h = torch.from_numpy(fr_h).pin_memory() if fr_h is not None else None
    out_h = torch.empty((w.B, w.H, 512), dtype=torch.float32).pin_memory()
    ql_d, qr_d = torch.empty_like(ql), torch.empty_like(qr)
    fresh_d = torch.empty_like(fresh) if fresh is not None else None

    def e2e_step():
        ql_d.copy_(ql_h, non_blocking=True)
        qr_d.copy_(qr_h, non_blocking=True)
        if fresh_d is not None:
            fresh_d.copy_(fresh_h, non_blocking=True)
            pkg.kv8_quantize_rows(fresh_d, codes, scales, dst_slot=fresh_slots)
        pkg.mla_absorb_decode_fp8_batch(ql_d, qr_d, codes, scales, bt, sl, w.sm_scale, out=out,
                                        workspace=ws, variant=variant)
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for k in range(args.steps):
        if do_flush:
            flush_l2(flush)
        e2e_evs[k][0].record(stream)
        e2e_step()
        e2e_evs[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in e2e_evs]))
    h2d = ql_h.numel() * 4 + qr_h.numel() * 4 + (fresh_h.numel() * 4 if fresh_h is not None else 0)
    d2h = out_h.numel() * 4

    # ---- max over ranks
    ms_step, ms_dec, e2e_ms = slowest_rank([ms_step, ms_dec, e2e_ms], dev)
    if rank != 0:
        return None

    kv_bytes = w.kv_bytes() * world
    tok_heads = w.total_tokens * w.H * world
    value = kv_bytes / (ms_step * 1e-3) / 1e9
    peaks = load_peaks()
    flops = FLOP_PER_TOKEN_HEAD * w.total_tokens * w.H
    if plan_variant in (pkg.KV8_DECODE_TCGEN05_PAIR, pkg.KV8_DECODE_TCGEN05_CTA):
        kernel = "decode_pair" if plan_variant == pkg.KV8_DECODE_TCGEN05_PAIR else "decode_tc"
        # both contractions on e4m3 operands: the e4m3 tensor peak is twice the measured
        # bf16 dense peak (the nominal fp8 / bf16 ratio)
        p8 = 2 * peaks["bf16_tflops"] * 1e12
        t_tensor = flops / p8
        t_hbm = w.kv_bytes() / (peaks["hbm_gbs"] * 1e9)
        if t_tensor >= t_hbm:
            roof = {"bound": "tensor", "achieved": flops / (ms_dec * 1e-3) / 1e12,
                    "peak": p8 / 1e12, "unit": "TFLOP/s",
                    "peak_note": f"{peaks['src']} bf16 dense burst x 2 (e4m3 operands)"}
        else:
            roof = {"bound": "hbm", "achieved": w.kv_bytes() / (ms_dec * 1e-3) / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "peak_note": f"{peaks['src']} copy",
                    "tensor_frac": flops / (ms_dec * 1e-3) / p8}
    else:
        kernel = "decode_simt"
        alu_peak = NUM_SMS * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12
        t_alu = flops / (alu_peak * 1e12)
        t_hbm = w.kv_bytes() / (peaks["hbm_gbs"] * 1e9)
        if t_alu >= t_hbm:
            roof = {"bound": "alu", "achieved": flops / (ms_dec * 1e-3) / 1e12, "peak": alu_peak,
                    "unit": "TFLOP/s",
                    "peak_note": "152 SMs x 128 FP32 lanes x 2 FLOP x max SM clock"}
        else:
            roof = {"bound": "hbm", "achieved": w.kv_bytes() / (ms_dec * 1e-3) / 1e9,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "peak_note": f"{peaks['src']} copy"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_for(kernel, args.workload)
    roof["kernel"] = kernel
    roof["ms_per_launch"] = ms_dec
    roof["algorithmic"] = {"bytes": w.kv_bytes(), "flops": flops,
                           "per_unit": "584 B and 2176*H FLOP per (token, sequence)"}

    res = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPES[plan_variant],
        "data": "synthetic (seeded; the workload's shapes, page layout and value mix)",
        "token_heads_per_s": tok_heads / (ms_step * 1e-3),
        "config": {"workload": args.workload, "scale": args.scale, "B": w.B, "H": w.H,
                   "T_total": w.total_tokens, "kv_lora": 512, "qk_rope": 64,
                   "variant": {1: "simt", 3: "tcgen05_cta", 4: "tcgen05_pair"}[plan_variant],
                   "l2": ("flushed between steps (256 MB written, then read)" if do_flush else
                          f"no flush: the step's inputs ({in_bytes / 1e6:.0f} MB) are over twice "
                          "L2 (129 MB)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "phases_ms": {"quantize": float(q_ms.mean()), "decode": ms_dec,
                      "combine": float(comb_ms.mean())},
        "roofline": roof,
        "e2e": {"value": kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        # per step: the fresh rows' quantizer (append), the query prep (tensor-core
        # kernels), the decode kernel and the combine kernel
        "gpu_launches": args.steps * ((1 if fresh is not None else 0) +
                                     (1 if plan_variant == pkg.KV8_DECODE_SIMT else 2) + 1),
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    return res, w


# the decode configs, in the order of the lines; the long-context one, the headline,
# comes last
DECODE_ORDER = ("tiny", "single", "batched", "append", "long")

# what each decode kernel computes in (the cache is e4m3 in every case)
DTYPES = {
    1: "e4m3 cache; f32 arithmetic on CUDA cores",
    3: "e4m3 cache; two-term e4m3 query and two-term e4m3 weights on tcgen05; f32 accumulation",
    4: "e4m3 cache; two-term e4m3 query and two-term e4m3 weights on tcgen05; f32 accumulation",
}


PRODUCE_METRIC = "fp8-latent fused producer (RMS norm + rotary + e4m3 quantize + paged write): GB/s"
PRODUCE_ROW_BYTES = 2304 + 8 + 8 + 576 + 8   # f32 row, position, slot in; codes, scales out


def run_produce(args, rank, world, local_rank):
    """The fused producer step of the append workload: 65536 raw rows -> cache slots."""
    import torch
    import fp8_mla_latent_gb300 as pkg
    from fp8_mla_latent_gb300 import workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    n = max(1, int(65536 * args.scale))
    p = workloads.producer_inputs(n)
    rows = torch.from_numpy(p.rows).to(dev)
    weight = torch.from_numpy(p.weight).to(dev)
    pos = torch.from_numpy(p.positions).to(dev)
    cos = torch.from_numpy(p.rope_cos).to(dev)
    sin = torch.from_numpy(p.rope_sin).to(dev)
    slots = torch.from_numpy(p.slots).to(dev)
    codes = torch.zeros((p.n_slots, 576), dtype=torch.uint8, device=dev)
    scales = torch.zeros((p.n_slots, 2), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def once():
        pkg.kv8_produce_rows(rows, weight, p.eps, pos, cos, sin, codes, scales, dst_slot=slots,
                             err_word=err)

    for _ in range(args.warmup):
        flush_l2(flush)
        once()
    torch.cuda.synchronize()
    rank_sync()
    sampler = ClockSampler(local_rank)
    sampler.start()
    times = []
    for _ in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        once()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    clocks = sampler.stop()
    rank_sync()
    ms, = slowest_rank([float(np.mean(times))], dev)
    nbytes = n * PRODUCE_ROW_BYTES
    value = world * nbytes / (ms * 1e-3) / 1e9
    # end to end: raw rows from pinned host memory, error word back
    host_rows = torch.from_numpy(p.rows).pin_memory()
    host_err = torch.zeros(1, dtype=torch.int32).pin_memory()
    e2e = []
    for k in range(args.warmup + args.steps):
        flush_l2(flush)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rows.copy_(host_rows, non_blocking=True)
        once()
        host_err.copy_(err, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    e2e_ms, = slowest_rank([float(np.mean(e2e))], dev)
    peaks = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    res = {
        "metric": PRODUCE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 in, e4m3 + f32 scales out",
        "data": "synthetic (seeded; the append workload's value mix)",
        "rows_per_s": world * n / (ms * 1e-3),
        "config": {"workload": "produce", "rows": n, "max_pos": int(p.rope_cos.shape[0]),
                   "l2": "flushed between steps (256 MB written, then read); rows > L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic_for("produce_rows", "produce") if n == 65536 else None,
                     "kernel": "produce_rows", "ms_per_launch": ms,
                     "peak_note": f"{peaks['src']} copy",
                     "algorithmic": {"bytes": nbytes, "per_unit": f"{PRODUCE_ROW_BYTES} B per row"}},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": n * 2304, "d2h_bytes_per_step": 4},
        "gpu_launches": args.steps,
        "clocks": clocks if clocks else {"note": "timed region shorter than the 50 ms sampling period"},
    }
    return res, p


WUV_METRIC = "fp8-latent MLA decode W_UV epilogue (per-head value projection): GB/s"


def run_wuv(args, rank, world, local_rank):
    """The W_UV epilogue after the long workload's decode: B=2 sequences, H=128, V=128."""
    import torch
    import fp8_mla_latent_gb300 as pkg

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    B, H, V = 2, 128, 128
    rng = np.random.default_rng(9)
    o = torch.from_numpy(rng.standard_normal((B, H, 512)).astype(np.float32)).to(dev)
    w = torch.from_numpy((rng.standard_normal((H, 512, V)) / np.sqrt(512)).astype(np.float32))
    w = w.to(torch.bfloat16).to(dev)
    y = torch.empty((B, H, V), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush_l2(flush)
        pkg.mla_wuv_epilogue(o, w, y)
    torch.cuda.synchronize()
    rank_sync()
    times = []
    for _ in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pkg.mla_wuv_epilogue(o, w, y)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    rank_sync()
    ms, = slowest_rank([float(np.mean(times))], dev)
    nbytes = H * 512 * V * 2 + B * H * 512 * 4 + B * H * V * 4
    peaks = load_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {
        "metric": WUV_METRIC, "value": world * achieved, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 weights, f32 accum",
        "data": "synthetic (seeded)",
        "config": {"workload": "wuv", "B": B, "H": H, "V": V, "l2": "flushed between steps (256 MB written, then read)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic_for("wuv", "wuv"),
                     "kernel": "wuv",
                     "ms_per_launch": ms, "peak_note": f"{peaks['src']} copy",
                     "algorithmic": {"bytes": nbytes, "per_unit": "H*512*V bf16 weights + B*H*(512+V) f32"}},
        "gpu_launches": args.steps,
        "clocks": {"note": "timed region shorter than the 50 ms sampling period"},
    }


PREFILL_METRIC = "fp8-latent non-absorbed prefill projection (cached latent x kv_b, rope keys): TFLOP/s"


def prefill_bytes(T, N):
    """Algorithmic bytes of one launch: the cached rows read once, W read once, Y and
    the rope keys written once."""
    return T * ROW_BYTES + 512 * N * 2 + T * N * 2 + T * 64 * 4


def run_prefill(args, rank, world, local_rank):
    """The projection of one 4096-token prompt chunk: Y = dequantized Lc x W_UKV
    (bf16 [512, 32768]) plus the dequantized rope keys."""
    import torch
    import fp8_mla_latent_gb300 as pkg
    from fp8_mla_latent_gb300 import workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T = max(128, int(4096 * args.scale))
    p = workloads.prefill_inputs(T)
    N = p.w_ukv.shape[1]
    codes = torch.zeros((p.n_slots, 576), dtype=torch.uint8, device=dev)
    scales = torch.zeros((p.n_slots, 2), dtype=torch.float32, device=dev)
    slots = torch.from_numpy(p.slots).to(dev)
    pkg.kv8_quantize_rows(torch.from_numpy(p.rows).to(dev), codes, scales, dst_slot=slots)
    w = torch.from_numpy(p.w_ukv).to(torch.bfloat16).to(dev)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    k_rope = torch.empty((T, 64), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def once():
        pkg.kv8_prefill_project(codes, scales, w, slots=slots, y=y, k_rope=k_rope, err_word=err)

    for _ in range(args.warmup):
        flush_l2(flush)
        once()
    torch.cuda.synchronize()
    rank_sync()
    sampler = ClockSampler(local_rank)
    sampler.start()
    times = []
    for _ in range(args.steps):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        once()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    clocks = sampler.stop()
    assert err.item() == 0, f"prefill error word {err.item()}"
    rank_sync()
    ms, = slowest_rank([float(np.mean(times))], dev)
    flops = 2.0 * T * 512 * N
    tflops = flops / (ms * 1e-3) / 1e12
    # end to end: the chunk's cache rows and slot map from pinned host memory, Y and
    # the rope keys back to pinned host memory
    h_codes = codes.cpu().pin_memory()
    h_scales = scales.cpu().pin_memory()
    h_slots = slots.cpu().pin_memory()
    h_y = torch.empty((T, N), dtype=torch.bfloat16).pin_memory()
    h_k = torch.empty((T, 64), dtype=torch.float32).pin_memory()
    e2e = []
    for k in range(args.warmup + args.steps):
        flush_l2(flush)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        codes.copy_(h_codes, non_blocking=True)
        scales.copy_(h_scales, non_blocking=True)
        slots.copy_(h_slots, non_blocking=True)
        once()
        h_y.copy_(y, non_blocking=True)
        h_k.copy_(k_rope, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e.append(e0.elapsed_time(e1))
    e2e_ms, = slowest_rank([float(np.mean(e2e))], dev)
    peaks = load_peaks()
    nbytes = prefill_bytes(T, N)
    res = {
        "metric": PREFILL_METRIC, "value": world * tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 operands (e4m3 codes exact), f32 accum, bf16 out",
        "data": "synthetic (seeded; Gaussian rows with log-normal channel gains, N(0,1/512) weights)",
        "tokens_per_s": world * T / (ms * 1e-3),
        "config": {"workload": "prefill", "T": T, "N": N, "heads": 128, "qk_nope": 128, "v_head": 128,
                   "l2": "flushed between steps (256 MB written, then read)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                     "traffic": traffic_for("prefill", "prefill") if T == 4096 else None,
                     "kernel": "prefill", "ms_per_launch": ms,
                     "peak_note": f"{peaks['src']} cuBLAS bf16 burst",
                     "algorithmic": {"flops": flops, "per_unit": "2 x 512 x N flops per token",
                                     "bytes": nbytes, "hbm_gbs": nbytes / (ms * 1e-3) / 1e9}},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": T * ROW_BYTES + T * 8 + 1024 * ROW_BYTES,
                "d2h_bytes_per_step": T * N * 2 + T * 64 * 4},
        "gpu_launches": args.steps,
        "clocks": clocks if clocks else {"note": "timed region shorter than the 50 ms sampling period"},
    }
    return res, p


def prefill_cpu_baseline(p, budget_s=8.0):
    """The float64 oracle on a bounded sample: the first n tokens of the chunk, all
    N columns, n grown until about budget_s of wall time."""
    import oracle
    T = p.rows.shape[0]
    codes, scales = oracle.quantize_rows(p.rows, dst_slot=p.slots, n_slots=p.n_slots)
    wb = oracle_bf16_bits(p.w_ukv)
    n, dt = 16, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.prefill_project(codes, scales, wb, slots=p.slots[:n])
        oracle.prefill_rope(codes, scales, p.slots[:n])
        dt = time.perf_counter() - t0
        if dt > budget_s / 4 or n >= T:
            break
        n = min(T, n * 4)
    N = wb.shape[1]
    value = 2.0 * n * 512 * N / dt / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} of {T} tokens x {N} columns, float64 numpy, {dt:.2f} s wall"}


def oracle_bf16_bits(w):
    """The bf16 bit patterns of the weights, rounded as the GPU arm rounds them."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


PERSIST_METRIC = "fp8 cache save + resume through the cache file (COLIKV2 records): GB/s"


def run_persist(args, rank, world, local_rank):
    """Append 65536 cache rows (the append workload's fresh rows, at scattered slots) to
    the cache file through a persistent handle and load them back into other slots: one
    step.  The calls are synchronous host I/O (page cache, no fsync), so the step is
    timed on the host."""
    import shutil
    import tempfile

    import torch
    import fp8_mla_latent_gb300 as pkg
    from fp8_mla_latent_gb300 import workloads

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    n = max(1, int(65536 * args.scale))
    p = workloads.producer_inputs(n)
    codes = torch.zeros((p.n_slots, 576), dtype=torch.uint8, device=dev)
    scales = torch.zeros((p.n_slots, 2), dtype=torch.float32, device=dev)
    slots = torch.from_numpy(p.slots).to(dev)
    pkg.kv8_quantize_rows(torch.from_numpy(p.rows).to(dev), codes, scales, dst_slot=slots)
    back = torch.from_numpy(np.random.default_rng(5).permutation(p.n_slots)[:n].astype(np.int64)).to(dev)
    c2, s2 = torch.zeros_like(codes), torch.zeros_like(scales)
    tmp = tempfile.mkdtemp(prefix=f"kv8_persist_{rank}_")
    staging = 4096
    # one persistent handle (opened outside the timed steps, as a server keeps it):
    # each step appends the rows and loads the rows it just appended back
    disk = pkg.Kv8Disk(os.path.join(tmp, "cache.kv"), staging_rows=staging)

    def step():
        t0 = time.perf_counter()
        disk.append(codes, scales, slots=slots)
        t1 = time.perf_counter()
        disk.load(c2, s2, first_row=disk.info()[0] - n, dst_slot=back)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    try:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        rank_sync()
        times = [step() for _ in range(args.steps)]
        rank_sync()
    finally:
        disk.close()
        shutil.rmtree(tmp, ignore_errors=True)
    ok = bool(torch.equal(c2[back], codes[slots]))
    save_ms = 1e3 * float(np.mean([a for a, _ in times]))
    load_ms = 1e3 * float(np.mean([b for _, b in times]))
    save_ms, load_ms = slowest_rank([save_ms, load_ms], dev)
    ms = save_ms + load_ms
    nbytes = 2 * n * 584
    value = world * nbytes / (ms * 1e-3) / 1e9
    chunks = (n + staging - 1) // staging
    return {
        "metric": PERSIST_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8 codes + f32 scales (bytes moved)",
        "data": "synthetic (seeded; the producer workload's rows, quantized, at scattered slots)",
        "config": {"workload": "persist", "rows": n, "staging_rows": staging,
                   "file": "one file on the host's temporary directory, one handle opened before the timed steps; each step appends the rows and loads them back (page cache, no fsync)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "phases_ms": {"save": save_ms, "load": load_ms},
        "save_gbs": n * 584 / (save_ms * 1e-3) / 1e9, "load_gbs": n * 584 / (load_ms * 1e-3) / 1e9,
        "round_trip_bit_exact": ok,
        "roofline": {"bound": "io", "achieved": value, "peak": None, "unit": "GB/s", "frac": None,
                     "traffic": None, "kernel": "gather_kernel / scatter_kernel + file I/O",
                     "note": "host file I/O through the page cache dominates; no device roofline",
                     "algorithmic": {"bytes": nbytes, "per_unit": "584 B per row, each way"}},
        "e2e": {"value": value, "unit": "GB/s", "ms_per_step": ms,
                "h2d_bytes_per_step": n * 584, "d2h_bytes_per_step": n * 584},
        "gpu_launches": 2 * chunks * args.steps,
        "clocks": {"note": "host-timed I/O step"},
    }, p


def persist_cpu_baseline(p, budget_s=4.0):
    """The oracle's writer and reader of the file on the same rows, from host arrays."""
    import tempfile
    import oracle
    from oracle import coli_kv
    codes, scales = oracle.quantize_rows(p.rows)
    n = codes.shape[0]
    d = tempfile.mkdtemp(prefix="kv8_persist_oracle_")
    path = os.path.join(d, "o.kv")
    t0 = time.time()
    k = 0
    while time.time() - t0 < budget_s and k < 20:
        coli_kv.write_v2(path, codes, scales)
        coli_kv.read(path)
        k += 1
    dt = time.time() - t0
    os.remove(path)
    os.rmdir(d)
    return {"value": 2 * k * n * 584 / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{k} save + read round trips of {n} rows, numpy + Python file I/O, {dt:.2f} s wall"}


def produce_cpu_baseline(p, budget_s=8.0):
    import oracle
    n = p.rows.shape[0]
    t0 = time.time()
    done = 0
    while time.time() - t0 < budget_s and done < 4 * n:
        oracle.produce_rows(p.rows, p.weight, p.eps, p.positions, p.rope_cos, p.rope_sin,
                            dst_slot=p.slots, n_slots=p.n_slots)
        done += n
    dt = time.time() - t0
    return {"value": done * PRODUCE_ROW_BYTES / dt / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "sample": f"{done} rows of the producer workload, plain C, {dt:.2f} s wall"}


def tc_built(pkg, dev):
    import torch
    try:
        q = torch.zeros((16, 512), device=dev)
        r = torch.zeros((16, 64), device=dev)
        c = torch.zeros((1, 576), dtype=torch.uint8, device=dev)
        s = torch.zeros((1, 2), device=dev)
        pkg.mla_absorb_decode_fp8(q, r, c, s, 1, 0.1, variant=pkg.KV8_DECODE_TCGEN05)
        torch.cuda.synchronize()
        return True
    except pkg.Kv8Error:
        return False


# ----------------------------------------------------------------- oracle (CPU) arm
def oracle_sample(w, budget_s, codes=None, scales=None, n_threads=None):
    """Time the f32 oracle (OpenMP over heads; all cores unless n_threads) on a
    bounded sample of the workload: sequence 0, the first n heads, n sized to about
    budget_s of wall time.  value is the sample's rate (KV bytes of the heads it
    covered per second), the same rate the whole job would run at."""
    import oracle
    if codes is None:
        codes, scales = oracle.quantize_rows(w.cache_rows, dst_slot=w.cache_slots,
                                             n_slots=w.n_slots)
        if w.fresh_rows is not None:
            oracle.quantize_rows(w.fresh_rows, dst_slot=w.fresh_slots, codes=codes, scales=scales)
    # the thread count is always passed explicitly: the OpenMP setting a call makes
    # outlives it, so asking the runtime after a one-core sample would answer 1
    cores = len(os.sched_getaffinity(0)) if n_threads is None else int(n_threads)
    b = 0
    T = int(w.seq_lens[b])

    def run(nh):
        t0 = time.perf_counter()
        oracle.attention_batch_f32(w.q_lat[b:b + 1, :nh], w.q_rope[b:b + 1, :nh], codes, scales,
                                   w.block_table[b:b + 1], w.seq_lens[b:b + 1], w.sm_scale,
                                   n_threads=cores)
        return time.perf_counter() - t0

    nh = min(w.H, cores)
    t1 = run(nh)
    per_head = t1 / nh
    n2 = int(max(1, min(w.H, budget_s / max(per_head, 1e-6))))
    if n2 > nh:
        nh, t1 = n2, run(n2)
    # the rate: KV bytes per (token, head) share, over the sample's time
    per_tok_head = t1 / (nh * T)
    t_full = per_tok_head * w.total_tokens * w.H
    value = w.kv_bytes() / t_full / 1e9
    sample = f"sequence 0 ({T} tokens) x {nh} of {w.H} heads, f32 oracle, {t1:.2f} s wall"
    return {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
            "seconds": t1, "projected_full_job_s": t_full}, (codes, scales)


def cpu_baselines(w, budget_s):
    """The oracle on all host cores (the reported value) and on one core."""
    allc, cache = oracle_sample(w, budget_s)
    one, _ = oracle_sample(w, budget_s, *cache, n_threads=1)
    res = {k: allc[k] for k in ("value", "unit", "cores", "kind", "sample")}
    res["one_core"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
    return res


def run_reference(args, world):
    from fp8_mla_latent_gb300 import workloads
    import oracle
    if args.workload == "persist":
        p = workloads.producer_inputs(max(1, int(65536 * args.scale)))
        persist_cpu_baseline(p, 0.5)
        vals = [persist_cpu_baseline(p, 1.0) for _ in range(args.steps)]
        value = float(np.mean([v["value"] for v in vals]))
        n = p.rows.shape[0]
        return {
            "impl": "reference", "metric": PERSIST_METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 2 * n * 584 / (value * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8 + f32",
            "data": "synthetic (seeded; same rows as our arm)",
            "config": {"workload": "persist", "rows": n},
            "cpu_baseline": dict(vals[-1], value=value),
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    if args.workload == "prefill":
        p = workloads.prefill_inputs(max(128, int(4096 * args.scale)))
        prefill_cpu_baseline(p, 0.5)
        vals = [prefill_cpu_baseline(p, 2.0) for _ in range(args.steps)]
        value = float(np.mean([v["value"] for v in vals]))
        T, N = p.rows.shape[0], p.w_ukv.shape[1]
        return {
            "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 2.0 * T * 512 * N / (value * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; same inputs as our arm)",
            "config": {"workload": "prefill", "T": T, "N": N},
            "cpu_baseline": dict(vals[-1], value=value),
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    if args.workload == "produce":
        p = workloads.producer_inputs(max(1, int(65536 * args.scale)))
        for _ in range(args.warmup):
            produce_cpu_baseline(p, 0.1)
        vals = [produce_cpu_baseline(p, 1.0) for _ in range(args.steps)]
        value = float(np.mean([v["value"] for v in vals]))
        return {
            "impl": "reference", "metric": PRODUCE_METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": p.rows.shape[0] * PRODUCE_ROW_BYTES / (value * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; same rows as our arm)",
            "config": {"workload": "produce", "rows": int(p.rows.shape[0])},
            "cpu_baseline": dict(vals[-1], value=value),
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    return ref_decode(args.workload, args, world, 1.0)


def ref_decode(name, args, world, budget_s):
    """The oracle arm on one decode workload: each step a bounded sample (sequence 0,
    as many heads as fit in budget_s).  ms_per_step is the measured time of the
    sample; value is its rate, which the whole job would run at."""
    from fp8_mla_latent_gb300 import workloads
    w = workloads.make(name)
    cache = None
    for _ in range(args.warmup):
        _, cache = oracle_sample(w, min(0.2, budget_s), *(cache or (None, None)))
    vals, secs = [], []
    cb = None
    for _ in range(args.steps):
        cb, cache = oracle_sample(w, budget_s, *cache)
        vals.append(cb["value"])
        secs.append(cb["seconds"])
    value = float(np.mean(vals))
    ms = float(np.mean(secs)) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; same workload as our arm)",
        "config": {"workload": name, "scale": args.scale, "B": w.B, "H": w.H,
                   "T_total": w.total_tokens},
        "step": "a bounded sample of the workload: " + cb["sample"] +
                "; ms_per_step is that sample's measured time",
        "projected_full_job_ms": w.kv_bytes() / (value * 1e9) * 1e3,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cb["cores"], "kind": "oracle",
                         "sample": cb["sample"] + f"; {args.steps} steps"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the CPU oracle (plain C, OpenMP over heads) stands in for the reference; "
                "the source pages ship no runnable implementation",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="all",
                    help="a decode workload, 'all' (one line per decode config, the long one "
                         "last), or produce / wuv / prefill / persist")
    ap.add_argument("--variant", default="auto", choices=["auto", "simt", "tcgen05", "tc_cta", "tc_pair"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="shrink token counts (profiling captures only; the bench line is scale 1)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            if args.workload == "all":
                for name in DECODE_ORDER:
                    print(json.dumps(ref_decode(name, args, world, 1.0 if name == "long" else 0.25)),
                          flush=True)
            else:
                print(json.dumps(run_reference(args, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.workload == "wuv":
        res = run_wuv(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
    elif args.workload == "persist":
        res, p = run_persist(args, rank, world, local_rank)
        if rank == 0:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = persist_cpu_baseline(p)
            print(json.dumps(res), flush=True)
    elif args.workload == "prefill":
        res, p = run_prefill(args, rank, world, local_rank)
        if rank == 0:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = prefill_cpu_baseline(p)
            print(json.dumps(res), flush=True)
    elif args.workload == "produce":
        res, p = run_produce(args, rank, world, local_rank)
        if rank == 0:
            if not args.no_cpu_baseline:
                res["cpu_baseline"] = produce_cpu_baseline(p)
            print(json.dumps(res), flush=True)
    else:
        import copy
        import torch
        names = DECODE_ORDER if args.workload == "all" else (args.workload,)
        for name in names:
            a = copy.copy(args)
            a.workload = name
            r = run_ours(a, rank, world, local_rank)
            if rank == 0:
                res, w = r
                if not args.no_cpu_baseline:
                    res["cpu_baseline"] = cpu_baselines(w, 6.0 if name == "long" else 3.0)
                print(json.dumps(res), flush=True)
            del r
            torch.cuda.empty_cache()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
