"""Shared set-up for the GPU parity tests: upload a workload, fill the cache
with the library's quantizer, run a decode variant, and compare sampled
(sequence, head) outputs with the f64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import fp8_mla_latent_gb300 as pkg
import oracle

# max-abs error <= TOL * max|out| per sequence against the f64 oracle on the same codes:
#   CUDA-core kernel (f32 operands and accumulation): 2e-3;
#   tensor-core kernels (reduced-precision MMA operands: the query as two e4m3 terms on a
#   per-head power-of-two scale for the scores, in both kernels, and the softmax weights as
#   two e4m3 terms for the context; f32 accumulation): 1e-2.
TOLS = {1: 2e-3, 2: 1e-2, 3: 1e-2, 4: 1e-2}
NAMES = {1: "simt", 2: "tcgen05", 3: "tcgen05_cta", 4: "tcgen05_pair"}
LSE_TOL = 2e-3   # natural-log units
WORST = {}       # variant -> worst observed err / max|out|, reported by the tests


def dev():
    return torch.device("cuda:0")


def upload_cache(w, quantize_fresh=True):
    """Quantize the workload's rows into a fresh device cache; returns tensors."""
    d = dev()
    codes = torch.zeros((w.n_slots, 576), dtype=torch.uint8, device=d)
    scales = torch.zeros((w.n_slots, 2), dtype=torch.float32, device=d)
    rows = torch.from_numpy(w.cache_rows).to(d)
    slots = torch.from_numpy(w.cache_slots).to(d)
    pkg.kv8_quantize_rows(rows, codes, scales, dst_slot=slots)
    if quantize_fresh and w.fresh_rows is not None:
        pkg.kv8_quantize_rows(torch.from_numpy(w.fresh_rows).to(d), codes, scales,
                              dst_slot=torch.from_numpy(w.fresh_slots).to(d))
    return codes, scales


def decode(w, codes, scales, variant, lse=True, contiguous=None):
    d = dev()
    ql = torch.from_numpy(w.q_lat).to(d)
    qr = torch.from_numpy(w.q_rope).to(d)
    contiguous = w.contiguous if contiguous is None else contiguous
    if contiguous:
        T = int(w.seq_lens[0])
        l = torch.empty((w.H,), dtype=torch.float32, device=d) if lse else None
        ws = pkg.alloc_workspace(pkg.mla_absorb_decode_fp8_workspace_size(T, w.H, variant), d)
        out = pkg.mla_absorb_decode_fp8(ql[0], qr[0], codes, scales, T, w.sm_scale, lse=l,
                                        workspace=ws, variant=variant)
        torch.cuda.synchronize()
        err = pkg.kv8_workspace_error(ws)
        assert err == 0, f"workspace error status {err}"
        return out[None].cpu().numpy(), (l[None].cpu().numpy() if lse else None)
    bt = torch.from_numpy(w.block_table).to(d)
    sl = torch.from_numpy(w.seq_lens).to(d)
    l = torch.empty((w.B, w.H), dtype=torch.float32, device=d) if lse else None
    ws = pkg.alloc_workspace(pkg.mla_absorb_decode_fp8_batch_workspace_size(
        w.B, w.H, w.max_blocks, variant=variant), d)
    out = pkg.mla_absorb_decode_fp8_batch(ql, qr, codes, scales, bt, sl, w.sm_scale, lse=l,
                                          workspace=ws, variant=variant)
    torch.cuda.synchronize()
    err = pkg.kv8_workspace_error(ws)
    assert err == 0, f"workspace error status {err}"
    return out.cpu().numpy(), (l.cpu().numpy() if lse else None)


def oracle_heads(w, codes_np, scales_np, b, heads):
    T = int(w.seq_lens[b])
    slots = None if w.contiguous else oracle.paged_slots(w.block_table, b, T)
    h0, h1 = heads
    return oracle.attention_f64(w.q_lat[b], w.q_rope[b], codes_np, scales_np, T, w.sm_scale,
                                slots=slots, heads=(h0, h1 - h0))


def check(w, out, lse, codes_np, scales_np, pairs, variant=1):
    """pairs: list of (b, (h0, h1)) blocks to compare; returns the worst err / max|out|."""
    TOL = TOLS[variant]
    worst = 0.0
    for b, (h0, h1) in pairs:
        ref, ref_lse = oracle_heads(w, codes_np, scales_np, b, (h0, h1))
        got = out[b, h0:h1].astype(np.float64)
        scale = np.abs(ref).max()
        err = np.abs(got - ref).max()
        if int(w.seq_lens[b]) == 0:
            assert np.all(got == 0) and (lse is None or np.all(np.isneginf(lse[b, h0:h1])))
            continue
        assert np.isfinite(got).all(), f"non-finite output b={b}"
        assert err <= TOL * scale, f"b={b} h={h0}:{h1} err {err:.3e} > {TOL} * {scale:.3e}"
        worst = max(worst, err / scale)
        if lse is not None:
            lerr = np.abs(lse[b, h0:h1] - ref_lse).max()
            assert lerr <= LSE_TOL * max(1.0, np.abs(ref_lse).max()), f"lse err {lerr}"
    WORST[variant] = max(WORST.get(variant, 0.0), worst)
    return worst


def custom_workload(seqs, q_lat, q_rope, sm_scale=None, shuffle=True, seed=0):
    """A paged workload from explicit f32 rows: seqs = list of [T_b, 576] arrays,
    q_lat [B, H, 512], q_rope [B, H, 64]; pages in a random order of one pool."""
    from fp8_mla_latent_gb300 import workloads
    rng = np.random.default_rng(seed)
    lens = np.array([s.shape[0] for s in seqs], np.int32)
    bt, n_slots, slots = workloads._paged_tables(rng, lens, shuffle=shuffle)
    rows = np.concatenate(seqs).astype(np.float32) if len(seqs) else np.zeros((0, 576), np.float32)
    B, H = q_lat.shape[:2]
    return workloads.Workload("custom", B, H, lens, bt, n_slots, rows, slots, None, None,
                              np.ascontiguousarray(q_lat, np.float32),
                              np.ascontiguousarray(q_rope, np.float32),
                              sm_scale=workloads.SM_SCALE if sm_scale is None else sm_scale)
