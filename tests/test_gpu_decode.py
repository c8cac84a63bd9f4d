"""GPU decode parity against the f64 oracle.

Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description (absorbed attention over the e4m3 latent rows, each row
scale applied outside its dot product) and closing note (split-T).  Tolerance:
max-abs error <= 2e-3 * max|out| per sequence for the CUDA-core kernel (f32 throughout) and
<= 1e-2 * max|out| for the tensor-core kernels (reduced-precision MMA operands:
the query as two e4m3 terms on a per-head power-of-two scale for the scores, in
both kernels, the softmax weights as two e4m3 terms for the context; f32
accumulation); lse within 2e-3.  Every test runs the three kernels: CUDA-core,
one-CTA tensor-core and SM-pair tensor-core (the last two forced at any H).
Caches are filled by the library's quantizer and the oracle reads the same
codes, so these tests isolate attention.
"""
import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
from fp8_mla_latent_gb300 import workloads

from gpu_helpers import check, decode, upload_cache

pytestmark = pytest.mark.gpu

VARIANTS = {"simt": pkg.KV8_DECODE_SIMT, "tc_cta": pkg.KV8_DECODE_TCGEN05_CTA,
            "tc_pair": pkg.KV8_DECODE_TCGEN05_PAIR}
TENSOR = (pkg.KV8_DECODE_TCGEN05_CTA, pkg.KV8_DECODE_TCGEN05_PAIR)


def tc_ready():
    try:
        d = torch.device("cuda:0")
        q = torch.zeros((16, 512), device=d)
        r = torch.zeros((16, 64), device=d)
        c = torch.zeros((1, 576), dtype=torch.uint8, device=d)
        s = torch.zeros((1, 2), device=d)
        pkg.mla_absorb_decode_fp8(q, r, c, s, 1, 0.1, variant=pkg.KV8_DECODE_TCGEN05)
        return True
    except pkg.Kv8Error as e:
        if e.status == -3:
            return False
        raise


@pytest.fixture(params=list(VARIANTS))
def variant(request):
    v = VARIANTS[request.param]
    if v in TENSOR and not tc_ready():
        pytest.skip("tensor-core decode not built in this library")
    return v


def all_pairs(w, head_block=None):
    hb = head_block or w.H
    return [(b, (h, min(h + hb, w.H))) for b in range(w.B) for h in range(0, w.H, hb)]


SMALL = [("tiny", 1.0), ("single", 0.25), ("batched", 0.03), ("long", 0.01), ("append", 0.05)]


@pytest.mark.parametrize("name,scale", SMALL)
def test_workloads_small(name, scale, variant):
    w = workloads.make(name, scale=scale)
    codes, scales = upload_cache(w)
    out, lse = decode(w, codes, scales, variant)
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    rng = np.random.default_rng(0)
    if w.H * int(w.seq_lens.sum()) <= 4_000_000:
        pairs = all_pairs(w)
    else:  # every sequence, a random block of 8 heads
        pairs = [(b, (h, h + 8)) for b in range(w.B)
                 for h in [int(rng.integers(0, max(1, w.H - 8)))]]
    check(w, out, lse, c, s, pairs, variant)


@pytest.mark.parametrize("T", [1, 2, 31, 33, 63, 64, 65, 127, 128, 129, 255, 300, 1000])
@pytest.mark.parametrize("H", [1, 3, 16, 17, 64, 100, 128])
def test_ragged_lengths_and_head_counts(T, H, variant):
    if H * T > 128 * 300 and T > 300:
        pytest.skip("covered by the workload tests")
    rng = np.random.default_rng(T * 1000 + H)
    w = workloads.make("tiny", scale=1.0, seed=T + H)
    x = rng.standard_normal((T, 576)).astype(np.float32) * np.exp(
        0.5 * rng.standard_normal(576)).astype(np.float32)
    w.cache_rows = x
    w.cache_slots = np.arange(T, dtype=np.int64)
    w.n_slots = ((T + 63) // 64) * 64
    w.seq_lens = np.array([T], np.int32)
    w.block_table = np.arange(w.n_slots // 64, dtype=np.int32)[None]
    w.H = H
    w.q_lat = rng.standard_normal((1, H, 512)).astype(np.float32)
    w.q_rope = rng.standard_normal((1, H, 64)).astype(np.float32)
    codes, scales = upload_cache(w)
    for contiguous in (True, False):
        out, lse = decode(w, codes, scales, variant, contiguous=contiguous)
        check(w, out, lse, codes.cpu().numpy(), scales.cpu().numpy(), all_pairs(w), variant)


def test_empty_cache_single(variant):
    d = torch.device("cuda:0")
    q = torch.randn((16, 512), device=d)
    r = torch.randn((16, 64), device=d)
    c = torch.zeros((1, 576), dtype=torch.uint8, device=d)
    s = torch.zeros((1, 2), device=d)
    lse = torch.empty(16, device=d)
    out = pkg.mla_absorb_decode_fp8(q, r, c, s, 0, 0.1, lse=lse, variant=variant)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_batch_with_empty_and_short_sequences(variant):
    w = workloads.make("batched", scale=0.01)
    w.seq_lens = w.seq_lens.copy()
    w.seq_lens[0] = 0
    w.seq_lens[1] = 1
    w.seq_lens[2] = 64
    codes, scales = upload_cache(w)
    out, lse = decode(w, codes, scales, variant)
    check(w, out, lse, codes.cpu().numpy(), scales.cpu().numpy(),
          [(b, (0, 16)) for b in range(6)], variant)


def test_paged_permutation_is_bitwise_identical(variant):
    """Same tokens in the same logical order: any physical page permutation gives
    the same bits."""
    w = workloads.make("long", scale=0.01)
    codes, scales = upload_cache(w)
    out_a, lse_a = decode(w, codes, scales, variant)
    rng = np.random.default_rng(1)
    nb = w.n_slots // 64
    perm = rng.permutation(nb).astype(np.int32)
    c2 = torch.empty_like(codes)
    s2 = torch.empty_like(scales)
    p = torch.from_numpy(perm.astype(np.int64)).to(codes.device)
    c2.view(nb, 64, 576)[p] = codes.view(nb, 64, 576)
    s2.view(nb, 64, 2)[p] = scales.view(nb, 64, 2)
    w.block_table = perm[w.block_table]
    out_b, lse_b = decode(w, c2, s2, variant)
    assert np.array_equal(out_a.view(np.uint32), out_b.view(np.uint32))
    assert np.array_equal(lse_a.view(np.uint32), lse_b.view(np.uint32))


def test_bad_block_table_and_seq_len_report_ebounds(variant):
    w = workloads.make("batched", scale=0.01)
    codes, scales = upload_cache(w)
    d = torch.device("cuda:0")
    bt = torch.from_numpy(w.block_table).to(d)
    bt[0, 0] = 10 ** 6
    bt[1, 1] = -5
    sl = torch.from_numpy(w.seq_lens).to(d)
    sl[2] = w.max_blocks * 64 + 1000
    ql = torch.from_numpy(w.q_lat).to(d)
    qr = torch.from_numpy(w.q_rope).to(d)
    ws = pkg.alloc_workspace(pkg.mla_absorb_decode_fp8_batch_workspace_size(
        w.B, w.H, w.max_blocks, variant=variant), d)
    out = pkg.mla_absorb_decode_fp8_batch(ql, qr, codes, scales, bt, sl, w.sm_scale,
                                          workspace=ws, variant=variant)
    assert pkg.kv8_workspace_error(ws) == -5
    assert torch.isfinite(out[3:]).all()
    # a clean call on the same workspace clears the error word
    pkg.mla_absorb_decode_fp8_batch(ql, qr, codes, scales, torch.from_numpy(w.block_table).to(d),
                                    torch.from_numpy(w.seq_lens).to(d), w.sm_scale, workspace=ws,
                                    variant=variant)
    assert pkg.kv8_workspace_error(ws) == 0


def test_split_phases_equal_the_fused_call(variant):
    w = workloads.make("append", scale=0.05)
    codes, scales = upload_cache(w)
    d = torch.device("cuda:0")
    ql = torch.from_numpy(w.q_lat).to(d)
    qr = torch.from_numpy(w.q_rope).to(d)
    bt = torch.from_numpy(w.block_table).to(d)
    sl = torch.from_numpy(w.seq_lens).to(d)
    ws = pkg.alloc_workspace(pkg.mla_absorb_decode_fp8_batch_workspace_size(
        w.B, w.H, w.max_blocks, variant=variant), d)
    ref = pkg.mla_absorb_decode_fp8_batch(ql, qr, codes, scales, bt, sl, w.sm_scale,
                                          workspace=ws, variant=variant).clone()
    out = torch.empty_like(ref)
    lse = torch.empty((w.B, w.H), device=d)
    pkg.mla_absorb_decode_fp8_batch_partials(ql, qr, codes, scales, bt, sl, w.sm_scale, ws,
                                             variant=variant)
    pkg.mla_absorb_decode_fp8_batch_combine(sl, w.H, w.max_blocks, out, lse, ws, variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("B,T,H", [(100, 640, 16), (100, 600, 16), (50, 1000, 64)])
def test_ranges_across_sequences(B, T, H):
    """Shapes where the one-CTA kernel cuts the tiles of all sequences into equal
    ranges (a range runs from one sequence into the next): every sequence, on both
    sides of each range boundary, against the oracle; and the automatic choice
    gives the forced kernel's bits."""
    if not tc_ready():
        pytest.skip("tensor-core decode not built in this library")
    rng = np.random.default_rng(B + T + H)
    w = workloads.make("batched", scale=0.01, seed=5)
    w.B, w.H = B, H
    nb = (T + 63) // 64
    w.seq_lens = np.full(B, T, np.int32)
    w.n_slots = B * nb * 64
    perm = rng.permutation(B * nb).astype(np.int32)
    w.block_table = perm.reshape(B, nb)
    rows = []
    slots = []
    for b in range(B):
        x = rng.standard_normal((T, 576)).astype(np.float32)
        rows.append(x)
        pages = w.block_table[b]
        slots.append(pages[np.arange(T) // 64].astype(np.int64) * 64 + np.arange(T) % 64)
    w.cache_rows = np.concatenate(rows)
    w.cache_slots = np.concatenate(slots)
    w.fresh_rows = None
    w.q_lat = rng.standard_normal((B, H, 512)).astype(np.float32)
    w.q_rope = rng.standard_normal((B, H, 64)).astype(np.float32)
    codes, scales = upload_cache(w)
    out, lse = decode(w, codes, scales, pkg.KV8_DECODE_TCGEN05_CTA)
    c, s_ = codes.cpu().numpy(), scales.cpu().numpy()
    bs = sorted(set([0, 1, B // 2, B - 2, B - 1] + list(rng.choice(B, size=6, replace=False))))
    check(w, out, lse, c, s_, [(int(b), (0, H)) for b in bs], pkg.KV8_DECODE_TCGEN05_CTA)
    out_a, lse_a = decode(w, codes, scales, pkg.KV8_DECODE_TCGEN05)
    assert np.array_equal(out_a.view(np.uint32), out.view(np.uint32))
    assert np.array_equal(lse_a.view(np.uint32), lse.view(np.uint32))


FULL = ["single", "long", "batched", "append"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name, variant):
    """Full-size workloads in the benchmark's launch configuration; sampled heads."""
    if variant == pkg.KV8_DECODE_SIMT and name in ("long", "batched"):
        pytest.skip("the CUDA-core kernel is checked at full size on the smaller workloads")
    w = workloads.make(name)
    codes, scales = upload_cache(w)
    out, lse = decode(w, codes, scales, variant)
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    rng = np.random.default_rng(7)
    bs = rng.choice(w.B, size=min(w.B, 2), replace=False)
    pairs = [(int(b), (h, h + 1)) for b in bs for h in rng.choice(w.H, size=2, replace=False)]
    check(w, out, lse, c, s, pairs, variant)
    assert np.isfinite(out).all()


@pytest.mark.parametrize("H", [16, 64, 65, 128])
def test_automatic_tensor_core_choice(H):
    """TCGEN05 runs the SM-pair kernel for H > 64 and the one-CTA kernel otherwise:
    bit for bit the forced kernel's result."""
    if not tc_ready():
        pytest.skip("tensor-core decode not built in this library")
    w = workloads.make("batched", scale=0.02)
    rng = np.random.default_rng(H)
    w.H = H
    w.q_lat = rng.standard_normal((w.B, H, 512)).astype(np.float32)
    w.q_rope = rng.standard_normal((w.B, H, 64)).astype(np.float32)
    codes, scales = upload_cache(w)
    out_a, lse_a = decode(w, codes, scales, pkg.KV8_DECODE_TCGEN05)
    forced = pkg.KV8_DECODE_TCGEN05_PAIR if H > 64 else pkg.KV8_DECODE_TCGEN05_CTA
    out_f, lse_f = decode(w, codes, scales, forced)
    assert np.array_equal(out_a.view(np.uint32), out_f.view(np.uint32))
    assert np.array_equal(lse_a.view(np.uint32), lse_f.view(np.uint32))


def test_report_worst_error():
    """Not a check: prints the worst err/max|out| seen per kernel in this session."""
    from gpu_helpers import NAMES, WORST
    print("worst err / max|out|: " + ", ".join(f"{NAMES[k]} {v:.2e}" for k, v in sorted(WORST.items())))


def test_wrappers_reject_host_buffers_and_bad_shapes():
    """Arguments a kernel would misread are refused in Python, before any launch: a
    host workspace (a host pointer in a kernel faults the device), and out / lse /
    seq_lens of the wrong shape or type."""
    d = torch.device("cuda:0")
    H, B, MB = 16, 2, 4
    codes = torch.zeros((B * MB * 64, 576), dtype=torch.uint8, device=d)
    scales = torch.zeros((B * MB * 64, 2), device=d)
    host_ws = torch.empty(1 << 20, dtype=torch.uint8)
    q = torch.zeros((H, 512), device=d)
    r = torch.zeros((H, 64), device=d)
    with pytest.raises(ValueError, match="^workspace"):
        pkg.mla_absorb_decode_fp8(q, r, codes, scales, 10, 0.1, workspace=host_ws)
    with pytest.raises(ValueError, match="^out"):
        pkg.mla_absorb_decode_fp8(q, r, codes, scales, 10, 0.1, out=torch.empty((H, 256), device=d))
    with pytest.raises(ValueError, match="^lse"):
        pkg.mla_absorb_decode_fp8(q, r, codes, scales, 10, 0.1, lse=torch.empty(H + 1, device=d))
    ql = torch.zeros((B, H, 512), device=d)
    qr = torch.zeros((B, H, 64), device=d)
    bt = torch.arange(B * MB, dtype=torch.int32, device=d).reshape(B, MB)
    sl = torch.full((B,), 100, dtype=torch.int32, device=d)
    with pytest.raises(ValueError, match="^workspace"):
        pkg.mla_absorb_decode_fp8_batch(ql, qr, codes, scales, bt, sl, 0.1, workspace=host_ws)
    with pytest.raises(ValueError, match="^workspace"):
        pkg.mla_absorb_decode_fp8_batch_partials(ql, qr, codes, scales, bt, sl, 0.1, host_ws)
    out = torch.empty((B, H, 512), device=d)
    lse = torch.empty((B, H), device=d)
    ws = pkg.alloc_workspace(1 << 20, d)
    with pytest.raises(ValueError, match="^workspace"):
        pkg.mla_absorb_decode_fp8_batch_combine(sl, H, MB, out, lse, host_ws)
    with pytest.raises(ValueError, match="^out"):
        pkg.mla_absorb_decode_fp8_batch_combine(sl, H + 1, MB, out, lse, ws)
    with pytest.raises(ValueError, match="^lse"):
        pkg.mla_absorb_decode_fp8_batch_combine(sl, H, MB, out, lse[:1], ws)
    with pytest.raises(TypeError, match="^seq_lens"):
        pkg.mla_absorb_decode_fp8_batch_combine(sl.long(), H, MB, out, lse, ws)
    with pytest.raises(ValueError, match="^workspace"):
        pkg.kv8_workspace_error(host_ws)
