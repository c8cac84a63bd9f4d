"""GPU prefill projection parity against the float64 oracle.

KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
description: the projection path dequantizes the cached Lc rows before the kv_b
up-projection.  The tensor-core kernel uses bf16 operands (the e4m3 values are
exact in bf16, the row scale is applied in the f32 epilogue), f32 accumulation
and a bf16 result.  Rounding Y to bf16 costs at most 2^-9 |Y| ~ 1.95e-3 |Y| and the
f32 sums far less, so max-abs error <= 3e-3 * max|Y|.  Ragged token counts, slot
maps, several column widths and the full size (4096 tokens x 32768 columns,
sampled rows) are covered.
"""
import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
import oracle

pytestmark = pytest.mark.gpu


def make_cache(rng, n_slots):
    d = torch.device("cuda:0")
    rows = (rng.standard_normal((n_slots, 576)) * np.exp(0.5 * rng.standard_normal(576))).astype(np.float32)
    codes = torch.zeros((n_slots, 576), dtype=torch.uint8, device=d)
    scales = torch.zeros((n_slots, 2), dtype=torch.float32, device=d)
    pkg.kv8_quantize_rows(torch.from_numpy(rows).to(d), codes, scales)
    return codes, scales


def weights(rng, N):
    w = torch.from_numpy((rng.standard_normal((512, N)) / np.sqrt(512)).astype(np.float32))
    return w.to(torch.bfloat16)


def check(y, ref, rows=None):
    got = y.float().cpu().numpy()
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= 3e-3, err
    return err


@pytest.mark.parametrize("T,N,mapped", [(1, 256, False), (128, 256, False), (300, 512, True),
                                        (1000, 768, True), (2048, 4096, False)])
def test_prefill_matches_oracle(T, N, mapped):
    rng = np.random.default_rng(T + N)
    d = torch.device("cuda:0")
    n_slots = T + 64
    codes, scales = make_cache(rng, n_slots)
    w = weights(rng, N)
    slots = rng.permutation(n_slots)[:T].astype(np.int64) if mapped else None
    k_rope = torch.full((T, 64), float("nan"), dtype=torch.float32, device=d)
    y = pkg.kv8_prefill_project(codes, scales, w.to(d), T=T,
                                slots=None if slots is None else torch.from_numpy(slots).to(d),
                                k_rope=k_rope)
    torch.cuda.synchronize()
    idx = slots if mapped else np.arange(T)
    c_np, s_np = codes.cpu().numpy(), scales.cpu().numpy()
    ref = oracle.prefill_project(c_np, s_np, w.view(torch.int16).numpy().view(np.uint16), slots=idx)
    check(y, ref)
    # rope keys: one rounding of an exact product on both sides -> bit-exact
    kr = oracle.prefill_rope(c_np, s_np, idx)
    assert np.array_equal(k_rope.cpu().numpy().view(np.uint32), kr.view(np.uint32))


def test_prefill_full_size_sampled_rows():
    """4096 tokens (one sequence of the single-sequence workload) x 128 heads x (128 + 128)."""
    rng = np.random.default_rng(5)
    d = torch.device("cuda:0")
    T, N = 4096, 32768
    codes, scales = make_cache(rng, T)
    w = weights(rng, N)
    y = pkg.kv8_prefill_project(codes, scales, w.to(d))
    torch.cuda.synchronize()
    rows = np.sort(rng.choice(T, 48, replace=False))
    ref = oracle.prefill_project(codes.cpu().numpy(), scales.cpu().numpy(),
                                 w.view(torch.int16).numpy().view(np.uint16), slots=rows)
    check(y, ref, rows)
    assert torch.isfinite(y.float()).all()


def test_prefill_bad_slot_gives_zero_row_and_flag():
    rng = np.random.default_rng(6)
    d = torch.device("cuda:0")
    codes, scales = make_cache(rng, 200)
    w = weights(rng, 256).to(d)
    slots = torch.arange(130, dtype=torch.int64, device=d)
    slots[7] = 10 ** 6
    slots[129] = -3
    err = torch.zeros(1, dtype=torch.int32, device=d)
    k_rope = torch.full((130, 64), 1.0, dtype=torch.float32, device=d)
    y = pkg.kv8_prefill_project(codes, scales, w, slots=slots, k_rope=k_rope, err_word=err)
    torch.cuda.synchronize()
    assert err.item() & 1
    assert torch.all(y[7] == 0) and torch.all(y[129] == 0)
    assert torch.all(k_rope[7] == 0) and torch.all(k_rope[129] == 0)
    ref = oracle.prefill_project(codes.cpu().numpy(), scales.cpu().numpy(),
                                 w.cpu().view(torch.int16).numpy().view(np.uint16), slots=np.arange(7))
    check(y[:7], ref)


@pytest.mark.parametrize("T,N", [(129, 256), (257, 512), (383, 256), (640, 1024), (1100, 2560)])
def test_prefill_ragged_pair_tiles(T, N):
    """Token counts that end inside the first or the second 128-token half of a
    256-token pair tile (the second CTA of the pair then holds no token, or a few),
    through a random slot map, with the rope keys."""
    rng = np.random.default_rng(1000 + T)
    d = torch.device("cuda:0")
    n_slots = 2 * T
    codes, scales = make_cache(rng, n_slots)
    w = weights(rng, N)
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    k_rope = torch.empty((T, 64), dtype=torch.float32, device=d)
    y = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device=d)
    pkg.kv8_prefill_project(codes, scales, w.to(d), slots=torch.from_numpy(slots).to(d), y=y,
                            k_rope=k_rope)
    torch.cuda.synchronize()
    c_np, s_np = codes.cpu().numpy(), scales.cpu().numpy()
    ref = oracle.prefill_project(c_np, s_np, w.view(torch.int16).numpy().view(np.uint16), slots=slots)
    check(y, ref)
    kr = oracle.prefill_rope(c_np, s_np, slots)
    assert np.array_equal(k_rope.cpu().numpy().view(np.uint32), kr.view(np.uint32))


def test_prefill_calls_with_changing_shapes():
    """Back-to-back calls with different token counts and widths on one stream."""
    rng = np.random.default_rng(77)
    d = torch.device("cuda:0")
    codes, scales = make_cache(rng, 600)
    c_np, s_np = codes.cpu().numpy(), scales.cpu().numpy()
    outs = []
    for T, N in ((600, 256), (5, 768), (300, 512)):
        w = weights(rng, N)
        outs.append((T, w, pkg.kv8_prefill_project(codes, scales, w.to(d), T=T)))
    torch.cuda.synchronize()
    for T, w, y in outs:
        ref = oracle.prefill_project(c_np, s_np, w.view(torch.int16).numpy().view(np.uint16),
                                     slots=np.arange(T))
        check(y, ref)
