"""Pins of the oracle's non-absorbed prefill projection (CPU only).

KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
description: the projection path dequantizes the cached Lc rows (LUT value times
the row scale) before the kv_b up-projection.  Pinned against a selection
matrix (it must return the dequantized channels), a brute-force triple loop, the
per-row scale and the slot map, so a dropped scale, a transposed weight or an
ignored slot map fails.
"""
import numpy as np

import oracle
from test_oracle_wuv import f32_to_bf16_bits


def cache(rng, n):
    rows = rng.standard_normal((n, 576)).astype(np.float32) * np.exp(rng.standard_normal((n, 1)))
    return oracle.quantize_rows(rows)


def test_selection_matrix_returns_the_dequantized_channels():
    rng = np.random.default_rng(0)
    codes, scales = cache(rng, 20)
    w = np.zeros((512, 6), np.float32)
    chans = [0, 5, 77, 256, 300, 511]
    for j, c in enumerate(chans):
        w[c, j] = 1.0
    y = oracle.prefill_project(codes, scales, f32_to_bf16_bits(w))
    lut = oracle.decode_table().astype(np.float64)
    for t in range(20):
        for j, c in enumerate(chans):
            assert y[t, j] == lut[codes[t, c]] * np.float64(scales[t, 0])


def test_brute_force_and_slot_map():
    rng = np.random.default_rng(1)
    codes, scales = cache(rng, 12)
    wb = f32_to_bf16_bits(rng.standard_normal((512, 3)))
    w = oracle.bf16_to_f32(wb).astype(np.float64)
    slots = np.array([11, 0, 5, 5, 2])
    y = oracle.prefill_project(codes, scales, wb, slots=slots)
    lut = oracle.decode_table().astype(np.float64)
    for t, sl in enumerate(slots):
        for n in range(3):
            ref = sum(lut[codes[sl, d]] * w[d, n] for d in range(512)) * float(scales[sl, 0])
            assert abs(y[t, n] - ref) <= 1e-12 * max(1.0, abs(ref))
    assert np.array_equal(y[2], y[3])    # same slot, same row


def test_rope_part_and_scale_of_rc_are_not_used():
    rng = np.random.default_rng(2)
    codes, scales = cache(rng, 4)
    wb = f32_to_bf16_bits(rng.standard_normal((512, 2)))
    y = oracle.prefill_project(codes, scales, wb)
    c2, s2 = codes.copy(), scales.copy()
    c2[:, 512:] = 0x33
    s2[:, 1] = 7.0
    assert np.array_equal(oracle.prefill_project(c2, s2, wb), y)
