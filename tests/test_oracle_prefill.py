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


def test_rope_keys_round_trip_within_half_an_e4m3_step():
    """Quantize then dequantize: every rope channel comes back within half a step of
    the e4m3 grid scaled by the row's Rc scale (3 mantissa bits: relative 2^-4 for
    normals, 2^-10 * sRc below the normal range).  Lc is 1000x larger than Rc in these
    rows, so using the Lc scale, or the Lc columns, fails the bound."""
    rng = np.random.default_rng(7)
    n = 40
    rows = rng.standard_normal((n, 576)).astype(np.float32)
    rows[:, :512] *= 1000.0
    rows[3, 512:] = 0.0            # all-zero rope segment
    codes, scales = oracle.quantize_rows(rows)
    k = oracle.prefill_rope(codes, scales)
    assert k.dtype == np.float32 and k.shape == (n, 64)
    x = rows[:, 512:].astype(np.float64)
    sR = scales[:, 1].astype(np.float64)[:, None]
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sR * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(k - x) <= bound)
    assert np.all(k[3] == 0)
    # the channel holding the amax decodes to 448 * sRc (code 0x7E, or 0xFE)
    j = np.argmax(np.abs(x), axis=1)
    for t in range(n):
        if t == 3:
            continue
        assert abs(k[t, j[t]]) == np.float32(448.0 * np.float64(scales[t, 1]))


def test_rope_keys_follow_the_slot_map():
    rng = np.random.default_rng(8)
    codes, scales = cache(rng, 10)
    slots = np.array([9, 2, 2, 0])
    k = oracle.prefill_rope(codes, scales, slots)
    full = oracle.prefill_rope(codes, scales)
    assert np.array_equal(k, full[slots])
    assert not np.array_equal(full[9], full[2])
