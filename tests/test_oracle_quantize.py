"""Pins for the oracle's per-row quantizer (CPU only).

Rules: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description and expanded summary: Lc and Rc each get an f32 scale
amax/448; c/kv_fp8.h item: rows whose amax is subnormal (448/amax would overflow
to +inf) are guarded.  Checked against numpy's
f32 division, torch's e4m3fn cast, the format's spacing bound and invariants.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DL, DR, D = 512, 64, 576
SEGS = ((0, 0, DL), (1, DL, D))


def rows(n, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return rng.standard_normal((n, D)).astype(np.float32)
    if kind == "t3":
        return rng.standard_t(3, size=(n, D)).astype(np.float32)
    raise ValueError(kind)


def torch_e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_scale_is_f32_amax_over_448_per_segment():
    x = rows(64, 1, "t3")
    x[3, 7] = np.nan
    codes, scales = oracle.quantize_rows(x)
    for seg, a, b in SEGS:
        amax = np.nanmax(np.abs(x[:, a:b]), axis=1).astype(np.float32)
        assert np.array_equal(scales[:, seg], amax / np.float32(448.0))


def test_codes_match_torch_cast_of_the_f32_product():
    x = rows(128, 2, "t3")
    x[5, 100] = np.nan
    x[6, 520] = -0.0
    codes, _ = oracle.quantize_rows(x)
    for seg, a, b in SEGS:
        amax = np.nanmax(np.abs(x[:, a:b]), axis=1).astype(np.float32)
        inv = np.float32(448.0) / amax
        prod = x[:, a:b] * inv[:, None]  # numpy f32 multiply: one rounding
        want = torch_e4m3(prod)
        ok = ~np.isnan(prod)
        assert np.array_equal(codes[:, a:b][ok], want[ok])
        assert np.all(codes[:, a:b][~ok] == 0x00)


def test_amax_element_encodes_to_plus_minus_448():
    x = rows(50, 3)
    codes, _ = oracle.quantize_rows(x)
    for _, a, b in SEGS:
        seg = x[:, a:b]
        idx = np.argmax(np.abs(seg), axis=1)
        v = seg[np.arange(len(seg)), idx]
        c = codes[:, a:b][np.arange(len(seg)), idx]
        assert np.all(np.where(v > 0, c == 0x7E, c == 0xFE))


def test_error_bound_half_spacing():
    x = rows(200, 4, "t3")
    codes, scales = oracle.quantize_rows(x)
    lut = oracle.decode_table().astype(np.float64)
    for seg, a, b in SEGS:
        amax = np.abs(x[:, a:b]).max(1, keepdims=True).astype(np.float64)
        y = np.abs(x[:, a:b].astype(np.float64)) * 448.0 / amax  # exact scaled magnitude
        # e4m3 spacing at magnitude y: 2^(floor(log2 y) - 3) for y >= 2^-6, else 2^-9
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
        spacing = 2.0 ** (e - 3)
        err = np.abs(y - np.abs(lut[codes[:, a:b]]))
        # half a spacing, plus the two f32 roundings (inv = 448/amax and x*inv)
        assert np.all(err <= spacing / 2 + y * 2.0 ** -22)
        # and the decoded row reproduces x within s * (half spacing + slack)
        s = scales[:, seg].astype(np.float64)[:, None]
        back = s * lut[codes[:, a:b]]
        assert np.all(np.abs(back - x[:, a:b]) <= s * (spacing / 2 + y * 2.0 ** -21) + 1e-30)


def test_all_zero_row_keeps_signs_and_scale_zero():
    x = np.zeros((2, D), np.float32)
    x[1, ::2] = -0.0
    codes, scales = oracle.quantize_rows(x)
    assert np.all(scales == 0.0)
    assert np.all(codes[0] == 0x00)
    assert np.all(codes[1, ::2] == 0x80) and np.all(codes[1, 1::2] == 0x00)


def test_subnormal_amax_guard():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((4, D)).astype(np.float32)
    x[0] *= np.float32(2.0 ** -140)  # amax deep in the f32 subnormal range
    x[1, :DL] = np.float32(1e-38) * np.sign(x[1, :DL])  # Lc normal but below 448/FLT_MAX
    codes, scales = oracle.quantize_rows(x)
    for r, a, b in ((0, 0, DL), (0, DL, D), (1, 0, DL)):
        seg = x[r, a:b]
        assert np.all(codes[r, a:b] == np.where(np.signbit(seg), 0x80, 0x00))
    amax0 = np.abs(x[0, :DL]).max()
    assert scales[0, 0] == amax0 / np.float32(448.0) and scales[0, 0] > 0
    # Rc of row 1 is ordinary and unaffected by the Lc guard
    assert np.any(codes[1, DL:] & 0x7F) and scales[1, 1] > 1e-3


def test_guard_threshold_is_where_448_over_amax_overflows():
    fmax = np.finfo(np.float32).max
    thr = np.float32(448.0) / np.float32(fmax)
    for amax, fires in ((thr, False), (np.nextafter(thr, np.float32(0)) * np.float32(0.5), True)):
        x = np.zeros((1, D), np.float32)
        x[0, 0] = amax
        x[0, 1] = -amax
        codes, _ = oracle.quantize_rows(x)
        with np.errstate(over="ignore"):
            inv = np.float32(448.0) / np.float32(amax)
        assert np.isfinite(inv) != fires
        if fires:
            assert codes[0, 0] == 0x00 and codes[0, 1] == 0x80
        else:
            assert codes[0, 0] == 0x7E and codes[0, 1] == 0xFE


def test_nan_entries_are_inert_zero_and_ignored_by_amax():
    x = rows(3, 7)
    y = x.copy()
    y[0, 10] = np.nan
    y[1, 530] = np.nan
    y[2, :DL] = np.nan
    cx, sx = oracle.quantize_rows(x)
    cy, sy = oracle.quantize_rows(y)
    assert cy[0, 10] == 0 and cy[1, 530] == 0 and np.all(cy[2, :DL] == 0) and sy[2, 0] == 0
    # rows whose amax is not the NaN position keep every other code
    for r, col in ((0, 10), (1, 530)):
        a, b = (0, DL) if col < DL else (DL, D)
        if np.nanmax(np.abs(y[r, a:b])) == np.abs(x[r, a:b]).max():
            m = np.ones(D, bool)
            m[col] = False
            assert np.array_equal(cy[r, m], cx[r, m])


def test_power_of_two_scaling_invariance():
    x = rows(40, 8)
    c0, s0 = oracle.quantize_rows(x)
    for k in (-20, -3, 5, 30):
        c1, s1 = oracle.quantize_rows(x * np.float32(2.0 ** k))
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1, s0 * np.float32(2.0 ** k))


def test_segments_are_independent():
    x = rows(10, 9)
    y = x.copy()
    y[:, DL:] *= 1000.0
    cx, sx = oracle.quantize_rows(x)
    cy, sy = oracle.quantize_rows(y)
    assert np.array_equal(cx[:, :DL], cy[:, :DL]) and np.array_equal(sx[:, 0], sy[:, 0])
    assert not np.array_equal(sx[:, 1], sy[:, 1])


def test_slot_scatter_and_row_stride():
    x = rows(6, 10)
    padded = np.zeros((6, 600), np.float32)
    padded[:, :D] = x
    slots = np.array([9, 2, 7, 0, 4, 11])
    codes = np.full((12, D), 0xAB, np.uint8)
    scales = np.full((12, 2), -1.0, np.float32)
    oracle.quantize_rows(padded, dst_slot=slots, codes=codes, scales=scales)
    cref, sref = oracle.quantize_rows(x)
    assert np.array_equal(codes[slots], cref) and np.array_equal(scales[slots], sref)
    untouched = np.setdiff1d(np.arange(12), slots)
    assert np.all(codes[untouched] == 0xAB) and np.all(scales[untouched] == -1.0)


def test_page_format_numbers():
    """The page's printed memory figures fix the row format: 576 e4m3 bytes plus
    two f32 scales per token per layer (tests/golden/kv8_page_numbers.txt)."""
    vals = {}
    with open(os.path.join(GOLDEN, "kv8_page_numbers.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()[:2]
                vals[k] = float(v)
    f32_row = D * 4
    fp8_row = D * 1 + 2 * 4
    assert round(f32_row / fp8_row, 1) == vals["kv_ram_ratio"]
    assert round(f32_row / (D + 4), 1) != vals["kv_ram_ratio"]  # one scale per row would not fit
    layers = round(vals["slot_f32_gb"] * 1e9 / (262144 * f32_row))
    assert round(layers * f32_row / 1000) == vals["disk_kb_per_tok_v1"]
    assert round(layers * fp8_row / 1000) == vals["disk_kb_per_tok_v2"]


@pytest.mark.parametrize("n", [0, 1, 33])
def test_row_counts(n):
    x = rows(max(n, 1), 12)[:n]
    codes, scales = oracle.quantize_rows(x, n_slots=n)
    assert codes.shape == (n, D) and scales.shape == (n, 2)
