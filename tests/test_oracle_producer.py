"""Pins of the oracle's fused producer (CPU only).

Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description, attention_rows item: the producer quantizes the fresh
normed/roped row.  The page names the steps only; the readings (RMS norm with a
weight over Lc, rotation of the Rc pairs (2j, 2j+1) by tabulated angles) are
pinned here against closed forms, float64 restatements and invariants, so that a
dropped mean, an eps outside the root, a wrong rotation sign or swapped pair
order fails.
"""
import math

import numpy as np
import pytest

import oracle

EPS = 1e-6


def f64_rmsnorm(x, w, eps):
    x = np.asarray(x, np.float64)
    return x / math.sqrt(np.mean(x * x) + eps) * np.asarray(w, np.float64)


def test_rmsnorm_closed_form_three_four():
    x = np.zeros(512, np.float32)
    x[0], x[1] = 3.0, 4.0
    w = np.ones(512, np.float32)
    y = oracle.rmsnorm_row(x, w, EPS)
    inv = 1.0 / math.sqrt(25.0 / 512.0 + EPS)
    assert y[0] == pytest.approx(3.0 * inv, rel=3e-7)
    assert y[1] == pytest.approx(4.0 * inv, rel=3e-7)
    assert np.all(y[2:] == 0.0)


def test_rmsnorm_uses_the_mean_and_eps_inside_the_root():
    w = np.ones(512, np.float32)
    ones = np.ones(512, np.float32)
    y = oracle.rmsnorm_row(ones, w, EPS)          # a sum instead of a mean would give 1/sqrt(512)
    assert np.allclose(y, 1.0 / math.sqrt(1.0 + EPS), rtol=2e-7)
    tiny = np.full(512, 1e-4, np.float32)         # ms = 1e-8 << eps: eps must sit inside the root
    y = oracle.rmsnorm_row(tiny, w, EPS)
    assert np.allclose(y, 1e-4 / math.sqrt(1e-8 + EPS), rtol=1e-6)


def test_rmsnorm_against_float64_and_unit_mean_square():
    rng = np.random.default_rng(3)
    for scale in (1e-3, 1.0, 37.0):
        x = (rng.standard_normal(512) * scale).astype(np.float32)
        w = (1.0 + 0.5 * rng.standard_normal(512)).astype(np.float32)
        y = oracle.rmsnorm_row(x, w, EPS)
        ref = f64_rmsnorm(x, w, EPS)
        assert np.max(np.abs(y - ref) / np.maximum(np.abs(ref), 1e-30)) < 4e-7
        y1 = oracle.rmsnorm_row(x, np.ones(512, np.float32), EPS)
        ms = np.mean(x.astype(np.float64) ** 2)
        assert np.mean(y1.astype(np.float64) ** 2) == pytest.approx(ms / (ms + EPS), rel=2e-6)


def test_rmsnorm_weight_is_a_per_channel_factor_bit_exact():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(512).astype(np.float32)
    w = rng.standard_normal(512).astype(np.float32)
    y1 = oracle.rmsnorm_row(x, np.ones(512, np.float32), EPS)
    yw = oracle.rmsnorm_row(x, w, EPS)
    assert np.array_equal(yw, (y1 * w).astype(np.float32))


def test_rmsnorm_zero_row_is_zero():
    y = oracle.rmsnorm_row(np.zeros(512, np.float32), np.ones(512, np.float32), EPS)
    assert np.all(y == 0.0)


def test_rope_identity_and_quarter_turn_exact():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(64).astype(np.float32)
    ident = oracle.rope_pairs(x, np.ones(32, np.float32), np.zeros(32, np.float32))
    assert np.array_equal(ident, x)
    quarter = oracle.rope_pairs(x, np.zeros(32, np.float32), np.ones(32, np.float32))
    # (x0, x1) -> (-x1, x0): the pair order and the sign of the sine term
    assert np.array_equal(quarter[0::2], -x[1::2])
    assert np.array_equal(quarter[1::2], x[0::2])


def test_rope_matches_float64_rotation_and_keeps_pair_norms():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(64).astype(np.float32)
    ang = rng.uniform(-math.pi, math.pi, 32)
    c, s = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    y = oracle.rope_pairs(x, c, s).astype(np.float64)
    x0, x1 = x[0::2].astype(np.float64), x[1::2].astype(np.float64)
    c64, s64 = c.astype(np.float64), s.astype(np.float64)
    assert np.allclose(y[0::2], x0 * c64 - x1 * s64, atol=1e-6)
    assert np.allclose(y[1::2], x0 * s64 + x1 * c64, atol=1e-6)
    assert np.allclose(y[0::2] ** 2 + y[1::2] ** 2, x0 ** 2 + x1 ** 2, rtol=2e-6)


def test_rope_composes_angles():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(64).astype(np.float32)
    a, b = rng.uniform(-1, 1, 32), rng.uniform(-1, 1, 32)
    tab = lambda t: (np.cos(t).astype(np.float32), np.sin(t).astype(np.float32))
    two = oracle.rope_pairs(oracle.rope_pairs(x, *tab(a)), *tab(b))
    one = oracle.rope_pairs(x, *tab(a + b))
    assert np.allclose(two, one, atol=2e-6)


def test_produce_is_norm_rope_then_quantize_into_slots():
    rng = np.random.default_rng(8)
    n, max_pos = 40, 100
    src = np.zeros((n, 600), np.float32)
    src[:, :576] = rng.standard_normal((n, 576)) * 3
    w = (1 + 0.1 * rng.standard_normal(512)).astype(np.float32)
    ang = np.outer(np.arange(max_pos), 10000.0 ** (-np.arange(32) / 32.0))
    cos, sin = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    pos = rng.integers(0, max_pos, n)
    pos[3] = -1          # out of range: skipped
    pos[7] = max_pos     # out of range: skipped
    slots = rng.permutation(64)[:n]
    codes, scales = oracle.produce_rows(src, w, EPS, pos, cos, sin, dst_slot=slots, n_slots=64)
    for r in range(n):
        s = slots[r]
        if r in (3, 7):
            assert np.all(codes[s] == 0) and np.all(scales[s] == 0)
            continue
        y = np.concatenate([oracle.rmsnorm_row(src[r, :512], w, EPS),
                            oracle.rope_pairs(src[r, 512:576], cos[pos[r]], sin[pos[r]])])
        c1, s1 = oracle.quantize_rows(y[None, :])
        assert np.array_equal(codes[s], c1[0]) and np.array_equal(scales[s], s1[0])
