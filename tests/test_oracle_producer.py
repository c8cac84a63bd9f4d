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


def np_rmsnorm_f32(x, w, eps, ss):
    """The f32 steps after the sum of squares, each rounded once (numpy float32
    scalars are IEEE single operations): ms = ss/512, inv = 1/sqrt(ms + eps),
    y = (x * inv) * w."""
    f = np.float32
    inv = f(1.0) / np.sqrt(f(f(ss) * f(1.0 / 512.0)) + f(eps))
    return ((x.astype(np.float32) * inv).astype(np.float32) * w).astype(np.float32)


def exact_ss(x):
    """f32 of the exactly rounded (math.fsum) double sum of the squares."""
    return np.float32(math.fsum(float(v) * float(v) for v in np.asarray(x, np.float64)))


def butterfly_ss(x):
    """The sum of squares in another f32 order (32 partial sums of 16, then a
    pairwise tree), which is not the oracle's definition."""
    sq = (x.astype(np.float32) ** 2).astype(np.float32).reshape(32, 16)
    p = np.zeros(32, np.float32)
    for k in range(16):
        p = (p + sq[:, k]).astype(np.float32)
    idx = np.arange(32)
    for o in (16, 8, 4, 2, 1):
        p = (p + p[idx ^ o]).astype(np.float32)
    return p[0]


def test_rmsnorm_sum_of_squares_is_the_exact_sum_rounded_once():
    """On rows where a reordered f32 sum of squares gives a different f32 total,
    the oracle still gives the f32 of the exact sum: its output equals the f32
    pipeline run from f32(fsum(x^2)) bit for bit, and not the one run from the
    reordered sum."""
    rng = np.random.default_rng(21)
    w = np.ones(512, np.float32)
    discriminating = 0
    for r in range(400):
        x = (rng.standard_normal(512) * np.exp(rng.uniform(-3, 3))).astype(np.float32)
        y = oracle.rmsnorm_row(x, w, EPS)
        ss = exact_ss(x)
        assert np.array_equal(y.view(np.uint32), np_rmsnorm_f32(x, w, EPS, ss).view(np.uint32)), r
        other = np_rmsnorm_f32(x, w, EPS, butterfly_ss(x))
        discriminating += not np.array_equal(y.view(np.uint32), other.view(np.uint32))
    # the pin discriminates: on these rows an f32 sum in another order gives other bits
    assert discriminating >= 20


def test_rmsnorm_sum_of_squares_hand_worked():
    """1 + 2^-24 * 511 (exactly): index-order f32 accumulation loses every 2^-24
    (1 + 2^-24 rounds back to 1), the exact sum is 1 + 511 * 2^-24, which rounds
    to 1 + 2^-23 * 256 = 1.0000305 in f32 (halfway cases are absent)."""
    x = np.zeros(512, np.float32)
    x[0] = 1.0
    x[1:] = np.float32(2.0 ** -12)          # squares: 2^-24 each
    ss = exact_ss(x)
    assert ss == np.float32(1.0 + 511 * 2.0 ** -24)
    seq = np.float32(0)
    for v in x:
        seq = np.float32(seq + np.float32(v * v))
    assert seq == np.float32(1.0) != ss      # naive f32 order differs from the definition
    y = oracle.rmsnorm_row(x, np.ones(512, np.float32), 0.0)
    assert np.array_equal(y.view(np.uint32), np_rmsnorm_f32(x, np.ones(512, np.float32), 0.0,
                                                             ss).view(np.uint32))


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
