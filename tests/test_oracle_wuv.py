"""Pins of the oracle's W_UV epilogue (CPU only).

The absorbed attention of the KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU +
CUDA) with .coli_kv v2", PR description: the latent is key and value at once in
the absorbed attention) leaves the context in latent space; the per-head
projection W_UV maps it to the value heads.  Pinned against the bf16 format's
definition, a selection matrix, a brute-force triple loop and linearity, so a
transposed weight or a swapped head index fails.
"""
import numpy as np

import oracle


def f32_to_bf16_bits(x):
    """Round-to-nearest-even f32 -> bf16 bits (for building exact test weights)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def test_bf16_decoding_is_exact():
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4049, 0x7F80, 0x0001], np.uint16)
    f = oracle.bf16_to_f32(bits)
    assert f[0] == 0 and np.signbit(f[1]) and f[2] == 1.0 and f[3] == -1.0
    assert f[4] == np.float32(3.140625) and np.isinf(f[5]) and f[6] == np.float32(2.0 ** -133)


def test_selection_matrix_picks_channels_per_head():
    rng = np.random.default_rng(0)
    B, H, V = 3, 4, 8
    o = rng.standard_normal((B, H, 512)).astype(np.float32)
    w = np.zeros((H, 512, V), np.float32)
    for h in range(H):
        for v in range(V):
            w[h, 7 * v + h, v] = 1.0        # head-dependent channel choice
    y = oracle.wuv_project(o, f32_to_bf16_bits(w))
    for h in range(H):
        assert np.array_equal(y[:, h, :], o[:, h, [7 * v + h for v in range(V)]].astype(np.float64))


def test_brute_force_and_linearity():
    rng = np.random.default_rng(1)
    B, H, V = 2, 3, 5
    o = rng.standard_normal((B, H, 512)).astype(np.float32)
    wb = f32_to_bf16_bits(rng.standard_normal((H, 512, V)))
    w = oracle.bf16_to_f32(wb).astype(np.float64)
    y = oracle.wuv_project(o, wb)
    for b in range(B):
        for h in range(H):
            for v in range(V):
                ref = sum(float(o[b, h, d]) * w[h, d, v] for d in range(512))
                assert abs(y[b, h, v] - ref) <= 1e-12 * max(1.0, abs(ref))
    y2 = oracle.wuv_project(2.0 * o, wb)
    assert np.allclose(y2, 2.0 * y, rtol=0, atol=1e-12)
