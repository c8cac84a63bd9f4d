"""Pins for the oracle's absorbed MLA decode attention (CPU only).

Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description: the latent is key and value at once in the absorbed
attention; attention_rows item: the score and context loops decode the codes as
they go, the row scale applied outside each dot product; Validation paragraph:
the fp8 path is checked against a reference on the host over dequantized rows.  The oracle is pinned to
torch's scaled-dot-product attention over explicitly dequantized rows (a
library routine), closed forms (T = 1, identical rows, q = 0), invariants
(permutation, split-T merge, paged layout) and its own f32/f64 agreement.
"""
import numpy as np
import pytest
import torch

import oracle

DL, DR, D = 512, 64, 576
SM = 1.0 / np.sqrt(192.0)


def make(T, H, seed, gain=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((max(T, 1), D)) * gain).astype(np.float32)[:T]
    codes, scales = oracle.quantize_rows(x, n_slots=T)
    ql = rng.standard_normal((H, DL)).astype(np.float32)
    qr = rng.standard_normal((H, DR)).astype(np.float32)
    return ql, qr, codes, scales


def dequant(codes, scales):
    lut = oracle.decode_table().astype(np.float64)
    v = lut[codes]
    v[:, :DL] *= scales[:, :1].astype(np.float64)
    v[:, DL:] *= scales[:, 1:].astype(np.float64)
    return v


@pytest.mark.parametrize("T,H,seed", [(1, 2, 0), (5, 2, 1), (8, 2, 2), (37, 3, 3)])
def test_equals_sdpa_over_dequantized_rows(T, H, seed):
    """Absorbed fp8 attention == standard softmax attention (torch SDPA, f64) with
    key = [sLc*dec(Lc), sRc*dec(Rc)] and value = sLc*dec(Lc)."""
    ql, qr, codes, scales = make(T, H, seed, gain=np.linspace(0.2, 3.0, D))
    scales[:, 1] *= 7.0  # make the two scales clearly different
    kv = dequant(codes, scales)
    q = torch.from_numpy(np.concatenate([ql, qr], 1).astype(np.float64))[None, :, None, :]
    k = torch.from_numpy(kv)[None, None].expand(1, H, T, D)
    v = torch.from_numpy(kv[:, :DL])[None, None].expand(1, H, T, DL)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=SM)[0, :, 0].numpy()
    z = (q[0, :, 0] @ torch.from_numpy(kv).T * SM)
    ref_lse = torch.logsumexp(z, dim=1).numpy()
    out, lse = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    out32, lse32 = oracle.attention_f32(ql, qr, codes, scales, T, SM)
    assert np.abs(out32 - ref).max() <= 1e-5 * np.abs(ref).max()
    np.testing.assert_allclose(lse32, ref_lse, rtol=1e-5, atol=1e-5)


def test_single_token_returns_its_value_row():
    ql, qr, codes, scales = make(1, 4, 5)
    out, lse = oracle.attention_f64(ql, qr, codes, scales, 1, SM)
    row = dequant(codes, scales)[0, :DL]
    assert np.array_equal(out, np.broadcast_to(row, out.shape))


def test_identical_rows_return_that_row():
    ql, qr, codes, scales = make(1, 3, 6)
    T = 50
    codes = np.repeat(codes, T, 0)
    scales = np.repeat(scales, T, 0)
    out, lse = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    row = dequant(codes[:1], scales[:1])[0, :DL]
    np.testing.assert_allclose(out, np.broadcast_to(row, out.shape), rtol=1e-13, atol=1e-13)


def test_zero_query_gives_mean_and_log_T():
    T = 123
    _, _, codes, scales = make(T, 1, 7)
    ql = np.zeros((2, DL), np.float32)
    qr = np.zeros((2, DR), np.float32)
    out, lse = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    mean = dequant(codes, scales)[:, :DL].mean(0)
    np.testing.assert_allclose(out[0], mean, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(T), rtol=1e-14)
    out32, lse32 = oracle.attention_f32(ql, qr, codes, scales, T, SM)
    np.testing.assert_allclose(out32[0], mean, rtol=1e-5, atol=1e-6)


def test_dominant_token_wins():
    ql, qr, codes, scales = make(20, 1, 8)
    # make token 13's score huge: its Lc equals sign(q_lat) at full scale
    codes[13, :DL] = np.where(ql[0] >= 0, 0x7E, 0xFE)
    scales[13, 0] = 1.0
    out, _ = oracle.attention_f64(ql, qr, codes, scales, 20, SM)
    np.testing.assert_allclose(out[0], dequant(codes, scales)[13, :DL], rtol=1e-9)


def test_rope_part_enters_the_score_with_its_own_scale():
    ql, qr, codes, scales = make(30, 2, 9)
    base, _ = oracle.attention_f64(ql, qr, codes, scales, 30, SM)
    s2 = scales.copy()
    s2[:, 1] *= 3.0
    changed, _ = oracle.attention_f64(ql, qr, codes, s2, 30, SM)
    assert np.abs(changed - base).max() > 1e-3
    qz = np.zeros_like(qr)
    a, _ = oracle.attention_f64(ql, qz, codes, scales, 30, SM)
    b, _ = oracle.attention_f64(ql, qz, codes, s2, 30, SM)
    np.testing.assert_array_equal(a, b)  # with q_rope = 0 the Rc scale cannot matter


def test_permutation_invariance():
    T = 64
    ql, qr, codes, scales = make(T, 2, 10)
    perm = np.random.default_rng(1).permutation(T)
    a, la = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    b, lb = oracle.attention_f64(ql, qr, codes[perm], scales[perm], T, SM)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=1e-13)


@pytest.mark.parametrize("cuts", [[100], [1, 2, 3], [37, 38, 200], [0, 150, 150, 299]])
def test_split_T_merge_equals_unsplit(cuts):
    T = 300
    ql, qr, codes, scales = make(T, 3, 11)
    edges = [0] + list(cuts) + [T]
    parts = [oracle.attention_partial_f64(ql, qr, codes, scales, a, b, SM)
             for a, b in zip(edges[:-1], edges[1:])]
    o = np.stack([p[0] for p in parts])
    m = np.stack([p[1] for p in parts])
    l = np.stack([p[2] for p in parts])
    out, lse = oracle.lse_merge_f64(o, m, l)
    ref, ref_lse = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)


def test_paged_layout_equals_contiguous():
    bs, nblk = 64, 5
    T = 4 * bs + 17
    ql, qr, codes, scales = make(T, 2, 12)
    rng = np.random.default_rng(2)
    phys = rng.permutation(nblk + 3)[:nblk]
    pool_c = np.zeros(((nblk + 3) * bs, D), np.uint8)
    pool_s = np.zeros(((nblk + 3) * bs, 2), np.float32)
    for j in range(nblk):
        n = min(bs, T - j * bs)
        if n > 0:
            pool_c[phys[j] * bs: phys[j] * bs + n] = codes[j * bs: j * bs + n]
            pool_s[phys[j] * bs: phys[j] * bs + n] = scales[j * bs: j * bs + n]
    bt = phys[None].astype(np.int32)
    slots = oracle.paged_slots(bt, 0, T, bs)
    a, la = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    b, lb = oracle.attention_f64(ql, qr, pool_c, pool_s, T, SM, slots=slots)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)
    ob, lseb = oracle.attention_batch_f32(ql[None], qr[None], pool_c, pool_s, bt,
                                          np.array([T], np.int32), SM)
    o32, l32 = oracle.attention_f32(ql, qr, codes, scales, T, SM)
    np.testing.assert_array_equal(ob[0], o32)
    np.testing.assert_array_equal(lseb[0], l32)


def test_batched_paged_oracle_per_sequence():
    """Several sequences of different lengths, their pages scattered through one
    pool: every sequence's output (batch index b > 0 included) equals the plain
    f32 attention over that sequence's own contiguous rows, and a sequence of
    length 0 gives out = 0, lse = -inf."""
    bs = 64
    lens = [0, 1, 64, 130, 3 * bs + 5]
    H = 3
    rng = np.random.default_rng(21)
    nblk = [(t + bs - 1) // bs for t in lens]
    maxb = max(nblk)
    n_pool = sum(nblk) + 4
    perm = rng.permutation(n_pool)
    pool_c = np.zeros((n_pool * bs, D), np.uint8)
    pool_s = np.zeros((n_pool * bs, 2), np.float32)
    bt = np.full((len(lens), maxb), -1, np.int32)
    qls, qrs, seqs = [], [], []
    used = 0
    for b, T in enumerate(lens):
        ql, qr, codes, scales = make(T, H, 30 + b)
        qls.append(ql)
        qrs.append(qr)
        seqs.append((codes, scales))
        for j in range(nblk[b]):
            phys = int(perm[used])
            used += 1
            bt[b, j] = phys
            n = min(bs, T - j * bs)
            pool_c[phys * bs: phys * bs + n] = codes[j * bs: j * bs + n]
            pool_s[phys * bs: phys * bs + n] = scales[j * bs: j * bs + n]
    bt[bt < 0] = 0  # entries past a sequence's pages are never read
    out, lse = oracle.attention_batch_f32(np.stack(qls), np.stack(qrs), pool_c, pool_s, bt,
                                          np.array(lens, np.int32), SM)
    for b, T in enumerate(lens):
        codes, scales = seqs[b]
        if T == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        o32, l32 = oracle.attention_f32(qls[b], qrs[b], codes, scales, T, SM)
        np.testing.assert_array_equal(out[b], o32)
        np.testing.assert_array_equal(lse[b], l32)


def test_empty_cache():
    ql, qr, codes, scales = make(0, 2, 13)
    out, lse = oracle.attention_f64(ql, qr, codes, scales, 0, SM)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out32, lse32 = oracle.attention_f32(ql, qr, codes, scales, 0, SM)
    assert np.all(out32 == 0) and np.all(np.isneginf(lse32))


def test_f32_and_f64_agree_on_a_larger_case():
    T, H = 2000, 4
    ql, qr, codes, scales = make(T, H, 14, gain=np.exp(0.5 * np.random.default_rng(3)
                                                      .standard_normal(D)))
    a, la = oracle.attention_f32(ql, qr, codes, scales, T, SM)
    b, lb = oracle.attention_f64(ql, qr, codes, scales, T, SM)
    assert np.abs(a - b).max() <= 1e-5 * np.abs(b).max()
    np.testing.assert_allclose(la, lb, rtol=1e-5)
