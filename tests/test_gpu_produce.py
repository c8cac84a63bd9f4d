"""GPU fused-producer parity against the oracle.

Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description, attention_rows item (the producer quantizes the fresh
normed/roped row).  Every f32 operation on both sides is rounded once, in the
same order, except the sum of squares of the RMS norm: the oracle takes the
plain sum (exact squares added in double, rounded to f32 once), the kernel its
warp's reduction (32 partial sums of 16 in index order, then an xor butterfly
16, 8, 4, 2, 1, all in f32).  So:
- on every row where the kernel's f32 sum of squares (restated here in numpy,
  only to sort the rows) equals the oracle's, codes and scales must match bit
  for bit -- the special rows (NaN entries, zero rows, subnormal and
  overflowing sums of squares) included;
- on the other rows the two sums differ by a relative d (a few ulps of f32).  The
  inverse RMS, every normed value and so the row's amax and scale move by d / 2,
  and each of the six rounded steps after the sum (adding eps, the square root,
  the reciprocal, the two products, the division of the amax by 448) may round
  the two sides one ulp apart: each Lc scale must agree within 6 + d / 2 ulps
  (an ulp of the scale is at least 2^-24 of it), the Rc scale (no norm) bit for
  bit, and every code, which does not move with a common factor on the row,
  within one e4m3 step.
The tests print how many rows fell in each class.
"""
import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
import oracle
from fp8_mla_latent_gb300 import workloads

pytestmark = pytest.mark.gpu
D = 576


def run(p, rows=None, positions=None, stride=D, slots="map", eps=None):
    d = torch.device("cuda:0")
    rows = p.rows if rows is None else rows
    positions = p.positions if positions is None else positions
    n = rows.shape[0]
    buf = torch.zeros((n, stride), dtype=torch.float32, device=d)
    buf[:, :D] = torch.from_numpy(rows).to(d)
    n_slots = p.n_slots if slots == "map" else n
    codes = torch.full((n_slots, D), 0xAB, dtype=torch.uint8, device=d)
    scales = torch.full((n_slots, 2), -1.0, dtype=torch.float32, device=d)
    st = torch.from_numpy(p.slots[:n]).to(d) if slots == "map" else None
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkg.kv8_produce_rows(buf, torch.from_numpy(p.weight).to(d), p.eps if eps is None else eps,
                         torch.from_numpy(np.asarray(positions, np.int64)).to(d),
                         torch.from_numpy(p.rope_cos).to(d), torch.from_numpy(p.rope_sin).to(d),
                         codes, scales, dst_slot=st, err_word=err)
    torch.cuda.synchronize()
    # the oracle writes into the same sentinel-filled pool
    rc = np.full((n_slots, D), 0xAB, np.uint8)
    rs = np.full((n_slots, 2), -1.0, np.float32)
    oracle.produce_rows(rows, p.weight, p.eps if eps is None else eps, positions, p.rope_cos,
                        p.rope_sin, dst_slot=p.slots[:n] if slots == "map" else None,
                        n_slots=n_slots, codes=rc, scales=rs)
    return codes.cpu().numpy(), scales.cpu().numpy(), rc, rs, int(err.item())


def kernel_order_ss(rows):
    """The kernel's documented f32 order for the sum of squares of Lc."""
    sq = (rows[:, :512].astype(np.float32) ** 2).astype(np.float32).reshape(-1, 32, 16)
    p = np.zeros(sq.shape[:2], np.float32)
    for k in range(16):
        p = (p + sq[:, :, k]).astype(np.float32)
    idx = np.arange(32)
    for o in (16, 8, 4, 2, 1):
        p = (p + p[:, idx ^ o]).astype(np.float32)
    return p[:, 0]


def oracle_ss(rows):
    """The oracle's definition: exact squares added in index order in double."""
    x = rows[:, :512].astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return np.cumsum(x * x, axis=1)[:, -1].astype(np.float32)


def code_rank(c):
    """Position of an e4m3 code on the number line (adjacent codes differ by 1)."""
    k = (c & 0x7F).astype(np.int32)
    return np.where(c & 0x80, -k, k)


def assert_parity(c, s, rc, rs, rows, slots):
    """Bit-exact on the rows whose sums of squares agree; on the others the Lc scale
    within 6 + d / 2 ulps (d = the sums' relative difference), the Rc scale bit for
    bit and every code within one e4m3 step."""
    with np.errstate(invalid="ignore", over="ignore"):
        a, b = kernel_order_ss(rows), oracle_ss(rows)
    same = (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))
    exact = slots[same]
    bad = exact[(c[exact] != rc[exact]).any(1) |
                (s[exact].view(np.uint32) != rs[exact].view(np.uint32)).any(1)]
    assert bad.size == 0, f"{bad.size} rows with equal sums of squares differ, first slot {bad[0]}"
    near = slots[~same]
    if near.size:
        du = np.abs(s[near].view(np.int32).astype(np.int64) - rs[near].view(np.int32).astype(np.int64))
        with np.errstate(invalid="ignore", divide="ignore"):
            d = np.abs(a[~same].astype(np.float64) - b[~same]) / np.abs(b[~same].astype(np.float64))
        bound = 6 + np.ceil(d * 2.0 ** 23)  # 6 + (d / 2) / 2^-24 ulps, for the Lc scale
        over = du[:, 0] > bound
        assert not over.any(), (f"Lc scale differs by {du[over, 0].max()} ulp where the bound is "
                                f"{bound[over].min():.0f}")
        assert du[:, 1].max() <= 0, f"Rc scale differs by {du[:, 1].max()} ulp"
        dc = np.abs(code_rank(c[near]) - code_rank(rc[near]))
        assert dc.max() <= 1, f"code differs by {dc.max()} steps"
    n_bits = int(((c[near] == rc[near]).all(1) &
                  (s[near].view(np.uint32) == rs[near].view(np.uint32)).all(1)).sum()) if near.size else 0
    print(f"producer rows: {exact.size} with equal sums of squares (bit-exact), {near.size} with "
          f"different sums ({n_bits} of them bit-exact anyway)")


def test_append_value_mix_bit_exact():
    p = workloads.producer_inputs(65536)
    c, s, rc, rs, err = run(p)
    assert err == 0
    assert_parity(c, s, rc, rs, p.rows, p.slots)


@pytest.mark.parametrize("stride,slots", [(D, None), (600, "map"), (1024, None)])
def test_strides_and_identity_slots(stride, slots):
    p = workloads.producer_inputs(3000, seed=11)
    c, s, rc, rs, _ = run(p, stride=stride, slots=slots)
    assert_parity(c, s, rc, rs, p.rows, p.slots if slots == "map" else np.arange(p.rows.shape[0]))


def test_positions_outside_the_table_are_skipped_and_flagged():
    p = workloads.producer_inputs(500, max_pos=64, seed=12)
    pos = p.positions.copy()
    pos[[3, 17, 499]] = [-1, 64, 1 << 40]
    c, s, rc, rs, err = run(p, positions=pos)
    assert err & 1
    for r in (3, 17, 499):
        assert np.all(c[p.slots[r]] == 0xAB) and np.all(s[p.slots[r]] == -1.0)
    keep = np.setdiff1d(np.arange(500), [3, 17, 499])
    assert_parity(c, s, rc, rs, p.rows[keep], p.slots[keep])


def test_special_rows_bit_exact():
    p = workloads.producer_inputs(64, seed=13)
    rows = np.random.default_rng(1).standard_normal((64, D)).astype(np.float32)
    rows[0] = 0.0                                   # zero row: y = 0
    rows[1, 5] = np.nan                             # NaN in Lc: the whole normed Lc is NaN
    rows[2, 520] = np.nan                           # NaN in Rc: one pair
    rows[3, :512] = 1e30                            # sum of squares overflows: inv = 0
    rows[4, :512] = 1e-30                           # sum of squares underflows: eps dominates
    rows[5, :512] = np.float32(1e-45)               # subnormal entries
    rows[6, 512:] = 3e38                            # rotation overflows to inf
    rows[7, :] = -0.0                               # negative zeros
    rows[8, :512] = np.inf                          # infinities (unsupported, must not fault)
    for eps in (1e-6, 0.0):
        c, s, rc, rs, _ = run(p, rows=rows, eps=eps)
        assert_parity(c, s, rc, rs, rows, p.slots[:64])


def test_empty_call():
    d = torch.device("cuda:0")
    p = workloads.producer_inputs(4)
    pkg.kv8_produce_rows(torch.zeros((0, D), device=d), torch.from_numpy(p.weight).to(d), 1e-6,
                         torch.zeros(0, dtype=torch.int64, device=d),
                         torch.from_numpy(p.rope_cos).to(d), torch.from_numpy(p.rope_sin).to(d),
                         torch.zeros((4, D), dtype=torch.uint8, device=d),
                         torch.zeros((4, 2), device=d))
    torch.cuda.synchronize()
