"""GPU fused-producer parity: bit-exact codes and scales against the oracle.

Method: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description, attention_rows item (the producer quantizes the fresh
normed/roped row).  Both sides round every f32 operation once in the same fixed
order, so every code and scale must match bit for bit, including the special
rows (NaN entries, zero rows, subnormal and overflowing sums of squares).
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


def assert_bits(c, s, rc, rs):
    bad = np.nonzero((c != rc).any(1) | (s.view(np.uint32) != rs.view(np.uint32)).any(1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first slot {bad[0]}"


def test_append_value_mix_bit_exact():
    p = workloads.producer_inputs(65536)
    c, s, rc, rs, err = run(p)
    assert err == 0
    assert_bits(c, s, rc, rs)


@pytest.mark.parametrize("stride,slots", [(D, None), (600, "map"), (1024, None)])
def test_strides_and_identity_slots(stride, slots):
    p = workloads.producer_inputs(3000, seed=11)
    c, s, rc, rs, _ = run(p, stride=stride, slots=slots)
    assert_bits(c, s, rc, rs)


def test_positions_outside_the_table_are_skipped_and_flagged():
    p = workloads.producer_inputs(500, max_pos=64, seed=12)
    pos = p.positions.copy()
    pos[[3, 17, 499]] = [-1, 64, 1 << 40]
    c, s, rc, rs, err = run(p, positions=pos)
    assert err & 1
    for r in (3, 17, 499):
        assert np.all(c[p.slots[r]] == 0xAB) and np.all(s[p.slots[r]] == -1.0)
    assert_bits(c, s, rc, rs)


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
        assert_bits(c, s, rc, rs)


def test_empty_call():
    d = torch.device("cuda:0")
    p = workloads.producer_inputs(4)
    pkg.kv8_produce_rows(torch.zeros((0, D), device=d), torch.from_numpy(p.weight).to(d), 1e-6,
                         torch.zeros(0, dtype=torch.int64, device=d),
                         torch.from_numpy(p.rope_cos).to(d), torch.from_numpy(p.rope_sin).to(d),
                         torch.zeros((4, D), dtype=torch.uint8, device=d),
                         torch.zeros((4, 2), device=d))
    torch.cuda.synchronize()
