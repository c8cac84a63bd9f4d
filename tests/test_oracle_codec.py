"""Pins for the oracle's e4m3 codec (CPU only).

The codec rules come from the KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU +
CUDA) with .coli_kv v2"), PR description, c/kv_fp8.h item and Tests item.  The
oracle is checked against things other than itself: the closed form of the
format, hand-worked tie cases (tests/golden/e4m3_rne_cases.txt), a brute-force
nearest-value search, an independent midpoint-bracket search over every f32 bit
pattern, and torch's float8_e4m3fn cast (a library routine).
"""
import os
import struct

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_from_bits(u):
    return struct.unpack("<f", struct.pack("<I", u))[0]


def test_decode_spot_values_closed_form():
    t = oracle.decode_table()
    assert t[0x38] == 1.0
    assert t[0x7E] == 448.0
    assert t[0x08] == 2.0 ** -6
    assert t[0x01] == 2.0 ** -9
    assert t[0x07] == 7 * 2.0 ** -9
    assert t[0x3F] == 1.875
    assert t[0x40] == 2.0
    assert t[0xC0] == -2.0
    assert t[0x00] == 0.0 and not np.signbit(t[0x00])
    assert t[0x80] == 0.0 and np.signbit(t[0x80])
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2


def test_decode_matches_torch_float8_e4m3fn():
    t = oracle.decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(t))
    assert np.array_equal(ref[~nan].view(np.uint32), t[~nan].view(np.uint32))  # signed zeros too


def test_exhaustive_256_code_round_trip():
    t = oracle.decode_table()
    back = oracle.encode(t)
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert back[c] == 0x00, "NaN codes re-encode as inert 0"
        else:
            assert back[c] == c, hex(c)


def _load_cases():
    cases = []
    with open(os.path.join(GOLDEN, "e4m3_rne_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            x = f32_from_bits(int(parts[0], 16)) if parts[0].startswith("0x") else float(parts[0])
            cases.append((parts[0], x, int(parts[1], 16)))
    return cases


@pytest.mark.parametrize("src,x,code", _load_cases())
def test_golden_rne_cases(src, x, code):
    assert int(oracle.encode(np.array([x], np.float32))[0]) == code, src


def test_every_midpoint_ties_to_even():
    t = oracle.decode_table()
    pos = t[:0x7F].astype(np.float64)  # 0x00..0x7E ascending
    assert np.all(np.diff(pos) > 0)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact
    got = oracle.encode(mids)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want.astype(np.uint8))
    assert np.array_equal(oracle.encode(-mids), (want | 0x80).astype(np.uint8))


def _near_patterns():
    """Code values and midpoints, each +-1 and +-2 ulp, both signs."""
    t = oracle.decode_table()
    pos = t[:0x7F].astype(np.float64)
    pts = np.concatenate([pos, (pos[:-1] + pos[1:]) / 2, [448.0, 464.0, 480.0]]).astype(np.float32)
    bits = pts.view(np.uint32).astype(np.int64)
    allb = np.concatenate([bits + d for d in (-2, -1, 0, 1, 2)])
    allb = allb[(allb >= 0) & (allb < 0x7F800000)]
    allb = np.concatenate([allb, allb | 0x80000000]).astype(np.uint32)
    return allb


def test_bitmath_equals_brute_force_near_ties():
    n, first = oracle.list_mismatches_nearest(_near_patterns())
    assert n == 0, hex(first)


def test_bitmath_equals_brute_force_random_patterns():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=1 << 19, dtype=np.uint64).astype(np.uint32)
    # bias half the sample into the finite e4m3 range, where rounding happens
    small = rng.integers(0x2F000000, 0x43E80000, size=1 << 19, dtype=np.uint64).astype(np.uint32)
    small ^= (rng.integers(0, 2, size=small.size, dtype=np.uint32) << 31).astype(np.uint32)
    n, first = oracle.list_mismatches_nearest(np.concatenate([bits, small]))
    assert n == 0, hex(first)


def test_bitmath_equals_bracket_on_all_2_32_patterns():
    """Every f32 bit pattern: bit-math encoder == independent midpoint-bracket encoder."""
    n, first = oracle.exhaustive_mismatches(0, 1 << 32)
    assert n == 0, hex(first)


def test_bitmath_matches_torch_cast_in_range():
    """torch's float8_e4m3fn cast rounds to nearest even; outside |q| <= 464 it
    returns NaN instead of saturating, and it keeps NaN, so compare in range."""
    rng = np.random.default_rng(5)
    mags = rng.integers(0, 0x43E80001, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    sgn = (rng.integers(0, 2, size=mags.size, dtype=np.uint32) << 31).astype(np.uint32)
    x = np.concatenate([(mags | sgn), _near_patterns()]).view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 464.0)]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.encode(x)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, (x[bad[:5]], ref[bad[:5]], got[bad[:5]])
