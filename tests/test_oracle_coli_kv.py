"""Pins of the oracle's cache-file reader and writer (CPU only).

KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
description, persistence item: version 2 starts with the magic COLIKV2 and keeps
its data type in the header; a row is the fp8 codes plus their scales (the page's
"~46 KB per token" is 79 layers x 584 B).  The byte layout beyond that is this
project's definition; the pins fix the page's facts and the layout's invariants.
"""
import struct

import numpy as np

import oracle
from oracle import coli_kv


def test_magic_and_data_type_are_in_the_header():
    h = coli_kv.header(2, 5)
    assert len(h) == 64 and h[:7] == b"COLIKV2"
    assert struct.unpack("<I", h[12:16])[0] == 2           # data type: e4m3 codes + scales
    assert coli_kv.header(1, 5)[:7] == b"COLIKV1"


def test_record_size_matches_the_page_per_token_figure():
    # the page's ~46 KB per token is the 584-byte row summed over the model's layers
    # (46 KB / 584 B is about 79 layers)
    assert coli_kv.RECORD[2] == 576 + 2 * 4
    assert abs(79 * coli_kv.RECORD[2] / 1000 - 46) < 0.5
    assert coli_kv.RECORD[1] == 4 * 576


def test_round_trip_and_layout(tmp_path):
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 256, (7, 576), dtype=np.uint8)
    scales = rng.standard_normal((7, 2)).astype(np.float32)
    p = str(tmp_path / "a.kv")
    coli_kv.write_v2(p, codes, scales)
    raw = open(p, "rb").read()
    assert len(raw) == 64 + 7 * 584
    # record r: its codes, then sLc and sRc as little-endian f32
    r = 3
    rec = raw[64 + r * 584: 64 + (r + 1) * 584]
    assert rec[:576] == codes[r].tobytes()
    assert struct.unpack("<ff", rec[576:]) == (float(scales[r, 0]), float(scales[r, 1]))
    v, c2, s2 = coli_kv.read(p)
    assert v == 2 and np.array_equal(c2, codes) and np.array_equal(s2.view(np.uint32), scales.view(np.uint32))


def test_torn_tail_is_not_content(tmp_path):
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, (4, 576), dtype=np.uint8)
    scales = np.ones((4, 2), np.float32)
    p = str(tmp_path / "b.kv")
    coli_kv.write_v2(p, codes, scales)
    with open(p, "ab") as f:
        f.write(b"\x55" * 300)                              # half a record, never committed
    v, c2, _ = coli_kv.read(p)
    assert v == 2 and c2.shape[0] == 4


def test_damaged_or_short_headers_are_rejected(tmp_path):
    assert coli_kv.parse_header(b"COLIKV2") is None
    bad = bytearray(coli_kv.header(2, 0))
    bad[0] = ord("X")
    assert coli_kv.parse_header(bytes(bad)) is None
    bad = bytearray(coli_kv.header(2, 0))
    bad[20] = 0                                             # record size != 584
    assert coli_kv.parse_header(bytes(bad)) is None


def test_version_one_rows_quantize_to_the_quantizer_codes(tmp_path):
    """A version-1 file holds f32 rows; resuming it gives the quantizer's codes."""
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((9, 576)).astype(np.float32)
    p = str(tmp_path / "c.kv")
    coli_kv.write_v1(p, rows)
    v, back, _ = coli_kv.read(p)
    assert v == 1 and np.array_equal(back.view(np.uint32), rows.view(np.uint32))
    codes, scales = oracle.quantize_rows(back)
    assert codes.shape == (9, 576) and np.all(np.abs(oracle.decode_table()[codes[:, :512]]).max(axis=1) == 448)
