"""GPU tests of the cache file: rows saved from a device cache and loaded back
through the library, checked byte for byte against the oracle's reader and
writer (an independent plain-Python statement of the file layout) and against
the oracle's quantizer for version-1 files."""
import os

import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
import oracle
from oracle import coli_kv

pytestmark = pytest.mark.gpu


def dev():
    return torch.device("cuda:0")


def device_cache(rng, n_slots):
    rows = (rng.standard_normal((n_slots, 576)) * np.exp(0.5 * rng.standard_normal(576))).astype(np.float32)
    codes = torch.zeros((n_slots, 576), dtype=torch.uint8, device=dev())
    scales = torch.zeros((n_slots, 2), dtype=torch.float32, device=dev())
    pkg.kv8_quantize_rows(torch.from_numpy(rows).to(dev()), codes, scales)
    return codes, scales


@pytest.mark.parametrize("staging", [4096, 37])
def test_append_then_load_round_trip(tmp_path, staging):
    rng = np.random.default_rng(staging)
    codes, scales = device_cache(rng, 1000)
    c_np, s_np = codes.cpu().numpy(), scales.cpu().numpy()
    path = str(tmp_path / "cache.kv")
    picks = rng.permutation(1000)[:300].astype(np.int64)
    with pkg.Kv8Disk(path, staging_rows=staging) as d:
        assert d.info() == (0, 2)
        d.append(codes, scales, slots=torch.from_numpy(picks[:120]).to(dev()))
        d.append(codes, scales, slots=torch.from_numpy(picks[120:]).to(dev()))
        assert d.info() == (300, 2)
    v, fc, fs = coli_kv.read(path)
    assert v == 2
    assert np.array_equal(fc, c_np[picks])
    assert np.array_equal(fs.view(np.uint32), s_np[picks].view(np.uint32))
    # resume into a fresh cache at other slots
    c2 = torch.zeros_like(codes)
    s2 = torch.zeros_like(scales)
    dst = 20 + rng.permutation(980)[:300].astype(np.int64)   # clear of slots 10..14 below
    with pkg.Kv8Disk(path, staging_rows=staging) as d:
        d.load(c2, s2, dst_slot=torch.from_numpy(dst).to(dev()))
        d.load(c2, s2, first_row=10, n=5)          # identity slots 10..14
    got_c, got_s = c2.cpu().numpy(), s2.cpu().numpy()
    assert np.array_equal(got_c[dst[15:]], c_np[picks[15:]])
    assert np.array_equal(got_c[10:15], c_np[picks[10:15]])
    assert np.array_equal(got_s[10:15].view(np.uint32), s_np[picks[10:15]].view(np.uint32))


def test_identity_append_and_torn_tail(tmp_path):
    rng = np.random.default_rng(3)
    codes, scales = device_cache(rng, 64)
    path = str(tmp_path / "t.kv")
    with pkg.Kv8Disk(path) as d:
        d.append(codes, scales, n=40)
    with open(path, "ab") as f:
        f.write(b"\x77" * 1000)                    # a torn append: not committed
    with pkg.Kv8Disk(path) as d:
        assert d.info() == (40, 2)
        d.append(codes, scales, slots=torch.arange(40, 64, dtype=torch.int64, device=dev()))
    v, fc, _ = coli_kv.read(path)
    assert v == 2 and np.array_equal(fc, codes.cpu().numpy())
    assert os.path.getsize(path) >= 64 + 64 * 584


def test_bad_slot_commits_nothing(tmp_path):
    rng = np.random.default_rng(4)
    codes, scales = device_cache(rng, 50)
    path = str(tmp_path / "b.kv")
    with pkg.Kv8Disk(path) as d:
        d.append(codes, scales, n=10)
        bad = torch.tensor([1, 2, 50], dtype=torch.int64, device=dev())
        with pytest.raises(pkg.Kv8Error) as e:
            d.append(codes, scales, slots=bad)
        assert e.value.status == -5
        assert d.info() == (10, 2)
        with pytest.raises(pkg.Kv8Error):
            d.load(codes, scales, dst_slot=torch.tensor([0, -1], dtype=torch.int64, device=dev()))
    assert coli_kv.read(path)[1].shape[0] == 10


def test_version_one_file_is_quantized_on_resume_and_rewritten_at_append(tmp_path):
    rng = np.random.default_rng(5)
    rows = (rng.standard_normal((70, 576)) * 3).astype(np.float32)
    rows[4] = 0.0
    rows[9, 7] = np.nan
    path = str(tmp_path / "v1.kv")
    coli_kv.write_v1(path, rows)
    ref_c, ref_s = oracle.quantize_rows(rows)
    c = torch.zeros((80, 576), dtype=torch.uint8, device=dev())
    s = torch.zeros((80, 2), dtype=torch.float32, device=dev())
    with pkg.Kv8Disk(path, staging_rows=16) as d:
        assert d.info() == (70, 1)
        d.load(c, s)                                # identity slots 0..69
        d.load(c, s, first_row=60, dst_slot=torch.arange(70, 80, dtype=torch.int64, device=dev()))
    assert np.array_equal(c.cpu().numpy()[:70], ref_c)
    assert np.array_equal(s.cpu().numpy()[:70].view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(c.cpu().numpy()[70:], ref_c[60:])
    assert coli_kv.read(path)[0] == 1               # untouched until the first append
    with pkg.Kv8Disk(path, staging_rows=16) as d:
        d.append(c, s, slots=torch.tensor([70, 71], dtype=torch.int64, device=dev()))
        assert d.info() == (72, 2)
    v, fc, fs = coli_kv.read(path)
    assert v == 2
    assert np.array_equal(fc[:70], ref_c) and np.array_equal(fc[70:], ref_c[60:62])
    assert np.array_equal(fs[:70].view(np.uint32), ref_s.view(np.uint32))


def test_open_repairs_a_damaged_magic_and_heals_an_empty_file(tmp_path):
    rng = np.random.default_rng(6)
    codes, scales = device_cache(rng, 8)
    path = str(tmp_path / "m.kv")
    coli_kv.write_v2(path, codes.cpu().numpy(), scales.cpu().numpy())
    with open(path, "r+b") as f:
        f.write(b"GARBAGE")                         # the magic only
    with pkg.Kv8Disk(path) as d:
        assert d.info() == (8, 2)
    assert coli_kv.read(path)[0] == 2
    empty = str(tmp_path / "e.kv")
    open(empty, "wb").write(b"COL")                 # torn at creation
    with pkg.Kv8Disk(empty) as d:
        assert d.info() == (0, 2)
    foreign = str(tmp_path / "f.kv")
    open(foreign, "wb").write(b"x" * 200)
    with pytest.raises(pkg.Kv8Error) as e:
        pkg.Kv8Disk(foreign)
    assert e.value.status == -10
