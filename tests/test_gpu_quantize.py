"""GPU quantizer parity: bit-exact codes and scales against the oracle.

Rules: KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv
v2"), PR description, c/kv_fp8.h item.  The encoder is exercised on every
non-negative f32 pattern up to 448 (rows whose amax is exactly 448 make the
inverse scale 1, so the stored code is the encoding of the pattern itself),
plus sampled negatives, the workloads' rows and hand-made special rows.
"""
import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
import oracle
from fp8_mla_latent_gb300 import workloads

pytestmark = pytest.mark.gpu
D, DL = 576, 512


def gpu_quant(x, n_slots=None, slots=None, stride=None):
    d = torch.device("cuda:0")
    n = x.shape[0]
    n_slots = n if n_slots is None else n_slots
    if stride is not None and stride != D:
        buf = torch.zeros((n, stride), dtype=torch.float32, device=d)
        buf[:, :D] = torch.from_numpy(x).to(d)
        src = buf
    else:
        src = torch.from_numpy(np.ascontiguousarray(x)).to(d)
    codes = torch.full((n_slots, D), 0xAB, dtype=torch.uint8, device=d)
    scales = torch.full((n_slots, 2), -1.0, dtype=torch.float32, device=d)
    st = None if slots is None else torch.from_numpy(np.asarray(slots, np.int64)).to(d)
    pkg.kv8_quantize_rows(src, codes, scales, dst_slot=st)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def assert_same(x, c, s, slots=None, n_slots=None):
    rc, rs = oracle.quantize_rows(x, dst_slot=slots, n_slots=n_slots)
    idx = np.arange(len(x)) if slots is None else np.asarray(slots)
    bad = np.nonzero((c[idx] != rc[idx]).any(1))[0]
    assert bad.size == 0, f"rows {bad[:5]} differ"
    assert np.array_equal(s[idx].view(np.uint32), rs[idx].view(np.uint32))


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_workload_rows_bit_exact(name):
    w = workloads.make(name, scale=0.05)
    x = w.cache_rows if w.fresh_rows is None else np.concatenate([w.cache_rows, w.fresh_rows])
    c, s = gpu_quant(x)
    assert_same(x, c, s)


def test_append_workload_full_size_bit_exact():
    """The 65536 fresh rows of the append workload at full size."""
    w = workloads.make("append")
    c, s = gpu_quant(w.fresh_rows)
    assert_same(w.fresh_rows, c, s)


def test_encoder_on_every_pattern_up_to_448():
    d = torch.device("cuda:0")
    per_row = DL - 1
    hi = 0x43E00000 + 1  # every non-negative pattern <= 448.0
    chunk_rows = 1 << 16
    codes = torch.empty((chunk_rows, D), dtype=torch.uint8, device=d)
    scales = torch.empty((chunk_rows, 2), dtype=torch.float32, device=d)
    src = torch.empty((chunk_rows, D), dtype=torch.float32, device=d)
    src[:, DL:] = 448.0  # Rc: amax 448 too
    src[:, 0] = 448.0    # Lc amax 448 -> inverse scale exactly 1
    start = 0
    step = chunk_rows * per_row
    while start < hi:
        n = min(step, hi - start)
        rows = (n + per_row - 1) // per_row
        pat = torch.arange(start, start + rows * per_row, dtype=torch.int64, device=d)
        pat = torch.clamp(pat, max=hi - 1).to(torch.int32).view(torch.float32)
        src[:rows, 1:DL] = pat.view(rows, per_row)
        pkg.kv8_quantize_rows(src[:rows], codes[:rows], scales[:rows])
        got = codes[:rows, 1:DL].reshape(-1).cpu().numpy()
        want = oracle.encode(pat.cpu().numpy())
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"pattern {hex(start + int(bad[0]))}: gpu {got[bad[0]]:#x} want {want[bad[0]]:#x}"
        start += step
    assert torch.all(scales[:1] == 1.0)


def test_encoder_negative_and_near_tie_patterns():
    t = oracle.decode_table().astype(np.float64)[:0x7F]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32).view(np.uint32).astype(np.int64)
    vals = t.astype(np.float32).view(np.uint32).astype(np.int64)
    pats = np.concatenate([m + d for m in (mids, vals) for d in (-1, 0, 1)])
    pats = np.clip(pats, 0, 0x43E00000).astype(np.uint32)
    rng = np.random.default_rng(3)
    pats = np.concatenate([pats, rng.integers(0, 0x43E00001, 200000, dtype=np.uint64)
                           .astype(np.uint32)])
    x = pats.view(np.float32)
    x = np.concatenate([x, -x])
    per_row = DL - 1
    rows = (x.size + per_row - 1) // per_row
    buf = np.zeros(rows * per_row, np.float32)
    buf[:x.size] = x
    src = np.zeros((rows, D), np.float32)
    src[:, 0] = 448.0
    src[:, 1:DL] = buf.reshape(rows, per_row)
    src[:, DL:] = -448.0
    c, s = gpu_quant(src)
    assert_same(src, c, s)


def test_special_rows():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((12, D)).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2, ::3] = -0.0
    x[2, 1::3] = 0.0
    x[3] *= np.float32(2.0 ** -140)                  # subnormal amax: guard
    x[4, :DL] = np.float32(1e-38)                     # below 448/FLT_MAX: guard
    x[5, 7] = np.nan
    x[5, 600 - 30] = np.nan
    x[6, :DL] = np.nan                                # all-NaN segment
    x[7, 3] = np.inf                                  # unsupported, must not fault
    x[8, 520] = -np.inf
    fmax = np.finfo(np.float32).max
    thr = np.float32(448.0) / np.float32(fmax)
    x[9, :] = thr
    x[10, :] = np.nextafter(thr, np.float32(0))
    x[11] *= np.float32(1e30)
    c, s = gpu_quant(x)
    assert_same(x, c, s)


def test_slot_scatter_skips_out_of_range_and_honours_stride():
    rng = np.random.default_rng(4)
    x = rng.standard_t(3, size=(40, D)).astype(np.float32)
    slots = rng.permutation(64)[:40].astype(np.int64)
    slots[5] = -1
    slots[9] = 64  # out of range: skipped
    c, s = gpu_quant(x, n_slots=64, slots=slots, stride=640)
    ok = (slots >= 0) & (slots < 64)
    assert_same(x[ok], c, s, slots=slots[ok], n_slots=64)
    untouched = np.setdiff1d(np.arange(64), slots[ok])
    assert np.all(c[untouched] == 0xAB) and np.all(s[untouched] == -1.0)


def test_zero_rows_is_a_no_op():
    d = torch.device("cuda:0")
    codes = torch.zeros((4, D), dtype=torch.uint8, device=d)
    scales = torch.zeros((4, 2), dtype=torch.float32, device=d)
    pkg.kv8_quantize_rows(torch.zeros((0, D), device=d), codes, scales)
    torch.cuda.synchronize()
    assert int(codes.sum()) == 0
