"""The Python binding's argument checks, on the host.

A tensor of the wrong shape, width or placement handed to a kernel is read or
written out of bounds (a host pointer in a kernel faults the device), so every
wrapper refuses such arguments by name before it calls the library.  Here the
device test is patched to accept host tensors and the library is replaced by a
stand-in that fails the test if any compute call reaches it: each bad argument
must raise, and the same call with that argument fixed must reach the library.
"""
import types

import pytest
import torch

import fp8_mla_latent_gb300 as pkg
from fp8_mla_latent_gb300 import _lib

S, H, B, MB, V, N = 256, 16, 2, 2, 128, 64  # cache slots, heads, sequences, blocks, widths
STREAM = types.SimpleNamespace(cuda_stream=0)


class Reached(Exception):
    pass


class NoLibrary:
    """The size queries answer; any other call raises Reached."""

    def __getattr__(self, name):
        if name.endswith("_workspace_size"):
            return lambda *a: 1 << 16

        def call(*a):
            raise Reached(name)
        return call


@pytest.fixture(autouse=True)
def host_as_device(monkeypatch):
    monkeypatch.setattr(_lib, "_is_device", lambda t: True)
    monkeypatch.setattr(_lib, "lib", lambda: NoLibrary())


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


def cache(slots=S, width=576, scale_rows=None):
    return (torch.zeros((slots, width), dtype=torch.uint8),
            f32(slots if scale_rows is None else scale_rows, 2))


def reaches(fn, *a, **k):
    with pytest.raises(Reached):
        fn(*a, stream=STREAM, **k)


def refuses(exc, name, fn, *a, **k):
    with pytest.raises(exc, match="^" + name):
        fn(*a, stream=STREAM, **k)


def test_quantize():
    codes, scales = cache()
    reaches(pkg.kv8_quantize_rows, f32(4, 576), codes, scales)
    reaches(pkg.kv8_quantize_rows, f32(4, 640), codes, scales)
    refuses(ValueError, "src", pkg.kv8_quantize_rows, f32(4, 512), codes, scales)
    refuses(ValueError, "kv_codes", pkg.kv8_quantize_rows, f32(4, 576), *cache(scale_rows=S - 1))
    refuses(ValueError, "kv_codes", pkg.kv8_quantize_rows, f32(4, 576), *cache(width=512))


def test_produce():
    codes, scales = cache()
    pos = torch.zeros(4, dtype=torch.int64)
    args = (f32(512), 1e-6, pos, f32(32, 32), f32(32, 32))
    reaches(pkg.kv8_produce_rows, f32(4, 576), *args, codes, scales)
    refuses(ValueError, "src", pkg.kv8_produce_rows, f32(4, 575), *args, codes, scales)
    refuses(ValueError, "kv_codes", pkg.kv8_produce_rows, f32(4, 576), *args,
            *cache(scale_rows=S + 1))
    refuses(ValueError, "err_word", pkg.kv8_produce_rows, f32(4, 576), *args, codes, scales,
            err_word=torch.zeros(0, dtype=torch.int32))


def test_prefill():
    codes, scales = cache()
    w = torch.zeros((512, N), dtype=torch.bfloat16)
    reaches(pkg.kv8_prefill_project, codes, scales, w, T=10)
    refuses(ValueError, "kv_codes", pkg.kv8_prefill_project, *cache(scale_rows=S - 1), w, T=10)
    refuses(ValueError, "y", pkg.kv8_prefill_project, codes, scales, w, T=10,
            y=torch.zeros((9, N), dtype=torch.bfloat16))


def test_wuv():
    w = torch.zeros((H, 512, V), dtype=torch.bfloat16)
    reaches(pkg.mla_wuv_epilogue, f32(B, H, 512), w)
    reaches(pkg.mla_wuv_epilogue, f32(B, H, 512), w, y=f32(B, H, V))
    refuses(ValueError, "y", pkg.mla_wuv_epilogue, f32(B, H, 512), w, y=f32(B, H, V - 1))
    refuses(ValueError, "y", pkg.mla_wuv_epilogue, f32(B, H, 512), w, y=f32(B + 1, H, V))


def test_single_decode():
    codes, scales = cache()
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    q, r = f32(H, 512), f32(H, 64)
    d = pkg.mla_absorb_decode_fp8
    reaches(d, q, r, codes, scales, 10, 0.1, workspace=ws)
    reaches(d, q, r, codes, scales, 10, 0.1, out=f32(H, 512), lse=f32(H), workspace=ws)
    refuses(ValueError, "kv_codes", d, q, r, *cache(width=512), 10, 0.1, workspace=ws)
    refuses(ValueError, "out", d, q, r, codes, scales, 10, 0.1, out=f32(H, 256), workspace=ws)
    refuses(ValueError, "lse", d, q, r, codes, scales, 10, 0.1, lse=f32(H + 1), workspace=ws)
    refuses(ValueError, "workspace", d, q, r, codes, scales, 10, 0.1, workspace=ws[::2])
    refuses(TypeError, "workspace", d, q, r, codes, scales, 10, 0.1, workspace=bytearray(64))


def test_batched_decode_and_its_phases():
    codes, scales = cache()
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    ql, qr = f32(B, H, 512), f32(B, H, 64)
    bt = torch.zeros((B, MB), dtype=torch.int32)
    sl = torch.zeros(B, dtype=torch.int32)
    inputs = (ql, qr, codes, scales, bt, sl, 0.1)
    reaches(pkg.mla_absorb_decode_fp8_batch, *inputs, workspace=ws)
    reaches(pkg.mla_absorb_decode_fp8_batch_noalloc, *inputs)
    reaches(pkg.mla_absorb_decode_fp8_batch_partials, *inputs, ws)
    refuses(ValueError, "kv_codes", pkg.mla_absorb_decode_fp8_batch, ql, qr,
            *cache(scale_rows=S - 1), bt, sl, 0.1, workspace=ws)
    refuses(ValueError, "out", pkg.mla_absorb_decode_fp8_batch_noalloc, *inputs,
            out=f32(B, H + 1, 512))
    refuses(ValueError, "block_table", pkg.mla_absorb_decode_fp8_batch_partials, ql, qr, codes,
            scales, bt[:1], sl, 0.1, ws)
    refuses(ValueError, "workspace", pkg.mla_absorb_decode_fp8_batch_partials, *inputs, ws[::2])
    out, lse = f32(B, H, 512), f32(B, H)
    c = pkg.mla_absorb_decode_fp8_batch_combine
    reaches(c, sl, H, MB, out, lse, ws)
    reaches(c, sl, H, MB, out, None, ws)
    refuses(ValueError, "out", c, sl, H + 1, MB, out, lse, ws)
    refuses(ValueError, "lse", c, sl, H, MB, out, lse[:1], ws)
    refuses(TypeError, "seq_lens", c, sl.long(), H, MB, out, lse, ws)
    refuses(ValueError, "workspace", c, sl, H, MB, out, lse, ws[::2])
