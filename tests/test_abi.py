"""The C ABI without a GPU: the library loads, exports every call the header
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import fp8_mla_latent_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8mla.h")

EINVAL, EALIGN, EUNSUPPORTED, EWORKSPACE = -1, -2, -3, -6


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for want in ("kv8_quantize_rows", "kv8_produce_rows", "mla_absorb_decode_fp8",
                 "mla_absorb_decode_fp8_batch",
                 "mla_absorb_decode_fp8_workspace_size",
                 "mla_absorb_decode_fp8_batch_workspace_size", "kv8_status_string",
                 "mla_wuv_epilogue", "kv8_prefill_project", "kv8_selftest_wait_timeout"):
        assert want in names


def test_library_exports_every_declared_symbol():
    L = pkg.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_status_strings_and_version():
    L = pkg.lib()
    assert L.kv8_abi_version() >= 100
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert L.kv8_status_string(s)
    assert L.kv8_status_string(12345) == b"unknown status"


def P(x):
    return ctypes.c_void_p(x)


def test_quantize_rejects_bad_arguments_on_host():
    L = pkg.lib()
    f = L.kv8_quantize_rows
    good = 1 << 20  # a 16-byte aligned fake address: never dereferenced because validation fails
    assert f(P(good), -1, 576, None, P(good), P(good), 10, None) == EINVAL
    assert f(None, 4, 576, None, P(good), P(good), 10, None) == EINVAL
    assert f(P(good), 4, 575, None, P(good), P(good), 10, None) == EINVAL
    assert f(P(good), 11, 576, None, P(good), P(good), 10, None) == EINVAL
    assert f(P(good + 4), 4, 576, None, P(good), P(good), 10, None) == EALIGN
    assert f(P(good), 4, 578, None, P(good), P(good), 10, None) == EALIGN
    assert f(P(good), 4, 576, None, P(good + 8), P(good), 10, None) == EALIGN
    assert f(P(good), 4, 576, None, P(good), P(good + 4), 10, None) == EALIGN
    assert f(P(good), 0, 576, None, None, None, 0, None) == 0  # nothing to do


def test_produce_rejects_bad_arguments_on_host():
    L = pkg.lib()
    f = L.kv8_produce_rows
    g = 1 << 20
    base = [P(g), 4, 576, P(g), 1e-6, P(g), P(g), P(g), 16, None, P(g), P(g), 10, None, None]

    def call(**kw):
        a = list(base)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return f(*a)
    assert call(a1=-1) == EINVAL
    assert call(a8=0) == EINVAL                      # max_pos < 1
    assert call(a4=-1.0) == EINVAL                   # negative eps
    assert call(a4=float("nan")) == EINVAL
    assert call(a0=None) == EINVAL
    assert call(a3=None) == EINVAL                   # norm weight
    assert call(a5=None) == EINVAL                   # positions
    assert call(a6=None) == EINVAL
    assert call(a2=575) == EINVAL
    assert call(a1=11) == EINVAL                     # identity slots past n_slots
    assert call(a0=P(g + 4)) == EALIGN
    assert call(a2=578) == EALIGN
    assert call(a3=P(g + 4)) == EALIGN
    assert call(a5=P(g + 4)) == EALIGN
    assert call(a10=P(g + 8)) == EALIGN
    assert call(a13=P(g + 2)) == EALIGN
    assert call(a1=0, a0=None, a3=None) == 0         # nothing to do


def test_wuv_rejects_bad_arguments_on_host():
    f = pkg.lib().mla_wuv_epilogue
    g = 1 << 20
    assert f(P(g), P(g), -1, 4, 128, P(g), None) == EINVAL
    assert f(P(g), P(g), 2, 0, 128, P(g), None) == EINVAL
    assert f(P(g), P(g), 2, 4, 0, P(g), None) == EINVAL
    assert f(P(g), P(g), 2, 4, 5000, P(g), None) == EINVAL
    assert f(None, P(g), 2, 4, 128, P(g), None) == EINVAL
    assert f(P(g + 2), P(g), 2, 4, 128, P(g), None) == EALIGN
    assert f(P(g), P(g + 1), 2, 4, 128, P(g), None) == EALIGN
    assert f(None, None, 0, 4, 128, None, None) == 0


def test_decode_rejects_bad_arguments_on_host():
    L = pkg.lib()
    g = 1 << 20
    d = L.mla_absorb_decode_fp8
    assert d(P(g), P(g), P(g), P(g), -1, 4, 0.1, P(g), None, P(g), 1 << 30, 0, None) == EINVAL
    assert d(P(g), P(g), P(g), P(g), 10, 0, 0.1, P(g), None, P(g), 1 << 30, 0, None) == EINVAL
    assert d(P(g), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g), 1 << 30, 7, None) == EINVAL
    assert d(P(g), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g), 1 << 30, 5, None) == EINVAL
    assert d(P(g), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g), 1 << 30, -1, None) == EINVAL
    # the softmax scale must be positive and finite
    for bad in (0.0, -0.1, float("nan"), float("inf"), -float("inf")):
        assert d(P(g), P(g), P(g), P(g), 10, 4, bad, P(g), None, P(g), 1 << 30, 0, None) == EINVAL
    # the row scales are read by TMA: 16-byte aligned
    assert d(P(g), P(g), P(g), P(g + 8), 10, 4, 0.1, P(g), None, P(g), 1 << 30, 0, None) == EALIGN
    assert d(None, P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g), 1 << 30, 0, None) == EINVAL
    assert d(P(g + 8), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g), 1 << 30, 0, None) == EALIGN
    assert d(P(g), P(g), P(g + 1), P(g), 10, 4, 0.1, P(g), None, P(g), 1 << 30, 0, None) == EALIGN
    need = L.mla_absorb_decode_fp8_workspace_size(10, 4, 0)
    assert need > 0
    assert d(P(g), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g), need - 1, 0, None) == EWORKSPACE
    assert d(P(g), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, None, need, 0, None) == EWORKSPACE
    assert d(P(g), P(g), P(g), P(g), 10, 4, 0.1, P(g), None, P(g + 16), need, 0, None) == EALIGN
    b = L.mla_absorb_decode_fp8_batch
    args = [P(g)] * 6 + [2, 4, 8, 64, 16, 0.1, P(g), None, P(g), 1 << 30, 0, None]
    a = list(args)
    a[9] = 32
    assert b(*a) == EUNSUPPORTED
    a = list(args)
    a[4] = None
    assert b(*a) == EINVAL
    a = list(args)
    a[10] = 0
    assert b(*a) == EINVAL
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        a = list(args)
        a[11] = bad
        assert b(*a) == EINVAL
        assert L.mla_absorb_decode_fp8_batch_partials(*(a[:12] + [P(g), 1 << 30, 0, None])) == EINVAL
        assert L.mla_absorb_decode_fp8_batch_noalloc(*(a[:14] + [0, None])) == EINVAL
    a = list(args)
    a[3] = P(g + 8)
    assert b(*a) == EALIGN
    assert b(*([P(g)] * 6 + [0, 4, 8, 64, 16, 0.1, P(g), None, P(g), 1 << 30, 0, None])) == 0


def test_wrappers_refuse_host_tensors_before_the_library():
    """A host pointer handed to a kernel would fault the device, so the binding
    refuses host tensors by name before anything reaches the library (without a
    GPU every tensor is a host tensor)."""
    ws = torch.empty(64, dtype=torch.uint8)
    with pytest.raises(ValueError, match="^workspace"):
        pkg.kv8_workspace_error(ws)
    with pytest.raises(TypeError, match="^workspace"):
        pkg.kv8_workspace_error(bytes(64))
    sl = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(TypeError, match="^seq_lens"):
        pkg.mla_absorb_decode_fp8_batch_combine(sl.long(), 4, 2, None, None, ws)
    with pytest.raises(ValueError, match="^seq_lens"):
        pkg.mla_absorb_decode_fp8_batch_combine(sl, 4, 2, None, None, ws)


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4])
def test_workspace_sizes(variant):
    L = pkg.lib()
    for T, H in ((0, 1), (1, 4), (256, 4), (4096, 128), (262144, 128)):
        n = L.mla_absorb_decode_fp8_workspace_size(T, H, variant)
        assert n >= 256 and n % 256 == 0
    assert L.mla_absorb_decode_fp8_workspace_size(-1, 4, variant) < 0
    assert L.mla_absorb_decode_fp8_batch_workspace_size(32, 128, 512, 64, variant) > 0
    assert L.mla_absorb_decode_fp8_batch_workspace_size(32, 128, 512, 32, variant) < 0
    # more tokens never needs a smaller workspace per split partial
    assert (L.mla_absorb_decode_fp8_batch_workspace_size(2, 128, 4096, 64, variant)
            >= L.mla_absorb_decode_fp8_batch_workspace_size(2, 128, 1, 64, variant))
    assert L.mla_absorb_decode_fp8_batch_workspace_size(2, 128, 4096, 64, 5) < 0


def test_tensor_core_workspace_covers_both_kernels():
    """The automatic tensor-core choice and the two forced kernels plan their own
    splits; each size query matches the kernel its call runs."""
    L = pkg.lib()
    for B, H in ((1, 16), (2, 64), (2, 65), (2, 128), (32, 128), (3, 200)):
        auto = L.mla_absorb_decode_fp8_batch_workspace_size(B, H, 512, 64, 2)
        cta = L.mla_absorb_decode_fp8_batch_workspace_size(B, H, 512, 64, 3)
        pair = L.mla_absorb_decode_fp8_batch_workspace_size(B, H, 512, 64, 4)
        assert auto == (pair if H > 64 else cta)


def test_selftest_rejects_bad_arguments_on_host():
    f = pkg.lib().kv8_selftest_wait_timeout
    g = 1 << 20
    assert f(P(g), 256, 0, None) == EINVAL
    assert f(P(g), 256, 20_000_000, None) == EINVAL
    assert f(None, 256, 1000, None) == EWORKSPACE
    assert f(P(g), 255, 1000, None) == EWORKSPACE
    assert f(P(g + 16), 256, 1000, None) == EALIGN


def test_prefill_rejects_bad_arguments_on_host():
    f = pkg.lib().kv8_prefill_project
    g = 1 << 20
    base = [P(g), P(g), 100, None, 64, P(g), 512, P(g), None, None, None]

    def call(**kw):
        a = list(base)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return f(*a)
    assert call(a4=-1) == EINVAL
    assert call(a6=300) == EINVAL          # N not a multiple of 256
    assert call(a6=0) == EINVAL
    assert call(a4=101) == EINVAL          # identity slots past the pool
    assert call(a0=None) == EINVAL
    assert call(a5=None) == EINVAL
    assert call(a0=P(g + 8)) == EALIGN
    assert call(a5=P(g + 8)) == EALIGN
    assert call(a7=P(g + 8)) == EALIGN
    assert call(a3=P(g + 4)) == EALIGN
    assert call(a8=P(g + 8)) == EALIGN      # k_rope
    assert call(a9=P(g + 2)) == EALIGN      # err_word
    assert call(a4=0, a0=None) == 0


def test_disk_rejects_bad_arguments_on_host():
    L = pkg.lib()
    h = ctypes.c_void_p()
    assert L.kv8_disk_open(None, 16, ctypes.byref(h)) == EINVAL
    assert L.kv8_disk_open(b"", 16, ctypes.byref(h)) == EINVAL
    assert L.kv8_disk_open(b"/tmp/x.kv", 0, ctypes.byref(h)) == EINVAL
    assert L.kv8_disk_open(b"/tmp/x.kv", 1 << 23, ctypes.byref(h)) == EINVAL
    assert L.kv8_disk_open(b"/tmp/x.kv", 16, None) == EINVAL
    n = ctypes.c_int64()
    assert L.kv8_disk_info(None, ctypes.byref(n), None) == EINVAL
    assert L.kv8_disk_append(None, None, None, 0, None, 0, None) == EINVAL
    assert L.kv8_disk_load(None, 0, 0, None, None, 0, None, None) == EINVAL
    assert L.kv8_disk_close(None) == 0
    assert L.kv8_status_string(-9) == b"cache file read, write or rename failed"
