"""ctypes binding of libfp8mla.so with the same names as the C ABI (include/fp8mla.h).

Argument marshalling only: tensors are checked for device, dtype and layout,
their device pointers and the current CUDA stream are passed through, and a
non-zero status raises.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU fallback, and a missing library or missing CUDA
device raises instead of computing anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

KV8_DL, KV8_DR, KV8_D, KV8_BLOCK = 512, 64, 576, 64
KV8_DECODE_AUTO, KV8_DECODE_SIMT, KV8_DECODE_TCGEN05 = 0, 1, 2
KV8_DECODE_TCGEN05_CTA, KV8_DECODE_TCGEN05_PAIR = 3, 4
STATUS = {0: "KV8_OK", -1: "KV8_EINVAL", -2: "KV8_EALIGN", -3: "KV8_EUNSUPPORTED",
          -4: "KV8_ECUDA", -5: "KV8_EBOUNDS", -6: "KV8_EWORKSPACE", -7: "KV8_ETIMEOUT",
          -8: "KV8_ESCRATCH", -9: "KV8_EIO", -10: "KV8_EFORMAT"}

_lock = threading.Lock()
_lib = None


class Kv8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().kv8_status_string(status).decode()
        if status in (-3, -4):
            msg += ", " + lib().kv8_last_cuda_error().decode()
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({msg})")


def lib() -> ctypes.CDLL:
    """Load libfp8mla.so, building it in-tree first if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            if not _build.up_to_date():
                _build.build()
            L = ctypes.CDLL(_build.LIB)
            P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            sig = {
                "kv8_quantize_rows": (i32, [P, i64, i64, P, P, P, i64, P]),
                "kv8_produce_rows": (i32, [P, i64, i64, P, ctypes.c_float, P, P, P, i64, P, P, P,
                                           i64, P, P]),
                "mla_wuv_epilogue": (i32, [P, P, i32, i32, i32, P, P]),
                "kv8_selftest_wait_timeout": (i32, [P, i64, i64, P]),
                "kv8_prefill_project": (i32, [P, P, i64, P, i64, P, i32, P, P, P, P]),
                "mla_absorb_decode_fp8_workspace_size": (i64, [i64, i32, i32]),
                "mla_absorb_decode_fp8": (i32, [P, P, P, P, i64, i32, f32, P, P, P, i64, i32, P]),
                "mla_absorb_decode_fp8_batch_workspace_size": (i64, [i32, i32, i32, i32, i32]),
                "mla_absorb_decode_fp8_batch": (i32, [P, P, P, P, P, P, i32, i32, i32, i32, i64, f32,
                                                      P, P, P, i64, i32, P]),
                "mla_absorb_decode_fp8_batch_partials": (i32, [P, P, P, P, P, P, i32, i32, i32, i32,
                                                               i64, f32, P, i64, i32, P]),
                "mla_absorb_decode_fp8_batch_combine": (i32, [P, i32, i32, i32, i32, P, P, P, i64,
                                                              i32, P]),
                "mla_absorb_decode_fp8_batch_noalloc": (i32, [P, P, P, P, P, P, i32, i32, i32, i32,
                                                              i64, f32, P, P, i32, P]),
                "kv8_noalloc_error": (i32, [P]),
                "kv8_workspace_error": (i32, [P, P]),
                "kv8_disk_open": (i32, [ctypes.c_char_p, i64, ctypes.POINTER(P)]),
                "kv8_disk_info": (i32, [P, ctypes.POINTER(i64), ctypes.POINTER(i32)]),
                "kv8_disk_append": (i32, [P, P, P, i64, P, i64, P]),
                "kv8_disk_load": (i32, [P, i64, i64, P, P, i64, P, P]),
                "kv8_disk_close": (i32, [P]),
                "kv8_status_string": (ctypes.c_char_p, [i32]),
                "kv8_last_cuda_error": (ctypes.c_char_p, []),
                "kv8_abi_version": (i32, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def library_path() -> str:
    return os.path.abspath(_build.LIB)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _is_device(t) -> bool:
    """Whether a tensor lives in device memory (the one place the binding asks)."""
    return t.is_cuda


def _need(t, name, dtype, ndim=None, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device and not _is_device(t):
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


def _need_cache(kv_codes, kv_scales):
    """The cache: codes uint8 [slots, 576] and their row scales f32 [slots, 2]."""
    _need(kv_codes, "kv_codes", torch.uint8, 2)
    _need(kv_scales, "kv_scales", torch.float32, 2)
    if kv_codes.shape[1] != KV8_D or tuple(kv_scales.shape) != (kv_codes.shape[0], 2):
        raise ValueError("kv_codes must be [slots,576] and kv_scales [slots,2]")


def _need_workspace(ws):
    """A caller's workspace: a contiguous CUDA tensor of any dtype (its size is
    checked by the library against the call's need)."""
    if not isinstance(ws, torch.Tensor):
        raise TypeError("workspace must be a torch.Tensor")
    if not _is_device(ws):
        raise ValueError("workspace must be a CUDA tensor (the library has no CPU path)")
    if not ws.is_contiguous():
        raise ValueError("workspace must be contiguous")


def _check(fn, status):
    if status != 0:
        raise Kv8Error(fn, status)


# ----------------------------------------------------------------- quantizer
def kv8_quantize_rows(src, kv_codes, kv_scales, dst_slot=None, stream=None):
    """Quantize f32 rows src [n, >=576] (row stride = src.stride(0)) into the cache."""
    if not (isinstance(src, torch.Tensor) and src.dtype == torch.float32 and _is_device(src)
            and src.dim() == 2 and src.stride(1) == 1
            and src.shape[1] >= KV8_D):
        raise ValueError("src must be a CUDA float32 [n, >=576] tensor with unit column stride")
    _need_cache(kv_codes, kv_scales)
    if dst_slot is not None:
        _need(dst_slot, "dst_slot", torch.int64, 1)
        if dst_slot.numel() != src.shape[0]:
            raise ValueError("dst_slot must have one entry per source row")
    st = lib().kv8_quantize_rows(_ptr(src), src.shape[0], src.stride(0), _ptr(dst_slot),
                                 _ptr(kv_codes), _ptr(kv_scales), kv_codes.shape[0],
                                 _stream(stream))
    _check("kv8_quantize_rows", st)


def kv8_produce_rows(src, norm_weight, eps, positions, rope_cos, rope_sin, kv_codes, kv_scales,
                     dst_slot=None, err_word=None, stream=None):
    """Fused producer: RMS norm (Lc) + rotary pairs (Rc) + quantize raw rows src [n, >=576]."""
    if not (isinstance(src, torch.Tensor) and src.dtype == torch.float32 and _is_device(src)
            and src.dim() == 2 and src.stride(1) == 1
            and src.shape[1] >= KV8_D):
        raise ValueError("src must be a CUDA float32 [n, >=576] tensor with unit column stride")
    _need(norm_weight, "norm_weight", torch.float32, 1)
    _need(positions, "positions", torch.int64, 1)
    _need(rope_cos, "rope_cos", torch.float32, 2)
    _need(rope_sin, "rope_sin", torch.float32, 2)
    _need_cache(kv_codes, kv_scales)
    if norm_weight.numel() != KV8_DL:
        raise ValueError("norm_weight must have 512 entries")
    if positions.numel() != src.shape[0]:
        raise ValueError("positions must have one entry per source row")
    if rope_cos.shape != rope_sin.shape or rope_cos.shape[1] != KV8_DR // 2:
        raise ValueError("rope_cos and rope_sin must both be [max_pos, 32]")
    if dst_slot is not None:
        _need(dst_slot, "dst_slot", torch.int64, 1)
        if dst_slot.numel() != src.shape[0]:
            raise ValueError("dst_slot must have one entry per source row")
    if err_word is not None and not (isinstance(err_word, torch.Tensor) and _is_device(err_word)
                                     and err_word.dtype == torch.int32 and err_word.numel() >= 1):
        raise ValueError("err_word must be a CUDA int32 tensor")
    st = lib().kv8_produce_rows(_ptr(src), src.shape[0], src.stride(0), _ptr(norm_weight),
                                float(eps), _ptr(positions), _ptr(rope_cos), _ptr(rope_sin),
                                rope_cos.shape[0], _ptr(dst_slot), _ptr(kv_codes),
                                _ptr(kv_scales), kv_codes.shape[0], _ptr(err_word),
                                _stream(stream))
    _check("kv8_produce_rows", st)


def kv8_prefill_project(kv_codes, kv_scales, w_ukv, T=None, slots=None, y=None, k_rope=None,
                        err_word=None, stream=None):
    """Y [T, N] bf16 = dequantized cached latent (slots or 0..T-1) @ W_UKV (bf16 [512, N]);
    k_rope (optional f32 [T, 64]) receives the dequantized rope keys."""
    _need_cache(kv_codes, kv_scales)
    if not (isinstance(w_ukv, torch.Tensor) and _is_device(w_ukv) and w_ukv.dim() == 2
            and w_ukv.dtype == torch.bfloat16 and w_ukv.is_contiguous() and w_ukv.shape[0] == KV8_DL):
        raise ValueError("w_ukv must be a contiguous CUDA bfloat16 [512, N] tensor")
    if slots is not None:
        _need(slots, "slots", torch.int64, 1)
        T = slots.numel()
    elif T is None:
        T = kv_codes.shape[0]
    N = w_ukv.shape[1]
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=kv_codes.device)
    if not (y.dtype == torch.bfloat16 and _is_device(y) and y.is_contiguous() and tuple(y.shape) == (T, N)):
        raise ValueError("y must be a contiguous CUDA bfloat16 [T, N] tensor")
    if k_rope is not None and not (k_rope.dtype == torch.float32 and _is_device(k_rope)
                                   and k_rope.is_contiguous() and tuple(k_rope.shape) == (T, KV8_DR)):
        raise ValueError("k_rope must be a contiguous CUDA float32 [T, 64] tensor")
    if err_word is not None and not (isinstance(err_word, torch.Tensor) and _is_device(err_word)
                                     and err_word.dtype == torch.int32 and err_word.numel() >= 1):
        raise ValueError("err_word must be a CUDA int32 tensor")
    st = lib().kv8_prefill_project(_ptr(kv_codes), _ptr(kv_scales), kv_codes.shape[0], _ptr(slots),
                                   int(T), _ptr(w_ukv), int(N), _ptr(y), _ptr(k_rope),
                                   _ptr(err_word), _stream(stream))
    _check("kv8_prefill_project", st)
    return y


def kv8_selftest_wait_timeout(workspace, limit_us: int, stream=None):
    """Run the bounded-wait failure check; afterwards kv8_workspace_error(workspace) is -7."""
    _need(workspace, "workspace", torch.uint8, 1)
    st = lib().kv8_selftest_wait_timeout(_ptr(workspace), workspace.numel(), int(limit_us),
                                         _stream(stream))
    _check("kv8_selftest_wait_timeout", st)


def mla_wuv_epilogue(o, w_uv, y=None, stream=None):
    """Per-head value projection y[b,h,:] = o[b,h,:] @ W_UV[h]; o f32 [B,H,512], w_uv bf16 [H,512,V]."""
    _need(o, "o", torch.float32, 3)
    if not (isinstance(w_uv, torch.Tensor) and _is_device(w_uv) and w_uv.dim() == 3
            and w_uv.dtype in (torch.bfloat16, torch.int16, torch.uint16)
            and w_uv.is_contiguous()):
        raise ValueError("w_uv must be a contiguous CUDA bfloat16 [H, 512, V] tensor")
    B, H, dl = o.shape
    if dl != KV8_DL or w_uv.shape[0] != H or w_uv.shape[1] != KV8_DL:
        raise ValueError("shapes must be o [B, H, 512] and w_uv [H, 512, V]")
    V = w_uv.shape[2]
    if y is None:
        y = torch.empty((B, H, V), dtype=torch.float32, device=o.device)
    _need(y, "y", torch.float32, 3)
    if tuple(y.shape) != (B, H, V):
        raise ValueError("y must be [B, H, V]")
    st = lib().mla_wuv_epilogue(_ptr(o), _ptr(w_uv), B, H, V, _ptr(y), _stream(stream))
    _check("mla_wuv_epilogue", st)
    return y


# ----------------------------------------------------------------- decode
def mla_absorb_decode_fp8_workspace_size(T: int, H: int, variant: int = KV8_DECODE_AUTO) -> int:
    n = lib().mla_absorb_decode_fp8_workspace_size(int(T), int(H), int(variant))
    if n < 0:
        raise ValueError("invalid T, H or variant")
    return int(n)


def mla_absorb_decode_fp8_batch_workspace_size(B: int, H: int, max_blocks: int,
                                               block_size: int = KV8_BLOCK,
                                               variant: int = KV8_DECODE_AUTO) -> int:
    n = lib().mla_absorb_decode_fp8_batch_workspace_size(int(B), int(H), int(max_blocks),
                                                         int(block_size), int(variant))
    if n < 0:
        raise ValueError("invalid B, H, max_blocks, block_size or variant")
    return int(n)


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def mla_absorb_decode_fp8(q_lat, q_rope, kv_codes, kv_scales, T, sm_scale, out=None, lse=None,
                          workspace=None, variant=KV8_DECODE_AUTO, stream=None):
    """One query (q_lat [H,512], q_rope [H,64]) against kv rows 0..T-1 -> out [H,512]."""
    _need(q_lat, "q_lat", torch.float32, 2)
    _need(q_rope, "q_rope", torch.float32, 2)
    _need_cache(kv_codes, kv_scales)
    H = q_lat.shape[0]
    if q_lat.shape[1] != KV8_DL or tuple(q_rope.shape) != (H, KV8_DR):
        raise ValueError("q_lat must be [H,512] and q_rope [H,64]")
    if T > kv_codes.shape[0] or T > kv_scales.shape[0]:
        raise ValueError("T exceeds the cache rows")
    if out is None:
        out = torch.empty((H, KV8_DL), dtype=torch.float32, device=q_lat.device)
    _need(out, "out", torch.float32, 2)
    if tuple(out.shape) != (H, KV8_DL):
        raise ValueError("out must be [H,512]")
    if lse is not None:
        _need(lse, "lse", torch.float32, 1)
        if lse.shape[0] != H:
            raise ValueError("lse must be [H]")
    need = mla_absorb_decode_fp8_workspace_size(T, H, variant)
    if workspace is None:
        workspace = alloc_workspace(need, q_lat.device)
    _need_workspace(workspace)
    st = lib().mla_absorb_decode_fp8(_ptr(q_lat), _ptr(q_rope), _ptr(kv_codes), _ptr(kv_scales),
                                     int(T), H, float(sm_scale), _ptr(out), _ptr(lse),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     int(variant), _stream(stream))
    _check("mla_absorb_decode_fp8", st)
    return out


def _batch_inputs(q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens, out=None, lse=None,
                  outputs=True):
    """The checks every batched decode wrapper runs: dtypes, shapes and one row per
    sequence (and of out / lse when the call writes them); returns (B, H, out), out
    allocated if None."""
    _need(q_lat, "q_lat", torch.float32, 3)
    _need(q_rope, "q_rope", torch.float32, 3)
    _need_cache(kv_codes, kv_scales)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, H = q_lat.shape[:2]
    if q_lat.shape[2] != KV8_DL or tuple(q_rope.shape) != (B, H, KV8_DR):
        raise ValueError("q_lat must be [B,H,512] and q_rope [B,H,64]")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table and seq_lens need one row per sequence")
    if not outputs:
        return B, H, None
    if out is None:
        out = torch.empty((B, H, KV8_DL), dtype=torch.float32, device=q_lat.device)
    _need(out, "out", torch.float32, 3)
    if tuple(out.shape) != (B, H, KV8_DL):
        raise ValueError("out must be [B,H,512]")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
        if tuple(lse.shape) != (B, H):
            raise ValueError("lse must be [B,H]")
    return B, H, out


def mla_absorb_decode_fp8_batch(q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens,
                                sm_scale, out=None, lse=None, workspace=None,
                                variant=KV8_DECODE_AUTO, block_size=KV8_BLOCK, stream=None):
    """B queries (q_lat [B,H,512], q_rope [B,H,64]) over a paged cache -> out [B,H,512]."""
    B, H, out = _batch_inputs(q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens, out, lse)
    max_blocks = block_table.shape[1]
    n_blocks = kv_codes.shape[0] // block_size
    need = mla_absorb_decode_fp8_batch_workspace_size(B, H, max_blocks, block_size, variant)
    if workspace is None:
        workspace = alloc_workspace(need, q_lat.device)
    _need_workspace(workspace)
    st = lib().mla_absorb_decode_fp8_batch(
        _ptr(q_lat), _ptr(q_rope), _ptr(kv_codes), _ptr(kv_scales), _ptr(block_table),
        _ptr(seq_lens), B, H, max_blocks, int(block_size), int(n_blocks), float(sm_scale),
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        int(variant), _stream(stream))
    _check("mla_absorb_decode_fp8_batch", st)
    return out


def mla_absorb_decode_fp8_batch_partials(q_lat, q_rope, kv_codes, kv_scales, block_table,
                                         seq_lens, sm_scale, workspace,
                                         variant=KV8_DECODE_AUTO, block_size=KV8_BLOCK,
                                         stream=None):
    """Split phase 1: the split-T kernel only; partials stay in ``workspace``."""
    B, H, _ = _batch_inputs(q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens,
                            outputs=False)
    _need_workspace(workspace)
    st = lib().mla_absorb_decode_fp8_batch_partials(
        _ptr(q_lat), _ptr(q_rope), _ptr(kv_codes), _ptr(kv_scales), _ptr(block_table),
        _ptr(seq_lens), B, H, block_table.shape[1], int(block_size),
        int(kv_codes.shape[0] // block_size), float(sm_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(variant), _stream(stream))
    _check("mla_absorb_decode_fp8_batch_partials", st)


def mla_absorb_decode_fp8_batch_combine(seq_lens, H, max_blocks, out, lse, workspace,
                                        variant=KV8_DECODE_AUTO, block_size=KV8_BLOCK,
                                        stream=None):
    """Split phase 2: merge the workspace partials into ``out`` / ``lse``."""
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B = seq_lens.shape[0]
    _need(out, "out", torch.float32, 3)
    if tuple(out.shape) != (B, int(H), KV8_DL):
        raise ValueError("out must be [B,H,512], B = len(seq_lens)")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
        if tuple(lse.shape) != (B, int(H)):
            raise ValueError("lse must be [B,H]")
    _need_workspace(workspace)
    st = lib().mla_absorb_decode_fp8_batch_combine(
        _ptr(seq_lens), seq_lens.shape[0], int(H), int(max_blocks), int(block_size), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), int(variant),
        _stream(stream))
    _check("mla_absorb_decode_fp8_batch_combine", st)


def kv8_workspace_error(workspace, stream=None) -> int:
    _need_workspace(workspace)
    return int(lib().kv8_workspace_error(_ptr(workspace), _stream(stream)))


def mla_absorb_decode_fp8_batch_noalloc(q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens,
                                        sm_scale, out=None, lse=None, variant=KV8_DECODE_AUTO,
                                        block_size=KV8_BLOCK, stream=None):
    """The batched decode without a caller workspace (for callers that cannot
    allocate device memory): partials go to the library's static device scratch."""
    B, H, out = _batch_inputs(q_lat, q_rope, kv_codes, kv_scales, block_table, seq_lens, out, lse)
    st = lib().mla_absorb_decode_fp8_batch_noalloc(
        _ptr(q_lat), _ptr(q_rope), _ptr(kv_codes), _ptr(kv_scales), _ptr(block_table),
        _ptr(seq_lens), B, H, block_table.shape[1], int(block_size),
        int(kv_codes.shape[0] // block_size), float(sm_scale), _ptr(out), _ptr(lse), int(variant),
        _stream(stream))
    _check("mla_absorb_decode_fp8_batch_noalloc", st)
    return out


# ----------------------------------------------------------------- cache file
class Kv8Disk:
    """An open cache file (the kv8_disk_* calls): save rows of a device cache to it,
    load them back.  Use as a context manager or call close()."""

    def __init__(self, path: str, staging_rows: int = 4096):
        h = ctypes.c_void_p()
        _check("kv8_disk_open", lib().kv8_disk_open(os.fsencode(path), int(staging_rows),
                                                    ctypes.byref(h)))
        self._h = h

    def info(self):
        """(committed rows, version)."""
        n, v = ctypes.c_int64(), ctypes.c_int()
        _check("kv8_disk_info", lib().kv8_disk_info(self._h, ctypes.byref(n), ctypes.byref(v)))
        return n.value, v.value

    def append(self, kv_codes, kv_scales, slots=None, n=None, stream=None):
        """Append the cache rows at device slots (int64 [n]) or slots 0..n-1."""
        _need(kv_codes, "kv_codes", torch.uint8, 2)
        _need(kv_scales, "kv_scales", torch.float32, 2)
        if slots is not None:
            _need(slots, "slots", torch.int64, 1)
            n = slots.numel()
        elif n is None:
            n = kv_codes.shape[0]
        _check("kv8_disk_append", lib().kv8_disk_append(self._h, _ptr(kv_codes), _ptr(kv_scales),
                                                        kv_codes.shape[0], _ptr(slots), int(n),
                                                        _stream(stream)))

    def load(self, kv_codes, kv_scales, first_row=0, n=None, dst_slot=None, stream=None):
        """Load committed rows [first_row, first_row + n) into the cache at device
        dst_slot (int64 [n]) or slots first_row + i."""
        _need(kv_codes, "kv_codes", torch.uint8, 2)
        _need(kv_scales, "kv_scales", torch.float32, 2)
        if dst_slot is not None:
            _need(dst_slot, "dst_slot", torch.int64, 1)
            n = dst_slot.numel()
        elif n is None:
            n = self.info()[0] - first_row
        _check("kv8_disk_load", lib().kv8_disk_load(self._h, int(first_row), int(n), _ptr(kv_codes),
                                                    _ptr(kv_scales), kv_codes.shape[0],
                                                    _ptr(dst_slot), _stream(stream)))

    def close(self):
        if self._h is not None and self._h.value is not None:
            _check("kv8_disk_close", lib().kv8_disk_close(self._h))
        self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
