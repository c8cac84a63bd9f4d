"""CPU oracle for the fp8 e4m3 latent KV cache and absorbed MLA decode.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product (``fp8_mla_latent_gb300``) never imports, links or runs it, and it
shares no code with the CUDA library.

The arithmetic lives in ``kv8_oracle.c`` (plain C, compiled with
``-O2 -ffp-contract=off``, no fast-math); this module only marshals numpy
arrays through ctypes.  Source of the method: the pull-request page
"KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2".

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, library routines (torch's e4m3fn cast,
torch's scaled-dot-product attention) and invariants; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv8_oracle.c")
_HDR = os.path.join(_HERE, "kv8_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DL, DR, D = 512, 64, 576


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64, i32, u32 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
            f32, f64 = ctypes.c_float, ctypes.c_double
            sig = {
                "orc_e4m3_decode": (f32, [ctypes.c_uint8]),
                "orc_e4m3_decode_table": (None, [P]),
                "orc_e4m3_encode": (ctypes.c_uint8, [f32]),
                "orc_e4m3_encode_nearest": (ctypes.c_uint8, [f32]),
                "orc_e4m3_encode_bracket": (ctypes.c_uint8, [f32]),
                "orc_e4m3_encode_array": (None, [P, i64, P, i32]),
                "orc_e4m3_exhaustive_mismatches": (i64, [ctypes.c_uint64, ctypes.c_uint64, P]),
                "orc_e4m3_list_mismatches_nearest": (i64, [P, i64, P]),
                "orc_quantize_row": (None, [P, P, P]),
                "orc_quantize_rows": (None, [P, i64, i64, P, P, P]),
                "orc_attention_f32": (None, [P, P, P, P, P, i64, i32, f32, P, P]),
                "orc_attention_f64": (None, [P, P, P, P, P, i64, i32, f64, P, P]),
                "orc_attention_heads_f64": (None, [P, P, P, P, P, i64, i32, i32, i32, f64, P, P]),
                "orc_attention_partial_f64": (None, [P, P, P, P, P, i64, i64, i32, f64, P, P, P]),
                "orc_lse_merge_f64": (None, [i32, i32, P, P, P, P, P]),
                "orc_paged_slots": (None, [P, i32, i32, i32, i64, P]),
                "orc_attention_batch_f32": (None, [P, P, P, P, P, P, i32, i32, i32, i32, f32, P, P,
                                                   i32]),
                "orc_max_threads": (i32, []),
                "orc_rmsnorm_row": (None, [P, P, f32, P]),
                "orc_rope_pairs": (None, [P, P, P, P]),
                "orc_produce_rows": (None, [P, i64, i64, P, f32, P, P, P, i64, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _ = u32
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codec
def decode_table() -> np.ndarray:
    out = np.empty(256, np.float32)
    lib().orc_e4m3_decode_table(_p(out))
    return out


def encode(x, method: str = "bitmath") -> np.ndarray:
    """Encode f32 values to e4m3 bytes (method: bitmath | nearest | bracket)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    which = {"bitmath": 0, "nearest": 1, "bracket": 2}[method]
    lib().orc_e4m3_encode_array(_p(x), x.size, _p(out), which)
    return out


def exhaustive_mismatches(lo: int, hi: int):
    first = ctypes.c_uint32(0)
    n = lib().orc_e4m3_exhaustive_mismatches(lo, hi, ctypes.byref(first))
    return int(n), int(first.value)


def list_mismatches_nearest(bits):
    bits = _c(bits, np.uint32)
    first = ctypes.c_uint32(0)
    n = lib().orc_e4m3_list_mismatches_nearest(_p(bits), bits.size, ctypes.byref(first))
    return int(n), int(first.value)


# ---------------------------------------------------------------- fused producer
def rmsnorm_row(x, weight, eps: float) -> np.ndarray:
    """RMS norm of the 512 Lc values of one row (fixed f32 order; see kv8_oracle.h)."""
    x = _c(x, np.float32)
    w = _c(weight, np.float32)
    y = np.empty(DL, np.float32)
    lib().orc_rmsnorm_row(_p(x), _p(w), float(eps), _p(y))
    return y


def rope_pairs(x, cos_row, sin_row) -> np.ndarray:
    """Rotation of the 32 Rc pairs (x[2j], x[2j+1]) by tabulated cos/sin."""
    x = _c(x, np.float32)
    y = np.empty(DR, np.float32)
    lib().orc_rope_pairs(_p(x), _p(_c(cos_row, np.float32)), _p(_c(sin_row, np.float32)), _p(y))
    return y


def produce_rows(src, norm_weight, eps, positions, rope_cos, rope_sin, dst_slot=None,
                 n_slots=None, codes=None, scales=None):
    """Fused producer: RMS norm (Lc) + rotary pairs (Rc) + quantize, into cache slots."""
    src = np.asarray(src, dtype=np.float32)
    assert src.ndim == 2 and src.shape[1] >= D and src.strides[1] == 4
    n = src.shape[0]
    stride = src.strides[0] // 4
    rope_cos = _c(rope_cos, np.float32)
    rope_sin = _c(rope_sin, np.float32)
    assert rope_cos.shape == rope_sin.shape and rope_cos.shape[1] == DR // 2
    if n_slots is None:
        n_slots = n if dst_slot is None else int(np.max(dst_slot)) + 1 if n else 0
    if codes is None:
        codes = np.zeros((n_slots, D), np.uint8)
    if scales is None:
        scales = np.zeros((n_slots, 2), np.float32)
    slots = None if dst_slot is None else _c(dst_slot, np.int64)
    lib().orc_produce_rows(src.ctypes.data_as(ctypes.c_void_p), n, stride,
                           _p(_c(norm_weight, np.float32)), float(eps),
                           _p(_c(positions, np.int64)), _p(rope_cos), _p(rope_sin),
                           rope_cos.shape[0], _p(slots), _p(codes), _p(scales))
    return codes, scales


# ---------------------------------------------------------------- W_UV epilogue
def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exactly (the upper half of an f32)."""
    bits = np.asarray(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def wuv_project(o, w_uv_bits) -> np.ndarray:
    """Per-head projection of the latent context (the step after the attention in the
    absorbed form): y[b][h][v] = sum_d o[b][h][d] * W_UV[h][d][v], in float64, with the
    bf16 weights taken exactly.  o: [B, H, 512]; w_uv_bits: uint16 [H, 512, V]."""
    o = np.asarray(o, np.float64)
    w = bf16_to_f32(w_uv_bits).astype(np.float64)
    return np.einsum("bhd,hdv->bhv", o, w)


# ---------------------------------------------------------------- prefill projection
def prefill_project(codes, scales, w_ukv_bits, slots=None) -> np.ndarray:
    """Non-absorbed path: the cached latent of T tokens, dequantized (dec(code) * sLc, as
    stored), times the up-projection W_UKV (bf16 [512, N], taken exactly), in float64:
    Y[t][n] = sLc_t * sum_d dec(Lc_t[d]) * W[d][n].  slots[t] is token t's cache slot
    (None: slot t)."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.float32)
    idx = np.arange(codes.shape[0]) if slots is None else np.asarray(slots, np.int64)
    lut = decode_table().astype(np.float64)
    lc = lut[codes[idx, :DL]] * scales[idx, 0].astype(np.float64)[:, None]
    w = bf16_to_f32(w_ukv_bits).astype(np.float64)
    return lc @ w


def prefill_rope(codes, scales, slots=None) -> np.ndarray:
    """Rope keys of the non-absorbed path: the cached Rc of each token dequantized,
    dec(Rc_t[j]) * sRc_t, the exact product (float64) rounded once to float32."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.float32)
    idx = np.arange(codes.shape[0]) if slots is None else np.asarray(slots, np.int64)
    lut = decode_table().astype(np.float64)
    return (lut[codes[idx, DL:]] * scales[idx, 1].astype(np.float64)[:, None]).astype(np.float32)


# ---------------------------------------------------------------- quantizer
def quantize_rows(src, dst_slot=None, n_slots=None, codes=None, scales=None):
    """Quantize f32 rows [n, >=576] into (codes [n_slots, 576] u8, scales [n_slots, 2] f32)."""
    src = np.asarray(src, dtype=np.float32)
    assert src.ndim == 2 and src.shape[1] >= D and src.strides[1] == 4
    n = src.shape[0]
    stride = src.strides[0] // 4
    if n_slots is None:
        n_slots = n if dst_slot is None else int(np.max(dst_slot)) + 1 if n else 0
    if codes is None:
        codes = np.zeros((n_slots, D), np.uint8)
    if scales is None:
        scales = np.zeros((n_slots, 2), np.float32)
    slots = None if dst_slot is None else _c(dst_slot, np.int64)
    lib().orc_quantize_rows(src.ctypes.data_as(ctypes.c_void_p), n, stride, _p(slots),
                            _p(codes), _p(scales))
    return codes, scales


# ---------------------------------------------------------------- attention
def _prep(q_lat, q_rope, codes, scales, slots):
    q_lat = _c(q_lat, np.float32)
    q_rope = _c(q_rope, np.float32)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    slots = None if slots is None else _c(slots, np.int64)
    return q_lat, q_rope, codes, scales, slots


def attention_f32(q_lat, q_rope, codes, scales, T, sm_scale, slots=None):
    """q_lat [H,512], q_rope [H,64] -> (out [H,512] f32, lse [H] f32)."""
    q_lat, q_rope, codes, scales, slots = _prep(q_lat, q_rope, codes, scales, slots)
    H = q_lat.shape[0]
    out = np.empty((H, DL), np.float32)
    lse = np.empty(H, np.float32)
    lib().orc_attention_f32(_p(q_lat), _p(q_rope), _p(codes), _p(scales), _p(slots), int(T), H,
                            float(sm_scale), _p(out), _p(lse))
    return out, lse


def attention_f64(q_lat, q_rope, codes, scales, T, sm_scale, slots=None, heads=None):
    """f64 twin.  heads=(h0, nh) restricts to a head range."""
    q_lat, q_rope, codes, scales, slots = _prep(q_lat, q_rope, codes, scales, slots)
    H = q_lat.shape[0]
    h0, nh = (0, H) if heads is None else heads
    out = np.empty((nh, DL), np.float64)
    lse = np.empty(nh, np.float64)
    lib().orc_attention_heads_f64(_p(q_lat), _p(q_rope), _p(codes), _p(scales), _p(slots),
                                  int(T), H, int(h0), int(nh), float(sm_scale), _p(out), _p(lse))
    return out, lse


def attention_partial_f64(q_lat, q_rope, codes, scales, t0, t1, sm_scale, slots=None):
    q_lat, q_rope, codes, scales, slots = _prep(q_lat, q_rope, codes, scales, slots)
    H = q_lat.shape[0]
    o = np.empty((H, DL), np.float64)
    m = np.empty(H, np.float64)
    l = np.empty(H, np.float64)
    lib().orc_attention_partial_f64(_p(q_lat), _p(q_rope), _p(codes), _p(scales), _p(slots),
                                    int(t0), int(t1), H, float(sm_scale), _p(o), _p(m), _p(l))
    return o, m, l


def lse_merge_f64(o_parts, m_parts, l_parts):
    o_parts = _c(o_parts, np.float64)
    m_parts = _c(m_parts, np.float64)
    l_parts = _c(l_parts, np.float64)
    S, H = m_parts.shape
    out = np.empty((H, DL), np.float64)
    lse = np.empty(H, np.float64)
    lib().orc_lse_merge_f64(S, H, _p(o_parts), _p(m_parts), _p(l_parts), _p(out), _p(lse))
    return out, lse


def paged_slots(block_table, b, T, block_size=64):
    bt = _c(block_table, np.int32)
    out = np.empty(int(T), np.int64)
    lib().orc_paged_slots(_p(bt), bt.shape[1], int(block_size), int(b), int(T), _p(out))
    return out


def attention_batch_f32(q_lat, q_rope, codes, scales, block_table, seq_lens, sm_scale,
                        block_size=64, n_threads=0):
    """q_lat [B,H,512], q_rope [B,H,64]; paged cache -> (out [B,H,512], lse [B,H])."""
    q_lat = _c(q_lat, np.float32)
    q_rope = _c(q_rope, np.float32)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    B, H = q_lat.shape[:2]
    out = np.empty((B, H, DL), np.float32)
    lse = np.empty((B, H), np.float32)
    lib().orc_attention_batch_f32(_p(q_lat), _p(q_rope), _p(codes), _p(scales), _p(bt), _p(sl),
                                  B, H, bt.shape[1], int(block_size), float(sm_scale), _p(out),
                                  _p(lse), int(n_threads))
    return out, lse


def max_threads() -> int:
    return int(lib().orc_max_threads())
