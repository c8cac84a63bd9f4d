"""Seeded synthetic inputs for the fp8 latent-KV MLA decode workloads.

This module only draws random numbers and lays out index tables; it holds none
of the method's arithmetic (no quantization, no attention), so both the CUDA
path and the CPU oracle can be fed from it.

Workloads (DeepSeek-V3-style MLA: kv_lora 512, qk_rope 64, softmax scale
1/sqrt(192) for every workload -- our reading, the source pages give no value):

  tiny      B=1,  H=4,   T=256              rows N(0,1), q N(0,1)               seed 0
  single    B=1,  H=128, T=4096             rows N(0,1) * g_c, g_c = exp(0.5 N(0,1)) per channel
  batched   B=32, H=128, T_b ~ U{1024..32768}, paged in 64-token blocks (random block
            permutation of one pool); values as "single"                          seed 2
  long      B=2,  H=128, T=262144 each; rows N(0,1) with each element x20 w.p. 0.001 seed 3
  append    65536 fresh rows (Student-t nu=3; 1% all-zero rows; 1% rows rescaled so
            amax lies in the f32 subnormal range; 0.1% NaN entries) appended 1024 per
            sequence after 7168 cached rows of the same kind; then decode B=64, H=16,
            T=8192, paged                                                       seed 4

``scale`` < 1 shrinks token counts (never below one 64-token block plus a ragged
tail) for parity tests that the oracle must finish in seconds.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

DL, DR, D = 512, 64, 576
BLOCK = 64
SM_SCALE = 1.0 / math.sqrt(192.0)

WORKLOADS = ("tiny", "single", "batched", "long", "append")


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    H: int
    seq_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, max_blocks]; physical block ids
    n_slots: int                  # rows in the cache pool (multiple of 64)
    cache_rows: np.ndarray        # f32 [n_cache, 576] rows written before the step
    cache_slots: np.ndarray       # int64 [n_cache] their slots
    fresh_rows: np.ndarray | None  # f32 [n_fresh, 576] rows appended inside the step
    fresh_slots: np.ndarray | None
    q_lat: np.ndarray             # f32 [B, H, 512]
    q_rope: np.ndarray            # f32 [B, H, 64]
    sm_scale: float = SM_SCALE
    contiguous: bool = False      # single sequence stored at slots 0..T-1

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def kv_bytes(self) -> int:
        return self.total_tokens * (D + 8)


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def _channel_gain(rng):
    return np.exp(0.5 * rng.standard_normal(D)).astype(np.float32)


def _paged_tables(rng, seq_lens, shuffle=True):
    nb = [(int(t) + BLOCK - 1) // BLOCK for t in seq_lens]
    total = sum(nb)
    max_blocks = max(max(nb), 1)
    phys = rng.permutation(total).astype(np.int32) if shuffle else np.arange(total, dtype=np.int32)
    bt = np.zeros((len(seq_lens), max_blocks), np.int32)
    slots = []
    k = 0
    for b, n in enumerate(nb):
        bt[b, :n] = phys[k:k + n]
        k += n
        t = np.arange(int(seq_lens[b]), dtype=np.int64)
        slots.append(bt[b, t // BLOCK].astype(np.int64) * BLOCK + t % BLOCK)
    return bt, max(total, 1) * BLOCK, (np.concatenate(slots) if slots else np.zeros(0, np.int64))


def _append_rows(rng, n):
    """Student-t(3) rows with the special rows of the append workload."""
    x = rng.standard_t(3, size=(n, D)).astype(np.float32)
    kind = rng.random(n)
    zero = kind < 0.01
    sub = (kind >= 0.01) & (kind < 0.02)
    x[zero] = 0.0
    if sub.any():
        # target amax uniform in log2 over [2^-149, 2^-126): scale each row so its amax lands there
        e = rng.uniform(-149.0, -126.0, size=int(sub.sum()))
        amax = np.abs(x[sub]).max(1)
        with np.errstate(over="ignore", under="ignore"):
            f = (np.exp2(e) / amax.astype(np.float64))
            x[sub] = (x[sub].astype(np.float64) * f[:, None]).astype(np.float32)
    nan = rng.random((n, D)) < 0.001
    x[nan] = np.nan
    return x


def make(name: str, scale: float = 1.0, seed: int | None = None) -> Workload:
    """Build a workload.  ``scale`` shrinks token counts for small parity cases."""
    seeds = {"tiny": 0, "single": 1, "batched": 2, "long": 3, "append": 4}
    rng = np.random.default_rng(seeds[name] if seed is None else seed)

    def sz(t, lo=BLOCK + 17):
        return t if scale >= 1.0 else max(lo, int(t * scale))

    if name in ("tiny", "single"):
        B, H = 1, (4 if name == "tiny" else 128)
        T = sz(256 if name == "tiny" else 4096)
        rows = _normal(rng, (T, D))
        if name == "single":
            rows *= _channel_gain(rng)
        seq = np.array([T], np.int32)
        nblk = (T + BLOCK - 1) // BLOCK
        bt = np.arange(nblk, dtype=np.int32)[None]
        q = _normal(rng, (B, H, D))
        return Workload(name, B, H, seq, bt, nblk * BLOCK, rows, np.arange(T, dtype=np.int64),
                        None, None, np.ascontiguousarray(q[..., :DL]),
                        np.ascontiguousarray(q[..., DL:]), contiguous=True)

    if name == "batched":
        B, H = 32, 128
        lo, hi = sz(1024), sz(32768, lo=2 * BLOCK + 17)
        seq = rng.integers(lo, hi + 1, size=B).astype(np.int32)
        gain = _channel_gain(rng)
        bt, n_slots, slots = _paged_tables(rng, seq)
        rows = _normal(rng, (slots.size, D)) * gain
        q = _normal(rng, (B, H, D))
        return Workload(name, B, H, seq, bt, n_slots, rows, slots, None, None,
                        np.ascontiguousarray(q[..., :DL]), np.ascontiguousarray(q[..., DL:]))

    if name == "long":
        B, H = 2, 128
        T = sz(262144)
        seq = np.full(B, T, np.int32)
        bt, n_slots, slots = _paged_tables(rng, seq, shuffle=False)  # each sequence contiguous
        rows = _normal(rng, (slots.size, D))
        out = rng.random(rows.shape) < 0.001
        rows[out] *= 20.0
        q = _normal(rng, (B, H, D))
        return Workload(name, B, H, seq, bt, n_slots, rows, slots, None, None,
                        np.ascontiguousarray(q[..., :DL]), np.ascontiguousarray(q[..., DL:]))

    if name == "append":
        B, H = 64, 16
        T = sz(8192, lo=2 * BLOCK + 17)
        fresh_per = max(1, T // 8)        # 1024 of 8192 at full size
        cached = T - fresh_per
        seq = np.full(B, T, np.int32)
        bt, n_slots, slots = _paged_tables(rng, seq)
        slots = slots.reshape(B, T)
        cache_slots = slots[:, :cached].reshape(-1)
        fresh_slots = slots[:, cached:].reshape(-1)
        cache_rows = _append_rows(rng, cache_slots.size)
        fresh_rows = _append_rows(rng, fresh_slots.size)
        q = _normal(rng, (B, H, D))
        return Workload(name, B, H, seq, bt, n_slots, cache_rows, cache_slots, fresh_rows,
                        fresh_slots, np.ascontiguousarray(q[..., :DL]),
                        np.ascontiguousarray(q[..., DL:]))

    raise ValueError(f"unknown workload {name!r}; choose from {WORKLOADS}")


@dataclasses.dataclass
class ProducerInputs:
    """Raw rows for the fused producer, with its tables (all seeded inputs)."""
    rows: np.ndarray        # f32 [n, 576]: pre-norm Lc, pre-rotation Rc
    weight: np.ndarray      # f32 [512] norm weight
    eps: float
    positions: np.ndarray   # int64 [n]
    rope_cos: np.ndarray    # f32 [max_pos, 32]
    rope_sin: np.ndarray    # f32 [max_pos, 32]
    slots: np.ndarray       # int64 [n]: distinct cache slots
    n_slots: int


def producer_inputs(n: int, max_pos: int = 16384, seed: int = 4, base: float = 10000.0,
                    eps: float = 1e-6) -> ProducerInputs:
    """Rows of the append workload's value mix (Student-t nu=3, 1% zero rows, 1%
    subnormal-amax rows, 0.1% NaN entries) before normalisation and rotation; a
    norm weight around 1; positions uniform in [0, max_pos); the rotation tables
    cos/sin(pos * base^(-j/32)) for the 32 pairs, computed in float64 and
    rounded to f32 (the caller's rope cache); slots a random injective map into a
    pool twice the size."""
    rng = np.random.default_rng(seed)
    rows = _append_rows(rng, n)
    weight = (1.0 + 0.1 * rng.standard_normal(DL)).astype(np.float32)
    positions = rng.integers(0, max_pos, n).astype(np.int64)
    ang = np.outer(np.arange(max_pos, dtype=np.float64), base ** (-np.arange(DR // 2) / (DR // 2)))
    n_slots = 2 * n
    slots = rng.permutation(n_slots)[:n].astype(np.int64)
    return ProducerInputs(rows, weight, eps, positions, np.cos(ang).astype(np.float32),
                          np.sin(ang).astype(np.float32), slots, n_slots)


@dataclasses.dataclass
class PrefillInputs:
    rows: np.ndarray        # f32 [T, 576]: latent rows to quantize into the cache
    slots: np.ndarray       # int64 [T]: cache slot of token t (a permutation of a pool)
    n_slots: int
    w_ukv: np.ndarray       # f32 [512, N]: up-projection weights (rounded to bf16 by the caller)


def prefill_inputs(T: int = 4096, N: int = 32768, seed: int = 11) -> PrefillInputs:
    """One prompt chunk of T tokens in a pool of T + 1024 slots (random injective map,
    as pages hand out slots), rows with the decode workloads' per-channel spread
    (Gaussian times a log-normal channel gain), and kv_b weights N(0, 1/512):
    N = 128 heads x (128 qk_nope + 128 v_head)."""
    rng = np.random.default_rng(seed)
    gain = np.exp(0.5 * rng.standard_normal(D))
    rows = (rng.standard_normal((T, D)) * gain).astype(np.float32)
    n_slots = T + 1024
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    w = (rng.standard_normal((DL, N)) / math.sqrt(DL)).astype(np.float32)
    return PrefillInputs(rows, slots, n_slots, w)
