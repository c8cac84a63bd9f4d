"""CPU oracle of the fp8 cache file (save / resume), written out in plain Python.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: only the tests, ``smoke()``
and ``bench.py``'s baseline legs use it, and it shares no code with the library.

KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU + CUDA) with .coli_kv v2"), PR
description, persistence item: the cache file of version 2 starts with the magic
``COLIKV2`` and records its data type in the header; its rows are the fp8 codes
with their scales (about 46 KB per token over all layers, i.e. 584 B per token
per layer); rows are appended through a persistent handle; a version-1 file
(f32 rows) is quantized on resume and rewritten as version 2 at the first
append; opening a file repairs a damaged magic.  The page gives no byte layout,
so the layout below is this project's definition (the library's header states
the same one):

  header, 64 bytes, little-endian:
    [0, 8)   magic  b"COLIKV2\\0" (version 2) or b"COLIKV1\\0" (version 1)
    [8, 12)  u32    header bytes = 64
    [12, 16) u32    data type: 2 = e4m3 codes + two f32 scales, 1 = f32 values
    [16, 20) u32    values per row = 576 (Lc 512, then Rc 64)
    [20, 24) u32    bytes per record: 584 (version 2) or 2304 (version 1)
    [24, 32) u64    rows committed
    [32, 64)        zero
  then `rows committed` records: version 2: the 576 code bytes, then sLc and sRc
  (f32); version 1: 576 f32 values.  Bytes past the last committed record (a torn
  append) are not part of the file's contents.
"""
from __future__ import annotations

import struct

import numpy as np

HEADER_BYTES = 64
D = 576
MAGIC = {2: b"COLIKV2\0", 1: b"COLIKV1\0"}
DTYPE = {2: 2, 1: 1}
RECORD = {2: D + 8, 1: D * 4}


def header(version: int, n_rows: int) -> bytes:
    """The 64 header bytes of a file of the given version holding n_rows rows."""
    h = MAGIC[version] + struct.pack("<IIIIQ", HEADER_BYTES, DTYPE[version], D, RECORD[version],
                                     n_rows)
    return h + bytes(HEADER_BYTES - len(h))


def parse_header(raw: bytes):
    """(version, n_rows) of a header, or None when the bytes are not one."""
    if len(raw) < HEADER_BYTES:
        return None
    magic = raw[:8]
    version = {v: k for k, v in MAGIC.items()}.get(magic)
    if version is None:
        return None
    hb, dt, d, rec, n = struct.unpack("<IIIIQ", raw[8:32])
    if hb != HEADER_BYTES or dt != DTYPE[version] or d != D or rec != RECORD[version]:
        return None
    return version, n


def records_v2(codes: np.ndarray, scales: np.ndarray) -> bytes:
    """Version-2 records of rows: codes u8 [n, 576], scales f32 [n, 2]."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, "<f4")
    n = codes.shape[0]
    rec = np.zeros((n, RECORD[2]), np.uint8)
    rec[:, :D] = codes
    rec[:, D:] = scales.view(np.uint8).reshape(n, 8)
    return rec.tobytes()


def write_v2(path: str, codes: np.ndarray, scales: np.ndarray) -> None:
    with open(path, "wb") as f:
        f.write(header(2, codes.shape[0]))
        f.write(records_v2(codes, scales))


def write_v1(path: str, rows: np.ndarray) -> None:
    rows = np.ascontiguousarray(rows, "<f4")
    assert rows.ndim == 2 and rows.shape[1] == D
    with open(path, "wb") as f:
        f.write(header(1, rows.shape[0]))
        f.write(rows.tobytes())


def read(path: str):
    """The committed contents of a file: (2, codes [n, 576] u8, scales [n, 2] f32) or
    (1, rows [n, 576] f32, None); None when the file has no valid header."""
    with open(path, "rb") as f:
        raw = f.read()
    h = parse_header(raw)
    if h is None:
        return None
    version, n = h
    body = raw[HEADER_BYTES:HEADER_BYTES + n * RECORD[version]]
    assert len(body) == n * RECORD[version], "file shorter than its committed rows"
    if version == 2:
        rec = np.frombuffer(body, np.uint8).reshape(n, RECORD[2])
        return 2, rec[:, :D].copy(), rec[:, D:].copy().view("<f4").reshape(n, 2).astype(np.float32)
    return 1, np.frombuffer(body, "<f4").reshape(n, D).astype(np.float32), None
