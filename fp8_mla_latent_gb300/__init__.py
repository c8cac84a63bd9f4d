"""fp8 e4m3 latent-KV absorbed MLA decode for one GB300 (sm_103a).

The product is the C-ABI library ``libfp8mla.so`` (sources in ``csrc/``, calls
declared in ``include/fp8mla.h``); this package holds its in-tree build step
(``build``), a ctypes binding with the same call names (``_lib``) and the seeded
synthetic workloads (``workloads``).
"""
from ._lib import (KV8_BLOCK, KV8_D, KV8_DECODE_AUTO, KV8_DECODE_SIMT, KV8_DECODE_TCGEN05,
                   KV8_DECODE_TCGEN05_CTA, KV8_DECODE_TCGEN05_PAIR,
                   KV8_DL, KV8_DR, Kv8Disk, Kv8Error, alloc_workspace, kv8_prefill_project, kv8_produce_rows, kv8_quantize_rows,
                   kv8_selftest_wait_timeout,
                   kv8_workspace_error, lib, library_path, mla_absorb_decode_fp8,
                   mla_absorb_decode_fp8_batch, mla_absorb_decode_fp8_batch_combine,
                   mla_absorb_decode_fp8_batch_noalloc, mla_absorb_decode_fp8_batch_partials,
                   mla_absorb_decode_fp8_batch_workspace_size,
                   mla_absorb_decode_fp8_workspace_size, mla_wuv_epilogue)

__all__ = [
    "KV8_BLOCK", "KV8_D", "KV8_DECODE_AUTO", "KV8_DECODE_SIMT", "KV8_DECODE_TCGEN05",
    "KV8_DECODE_TCGEN05_CTA", "KV8_DECODE_TCGEN05_PAIR", "KV8_DL",
    "KV8_DR", "Kv8Disk", "Kv8Error", "alloc_workspace", "kv8_prefill_project", "kv8_produce_rows", "kv8_quantize_rows",
    "kv8_selftest_wait_timeout", "kv8_workspace_error", "lib",
    "library_path", "mla_absorb_decode_fp8", "mla_absorb_decode_fp8_batch",
    "mla_absorb_decode_fp8_batch_combine", "mla_absorb_decode_fp8_batch_noalloc",
    "mla_absorb_decode_fp8_batch_partials",
    "mla_absorb_decode_fp8_batch_workspace_size", "mla_absorb_decode_fp8_workspace_size",
    "mla_wuv_epilogue",
]
