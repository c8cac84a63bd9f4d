"""The no-allocation decode entry point, called through the C ABI.

Some callers cannot allocate device memory (a host runtime that owns every
buffer and hands the library only inputs and outputs, or a loop whose memory
budget is fixed in advance), so they cannot pass a workspace.
mla_absorb_decode_fp8_batch_noalloc serves them from a static device scratch
array.  This test checks that two calls in a row give what the workspace call
gives, bit for bit (both run the same kernels on the same split plan), and
that a problem too large for the scratch is refused.  It lives in its own file so pytest collects
it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
from fp8_mla_latent_gb300 import workloads

from gpu_helpers import upload_cache

pytestmark = pytest.mark.gpu

ESCRATCH = -8


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


@pytest.mark.parametrize("variant", [pkg.KV8_DECODE_SIMT, pkg.KV8_DECODE_TCGEN05_CTA,
                                     pkg.KV8_DECODE_TCGEN05_PAIR])
def test_noalloc_matches_workspace_call_twice(variant):
    d = torch.device("cuda:0")
    w = workloads.make("batched", scale=0.02)
    codes, scales = upload_cache(w)
    ql = torch.from_numpy(w.q_lat).to(d)
    qr = torch.from_numpy(w.q_rope).to(d)
    bt = torch.from_numpy(w.block_table).to(d)
    sl = torch.from_numpy(w.seq_lens).to(d)
    ref_lse = torch.empty((w.B, w.H), device=d)
    ref = pkg.mla_absorb_decode_fp8_batch(ql, qr, codes, scales, bt, sl, w.sm_scale, lse=ref_lse,
                                          variant=variant)
    torch.cuda.synchronize()
    ref_np, ref_lse_np = ref.cpu().numpy(), ref_lse.cpu().numpy()
    L = pkg.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full((w.B, w.H, 512), float("nan"), device=d)
        lse = torch.full((w.B, w.H), float("nan"), device=d)
        st = L.mla_absorb_decode_fp8_batch_noalloc(
            _p(ql), _p(qr), _p(codes), _p(scales), _p(bt), _p(sl), w.B, w.H, w.max_blocks, 64,
            codes.shape[0] // 64, w.sm_scale, _p(out), _p(lse), variant, stream)
        assert st == 0, f"call {call}: status {st}"
        assert L.kv8_noalloc_error(stream) == 0
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref_np.view(np.uint32)), call
        assert np.array_equal(lse.cpu().numpy().view(np.uint32), ref_lse_np.view(np.uint32)), call


def test_noalloc_refuses_problems_larger_than_its_scratch():
    d = torch.device("cuda:0")
    B, H, max_blocks = 256, 128, 64  # one split per sequence: 67 MB of partials, beyond 32 MiB
    need = pkg.mla_absorb_decode_fp8_batch_workspace_size(B, H, max_blocks)
    assert need > (32 << 20)
    q = torch.zeros((B, H, 512), device=d)
    r = torch.zeros((B, H, 64), device=d)
    codes = torch.zeros((64, 576), dtype=torch.uint8, device=d)
    scales = torch.zeros((64, 2), device=d)
    bt = torch.zeros((B, max_blocks), dtype=torch.int32, device=d)
    sl = torch.zeros((B,), dtype=torch.int32, device=d)
    out = torch.zeros((B, H, 512), device=d)
    st = pkg.lib().mla_absorb_decode_fp8_batch_noalloc(
        _p(q), _p(r), _p(codes), _p(scales), _p(bt), _p(sl), B, H, max_blocks, 64, 1, 0.1,
        _p(out), None, pkg.KV8_DECODE_AUTO, None)
    assert st == ESCRATCH
    with pytest.raises(pkg.Kv8Error):
        pkg.mla_absorb_decode_fp8_batch_noalloc(q, r, codes, scales, bt, sl, 0.1, out=out)
