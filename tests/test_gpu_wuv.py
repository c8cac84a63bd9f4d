"""GPU W_UV epilogue parity against the float64 oracle.

The absorbed attention of the KV8 page ("KV8=1: fp8 e4m3 latent KV cache (CPU +
CUDA) with .coli_kv v2", PR description) leaves a latent context per head; the
epilogue applies each head's value projection.  Tolerance: max-abs error
<= 1e-5 * max|y| (f32 sums of 512 products against float64).
"""
import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg
import oracle

pytestmark = pytest.mark.gpu


def bf16_weights(rng, H, V):
    w = torch.from_numpy((rng.standard_normal((H, 512, V)) / np.sqrt(512)).astype(np.float32))
    return w.to(torch.bfloat16)


@pytest.mark.parametrize("B,H,V", [(1, 1, 1), (2, 128, 128), (3, 16, 128), (32, 128, 128),
                                   (17, 7, 200), (64, 128, 64), (5, 3, 513), (3, 2, 8),
                                   (33, 4, 4096), (1, 1024, 16)])
def test_wuv_matches_oracle(B, H, V):
    rng = np.random.default_rng(B * 1000 + H * 10 + V)
    d = torch.device("cuda:0")
    o = rng.standard_normal((B, H, 512)).astype(np.float32)
    w = bf16_weights(rng, H, V)
    y = pkg.mla_wuv_epilogue(torch.from_numpy(o).to(d), w.to(d))
    torch.cuda.synchronize()
    ref = oracle.wuv_project(o, w.view(torch.int16).numpy().view(np.uint16))
    err = np.abs(y.cpu().numpy() - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= 1e-5, err


def test_wuv_after_decode_output():
    """The epilogue on the decode call's own output tensor (shape and layout contract)."""
    from fp8_mla_latent_gb300 import workloads
    from gpu_helpers import decode, upload_cache
    w = workloads.make("batched", scale=0.02)
    codes, scales = upload_cache(w)
    out, _ = decode(w, codes, scales, pkg.KV8_DECODE_TCGEN05)
    rng = np.random.default_rng(2)
    wt = bf16_weights(rng, w.H, 128)
    d = torch.device("cuda:0")
    y = pkg.mla_wuv_epilogue(torch.from_numpy(out).to(d), wt.to(d))
    torch.cuda.synchronize()
    ref = oracle.wuv_project(out, wt.view(torch.int16).numpy().view(np.uint16))
    assert np.abs(y.cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()


def test_wuv_deterministic():
    """A fixed summation order: two calls give the same bits."""
    rng = np.random.default_rng(5)
    d = torch.device("cuda:0")
    o = torch.from_numpy(rng.standard_normal((9, 64, 512)).astype(np.float32)).to(d)
    w = bf16_weights(rng, 64, 136).to(d)
    y1 = pkg.mla_wuv_epilogue(o, w)
    y2 = pkg.mla_wuv_epilogue(o, w)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_wuv_weights_not_16_byte_aligned():
    """Weights 2 bytes past a 16-byte boundary take the plain path (no bulk copies)."""
    rng = np.random.default_rng(11)
    d = torch.device("cuda:0")
    B, H, V = 3, 4, 128
    o = rng.standard_normal((B, H, 512)).astype(np.float32)
    w = bf16_weights(rng, H, V)
    flat = torch.empty(H * 512 * V + 8, dtype=torch.bfloat16, device=d)
    wd = flat[1:1 + H * 512 * V].view(H, 512, V)
    wd.copy_(w.to(d))
    assert wd.data_ptr() % 16 == 2
    y = pkg.mla_wuv_epilogue(torch.from_numpy(o).to(d), wd)
    torch.cuda.synchronize()
    ref = oracle.wuv_project(o, w.view(torch.int16).numpy().view(np.uint16))
    err = np.abs(y.cpu().numpy() - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= 1e-5, err
