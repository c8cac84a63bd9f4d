"""The device-side failure path, exercised without a GPU fault.

The decode pipelines wait on mbarriers with a time limit; a wait that runs out
must flag the workspace error word (KV8_ETIMEOUT) and return, leaving the
context usable.  The self-test makes such a wait run out (a barrier nothing
arrives at) with a short limit.
"""
import time

import numpy as np
import pytest
import torch

import fp8_mla_latent_gb300 as pkg

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    d = torch.device("cuda:0")
    ws = pkg.alloc_workspace(256, d)
    t0 = time.time()
    pkg.kv8_selftest_wait_timeout(ws, 5000)   # 5 ms
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert pkg.kv8_workspace_error(ws) == -7
    assert 0.004 <= dt < 2.0
    # the context still runs work: a small decode gives finite results and a clean error word
    q = torch.randn((16, 512), device=d)
    r = torch.randn((16, 64), device=d)
    codes = torch.zeros((256, 576), dtype=torch.uint8, device=d)
    scales = torch.zeros((256, 2), device=d)
    rows = torch.randn((256, 576), device=d)
    pkg.kv8_quantize_rows(rows, codes, scales)
    ws2 = pkg.alloc_workspace(pkg.mla_absorb_decode_fp8_workspace_size(256, 16), d)
    out = pkg.mla_absorb_decode_fp8(q, r, codes, scales, 256, 0.07, workspace=ws2)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert pkg.kv8_workspace_error(ws2) == 0
