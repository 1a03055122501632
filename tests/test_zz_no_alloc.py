"""fa_decode_static: decode with the library's static scratch array, no
allocation anywhere in the call.

The file name sorts last, so in a full run these tests come after every
other test of the session; they also pass alone in a fresh process (the
first call on the device then does the scratch address lookup).
"""
import ctypes

import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa

from _parity import MAX_DLSE, MAX_DO, MEAN_DO

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 8 << 20  # FA_DECODE_STATIC_SCRATCH_BYTES in include/fa.h


def call_static(q, k, v, o, lse, causal, scale):
    B, H, Nq, d = (int(s) for s in q.shape)
    Nk = int(k.shape[2])
    vp = ctypes.c_void_p
    return fa.library().fa_decode_static(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
                                         vp(lse.data_ptr()), B, H, Nq, Nk, d, int(bool(causal)), float(scale),
                                         vp(torch.cuda.current_stream().cuda_stream))


def rand(B, H, Nq, Nk, d, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16).cuda()
    k = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16).cuda()
    return q, k, v


@pytest.mark.parametrize("B, H, Nq, Nk, d, causal", [
    (1, 2, 1, 20000, 128, False),   # one head over many chunks
    (2, 3, 4, 3000, 64, True),
    (8, 32, 1, 32768, 128, False),  # the decode bench workload's shape
])
def test_static_scratch_matches_the_workspace_entry_twice(B, H, Nq, Nk, d, causal):
    q, k, v = rand(B, H, Nq, Nk, d, seed=B + H + Nq + Nk + d)
    scale = 1.0 / np.sqrt(d)
    # These sizes split the key range, so the scratch is really used.
    assert 0 < fa.decode_workspace_bytes(B, H, Nq, Nk, d, causal) <= STATIC_SCRATCH_BYTES
    o_ref, lse_ref = fa.decode(q, k, v, causal=causal, scale=scale)
    for _ in range(2):  # two calls in a row on the same scratch
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
        assert call_static(q, k, v, o, lse, causal, scale) == 0
        torch.cuda.synchronize()
        assert fa.check_device_status() == 0
        do = (o.float() - o_ref.float()).abs()
        assert torch.isfinite(do).all()
        assert do.max().item() <= MAX_DO and do.mean().item() <= MEAN_DO
        assert (lse - lse_ref).abs().max().item() <= MAX_DLSE


def test_sizes_beyond_the_static_scratch_are_refused():
    B, H, Nq, Nk, d = 10, 100, 8, 4096, 128  # at least 11.8 MB of partial results at any occupancy
    need = fa.decode_workspace_bytes(B, H, Nq, Nk, d, False)
    if need <= STATIC_SCRATCH_BYTES:
        pytest.skip("this device's split plan fits these sizes into the static scratch")
    q = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, H, Nk, d), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    assert call_static(q, k, v, o, lse, False, 0.088) == 5  # FA_ERR_TOO_LARGE, nothing enqueued
    assert fa.STATUS[5] == "FA_ERR_TOO_LARGE"
