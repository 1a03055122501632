"""Shared helpers for the GPU parity tests (comparison and tolerances).

Tolerances for bf16 inputs with fp32 accumulation, against the fp64 oracle:
max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3.
"""
import numpy as np
import torch

import io_aware_attention_gb300 as fa

MAX_DO = 1e-2
MEAN_DO = 1e-3
MAX_DLSE = 1e-3
GUARD = 64  # elements of canary on each side of every output


def assert_close(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, np.float64)
    lse = np.asarray(lse, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    assert np.isfinite(lse).all(), f"{what}: non-finite LSE"
    do = np.abs(o - o_ref)
    dl = np.abs(lse - lse_ref)
    worst = np.unravel_index(np.argmax(do), do.shape)
    msg = (f"{what}: max|dO|={do.max():.3e} at {tuple(int(i) for i in worst)} "
           f"(|O_ref|={abs(o_ref[worst]):.3f}) mean|dO|={do.mean():.3e} "
           f"max|dLSE|={dl.max():.3e} at {np.unravel_index(np.argmax(dl), dl.shape)}")
    assert do.max() <= MAX_DO and do.mean() <= MEAN_DO and dl.max() <= MAX_DLSE, msg
    return do.max(), do.mean(), dl.max()


def run_guarded(q, k, v, causal, scale, stream=None):
    """fa.fwd_into with NaN-filled outputs surrounded by canary bands; checks
    that every output element was written and nothing outside was touched."""
    B, H, N, d = q.shape
    no, nl = B * H * N * d, B * H * N
    obuf = torch.full((no + 2 * GUARD,), float("nan"), dtype=torch.bfloat16, device=q.device)
    obuf.view(torch.int16)[:GUARD] = 0x7FC1  # a NaN payload the kernel never produces
    obuf.view(torch.int16)[-GUARD:] = 0x7FC1
    lbuf = torch.full((nl + 2 * GUARD,), float("nan"), dtype=torch.float32, device=q.device)
    lbuf[:GUARD] = -12345.0
    lbuf[-GUARD:] = -12345.0
    o = obuf[GUARD:GUARD + no].view(B, H, N, d)
    lse = lbuf[GUARD:GUARD + nl].view(B, H, N)
    fa.fwd_into(q, k, v, o, lse, causal, scale, stream)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0, "a kernel wait timed out"
    ob = obuf.view(torch.int16).cpu()
    assert (ob[:GUARD] == 0x7FC1).all() and (ob[-GUARD:] == 0x7FC1).all(), "O guard band overwritten"
    lb = lbuf.cpu()
    assert (lb[:GUARD] == -12345.0).all() and (lb[-GUARD:] == -12345.0).all(), "LSE guard overwritten"
    return o, lse
