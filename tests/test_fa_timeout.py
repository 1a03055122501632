"""The failure path: a pipeline wait that runs out ends the kernel cleanly.

A test hook makes the producer of the first CTA skip one K tile (forward) or
one step's Q / dO tile (backward); the MMA warp's bounded wait for it gives
up after a short limit, every role drains and leaves -- in the backward still
meeting each of its named barriers, as bar.sync after the abort -- and the
host reads FA_ERR_TIMEOUT from the device status word.  No fault, trap or
hang is involved.  The context stays usable: the next launch without the hook
is correct.
"""
import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa
import oracle
from io_aware_attention_gb300.workloads import make_random_qkv

from _parity import assert_close
from test_bwd import check_heads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
def test_wait_timeout_is_reported_and_recoverable(causal):
    q, k, v = make_random_qkv(1, 2, 640, 128, seed=21)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert fa.check_device_status() == 0
    fa.set_wait_limit_ns(20_000_000)  # 20 ms
    fa.debug_skip_k_tile(1)
    try:
        fa.fwd(qd, kd, vd, causal=causal)
        torch.cuda.synchronize()
        assert fa.check_device_status() == 4  # FA_ERR_TIMEOUT
    finally:
        fa.debug_skip_k_tile(-1)
        fa.set_wait_limit_ns(0)
    # the status was cleared and the device works
    assert fa.check_device_status() == 0
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    o_ref, lse_ref = oracle.attention(q, k, v, causal, 1.0 / np.sqrt(128))
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "after timeout")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tile", [0, 1])
def test_bwd_wait_timeout_is_reported_and_recoverable(causal, tile):
    B, H, N, d = 1, 2, 640, 128
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, seed=22))
    do = make_random_qkv(B, H, N, d, seed=23)[0].cuda()
    scale = d ** -0.5
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    fa.set_wait_limit_ns(20_000_000)  # 20 ms
    fa.debug_skip_k_tile(tile)
    try:
        fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert fa.check_device_status() == 4  # FA_ERR_TIMEOUT
    finally:
        fa.debug_skip_k_tile(-1)
        fa.set_wait_limit_ns(0)
    assert fa.check_device_status() == 0
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    check_heads(q, k, v, do, causal, scale, dq, dk, dv, range(B * H), "after timeout")


def test_get_device_status_reports_and_clears():
    """fa_get_device_status, the short form: FA_ERR_TIMEOUT once, then FA_OK."""
    q, k, v = (t.cuda() for t in make_random_qkv(1, 2, 640, 128, seed=24))
    assert fa.get_device_status() == 0
    fa.set_wait_limit_ns(20_000_000)  # 20 ms
    fa.debug_skip_k_tile(1)
    try:
        fa.fwd(q, k, v, causal=False)
        assert fa.get_device_status() == 4  # FA_ERR_TIMEOUT
    finally:
        fa.debug_skip_k_tile(-1)
        fa.set_wait_limit_ns(0)
    assert fa.get_device_status() == 0
    fa.fwd(q, k, v, causal=False)
    assert fa.get_device_status() == 0
