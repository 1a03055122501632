"""Head sizes other than 64 and 128 (multiples of 8 up to 128) on the GPU.

They run in the 64- or 128-column kernels with the columns past d read as
zeros by the TMA loads; only d columns are written.  Forward outputs are
compared with the fp64 oracle within the forward tolerances, gradients
within the backward's rounding bound (see test_bwd.py), with canary bands
around every output so that a write past the d columns or with the padded
row stride shows.
"""
import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa
import oracle
from _parity import assert_close, run_guarded
from io_aware_attention_gb300.workloads import make_random_qkv
from test_bwd import check_heads, run_bwd

pytestmark = pytest.mark.gpu

FWD_CASES = [  # (B, H, N, d, causal)
    (1, 2, 200, 8, True), (1, 2, 256, 32, False), (2, 2, 130, 40, True), (1, 2, 300, 56, False),
    (1, 2, 257, 80, True), (2, 1, 384, 96, False), (1, 2, 129, 112, True), (1, 1, 1, 24, True),
]


@pytest.mark.parametrize("B,H,N,d,causal", FWD_CASES,
                         ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in FWD_CASES])
def test_fwd_padded_head_sizes(B, H, N, d, causal):
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 12000 + N + d))
    scale = d ** -0.5
    o, lse = run_guarded(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"d={d} N={N} causal={causal}")


BWD_CASES = [  # (B, H, N, d, causal)
    (1, 2, 256, 32, True), (1, 2, 200, 40, False), (2, 1, 333, 80, True), (1, 2, 256, 96, False),
    (1, 1, 130, 112, True), (1, 1, 1, 8, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", BWD_CASES,
                         ids=[f"b{b}h{h}n{n}d{d}{'c' if c else ''}" for b, h, n, d, c in BWD_CASES])
def test_bwd_padded_head_sizes(B, H, N, d, causal):
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 13000 + N + d))
    do = make_random_qkv(B, H, N, d, 13500 + N + d)[0].cuda()
    scale = d ** -0.5
    dq, dk, dv = run_bwd(q, k, v, do, causal, scale)
    check_heads(q, k, v, do, causal, scale, dq, dk, dv, range(B * H), f"d={d} N={N} causal={causal}")


def test_padded_matches_explicit_zero_padding():
    """d = 96 equals d = 128 with the last 32 columns of q, k, v zero (and
    the scale kept): the padding is exact, so O agrees to the bit on the
    first 96 columns and the padded columns of the d = 128 run are zero."""
    B, H, N, d = 1, 2, 300, 96
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 14001))
    pad = lambda t: torch.nn.functional.pad(t, (0, 128 - d)).contiguous()
    for causal in (False, True):
        o96, l96 = fa.fwd(q, k, v, causal=causal, scale=d ** -0.5)
        o128, l128 = fa.fwd(pad(q), pad(k), pad(v), causal=causal, scale=d ** -0.5)
        torch.cuda.synchronize()
        assert torch.equal(o96, o128[..., :d].contiguous())
        assert torch.equal(l96, l128)
        assert (o128[..., d:] == 0).all()
