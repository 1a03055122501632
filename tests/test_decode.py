"""Decode attention (fa_decode): a few query rows against a long KV cache.

Parity with the fp64 oracle on the same seeded inputs, element by element,
over head sizes, query counts, cache lengths that are not multiples of the
kernel's rounds (ragged tails, a single key), both masks, and split and
unsplit key ranges; the full-size cache on sampled rows plus properties that
hold at any size.  Cross-check: causal decode of the last Nq rows equals the
forward kernel's last Nq rows.
"""
import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa
import oracle
from io_aware_attention_gb300.workloads import (DECODE_WORKLOADS, make_decode_qkv, make_random_qkv,
                                                sample_decode_rows)

from _parity import GUARD, MAX_DLSE, MAX_DO, MEAN_DO, assert_close

pytestmark = pytest.mark.gpu


def rand(B, H, Nq, Nk, d, seed, q_mult=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    q = (torch.randn((B, H, Nq, d), generator=g) * q_mult).to(torch.bfloat16)
    k = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H, Nk, d), generator=g).to(torch.bfloat16)
    return q, k, v


def run_guarded(q, k, v, causal, scale):
    """fa.decode_into with NaN-filled outputs inside canary bands."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    no, nl = B * H * Nq * d, B * H * Nq
    obuf = torch.full((no + 2 * GUARD,), float("nan"), dtype=torch.bfloat16, device="cuda")
    obuf.view(torch.int16)[:GUARD] = 0x7FC1
    obuf.view(torch.int16)[-GUARD:] = 0x7FC1
    lbuf = torch.full((nl + 2 * GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    lbuf[:GUARD] = -12345.0
    lbuf[-GUARD:] = -12345.0
    o = obuf[GUARD:GUARD + no].view(B, H, Nq, d)
    lse = lbuf[GUARD:GUARD + nl].view(B, H, Nq)
    nbytes = fa.decode_workspace_bytes(B, H, Nq, Nk, d, causal)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda") if nbytes else None
    fa.decode_into(q, k, v, o, lse, ws, causal, scale)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    ob = obuf.view(torch.int16).cpu()
    assert (ob[:GUARD] == 0x7FC1).all() and (ob[-GUARD:] == 0x7FC1).all(), "O guard band overwritten"
    lb = lbuf.cpu()
    assert (lb[:GUARD] == -12345.0).all() and (lb[-GUARD:] == -12345.0).all(), "LSE guard overwritten"
    return o, lse, nbytes


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("nk", [1, 17, 128, 129, 1000, 4097, 20000])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_matches_oracle(d, nq, nk, causal):
    if causal and nq > nk:
        pytest.skip("the causal window needs Nq <= Nk")
    q, k, v = rand(2, 3, nq, nk, d, seed=nq * 1000 + nk + d + int(causal))
    scale = 1.0 / np.sqrt(d)
    o, lse, _ = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    o_ref, lse_ref = oracle.attention_rect(q, k, v, causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"d{d} nq{nq} nk{nk} c{int(causal)}")


@pytest.mark.parametrize("d", [8, 40, 80, 96, 112])
@pytest.mark.parametrize("nq", [1, 5])
@pytest.mark.parametrize("nk", [129, 4097])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_padded_head_sizes(d, nq, nk, causal):
    """Head sizes other than 64 and 128 (multiples of 8) run in the 64- or
    128-column kernel with the columns past d read as zeros; canary bands
    around the outputs show any write past d columns or with the padded
    row stride."""
    q, k, v = rand(2, 3, nq, nk, d, seed=7000 + nq * 100 + nk + d + int(causal))
    scale = 1.0 / np.sqrt(d)
    o, lse, _ = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    o_ref, lse_ref = oracle.attention_rect(q, k, v, causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"d{d} nq{nq} nk{nk} c{int(causal)}")


def test_decode_padding_is_exact():
    """d = 96 equals d = 128 with the last 32 columns of q, k, v zero (the
    scale kept), bit for bit, both with one split and with many; the padded
    columns of the d = 128 output are zero."""
    pad = lambda t: torch.nn.functional.pad(t, (0, 128 - 96)).contiguous()
    for B, H, nk in ((64, 16, 3000), (1, 1, 20000)):
        q, k, v = (t.cuda() for t in rand(B, H, 3, nk, 96, seed=B + nk))
        o96, l96 = fa.decode(q, k, v, causal=True, scale=96 ** -0.5)
        o128, l128 = fa.decode(pad(q), pad(k), pad(v), causal=True, scale=96 ** -0.5)
        torch.cuda.synchronize()
        assert torch.equal(o96, o128[..., :96].contiguous())
        assert torch.equal(l96, l128)
        assert (o128[..., 96:] == 0).all()


def test_split_and_unsplit_key_ranges():
    """Many heads (a few chunks each) and one head (many chunks) give the
    oracle."""
    for B, H in ((64, 16), (1, 1)):
        q, k, v = rand(B, H, 1, 6000, 128, seed=B * 7 + H)
        o, lse, nbytes = run_guarded(q.cuda(), k.cuda(), v.cuda(), False, 0.088)
        if (B, H) == (1, 1):
            assert nbytes > 0  # a single head is split across CTAs
        bh = np.arange(B * H, dtype=np.int64)
        o_ref, lse_ref = oracle.attention_rect_rows(q, k, v, False, 0.088, bh, np.zeros_like(bh))
        assert_close(o.float().cpu().numpy().reshape(-1, 128), lse.cpu().numpy().reshape(-1), o_ref, lse_ref,
                     f"B{B} H{H}")


def test_large_scores_merge_across_splits():
    """A few dominant keys spread over distant chunks: the merge by logsumexp
    must weigh the chunks exactly."""
    q, k, v = rand(1, 2, 2, 30000, 64, seed=5, q_mult=4.0)
    k[:, :, 7::9001] *= 8.0  # exact in bf16
    o, lse, _ = run_guarded(q.cuda(), k.cuda(), v.cuda(), False, 0.125)
    o_ref, lse_ref = oracle.attention_rect(q, k, v, False, 0.125)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "spiky")


def test_single_key_returns_its_value():
    q, k, v = rand(2, 2, 1, 1, 128, seed=9)
    o, lse, _ = run_guarded(q.cuda(), k.cuda(), v.cuda(), False, 0.1)
    assert torch.equal(o.cpu(), v)  # one visible key: O = v_0 exactly


def test_causal_decode_matches_forward_last_rows():
    """Query rows Nk-Nq .. Nk-1 of a causal prefill equal causal decode of those rows."""
    q, k, v = make_random_qkv(2, 4, 777, 128, seed=11)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_f, l_f = fa.fwd(qd, kd, vd, causal=True)
    for nq in (1, 5):
        o_d, l_d = fa.decode(qd[:, :, -nq:].contiguous(), kd, vd, causal=True)
        torch.cuda.synchronize()
        do = (o_d.float() - o_f[:, :, -nq:].float()).abs()
        assert do.max().item() <= 2 * MAX_DO and do.mean().item() <= 2 * MEAN_DO
        assert (l_d - l_f[:, :, -nq:]).abs().max().item() <= 2 * MAX_DLSE


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_workload(name):
    w = DECODE_WORKLOADS[name]
    q, k, v = make_decode_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.decode(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    # O is a convex combination of the visible value rows (columnwise range).
    vf = vd.float()
    assert bool((o.float() <= vf.amax(dim=2, keepdim=True) + 1e-2).all())
    assert bool((o.float() >= vf.amin(dim=2, keepdim=True) - 1e-2).all())
    if w.sample_rows == 0:
        o_ref, lse_ref = oracle.attention_rect(q, k, v, w.causal, w.scale)
        assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, name)
        return
    bh, row = sample_decode_rows(w)
    o_ref, lse_ref = oracle.attention_rect_rows(q, k, v, w.causal, w.scale, bh, row)
    of = o.view(w.B * w.H, w.Nq, w.d)
    lf = lse.view(w.B * w.H, w.Nq)
    bh_t, row_t = torch.from_numpy(bh).cuda(), torch.from_numpy(row).cuda()
    assert_close(of[bh_t, row_t].float().cpu().numpy(), lf[bh_t, row_t].cpu().numpy(), o_ref, lse_ref, name)
