"""GPU kernel vs the fp64 oracle on small shapes, element by element.

Shapes span several 128-row tiles and ragged tails (N not a multiple of the
tile, "Writing and Benchmarking Custom Kernels" §10.3.1: the final partial
tile), both head sizes, causal and not, plus the method's degenerate cases.
"""
import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa
import oracle
from io_aware_attention_gb300.workloads import make_random_qkv

from _parity import assert_close, run_guarded

pytestmark = pytest.mark.gpu

NS = [1, 2, 17, 64, 127, 128, 129, 200, 256, 383, 640]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", NS)
def test_small_shapes(N, d, causal):
    q, k, v = make_random_qkv(1, 2, N, d, seed=100 + N + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
                 f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_many_heads(d):
    q, k, v = make_random_qkv(3, 5, 300, d, seed=7)
    for causal in (False, True):
        o, lse = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, 0.1)
        o_ref, lse_ref = oracle.attention(q, k, v, causal, 0.1)
        assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"d={d} {causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_causal_row0_is_v0(d):
    """Row 0 sees key 0 only: O_0 = V_0 bit for bit, L_0 = scale * q_0 . k_0."""
    q, k, v = make_random_qkv(2, 3, 257, d, seed=8)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])
    ref = scale * (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1)
    assert (lse[:, :, 0].cpu().double() - ref).abs().max().item() <= 1e-4


@pytest.mark.parametrize("d", [64, 128])
def test_causal_last_row_equals_full_row(d):
    """The mask leaves the last query row every key: the causal kernel's last
    row must match the oracle's non-causal last row, computed by the oracle
    without any mask."""
    B, H, N = 1, 4, 333
    q, k, v = make_random_qkv(B, H, N, d, seed=9)
    scale = 1.0 / np.sqrt(d)
    oc, lc = run_guarded(q.cuda(), k.cuda(), v.cuda(), True, scale)
    bh = np.arange(B * H, dtype=np.int64)
    row = np.full(B * H, N - 1, dtype=np.int64)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, False, scale, bh, row)
    got_o = oc.view(B * H, N, d)[:, -1].float().cpu().numpy()
    got_l = lc.view(B * H, N)[:, -1].cpu().numpy()
    assert_close(got_o, got_l, o_ref, lse_ref, f"last causal row d={d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rescale_stress(d, causal):
    """Large scores whose row max jumps late in the row (Q x4, every 64th key x8
    and the last key x16): the running max must rescale O and l."""
    q, k, v = make_random_qkv(1, 2, 1000, d, seed=10, q_mult=4.0)
    k = k.clone()
    k[:, :, 63::64] *= 8
    k[:, :, -1] *= 16
    scale = 1.0 / np.sqrt(d)
    o, lse = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "stress")


def test_constant_values_pass_through():
    q, k, _ = make_random_qkv(1, 2, 500, 128, seed=11)
    v = torch.full_like(q, 0.7109375)  # exactly representable in bf16
    o, _ = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert (o.float() - 0.7109375).abs().max().item() <= 2 ** -8


def test_side_stream_and_repeatability():
    q, k, v = (t.cuda() for t in make_random_qkv(2, 2, 700, 128, seed=12))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = fa.fwd(q, k, v, causal=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_python_checks_reject_bad_tensors():
    q, k, v = (t.cuda() for t in make_random_qkv(1, 1, 64, 64, seed=13))
    with pytest.raises(ValueError):
        fa.fwd(q.float(), k, v)
    with pytest.raises(ValueError):
        fa.fwd(q.transpose(2, 3), k, v)
    with pytest.raises(fa.FaError) as e:
        # head sizes must be multiples of 8 (up to 128)
        fa.fwd(q[..., :36].contiguous(), k[..., :36].contiguous(), v[..., :36].contiguous())
    assert e.value.code == 2


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("pos", [0, 1, 31, 63, 64, 65, 96, 127])
def test_row_max_at_each_column(pos, causal, d):
    """The row max of a tile comes back with the TMEM load of the scores; put
    it on a chosen key column of every tile (the first and last of each
    64-column half among them) by scaling that key up, with a tie in the
    other half, and compare with the oracle.  The planted keys dominate their
    rows, so O comes close to single value rows; V is halved (exactly, in
    bf16) so that |O| stays where the bf16 rounding of the output (half an
    ulp: 2^-8 |O|) is within the absolute tolerance."""
    N = 640
    q, k, v = make_random_qkv(1, 2, N, d, seed=300 + pos + d)
    k, v = k.clone(), v * 0.5
    k[:, :, pos::128] *= 6
    k[:, :, (pos + 64) % 128::128] = k[:, :, pos::128][:, :, : k[:, :, (pos + 64) % 128::128].shape[2]]
    scale = 1.0 / np.sqrt(d)
    o, lse = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"max at column {pos}")


@pytest.mark.parametrize("d", [64, 128, 40])
@pytest.mark.parametrize("causal", [False, True])
def test_many_single_tile_items(d, causal):
    """Thousands of heads of a few rows: every item is one tile, so the
    statistics slots, the O hand-over to the epilogue warps and the Q loads
    turn over at every tile, on every CTA, many times over.  Full tensors
    against the oracle.  The first causal rows see one to three keys, so O
    is close to single value rows; V is halved (exactly, in bf16) so that
    |O| stays where the bf16 rounding of the output fits the absolute
    tolerance over these 2048 heads."""
    B, H, N = 32, 64, 17
    q, k, v = make_random_qkv(B, H, N, d, seed=500 + d + int(causal))
    v = v * 0.5
    scale = 1.0 / np.sqrt(d)
    o, lse = run_guarded(q.cuda(), k.cuda(), v.cuda(), causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal, scale)
    assert_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"{B * H} heads of N={N}")
