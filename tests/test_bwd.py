"""GPU parity of the attention backward (fa_bwd) with the fp64 oracle.

The forward runs on the GPU (fa_fwd), its O and logsumexp feed fa_bwd, and
dQ, dK, dV are compared with the oracle's exact gradients of the same bf16
inputs ("Writing and Benchmarking Custom Kernels" §10.3.2).

Tolerance (no page states one for gradients; derived from the kernel's
arithmetic).  The kernel rounds P and dS to bf16 (unit roundoff u = 2^-8) for
the tensor cores, takes D from the bf16 forward output, accumulates in fp32
and rounds the gradients to bf16.  To first order every gradient element G
is then off by at most u * (|G| + A), where A sums the absolute values of the
terms a rounded operand enters:
    A(dV_j) = sum_i P_ij |dO_i|
    A(dK_j) = scale * sum_i E_ij |Q_i|,   A(dQ_i) = scale * sum_j E_ij |K_j|
    E_ij    = |dS_ij| + P_ij * sum_c |dO_ic O_ic|   (rounded dS, and D from rounded O)
(fp32 accumulation and the exp2 approximation add orders of magnitude less).
Each element must lie within 2u * (|G| + A), and the mean error within
8e-3 * rms(G) (rms floored at 1e-2; one key makes dQ and dK exactly zero).
Replaying exactly the kernel's roundings in fp64 on these shapes reaches at
most 0.93 of u * (|G| + A) and a mean of 3.4e-3 * rms(G).
"""
import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa
import oracle
from io_aware_attention_gb300.workloads import make_random_qkv

pytestmark = pytest.mark.gpu

U = 2.0 ** -8      # bf16 unit roundoff
BOUND_FACTOR = 2.0
MEAN_RMS = 8e-3
RMS_FLOOR = 1e-2
GUARD = 64


def rounding_terms(q, k, v, do, causal, scale):
    """A(dQ), A(dK), A(dV) of one head (inputs (1, 1, N, d) bf16): the sums of
    absolute terms the tolerance scales with.  Uses the oracle's P and O."""
    Q, K, V, dO = (oracle.bf16_to_f64(t)[0, 0] for t in (q, k, v, do))
    o, _, P = oracle.attention(q, k, v, causal, scale, return_probs=True)
    o, P = o[0, 0], P[0, 0]
    D = (dO * o).sum(-1)
    E = np.abs(P * (dO @ V.T - D[:, None])) + P * np.abs(dO * o).sum(-1)[:, None]
    return scale * (E @ np.abs(K)), scale * (E.T @ np.abs(Q)), P.T @ np.abs(dO)


def grad_close(g, ref, terms, what):
    g = np.asarray(g, np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    rms = max(float(np.sqrt((ref ** 2).mean())), RMS_FLOOR)
    err = np.abs(g - ref)
    bound = BOUND_FACTOR * U * (np.abs(ref) + terms)
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), err.shape)
    msg = (f"{what}: worst |d|={err[worst]:.3e} at {tuple(int(i) for i in worst)} (|ref|={abs(ref[worst]):.3e}, "
           f"bound {bound[worst]:.3e}), max err/bound={ratio.max():.3f}, mean|d|/rms={err.mean() / rms:.3e}")
    assert ratio.max() <= 1.0 and err.mean() <= MEAN_RMS * rms, msg
    return ratio.max(), err.mean() / rms


def run_bwd(q, k, v, do, causal, scale):
    """fa.fwd, then fa.bwd_into with canary bands around every output and a
    NaN-filled workspace (nothing in it may need to start at zero)."""
    B, H, N, d = q.shape
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    n = B * H * N * d
    bufs = []
    for _ in range(3):
        b = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.bfloat16, device=q.device)
        b.view(torch.int16)[:GUARD] = 0x7FC1
        b.view(torch.int16)[-GUARD:] = 0x7FC1
        bufs.append(b)
    dq, dk, dv = (b[GUARD:GUARD + n].view(B, H, N, d) for b in bufs)
    ws = torch.full((fa.bwd_workspace_bytes(B, H, N, d),), 0xFF, dtype=torch.uint8, device=q.device)
    fa.bwd_into(q, k, v, o, lse, do, dq, dk, dv, ws, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0, "a kernel wait timed out"
    for b in bufs:
        bb = b.view(torch.int16).cpu()
        assert (bb[:GUARD] == 0x7FC1).all() and (bb[-GUARD:] == 0x7FC1).all(), "guard band overwritten"
    return dq, dk, dv


def check_heads(q, k, v, do, causal, scale, dq, dk, dv, heads, what):
    """Compares the listed flattened heads (b*H + h) with the oracle."""
    B, H, N, d = q.shape
    flat = lambda t: t.reshape(B * H, 1, 1, N, d)
    for bh in heads:
        ins = [flat(t.cpu())[bh].contiguous() for t in (q, k, v, do)]
        rq, rk, rv, _ = oracle.attention_bwd(*ins, causal, scale)
        terms = rounding_terms(*ins, causal, scale)
        for name, mine, ref, a in zip(("dq", "dk", "dv"), (dq, dk, dv), (rq, rk, rv), terms):
            grad_close(flat(mine.float().cpu())[bh].numpy()[0, 0], ref[0, 0], a, f"{what} head {bh} {name}")


SHAPES = [  # (B, H, N, causal)
    (1, 2, 256, True), (1, 2, 256, False), (2, 3, 384, True), (2, 3, 384, False),
    (1, 1, 1, True), (1, 1, 1, False), (1, 2, 63, True), (1, 2, 64, False), (1, 2, 65, True),
    (1, 1, 130, False), (1, 1, 200, True), (1, 2, 333, False), (2, 2, 1000, True), (1, 1, 1000, False),
]


@pytest.mark.parametrize("B,H,N,causal", SHAPES, ids=[f"b{b}h{h}n{n}{'c' if c else ''}" for b, h, n, c in SHAPES])
def test_bwd_parity(B, H, N, causal):
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, 128, 9000 + N + B))
    do = make_random_qkv(B, H, N, 128, 9500 + N + B)[0].cuda()
    scale = 128 ** -0.5
    dq, dk, dv = run_bwd(q, k, v, do, causal, scale)
    check_heads(q, k, v, do, causal, scale, dq, dk, dv, range(B * H), f"N={N} causal={causal}")


SHAPES_D64 = [  # (B, H, N, causal), head size 64
    (1, 2, 256, False), (1, 2, 256, True), (1, 1, 1, True), (1, 2, 65, False), (2, 2, 333, True),
    (1, 1, 1000, False),
]


@pytest.mark.parametrize("B,H,N,causal", SHAPES_D64, ids=[f"d64b{b}h{h}n{n}{'c' if c else ''}" for b, h, n, c in SHAPES_D64])
def test_bwd_parity_d64(B, H, N, causal):
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, 64, 9800 + N + B))
    do = make_random_qkv(B, H, N, 64, 9850 + N + B)[0].cuda()
    scale = 64 ** -0.5
    dq, dk, dv = run_bwd(q, k, v, do, causal, scale)
    check_heads(q, k, v, do, causal, scale, dq, dk, dv, range(B * H), f"d=64 N={N} causal={causal}")


def test_bwd_d64_stress_workload_sampled_heads():
    """The d = 64 rescale-stress workload (B16 H16 N8192, Q x4, every 512th
    key x8, non-causal): whole sampled heads against the oracle."""
    from io_aware_attention_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS["b16_h16_n8192_d64_spiky"]
    q, k, v = (t.cuda() for t in make_qkv(w))
    do = make_random_qkv(w.B, w.H, w.N, w.d, w.seed + 500)[0].cuda()
    o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    check_heads(q, k, v, do, w.causal, w.scale, dq, dk, dv, [w.B * w.H - 1], "d=64 stress")


def test_bwd_spiky_scores():
    """Large scores (Q = 4 N(0,1)) and every 16th key scaled by 8, so rows are
    dominated by a few keys and P spans many binades."""
    q, k, v = (t.cuda() for t in make_random_qkv(1, 2, 512, 128, 9601, q_mult=4.0))
    k[:, :, ::16] *= 8
    do = make_random_qkv(1, 2, 512, 128, 9602)[0].cuda()
    for causal in (False, True):
        dq, dk, dv = run_bwd(q, k, v, do, causal, 128 ** -0.5)
        check_heads(q, k, v, do, causal, 128 ** -0.5, dq, dk, dv, range(2), f"spiky causal={causal}")


def test_bwd_other_scale():
    q, k, v = (t.cuda() for t in make_random_qkv(1, 2, 300, 128, 9603))
    do = make_random_qkv(1, 2, 300, 128, 9604)[0].cuda()
    dq, dk, dv = run_bwd(q, k, v, do, True, 0.05)
    check_heads(q, k, v, do, True, 0.05, dq, dk, dv, range(2), "scale=0.05")


def test_bwd_dk_dv_deterministic():
    """dK and dV come from one CTA each (no atomics): bitwise equal across runs."""
    q, k, v = (t.cuda() for t in make_random_qkv(2, 4, 1024, 128, 9605))
    do = make_random_qkv(2, 4, 1024, 128, 9606)[0].cuda()
    o, lse = fa.fwd(q, k, v, causal=True)
    a = fa.bwd(q, k, v, o, lse, do, causal=True)
    b = fa.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ is summed with atomics in fp32: equal up to its rounding to bf16.
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2 ** -7 * a[0].float().abs().max().item()


@pytest.mark.parametrize("B,H,N,causal,heads", [
    (4, 16, 2048, True, [0, 63]),
    (8, 32, 4096, True, [255]),
    (8, 32, 4096, False, [0]),
], ids=["b4h16n2048c", "b8h32n4096c", "b8h32n4096"])
def test_bwd_full_size_sampled_heads(B, H, N, causal, heads):
    """The benchmark shapes; whole heads compared (a head's gradients need
    every row of it)."""
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, 128, 9700 + N))
    do = make_random_qkv(B, H, N, 128, 9701 + N)[0].cuda()
    o, lse = fa.fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    check_heads(q, k, v, do, causal, 128 ** -0.5, dq, dk, dv, heads, f"B={B} H={H} N={N}")


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_many_short_heads(d, causal):
    """1024 heads of 65 rows: every item is one key block of two query steps,
    so each CTA turns items over every other step (the dK / dV read-out and
    the item barriers at their fastest).  64 heads, the first and last among
    them, against the oracle."""
    B, H, N = 16, 64, 65
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 9900 + d + int(causal)))
    do = make_random_qkv(B, H, N, d, 9950 + d + int(causal))[0].cuda()
    scale = d ** -0.5
    dq, dk, dv = run_bwd(q, k, v, do, causal, scale)
    rng = np.random.default_rng(9900 + d)
    heads = sorted({0, B * H - 1, *rng.integers(0, B * H, size=62).tolist()})
    check_heads(q, k, v, do, causal, scale, dq, dk, dv, heads, f"{B * H} heads of N={N}")
