"""Pins for the CPU oracle, checked against things other than itself.

Each pin is a plain function taking an oracle instance, so that the same
battery can be run against copies of the oracle with a planted mistake
(``test_planted_mistakes_are_caught``): every plausible slip -- a mask off by
one, a transposed operand, a dropped scale or normalisation, a wrong sign, a
wrong logarithm base, a missing rescale in the recurrence -- must fail at
least one pin.

What pins what (the statements are those of "Kernels — fusion and
FlashAttention" §2–§3, "Fusion and IO-aware kernels" § FlashAttention, and
"Writing and Benchmarking Custom Kernels" §10.3):
  * library softmax / logsumexp (scipy) on tiny inputs -- the whole definition;
  * exact closed forms: one key (O = V, L = scale·q·k), equal scores (O = mean
    of the visible values, L = ln n), two keys (logistic weights);
  * invariants: probability rows sum to one, constant values pass through,
    a per-row score shift leaves O alone and moves L by the shift, key
    permutation leaves non-causal rows alone, a causal row equals the
    unmasked problem on its prefix, huge scores do not overflow;
  * the tile-by-tile online recurrence reaches the two-pass result for every
    tile size, including 1, sizes that do not divide N, and sizes above N.

The backward (gradients dQ, dK, dV for a given dO; "Writing and Benchmarking
Custom Kernels" §10.3.2) is pinned by:
  * torch's fp64 autograd of the plain masked softmax(QK^T)V expression;
  * central finite differences (Richardson-extrapolated) of the forward
    oracle's sum(O * dO), on inputs that are multiples of 2^-7 below 2 in
    magnitude so that every perturbed input is still exactly a bf16 value;
  * invariants: the softmax gradient rows sum to zero, so the key gradients
    sum to zero over keys; the value gradients sum to the summed dO; D_i
    equals dO_i . O_i (the page's form of the row scalar); a single key gives
    dV = dO and dQ = dK = 0; under the causal mask keys after the last row
    with a nonzero dO get no gradient; key permutation permutes dK, dV.

The fused elementwise chain (bias + GELU + dropout; "Fusion and IO-aware
kernels", "Writing and Benchmarking Custom Kernels" §10.2.1) is pinned by:
  * the exact GELU x·Phi(x) (scipy's normal cdf) within 4.8e-4 over
    [-8, 8]: the tanh form's own maximum departure is 4.73e-4;
  * the exact identity g(-h) = g(h) - h (tanh is odd), g(0) = 0, g(h) = h and
    g(-h) = 0 far out, and (g(h) - h/2) / h^2 -> 1/sqrt(2 pi) as h -> 0;
  * bias broadcast: on integer data (exact in bf16) x + bias through the
    oracle equals the sum fed in with a zero bias, with rows != cols;
  * dropout: kept elements are the undropped values divided by (1 - p),
    dropped ones exactly 0, and the mask bit of element e is bit e % 32 of
    word e // 32.
"""
import math
import os
import re
import shutil
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from io_aware_attention_gb300.workloads import make_random_qkv

HERE = os.path.dirname(os.path.abspath(__file__))


def f64(x):
    return oracle.bf16_to_f64(x)


def bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


# --------------------------------------------------------------------------- pins


def pin_library_softmax(orc):
    """scipy softmax / logsumexp of the masked, scaled score matrix."""
    for (B, H, N, d, causal, seed) in [(1, 1, 1, 8, False, 1), (1, 2, 5, 8, True, 2),
                                        (2, 1, 17, 64, False, 3), (1, 1, 17, 64, True, 4),
                                        (1, 1, 9, 1, True, 5)]:
        q, k, v = make_random_qkv(B, H, N, d, seed)
        scale = 0.37
        o, lse = orc.attention(q, k, v, causal, scale)
        Q, K, V = f64(q), f64(k), f64(v)
        S = scale * np.einsum("bhid,bhjd->bhij", Q, K)
        if causal:
            S = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, S)
        P = scipy.special.softmax(S, axis=-1)
        np.testing.assert_allclose(o, P @ V, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, scipy.special.logsumexp(S, axis=-1), rtol=1e-13,
                                   atol=1e-13)


def pin_single_key(orc):
    """N = 1: the one key gets all the weight; L = scale·q·k exactly."""
    q, k, v = make_random_qkv(2, 3, 1, 64, 11)
    scale = 0.125
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, scale)
        np.testing.assert_array_equal(o, f64(v))
        Q, K = f64(q), f64(k)
        for b in range(2):
            for h in range(3):
                exact = Fraction(scale) * sum(Fraction(float(a)) * Fraction(float(c))
                                              for a, c in zip(Q[b, h, 0], K[b, h, 0]))
                assert abs(lse[b, h, 0] - float(exact)) <= 1e-13 * max(1.0, abs(float(exact)))


def pin_equal_scores(orc):
    """Q = 0: all visible scores are 0, O = mean of the visible values, L = ln n."""
    _, k, v = make_random_qkv(1, 2, 13, 16, 12)
    q = torch.zeros_like(k)
    V = f64(v)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.5)
        for i in range(13):
            n = i + 1 if causal else 13
            mean = np.array([[float(sum(Fraction(float(x)) for x in V[0, h, :n, c]) / n)
                              for c in range(16)] for h in range(2)])
            np.testing.assert_allclose(o[0, :, i], mean, rtol=1e-14, atol=1e-15)
            np.testing.assert_allclose(lse[0, :, i], math.log(n), rtol=1e-15, atol=1e-15)


def pin_two_keys(orc):
    """N = 2: weights are the logistic function of the score gap."""
    q, k, v = make_random_qkv(1, 1, 2, 8, 13, q_mult=2.0)
    scale = 0.3
    Q, K, V = f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0]
    o, lse = orc.attention(q, k, v, False, scale)
    oc, lsec = orc.attention(q, k, v, True, scale)
    for i in range(2):
        s0, s1 = scale * float(Q[i] @ K[0]), scale * float(Q[i] @ K[1])
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(o[0, 0, i], w0 * V[0] + (1.0 - w0) * V[1], rtol=1e-13,
                                   atol=1e-14)
        hi = max(s0, s1)
        assert abs(lse[0, 0, i] - (hi + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-13
    # causal: row 0 sees key 0 only, row 1 sees both
    np.testing.assert_array_equal(oc[0, 0, 0], V[0])
    assert abs(lsec[0, 0, 0] - scale * float(Q[0] @ K[0])) < 1e-13
    np.testing.assert_allclose(oc[0, 0, 1], o[0, 0, 1], rtol=1e-15, atol=1e-15)


def pin_probability_rows(orc):
    """P >= 0, rows sum to 1, and the causal mask zeroes exactly j > i."""
    q, k, v = make_random_qkv(1, 2, 23, 32, 14)
    for causal in (False, True):
        _, _, p = orc.attention(q, k, v, causal, 0.2, return_probs=True)
        assert (p >= 0).all()
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
        upper = np.triu(np.ones((23, 23), bool), 1)
        if causal:
            assert (p[..., upper] == 0).all()
            assert (p[..., ~upper] > 0).all()
        else:
            assert (p > 0).all()


def pin_constant_values(orc):
    """Every value row equal to c: O = c whatever the weights."""
    q, k, _ = make_random_qkv(1, 2, 31, 64, 15)
    c = make_random_qkv(1, 2, 1, 64, 16)[2]
    v = c.expand(1, 2, 31, 64).contiguous()
    for causal in (False, True):
        o, _ = orc.attention(q, k, v, causal, 0.125)
        np.testing.assert_allclose(o, np.broadcast_to(f64(c), o.shape), rtol=1e-14, atol=1e-15)


def pin_score_shift(orc):
    """Adding u to every key row shifts row i's scores by scale·q_i·u: O stays,
    L moves by exactly that shift (integer-valued data keeps K + u exact)."""
    rng = np.random.default_rng(17)
    N, d, scale = 12, 8, 0.25
    Qi = rng.integers(-3, 4, size=(1, 1, N, d))
    Ki = rng.integers(-4, 5, size=(1, 1, N, d))
    u = rng.integers(-2, 3, size=(d,))
    Vv = rng.standard_normal((1, 1, N, d))
    q, k, k2, v = bf16(Qi), bf16(Ki), bf16(Ki + u), bf16(Vv)
    for causal in (False, True):
        o1, l1 = orc.attention(q, k, v, causal, scale)
        o2, l2 = orc.attention(q, k2, v, causal, scale)
        np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(l2 - l1, scale * (Qi @ u), rtol=0, atol=1e-12)


def pin_key_permutation(orc):
    """Non-causal rows do not depend on the order of the (key, value) pairs."""
    q, k, v = make_random_qkv(1, 1, 19, 16, 18)
    perm = torch.from_numpy(np.random.default_rng(19).permutation(19))
    o1, l1 = orc.attention(q, k, v, False, 0.25)
    o2, l2 = orc.attention(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, 0.25)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l2, l1, rtol=1e-14, atol=1e-14)


def pin_causal_prefix(orc):
    """Causal row i equals the unmasked problem on keys 0..i (last row there)."""
    q, k, v = make_random_qkv(1, 1, 9, 16, 20)
    oc, lc = orc.attention(q, k, v, True, 0.25)
    for i in range(9):
        sl = slice(0, i + 1)
        o, l = orc.attention(q[:, :, sl].contiguous(), k[:, :, sl].contiguous(),
                             v[:, :, sl].contiguous(), False, 0.25)
        np.testing.assert_allclose(oc[0, 0, i], o[0, 0, i], rtol=1e-14, atol=1e-15)
        assert abs(lc[0, 0, i] - l[0, 0, i]) < 1e-13


def pin_huge_scores(orc):
    """Scores in the thousands: with the max subtracted nothing overflows; the
    row collapses onto the best key and L is the largest score."""
    q, k, v = make_random_qkv(1, 1, 16, 64, 21, q_mult=64.0)
    k = k * 8
    o, lse = orc.attention(q, k, v, False, 1.0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    S = f64(q)[0, 0] @ f64(k)[0, 0].T
    assert S.max() > 1000.0
    best = S.argmax(-1)
    top2 = np.sort(S, -1)[:, -2:]
    assert (top2[:, 1] - top2[:, 0] > 40).all()  # the runner-up weighs < e^-40
    np.testing.assert_allclose(o[0, 0], f64(v)[0, 0][best], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], S.max(-1), rtol=1e-15, atol=1e-12)


def pin_rows_entry(orc):
    """Selected rows equal the same rows of the full computation."""
    q, k, v = make_random_qkv(2, 3, 37, 16, 22)
    bh = np.array([0, 5, 3, 2, 4, 1], np.int64)
    row = np.array([0, 36, 17, 1, 35, 20], np.int64)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.3)
        orow, lrow = orc.attention_rows(q, k, v, causal, 0.3, bh, row)
        np.testing.assert_array_equal(orow, o.reshape(6, 37, 16)[bh, row])
        np.testing.assert_array_equal(lrow, lse.reshape(6, 37)[bh, row])


def pin_online_recurrence(orc):
    """The tile-by-tile recurrence reaches the two-pass result for any tile size."""
    q, k, v = make_random_qkv(1, 2, 100, 32, 23, q_mult=3.0)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.4)
        for tile in (1, 3, 16, 64, 100, 105):
            o2, l2 = orc.attention_online(q, k, v, causal, 0.4, tile)
            np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(l2, lse, rtol=1e-13, atol=1e-12)


def pin_rect_is_square_when_nq_is_nk(orc):
    """Decode attention with as many queries as keys is the square case."""
    q, k, v = make_random_qkv(2, 2, 29, 16, 31)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.3)
        o2, l2 = orc.attention_rect(q, k, v, causal, 0.3)
        np.testing.assert_array_equal(o2, o)
        np.testing.assert_array_equal(l2, lse)


def pin_rect_bottom_right(orc):
    """Causal decode: the Nq queries are the last Nq positions of the sequence,
    so their rows equal the last Nq rows of square causal attention."""
    q, k, v = make_random_qkv(1, 3, 40, 16, 32)
    for nq in (1, 3, 7):
        o, lse = orc.attention(q, k, v, True, 0.3)
        o2, l2 = orc.attention_rect(q[:, :, -nq:].contiguous(), k, v, True, 0.3)
        np.testing.assert_array_equal(o2, o[:, :, -nq:])
        np.testing.assert_array_equal(l2, lse[:, :, -nq:])


def pin_rect_single_query_library(orc):
    """One query against the whole cache: scipy's softmax and logsumexp."""
    q, k, v = make_random_qkv(1, 2, 50, 16, 33, q_mult=2.0)
    q1 = q[:, :, 5:6].contiguous()
    o, lse = orc.attention_rect(q1, k, v, False, 0.4)
    S = 0.4 * np.einsum("bhqc,bhkc->bhqk", f64(q1), f64(k))
    np.testing.assert_allclose(o, np.einsum("bhqk,bhkc->bhqc", scipy.special.softmax(S, axis=-1), f64(v)),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(S, axis=-1), rtol=1e-13, atol=1e-12)


def pin_rect_rows_entry(orc):
    """Selected decode rows equal the same rows of the full computation."""
    q, k, v = make_random_qkv(2, 2, 33, 16, 34)
    q4 = q[:, :, :4].contiguous()
    bh = np.array([0, 3, 1, 2, 3], np.int64)
    row = np.array([0, 3, 2, 1, 0], np.int64)
    for causal in (False, True):
        o, lse = orc.attention_rect(q4, k, v, causal, 0.3)
        orow, lrow = orc.attention_rect_rows(q4, k, v, causal, 0.3, bh, row)
        np.testing.assert_array_equal(orow, o.reshape(4, 4, 16)[bh, row])
        np.testing.assert_array_equal(lrow, lse.reshape(4, 4)[bh, row])


def _bwd_inputs(B, H, N, d, seed):
    """bf16 q, k, v whose entries are multiples of 2^-7 in (-1.9, 1.9), so that
    x +- 2^-7 and x +- 2^-6 are bf16 values too; dO any bf16."""
    rng = np.random.default_rng(seed)
    grid = lambda: bf16(np.clip(np.round(rng.standard_normal((B, H, N, d)) * 0.7 * 128) / 128,
                                -1.875, 1.875))
    q, k, v = grid(), grid(), grid()
    do = bf16(rng.standard_normal((B, H, N, d)))
    return q, k, v, do


def pin_bwd_autograd(orc):
    """torch fp64 autograd of softmax(scale*QK^T + mask) V with output gradient dO."""
    for (B, H, N, d, causal, seed) in [(1, 1, 1, 8, True, 41), (1, 2, 6, 8, True, 42),
                                        (2, 1, 11, 16, False, 43), (1, 1, 13, 32, True, 44)]:
        q, k, v = make_random_qkv(B, H, N, d, seed, q_mult=1.5)
        do = make_random_qkv(B, H, N, d, seed + 100)[0]
        scale = 0.31
        dq, dk, dv, dsum = orc.attention_bwd(q, k, v, do, causal, scale)
        Q, K, V = (torch.from_numpy(f64(t)).requires_grad_() for t in (q, k, v))
        S = scale * Q @ K.transpose(-1, -2)
        if causal:
            S = S.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        O = torch.softmax(S, dim=-1) @ V
        O.backward(torch.from_numpy(f64(do)))
        for mine, ref in ((dq, Q.grad), (dk, K.grad), (dv, V.grad)):
            np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-11, atol=1e-12)


def pin_bwd_finite_differences(orc):
    """Every gradient entry against (8(f(x+h)-f(x-h)) - (f(x+2h)-f(x-2h))) / 12h of
    f = sum(O * dO) through the forward oracle, h = 2^-7 (error O(h^4))."""
    h = 2.0 ** -7
    for (N, d, causal, seed) in [(5, 4, True, 45), (4, 3, False, 46)]:
        q, k, v, do = _bwd_inputs(1, 1, N, d, seed)
        scale = 0.35
        dq, dk, dv, _ = orc.attention_bwd(q, k, v, do, causal, scale)
        dO = f64(do)

        def f(qq, kk, vv):
            return float((orc.attention(qq, kk, vv, causal, scale)[0] * dO).sum())

        for which, grad in ((0, dq), (1, dk), (2, dv)):
            for i in range(N):
                for c in range(d):
                    vals = []
                    for step in (h, -h, 2 * h, -2 * h):
                        ins = [q.clone(), k.clone(), v.clone()]
                        ins[which][0, 0, i, c] = ins[which][0, 0, i, c].float() + step
                        assert float(ins[which][0, 0, i, c]) == float(
                            [q, k, v][which][0, 0, i, c]) + step  # perturbation is exact
                        vals.append(f(*ins))
                    fd = (8 * (vals[0] - vals[1]) - (vals[2] - vals[3])) / (12 * h)
                    assert abs(grad[0, 0, i, c] - fd) <= 1e-7 + 1e-6 * abs(fd), (which, i, c)


def pin_bwd_invariants(orc):
    """Rows of the softmax gradient sum to zero (so sum_j dK_j = 0), sum_j dV_j
    = sum_i dO_i, and D_i = dO_i . O_i."""
    q, k, v = make_random_qkv(2, 2, 21, 16, 47, q_mult=2.0)
    do = make_random_qkv(2, 2, 21, 16, 48)[0]
    for causal in (False, True):
        dq, dk, dv, dsum = orc.attention_bwd(q, k, v, do, causal, 0.4)
        o, _ = orc.attention(q, k, v, causal, 0.4)
        scale_dk = np.abs(dk).max()
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-13 * 21 * max(1.0, scale_dk))
        np.testing.assert_allclose(dv.sum(axis=2), f64(do).sum(axis=2), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dsum, (f64(do) * o).sum(-1), rtol=1e-12, atol=1e-12)


def pin_bwd_single_key(orc):
    """N = 1: P = 1, so dV = dO and the score gradient, hence dQ and dK, is zero."""
    q, k, v = make_random_qkv(2, 2, 1, 32, 49)
    do = make_random_qkv(2, 2, 1, 32, 50)[0]
    for causal in (False, True):
        dq, dk, dv, _ = orc.attention_bwd(q, k, v, do, causal, 0.2)
        np.testing.assert_array_equal(dv, f64(do))
        np.testing.assert_array_equal(dq, 0.0)
        np.testing.assert_array_equal(dk, 0.0)


def pin_bwd_causal_tail(orc):
    """Causal, dO zero from row t on: keys t.. are seen only by those rows, so
    their dK and dV are zero; rows before t match the problem cut at t."""
    q, k, v = make_random_qkv(1, 2, 17, 16, 51)
    do = make_random_qkv(1, 2, 17, 16, 52)[0]
    t = 9
    do[:, :, t:] = 0
    dq, dk, dv, _ = orc.attention_bwd(q, k, v, do, True, 0.3)
    np.testing.assert_array_equal(dk[:, :, t:], 0.0)
    np.testing.assert_array_equal(dv[:, :, t:], 0.0)
    np.testing.assert_array_equal(dq[:, :, t:], 0.0)
    cut = [x[:, :, :t].contiguous() for x in (q, k, v, do)]
    dq2, dk2, dv2, _ = orc.attention_bwd(*cut, True, 0.3)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        np.testing.assert_allclose(a[:, :, :t], b, rtol=1e-13, atol=1e-14)


def pin_bwd_key_permutation(orc):
    """Non-causal: permuting the (key, value) pairs permutes dK and dV the same
    way and leaves dQ alone."""
    q, k, v = make_random_qkv(1, 1, 15, 8, 53)
    do = make_random_qkv(1, 1, 15, 8, 54)[0]
    perm = torch.from_numpy(np.random.default_rng(55).permutation(15))
    dq, dk, dv, _ = orc.attention_bwd(q, k, v, do, False, 0.5)
    dq2, dk2, dv2, _ = orc.attention_bwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(),
                                         do, False, 0.5)
    np.testing.assert_allclose(dq2, dq, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk2, dk[:, :, perm.numpy()], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv2, dv[:, :, perm.numpy()], rtol=1e-12, atol=1e-13)


def _ew_inputs(rows, cols, seed):
    rng = np.random.default_rng(seed)
    return bf16(rng.standard_normal((rows, cols)) * 2.0), bf16(rng.standard_normal(cols))


def pin_gelu_exact_library(orc):
    """The tanh form stays within its known 4.73e-4 of x*Phi(x) (scipy.special.ndtr)."""
    x = bf16(np.linspace(-8, 8, 4097).reshape(1, -1))
    y = orc.bias_gelu_dropout(x, bf16(np.zeros(4097)), None, 0.0)
    X = f64(x)
    assert np.abs(y - X * scipy.special.ndtr(X)).max() <= 4.8e-4


def pin_gelu_identities(orc):
    """g(-h) = g(h) - h; g(0) = 0; g far out; the h^2 coefficient at 0."""
    x = bf16(np.linspace(-5, 5, 513).reshape(1, -1))
    zero = bf16(np.zeros(513))
    g = orc.bias_gelu_dropout(x, zero, None, 0.0)
    gn = orc.bias_gelu_dropout(bf16(-f64(x)), zero, None, 0.0)
    np.testing.assert_allclose(gn, g - f64(x), rtol=0, atol=1e-14)
    t = bf16(np.array([[0.0, 9.0, -9.0, 2.0 ** -12]]))
    y = orc.bias_gelu_dropout(t, bf16(np.zeros(4)), None, 0.0)[0]
    assert y[0] == 0.0 and abs(y[1] - 9.0) < 1e-14 and abs(y[2]) < 1e-14
    h = 2.0 ** -12
    assert abs((y[3] - h / 2) / h ** 2 - 1 / math.sqrt(2 * math.pi)) < 1e-3


def pin_bias_broadcast(orc):
    """Integer data (exact in bf16): gelu(x + bias) with bias per column equals
    gelu of the materialised sum with a zero bias."""
    rng = np.random.default_rng(61)
    xi = rng.integers(-4, 5, size=(5, 7)).astype(np.float64)
    bi = rng.integers(-3, 4, size=(7,)).astype(np.float64)
    y1 = orc.bias_gelu_dropout(bf16(xi), bf16(bi), None, 0.0)
    y2 = orc.bias_gelu_dropout(bf16(xi + bi), bf16(np.zeros(7)), None, 0.0)
    np.testing.assert_array_equal(y1, y2)


def pin_dropout_mask(orc):
    """Kept: undropped / (1 - p); dropped: exactly 0; bit e % 32 of word e // 32."""
    x, b = _ew_inputs(6, 40, 62)
    n = 6 * 40
    words = np.random.default_rng(63).integers(0, 2 ** 32, size=(n + 31) // 32 + 32, dtype=np.uint64).astype(np.uint32)
    p = 0.25
    full = orc.bias_gelu_dropout(x, b, None, 0.0)
    y = orc.bias_gelu_dropout(x, b, words, p)
    bits = np.array([(int(words[e >> 5]) >> (e & 31)) & 1 for e in range(n)], bool).reshape(6, 40)
    assert (y[~bits] == 0).all()
    np.testing.assert_allclose(y[bits], full[bits] / (1 - p), rtol=1e-15, atol=0)
    one = np.zeros_like(words)
    one[37 >> 5] = np.uint32(1 << (37 & 31))
    y1 = orc.bias_gelu_dropout(x, b, one, 0.5)
    assert np.count_nonzero(y1) == (1 if full.flat[37] != 0 else 0) and y1.flat[37] == full.flat[37] * 2


PINS = [pin_library_softmax, pin_single_key, pin_equal_scores, pin_two_keys,
        pin_probability_rows, pin_constant_values, pin_score_shift, pin_key_permutation,
        pin_causal_prefix, pin_huge_scores, pin_rows_entry, pin_online_recurrence,
        pin_rect_is_square_when_nq_is_nk, pin_rect_bottom_right, pin_rect_single_query_library,
        pin_rect_rows_entry, pin_bwd_autograd, pin_bwd_finite_differences, pin_bwd_invariants,
        pin_bwd_single_key, pin_bwd_causal_tail, pin_bwd_key_permutation, pin_gelu_exact_library,
        pin_gelu_identities, pin_bias_broadcast, pin_dropout_mask]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle)


# --------------------------------------------------------- planted mistakes

# (description, text to replace, replacement) -- each applied alone to a copy
# of attn_ref.c.  Indexes stay in bounds so a mutant cannot crash the test.
MUTANTS = [
    ("mask off by one (diagonal hidden)", "if (causal && j > i) {\n            s_row[j]",
     "if (causal && j >= i) {\n            s_row[j]"),
    ("mask the wrong triangle", "if (causal && j > i) {\n            s_row[j]",
     "if (causal && j < i) {\n            s_row[j]"),
    ("transposed score operands", "q[i * d + c]) * bf16_bits_to_f64(k[j * d + c])",
     "q[j * d + c]) * bf16_bits_to_f64(k[i * d + c])"),
    ("scale dropped", "s_row[j] = scale * acc;", "s_row[j] = acc;"),
    ("exp sign flipped", "s_row[j] = exp(s_row[j] - m);", "s_row[j] = exp(m - s_row[j]);"),
    ("no normalisation", "for (int64_t j = 0; j < N; ++j) s_row[j] /= l;", ""),
    ("values of the query row", "o_row[c] += p * bf16_bits_to_f64(v[j * d + c])",
     "o_row[c] += p * bf16_bits_to_f64(v[i * d + c])"),
    ("lse in base 2", "*lse = m + log(l);", "*lse = m + log2(l);"),
    ("lse without the max", "*lse = m + log(l);", "*lse = log(l);"),
    ("max not subtracted", "double m = -INFINITY;\n    for (int64_t j = 0; j < N; ++j)\n        if",
     "double m = 0.0;\n    for (int64_t j = 0; j < N; ++j)\n        if (0) if"),
    ("recurrence: output not rescaled", "for (int64_t c = 0; c < d; ++c) acc[c] *= corr;", ""),
    ("recurrence: denominator not rescaled", "l = l * corr + psum;", "l = l + psum;"),
    ("recurrence: causal tile skip off by one", "if (causal && j0 > i) break;",
     "if (causal && j0 >= i) break;"),
    ("decode: the query's own key masked", "if (j > last_key) {", "if (j >= last_key) {"),
    ("decode: causal window aligned top-left",
     "const int64_t bh = r / Nq, i = r % Nq;\n            const int64_t last = causal ? Nk - Nq + i : Nk - 1;",
     "const int64_t bh = r / Nq, i = r % Nq;\n            const int64_t last = causal ? i : Nk - 1;"),
    ("decode: every row uses the head's first query", "attention_row_keys(q + r * d, k + bh * Nk * d",
     "attention_row_keys(q + bh * Nq * d, k + bh * Nk * d"),
    ("backward: D dropped", "dSi[j] = j < visible ? Pi[j] * (dP[j] - Di) : 0.0;",
     "dSi[j] = j < visible ? Pi[j] * dP[j] : 0.0;"),
    ("backward: score gradient sign", "dSi[j] = j < visible ? Pi[j] * (dP[j] - Di) : 0.0;",
     "dSi[j] = j < visible ? Pi[j] * (Di - dP[j]) : 0.0;"),
    ("backward: D without the probabilities", "Di += Pi[j] * g;", "Di += g;"),
    ("backward: dQ scale dropped", "dq[base + i * d + c] = scale * acc;", "dq[base + i * d + c] = acc;"),
    ("backward: dQ from the values", "acc += dSi[j] * Kw[j * d + c];", "acc += dSi[j] * Vw[j * d + c];"),
    ("backward: dK from dS untransposed", "gk += dS[i * N + j] * Qw[i * d + c];",
     "gk += dS[j * N + i] * Qw[i * d + c];"),
    ("backward: dK from dO", "gk += dS[i * N + j] * Qw[i * d + c];", "gk += dS[i * N + j] * dOw[i * d + c];"),
    ("backward: dV from P untransposed", "gv += P[i * N + j] * dOw[i * d + c];",
     "gv += P[j * N + i] * dOw[i * d + c];"),
    ("backward: diagonal masked", "const int64_t visible = causal ? i + 1 : N;",
     "const int64_t visible = causal ? (i > 0 ? i : 1) : N;"),
    ("backward: dP from the keys", "for (int64_t c = 0; c < d; ++c) g += dOw[i * d + c] * Vw[j * d + c];",
     "for (int64_t c = 0; c < d; ++c) g += dOw[i * d + c] * Kw[j * d + c];"),
    ("gelu: the one half dropped", "const double g = 0.5 * h * (1.0 + tanh(", "const double g = h * (1.0 + tanh("),
    ("gelu: tanh sign", "const double g = 0.5 * h * (1.0 + tanh(", "const double g = 0.5 * h * (1.0 - tanh("),
    ("gelu: cubic term dropped", "(h + 0.044715 * h * h * h)", "(h)"),
    ("gelu: sqrt(2/pi) dropped", "tanh(k0 * (h + ", "tanh(1.0 * (h + "),
    ("bias indexed by row", "bf16_bits_to_f64(bias[c])", "bf16_bits_to_f64(bias[r % cols])"),
    ("mask bit order reversed", "(keep[e >> 5] >> (e & 31))", "(keep[e >> 5] >> (31 - (e & 31)))"),
    ("dropout scale inverted", "y[e] = kept ? g / (1.0 - p) : 0.0;", "y[e] = kept ? g * (1.0 - p) : 0.0;"),
    ("dropout keeps dropped values", "y[e] = kept ? g / (1.0 - p) : 0.0;", "y[e] = kept ? g / (1.0 - p) : g;"),
]


def test_planted_mistakes_are_caught(tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_ref.c")).read()
    # the unmodified source, compiled the same way, passes every pin
    clean = tmp_path / "clean.c"
    clean.write_text(src)
    orc = oracle.from_source(str(clean), str(tmp_path / "clean.so"))
    for pin in PINS:
        pin(orc)
    for n, (what, old, new) in enumerate(MUTANTS):
        assert src.count(old) == 1, f"mutation site not unique/found: {what}"
        path = tmp_path / f"m{n}.c"
        path.write_text(src.replace(old, new))
        mut = oracle.from_source(str(path), str(tmp_path / f"m{n}.so"))
        caught = []
        with np.errstate(all="ignore"):
            for pin in PINS:
                try:
                    pin(mut)
                except (AssertionError, RuntimeError, FloatingPointError, ValueError):
                    caught.append(pin.__name__)
        assert caught, f"no pin catches the planted mistake: {what}"
