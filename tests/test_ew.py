"""GPU parity of the fused bias + GELU + dropout chain (fa_bias_gelu_dropout)
with the fp64 oracle, element by element.

Tolerance, from the arithmetic: a dropped element is exactly 0 on both sides.
A kept one is computed in fp32 from the exact sum x + bias (two bf16 values
add exactly in fp32 at these magnitudes), through h / (1 + 2^z) with ex2.approx
(relative error 2^-22) and a fast division (2 ulp), then rounded to bf16
(relative half-ulp 2^-9); the exponent clamp at 2^64 changes only values
below 2^-64 |h|.  Every kept element must lie within 2^-8 |y| + 1e-12.
"""
import numpy as np
import pytest
import torch

import io_aware_attention_gb300 as fa
import oracle
from io_aware_attention_gb300.workloads import EW_WORKLOADS, make_ew_inputs

pytestmark = pytest.mark.gpu

RTOL = 2.0 ** -8
ATOL = 1e-12
GUARD = 64


def check(y, ref, keep_words, n, what):
    y = y.float().cpu().numpy().astype(np.float64).reshape(-1)
    ref = ref.reshape(-1)
    assert np.isfinite(y).all(), what
    if keep_words is not None:
        w = keep_words.cpu().numpy().view(np.uint32)
        bits = np.unpackbits(w.view(np.uint8), bitorder="little")[:n].astype(bool)
        assert (y[~bits] == 0).all() and (ref[~bits] == 0).all(), f"{what}: dropped element not zero"
    err = np.abs(y - ref)
    bound = RTOL * np.abs(ref) + ATOL
    worst = int(np.argmax(err / bound))
    assert (err <= bound).all(), f"{what}: element {worst}: {y[worst]!r} vs {ref[worst]!r}"


def run_guarded(x, b, keep, p):
    rows, cols = x.shape
    n = rows * cols
    buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.bfloat16, device=x.device)
    buf.view(torch.int16)[:GUARD] = 0x7FC1
    buf.view(torch.int16)[-GUARD:] = 0x7FC1
    y = buf[GUARD:GUARD + n].view(rows, cols)
    fa.bias_gelu_dropout(x, b, keep, p, out=y)
    torch.cuda.synchronize()
    bb = buf.view(torch.int16).cpu()
    assert (bb[:GUARD] == 0x7FC1).all() and (bb[-GUARD:] == 0x7FC1).all(), "guard band overwritten"
    return y


CASES = [  # (rows, cols, p, with mask)
    (1, 8, 0.0, False), (1, 8, 0.5, True), (3, 40, 0.25, True), (7, 24, 0.1, True), (33, 1000, 0.1, True),
    (128, 4096, 0.1, True), (2, 65536, 0.9, True), (1000, 8, 0.3, True), (5, 4104, 0.0, False), (17, 2056, 0.0, True),
]


@pytest.mark.parametrize("rows,cols,p,masked", CASES, ids=[f"{r}x{c}p{p}{'m' if m else ''}" for r, c, p, m in CASES])
def test_ew_parity(rows, cols, p, masked):
    x, b, keep = make_ew_inputs(rows, cols, p, 3100 + rows + cols)
    kw = keep if masked else None
    y = run_guarded(x.cuda(), b.cuda(), kw.cuda() if kw is not None else None, p)
    ref = oracle.bias_gelu_dropout(x, b, kw.numpy().view(np.uint32) if kw is not None else None, p)
    check(y, ref, kw, rows * cols, f"{rows}x{cols} p={p}")


def test_ew_extreme_inputs():
    """Large magnitudes: the GELU tails (y -> h, y -> 0 from below) and the
    exponent clamp."""
    vals = np.array([-60, -20, -9, -6.5, -3, -1e-3, 0, 1e-3, 3, 6.5, 9, 20, 60, 300, -300, 1e4], np.float32)
    x = torch.from_numpy(np.tile(vals, 8).reshape(8, 16)).to(torch.bfloat16)
    b = torch.zeros(16, dtype=torch.bfloat16)
    y = run_guarded(x.cuda(), b.cuda(), None, 0.0)
    ref = oracle.bias_gelu_dropout(x, b, None, 0.0)
    check(y, ref, None, 128, "extremes")


@pytest.mark.parametrize("name", sorted(EW_WORKLOADS))
def test_ew_workloads_full(name):
    w = EW_WORKLOADS[name]
    x, b, keep = make_ew_inputs(w.rows, w.cols, w.p, w.seed)
    y = fa.bias_gelu_dropout(x.cuda(), b.cuda(), keep.cuda(), w.p)
    torch.cuda.synchronize()
    ref = oracle.bias_gelu_dropout(x, b, keep.numpy().view(np.uint32), w.p)
    check(y, ref, keep, w.rows * w.cols, name)
