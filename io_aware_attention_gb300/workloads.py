"""Seeded synthetic inputs for the attention forward.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both take their
inputs from it without sharing any of the method.

Every workload is (B, H, N, d) bf16 Q, K, V drawn i.i.d. N(0, 1) from
``torch.Generator('cpu').manual_seed(seed)`` in the order Q, K, V (fp32, then
rounded to bf16).  The rescale-stress workload also multiplies Q by 4 and
every 512th key row (0-based index j with j % 512 == 511) by 8; both factors
are powers of two, so they commute with the rounding to bf16.

The shapes follow the pages' running example ("Kernels — fusion and
FlashAttention" §2: B = 8, h = 32 heads, bf16, where a naive score matrix
takes 8.6 GB at T = 4096) and head sizes d in {64, 128} ("Writing and
Benchmarking Custom Kernels" §10.3.1 worked example: d_head = 128, 32 heads).
No public dataset is involved.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    q_mult: float = 1.0
    spike_every: int = 0       # every spike_every-th key row is multiplied ...
    spike_mult: float = 1.0    # ... by spike_mult
    sample_rows: int = 0       # rows compared with the oracle; 0 = the full tensor

    @property
    def shape(self):
        return (self.B, self.H, self.N, self.d)

    @property
    def scale(self) -> float:
        """1/sqrt(d) rounded to fp32, the value both sides are given."""
        return float(np.float32(1.0 / np.sqrt(self.d)))


WORKLOADS = {
    w.name: w
    for w in (
        Workload("b1_h2_n256_d64", 1, 2, 256, 64, False, 1001),
        Workload("b4_h16_n2048_d128_causal", 4, 16, 2048, 128, True, 1002),
        Workload("b8_h32_n4096_d128_causal", 8, 32, 4096, 128, True, 1003, sample_rows=512),
        Workload("b8_h32_n4096_d128", 8, 32, 4096, 128, False, 1006, sample_rows=512),
        Workload("b1_h32_n32768_d128_causal", 1, 32, 32768, 128, True, 1004, sample_rows=256),
        Workload("b16_h16_n8192_d64_spiky", 16, 16, 8192, 64, False, 1005, q_mult=4.0,
                 spike_every=512, spike_mult=8.0, sample_rows=512),
        # Sequence lengths that are not a multiple of the 128-row tile ("Writing
        # and Benchmarking Custom Kernels" §10.3.1: the final partial tile):
        # 4000 = 31 tiles + 32 rows, 4097 = 32 tiles + 1 row.
        Workload("b8_h32_n4000_d128_causal", 8, 32, 4000, 128, True, 1007, sample_rows=512),
        Workload("b8_h32_n4000_d128", 8, 32, 4000, 128, False, 1008, sample_rows=512),
        Workload("b8_h32_n4097_d128_causal", 8, 32, 4097, 128, True, 1009, sample_rows=512),
        Workload("b8_h32_n4097_d128", 8, 32, 4097, 128, False, 1010, sample_rows=512),
    )
}

# The workload the throughput line is quoted on: the pages' B = 8, h = 32
# example at T = 4096, d_head = 128, causal.
HEADLINE = "b8_h32_n4096_d128_causal"


def make_qkv(w: Workload, device="cpu"):
    """Seeded bf16 (Q, K, V) of shape (B, H, N, d), generated on the CPU."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = torch.randn(w.shape, generator=g, dtype=torch.float32)
    k = torch.randn(w.shape, generator=g, dtype=torch.float32)
    v = torch.randn(w.shape, generator=g, dtype=torch.float32)
    if w.q_mult != 1.0:
        q.mul_(w.q_mult)
    if w.spike_every:
        k[:, :, w.spike_every - 1 :: w.spike_every, :] *= w.spike_mult
    out = [t.to(torch.bfloat16) for t in (q, k, v)]
    del q, k, v
    if device != "cpu":
        out = [t.to(device) for t in out]
    return tuple(out)


def make_random_qkv(B, H, N, d, seed, q_mult=1.0, device="cpu"):
    """Seeded i.i.d. N(0,1) bf16 tensors of an arbitrary shape (test cases)."""
    return make_qkv(Workload("adhoc", B, H, N, d, False, seed, q_mult=q_mult), device)


def sample_rows(w: Workload, n: int | None = None):
    """Seeded (bh, row) pairs to compare with the oracle.

    Always holds the first row of the first head and the last row of the last
    head; the rest are drawn with ``numpy.random.default_rng(seed + 1)``.
    Returns two int64 arrays (bh index = b*H + h, query row).
    """
    n = w.sample_rows if n is None else n
    rng = np.random.default_rng(w.seed + 1)
    bh = rng.integers(0, w.B * w.H, size=n, dtype=np.int64)
    row = rng.integers(0, w.N, size=n, dtype=np.int64)
    if n >= 1:
        bh[0], row[0] = 0, 0
    if n >= 2:
        bh[1], row[1] = w.B * w.H - 1, w.N - 1
    return bh, row


# ----------------------------------------------------------------- decode
@dataclass(frozen=True)
class DecodeWorkload:
    """Nq query rows per (batch, head) against a cache of Nk keys.

    Drawn like :class:`Workload`: ``torch.Generator('cpu').manual_seed(seed)``,
    ``torch.randn`` in fp32 in the order Q (B, H, Nq, d), K, V (B, H, Nk, d),
    then rounded to bf16.
    """
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    sample_rows: int = 0  # rows compared with the oracle; 0 = all

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / np.sqrt(self.d)))


DECODE_WORKLOADS = {
    w.name: w
    for w in (
        # One new token per sequence against a 32k-token cache of the pages'
        # B = 8, h = 32, d_head = 128 model: 4.3 GB of K and V per step.
        DecodeWorkload("decode_b8_h32_nk32768_d128", 8, 32, 1, 32768, 128, False, 2001, sample_rows=64),
        DecodeWorkload("decode_b2_h4_nq4_nk1000_d64_causal", 2, 4, 4, 1000, 64, True, 2002),
    )
}


def make_decode_qkv(w: DecodeWorkload, device="cpu"):
    """Seeded bf16 q (B, H, Nq, d) and cache k, v (B, H, Nk, d)."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    q = torch.randn((w.B, w.H, w.Nq, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.H, w.Nk, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.H, w.Nk, w.d), generator=g, dtype=torch.float32)
    out = [t.to(torch.bfloat16) for t in (q, k, v)]
    del q, k, v
    if device != "cpu":
        out = [t.to(device) for t in out]
    return tuple(out)


def sample_decode_rows(w: DecodeWorkload, n: int | None = None):
    """Seeded (bh, query row) pairs, including the first and the last."""
    n = w.sample_rows if n is None else n
    rng = np.random.default_rng(w.seed + 1)
    bh = rng.integers(0, w.B * w.H, size=n, dtype=np.int64)
    row = rng.integers(0, w.Nq, size=n, dtype=np.int64)
    if n >= 1:
        bh[0], row[0] = 0, 0
    if n >= 2:
        bh[1], row[1] = w.B * w.H - 1, w.Nq - 1
    return bh, row


# ------------------------------------------------------- elementwise chain
@dataclass(frozen=True)
class EwWorkload:
    """A bias + GELU + dropout problem: x (rows, cols), bias (cols,), keep mask
    with keep probability 1 - p."""

    name: str
    rows: int
    cols: int
    p: float
    seed: int


EW_WORKLOADS = {
    w.name: w
    for w in [
        # "Fusion and IO-aware kernels", § Why elementwise chains are pure
        # traffic: the residual-stream activation (B, T, d) = (8, 4096, 4096)
        # in bf16 (268 MB), here with bias + GELU + dropout; larger than L2.
        EwWorkload("ew_b8_t4096_d4096_p0.1", 8 * 4096, 4096, 0.1, 3001),
        # the 4096 x 8192 activation of the page's fusion.py byte count
        EwWorkload("ew_4096x8192_p0.1", 4096, 8192, 0.1, 3002),
    ]
}


def make_ew_inputs(rows: int, cols: int, p: float, seed: int, device="cpu"):
    """Seeded x ~ N(0, 4) and bias ~ N(0, 1) in bf16, and a packed keep mask
    (uint32 words as int32, bit e % 32 of word e // 32 keeps flat element e,
    each kept with probability 1 - p) from numpy's default_rng(seed)."""
    import torch

    rng = np.random.default_rng(seed)
    x = torch.from_numpy((rng.standard_normal((rows, cols), dtype=np.float32) * 2.0)).to(torch.bfloat16)
    bias = torch.from_numpy(rng.standard_normal(cols, dtype=np.float32)).to(torch.bfloat16)
    n = rows * cols
    keep_bits = rng.random(((n + 31) // 32) * 32, dtype=np.float32) >= p
    words = np.packbits(keep_bits.reshape(-1, 8), axis=1, bitorder="little").reshape(-1).view(np.uint32)
    keep = torch.from_numpy(words.view(np.int32).copy())
    return x.to(device), bias.to(device), keep.to(device)
