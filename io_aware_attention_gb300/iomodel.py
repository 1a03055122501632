"""FLOP and HBM-byte model of the attention forward (host-side arithmetic).

These are the counts the benchmark divides by and the profiles compare the
measured DRAM traffic against.

* FLOPs: each score costs a d-long dot product (2d FLOPs) and each
  probability weights a d-long value row (2d FLOPs), so 4·N²·d per (batch,
  head); under the causal mask half of that is counted, the convention the
  metric is quoted in.
* Minimum bytes the method must move ("Kernels — fusion and FlashAttention"
  §4: HBM traffic of O(T·d) from streaming K, V once): Q, K, V read and O
  written once in bf16, plus one fp32 logsumexp per row.
* The standard (unfused) attention count of "Fusion and IO-aware kernels",
  section "FlashAttention" / "Code": Q, K, V and O once, plus four passes over
  the N×N score and probability matrices (write S, read S, write P, read P).
  Its printed program output pins both this count and the elementwise-chain
  count below.
* K/V re-reads: a query block of ``block_rows`` rows reads the K and V rows
  it attends to once, so each K and V element is read about N / block_rows
  times ("Fusion and IO-aware kernels", "Try it" 1).
"""
from __future__ import annotations

BF16 = 2
FP32 = 4


def attention_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """4·B·H·N²·d, halved under the causal mask."""
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f


def attention_min_bytes(B: int, H: int, N: int, d: int) -> int:
    """Q, K, V read once and O written once (bf16) + fp32 logsumexp per row."""
    return 4 * B * H * N * d * BF16 + B * H * N * FP32


def qkvo_bytes(seq: int, d: int, heads: int, batch: int, elem: int = BF16) -> int:
    """Q, K, V and O, each touched once."""
    return 4 * batch * heads * seq * d * elem


def standard_attention_bytes(seq: int, d: int, heads: int, batch: int, elem: int = BF16) -> int:
    """Unfused attention: Q, K, V, O once plus S written, S read, P written, P read."""
    score_matrix = batch * heads * seq * seq * elem
    return qkvo_bytes(seq, d, heads, batch, elem) + 4 * score_matrix


def elementwise_chain_bytes(n: int, ops: int, elem: int = BF16) -> tuple[int, int]:
    """(unfused, fused) bytes for a chain of ``ops`` elementwise ops on n values.

    Unfused, each op reads and writes the whole tensor; fused, the chain reads
    it once and writes it once.
    """
    one_round_trip = 2 * n * elem
    return ops * one_round_trip, one_round_trip


def kv_reread_bytes(B: int, H: int, N: int, d: int, block_rows: int, causal: bool) -> int:
    """K and V bytes read when every query block streams the K/V rows it needs.

    Non-causal: every block reads all N rows of K and V.  Causal: block i
    (rows [i·block_rows, (i+1)·block_rows)) reads rows [0, min(N, (i+1)·block_rows)).
    """
    nblk = -(-N // block_rows)
    rows = 0
    for i in range(nblk):
        rows += min(N, (i + 1) * block_rows) if causal else N
    return 2 * B * H * rows * d * BF16


def hbm_time_us(nbytes: float, bandwidth_bytes_per_s: float) -> float:
    return nbytes / bandwidth_bytes_per_s * 1e6
