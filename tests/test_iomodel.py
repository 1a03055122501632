"""The byte/FLOP model against the numbers the pages print.

Golden values: tests/golden/fusion_bytes.txt, the printed run of the byte
counter on "Fusion and IO-aware kernels" (section "Code").  The model must
reproduce every printed figure at the page's rounding.
"""
import os

import pytest

from io_aware_attention_gb300 import iomodel

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fusion_bytes.txt")
PAGE_HBM = 3.35e12  # the page's H100 model bandwidth, B/s


def _rows(kind):
    out = []
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if line and line[0] == kind:
            out.append(line[1:])
    return out


def test_golden_file_has_all_rows():
    assert len(_rows("chain")) == 2 and len(_rows("attention")) == 3


@pytest.mark.parametrize("row", _rows("chain"))
def test_elementwise_chain_matches_page(row):
    ops, u_mb, u_us, f_mb, f_us, ratio = row
    n = 4096 * 8192
    u, f = iomodel.elementwise_chain_bytes(n, int(ops))
    assert f"{u / 1e6:.0f}" == u_mb
    assert f"{f / 1e6:.0f}" == f_mb
    assert f"{iomodel.hbm_time_us(u, PAGE_HBM):.0f}" == u_us
    assert f"{iomodel.hbm_time_us(f, PAGE_HBM):.0f}" == f_us
    assert f"{u / f:.1f}" == ratio


@pytest.mark.parametrize("row", _rows("attention"))
def test_attention_bytes_match_page(row):
    seq, std_gb, io_gb, ratio = row
    s = iomodel.standard_attention_bytes(int(seq), 128, 32, 1)
    f = iomodel.qkvo_bytes(int(seq), 128, 32, 1)
    assert f"{s / 1e9:.2f}" == std_gb
    assert f"{f / 1e9:.2f}" == io_gb
    assert f"{s / f:.1f}" == ratio


def test_score_matrix_of_the_running_example():
    # "Kernels — fusion and FlashAttention" §2: B = 8, h = 32, T = 4096, bf16
    # score matrix ~ 8.6 GB (the printed formula is lost; B·h·T²·2 gives it).
    assert round(8 * 32 * 4096 * 4096 * 2 / 1e9, 1) == 8.6


def test_flops_and_min_bytes():
    assert iomodel.attention_flops(1, 1, 4, 2, False) == 4 * 16 * 2
    assert iomodel.attention_flops(1, 1, 4, 2, True) == 4 * 16 * 2 / 2
    # B8 H32 N4096 d128 causal: 1099.5 GFLOP
    assert round(iomodel.attention_flops(8, 32, 4096, 128, True) / 1e9, 1) == 1099.5
    assert iomodel.attention_min_bytes(1, 1, 10, 4) == 4 * 10 * 4 * 2 + 10 * 4


def test_kv_reread():
    # non-causal: every one of N/128 blocks reads all of K and V
    assert iomodel.kv_reread_bytes(1, 1, 1024, 128, 128, False) == 8 * 2 * 1024 * 128 * 2
    # causal: block i reads (i+1)*128 rows; ragged last block reads N rows
    assert iomodel.kv_reread_bytes(1, 1, 300, 8, 128, True) == 2 * (128 + 256 + 300) * 8 * 2
