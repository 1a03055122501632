"""bench.py's roofline arithmetic on the host (no GPU): every fraction
recomputes from the block's own launch time, and the tighter of the tensor
and exponential bounds is the one named."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from io_aware_attention_gb300 import iomodel  # noqa: E402
from io_aware_attention_gb300.workloads import WORKLOADS  # noqa: E402

PEAKS = {"bf16_tflops": 1888.1, "bf16_tflops_sustained": 1712.9, "hbm_gbs": 6793.4}


def test_headline_roofline_fractions():
    w = WORKLOADS["b8_h32_n4096_d128_causal"]
    flops = iomodel.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    assert flops == 4 * 8 * 32 * 4096 ** 2 * 128 / 2
    ms = 0.87071
    roof = bench.tensor_roofline(w, flops, ms, PEAKS, "measured", {"sm_mhz": 2070.0}, 152, "k")
    achieved = flops / (ms * 1e-3) / 1e12
    assert roof["achieved"] == pytest.approx(achieved, abs=0.05)
    assert roof["frac"] == pytest.approx(achieved / 1888.1, abs=1e-4)
    assert roof["frac_of_sustained"] == pytest.approx(achieved / 1712.9, abs=1e-4)
    assert roof["frac_of_datasheet"] == pytest.approx(achieved / 2250.0, abs=1e-4)
    # d = 128: 1088 tensor cycles per 128 x 128 tile against 538 of ex2, so
    # the tensor core binds
    assert roof["binding"] == "tensor"
    assert roof["frac_of_binding"] == pytest.approx(roof["tensor_bound_ms"] / ms, abs=1e-3)


def test_exponential_bound():
    w = WORKLOADS["b16_h16_n8192_d64_spiky"]
    mufu = bench.mufu_bound(w, 5.0, 2000.0, 152)
    scores = 16 * 16 * 8192 ** 2
    rate = 152 * 4 * 32 / 4.2 * 2000e6
    assert mufu["scores_per_launch"] == scores
    assert mufu["bound_ms"] == pytest.approx(scores / rate * 1e3, rel=1e-4)
    assert mufu["frac"] == pytest.approx(mufu["bound_ms"] / 5.0, abs=1e-4)
    # causal halves the scores; no clock sample, no bound
    wc = WORKLOADS["b8_h32_n4096_d128_causal"]
    assert bench.mufu_bound(wc, 1.0, 2000.0, 152)["scores_per_launch"] == 8 * 32 * 4096 ** 2 / 2
    assert bench.mufu_bound(w, 5.0, None, 152) is None


def test_binding_bound_switches_with_the_clock():
    """At d = 64 the exponentials take almost as long as the tensor work: at a
    low enough SM clock they bind instead."""
    w = WORKLOADS["b16_h16_n8192_d64_spiky"]
    flops = iomodel.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    fast = bench.tensor_roofline(w, flops, 5.0, PEAKS, "measured", {"sm_mhz": 2070.0}, 152, "k")
    slow = bench.tensor_roofline(w, flops, 5.0, PEAKS, "measured", {"sm_mhz": 1000.0}, 152, "k")
    assert fast["binding"] == "tensor" and slow["binding"] == "mufu"
    assert slow["frac_of_binding"] == pytest.approx(slow["mufu"]["bound_ms"] / 5.0, abs=1e-3)


def test_executed_tensor_work():
    """The forward executes whole tiles and the l~ columns: at the headline
    (d = 128, N = 4096 causal) 1 + 8/128 for the ones block times 33/32 for
    the diagonal tiles over the algorithmic count; non-causal d = 64 only the
    ones block (1 + 8/64); a padded head size counts the padded columns."""
    w = WORKLOADS["b8_h32_n4096_d128_causal"]
    flops = iomodel.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    assert bench.executed_flops(w) / flops == pytest.approx((1 + 8 / 128) * 33 / 32, rel=1e-12)
    w64 = WORKLOADS["b16_h16_n8192_d64_spiky"]
    assert bench.executed_flops(w64) / iomodel.attention_flops(w64.B, w64.H, w64.N, w64.d, w64.causal) == \
        pytest.approx(1 + 8 / 64, rel=1e-12)
    from io_aware_attention_gb300.workloads import Workload
    w40 = Workload("d40", 1, 1, 256, 40, False, 1)
    assert bench.executed_flops(w40) == 1 * 1 * 4 * 2 * 128 * 128 * (2 * 64 + 16)
    roof = bench.tensor_roofline(w, flops, 0.8, PEAKS, "measured", {"sm_mhz": 2070.0}, 152, "k")
    assert roof["executed_over_algorithmic"] == pytest.approx(1.0957, abs=1e-4)
    assert roof["executed_frac"] == pytest.approx(bench.executed_flops(w) / 0.8e-3 / 1e12 / 1888.1, abs=1e-4)
