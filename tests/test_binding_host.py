"""Host-side logic of the Python binding (CPU only, no library loaded).

The binding checks the call's tensors in one pass (_fast_ok) and falls back
to the detailed checks, which name the problem, when that pass fails; a
tensor that is not a CUDA tensor is refused before the C library is even
loaded, so nothing is launched.
"""
import pytest
import torch

import io_aware_attention_gb300 as fa


def _t(shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def test_fast_check_accepts_only_matching_tensors():
    s = (1, 2, 8, 16)
    a, b = _t(s), _t(s)
    dev = a.get_device()  # -1 on the CPU
    assert fa._fast_ok(dev, a.shape, torch.bfloat16, a, b)
    assert not fa._fast_ok(dev, a.shape, torch.bfloat16, a, _t((1, 2, 8, 8)))         # shape
    assert not fa._fast_ok(dev, a.shape, torch.bfloat16, a, _t(s, torch.float16))     # dtype
    assert not fa._fast_ok(dev, a.shape, torch.bfloat16, a, _t((1, 2, 16, 8)).transpose(2, 3))  # strides
    assert not fa._fast_ok(0, a.shape, torch.bfloat16, a, b)                          # device


def test_stream_handle_of_an_explicit_stream():
    class FakeStream:
        cuda_stream = 0x1234
    assert fa._stream_handle(FakeStream()) == 0x1234


@pytest.mark.parametrize("call", ["fwd", "fwd_into", "bias_gelu_dropout"])
def test_cpu_tensors_are_refused_before_the_library_loads(call, monkeypatch):
    def no_library():
        raise AssertionError("the library was loaded for a call that must be refused")
    monkeypatch.setattr(fa, "library", no_library)
    s = (1, 2, 8, 16)
    q, k, v = _t(s), _t(s), _t(s)
    with pytest.raises(ValueError):
        if call == "fwd":
            fa.fwd(q, k, v)
        elif call == "fwd_into":
            fa.fwd_into(q, k, v, _t(s), _t(s[:3], torch.float32))
        else:
            fa.bias_gelu_dropout(_t((4, 16)), _t((16,)))
