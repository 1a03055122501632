"""The Python binding checks the caller's output tensors before any launch.

The C ABI sees only pointers and sizes, so an output tensor of the wrong
shape, dtype or device would be written out of bounds; the binding refuses it
with ValueError and nothing runs (the tensor keeps its contents).
"""
import pytest
import torch

import io_aware_attention_gb300 as fa

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 2, 130, 64


def _qkv():
    g = torch.Generator("cpu").manual_seed(5)
    return [torch.randn(B, H, N, D, generator=g).to(torch.bfloat16).cuda() for _ in range(3)]


def _untouched(t, fill):
    torch.cuda.synchronize()
    return bool((t.float() == fill).all())


@pytest.mark.parametrize("bad", ["o_shape", "o_dtype", "o_strided", "lse_shape", "lse_dtype", "o_cpu"])
def test_fwd_into_rejects_bad_outputs(bad):
    q, k, v = _qkv()
    o = torch.full((B, H, N, D), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, N), 3.0, dtype=torch.float32, device="cuda")
    if bad == "o_shape":
        o = torch.full((B, H, N - 1, D), 3.0, dtype=torch.bfloat16, device="cuda")
    elif bad == "o_dtype":
        o = torch.full((B, H, N, D), 3.0, dtype=torch.float16, device="cuda")
    elif bad == "o_strided":
        o = torch.full((B, H, D, N), 3.0, dtype=torch.bfloat16, device="cuda").transpose(2, 3)
    elif bad == "lse_shape":
        lse = torch.full((B * H * N,), 3.0, dtype=torch.float32, device="cuda")
    elif bad == "lse_dtype":
        lse = torch.full((B, H, N), 3.0, dtype=torch.float64, device="cuda")
    elif bad == "o_cpu":
        o = torch.full((B, H, N, D), 3.0, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd_into(q, k, v, o, lse, causal=True)
    assert _untouched(o, 3.0) and _untouched(lse, 3.0)


def test_fwd_into_accepts_a_contiguous_view():
    q, k, v = _qkv()
    buf = torch.zeros(B * H * N * D + 64, dtype=torch.bfloat16, device="cuda")
    o = buf[64:].view(B, H, N, D)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda")
    fa.fwd_into(q, k, v, o, lse, causal=False)
    o_ref, lse_ref = fa.fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("bad", ["o_shape", "lse_shape"])
def test_decode_into_rejects_bad_outputs(bad):
    g = torch.Generator("cpu").manual_seed(6)
    q = torch.randn(B, H, 1, D, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(B, H, 4096, D, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, H, 4096, D, generator=g).to(torch.bfloat16).cuda()
    o = torch.full((B, H, 1, D), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, 1), 3.0, dtype=torch.float32, device="cuda")
    if bad == "o_shape":
        o = torch.full((B, H, 2, D), 3.0, dtype=torch.bfloat16, device="cuda")
    else:
        lse = torch.full((B, H, 2), 3.0, dtype=torch.float32, device="cuda")
    nbytes = fa.decode_workspace_bytes(B, H, 1, 4096, D, True)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        fa.decode_into(q, k, v, o, lse, ws, causal=True)
    assert _untouched(o, 3.0) and _untouched(lse, 3.0)


def test_bwd_into_rejects_bad_lse_and_workspace():
    q, k, v = _qkv()
    o, lse = fa.fwd(q, k, v, causal=True)
    do = torch.randn_like(q, dtype=torch.float32).to(torch.bfloat16)
    dq, dk, dv = (torch.full_like(q, 3.0) for _ in range(3))
    ws = torch.empty(fa.bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        fa.bwd_into(q, k, v, o, lse.view(-1), do, dq, dk, dv, ws, causal=True)
    with pytest.raises(ValueError):
        fa.bwd_into(q, k, v, o, lse, do, dq, dk, dv, ws.cpu(), causal=True)
    assert _untouched(dq, 3.0) and _untouched(dk, 3.0) and _untouched(dv, 3.0)


def test_bias_gelu_dropout_rejects_a_bad_out():
    x = torch.ones(64, 256, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(256, dtype=torch.bfloat16, device="cuda")
    out = torch.full((64, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.bias_gelu_dropout(x, b, None, 0.0, out=out)
    assert _untouched(out, 3.0)
