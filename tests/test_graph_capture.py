"""The library's calls captured in a CUDA graph and replayed.

A serving loop captures its step once and replays it.  The forward, decode
and elementwise kernels are launched as programmatic dependents (their
launch attribute becomes a programmatic edge of the graph), the backward's
kernels plainly.  One graph holds a chain of calls that read one another's
outputs; each replay, on new inputs copied into the captured buffers, must
give the same bits as the same calls made eagerly.  (The first call on a
device does one-time set-up, so every call runs once before capture.)
"""
import pytest
import torch

import io_aware_attention_gb300 as fa
from io_aware_attention_gb300.workloads import make_ew_inputs, make_random_qkv

pytestmark = pytest.mark.gpu

B, H, N, D = 2, 4, 1000, 128
NQ = 4  # decode query rows


def _buffers():
    q, k, v = (torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    do = torch.empty_like(q)
    x = torch.empty(512, 1024, dtype=torch.bfloat16, device="cuda")
    bias = torch.empty(1024, dtype=torch.bfloat16, device="cuda")
    keep = torch.empty((512 * 1024 + 31) // 32, dtype=torch.int32, device="cuda")
    return dict(q=q, k=k, v=v, do=do, x=x, bias=bias, keep=keep)


def _fill(buf, seed):
    q, k, v = make_random_qkv(B, H, N, D, seed)
    do = make_random_qkv(B, H, N, D, seed + 1)[0]
    x, bias, keep = make_ew_inputs(512, 1024, 0.1, seed + 2)
    for name, t in dict(q=q, k=k, v=v, do=do, x=x, bias=bias, keep=keep).items():
        buf[name].copy_(t)


def _outputs():
    o = torch.empty(B, H, N, D, dtype=torch.bfloat16, device="cuda")
    return dict(
        o=o, lse=torch.empty(B, H, N, device="cuda"), o2=torch.empty_like(o), lse2=torch.empty(B, H, N, device="cuda"),
        dq=torch.empty_like(o), dk=torch.empty_like(o), dv=torch.empty_like(o),
        ws=torch.empty(fa.bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8, device="cuda"),
        od=torch.empty(B, H, NQ, D, dtype=torch.bfloat16, device="cuda"), ld=torch.empty(B, H, NQ, device="cuda"),
        dws=torch.empty(max(fa.decode_workspace_bytes(B, H, NQ, N, D, True), 16), dtype=torch.uint8, device="cuda"),
        y=torch.empty(512, 1024, dtype=torch.bfloat16, device="cuda"))


def _step(i, out):
    """forward -> forward on its output -> backward -> decode of the first
    output's last rows -> the elementwise chain."""
    fa.fwd_into(i["q"], i["k"], i["v"], out["o"], out["lse"], causal=True)
    fa.fwd_into(out["o"], i["k"], i["v"], out["o2"], out["lse2"], causal=False)
    fa.bwd_into(i["q"], i["k"], i["v"], out["o"], out["lse"], i["do"], out["dq"], out["dk"], out["dv"], out["ws"],
                causal=True)
    fa.decode_into(out["o"][:, :, -NQ:].contiguous(), i["k"], i["v"], out["od"], out["ld"], out["dws"], causal=True)
    fa.bias_gelu_dropout(i["x"], i["bias"], i["keep"], 0.1, out=out["y"])


def test_captured_chain_replays_like_eager_calls():
    buf, out = _buffers(), _outputs()
    _fill(buf, 41000)
    _step(buf, out)  # one-time set-up of every kernel before capture
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            _step(buf, out)
    torch.cuda.current_stream().wait_stream(side)

    for seed in (42000, 43000):
        _fill(buf, seed)
        eager = _outputs()
        _step(buf, eager)
        torch.cuda.synchronize()
        for t in out.values():
            t.fill_(0) if t.dtype == torch.uint8 else t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert fa.check_device_status() == 0
        for name in ("o", "lse", "o2", "lse2", "dk", "dv", "od", "ld", "y"):
            assert torch.equal(out[name], eager[name]), f"{name} differs between the replay and eager calls"
        # dQ is summed by reduce-adds in L2 in no fixed order: within rounding
        a, b = out["dq"].float(), eager["dq"].float()
        assert not torch.isnan(a).any() and ((a - b).abs() <= 2.0 ** -6 * b.abs() + 1e-3).all()
