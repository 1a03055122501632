"""Launches that feed one another on one stream, with no synchronisation in
between.

The forward, decode and elementwise kernels are launched as programmatic
dependents of the kernel before them on the stream: their blocks may start
while that kernel's last blocks still run, and must read and write device
memory only after it has completed (griddepcontrol.wait).  Each chain here
makes a call consume what the call just before it wrote -- the consumer's
output buffers filled with NaN beforehand -- and is compared bit for bit with
the same chain synchronised after every call (each call alone is checked
against the oracle by the other tests).  A read of a buffer before its
producer finished would show as NaN or as different bits.
"""
import pytest
import torch

import io_aware_attention_gb300 as fa
from io_aware_attention_gb300.workloads import make_ew_inputs, make_random_qkv

pytestmark = pytest.mark.gpu


def _nan_like(t):
    return torch.full_like(t, float("nan"))


def _fwd_chain(q, k, v, steps, causal, sync):
    """o_1 = attn(q, k, v); o_{i+1} = attn(o_i, k, v): each call reads the
    previous call's output as its queries."""
    outs = []
    x = q
    for _ in range(steps):
        o, lse = _nan_like(q), torch.full(q.shape[:3], float("nan"), device=q.device)
        fa.fwd_into(x, k, v, o, lse, causal=causal)
        if sync:
            torch.cuda.synchronize()
        outs.append((o, lse))
        x = o
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("shape,causal", [((8, 32, 2048, 128), True), ((2, 4, 1000, 64), False),
                                          ((1, 2, 300, 96), True)],
                         ids=["b8h32n2048d128c", "b2h4n1000d64", "b1h2n300d96c"])
def test_forward_chain(shape, causal):
    B, H, N, d = shape
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 31000 + N))
    ref = _fwd_chain(q, k, v, 4, causal, sync=True)
    got = _fwd_chain(q, k, v, 4, causal, sync=False)
    assert fa.check_device_status() == 0
    for i, ((o, l), (o_r, l_r)) in enumerate(zip(got, ref)):
        assert not torch.isnan(o).any() and not torch.isnan(l).any(), f"step {i}: unwritten or stale output"
        assert torch.equal(o, o_r) and torch.equal(l, l_r), f"step {i} differs from the synchronised chain"


def test_large_forward_then_small_consumer():
    """A long launch, then a small one that reads its last head -- among the
    last rows the long launch writes -- as queries: the small launch's blocks
    are started while the long one's last blocks still run."""
    q, k, v = (t.cuda() for t in make_random_qkv(8, 32, 4096, 128, 31100))
    ks, vs = k[7:8, 31:32], v[7:8, 31:32]  # contiguous slices: the last head
    o, lse = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    o_ref, l_ref = fa.fwd(o[7:8, 31:32], ks, vs, causal=False)
    torch.cuda.synchronize()
    big_o, big_l = _nan_like(o), torch.full_like(lse, float("nan"))
    out2, l2 = _nan_like(o_ref), torch.full_like(l_ref, float("nan"))
    fa.fwd_into(q, k, v, big_o, big_l, causal=True)
    fa.fwd_into(big_o[7:8, 31:32], ks, vs, out2, l2, causal=False)
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    assert torch.equal(big_o, o) and torch.equal(big_l, lse)
    assert torch.equal(out2, o_ref) and torch.equal(l2, l_ref)


def test_forward_then_decode_then_forward():
    """decode's queries are the forward's last output rows; the next forward's
    keys include decode's output."""
    B, H, N, d = 2, 8, 3000, 128
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 31200))

    def chain(sync):
        o, lse = _nan_like(q), torch.full((B, H, N), float("nan"), device="cuda")
        fa.fwd_into(q, k, v, o, lse, causal=True)
        if sync:
            torch.cuda.synchronize()
        qd = o[:, :, -4:].contiguous()
        od, ld = fa.decode(qd, k, v, causal=True)
        if sync:
            torch.cuda.synchronize()
        k2 = torch.cat([k[:, :, :-4], od], dim=2).contiguous()
        o2, l2 = _nan_like(q), torch.full((B, H, N), float("nan"), device="cuda")
        fa.fwd_into(q, k2, v, o2, l2, causal=False)
        torch.cuda.synchronize()
        return o, lse, od, ld, o2, l2

    ref = chain(True)
    got = chain(False)
    assert fa.check_device_status() == 0
    for i, (a, b) in enumerate(zip(got, ref)):
        assert not torch.isnan(a).any(), f"output {i}: unwritten or stale"
        assert torch.equal(a, b), f"output {i} differs from the synchronised chain"


def test_elementwise_chain():
    """y_1 = f(x), y_{i+1} = f(y_i): each launch reads the previous one's
    output."""
    rows, cols = 8192, 4096
    x, bias, keep = make_ew_inputs(rows, cols, 0.1, 31300, device="cuda")

    def chain(sync):
        outs, cur = [], x
        for _ in range(5):
            y = _nan_like(x)
            fa.bias_gelu_dropout(cur, bias, keep, 0.1, out=y)
            if sync:
                torch.cuda.synchronize()
            outs.append(y)
            cur = y
        torch.cuda.synchronize()
        return outs

    ref = chain(True)
    got = chain(False)
    for i, (a, b) in enumerate(zip(got, ref)):
        assert not torch.isnan(a).any() and torch.equal(a, b), f"step {i}"


def test_forward_backward_forward():
    """The backward's plain launches after a programmatic forward, and a
    programmatic forward after the backward, reading its dQ.  dQ is summed by
    reduce-adds in L2, whose order varies, so dQ and the forward that reads
    it are compared within a tolerance; everything else to the bit."""
    B, H, N, d = 2, 4, 1000, 128
    q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, 31400))
    do = make_random_qkv(B, H, N, d, 31401)[0].cuda()

    def chain(sync):
        o, lse = _nan_like(q), torch.full((B, H, N), float("nan"), device="cuda")
        fa.fwd_into(q, k, v, o, lse, causal=True)
        if sync:
            torch.cuda.synchronize()
        dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
        if sync:
            torch.cuda.synchronize()
        o2, l2 = _nan_like(q), torch.full((B, H, N), float("nan"), device="cuda")
        fa.fwd_into(dq, k, v, o2, l2, causal=True)
        torch.cuda.synchronize()
        return o, lse, dq, dk, dv, o2, l2

    ref = chain(True)
    got = chain(False)
    assert fa.check_device_status() == 0
    names = ["o", "lse", "dq", "dk", "dv", "o2", "lse2"]
    for name, a, b in zip(names, got, ref):
        assert not torch.isnan(a).any(), f"{name}: unwritten or stale"
        if name in ("dq", "o2", "lse2"):
            a, b = a.float(), b.float()
            assert ((a - b).abs() <= 2.0 ** -6 * b.abs() + 1e-3).all(), f"{name} differs from the synchronised chain"
        else:
            assert torch.equal(a, b), f"{name} differs from the synchronised chain"


def test_concurrent_streams_and_host_threads():
    """Two host threads, each on its own stream with its own inputs, call the
    forward and the decode in a loop at the same time (the tensor-map cache
    is per host thread, the device status word shared): every result equals
    the same call made alone."""
    import threading

    shapes = [(2, 8, 2048, 128, True, 32000), (4, 4, 1000, 64, False, 33000)]
    data, ref = [], []
    for B, H, N, d, causal, seed in shapes:
        q, k, v = (t.cuda() for t in make_random_qkv(B, H, N, d, seed))
        data.append((q, k, v, causal))
        o, lse = fa.fwd(q, k, v, causal=causal)
        od, ld = fa.decode(q[:, :, -2:].contiguous(), k, v, causal=True)
        ref.append((o, lse, od, ld))
    torch.cuda.synchronize()
    errors = []

    def worker(idx):
        try:
            q, k, v, causal = data[idx]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                qd = q[:, :, -2:].contiguous()
                for _ in range(20):
                    o, lse = fa.fwd(q, k, v, causal=causal)
                    od, ld = fa.decode(qd, k, v, causal=True)
                s.synchronize()
            r = ref[idx]
            if not (torch.equal(o, r[0]) and torch.equal(lse, r[1]) and torch.equal(od, r[2]) and torch.equal(ld, r[3])):
                errors.append(f"thread {idx}: results differ")
        except Exception as e:  # reported below
            errors.append(f"thread {idx}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert fa.check_device_status() == 0
