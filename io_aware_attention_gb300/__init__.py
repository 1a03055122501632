"""GB300 (sm_103a) IO-aware attention: Python binding of the C ABI in include/fa.h.

Only argument marshalling happens here; every step of the computation runs in
the CUDA kernels of ``libfa_gb300.so``.  There is no fallback: if the library
is missing or the device is not sm_103, calls raise.

    o, lse = io_aware_attention_gb300.fwd(q, k, v, causal=True)

q, k, v: CUDA bf16 tensors of shape (B, H, N, d), contiguous, d a multiple of
8 from 8 to 128.
Returns o (bf16, same shape) and lse (fp32, (B, H, N)), the natural-log
logsumexp of each row's scaled, masked scores.

    dq, dk, dv = io_aware_attention_gb300.bwd(q, k, v, o, lse, do, causal=True)

gives the gradients for the output gradient ``do`` (the same head sizes),
recomputing the probabilities from ``lse``.

    o, lse = io_aware_attention_gb300.decode(q, k_cache, v_cache, causal=True)

is split-KV decode of up to 8 query rows against a long cache (the same head
sizes).

    y = io_aware_attention_gb300.bias_gelu_dropout(x, bias, keep, p)

is the fused elementwise chain (bias add, tanh GELU, dropout with a packed
keep mask drawn by the caller) in one HBM read and one write.

The ``*_into`` forms write into caller-provided tensors; their shapes, dtypes
and devices are checked here, because the C ABI sees only pointers and sizes.
Work is enqueued on ``stream``, by default the current stream, of the current
CUDA device, which must be the tensors' device (``fwd``, ``bwd`` and
``decode`` switch to it themselves).  The checks of a ``fwd_into`` call take
one pass over its tensors (a few microseconds of host time per call).
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

__all__ = ["fwd", "fwd_into", "bwd", "bwd_into", "bwd_workspace_bytes", "bias_gelu_dropout", "decode", "decode_into", "decode_workspace_bytes", "check_device_status", "get_device_status",
           "set_wait_limit_ns", "debug_skip_k_tile", "debug_set_schedule", "FaError", "library", "library_path", "version", "STATUS"]

STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
          4: "FA_ERR_TIMEOUT", 5: "FA_ERR_TOO_LARGE"}
EXPORTS = ["fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_bias_gelu_dropout", "fa_decode", "fa_decode_workspace_bytes", "fa_decode_static", "fa_check_device_status", "fa_get_device_status",
           "fa_set_wait_limit_ns", "fa_debug_skip_k_tile", "fa_debug_set_schedule", "fa_debug_decode_plan", "fa_status_string",
           "fa_version"]


class FaError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        self.name = STATUS.get(code, f"status {code}")
        super().__init__(f"{what}: {self.name}" if what else self.name)


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def library():
    """Load ``libfa_gb300.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as "
                           "g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float, vp]
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                           vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_int
    lib.fa_bias_gelu_dropout.argtypes = [vp, vp, vp, vp, i64, i64, ctypes.c_float, vp]
    lib.fa_bias_gelu_dropout.restype = ctypes.c_int
    lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float, vp,
                              ctypes.c_size_t, vp]
    lib.fa_decode.restype = ctypes.c_int
    lib.fa_decode_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_size_t)]
    lib.fa_decode_workspace_bytes.restype = ctypes.c_int
    lib.fa_decode_static.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_float,
                                     vp]
    lib.fa_decode_static.restype = ctypes.c_int
    lib.fa_check_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.fa_check_device_status.restype = ctypes.c_int
    lib.fa_get_device_status.argtypes = [vp]
    lib.fa_get_device_status.restype = ctypes.c_int
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.fa_set_wait_limit_ns.restype = ctypes.c_int
    lib.fa_debug_skip_k_tile.argtypes = [ctypes.c_int]
    lib.fa_debug_skip_k_tile.restype = ctypes.c_int
    lib.fa_debug_set_schedule.argtypes = [ctypes.c_int]
    lib.fa_debug_set_schedule.restype = ctypes.c_int
    lib.fa_debug_decode_plan.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int)]
    lib.fa_debug_decode_plan.restype = ctypes.c_int
    lib.fa_status_string.argtypes = [ctypes.c_int]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = ctypes.c_int
    _lib = lib
    return lib


def version() -> int:
    return int(library().fa_version())


def _stream_handle(stream, device: int | None = None):
    """The raw cudaStream_t of ``stream`` as an int, else the current stream
    of ``device`` (default: the current device)."""
    import torch

    if stream is not None:
        return int(stream.cuda_stream)
    if device is None:
        device = torch.cuda.current_device()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return int(raw(device))
    return int(torch.cuda.current_stream(device).cuda_stream)


def _on_current_device(dev: int) -> None:
    """The C entry points launch on the calling thread's current device, so
    the tensors must live there."""
    import torch

    cur = torch.cuda.current_device()
    if dev != cur:
        raise ValueError(f"tensors are on cuda:{dev} but the current device is cuda:{cur}: "
                         f"call under torch.cuda.device({dev})")


def _fast_ok(dev: int, shape, dtype, *ts) -> bool:
    """One pass over tensors that must all be contiguous, of this dtype and
    shape, on CUDA device dev (the common case; any failure is reported by
    the detailed checks)."""
    for t in ts:
        if t.get_device() != dev or t.dtype is not dtype or t.shape != shape or not t.is_contiguous():
            return False
    return True


def _check(q, k, v):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bf16, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.dim() != 4:
            raise ValueError(f"{name} must be (B, H, N, d), got shape {tuple(t.shape)}")
    if not (q.shape == k.shape == v.shape):
        raise ValueError(f"q, k, v shapes differ: {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")


def _check_out(name, t, shape, dtype, device):
    """An output tensor the kernels write: CUDA, contiguous, of exactly this
    shape and dtype, on the inputs' device."""
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def fwd_into(q, k, v, o, lse, causal: bool = False, scale: float | None = None, stream=None):
    """Runs the kernel into caller-provided ``o`` (bf16, the shape of q) and
    ``lse`` (fp32, (B, H, N))."""
    import torch

    shape = q.shape
    dev = q.get_device()
    if not (dev >= 0 and len(shape) == 4 and _fast_ok(dev, shape, torch.bfloat16, q, k, v, o)
            and lse.get_device() == dev and lse.dtype is torch.float32 and lse.shape == shape[:3]
            and lse.is_contiguous()):
        _check(q, k, v)
        _check_out("o", o, q.shape, torch.bfloat16, q.device)
        _check_out("lse", lse, tuple(q.shape[:3]), torch.float32, q.device)
    _on_current_device(dev)
    B, H, N, d = shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                          1 if causal else 0, float(scale), _stream_handle(stream, dev))
    if rc != 0:
        raise FaError(rc, "fa_fwd")
    return o, lse


def fwd(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Attention forward; returns ``(o, lse)`` (see module docstring)."""
    import torch

    _check(q, k, v)
    B, H, N, d = (int(s) for s in q.shape)
    with torch.cuda.device(q.device):
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        return fwd_into(q, k, v, o, lse, causal, scale, stream)


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    """Workspace bytes fa_bwd needs for these sizes."""
    out = ctypes.c_size_t(0)
    rc = library().fa_bwd_workspace_bytes(int(B), int(H), int(N), int(d), ctypes.byref(out))
    if rc != 0:
        raise FaError(rc, "fa_bwd_workspace_bytes")
    return int(out.value)


def bwd_into(q, k, v, o, lse, do, dq, dk, dv, workspace, causal: bool = False, scale: float | None = None,
             stream=None):
    """Backward into caller-provided dq, dk, dv (bf16) and workspace (a CUDA
    tensor of at least bwd_workspace_bytes bytes)."""
    import torch

    _check(q, k, v)
    _check(o, do, dq)
    _check(dk, dv, dq)
    if not (q.shape == o.shape == do.shape == dq.shape):
        raise ValueError("o, do, dq, dk, dv must have the shape of q")
    B, H, N, d = (int(s) for s in q.shape)
    if not (q.device == o.device == do.device == dq.device == dk.device == dv.device):
        raise ValueError("q, k, v, o, do, dq, dk, dv must be on one device")
    _check_out("lse", lse, (B, H, N), torch.float32, q.device)
    if not workspace.is_cuda or workspace.device != q.device or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor on the inputs' device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws_bytes = workspace.numel() * workspace.element_size()
    dev = q.get_device()
    _on_current_device(dev)
    vp = ctypes.c_void_p
    rc = library().fa_bwd(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
                          vp(lse.data_ptr()), vp(do.data_ptr()), vp(dq.data_ptr()), vp(dk.data_ptr()),
                          vp(dv.data_ptr()), B, H, N, d, int(bool(causal)), float(scale), vp(workspace.data_ptr()),
                          ws_bytes, _stream_handle(stream, dev))
    if rc != 0:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def bwd(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, stream=None):
    """Gradients ``(dq, dk, dv)`` of the attention forward (o, lse from
    :func:`fwd` with the same causal and scale) for the output gradient do."""
    import torch

    _check(q, k, v)
    B, H, N, d = (int(s) for s in q.shape)
    with torch.cuda.device(q.device):
        ws = torch.empty(bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        return bwd_into(q, k, v, o, lse, do, dq, dk, dv, ws, causal, scale, stream)


def bias_gelu_dropout(x, bias, keep=None, p: float = 0.0, out=None, stream=None):
    """y = dropout(gelu(x + bias)) for x (rows, cols) bf16 and bias (cols,) bf16
    on the GPU; keep: int32/uint32 CUDA tensor of ceil(rows*cols/32) words of
    keep bits (bit e % 32 of word e // 32 keeps flat element e), or None to
    keep all; kept values are scaled by 1/(1-p).  Returns y (bf16, like x)."""
    import torch

    for name, t in (("x", x), ("bias", bias)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor")
    if x.dim() != 2 or bias.shape != (x.shape[1],):
        raise ValueError(f"x (rows, cols) and bias (cols,) expected: {tuple(x.shape)} {tuple(bias.shape)}")
    rows, cols = (int(s) for s in x.shape)
    if keep is not None:
        if not keep.is_cuda or keep.dtype not in (torch.int32, torch.uint32) or not keep.is_contiguous():
            raise ValueError("keep must be a contiguous CUDA int32/uint32 tensor of mask words")
        if keep.numel() * 32 < rows * cols:
            raise ValueError("keep holds fewer bits than x has elements")
    if (keep is not None and keep.device != x.device) or bias.device != x.device:
        raise ValueError("x, bias and keep must be on one device")
    if out is not None:
        _check_out("out", out, x.shape, torch.bfloat16, x.device)
    dev = x.get_device()
    _on_current_device(dev)
    y = torch.empty_like(x) if out is None else out
    vp = ctypes.c_void_p
    rc = library().fa_bias_gelu_dropout(vp(x.data_ptr()), vp(bias.data_ptr()),
                                        vp(keep.data_ptr() if keep is not None else 0), vp(y.data_ptr()), rows,
                                        cols, float(p), _stream_handle(stream, dev))
    if rc != 0:
        raise FaError(rc, "fa_bias_gelu_dropout")
    return y


def _check_decode(q, k, v):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous CUDA bf16 (B, H, N, d) tensor")
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError(f"q (B, H, Nq, d) and k, v (B, H, Nk, d) expected: {tuple(q.shape)} {tuple(k.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")


def decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool = False) -> int:
    """Workspace bytes fa_decode needs for these sizes on the current device."""
    out = ctypes.c_size_t(0)
    rc = library().fa_decode_workspace_bytes(int(B), int(H), int(Nq), int(Nk), int(d), int(bool(causal)),
                                             ctypes.byref(out))
    if rc != 0:
        raise FaError(rc, "fa_decode_workspace_bytes")
    return int(out.value)


def decode_into(q, k, v, o, lse, workspace, causal: bool = False, scale: float | None = None, stream=None):
    """Decode attention into caller-provided o (bf16, the shape of q), lse
    (fp32, (B, H, Nq)) and workspace (a CUDA tensor of at least
    decode_workspace_bytes bytes, or None when that is 0)."""
    import torch

    _check_decode(q, k, v)
    B, H, Nq, d = (int(s) for s in q.shape)
    Nk = int(k.shape[2])
    _check_out("o", o, q.shape, torch.bfloat16, q.device)
    _check_out("lse", lse, (B, H, Nq), torch.float32, q.device)
    if workspace is not None and (not workspace.is_cuda or workspace.device != q.device
                                  or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on the inputs' device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q.get_device()
    _on_current_device(dev)
    ws_ptr = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = library().fa_decode(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                             ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                             ctypes.c_void_p(lse.data_ptr()), B, H, Nq, Nk, d, int(bool(causal)), float(scale),
                             ws_ptr, ws_bytes, _stream_handle(stream, dev))
    if rc != 0:
        raise FaError(rc, "fa_decode")
    return o, lse


def decode(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Attention of q (B, H, Nq, d), Nq <= 8, against the cache k, v
    (B, H, Nk, d); query i stands at key position Nk - Nq + i.  Returns
    ``(o (B, H, Nq, d) bf16, lse (B, H, Nq) fp32)``."""
    import torch

    _check_decode(q, k, v)
    B, H, Nq, d = (int(s) for s in q.shape)
    with torch.cuda.device(q.device):
        nbytes = decode_workspace_bytes(B, H, Nq, int(k.shape[2]), d, causal)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if nbytes else None
        o = torch.empty_like(q)
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
        return decode_into(q, k, v, o, lse, ws, causal, scale, stream)


def check_device_status(stream=None) -> int:
    """Synchronises the stream and returns the device status (0 = ok, 4 = a wait
    timed out); raises FaError on a CUDA error."""
    where = ctypes.c_uint32(0)
    rc = library().fa_check_device_status(_stream_handle(stream), ctypes.byref(where))
    if rc == 3:
        raise FaError(rc, "fa_check_device_status")
    return rc


def get_device_status(stream=None) -> int:
    """fa_get_device_status: synchronises the stream and returns the device
    status (0 = ok, 4 = a wait timed out); raises FaError on a CUDA error."""
    rc = library().fa_get_device_status(_stream_handle(stream))
    if rc == 3:
        raise FaError(rc, "fa_get_device_status")
    return rc


def set_wait_limit_ns(ns: int) -> None:
    library().fa_set_wait_limit_ns(int(ns))


def debug_skip_k_tile(tile: int) -> None:
    """Test hook: see fa_debug_skip_k_tile in include/fa.h (-1 turns it off)."""
    rc = library().fa_debug_skip_k_tile(int(tile))
    if rc != 0:
        raise FaError(rc, "fa_debug_skip_k_tile")


def debug_set_schedule(order: int) -> None:
    """Test hook: see fa_debug_set_schedule in include/fa.h (-1: the order by
    size, 0: heavy/light pairs, 1: cost order)."""
    rc = library().fa_debug_set_schedule(int(order))
    if rc != 0:
        raise FaError(rc, "fa_debug_set_schedule")


def debug_decode_plan(B: int, H: int, Nq: int, Nk: int, d: int, wave: int) -> tuple[int, int]:
    """Test hook: the (splits, keys per chunk) that fa_decode would use if
    ``wave`` CTAs of its partial kernel were resident at once (host
    arithmetic only; see fa_debug_decode_plan in include/fa.h)."""
    splits, chunk = ctypes.c_int(0), ctypes.c_int(0)
    rc = library().fa_debug_decode_plan(B, H, Nq, Nk, d, wave, ctypes.byref(splits), ctypes.byref(chunk))
    if rc != 0:
        raise FaError(rc, "fa_debug_decode_plan")
    return splits.value, chunk.value
