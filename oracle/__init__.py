"""Oracle for softmax attention: plain fp64 CPU code, TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product path (``io_aware_attention_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``attn_ref.c`` (compiled with gcc into
``liboracle.so`` next to it); this module only marshals arrays.  What it
computes, per (batch, head) and query row i (the plain definition of the
attention the pages describe -- "Kernels — fusion and FlashAttention" §2–§3
and "Writing and Benchmarking Custom Kernels" §10.3.1):

    S = scale * Q K^T, causal: S_ij = -inf for j > i,
    P = softmax(S) by the two-pass rule (row max, exp, row sum),
    O = P V,  L_i = m_i + ln l_i.

``attention_online`` runs the tile-by-tile online-softmax recurrence of
"Kernels — fusion and FlashAttention" §3 instead, in fp64.

``attention_bwd`` gives the gradients dQ, dK, dV (and the per-row scalar
D_i) for a given dO, by the softmax/matrix-product chain rule that
"Writing and Benchmarking Custom Kernels" §10.3.2 describes.

``bias_gelu_dropout`` is the elementwise chain of "Fusion and IO-aware
kernels" (bias add, GELU in the tanh form of "Writing and Benchmarking
Custom Kernels" §10.2.1, dropout with a passed-in keep mask), in fp64.

Inputs are torch bf16 CPU tensors (or numpy uint16 arrays of bf16 bits) of
shape (B, H, N, d), contiguous.  Outputs are numpy float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``attn_ref.c`` into ``liboracle.so`` (gcc, OpenMP) if stale."""
    with _lock:
        stale = (not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src))
        if force or stale:
            tmp = out + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, out)
    return out


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 numpy array of bf16 bits."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 arrays of bf16 bits")
        return np.ascontiguousarray(x)
    import torch  # local: torch is only needed for tensor inputs

    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bf16 tensor, got {x.dtype}")
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def _shape4(q, k, v):
    if not (q.shape == k.shape == v.shape) or q.ndim != 4:
        raise ValueError(f"q, k, v must share one (B, H, N, d) shape: {q.shape} {k.shape} {v.shape}")
    return tuple(int(s) for s in q.shape)


class Oracle:
    """The oracle's entry points, bound to one compiled ``attn_ref.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64, c_int, c_dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        head = [u16p, u16p, u16p, i64, i64, i64, i64, c_int, c_dbl]
        lib.oracle_attn_f64.argtypes = head + [f64p, f64p, f64p, c_int]
        lib.oracle_attn_rows_f64.argtypes = head + [i64p, i64p, i64, f64p, f64p, c_int]
        lib.oracle_attn_online_f64.argtypes = head + [i64, f64p, f64p, c_int]
        lib.oracle_max_threads.argtypes = []
        rect = [u16p, u16p, u16p, i64, i64, i64, i64, i64, c_int, c_dbl]
        lib.oracle_attn_rect_f64.argtypes = rect + [f64p, f64p, c_int]
        lib.oracle_attn_rect_rows_f64.argtypes = rect + [i64p, i64p, i64, f64p, f64p, c_int]
        lib.oracle_attn_bwd_f64.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, i64, c_int,
                                            c_dbl, f64p, f64p, f64p, f64p, c_int]
        lib.oracle_bias_gelu_dropout_f64.argtypes = [u16p, u16p, ctypes.POINTER(ctypes.c_uint32), i64, i64,
                                                     c_dbl, f64p, c_int]
        for fn in (lib.oracle_attn_f64, lib.oracle_attn_rows_f64, lib.oracle_attn_online_f64,
                   lib.oracle_max_threads, lib.oracle_attn_rect_f64, lib.oracle_attn_rect_rows_f64,
                   lib.oracle_attn_bwd_f64, lib.oracle_bias_gelu_dropout_f64):
            fn.restype = c_int
        self.lib = lib

    def max_threads(self) -> int:
        """Number of OpenMP threads the oracle uses by default."""
        return int(self.lib.oracle_max_threads())

    def attention(self, q, k, v, causal: bool, scale: float, return_probs: bool = False,
                  threads: int = 0):
        """Two-pass fp64 attention over the full tensor.

        Returns ``(o, lse)`` or ``(o, lse, p)``; o is (B, H, N, d), lse
        (B, H, N), p (B, H, N, N), all float64.
        """
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        B, H, N, d = _shape4(qb, kb, vb)
        o = np.empty((B, H, N, d), np.float64)
        lse = np.empty((B, H, N), np.float64)
        p = np.empty((B, H, N, N), np.float64) if return_probs else None
        rc = self.lib.oracle_attn_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                      _ptr(vb, ctypes.c_uint16), B, H, N, d, int(bool(causal)),
                                      float(scale), _ptr(o, ctypes.c_double),
                                      _ptr(lse, ctypes.c_double), _ptr(p, ctypes.c_double),
                                      int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_f64 failed ({rc})")
        return (o, lse, p) if return_probs else (o, lse)

    def attention_rows(self, q, k, v, causal: bool, scale: float, bh_idx, row_idx,
                       threads: int = 0):
        """Two-pass fp64 attention for selected rows.

        Row t is query ``row_idx[t]`` of flattened head ``bh_idx[t]``
        (= b*H + h).  Returns ``(o_rows (n, d), lse_rows (n,))`` float64.
        """
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        B, H, N, d = _shape4(qb, kb, vb)
        bh = np.ascontiguousarray(np.asarray(bh_idx, dtype=np.int64))
        rows = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
        if bh.shape != rows.shape or bh.ndim != 1:
            raise ValueError("bh_idx and row_idx must be 1-D and of equal length")
        n = int(bh.shape[0])
        o = np.empty((n, d), np.float64)
        lse = np.empty((n,), np.float64)
        rc = self.lib.oracle_attn_rows_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                           _ptr(vb, ctypes.c_uint16), B, H, N, d,
                                           int(bool(causal)), float(scale),
                                           _ptr(bh, ctypes.c_int64), _ptr(rows, ctypes.c_int64),
                                           n, _ptr(o, ctypes.c_double),
                                           _ptr(lse, ctypes.c_double), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_rows_f64 failed ({rc})")
        return o, lse

    def attention_online(self, q, k, v, causal: bool, scale: float, tile: int,
                         threads: int = 0):
        """The online-softmax recurrence with ``tile`` keys per step, fp64.

        Returns ``(o, lse)`` like :meth:`attention`.
        """
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        B, H, N, d = _shape4(qb, kb, vb)
        o = np.empty((B, H, N, d), np.float64)
        lse = np.empty((B, H, N), np.float64)
        rc = self.lib.oracle_attn_online_f64(_ptr(qb, ctypes.c_uint16),
                                             _ptr(kb, ctypes.c_uint16),
                                             _ptr(vb, ctypes.c_uint16), B, H, N, d,
                                             int(bool(causal)), float(scale), int(tile),
                                             _ptr(o, ctypes.c_double),
                                             _ptr(lse, ctypes.c_double), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_online_f64 failed ({rc})")
        return o, lse


    def attention_rect(self, q, k, v, causal: bool, scale: float, threads: int = 0):
        """Decode attention: q (B, H, Nq, d) against k, v (B, H, Nk, d); query i
        stands at key position Nk - Nq + i (the causal window ends there).

        Returns ``(o (B, H, Nq, d), lse (B, H, Nq))`` float64.
        """
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        B, H, Nq, d, Nk = _shape_rect(qb, kb, vb)
        o = np.empty((B, H, Nq, d), np.float64)
        lse = np.empty((B, H, Nq), np.float64)
        rc = self.lib.oracle_attn_rect_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                           _ptr(vb, ctypes.c_uint16), B, H, Nq, Nk, d,
                                           int(bool(causal)), float(scale), _ptr(o, ctypes.c_double),
                                           _ptr(lse, ctypes.c_double), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_rect_f64 failed ({rc})")
        return o, lse

    def attention_rect_rows(self, q, k, v, causal: bool, scale: float, bh_idx, row_idx,
                            threads: int = 0):
        """Selected rows of :meth:`attention_rect` (query ``row_idx[t]`` of
        flattened head ``bh_idx[t]``)."""
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        B, H, Nq, d, Nk = _shape_rect(qb, kb, vb)
        bh = np.ascontiguousarray(np.asarray(bh_idx, dtype=np.int64))
        rows = np.ascontiguousarray(np.asarray(row_idx, dtype=np.int64))
        if bh.shape != rows.shape or bh.ndim != 1:
            raise ValueError("bh_idx and row_idx must be 1-D and of equal length")
        n = int(bh.shape[0])
        o = np.empty((n, d), np.float64)
        lse = np.empty((n,), np.float64)
        rc = self.lib.oracle_attn_rect_rows_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                                _ptr(vb, ctypes.c_uint16), B, H, Nq, Nk, d,
                                                int(bool(causal)), float(scale), _ptr(bh, ctypes.c_int64),
                                                _ptr(rows, ctypes.c_int64), n, _ptr(o, ctypes.c_double),
                                                _ptr(lse, ctypes.c_double), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_rect_rows_f64 failed ({rc})")
        return o, lse

    def attention_bwd(self, q, k, v, do, causal: bool, scale: float, threads: int = 0):
        """Gradients of square attention for the output gradient ``do``.

        q, k, v, do: bf16 (B, H, N, d).  Returns ``(dq, dk, dv, D)``, the
        first three (B, H, N, d) and D (B, H, N), all float64.
        """
        qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(do)
        B, H, N, d = _shape4(qb, kb, vb)
        if db.shape != qb.shape:
            raise ValueError(f"do must have the shape of q: {db.shape} vs {qb.shape}")
        dq = np.empty((B, H, N, d), np.float64)
        dk = np.empty((B, H, N, d), np.float64)
        dv = np.empty((B, H, N, d), np.float64)
        dsum = np.empty((B, H, N), np.float64)
        rc = self.lib.oracle_attn_bwd_f64(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                                          _ptr(vb, ctypes.c_uint16), _ptr(db, ctypes.c_uint16),
                                          B, H, N, d, int(bool(causal)), float(scale),
                                          _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                          _ptr(dv, ctypes.c_double), _ptr(dsum, ctypes.c_double),
                                          int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_attn_bwd_f64 failed ({rc})")
        return dq, dk, dv, dsum

    def bias_gelu_dropout(self, x, bias, keep, p: float, threads: int = 0):
        """y = dropout(gelu(x + bias)) in fp64 for x (rows, cols) and bias (cols,),
        bf16; keep: uint32 words of keep bits over the flat index (bit e % 32 of
        word e // 32), or None to keep every element.  Returns (rows, cols) float64."""
        xb, bb = _bits(x), _bits(bias)
        if xb.ndim != 2 or bb.shape != (xb.shape[1],):
            raise ValueError(f"x (rows, cols) and bias (cols,) expected: {xb.shape} {bb.shape}")
        rows, cols = (int(s) for s in xb.shape)
        kw = None
        if keep is not None:
            kw = np.ascontiguousarray(np.asarray(keep, dtype=np.uint32))
            if kw.size * 32 < rows * cols:
                raise ValueError("keep mask too short")
        y = np.empty((rows, cols), np.float64)
        rc = self.lib.oracle_bias_gelu_dropout_f64(_ptr(xb, ctypes.c_uint16), _ptr(bb, ctypes.c_uint16),
                                                   _ptr(kw, ctypes.c_uint32), rows, cols, float(p),
                                                   _ptr(y, ctypes.c_double), int(threads))
        if rc != 0:
            raise RuntimeError(f"oracle_bias_gelu_dropout_f64 failed ({rc})")
        return y


def _shape_rect(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError(f"q (B, H, Nq, d) and k, v (B, H, Nk, d) expected: {q.shape} {k.shape} {v.shape}")
    B, H, Nq, d = (int(s) for s in q.shape)
    return B, H, Nq, d, int(k.shape[2])


_default = None


def _oracle() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def from_source(src: str, out: str) -> Oracle:
    """Compile another copy of the oracle source (tests plant mistakes this way)."""
    return Oracle(build(force=True, src=src, out=out))


def max_threads() -> int:
    return _oracle().max_threads()


def attention(q, k, v, causal, scale, return_probs=False, threads=0):
    return _oracle().attention(q, k, v, causal, scale, return_probs, threads)


def attention_rows(q, k, v, causal, scale, bh_idx, row_idx, threads=0):
    return _oracle().attention_rows(q, k, v, causal, scale, bh_idx, row_idx, threads)


def attention_online(q, k, v, causal, scale, tile, threads=0):
    return _oracle().attention_online(q, k, v, causal, scale, tile, threads)


def bf16_to_f64(x) -> np.ndarray:
    """Exact widening of bf16 values (tensor or bits) to float64."""
    b = _bits(x).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def attention_rect(q, k, v, causal, scale, threads=0):
    return _oracle().attention_rect(q, k, v, causal, scale, threads)


def attention_rect_rows(q, k, v, causal, scale, bh_idx, row_idx, threads=0):
    return _oracle().attention_rect_rows(q, k, v, causal, scale, bh_idx, row_idx, threads)


def attention_bwd(q, k, v, do, causal, scale, threads=0):
    return _oracle().attention_bwd(q, k, v, do, causal, scale, threads)


def bias_gelu_dropout(x, bias, keep, p, threads=0):
    return _oracle().bias_gelu_dropout(x, bias, keep, p, threads)
