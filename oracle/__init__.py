"""The oracle: a plain fp64 CPU evaluation of the sink-bias attention forward.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers; the product library never
imports or links anything here, and nothing here imports the product.

The arithmetic lives in ``sinkattn_oracle.c`` (see its header for the passages
of the MiMo-V2-Flash Technical Report it follows).  This module only builds the
shared object with gcc and marshals numpy/torch CPU arrays into it.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sinkattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", _LIB, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("dqk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("drot", ctypes.c_int32), ("rope_style", ctypes.c_int32),
                ("window", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("rope_base", ctypes.c_double), ("scale", ctypes.c_double),
                ("k_rotated", ctypes.c_int32)]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.oracle_prefill.argtypes = [P, P, P, P, P, i32, i32, i32, ctypes.POINTER(_Cfg),
                                       P, i64, P, P, ctypes.c_int]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32,
                                      ctypes.POINTER(_Cfg), P, i64, P, P, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_prefill_backward.argtypes = [P, P, P, P, P, i32, i32, i32,
                                                ctypes.POINTER(_Cfg), P, P, P, P, P, ctypes.c_int]
        lib.oracle_prefill_backward.restype = ctypes.c_int
        lib.oracle_rope.argtypes = [P, i32, i32, i32, ctypes.c_double, ctypes.c_double, P]
        lib.oracle_rope.restype = None
        lib.oracle_rope_rows.argtypes = [P, i64, i32, i32, i32, ctypes.c_double, P, P]
        lib.oracle_rope_rows.restype = None
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_input(x):
    """-> (contiguous numpy array, dtype code): bf16 bit patterns or fp64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), 0
            return x.to(torch.float64).numpy(), 1
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        return a, 0
    return np.ascontiguousarray(a, dtype=np.float64), 1


def _f32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().cpu().to(torch.float32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.float32)


def _i32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().cpu().to(torch.int32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.int32)


def _cfg(dqk, dv, drot, rope_style, window, dtype, rope_base, scale, k_rotated=False):
    return _Cfg(int(dqk), int(dv), int(drot), int(rope_style), int(window), int(dtype),
                float(rope_base), float(scale), int(bool(k_rotated)))


def prefill(q, k, v, sink, cu_seqlens, *, window: int, rope_base: float,
            scale: float | None = None, drot: int = 64, rope_style: int = 0,
            rows=None, nthreads: int = 0):
    """Eqs. (1)-(3) over packed sequences.

    q [total, Hq, dqk], k [total, Hkv, dqk], v [total, Hkv, dv] (bf16 torch
    tensors, uint16 bit patterns or float arrays), sink [Hq], cu_seqlens [B+1].
    rows: flat indices token*Hq + h to evaluate (None = all).
    Returns (out fp64 [n, dv], lse fp64 [n]); with rows=None they are shaped
    [total, Hq, dv] and [total, Hq].
    """
    qa, dt_q = _as_input(q)
    ka, dt_k = _as_input(k)
    va, dt_v = _as_input(v)
    if not (dt_q == dt_k == dt_v):
        raise ValueError("q, k, v must share one dtype")
    total, Hq, dqk = qa.shape
    Hkv, dv = ka.shape[1], va.shape[2]
    sk = _f32(sink)
    cu = _i32(cu_seqlens)
    B = cu.shape[0] - 1
    if scale is None:
        scale = 1.0 / math.sqrt(dqk)
    cfg = _cfg(dqk, dv, drot, rope_style, window, dt_q, rope_base, scale)
    if rows is None:
        ra, n = None, total * Hq
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        n = ra.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_prefill(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, sk.ctypes.data,
                                cu.ctypes.data, B, Hq, Hkv, ctypes.byref(cfg),
                                None if ra is None else ra.ctypes.data, n,
                                out.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill failed with {rc}")
    if rows is None:
        return out.reshape(total, Hq, dv), lse.reshape(total, Hq)
    return out, lse


def prefill_backward(q, k, v, sink, cu_seqlens, dout, *, window: int, rope_base: float,
                     scale: float | None = None, drot: int = 64, rope_style: int = 0,
                     nthreads: int = 0):
    """Gradients of L = sum(dout * o) for the prefill above, by the chain rule
    through eqs. (1)-(3): returns (dq [total, Hq, dqk], dk [total, Hkv, dqk],
    dv [total, Hkv, dv], dsink [Hq]) as fp64 numpy arrays."""
    qa, dt_q = _as_input(q)
    ka, dt_k = _as_input(k)
    va, dt_v = _as_input(v)
    da, dt_d = _as_input(dout)
    if not (dt_q == dt_k == dt_v == dt_d):
        raise ValueError("q, k, v, dout must share one dtype")
    total, Hq, dqk = qa.shape
    Hkv, dv = ka.shape[1], va.shape[2]
    sk = _f32(sink)
    cu = _i32(cu_seqlens)
    B = cu.shape[0] - 1
    if scale is None:
        scale = 1.0 / math.sqrt(dqk)
    cfg = _cfg(dqk, dv, drot, rope_style, window, dt_q, rope_base, scale)
    dq = np.zeros((total, Hq, dqk), dtype=np.float64)
    dk = np.zeros((total, Hkv, dqk), dtype=np.float64)
    dvv = np.zeros((total, Hkv, dv), dtype=np.float64)
    ds = np.zeros((Hq,), dtype=np.float64)
    rc = _load().oracle_prefill_backward(qa.ctypes.data, ka.ctypes.data, va.ctypes.data,
                                         sk.ctypes.data, cu.ctypes.data, B, Hq, Hkv,
                                         ctypes.byref(cfg), da.ctypes.data, dq.ctypes.data,
                                         dk.ctypes.data, dvv.ctypes.data, ds.ctypes.data,
                                         int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill_backward failed with {rc}")
    return dq, dk, dvv, ds


def decode(q, kcache, vcache, seqlens, sink, *, window: int, rope_base: float,
           scale: float | None = None, drot: int = 64, rope_style: int = 0,
           rows=None, nthreads: int = 0, k_rotated: bool = False):
    """MTP-verify decode: q [B, T, Hq, dqk] against kcache [B, S_cap, Hkv, dqk] and
    vcache [B, S_cap, Hkv, dv]; seqlens [B] counts cached tokens including the T
    new ones.  rows: flat indices (b*T + t)*Hq + h (None = all).  k_rotated: the
    cache holds keys already rotated at their positions (only q is rotated).
    Returns (out [n, dv], lse [n]) or, with rows=None, [B, T, Hq, dv] and [B, T, Hq]."""
    qa, dt_q = _as_input(q)
    ka, dt_k = _as_input(kcache)
    va, dt_v = _as_input(vcache)
    if not (dt_q == dt_k == dt_v):
        raise ValueError("q, kcache, vcache must share one dtype")
    B, T, Hq, dqk = qa.shape
    S_cap, Hkv = ka.shape[1], ka.shape[2]
    dv = va.shape[3]
    sk = _f32(sink)
    sl = _i32(seqlens)
    if scale is None:
        scale = 1.0 / math.sqrt(dqk)
    cfg = _cfg(dqk, dv, drot, rope_style, window, dt_q, rope_base, scale, k_rotated)
    if rows is None:
        ra, n = None, B * T * Hq
    else:
        ra = np.ascontiguousarray(rows, dtype=np.int64)
        n = ra.shape[0]
    out = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_decode(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, sl.ctypes.data,
                               sk.ctypes.data, B, T, S_cap, Hq, Hkv, ctypes.byref(cfg),
                               None if ra is None else ra.ctypes.data, n,
                               out.ctypes.data, lse.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed with {rc}")
    if rows is None:
        return out.reshape(B, T, Hq, dv), lse.reshape(B, T, Hq)
    return out, lse


def rope(x, pos: float, *, base: float, drot: int = 64, rope_style: int = 0):
    """The oracle's rotary embedding of one fp64 vector (exposed for its pins)."""
    xa = np.ascontiguousarray(x, dtype=np.float64)
    y = np.zeros_like(xa)
    _load().oracle_rope(xa.ctypes.data, xa.shape[0], int(drot), int(rope_style),
                        float(base), float(pos), y.ctypes.data)
    return y


def rope_rows(x, pos, *, base: float, drot: int = 64, rope_style: int = 0):
    """The oracle's rotary embedding of many fp64 rows: x [..., d] with one
    position per row, pos broadcastable to x.shape[:-1].  Returns fp64 [..., d]."""
    xa = np.ascontiguousarray(x, dtype=np.float64)
    d = xa.shape[-1]
    pa = np.ascontiguousarray(np.broadcast_to(np.asarray(pos, dtype=np.float64), xa.shape[:-1]))
    y = np.zeros_like(xa)
    n = int(np.prod(xa.shape[:-1]))
    _load().oracle_rope_rows(xa.ctypes.data, n, d, int(drot), int(rope_style), float(base),
                             pa.ctypes.data, y.ctypes.data)
    return y
