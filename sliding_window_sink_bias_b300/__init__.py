"""sink-bias GQA attention forward for B300 (sm_103a): a thin Python binding.

The work happens in ``libsinkattn.so`` (hand-written CUDA, C ABI declared in
``include/sinkattn.h``).  This module only checks tensor dtypes/shapes and
passes raw device pointers and the current CUDA stream through ctypes.  There
is no fallback: if the library is missing, every call raises.

    out, lse = prefill(q, k, v, sink, cu_seqlens, max_seqlen=..., window=128, rope_base=1e4)
    out, lse = decode(q, kcache, vcache, seqlens, sink, max_seqlen=..., window=0, rope_base=5e6)
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# SINKATTN_LIBRARY may name another build of the same sources (the checking
# test build, to run a test suite with every in-kernel bounds check on)
LIB_PATH = os.environ.get("SINKATTN_LIBRARY") or os.path.join(_HERE, "libsinkattn.so")

# status codes of include/sinkattn.h
OK, EINVAL, EUNSUPPORTED, EWORKSPACE, ECUDA, ETIMEOUT, ECHECK = range(7)

EXPORTED = (
    "sinkattn_prefill", "sinkattn_prefill_ex", "sinkattn_decode_workspace_size",
    "sinkattn_decode", "sinkattn_decode_ex", "sinkattn_status_string",
    "sinkattn_get_device_status", "sinkattn_version", "sinkattn_decode_noalloc",
    "sinkattn_prefill_backward_workspace_size", "sinkattn_prefill_backward",
    "sinkattn_decode_fp8",
)

# bytes of the library's fixed decode scratch (include/sinkattn.h)
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class SinkAttnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class Params(ctypes.Structure):
    """sinkattn_params: scale (0 = 1/sqrt(192)), rope_off, rope_style, kv_ring, k_rotated."""
    _fields_ = [("scale", ctypes.c_float), ("rope_off", ctypes.c_int32),
                ("rope_style", ctypes.c_int32), ("kv_ring", ctypes.c_int32),
                ("k_rotated", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libsinkattn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m sliding_window_sink_bias_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        L.sinkattn_prefill.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, P]
        L.sinkattn_prefill_ex.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32,
                                          ctypes.POINTER(Params), P, P, P]
        L.sinkattn_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.sinkattn_decode_workspace_size.restype = ctypes.c_size_t
        L.sinkattn_decode.argtypes = [P, P, P, P, P, i32, f32, i32, i32, i32, i32, i32, i32,
                                      P, ctypes.c_size_t, P, P, P]
        L.sinkattn_decode_ex.argtypes = [P, P, P, P, P, i32, f32, i32, i32, i32, i32, i32, i32,
                                         ctypes.POINTER(Params), P, ctypes.c_size_t, P, P, P]
        L.sinkattn_decode_noalloc.argtypes = [P, P, P, P, P, i32, f32, i32, i32, i32, i32, i32, i32,
                                              P, P, P]
        L.sinkattn_prefill_backward_workspace_size.argtypes = [i32, i32, i32]
        L.sinkattn_prefill_backward_workspace_size.restype = ctypes.c_size_t
        L.sinkattn_prefill_backward.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32,
                                                ctypes.POINTER(Params), P, P, P, P,
                                                ctypes.c_size_t, P, P, P, P, P]
        L.sinkattn_decode_fp8.argtypes = [P, P, P, P, P, P, P, i32, f32, i32, i32, i32, i32, i32,
                                          i32, ctypes.POINTER(Params), P, ctypes.c_size_t, P, P, P]
        L.sinkattn_status_string.argtypes = [i32]
        L.sinkattn_status_string.restype = ctypes.c_char_p
        L.sinkattn_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        L.sinkattn_version.restype = i32
        for name in ("sinkattn_prefill", "sinkattn_prefill_ex", "sinkattn_decode",
                     "sinkattn_decode_ex", "sinkattn_get_device_status", "sinkattn_decode_noalloc",
                     "sinkattn_prefill_backward", "sinkattn_decode_fp8"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != OK:
        raise SinkAttnError(fn, status, lib().sinkattn_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _params(scale, rope_style, rope_off, kv_ring=False, k_rotated=False):
    if scale is None and rope_style == 0 and not rope_off and not kv_ring and not k_rotated:
        return None
    return Params(float(scale or 0.0), int(bool(rope_off)), int(rope_style), int(bool(kv_ring)),
                  int(bool(k_rotated)))


def _require(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _outputs(out, lse, out_shape, lse_shape, device):
    """The caller's out/lse (checked: dtype, contiguity, exact shape), or new ones."""
    if out is None:
        out = torch.empty(*out_shape, dtype=torch.bfloat16, device=device)
    if lse is None:
        lse = torch.empty(*lse_shape, dtype=torch.float32, device=device)
    _require(out, "out", torch.bfloat16, len(out_shape))
    _require(lse, "lse", torch.float32, len(lse_shape))
    _shape(out, "out", out_shape)
    _shape(lse, "lse", lse_shape)
    return out, lse


def prefill(q, k, v, sink, cu_seqlens, *, max_seqlen: int, window: int, rope_base: float,
            out=None, lse=None, scale=None, rope_style: int = 0, rope_off: bool = False,
            stream=None):
    """Varlen prefill (one SWA or GA layer).  q [total, Hq, 192], k [total, Hkv, 192],
    v [total, Hkv, 128] bf16; sink fp32 [Hq]; cu_seqlens int32 [B+1] on the device.
    Returns (out bf16 [total, Hq, 128], lse fp32 [total, Hq])."""
    _require(q, "q", torch.bfloat16, 3)
    _require(k, "k", torch.bfloat16, 3)
    _require(v, "v", torch.bfloat16, 3)
    _require(sink, "sink", torch.float32, 1)
    _require(cu_seqlens, "cu_seqlens", torch.int32, 1)
    total, hq, dqk = q.shape
    hkv = k.shape[1]
    if dqk != 192 or k.shape != (total, hkv, 192) or v.shape != (total, hkv, 128):
        raise ValueError("expected q [T,Hq,192], k [T,Hkv,192], v [T,Hkv,128]")
    _shape(sink, "sink", (hq,))
    if cu_seqlens.shape[0] < 1:
        raise ValueError("cu_seqlens must have batch + 1 >= 1 entries")
    out, lse = _outputs(out, lse, (total, hq, 128), (total, hq), q.device)
    p = _params(scale, rope_style, rope_off)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(cu_seqlens), cu_seqlens.shape[0] - 1,
            total, int(max_seqlen), hq, hkv, int(window), float(rope_base))
    if p is None:
        st = lib().sinkattn_prefill(*args, _ptr(out), _ptr(lse), _stream(stream))
    else:
        st = lib().sinkattn_prefill_ex(*args, ctypes.byref(p), _ptr(out), _ptr(lse),
                                       _stream(stream))
    _check("sinkattn_prefill", st)
    return out, lse


def decode_workspace_size(batch: int, t: int, hq: int, hkv: int, max_seqlen: int,
                          window: int) -> int:
    return int(lib().sinkattn_decode_workspace_size(batch, t, hq, hkv, max_seqlen, window))


def prefill_backward_workspace_size(total: int, hq: int, hkv: int) -> int:
    return int(lib().sinkattn_prefill_backward_workspace_size(total, hq, hkv))


def prefill_backward(q, k, v, sink, cu_seqlens, out, lse, dout, *, max_seqlen: int, window: int,
                     rope_base: float, scale=None, rope_style: int = 0, rope_off: bool = False,
                     workspace=None, dq=None, dk=None, dv=None, dsink=None, stream=None):
    """Backward of prefill() for the loss sum(dout * out): returns (dq bf16 [T, Hq, 192],
    dk bf16 [T, Hkv, 192], dv bf16 [T, Hkv, 128], dsink fp32 [Hq]).  out and lse are the
    forward's results for the same inputs."""
    _require(q, "q", torch.bfloat16, 3)
    _require(k, "k", torch.bfloat16, 3)
    _require(v, "v", torch.bfloat16, 3)
    _require(sink, "sink", torch.float32, 1)
    _require(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _require(out, "out", torch.bfloat16, 3)
    _require(lse, "lse", torch.float32, 2)
    _require(dout, "dout", torch.bfloat16, 3)
    total, hq, _ = q.shape
    hkv = k.shape[1]
    if q.shape[2] != 192 or k.shape != (total, hkv, 192) or v.shape != (total, hkv, 128):
        raise ValueError("expected q [T,Hq,192], k [T,Hkv,192], v [T,Hkv,128]")
    _shape(sink, "sink", (hq,))
    _shape(out, "out", (total, hq, 128))
    _shape(dout, "dout", (total, hq, 128))
    _shape(lse, "lse", (total, hq))
    if cu_seqlens.shape[0] < 1:
        raise ValueError("cu_seqlens must have batch + 1 >= 1 entries")
    need = prefill_backward_workspace_size(total, hq, hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    dev = q.device
    grads = []
    for name, t, shape, dtype in (("dq", dq, (total, hq, 192), torch.bfloat16),
                                  ("dk", dk, (total, hkv, 192), torch.bfloat16),
                                  ("dv", dv, (total, hkv, 128), torch.bfloat16),
                                  ("dsink", dsink, (hq,), torch.float32)):
        if t is None:
            t = torch.empty(*shape, dtype=dtype, device=dev)
        _require(t, name, dtype, len(shape))
        _shape(t, name, shape)
        grads.append(t)
    dq, dk, dv, dsink = grads
    p = _params(scale, rope_style, rope_off)
    st = lib().sinkattn_prefill_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(cu_seqlens), cu_seqlens.shape[0] - 1, total,
        int(max_seqlen), hq, hkv, int(window), float(rope_base),
        None if p is None else ctypes.byref(p), _ptr(out), _ptr(lse), _ptr(dout),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(dsink), _stream(stream))
    _check("sinkattn_prefill_backward", st)
    return dq, dk, dv, dsink


def decode(q, kcache, vcache, seqlens, sink, *, max_seqlen: int, window: int, rope_base: float,
           workspace=None, out=None, lse=None, scale=None, rope_style: int = 0,
           rope_off: bool = False, kv_ring: bool = False, k_rotated: bool = False, stream=None):
    """MTP-verify decode.  q [B, T, Hq, 192]; kcache [B, S_cap, Hkv, 192];
    vcache [B, S_cap, Hkv, 128] bf16; seqlens int32 [B] (cached tokens including
    the T new ones); sink fp32 [Hq].  Returns (out [B, T, Hq, 128], lse [B, T, Hq]).
    kv_ring=True: the caches are rings of S_cap slots, position j at slot
    j % S_cap (sliding-window layers; seqlens may exceed S_cap).
    k_rotated=True: kcache holds keys already rotated at their positions."""
    _require(q, "q", torch.bfloat16, 4)
    _require(kcache, "kcache", torch.bfloat16, 4)
    _require(vcache, "vcache", torch.bfloat16, 4)
    _require(seqlens, "seqlens", torch.int32, 1)
    _require(sink, "sink", torch.float32, 1)
    b, t, hq, dqk = q.shape
    s_cap, hkv = kcache.shape[1], kcache.shape[2]
    if dqk != 192 or kcache.shape != (b, s_cap, hkv, 192) or vcache.shape != (b, s_cap, hkv, 128):
        raise ValueError("expected q [B,T,Hq,192], kcache [B,S,Hkv,192], vcache [B,S,Hkv,128]")
    _shape(sink, "sink", (hq,))
    _shape(seqlens, "seqlens", (b,))
    need = decode_workspace_size(b, t, hq, hkv, max_seqlen, window)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    out, lse = _outputs(out, lse, (b, t, hq, 128), (b, t, hq), q.device)
    p = _params(scale, rope_style, rope_off, kv_ring, k_rotated)
    args = (_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(sink), int(window),
            float(rope_base), b, t, s_cap, int(max_seqlen), hq, hkv)
    tail = (_ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse),
            _stream(stream))
    if p is None:
        st = lib().sinkattn_decode(*args, *tail)
    else:
        st = lib().sinkattn_decode_ex(*args, ctypes.byref(p), *tail)
    _check("sinkattn_decode", st)
    return out, lse


def decode_fp8(q, kcache, vcache, k_scale, v_scale, seqlens, sink, *, max_seqlen: int,
               window: int, rope_base: float, workspace=None, out=None, lse=None, scale=None,
               rope_style: int = 0, rope_off: bool = False, k_rotated: bool = False,
               stream=None):
    """MTP-verify decode over an FP8 (E4M3) cache: kcache [B, S_cap, Hkv, 192] and
    vcache [B, S_cap, Hkv, 128] as torch.float8_e4m3fn (or uint8 bit patterns),
    k_scale / v_scale fp32 [Hkv] (key = e4m3 * k_scale[kv head]).  Other arguments
    and the results as decode() (k_rotated: the E4M3 keys are already rotated)."""
    _require(q, "q", torch.bfloat16, 4)
    for name, t in (("kcache", kcache), ("vcache", vcache)):
        if not isinstance(t, torch.Tensor) or t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must be a float8_e4m3fn/uint8 tensor")
        _require(t, name, t.dtype, 4)
    _require(k_scale, "k_scale", torch.float32, 1)
    _require(v_scale, "v_scale", torch.float32, 1)
    _require(seqlens, "seqlens", torch.int32, 1)
    _require(sink, "sink", torch.float32, 1)
    b, t, hq, dqk = q.shape
    s_cap, hkv = kcache.shape[1], kcache.shape[2]
    if dqk != 192 or kcache.shape != (b, s_cap, hkv, 192) or vcache.shape != (b, s_cap, hkv, 128):
        raise ValueError("expected q [B,T,Hq,192], kcache [B,S,Hkv,192], vcache [B,S,Hkv,128]")
    _shape(k_scale, "k_scale", (hkv,))
    _shape(v_scale, "v_scale", (hkv,))
    _shape(sink, "sink", (hq,))
    _shape(seqlens, "seqlens", (b,))
    need = decode_workspace_size(b, t, hq, hkv, max_seqlen, window)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    out, lse = _outputs(out, lse, (b, t, hq, 128), (b, t, hq), q.device)
    p = _params(scale, rope_style, rope_off, k_rotated=k_rotated)
    st = lib().sinkattn_decode_fp8(
        _ptr(q), kcache.data_ptr(), vcache.data_ptr(), _ptr(k_scale), _ptr(v_scale),
        _ptr(seqlens), _ptr(sink), int(window), float(rope_base), b, t, s_cap, int(max_seqlen),
        hq, hkv, None if p is None else ctypes.byref(p), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    _check("sinkattn_decode_fp8", st)
    return out, lse


def decode_noalloc(q, kcache, vcache, seqlens, sink, *, max_seqlen: int, window: int,
                   rope_base: float, out=None, lse=None, stream=None):
    """MTP-verify decode through sinkattn_decode_noalloc: same inputs and results
    as decode(), but the split-KV partials go to the library's fixed device
    buffer (NOALLOC_SCRATCH_BYTES per GPU) instead of a workspace, so the call
    itself allocates nothing.  For callers that cannot allocate device memory
    where they decode.  Calls that overlap on the GPU share that buffer and
    race; the first call on a device should come before any stream capture.
    out / lse are the caller's outputs (allocated here only if not given)."""
    _require(q, "q", torch.bfloat16, 4)
    _require(kcache, "kcache", torch.bfloat16, 4)
    _require(vcache, "vcache", torch.bfloat16, 4)
    _require(seqlens, "seqlens", torch.int32, 1)
    _require(sink, "sink", torch.float32, 1)
    b, t, hq, dqk = q.shape
    s_cap, hkv = kcache.shape[1], kcache.shape[2]
    if dqk != 192 or kcache.shape != (b, s_cap, hkv, 192) or vcache.shape != (b, s_cap, hkv, 128):
        raise ValueError("expected q [B,T,Hq,192], kcache [B,S,Hkv,192], vcache [B,S,Hkv,128]")
    _shape(sink, "sink", (hq,))
    _shape(seqlens, "seqlens", (b,))
    out, lse = _outputs(out, lse, (b, t, hq, 128), (b, t, hq), q.device)
    st = lib().sinkattn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens),
                                       _ptr(sink), int(window), float(rope_base), b, t, s_cap,
                                       int(max_seqlen), hq, hkv, _ptr(out), _ptr(lse),
                                       _stream(stream))
    _check("sinkattn_decode_noalloc", st)
    return out, lse


def device_status():
    """(status, raw word) of the device status word; synchronises the device."""
    w = ctypes.c_uint32(0)
    st = lib().sinkattn_get_device_status(ctypes.byref(w))
    return int(st), int(w.value)


def version() -> int:
    return int(lib().sinkattn_version())
