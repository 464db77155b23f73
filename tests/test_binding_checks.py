"""Host-only checks of the Python binding: a tensor of the wrong shape (out,
lse, sink, seqlens, a gradient, an FP8 scale) is refused with ValueError before
the C library is called, so no kernel ever reads or writes past a tensor's end.

There is no GPU here, so the binding's CUDA-device check is relaxed for these
calls (CPU tensors stand in for device tensors); the library itself is never
reached: its entry points are replaced by functions that fail the test."""
import pytest
import torch

import sliding_window_sink_bias_b300 as sa


class _NoCall:
    """Stands in for the loaded library: the size queries go to the real one,
    every other entry point fails the test."""

    def __init__(self, real):
        self._real = real

    def __getattr__(self, name):
        if name.startswith("sinkattn_") and not name.endswith("workspace_size"):
            def fail(*a, **k):
                raise AssertionError(f"{name} reached with a mis-shaped argument")
            return fail
        return getattr(self._real, name)


@pytest.fixture
def host_binding(monkeypatch):
    def require(t, name, dtype, ndim):
        if not isinstance(t, torch.Tensor):
            raise TypeError(name)
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}")
        if t.dim() != ndim:
            raise ValueError(f"{name} must have {ndim} dims")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    monkeypatch.setattr(sa, "_require", require)
    nocall = _NoCall(sa.lib())
    monkeypatch.setattr(sa, "lib", lambda: nocall)
    yield


def bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def f32(*shape):
    return torch.zeros(*shape, dtype=torch.float32)


def i32(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


def _prefill_args(total=32, hq=64, hkv=8):
    return (bf(total, hq, 192), bf(total, hkv, 192), bf(total, hkv, 128), f32(hq),
            torch.tensor([0, total], dtype=torch.int32))


def test_prefill_rejects_wrong_shapes(host_binding):
    kw = dict(max_seqlen=32, window=128, rope_base=1e4)
    q, k, v, sink, cu = _prefill_args()
    for bad in (dict(out=bf(32, 64, 127)), dict(out=bf(31, 64, 128)), dict(lse=f32(32, 63)),
                dict(lse=f32(33, 64))):
        with pytest.raises(ValueError):
            sa.prefill(q, k, v, sink, cu, **kw, **bad)
    with pytest.raises(ValueError):
        sa.prefill(q, k, v, f32(32), cu, **kw)
    with pytest.raises(ValueError):
        sa.prefill(q, k[:16], v, sink, cu, **kw)


def test_backward_rejects_wrong_shapes(host_binding):
    kw = dict(max_seqlen=32, window=128, rope_base=1e4)
    q, k, v, sink, cu = _prefill_args()
    out, lse, dout = bf(32, 64, 128), f32(32, 64), bf(32, 64, 128)
    for bad in (dict(dq=bf(32, 64, 128)), dict(dk=bf(32, 4, 192)), dict(dv=bf(16, 8, 128)),
                dict(dsink=f32(8))):
        with pytest.raises(ValueError):
            sa.prefill_backward(q, k, v, sink, cu, out, lse, dout, **kw, **bad)
    with pytest.raises(ValueError):
        sa.prefill_backward(q, k, v, sink, cu, out, f32(32, 8), dout, **kw)
    with pytest.raises(ValueError):
        sa.prefill_backward(q, k, v, sink, cu, out, lse, bf(32, 64, 64), **kw)


def _decode_args(b=3, t=4, hq=64, hkv=4, s_cap=256):
    return (bf(b, t, hq, 192), bf(b, s_cap, hkv, 192), bf(b, s_cap, hkv, 128), i32(b), f32(hq))


@pytest.mark.parametrize("fn", ["decode", "decode_noalloc"])
def test_decode_rejects_wrong_shapes(host_binding, fn):
    call = getattr(sa, fn)
    kw = dict(max_seqlen=256, window=0, rope_base=5e6)
    q, kc, vc, sl, sink = _decode_args()
    for bad in (dict(out=bf(3, 4, 64, 64)), dict(out=bf(3, 3, 64, 128)), dict(lse=f32(3, 4, 32)),
                dict(lse=f32(2, 4, 64))):
        with pytest.raises(ValueError):
            call(q, kc, vc, sl, sink, **kw, **bad)
    with pytest.raises(ValueError):
        call(q, kc, vc, i32(2), sink, **kw)      # one length per sequence
    with pytest.raises(ValueError):
        call(q, kc, vc, sl, f32(16), **kw)       # one sink per query head


def test_decode_fp8_rejects_wrong_shapes(host_binding):
    kw = dict(max_seqlen=256, window=0, rope_base=5e6)
    q, kc, vc, sl, sink = _decode_args()
    k8 = torch.zeros(kc.shape, dtype=torch.uint8)
    v8 = torch.zeros(vc.shape, dtype=torch.uint8)
    ks, vs = f32(4), f32(4)
    with pytest.raises(ValueError):
        sa.decode_fp8(q, k8, v8, f32(8), vs, sl, sink, **kw)
    with pytest.raises(ValueError):
        sa.decode_fp8(q, k8, v8, ks, f32(1), sl, sink, **kw)
    with pytest.raises(ValueError):
        sa.decode_fp8(q, k8, v8, ks, vs, sl, sink, **kw, out=bf(3, 4, 64, 127))
    with pytest.raises(ValueError):
        sa.decode_fp8(q, k8, v8, ks, vs, i32(5), sink, **kw)
