"""Host-only checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/sinkattn.h declares, and rejects bad arguments before
touching the GPU (these calls never reach a CUDA API)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sinkattn.h")


@pytest.fixture(scope="module")
def L():
    from sliding_window_sink_bias_b300 import build
    build.build()
    import sliding_window_sink_bias_b300 as sa
    return sa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(sinkattn_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_lists_the_api():
    names = declared_functions()
    for n in ("sinkattn_prefill", "sinkattn_decode", "sinkattn_decode_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    import sliding_window_sink_bias_b300 as sa
    for n in declared_functions():
        assert hasattr(L, n), n
    assert set(sa.EXPORTED) == set(declared_functions())


def test_status_strings_and_version(L):
    import sliding_window_sink_bias_b300 as sa
    assert sa.version() >= 100
    for code in range(6):
        s = L.sinkattn_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.sinkattn_status_string(99).decode() == "unknown status"


def _prefill(L, q=1, k=1, v=1, sink=1, cu=1, batch=1, total=16, max_seqlen=16, hq=64, hkv=8,
             window=128, base=1e4, out=1, lse=1):
    P = ctypes.c_void_p
    f = lambda x: None if x is None else P(16 * x)  # fake, 16-byte-aligned pointers
    return L.sinkattn_prefill(f(q), f(k), f(v), f(sink), f(cu), batch, total, max_seqlen, hq, hkv,
                              window, base, f(out), f(lse), None)


def test_prefill_argument_checks(L):
    import sliding_window_sink_bias_b300 as sa
    assert _prefill(L, batch=-1) == sa.EINVAL
    assert _prefill(L, total=-5) == sa.EINVAL
    assert _prefill(L, window=-1) == sa.EINVAL
    assert _prefill(L, hq=64, hkv=5) == sa.EINVAL         # not a multiple
    assert _prefill(L, hq=0) == sa.EINVAL
    assert _prefill(L, hq=24, hkv=8) == sa.EUNSUPPORTED   # group of 3
    assert _prefill(L, hq=256, hkv=1) == sa.EUNSUPPORTED  # group above 128
    assert _prefill(L, q=None) == sa.EINVAL
    assert _prefill(L, lse=None) == sa.EINVAL
    assert _prefill(L, max_seqlen=0) == sa.EINVAL
    assert _prefill(L, base=0.0) == sa.EINVAL
    assert _prefill(L, base=float("nan")) == sa.EINVAL
    # nothing to do: no launch, no CUDA call
    assert _prefill(L, batch=0, total=0, max_seqlen=0, q=None) == sa.OK
    assert _prefill(L, total=0, max_seqlen=0, q=None) == sa.OK
    # misaligned q (8 bytes off)
    P = ctypes.c_void_p
    st = L.sinkattn_prefill(P(24), P(16), P(16), P(16), P(16), 1, 16, 16, 64, 8, 128, 1e4,
                            P(16), P(16), None)
    assert st == sa.EINVAL


def test_prefill_ex_params_checks(L):
    import sliding_window_sink_bias_b300 as sa
    P = ctypes.c_void_p
    bad = sa.Params(0.0, 0, 7, 0)
    st = L.sinkattn_prefill_ex(P(16), P(16), P(16), P(16), P(16), 1, 16, 16, 64, 8, 128, 1e4,
                               ctypes.byref(bad), P(16), P(16), None)
    assert st == sa.EINVAL
    inf_scale = sa.Params(float("inf"), 0, 0, 0)
    st = L.sinkattn_prefill_ex(P(16), P(16), P(16), P(16), P(16), 1, 16, 16, 64, 8, 128, 1e4,
                               ctypes.byref(inf_scale), P(16), P(16), None)
    assert st == sa.EINVAL


def test_decode_workspace_size(L):
    ws = L.sinkattn_decode_workspace_size
    assert ws(0, 4, 64, 4, 1000, 0) == 0
    assert ws(2, 0, 64, 4, 1000, 0) == 0
    assert ws(2, 9, 64, 4, 1000, 0) == 0        # 9 tokens x 16 heads > 128 rows
    assert ws(2, 4, 64, 5, 1000, 0) == 0
    a = ws(64, 4, 64, 4, 262144, 0)
    b = ws(64, 4, 64, 4, 65536, 0)
    # the layout does not depend on the cache lengths or the window: one 64-bit
    # ticket per unit (batch*Hkv, padded to 256 bytes), then two partial slots
    # of T*G rows x 132 fp32 (128 values, max, sum, pad) per CTA for at most
    # 160 CTAs
    assert a == b == ws(64, 4, 64, 4, 262144, 128)
    tab = (64 * 4 * 8 + 255) // 256 * 256
    assert a == tab + 160 * 2 * (4 * 16) * 132 * 4
    tab8 = (64 * 8 * 8 + 255) // 256 * 256
    assert ws(64, 4, 64, 8, 262144, 128) == tab8 + 160 * 2 * (4 * 8) * 132 * 4


def _decode(L, q=1, kc=1, vc=1, sl=1, sink=1, window=0, base=5e6, b=2, t=4, s_cap=100,
            max_seqlen=100, hq=64, hkv=4, ws=1, ws_bytes=None, out=1, lse=1):
    P = ctypes.c_void_p
    f = lambda x: None if x is None else P(256 * x)
    if ws_bytes is None:
        ws_bytes = L.sinkattn_decode_workspace_size(b, t, hq, hkv, max_seqlen, window)
    return L.sinkattn_decode(f(q), f(kc), f(vc), f(sl), f(sink), window, base, b, t, s_cap,
                             max_seqlen, hq, hkv, f(ws), ws_bytes, f(out), f(lse), None)


def test_decode_argument_checks(L):
    import sliding_window_sink_bias_b300 as sa
    assert _decode(L, t=0) == sa.EINVAL
    assert _decode(L, b=-1) == sa.EINVAL
    assert _decode(L, max_seqlen=101) == sa.EINVAL     # longer than the cache
    assert _decode(L, hkv=3) == sa.EINVAL
    assert _decode(L, t=9) == sa.EUNSUPPORTED          # 9 x 16 rows > 128
    assert _decode(L, kc=None) == sa.EINVAL
    assert _decode(L, ws=None) == sa.EWORKSPACE
    assert _decode(L, ws_bytes=8) == sa.EWORKSPACE
    assert _decode(L, b=0) == sa.OK


def test_decode_rejects_non_positive_scale(L):
    """The decode softmax scales the logits after taking their max, so a scale
    <= 0 is refused before anything is launched."""
    import sliding_window_sink_bias_b300 as sa
    P = ctypes.c_void_p
    f = lambda x: P(256 * x)
    ws = L.sinkattn_decode_workspace_size(2, 4, 64, 4, 100, 0)
    for scale in (-0.5, -1e-3):
        p = sa.Params(scale, 0, 0, 0)
        st = L.sinkattn_decode_ex(f(1), f(1), f(1), f(1), f(1), 0, 5e6, 2, 4, 100, 100, 64, 4,
                                  ctypes.byref(p), f(1), ws, f(1), f(1), None)
        assert st == sa.EINVAL


def test_ring_cache_argument_checks(L):
    """A ring KV cache (params kv_ring = 1) is a decode-only option for windowed
    layers; its slot count must hold the T + W - 1 visible positions and be a
    multiple of 16.  Everything here is refused on the host, before any launch."""
    import sliding_window_sink_bias_b300 as sa
    P = ctypes.c_void_p
    f = lambda x: P(256 * x)
    ws = L.sinkattn_decode_workspace_size(2, 4, 64, 8, 5000, 128)

    def dec(window, s_cap, max_seqlen, ring=1, t=4):
        p = sa.Params(0.0, 0, 0, ring)
        return L.sinkattn_decode_ex(f(1), f(1), f(1), f(1), f(1), window, 1e4, 2, t, s_cap,
                                    max_seqlen, 64, 8, ctypes.byref(p), f(1), ws, f(1), f(1),
                                    None)

    assert dec(0, 256, 5000) == sa.EINVAL      # global attention has no ring
    assert dec(128, 130, 5000) == sa.EINVAL    # fewer slots than T + W - 1 = 131
    assert dec(128, 136, 5000) == sa.EINVAL    # not a multiple of 16
    assert dec(128, 256, 5000, ring=2) == sa.EINVAL
    assert dec(128, 256, 5000, ring=0) == sa.EINVAL  # a plain cache must hold max_seqlen
    # the prefill reads no cache
    p = sa.Params(0.0, 0, 0, 1)
    st = L.sinkattn_prefill_ex(f(1), f(1), f(1), f(1), f(1), 1, 16, 16, 64, 8, 128, 1e4,
                               ctypes.byref(p), f(1), f(1), None)
    assert st == sa.EINVAL


def test_fp8_decode_argument_checks(L):
    """The FP8 decode needs both scale vectors and has no ring-cache form."""
    import sliding_window_sink_bias_b300 as sa
    P = ctypes.c_void_p
    f = lambda x: P(256 * x)
    ws = L.sinkattn_decode_workspace_size(2, 4, 64, 4, 100, 0)

    def dec(ks=1, vs=1, ring=0, window=0, s_cap=256):
        p = sa.Params(0.0, 0, 0, ring)
        return L.sinkattn_decode_fp8(f(1), f(1), f(1), None if ks is None else f(ks),
                                     None if vs is None else f(vs), f(1), f(1), window, 5e6, 2, 4,
                                     s_cap, 100, 64, 4, ctypes.byref(p), f(1), ws, f(1), f(1), None)

    assert dec(ks=None) == sa.EINVAL
    assert dec(vs=None) == sa.EINVAL
    assert dec(ring=1, window=128) == sa.EINVAL


def test_backward_workspace_size(L):
    sz = L.sinkattn_prefill_backward_workspace_size
    assert sz(4096, 64, 8) > sz(1024, 64, 8) > 0
    assert sz(-1, 64, 8) == 0 and sz(16, 64, 0) == 0 and sz(16, 12, 8) == 0


def test_backward_argument_checks(L):
    """Rejections that happen before any CUDA call (batch and total are
    non-zero here: an empty batch only clears dsink, on the device)."""
    import sliding_window_sink_bias_b300 as sa
    P = ctypes.c_void_p
    f = lambda x: None if x is None else P(256 * x)
    ws_ok = L.sinkattn_prefill_backward_workspace_size(16, 64, 8)

    def bwd(q=1, dq=1, total=16, max_seqlen=16, hq=64, hkv=8, scale=0.0, ring=0, ws=1,
            ws_bytes=None, q_off=0):
        p = sa.Params(scale, 0, 0, ring)
        qp = P(256 * q + q_off) if q is not None else None
        return L.sinkattn_prefill_backward(
            qp, f(1), f(1), f(1), f(1), 1, total, max_seqlen, hq, hkv, 128, 1e4, ctypes.byref(p),
            f(1), f(1), f(1), f(ws), ws_ok if ws_bytes is None else ws_bytes, f(dq), f(1), f(1),
            f(1), None)

    assert bwd(total=-1) == sa.EINVAL
    assert bwd(hq=64, hkv=7) == sa.EINVAL            # Hq not a multiple of Hkv
    assert bwd(hq=48, hkv=16) == sa.EUNSUPPORTED     # group of 3
    assert bwd(hq=128, hkv=1) == sa.EUNSUPPORTED     # group above 64
    assert bwd(ring=1) == sa.EINVAL                  # no ring cache in prefill
    assert bwd(max_seqlen=0) == sa.EINVAL
    assert bwd(scale=-1.0) == sa.EINVAL
    assert bwd(q=None) == sa.EINVAL
    assert bwd(dq=None) == sa.EINVAL
    assert bwd(q_off=8) == sa.EINVAL                 # q not 16-byte aligned
    assert bwd(ws=None) == sa.EWORKSPACE
    assert bwd(ws_bytes=ws_ok - 1) == sa.EWORKSPACE


def test_rotated_cache_argument_checks(L):
    """params k_rotated (a cache of keys already rotated at their positions) is a
    decode-only option taking 0 or 1; the prefill and the backward take raw keys
    and refuse it.  All refused on the host, before any launch."""
    import sliding_window_sink_bias_b300 as sa
    P = ctypes.c_void_p
    f = lambda x: P(256 * x)
    ws = L.sinkattn_decode_workspace_size(2, 4, 64, 4, 100, 0)
    p = sa.Params(0.0, 0, 0, 0, 2)
    assert L.sinkattn_decode_ex(f(1), f(1), f(1), f(1), f(1), 0, 5e6, 2, 4, 100, 100, 64, 4,
                                ctypes.byref(p), f(1), ws, f(1), f(1), None) == sa.EINVAL
    assert L.sinkattn_decode_fp8(f(1), f(1), f(1), f(1), f(1), f(1), f(1), 0, 5e6, 2, 4, 256,
                                 100, 64, 4, ctypes.byref(p), f(1), ws, f(1), f(1),
                                 None) == sa.EINVAL
    p = sa.Params(0.0, 0, 0, 0, 1)
    assert L.sinkattn_prefill_ex(f(1), f(1), f(1), f(1), f(1), 1, 16, 16, 64, 8, 128, 1e4,
                                 ctypes.byref(p), f(1), f(1), None) == sa.EINVAL
    wsb = L.sinkattn_prefill_backward_workspace_size(16, 64, 8)
    assert L.sinkattn_prefill_backward(
        f(1), f(1), f(1), f(1), f(1), 1, 16, 16, 64, 8, 128, 1e4, ctypes.byref(p), f(1), f(1),
        f(1), f(1), wsb, f(1), f(1), f(1), f(1), None) == sa.EINVAL
