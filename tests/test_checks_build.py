"""The checking build of the library (SINKATTN_CHECKS), on the GPU, without a fault.

libsinkattn_test.so is the same sources compiled with SINKATTN_CHECKS (and the
test hooks): inside every kernel, before the access, it checks each TMA copy's
x coordinate and shared-memory destination, each tcgen05.ld/st and MMA
operand's TMEM lane and columns (and that an MMA's two operands share a type),
and each global store's index against its tensor's extent.  A failed check
records SINKATTN_ECHECK with its site in the device status word and skips that
one access; barrier arrivals and MMA commits still happen.

The tests here
  * run one case of every kernel through the checking build: no check may
    fire, and the results must be the product build's bits exactly (the checks
    only guard accesses, they change no arithmetic);
  * make the checks fire without any access out of bounds: a test hook makes
    every extent look one row shorter (the last row's stores are skipped and
    nothing else changes) or admits fewer TMEM columns; the next call with the
    true limits is clean again.
The whole GPU suite can also run on the checking build:
SINKATTN_LIBRARY=<path of libsinkattn_test.so> pytest -m gpu."""
import ctypes
import os

import pytest
import torch

from helpers import assert_parity
from sliding_window_sink_bias_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sliding_window_sink_bias_b300")
TEST_LIB = os.path.join(PKG, "libsinkattn_test.so")
PROD_LIB = os.path.join(PKG, "libsinkattn.so")
DEV = "cuda"
# check sites (csrc/ptx.cuh and the kernels' stores)
TMEM_SITES = {0x03, 0x04, 0x05, 0x06}
BAND_STORE_SITES = {0x11, 0x12}
DECODE_STORE_SITES = {0x20, 0x21, 0x24}


def test_only_the_test_build_has_checks():
    from sliding_window_sink_bias_b300 import build
    build.build()
    assert not hasattr(ctypes.CDLL(PROD_LIB), "sinkattn_test_set_check_limits")
    assert hasattr(ctypes.CDLL(TEST_LIB), "sinkattn_test_set_check_limits")


def _use(monkeypatch, path):
    import sliding_window_sink_bias_b300 as sa
    monkeypatch.setattr(sa, "LIB_PATH", path)
    monkeypatch.setattr(sa, "_lib", None)
    return sa.lib()


def _set_limits(L, shrink, cols):
    L.sinkattn_test_set_check_limits.argtypes = [ctypes.c_int64, ctypes.c_uint32]
    L.sinkattn_test_set_check_limits.restype = ctypes.c_int
    assert L.sinkattn_test_set_check_limits(shrink, cols) == 0


# ---------------------------------------------------------------- the cases
def _prefill_case(hq, hkv, lens, window, base, seed, scale=None):
    inp = synth.prefill_inputs(lens, hq, hkv, window=window, rope_base=base, seed=seed, device="cpu")

    def run(sa, out=None, lse=None):
        return sa.prefill(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.sink.to(DEV),
                          inp.cu_seqlens.to(DEV), max_seqlen=max(lens), window=window,
                          rope_base=base, out=out, lse=lse, scale=scale)

    def oracle(om):
        return om.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, window=window,
                          rope_base=base, scale=scale)
    return run, oracle


def _decode_case(hkv, lens, t, s_cap, window, base, seed, ring=False):
    inp = synth.decode_inputs(lens, t, s_cap, 64, hkv, window=window, rope_base=base, seed=seed,
                              device="cpu")
    kc, vc = inp.kcache, inp.vcache
    if ring:
        # position j of sequence b at slot j % s_cap of a ring of s_cap slots
        kfull = synth.randn_bf16((len(lens), max(lens), hkv, 192), seed, "kcache")
        vfull = synth.randn_bf16((len(lens), max(lens), hkv, 128), seed, "vcache")
        kc = torch.zeros(len(lens), s_cap, hkv, 192, dtype=torch.bfloat16)
        vc = torch.zeros(len(lens), s_cap, hkv, 128, dtype=torch.bfloat16)
        for b, L in enumerate(lens):
            for j in range(max(0, L - s_cap), L):
                kc[b, j % s_cap] = kfull[b, j]
                vc[b, j % s_cap] = vfull[b, j]

    def run(sa, out=None, lse=None):
        return sa.decode(inp.q.to(DEV), kc.to(DEV), vc.to(DEV), inp.seqlens.to(DEV),
                         inp.sink.to(DEV), max_seqlen=max(lens), window=window, rope_base=base,
                         out=out, lse=lse, kv_ring=ring)

    def oracle(om):
        if ring:
            return om.decode(inp.q.to(torch.float64), kfull.to(torch.float64),
                             vfull.to(torch.float64), inp.seqlens, inp.sink, window=window,
                             rope_base=base)
        return om.decode(inp.q.to(torch.float64), kc.to(torch.float64), vc.to(torch.float64),
                         inp.seqlens, inp.sink, window=window, rope_base=base)
    return run, oracle


def _fp8_case(lens, seed):
    inp = synth.decode_inputs(lens, 4, max(lens), 64, 4, window=0, rope_base=5e6, seed=seed,
                              device="cpu")

    def q8(x, s):
        amax = x.float().abs().amax(dim=(0, 1, 3)).clamp_min(1e-6)
        sc = (amax / 224.0) * (0.5 + torch.rand(x.shape[2], generator=torch.Generator().manual_seed(s)))
        return (x.float() / sc[None, None, :, None]).to(torch.float8_e4m3fn), sc.float()
    k8, ks = q8(inp.kcache, seed)
    v8, vs = q8(inp.vcache, seed + 1)

    def run(sa, out=None, lse=None):
        return sa.decode_fp8(inp.q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV),
                             inp.seqlens.to(DEV), inp.sink.to(DEV), max_seqlen=max(lens),
                             window=0, rope_base=5e6, out=out, lse=lse)

    def oracle(om):
        deq = lambda a, s: a.to(torch.float64) * s.to(torch.float64)[None, None, :, None]
        return om.decode(inp.q.to(torch.float64), deq(k8, ks), deq(v8, vs), inp.seqlens,
                         inp.sink, window=0, rope_base=5e6)
    return run, oracle


CASES = {
    # band kernel (8 heads a KV head, W <= 128), ragged lengths
    "swa_band": lambda: _prefill_case(64, 8, [200, 57, 1, 300], 128, 1e4, 61),
    # causal kernel with 2 heads a KV head and a window, 1 head a KV head global
    "causal_g2_window": lambda: _prefill_case(16, 8, [150, 33], 64, 1e4, 62),
    "causal_g1_global": lambda: _prefill_case(8, 8, [140, 9], 0, 5e6, 63),
    # general kernel: a negative logit scale
    "general_neg_scale": lambda: _prefill_case(64, 8, [150, 33], 128, 1e4, 71, scale=-0.05),
    # causal kernel: global, several sequences; and with a window past one block
    "ga_causal": lambda: _prefill_case(64, 4, [300, 129, 5], 0, 5e6, 64),
    "causal_window": lambda: _prefill_case(64, 8, [700, 129, 1], 256, 1e4, 70),
    # decode: long caches cut over many CTAs (partials merged in the launch)
    "decode_ga_split": lambda: _decode_case(4, [20000, 9000, 0, 3], 4, 20000, 0, 5e6, 65),
    "decode_swa_ring": lambda: _decode_case(8, [5000, 131, 2], 4, 144, 128, 1e4, 66, ring=True),
    "decode_fp8": lambda: _fp8_case([3000, 64, 65], 67),
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_no_check_fires_and_results_match_product_bits(oracle_mod, monkeypatch, name):
    run, oracle = CASES[name]()
    sa_prod = _use(monkeypatch, PROD_LIB)
    import sliding_window_sink_bias_b300 as sa
    o_p, l_p = run(sa)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    L = _use(monkeypatch, TEST_LIB)
    _set_limits(L, 0, 512)
    o_c, l_c = run(sa)
    st, word = sa.device_status()
    assert st == sa.OK, (name, hex(word))
    assert torch.equal(o_c.view(torch.int16), o_p.view(torch.int16)), name
    assert torch.equal(l_c.view(torch.int32), l_p.view(torch.int32)), name
    ro, rl = oracle(oracle_mod)
    assert_parity(o_c, l_c, ro, rl, name)
    del sa_prod


@pytest.mark.gpu
def test_backward_no_check_fires_and_matches_product_bits(monkeypatch):
    import sliding_window_sink_bias_b300 as sa
    for hq, hkv, lens, window, base, seed in [(64, 8, [300, 77], 128, 1e4, 68),
                                              (64, 4, [257, 31], 0, 5e6, 69)]:
        inp = synth.prefill_inputs(lens, hq, hkv, window=window, rope_base=base, seed=seed,
                                   device=DEV)
        dout = synth.randn_bf16((inp.total, hq, 128), seed, "v", DEV)
        kw = dict(max_seqlen=max(lens), window=window, rope_base=base)
        res = []
        for path in (PROD_LIB, TEST_LIB):
            L = _use(monkeypatch, path)
            if path == TEST_LIB:
                _set_limits(L, 0, 512)
            out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, **kw)
            grads = sa.prefill_backward(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, out, lse,
                                        dout, **kw)
            st, word = sa.device_status()
            assert st == sa.OK, (path, hex(word))
            res.append([out, lse, *grads])
        for a, b in zip(*res):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (hq, hkv, window)


@pytest.mark.gpu
@pytest.mark.parametrize("name,sites", [("swa_band", BAND_STORE_SITES),
                                        ("decode_ga_split", DECODE_STORE_SITES)])
def test_shrunk_extent_skips_exactly_the_last_row(monkeypatch, name, sites):
    """With every extent one row short, the checks skip the last output row's
    stores (out and lse keep what the caller put there) and record the site;
    every other row is the normal result, bit for bit."""
    import sliding_window_sink_bias_b300 as sa
    run, _ = CASES[name]()
    L = _use(monkeypatch, TEST_LIB)
    _set_limits(L, 0, 512)
    o_ref, l_ref = run(sa)
    assert sa.device_status()[0] == sa.OK
    out = torch.full_like(o_ref, 7.0)
    lse = torch.full_like(l_ref, 7.0)
    try:
        _set_limits(L, 1, 512)
        run(sa, out=out, lse=lse)
        st, word = sa.device_status()
    finally:
        _set_limits(L, 0, 512)
    assert st == sa.ECHECK and word & 2, hex(word)
    assert ((word >> 16) & 0xFF) in sites, hex(word)
    of, lf = out.reshape(-1, 128), lse.reshape(-1)
    assert torch.all(of[-1] == 7.0) and float(lf[-1]) == 7.0
    assert torch.equal(of[:-1].view(torch.int16), o_ref.reshape(-1, 128)[:-1].view(torch.int16))
    assert torch.equal(lf[:-1].view(torch.int32), l_ref.reshape(-1)[:-1].view(torch.int32))
    # the true limits again: clean, same bits
    o2, l2 = run(sa)
    assert sa.device_status()[0] == sa.OK
    assert torch.equal(o2.view(torch.int16), o_ref.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["swa_band", "ga_causal", "decode_ga_split"])
def test_fewer_tmem_columns_fire_tmem_checks(monkeypatch, name):
    """Admitting 256 of the 512 TMEM columns makes the accesses to the upper
    half (every kernel keeps accumulators or operands there) fail their checks;
    they are skipped, the launch still ends by itself, the status names a TMEM
    site, and the next call is clean with the normal bits."""
    import sliding_window_sink_bias_b300 as sa
    run, _ = CASES[name]()
    L = _use(monkeypatch, TEST_LIB)
    _set_limits(L, 0, 512)
    o_ref, l_ref = run(sa)
    assert sa.device_status()[0] == sa.OK
    try:
        _set_limits(L, 0, 256)
        run(sa)
        st, word = sa.device_status()
    finally:
        _set_limits(L, 0, 512)
    assert st == sa.ECHECK and word & 2 and not word & 1, hex(word)
    assert ((word >> 16) & 0xFF) in TMEM_SITES, hex(word)
    o2, l2 = run(sa)
    assert sa.device_status()[0] == sa.OK
    assert torch.equal(o2.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(l2.view(torch.int32), l_ref.view(torch.int32))
