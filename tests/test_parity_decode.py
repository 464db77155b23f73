"""GPU parity: sinkattn_decode (MTP verify, split-KV with the merge of cut units) against the oracle."""
import math

import numpy as np
import pytest
import torch

from helpers import assert_parity
from sliding_window_sink_bias_b300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run_decode(oracle_mod, seqlens, t, s_cap, hq, hkv, window, base, *, seed=0, sink=None,
               **kw):
    import sliding_window_sink_bias_b300 as sa
    inp = synth.decode_inputs(seqlens, t, s_cap, hq, hkv, window=window, rope_base=base,
                              seed=seed, device="cpu")
    if sink is not None:
        inp.sink = torch.tensor(sink, dtype=torch.float32)
    out, lse = sa.decode(inp.q.to(DEV), inp.kcache.to(DEV), inp.vcache.to(DEV),
                         inp.seqlens.to(DEV), inp.sink.to(DEV), max_seqlen=max(seqlens),
                         window=window, rope_base=base, **kw)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    okw = {}
    if kw.get("rope_style"):
        okw["rope_style"] = kw["rope_style"]
    ro, rl = oracle_mod.decode(inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink,
                               window=window, rope_base=base, **okw)
    return out, lse, ro, rl


@pytest.mark.parametrize("window,hkv,base", [(0, 4, 5e6), (128, 8, 1e4)])
def test_mtp_verify_small(oracle_mod, window, hkv, base):
    seqlens = [4, 5, 1000, 2999, 3000, 131, 132]
    o, l, ro, rl = run_decode(oracle_mod, seqlens, 4, 3000, 64, hkv, window, base, seed=1)
    assert_parity(o, l, ro, rl, f"decode W={window}")


@pytest.mark.parametrize("window,hkv,base", [(0, 4, 5e6), (128, 8, 1e4), (16, 4, 1e4)])
def test_lengths_at_block_edges(oracle_mod, window, hkv, base):
    # cache lengths on both sides of the 64-key block edges: the blocks are cut
    # across CTAs, so some CTA segments hold keys that some query rows cannot
    # see (e.g. a query at position 127 against keys 128..130)
    seqlens = [1, 2, 3, 4, 5, 63, 64, 65, 66, 67, 68, 127, 128, 129, 130, 131, 132, 191, 192, 193,
               255, 256, 257]
    o, l, ro, rl = run_decode(oracle_mod, seqlens, 4, 257, 64, hkv, window, base, seed=9)
    assert_parity(o, l, ro, rl, f"block edges W={window}")


@pytest.mark.parametrize("t", [1, 2, 3, 8])
def test_token_counts(oracle_mod, t):
    o, l, ro, rl = run_decode(oracle_mod, [t, 700, 1500], t, 1600, 64, 4, 0, 5e6, seed=t)
    assert_parity(o, l, ro, rl, f"T={t}")


def test_many_splits_long_cache(oracle_mod):
    # 20000 keys -> many chunks per (sequence, kv head): the merge must count the sink once
    o, l, ro, rl = run_decode(oracle_mod, [20000, 9000], 4, 20000, 64, 4, 0, 5e6, seed=2)
    assert_parity(o, l, ro, rl, "long cache")


def test_sink_extremes_decode(oracle_mod):
    sinks = [(-math.inf, -20.0, 0.0, 20.0)[h % 4] for h in range(64)]
    for window, hkv in ((0, 4), (128, 8)):
        o, l, ro, rl = run_decode(oracle_mod, [600, 4], 4, 600, 64, hkv, window, 1e4, seed=3,
                                  sink=sinks)
        assert_parity(o, l, ro, rl, f"decode sinks W={window}")


def test_short_cache_rows_empty(oracle_mod):
    # seqlen < T: queries at negative positions see nothing -> out 0, lse sink
    o, l, ro, rl = run_decode(oracle_mod, [2, 0, 9], 4, 16, 64, 4, 0, 5e6, seed=4)
    assert_parity(o, l, ro, rl, "short cache")


def test_rope_half_split_decode(oracle_mod):
    o, l, ro, rl = run_decode(oracle_mod, [333, 1000], 4, 1000, 64, 4, 0, 5e6, seed=5,
                              rope_style=1)
    assert_parity(o, l, ro, rl, "decode half-split rope")


def test_decode_deterministic():
    import sliding_window_sink_bias_b300 as sa
    inp = synth.decode_inputs([5000, 70], 4, 5000, 64, 4, window=0, rope_base=5e6, seed=6,
                              device=DEV)
    args = (inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink)
    o1, l1 = sa.decode(*args, max_seqlen=5000, window=0, rope_base=5e6)
    o2, l2 = sa.decode(*args, max_seqlen=5000, window=0, rope_base=5e6)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


@pytest.mark.slow
def test_mtp_decode_full_size_sampled(oracle_mod):
    """B=64, T=4, S_cap=262144, seqlens U[65536, 262144]: GA (4 KV heads) and SWA
    (8 KV heads, W=128) layers; a few sequences checked against the oracle."""
    import sliding_window_sink_bias_b300 as sa
    for name in ("mtp_decode_ga_b64_t4", "mtp_decode_swa_b64_t4"):
        wl = synth.WORKLOADS[name]
        lens = synth.uniform_lengths(wl["batch"], wl["len_lo"], wl["len_hi"], seed=0)
        inp = synth.decode_inputs(lens, wl["t"], wl["s_cap"], wl["hq"], wl["hkv"],
                                  window=wl["window"], rope_base=wl["rope_base"], seed=0,
                                  device=DEV)
        out, lse = sa.decode(inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink,
                             max_seqlen=max(lens), window=wl["window"],
                             rope_base=wl["rope_base"])
        torch.cuda.synchronize()
        assert sa.device_status()[0] == sa.OK
        picks = [int(np.argmax(lens)), int(np.argmin(lens)), 17]
        for b in picks:
            L = lens[b]
            ro, rl = oracle_mod.decode(inp.q[b:b + 1].cpu(), inp.kcache[b:b + 1, :L].cpu(),
                                       inp.vcache[b:b + 1, :L].cpu(),
                                       torch.tensor([L], dtype=torch.int32), inp.sink.cpu(),
                                       window=wl["window"], rope_base=wl["rope_base"])
            assert_parity(out[b:b + 1], lse[b:b + 1], ro, rl, f"{name} b={b}")
        del inp, out, lse
        torch.cuda.empty_cache()


def _nan_past_end(cache, seqlens):
    for b, L in enumerate(seqlens):
        cache[b, L:] = float("nan")


@pytest.mark.parametrize("window,hkv,base", [(0, 4, 5e6), (128, 8, 1e4)])
def test_cache_rows_past_the_end_are_never_used(oracle_mod, window, hkv, base):
    """Rows at or past seqlens[b] may hold anything (NaN here): the last 64-key
    block of a sequence reads some of them, and the result must not change."""
    import sliding_window_sink_bias_b300 as sa
    seqlens = [4, 65, 130, 1000, 1001, 77]
    inp = synth.decode_inputs(seqlens, 4, 1100, 64, hkv, window=window, rope_base=base, seed=11,
                              device="cpu")
    _nan_past_end(inp.kcache, seqlens)
    _nan_past_end(inp.vcache, seqlens)
    out, lse = sa.decode(inp.q.to(DEV), inp.kcache.to(DEV), inp.vcache.to(DEV),
                         inp.seqlens.to(DEV), inp.sink.to(DEV), max_seqlen=max(seqlens),
                         window=window, rope_base=base)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.decode(inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink,
                               window=window, rope_base=base)
    assert_parity(out, lse, ro, rl, f"NaN past the end W={window}")


def _ring_of(full, seqlens, cap, keep):
    """The ring a sliding-window layer keeps: slot j % cap holds position j for
    the last `keep` positions; every other slot holds NaN."""
    ring = torch.full((full.shape[0], cap) + tuple(full.shape[2:]), float("nan"),
                      dtype=full.dtype)
    for b, L in enumerate(seqlens):
        idx = torch.arange(max(0, L - keep), L)
        ring[b, idx % cap] = full[b, idx]
    return ring


@pytest.mark.parametrize("cap,window,t", [(144, 128, 4), (256, 128, 4), (144, 128, 1),
                                          (144, 128, 8), (32, 16, 4)])
def test_ring_cache_matches_full_cache(oracle_mod, cap, window, t):
    """A ring of `cap` slots holding only the last T + W - 1 positions gives the
    decode of the full cache; lengths below, at and far past the ring size put
    the ring's seam at every offset of the 64-key blocks."""
    import sliding_window_sink_bias_b300 as sa
    seqlens = [t, 100, cap - 1, cap, cap + 1, 300, 1000, 5003, 4099 + t]
    full = synth.decode_inputs(seqlens, t, max(seqlens), 64, 8, window=window, rope_base=1e4,
                               seed=12 + t, device="cpu")
    keep = window + t - 1
    kr, vr = _ring_of(full.kcache, seqlens, cap, keep), _ring_of(full.vcache, seqlens, cap, keep)
    out, lse = sa.decode(full.q.to(DEV), kr.to(DEV), vr.to(DEV), full.seqlens.to(DEV),
                         full.sink.to(DEV), max_seqlen=max(seqlens), window=window,
                         rope_base=1e4, kv_ring=True)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.decode(full.q, full.kcache, full.vcache, full.seqlens, full.sink,
                               window=window, rope_base=1e4)
    assert_parity(out, lse, ro, rl, f"ring cap={cap} W={window} T={t}")


# ------------------------------------------------ cache of keys already rotated
def rotated_cache(oracle_mod, kcache, base, rope_style=0):
    """The cache a serving layer would keep if it stored keys after RoPE: every
    key rotated at its own position (slot j = position j) by the oracle's fp64
    rotation, then rounded to bf16."""
    pos = np.arange(kcache.shape[1], dtype=np.float64)[None, :, None]
    kr = oracle_mod.rope_rows(kcache.to(torch.float64).numpy(), pos, base=base,
                              rope_style=rope_style)
    return torch.from_numpy(kr).to(torch.bfloat16)


@pytest.mark.parametrize("window,hkv,base,style", [(0, 4, 5e6, 0), (128, 8, 1e4, 0),
                                                   (0, 4, 1e4, 1)])
def test_rotated_cache(oracle_mod, window, hkv, base, style):
    """k_rotated: the kernel reads keys a cache already holds rotated (in bf16)
    and rotates only q; compared with the oracle on that same rotated cache."""
    import sliding_window_sink_bias_b300 as sa
    seqlens = [4, 5, 63, 64, 65, 1000, 2999, 3000, 131]
    inp = synth.decode_inputs(seqlens, 4, 3000, 64, hkv, window=window, rope_base=base, seed=31,
                              device="cpu")
    kc = rotated_cache(oracle_mod, inp.kcache, base, style)
    _nan_past_end(kc, seqlens)
    out, lse = sa.decode(inp.q.to(DEV), kc.to(DEV), inp.vcache.to(DEV), inp.seqlens.to(DEV),
                         inp.sink.to(DEV), max_seqlen=max(seqlens), window=window,
                         rope_base=base, rope_style=style, k_rotated=True)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.decode(inp.q, kc, inp.vcache, inp.seqlens, inp.sink, window=window,
                               rope_base=base, rope_style=style, k_rotated=True)
    assert_parity(out, lse, ro, rl, f"rotated cache W={window} style={style}")


@pytest.mark.parametrize("cap,t", [(144, 4), (32, 1)])
def test_rotated_ring_cache(oracle_mod, cap, t):
    """A ring cache of keys rotated at their absolute positions (slot j % cap
    holds position j, rotated at j)."""
    import sliding_window_sink_bias_b300 as sa
    window = 128 if cap >= 131 else 16
    seqlens = [t, 100, cap - 1, cap, cap + 1, 1000, 4099 + t]
    full = synth.decode_inputs(seqlens, t, max(seqlens), 64, 8, window=window, rope_base=1e4,
                               seed=33 + t, device="cpu")
    kfull = rotated_cache(oracle_mod, full.kcache, 1e4)
    keep = window + t - 1
    kr, vr = _ring_of(kfull, seqlens, cap, keep), _ring_of(full.vcache, seqlens, cap, keep)
    out, lse = sa.decode(full.q.to(DEV), kr.to(DEV), vr.to(DEV), full.seqlens.to(DEV),
                         full.sink.to(DEV), max_seqlen=max(seqlens), window=window,
                         rope_base=1e4, kv_ring=True, k_rotated=True)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.decode(full.q, kfull, full.vcache, full.seqlens, full.sink,
                               window=window, rope_base=1e4, k_rotated=True)
    assert_parity(out, lse, ro, rl, f"rotated ring cap={cap} T={t}")
