"""GPU parity: sinkattn_decode (MTP verify, split-KV + combine) against the oracle."""
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
    # 20000 keys -> many chunks per (sequence, kv head): the combine must count the sink once
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
