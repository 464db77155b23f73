"""GPU parity: sinkattn_prefill (through the C ABI) against the fp64 oracle.

Inputs come from the seeded generators of sliding_window_sink_bias_b300.synth;
the same bf16 tensors go to the kernel (on the GPU) and to the oracle (on the
CPU).  Gate: max-abs error of out <= 1e-2 and of lse <= 2e-3.
"""
import math

import numpy as np
import pytest
import torch

from helpers import assert_parity, sample_rows
from sliding_window_sink_bias_b300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run_case(oracle_mod, seqlens, hq, hkv, window, base, *, seed=0, sink=None, rows=None,
             rope_style=0, rope_off=False, scale=None):
    import sliding_window_sink_bias_b300 as sa
    inp = synth.prefill_inputs(seqlens, hq, hkv, window=window, rope_base=base, seed=seed,
                               device="cpu")
    if sink is not None:
        inp.sink = torch.tensor(sink, dtype=torch.float32)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    out, lse = sa.prefill(q, k, v, inp.sink.to(DEV), inp.cu_seqlens.to(DEV),
                          max_seqlen=max(seqlens) if seqlens else 0, window=window,
                          rope_base=base, rope_style=rope_style, rope_off=rope_off, scale=scale)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, window=window,
                                rope_base=base, rope_style=rope_style,
                                drot=0 if rope_off else 64, scale=scale, rows=rows)
    if rows is None:
        return out, lse, ro, rl
    tok = torch.as_tensor(rows // hq)
    hd = torch.as_tensor(rows % hq)
    return out.cpu()[tok, hd], lse.cpu()[tok, hd], ro, rl


def test_tiny_swa_prefill_full(oracle_mod):
    # batch 1 x 512 tokens, 64/8 heads, window 128, base 1e4, seed 0: every row
    o, l, ro, rl = run_case(oracle_mod, [512], 64, 8, 128, 1e4)
    assert_parity(o, l, ro, rl, "tiny swa")


def test_ga_small_varlen_full(oracle_mod):
    o, l, ro, rl = run_case(oracle_mod, [300, 1, 700, 129], 64, 4, 0, 5e6, seed=1)
    assert_parity(o, l, ro, rl, "ga varlen")


@pytest.mark.parametrize("window", [1, 16, 127, 128, 129, 144, 200, 1000])
def test_window_sweep(oracle_mod, window):
    o, l, ro, rl = run_case(oracle_mod, [257, 16, 0, 33, 300], 64, 8, window, 1e4, seed=2)
    assert_parity(o, l, ro, rl, f"window {window}")


@pytest.mark.parametrize("hq,hkv,window", [(64, 16, 129), (64, 8, 256), (64, 4, 300),
                                           (32, 2, 150), (64, 1, 513), (64, 8, 700)])
def test_causal_kernel_windows(oracle_mod, hq, hkv, window):
    """Windows too wide for one 144-key block with G >= 4 run on the causal
    kernel: an item's first key block is the one its window reaches and the
    window's low edge is masked; ragged sequences, windows across block edges."""
    o, l, ro, rl = run_case(oracle_mod, [700, 129, 1, 300], hq, hkv, window, 1e4, seed=window)
    assert_parity(o, l, ro, rl, f"Hq={hq} Hkv={hkv} W={window}")


@pytest.mark.parametrize("L", [1, 2, 15, 16, 17, 127, 128, 129, 255, 300])
@pytest.mark.parametrize("window", [0, 128])
def test_ragged_lengths(oracle_mod, L, window):
    hkv = 8 if window else 4
    o, l, ro, rl = run_case(oracle_mod, [L, 3], 64, hkv, window, 1e4, seed=L)
    assert_parity(o, l, ro, rl, f"L={L} W={window}")


def test_sink_extremes(oracle_mod):
    sinks = [(-math.inf, -20.0, 0.0, 20.0)[h % 4] for h in range(64)]
    for window, hkv in ((128, 8), (0, 4)):
        o, l, ro, rl = run_case(oracle_mod, [200, 77], 64, hkv, window, 1e4, seed=3, sink=sinks)
        assert_parity(o, l, ro, rl, f"sinks W={window}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 2), (64, 1), (128, 1), (4, 4)])
def test_group_sizes(oracle_mod, hq, hkv):
    for window in (0, 64):
        o, l, ro, rl = run_case(oracle_mod, [190, 64], hq, hkv, window, 1e4, seed=hq + hkv)
        assert_parity(o, l, ro, rl, f"Hq={hq} Hkv={hkv} W={window}")


def test_rope_variants_and_scale(oracle_mod):
    for kw in (dict(rope_style=1), dict(rope_off=True), dict(scale=0.11)):
        # band, causal, causal with a window, general
        for window, hkv in ((128, 8), (0, 4), (300, 16), (64, 32)):
            o, l, ro, rl = run_case(oracle_mod, [150], 64, hkv, window, 1e4, seed=4, **kw)
            assert_parity(o, l, ro, rl, f"{kw} W={window}")


@pytest.mark.parametrize("window,hkv", [(128, 8), (0, 4), (64, 32), (0, 64), (300, 16)])
def test_negative_scale(oracle_mod, window, hkv):
    """A logit scale < 0 (the general kernel: the running max over the scaled
    logits) on the band's, the causal kernel's and 1-2 heads a KV head's
    shapes."""
    for scale in (-0.05, -1.0 / 192 ** 0.5):
        o, l, ro, rl = run_case(oracle_mod, [150, 1, 70], 64, hkv, window, 1e4, seed=8,
                                scale=scale)
        assert_parity(o, l, ro, rl, f"scale={scale:.3f} W={window} Hkv={hkv}")


def test_long_positions_rope(oracle_mod):
    # large positions stress the RoPE angle: GA base 5e6, rows near the end of 20000 tokens
    L = 20000
    toks, rows = sample_rows(L, 64, 24, seed=5, must=(L - 1, L - 2, 16383, 0))
    o, l, ro, rl = run_case(oracle_mod, [L], 64, 4, 0, 5e6, seed=5, rows=rows)
    assert_parity(o, l, ro.reshape(-1, 128), rl, "long GA")
    o, l, ro, rl = run_case(oracle_mod, [L], 64, 8, 128, 1e4, seed=6, rows=rows)
    assert_parity(o, l, ro.reshape(-1, 128), rl, "long SWA")


def test_deterministic_bits():
    import sliding_window_sink_bias_b300 as sa
    for window, hkv, base in ((128, 8, 1e4), (0, 4, 5e6)):
        inp = synth.prefill_inputs([1000, 37], 64, hkv, window=window, rope_base=base, seed=7,
                                   device=DEV)
        args = (inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens)
        o1, l1 = sa.prefill(*args, max_seqlen=1000, window=window, rope_base=base)
        o2, l2 = sa.prefill(*args, max_seqlen=1000, window=window, rope_base=base)
        torch.cuda.synchronize()
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_empty_batch_is_noop():
    import sliding_window_sink_bias_b300 as sa
    inp = synth.prefill_inputs([0, 0], 64, 8, window=128, rope_base=1e4, device=DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, max_seqlen=0,
                          window=128, rope_base=1e4)
    assert out.numel() == 0 and lse.numel() == 0


# ------------------------------------------------------------- full size, sampled
@pytest.mark.slow
def test_swa_prefill_bulk_sampled(oracle_mod):
    """4 x 32768 tokens, 64/8 heads, W=128: the benchmark's launch, sampled rows."""
    import sliding_window_sink_bias_b300 as sa
    wl = synth.WORKLOADS["swa_prefill_4x32768"]
    inp = synth.prefill_inputs(wl["seqlens"], wl["hq"], wl["hkv"], window=wl["window"],
                               rope_base=wl["rope_base"], seed=0, device=DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens,
                          max_seqlen=inp.max_seqlen, window=wl["window"],
                          rope_base=wl["rope_base"])
    torch.cuda.synchronize()
    for b in (0, 3):
        s0 = b * 32768
        toks, rows = sample_rows(32768, 64, 24, seed=10 + b, must=(0, 1, 127, 128, 32767))
        sl = slice(s0, s0 + 32768)
        ro, rl = oracle_mod.prefill(inp.q[sl].cpu(), inp.k[sl].cpu(), inp.v[sl].cpu(),
                                    inp.sink.cpu(), np.array([0, 32768], dtype=np.int32),
                                    window=128, rope_base=1e4, rows=rows)
        tok = torch.as_tensor(rows // 64) + s0
        hd = torch.as_tensor(rows % 64)
        assert_parity(out[tok.to(DEV), hd.to(DEV)], lse[tok.to(DEV), hd.to(DEV)], ro, rl,
                      f"swa bulk seq {b}")


@pytest.mark.slow
def test_swa_w512_prefill_sampled(oracle_mod):
    """1 x 32768 tokens, 64/8 heads, W=512 (the causal kernel with a window, as
    the benchmark runs it): sampled rows, including both sides of the window's
    edge and of block boundaries."""
    import sliding_window_sink_bias_b300 as sa
    wl = synth.WORKLOADS["swa_w512_prefill_1x32768"]
    inp = synth.prefill_inputs(wl["seqlens"], wl["hq"], wl["hkv"], window=wl["window"],
                               rope_base=wl["rope_base"], seed=0, device=DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens,
                          max_seqlen=inp.max_seqlen, window=wl["window"],
                          rope_base=wl["rope_base"])
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    L = 32768
    toks, rows = sample_rows(L, 64, 24, seed=30,
                             must=(0, 15, 16, 127, 128, 511, 512, 513, 639, 640, L - 1))
    ro, rl = oracle_mod.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.sink.cpu(),
                                np.array([0, L], dtype=np.int32), window=512,
                                rope_base=wl["rope_base"], rows=rows)
    tok = torch.as_tensor(rows // 64).to(DEV)
    hd = torch.as_tensor(rows % 64).to(DEV)
    assert_parity(out[tok, hd], lse[tok, hd], ro, rl, "swa w512")


@pytest.mark.slow
def test_swa_g2_prefill_sampled(oracle_mod):
    """1 x 32768 tokens, 64/32 heads, W=128 (the causal kernel with tiles of
    64 tokens x 2 heads, a lane quad's rows two tokens apart): sampled rows."""
    import sliding_window_sink_bias_b300 as sa
    wl = synth.WORKLOADS["swa_g2_prefill_1x32768"]
    inp = synth.prefill_inputs(wl["seqlens"], wl["hq"], wl["hkv"], window=wl["window"],
                               rope_base=wl["rope_base"], seed=0, device=DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens,
                          max_seqlen=inp.max_seqlen, window=wl["window"],
                          rope_base=wl["rope_base"])
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    L = 32768
    toks, rows = sample_rows(L, 64, 24, seed=31, must=(0, 63, 64, 127, 128, 191, 192, L - 1))
    ro, rl = oracle_mod.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.sink.cpu(),
                                np.array([0, L], dtype=np.int32), window=128,
                                rope_base=wl["rope_base"], rows=rows)
    tok = torch.as_tensor(rows // 64).to(DEV)
    hd = torch.as_tensor(rows % 64).to(DEV)
    assert_parity(out[tok, hd], lse[tok, hd], ro, rl, "swa g2")


@pytest.mark.slow
def test_ga_prefill_long_sampled(oracle_mod):
    """1 x 131072 tokens, 64/4 heads, global, base 5e6: sampled rows."""
    import sliding_window_sink_bias_b300 as sa
    wl = synth.WORKLOADS["ga_prefill_1x131072"]
    inp = synth.prefill_inputs(wl["seqlens"], wl["hq"], wl["hkv"], window=0,
                               rope_base=wl["rope_base"], seed=0, device=DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens,
                          max_seqlen=inp.max_seqlen, window=0, rope_base=wl["rope_base"])
    torch.cuda.synchronize()
    L = 131072
    toks, rows = sample_rows(L, 64, 10, seed=20, must=(0, 7, 8, 65535, L - 1))
    ro, rl = oracle_mod.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), inp.sink.cpu(),
                                np.array([0, L], dtype=np.int32), window=0,
                                rope_base=wl["rope_base"], rows=rows)
    tok = torch.as_tensor(rows // 64).to(DEV)
    hd = torch.as_tensor(rows % 64).to(DEV)
    assert_parity(out[tok, hd], lse[tok, hd], ro, rl, "ga long")


@pytest.mark.slow
@pytest.mark.parametrize("layer", ["swa", "ga"])
def test_hybrid_block_ragged_sampled(oracle_mod, layer):
    """The ragged hybrid block at full size (8 sequences of log-uniform lengths in
    [4096, 131072], seed 0, packed through cu_seqlens): one SWA layer (64/8, W=128,
    base 1e4) and the GA layer (64/4, global, base 5e6), each with its own sink,
    the inputs and sinks the benchmark draws.  Every sequence is sampled: its
    first and last rows, rows 127 and 128 (the window's edge), and 16 more, all
    64 heads.  This reaches the band kernel's ring refill at every sequence
    boundary and the causal kernel's longest-first schedule across sequences."""
    import sliding_window_sink_bias_b300 as sa
    wl = synth.WORKLOADS["hybrid_block_ragged_8seq"]
    lens = synth.log_uniform_lengths(wl["n_seq"], wl["len_lo"], wl["len_hi"], seed=0)
    hq = wl["hq"]
    if layer == "swa":
        hkv, window, base, seed, sink_seed = wl["swa_hkv"], wl["window"], wl["swa_base"], 0, 10
    else:
        hkv, window, base, seed, sink_seed = wl["ga_hkv"], 0, wl["ga_base"], 1, 10 + wl["swa_layers"]
    inp = synth.prefill_inputs(lens, hq, hkv, window=window, rope_base=base, seed=seed,
                               device=DEV)
    sink = synth.sink_vector(hq, seed=sink_seed, device=DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, sink, inp.cu_seqlens, max_seqlen=max(lens),
                          window=window, rope_base=base)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    cu = np.concatenate([[0], np.cumsum(lens)])
    for b, L in enumerate(lens):
        s0 = int(cu[b])
        toks, rows = sample_rows(L, hq, 20, seed=30 + b, must=(0, 127, 128, L - 1))
        hi = int(toks.max()) + 1  # keys past the last sampled row are never seen
        sl = slice(s0, s0 + hi)
        ro, rl = oracle_mod.prefill(inp.q[sl].cpu(), inp.k[sl].cpu(), inp.v[sl].cpu(),
                                    sink.cpu(), np.array([0, hi], dtype=np.int32),
                                    window=window, rope_base=base, rows=rows)
        tok = (torch.as_tensor(rows // hq) + s0).to(DEV)
        hd = torch.as_tensor(rows % hq).to(DEV)
        assert_parity(out[tok, hd], lse[tok, hd], ro, rl, f"hybrid {layer} seq {b} (L={L})")
