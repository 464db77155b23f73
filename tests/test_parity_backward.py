"""GPU parity: sinkattn_prefill_backward against the oracle's fp64 backward.

Tolerance (the target states none for the backward; derived from the
arithmetic): every gradient is a sum of products of bf16 values with fp32
accumulation, where P and dS are rounded to bf16 (relative 2^-9 each), the
rotated q and k are rounded to bf16 (2^-9), D = dO . o comes from the bf16
forward output (2^-9), and the result is rounded to bf16 (2^-9).  Those five
roundings give a worst-case relative error near 5 * 2^-9 = 1e-2 of the
gradient's scale.  The bounds are per row (one token and head):
  dk, dv: |error| <= 2e-2 (|row| + 0.05 |tensor|), where |row| is the row's
          largest reference magnitude and |tensor| the tensor's: every row is
          held to its own scale down to 5% of the tensor's (measured: within
          0.7% of that sum);
  dq:     |error| <= 2e-2 |row| + 1e-2 |tensor|.  A row of dq whose rotated
          keys cancel (dP close to D for every key it sees) is a small
          difference of large bf16-rounded terms, so its error follows the
          terms, i.e. the tensor's scale (measured: up to 4.5e-3 of it), not
          its own magnitude.
dsink is an fp32 sum over tokens of exp(sink - lse) D: 1e-2 relative.
"""
import numpy as np
import pytest
import torch

from sliding_window_sink_bias_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL = 2e-2


def _run(oracle_mod, lens, hq, hkv, window, base, seed, **kw):
    import sliding_window_sink_bias_b300 as sa
    inp = synth.prefill_inputs(lens, hq, hkv, window=window, rope_base=base, seed=seed,
                               device=DEV)
    g = torch.Generator(device="cpu").manual_seed(1000 + seed)
    dout = torch.randn(inp.total, hq, 128, generator=g).to(torch.bfloat16).to(DEV)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens,
                          max_seqlen=inp.max_seqlen, window=window, rope_base=base, **kw)
    dq, dk, dv, ds = sa.prefill_backward(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, out, lse,
                                         dout, max_seqlen=inp.max_seqlen, window=window,
                                         rope_base=base, **kw)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    okw = {}
    if kw.get("rope_style"):
        okw["rope_style"] = kw["rope_style"]
    if kw.get("scale") is not None:
        okw["scale"] = kw["scale"]
    rq, rk, rv, rs = oracle_mod.prefill_backward(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(),
                                                 inp.sink.cpu(), inp.cu_seqlens.cpu(),
                                                 dout.cpu(), window=window, rope_base=base,
                                                 **okw)
    return (dq, dk, dv, ds), (rq, rk, rv, rs)


def _check(got, ref, what):
    names = ("dq", "dk", "dv")
    for name, g, r in zip(names, got[:3], ref[:3]):
        g = g.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        tmax = max(np.max(np.abs(r)), 1e-30)
        err_row = np.max(np.abs(g - r), axis=-1)
        row = np.max(np.abs(r), axis=-1)
        bound = REL * row + (1e-2 * tmax if name == "dq" else REL * 0.05 * tmax)
        worst = np.unravel_index(np.argmax(err_row - bound), err_row.shape)
        assert np.all(err_row <= bound), (
            f"{what} {name}: row {worst} err {err_row[worst]:.3e} > bound {bound[worst]:.3e} "
            f"(row scale {row[worst]:.3e}, tensor scale {tmax:.3e})")
    gs = got[3].cpu().numpy().astype(np.float64)
    rs = ref[3]
    err = np.max(np.abs(gs - rs))
    assert err <= 1e-2 * max(np.max(np.abs(rs)), 1e-6), f"{what} dsink: {err:.3e}"


@pytest.mark.parametrize("lens,window,hkv,base", [
    ([300, 77], 128, 8, 1e4),          # SWA shape (G = 8)
    ([257, 130, 5], 0, 4, 5e6),        # GA shape (G = 16)
    ([200], 16, 8, 1e4),               # a narrow window
    ([129, 64, 1], 0, 8, 1e4),         # global with G = 8
])
def test_backward_small(oracle_mod, lens, window, hkv, base):
    got, ref = _run(oracle_mod, lens, 64, hkv, window, base, seed=sum(lens) + window)
    _check(got, ref, f"lens={lens} W={window} Hkv={hkv}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (16, 4), (64, 1)])
def test_backward_group_sizes(oracle_mod, hq, hkv):
    got, ref = _run(oracle_mod, [150, 33], hq, hkv, 0, 1e4, seed=hq + hkv)
    _check(got, ref, f"G={hq // hkv}")


def test_backward_rope_style_and_scale(oracle_mod):
    got, ref = _run(oracle_mod, [190], 64, 8, 100, 1e4, seed=5, rope_style=1, scale=0.05)
    _check(got, ref, "half-split rope, scale 0.05")


def test_backward_deterministic():
    import sliding_window_sink_bias_b300 as sa
    inp = synth.prefill_inputs([400, 99], 64, 8, window=128, rope_base=1e4, seed=3, device=DEV)
    dout = torch.randn(inp.total, 64, 128, device=DEV).to(torch.bfloat16)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, max_seqlen=400,
                          window=128, rope_base=1e4)
    a = sa.prefill_backward(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, out, lse, dout,
                            max_seqlen=400, window=128, rope_base=1e4)
    b = sa.prefill_backward(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, out, lse, dout,
                            max_seqlen=400, window=128, rope_base=1e4)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
