"""GPU parity at the edges of the rotated dims' storage range.

The kernels re-store the rotated dims 0..63 of q and k as fp16 (11 significant
bits, finite up to 65504; below 2^-14 = 6.1e-5 values are fp16 subnormals with
an absolute step of 2^-24), and the FP8-cache decode rounds all of q to fp16.
A rotation keeps each pair's length, so a rotated value never exceeds
sqrt(x^2 + y^2) of its input pair.  These cases put one operand's dims 0..63 at
large magnitudes (|N(0,1)| clipped at 1.5, times 30000 or 10000: up to 45056,
pair lengths up to 63718, still finite in fp16) and the other's at small ones
(times 1/30000, all below 5e-5 and so all fp16 subnormals; or times 1e-4, about
half of them subnormals), both ways round, and check the results against the
fp64 oracle with the usual gates.  The two magnitudes are paired so that each
product q_d k_d keeps the size it has for N(0,1) inputs: the logits, and with
them the peakedness of the attention and the bf16 rounding of the output, stay
those of the model's workload, and the test measures the fp16 storage alone.
"""
import numpy as np
import pytest
import torch

from helpers import assert_parity
from sliding_window_sink_bias_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
# (large, small) magnitude pairs with large * small = 1
PAIRS = [(30000.0, 1.0 / 30000.0), (10000.0, 1e-4)]
MAGS = [(a, b) for a, b in PAIRS] + [(b, a) for a, b in PAIRS]
MAG_IDS = ["q3e4_k3e-5", "q1e4_k1e-4", "q3e-5_k3e4", "q1e-4_k1e4"]


def _edge(x, mag):
    """Dims 0..63 of x scaled to the given magnitude (|N(0,1)| clipped at 1.5), bf16."""
    y = x.float().clone()
    y[..., :64] = y[..., :64].clamp(-1.5, 1.5) * mag
    return y.to(torch.bfloat16)


@pytest.mark.parametrize("q_mag,k_mag", MAGS, ids=MAG_IDS)
@pytest.mark.parametrize("hq,hkv,window,base", [(64, 8, 128, 1e4), (64, 4, 0, 5e6),
                                                (64, 16, 64, 1e4), (8, 4, 32, 1e4)],
                         ids=["band", "causal", "causal_window", "generic"])
def test_prefill_rotated_dims_at_fp16_edges(oracle_mod, q_mag, k_mag, hq, hkv, window, base):
    import sliding_window_sink_bias_b300 as sa
    lens = [300, 77]
    inp = synth.prefill_inputs(lens, hq, hkv, window=window, rope_base=base, seed=40, device="cpu")
    q, k = _edge(inp.q, q_mag), _edge(inp.k, k_mag)
    out, lse = sa.prefill(q.to(DEV), k.to(DEV), inp.v.to(DEV), inp.sink.to(DEV),
                          inp.cu_seqlens.to(DEV), max_seqlen=max(lens), window=window,
                          rope_base=base)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.prefill(q, k, inp.v, inp.sink, inp.cu_seqlens, window=window,
                                rope_base=base)
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert_parity(out, lse, ro, rl, f"prefill edges q={q_mag} k={k_mag} W={window}")


@pytest.mark.parametrize("q_mag,k_mag", MAGS, ids=MAG_IDS)
@pytest.mark.parametrize("hkv,window,base", [(4, 0, 5e6), (8, 128, 1e4)], ids=["ga", "swa"])
def test_decode_rotated_dims_at_fp16_edges(oracle_mod, q_mag, k_mag, hkv, window, base):
    import sliding_window_sink_bias_b300 as sa
    lens = [1000, 131, 4]
    inp = synth.decode_inputs(lens, 4, 1000, 64, hkv, window=window, rope_base=base, seed=41,
                              device="cpu")
    q, kc = _edge(inp.q, q_mag), _edge(inp.kcache, k_mag)
    out, lse = sa.decode(q.to(DEV), kc.to(DEV), inp.vcache.to(DEV), inp.seqlens.to(DEV),
                         inp.sink.to(DEV), max_seqlen=max(lens), window=window, rope_base=base)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.decode(q, kc, inp.vcache, inp.seqlens, inp.sink, window=window,
                               rope_base=base)
    assert_parity(out, lse, ro, rl, f"decode edges q={q_mag} k={k_mag} W={window}")


def test_fp8_decode_q_at_fp16_edges(oracle_mod):
    """FP8 cache: all of q is rounded to fp16, so q's dims 0..63 at up to 45056
    and its dims 64..191 at about 1e-4 (many fp16 subnormals) are its edges; the
    keys carry the inverse magnitudes (dims 0..63 about 3e-5, dims 64..191 up
    to 15000) and the cache holds E4M3 values with one scale per KV head."""
    import sliding_window_sink_bias_b300 as sa
    lens = [700, 64, 5]
    inp = synth.decode_inputs(lens, 4, 700, 64, 4, window=0, rope_base=5e6, seed=42, device="cpu")
    q = inp.q.float().clone()
    q[..., :64] = q[..., :64].clamp(-1.5, 1.5) * 30000.0
    q[..., 64:] = q[..., 64:] * 1e-4
    q = q.to(torch.bfloat16)
    kc = inp.kcache.float().clone()
    kc[..., :64] = kc[..., :64] / 30000.0
    kc[..., 64:] = kc[..., 64:].clamp(-1.5, 1.5) * 1e4
    ks = (kc.abs().amax(dim=(0, 1, 3)) / 224.0).float()
    k8 = (kc / ks[None, None, :, None]).to(torch.float8_e4m3fn)
    vs = (inp.vcache.float().abs().amax(dim=(0, 1, 3)) / 224.0).float()
    v8 = (inp.vcache.float() / vs[None, None, :, None]).to(torch.float8_e4m3fn)
    out, lse = sa.decode_fp8(q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV),
                             inp.seqlens.to(DEV), inp.sink.to(DEV), max_seqlen=max(lens),
                             window=0, rope_base=5e6)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    kd = k8.to(torch.float64) * ks.double()[None, None, :, None]
    vd = v8.to(torch.float64) * vs.double()[None, None, :, None]
    ro, rl = oracle_mod.decode(q.to(torch.float64), kd, vd, inp.seqlens, inp.sink, window=0,
                               rope_base=5e6)
    assert_parity(out, lse, ro, rl, "fp8 decode q edges")
