"""GPU parity: sinkattn_decode_fp8 (E4M3 KV cache, one scale per KV head) against
the oracle run on the exactly dequantised cache (e4m3 * scale in fp64).  The
kernel converts the cache to fp16 exactly and rounds q (bf16) to fp16, which is
exact in the normal range, so the bf16 decode's tolerances apply unchanged."""
import pytest
import torch

from helpers import assert_parity
from sliding_window_sink_bias_b300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _quantize(cache, seed):
    """-> (E4M3 tensor, fp32 scale per KV head): the scale maps each head's
    largest magnitude to 224 (half the E4M3 range), times a per-head factor."""
    hkv = cache.shape[2]
    amax = cache.float().abs().amax(dim=(0, 1, 3)).clamp_min(1e-6)
    g = torch.Generator().manual_seed(seed)
    scale = (amax / 224.0) * (0.5 + torch.rand(hkv, generator=g))
    q8 = (cache.float() / scale[None, None, :, None]).to(torch.float8_e4m3fn)
    return q8, scale.to(torch.float32)


def _dequant(q8, scale):
    return q8.to(torch.float64) * scale.to(torch.float64)[None, None, :, None]


def _run(oracle_mod, seqlens, t, s_cap, hkv, window, base, seed, nan_past_end=False, **kw):
    import sliding_window_sink_bias_b300 as sa
    inp = synth.decode_inputs(seqlens, t, s_cap, 64, hkv, window=window, rope_base=base, seed=seed,
                              device="cpu")
    k8, ks = _quantize(inp.kcache, seed)
    v8, vs = _quantize(inp.vcache, seed + 1)
    if nan_past_end:
        for b, L in enumerate(seqlens):
            k8.view(torch.uint8)[b, L:] = 0x7F  # E4M3 NaN
            v8.view(torch.uint8)[b, L:] = 0x7F
    out, lse = sa.decode_fp8(inp.q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV),
                             inp.seqlens.to(DEV), inp.sink.to(DEV), max_seqlen=max(seqlens),
                             window=window, rope_base=base, **kw)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    okw = {"rope_style": kw["rope_style"]} if kw.get("rope_style") else {}
    ro, rl = oracle_mod.decode(inp.q.to(torch.float64), _dequant(k8, ks), _dequant(v8, vs),
                               inp.seqlens, inp.sink, window=window, rope_base=base, **okw)
    return out, lse, ro, rl


@pytest.mark.parametrize("window,hkv,base", [(0, 4, 5e6), (128, 8, 1e4)])
def test_fp8_mtp_verify(oracle_mod, window, hkv, base):
    o, l, ro, rl = _run(oracle_mod, [4, 5, 1000, 2999, 3000, 131, 132], 4, 3000, hkv, window, base,
                        seed=21)
    assert_parity(o, l, ro, rl, f"fp8 decode W={window}")


@pytest.mark.parametrize("window,hkv", [(0, 4), (128, 8)])
def test_fp8_block_edges_and_nan_tail(oracle_mod, window, hkv):
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 191, 192, 193, 255, 256, 257]
    o, l, ro, rl = _run(oracle_mod, lens, 4, 300, hkv, window, 1e4, seed=22, nan_past_end=True)
    assert_parity(o, l, ro, rl, f"fp8 edges W={window}")


@pytest.mark.parametrize("t,hkv", [(5, 4), (8, 4), (8, 8), (16, 8)])
def test_fp8_tile_sizes(oracle_mod, t, hkv):
    """Query tiles of T * G = 80 and 128 rows as well as 64: more MTP tokens
    than the verify step's four, over the same caches."""
    o, l, ro, rl = _run(oracle_mod, [1, 64, 700, 1500, 1501], t, 1501, hkv, 0, 5e6, seed=26)
    assert_parity(o, l, ro, rl, f"fp8 T={t} G={64 // hkv}")


def test_fp8_half_split_rope_and_tokens(oracle_mod):
    o, l, ro, rl = _run(oracle_mod, [333, 1000, 2], 2, 1000, 4, 0, 5e6, seed=23, rope_style=1)
    assert_parity(o, l, ro, rl, "fp8 half-split")


def test_fp8_long_cache_many_splits(oracle_mod):
    o, l, ro, rl = _run(oracle_mod, [20000, 9000], 4, 20000, 4, 0, 5e6, seed=24)
    assert_parity(o, l, ro, rl, "fp8 long cache")


@pytest.mark.parametrize("window,hkv,base", [(0, 4, 5e6), (128, 8, 1e4)])
def test_fp8_rotated_cache(oracle_mod, window, hkv, base):
    """An E4M3 cache of keys already rotated at their positions (rotated in fp64
    by the oracle, then quantised): the kernel converts them without rotating;
    the oracle decodes the exactly dequantised cache with k_rotated."""
    import numpy as np

    import sliding_window_sink_bias_b300 as sa
    seqlens = [4, 64, 65, 1000, 2999, 3000, 131]
    inp = synth.decode_inputs(seqlens, 4, 3000, 64, hkv, window=window, rope_base=base, seed=25,
                              device="cpu")
    pos = np.arange(3000, dtype=np.float64)[None, :, None]
    krot = torch.from_numpy(oracle_mod.rope_rows(inp.kcache.to(torch.float64).numpy(), pos,
                                                 base=base))
    k8, ks = _quantize(krot, 25)
    v8, vs = _quantize(inp.vcache, 26)
    out, lse = sa.decode_fp8(inp.q.to(DEV), k8.to(DEV), v8.to(DEV), ks.to(DEV), vs.to(DEV),
                             inp.seqlens.to(DEV), inp.sink.to(DEV), max_seqlen=max(seqlens),
                             window=window, rope_base=base, k_rotated=True)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.decode(inp.q.to(torch.float64), _dequant(k8, ks), _dequant(v8, vs),
                               inp.seqlens, inp.sink, window=window, rope_base=base,
                               k_rotated=True)
    assert_parity(out, lse, ro, rl, f"fp8 rotated cache W={window}")
