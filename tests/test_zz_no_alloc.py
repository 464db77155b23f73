"""sinkattn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers may not allocate device memory at the point where they decode: a
serving loop inside a fixed memory pool that must not grow, a real-time path
that forbids cudaMalloc (and the synchronisation it implies), or a host program
that owns no device allocator.  The entry point keeps its split-KV partials in a
fixed buffer inside the library's device image instead of a caller-supplied
workspace.  These checks call it through the C ABI and compare it with
sinkattn_decode (which takes a workspace) on the same inputs.  Both run the same
deterministic kernels, so the results must be identical bit for bit.  Each case
makes two calls in a row on the same shapes with different inputs: the second
call runs on the buffer the first one left behind, and is also checked against
the fp64 oracle within the parity tolerances.  The file is named to run last, so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from helpers import assert_parity
from sliding_window_sink_bias_b300 import synth

DEV = "cuda"


def test_noalloc_rejects_sizes_beyond_its_buffer():
    """Host-side check, no GPU needed: a problem whose partials exceed the fixed
    buffer is refused with SINKATTN_EWORKSPACE before anything is launched, and
    arguments the workspace decode rejects get its status."""
    import sliding_window_sink_bias_b300 as sa
    L = sa.lib()
    # 8 query tokens x 16 heads = 128 partial rows per unit: more than the buffer holds
    need = sa.decode_workspace_size(64, 8, 64, 4, 262144, 0)
    assert need > sa.NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    st = L.sinkattn_decode_noalloc(P(256), P(256), P(256), P(256), P(256), 0, 5e6, 64, 8, 262144,
                                   262144, 64, 4, P(256), P(256), None)
    assert st == sa.EWORKSPACE
    # invalid sizes (T = 0; a group of 3 heads) and an empty batch: no CUDA call at all
    assert L.sinkattn_decode_noalloc(P(256), P(256), P(256), P(256), P(256), 0, 5e6, 4, 0, 1024,
                                     1024, 64, 4, P(256), P(256), None) == sa.EINVAL
    assert L.sinkattn_decode_noalloc(P(256), P(256), P(256), P(256), P(256), 0, 5e6, 4, 4, 1024,
                                     1024, 24, 8, P(256), P(256), None) == sa.EUNSUPPORTED
    assert L.sinkattn_decode_noalloc(None, None, None, None, None, 0, 5e6, 0, 4, 1024, 1024, 64,
                                     4, None, None, None) == sa.OK


CASES = [
    # GA layer: 4 KV heads, global causal, long enough for several splits
    dict(seqlens=[3000, 4, 1777, 2500], s_cap=3000, hkv=4, window=0, base=5e6, seed=11),
    # SWA layer: 8 KV heads, window 128
    dict(seqlens=[700, 129, 2000], s_cap=2000, hkv=8, window=128, base=1e4, seed=12),
]


@pytest.mark.gpu
@pytest.mark.parametrize("c", CASES, ids=["ga", "swa"])
def test_noalloc_decode_equals_workspace_decode_twice(c, oracle_mod):
    import sliding_window_sink_bias_b300 as sa
    need = sa.decode_workspace_size(len(c["seqlens"]), 4, 64, c["hkv"], max(c["seqlens"]),
                                    c["window"])
    assert 0 < need <= sa.NOALLOC_SCRATCH_BYTES
    kw = dict(max_seqlen=max(c["seqlens"]), window=c["window"], rope_base=c["base"])
    for call, seed in enumerate((c["seed"], c["seed"] + 100)):
        inp = synth.decode_inputs(c["seqlens"], 4, c["s_cap"], 64, c["hkv"], window=c["window"],
                                  rope_base=c["base"], seed=seed, device=DEV)
        args = (inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink)
        ref_out, ref_lse = sa.decode(*args, **kw)
        out, lse = sa.decode_noalloc(*args, **kw)
        torch.cuda.synchronize()
        assert sa.device_status()[0] == sa.OK
        assert torch.equal(out, ref_out), f"call {call}: out differs from sinkattn_decode"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from sinkattn_decode"
        if call == 1:
            ro, rl = oracle_mod.decode(inp.q.cpu(), inp.kcache.cpu(), inp.vcache.cpu(),
                                       inp.seqlens.cpu(), inp.sink.cpu(), window=c["window"],
                                       rope_base=c["base"])
            assert_parity(out, lse, ro, rl, f"noalloc second call {c['seqlens']}")
