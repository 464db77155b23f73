"""sinkattn_decode_noalloc: decode for callers that cannot allocate device memory.

The entry point keeps its split-KV partials in a fixed buffer inside the
library's device image instead of a caller-supplied workspace.  These checks
call it through the C ABI and compare it with sinkattn_decode (which takes a
workspace) on the same inputs, within the parity tolerances used everywhere
else, on two calls in a row (the second call reuses the buffer the first one
left behind).  The file is named to run last, so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from helpers import LSE_TOL, OUT_TOL, max_abs
from sliding_window_sink_bias_b300 import synth

DEV = "cuda"


def test_noalloc_rejects_sizes_beyond_its_buffer():
    """Host-side check, no GPU needed: a problem whose partials exceed the fixed
    buffer is refused with SINKATTN_EWORKSPACE before anything is launched."""
    import sliding_window_sink_bias_b300 as sa
    L = sa.lib()
    # 8 query tokens x 16 heads = 128 partial rows per unit: more than the buffer holds
    need = sa.decode_workspace_size(64, 8, 64, 4, 262144, 0)
    assert need > sa.NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    st = L.sinkattn_decode_noalloc(P(256), P(256), P(256), P(256), P(256), 0, 5e6, 64, 8, 262144,
                                   262144, 64, 4, P(256), P(256), None)
    assert st == sa.EWORKSPACE


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_twice():
    import sliding_window_sink_bias_b300 as sa
    cases = [
        # GA layer: 4 KV heads, global causal, long enough for several splits
        dict(seqlens=[3000, 4, 1777, 2500], s_cap=3000, hkv=4, window=0, base=5e6, seed=11),
        # SWA layer: 8 KV heads, window 128
        dict(seqlens=[700, 129, 2000], s_cap=2000, hkv=8, window=128, base=1e4, seed=12),
    ]
    for c in cases:
        need = sa.decode_workspace_size(len(c["seqlens"]), 4, 64, c["hkv"], max(c["seqlens"]),
                                        c["window"])
        assert 0 < need <= sa.NOALLOC_SCRATCH_BYTES
        inp = synth.decode_inputs(c["seqlens"], 4, c["s_cap"], 64, c["hkv"], window=c["window"],
                                  rope_base=c["base"], seed=c["seed"], device=DEV)
        args = (inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink)
        kw = dict(max_seqlen=max(c["seqlens"]), window=c["window"], rope_base=c["base"])
        ref_out, ref_lse = sa.decode(*args, **kw)
        out, lse = sa.decode_noalloc(*args, **kw)
        torch.cuda.synchronize()
        assert sa.device_status()[0] == sa.OK
        eo = max_abs(out.float().cpu().numpy(), ref_out.float().cpu().numpy())
        el = max_abs(lse.cpu().numpy(), ref_lse.cpu().numpy())
        assert eo <= OUT_TOL and el <= LSE_TOL, f"{c}: out err {eo:.3e}, lse err {el:.3e}"
