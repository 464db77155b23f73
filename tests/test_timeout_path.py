"""The timeout path of the kernels' bounded waits, on the GPU, without a fault.

Every mbarrier wait in the kernels is bounded: a wait that runs out sets the
CTA's abort flag and SINKATTN_ETIMEOUT (with the wait site) in the device status
word; the other roles of the CTA see the flag and leave their loops, the copy
and MMA threads wait (boundedly) for what they issued, TMEM is freed and the
kernel returns.  To run that path, the test loads the test build of the library
(libsinkattn_test.so: the same sources compiled with SINKATTN_TEST_HOOKS; the
product library has no such hook), which can make the SWA prefill kernel's MMA
thread first wait, for 20 ms at most, on a barrier nothing can complete yet.
The launch must end by itself, the status must read ETIMEOUT at that site, and
the next launch, with the stall off, must give SINKATTN_OK and results equal
to the oracle's."""
import ctypes
import os
import time

import pytest
import torch

from helpers import assert_parity
from sliding_window_sink_bias_b300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TEST_LIB = os.path.join(ROOT, "sliding_window_sink_bias_b300", "libsinkattn_test.so")
STALL_SITE = 0x7E
DEV = "cuda"


def test_product_library_has_no_test_hook():
    from sliding_window_sink_bias_b300 import build
    build.build()
    assert not hasattr(ctypes.CDLL(build.LIB), "sinkattn_test_set_stall_ns")
    assert hasattr(ctypes.CDLL(TEST_LIB), "sinkattn_test_set_stall_ns")


@pytest.mark.gpu
def test_timed_out_wait_aborts_cleanly_and_next_call_is_correct(oracle_mod, monkeypatch):
    import sliding_window_sink_bias_b300 as sa
    # run the binding against the test build for this test only
    monkeypatch.setattr(sa, "LIB_PATH", TEST_LIB)
    monkeypatch.setattr(sa, "_lib", None)
    L = sa.lib()
    L.sinkattn_test_set_stall_ns.argtypes = [ctypes.c_uint64]
    L.sinkattn_test_set_stall_ns.restype = ctypes.c_int
    lens = [200, 57]
    inp = synth.prefill_inputs(lens, 64, 8, window=128, rope_base=1e4, seed=50, device="cpu")
    args = (inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.sink.to(DEV), inp.cu_seqlens.to(DEV))
    kw = dict(max_seqlen=max(lens), window=128, rope_base=1e4)
    assert sa.device_status()[0] == sa.OK
    try:
        assert L.sinkattn_test_set_stall_ns(20_000_000) == 0
        t0 = time.perf_counter()
        sa.prefill(*args, **kw)
        st, word = sa.device_status()  # synchronises: the launch ended by itself
        dt = time.perf_counter() - t0
    finally:
        assert L.sinkattn_test_set_stall_ns(0) == 0
    assert st == sa.ETIMEOUT, (st, hex(word))
    assert word & 1 and ((word >> 8) & 0xFF) == STALL_SITE, hex(word)
    assert dt < 5.0
    # the status word was cleared by the read; the context is usable
    out, lse = sa.prefill(*args, **kw)
    torch.cuda.synchronize()
    assert sa.device_status()[0] == sa.OK
    ro, rl = oracle_mod.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, window=128,
                                rope_base=1e4)
    assert_parity(out, lse, ro, rl, "prefill after a timed-out launch")
