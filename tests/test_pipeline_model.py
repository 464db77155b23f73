"""The barrier protocols of the prefill, decode and backward kernels, checked
on a CPU model (tests/pipeline_model.py) over many random interleavings: no
deadlock, no parity wait whose barrier is two phases past or two phases short
of the awaited one, and no MMA or thread that reads a shared-memory stage or
TMEM region before the data it expects has landed or after the next write
replaced it.  The model transcribes the roles of sinkattn_band_kernel
(band_kernel.cuh), sinkattn_causal_kernel (causal_kernel.cuh),
sinkattn_fwd_kernel (attn_kernel.cuh, both instances),
sinkattn_decode_kernel (decode_kernel.cuh), bwd_dq_kernel and bwd_dkdv_kernel
(backward_kernel.cuh); a wait left out of it must be caught, which the
*_missing_wait_* tests check.  Run with random timeouts, every kernel's abort
path must leave nothing in flight (the *_abort_* and *_missing_drain_* tests)."""
import random

import pytest

from pipeline_model import (ModelError, band_roles, causal_roles, decode_roles, dkdv_roles, dq_roles,
                            general_roles, run)

SIZES = [[1], [2], [3], [1, 1, 1], [1, 2, 1, 3], [3, 3, 3], [5, 1, 4], [2, 7], [1] * 6]


def _random_sizes(rng):
    return [rng.choice([1, 1, 2, 3, 4, 6]) for _ in range(rng.randint(1, 5))]


@pytest.mark.parametrize("sizes", SIZES)
def test_dq_pipeline(sizes):
    for seed in range(60):
        run(dq_roles, sizes, seed)


@pytest.mark.parametrize("sizes", SIZES)
def test_dkdv_pipeline(sizes):
    for seed in range(60):
        run(dkdv_roles, sizes, seed)


def test_random_item_lists():
    rng = random.Random(7)
    for seed in range(200):
        sizes = _random_sizes(rng)
        run(dq_roles, sizes, seed)
        run(dkdv_roles, sizes, seed)


def _caught(make_roles, skip, sizes=(3, 2, 4)):
    for seed in range(400):
        try:
            run(make_roles, list(sizes), seed, skip=skip)
        except ModelError:
            return True
    return False


@pytest.mark.parametrize("skip,sizes", [("producer_kve", (3, 2, 4)), ("rows_accf", (3, 2, 4)),
                                        ("issuer_dsr", (1, 2, 1, 3)),
                                        ("producer_qe", (1, 1, 2, 1))])
def test_dq_missing_wait_is_caught(skip, sizes):
    assert _caught(dq_roles, (skip,), sizes)


@pytest.mark.parametrize("skip", ["producer_kve", "producer_qse", "issuer_pr", "issuer_sr",
                                  "rows_lf", "rows_mm2"])
def test_dkdv_missing_wait_is_caught(skip):
    assert _caught(dkdv_roles, (skip,))


@pytest.mark.parametrize("f8", [False, True])
@pytest.mark.parametrize("sizes", [[1], [2], [5], [1, 1, 1], [3, 1, 4], [2, 6, 1, 2]])
def test_decode_pipeline(f8, sizes):
    for seed in range(60):
        run(lambda s, sk: decode_roles(s, f8, sk), sizes, seed)


@pytest.mark.parametrize("f8,skip", [(False, "producer_kvempty"), (True, "convert_kvempty"),
                                     (False, "softmax_pvdone"), (True, "softmax_pvdone")])
def test_decode_missing_wait_is_caught(f8, skip):
    assert _caught(lambda s, sk: decode_roles(s, f8, sk), (skip,), (5, 3, 6))


@pytest.mark.parametrize("f8", [False, True])
def test_decode_missing_qtfree_is_caught(f8):
    # with one-block units the K stages do not order a unit's QK^T before the
    # Q copy of the unit two later: only the buffer-free commit does
    assert _caught(lambda s, sk: decode_roles(s, f8, sk), ("convert_qtfree",), (1, 1, 1, 1, 1, 1))


@pytest.mark.parametrize("sizes", [[1], [2], [4], [1, 1, 1], [3, 1, 2], [2, 5, 1, 3]])
def test_causal_pipeline(sizes):
    for seed in range(60):
        run(causal_roles, sizes, seed)


@pytest.mark.parametrize("skip", ["producer_kempty", "vloader_vempty", "mma_pfull", "rope_kfull"])
def test_causal_missing_wait_is_caught(skip):
    assert _caught(causal_roles, (skip,), (3, 2, 4))


BAND_RANGES = [[(0, 1)], [(0, 12)], [(5, 3)], [(0, 20)], [(7, 4), (0, 3)],
               [(30, 2), (0, 12), (0, 1)], [(0, 1), (0, 1), (0, 2)]]


@pytest.mark.parametrize("lanes", BAND_RANGES)
def test_band_pipeline(lanes):
    for seed in range(60):
        run(band_roles, lanes, seed)


@pytest.mark.parametrize("R", [10, 11])
def test_band_pipeline_smaller_rings(R):
    # the kernel's ring is the 9-segment window plus the 3 segments the Q
    # double buffer lets the copy thread run ahead; smaller rings only wait more
    for lanes in BAND_RANGES:
        for seed in range(20):
            run(lambda s, sk: band_roles(s, sk, R=R), lanes, seed)


@pytest.mark.parametrize("skip,R", [("mma_oempty", 12), ("softmax_pair", 12),
                                    # with 12 slots the segment-empty wait never
                                    # blocks (see above); with 10 it must
                                    ("producer_segempty", 10)])
def test_band_missing_wait_is_caught(skip, R):
    assert _caught(lambda s, sk: band_roles(s, sk, R=R), (skip,), [(3, 14), (0, 4)])


# ------------------------------------------------ abort and drain (band kernel)
@pytest.mark.parametrize("lanes", [[(0, 1)], [(0, 5)], [(3, 14), (0, 4)], [(0, 1), (0, 1), (2, 3)]])
def test_band_abort_drains_everything(lanes):
    """A bounded wait runs out at a random moment: the CTA's abort flag is set
    and every later unsatisfied wait gives up.  No role may then wait forever,
    no read may see the wrong data, and when every role is done no copy may
    still be landing and no MMA still running (the kernel frees its shared
    memory and TMEM there)."""
    aborted = 0
    for seed in range(300):
        sim = run(band_roles, lanes, seed, aborts=True)
        aborted += sim.aborted
    assert aborted > 50  # most runs took the abort path somewhere


@pytest.mark.parametrize("skip", ["producer_drain", "mma_drain"])
def test_band_missing_drain_is_caught(skip):
    """Leaving out the copy thread's or the MMA thread's drain lets the CTA
    finish with work in flight: the model notices."""
    caught = False
    for seed in range(400):
        try:
            run(band_roles, [(3, 14), (0, 4)], seed, skip=(skip,), aborts=True)
        except ModelError:
            caught = True
            break
    assert caught


@pytest.mark.parametrize("lanes", [[(0, 1)], [(0, 5)], [(3, 14), (0, 4)]])
def test_band_stalled_mma_thread_drains(lanes):
    """The test build's stall: the MMA thread's first wait can only run out.
    The CTA must abort, every role must leave, and the copies already issued
    must land before the exit, whatever the interleaving."""
    for seed in range(200):
        sim = run(lambda s, sk: band_roles(s, sk, stall=True), lanes, seed, aborts=True)
        assert sim.aborted


# ------------------------------------------------ abort and drain (backward kernels)
@pytest.mark.parametrize("make_roles", [dq_roles, dkdv_roles], ids=["dq", "dkdv"])
@pytest.mark.parametrize("sizes", [[1], [3], [1, 2, 1, 3], [2, 7], [5, 1, 4]])
def test_backward_abort_drains_everything(make_roles, sizes):
    """The dq and dk/dv kernels with a bounded wait running out at a random
    moment: no role waits forever, no read sees the wrong data, and when every
    role is done no copy is landing and no MMA running."""
    aborted = 0
    for seed in range(300):
        sim = run(make_roles, sizes, seed, aborts=True)
        aborted += sim.aborted
    assert aborted > 50


@pytest.mark.parametrize("make_roles", [dq_roles, dkdv_roles], ids=["dq", "dkdv"])
@pytest.mark.parametrize("skip", ["producer_drain", "mma_drain"])
def test_backward_missing_drain_is_caught(make_roles, skip):
    caught = False
    for seed in range(400):
        try:
            run(make_roles, [3, 2, 4], seed, skip=(skip,), aborts=True)
        except ModelError:
            caught = True
            break
    assert caught


# ------------------------------------------------ abort and drain (causal and decode kernels)
_ABORT_ROLES = {
    "causal": causal_roles,
    "decode": lambda s, sk: decode_roles(s, False, sk),
    "decode_fp8": lambda s, sk: decode_roles(s, True, sk),
}


@pytest.mark.parametrize("name", sorted(_ABORT_ROLES))
@pytest.mark.parametrize("sizes", [[1], [3], [1, 2, 1, 3], [2, 7]])
def test_forward_abort_drains_everything(name, sizes):
    """The GA prefill and decode kernels with a bounded wait running out at a
    random moment: every role leaves, nothing is read wrong, and no copy or
    MMA is in flight when the last role is done."""
    aborted = 0
    for seed in range(300):
        sim = run(_ABORT_ROLES[name], sizes, seed, aborts=True)
        aborted += sim.aborted
    assert aborted > 50


@pytest.mark.parametrize("name", sorted(_ABORT_ROLES))
@pytest.mark.parametrize("skip", ["producer_drain", "mma_drain"])
def test_forward_missing_drain_is_caught(name, skip):
    caught = False
    for seed in range(400):
        try:
            run(_ABORT_ROLES[name], [3, 2, 4], seed, skip=(skip,), aborts=True)
        except ModelError:
            caught = True
            break
    assert caught


# ------------------------------------------------ the general prefill kernel
_GENERAL = {"one_kv_stage": dict(NQ=2, NKV=1), "two_kv_stages": dict(NQ=1, NKV=2)}


@pytest.mark.parametrize("variant", sorted(_GENERAL))
@pytest.mark.parametrize("sizes", SIZES)
def test_general_pipeline(variant, sizes):
    for seed in range(60):
        run(lambda s, sk: general_roles(s, sk, **_GENERAL[variant]), sizes, seed)


@pytest.mark.parametrize("variant,skip", [(v, k) for v in sorted(_GENERAL)
                                          for k in ("producer_kvempty", "rope_kvfull")]
                         + [("two_kv_stages", "softmax_pvdone")])
def test_general_missing_wait_is_caught(variant, skip):
    # (with one K/V stage PV(j-1) goes out before QK^T(j), so S_FULL(j) implies
    # PV_DONE(j-1) and the softmax's own wait for it cannot be caught missing;
    # the MMA thread's O_EMPTY wait is implied by P_FULL in both variants)
    assert _caught(lambda s, sk: general_roles(s, sk, **_GENERAL[variant]), (skip,))


@pytest.mark.parametrize("variant", sorted(_GENERAL))
def test_general_abort_drains_everything(variant):
    aborted = 0
    for seed in range(300):
        sim = run(lambda s, sk: general_roles(s, sk, **_GENERAL[variant]), [1, 2, 1, 3], seed,
                  aborts=True)
        aborted += sim.aborted
    assert aborted > 50
