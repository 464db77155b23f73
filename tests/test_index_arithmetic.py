"""CPU checks of index arithmetic in the backward and causal kernels, restated
here from the kernel sources and compared with the plain rule each implements
(no GPU).  A wrong offset in these formulas would skip or double-count a key,
an angle or an output row without failing at run time.

- bwd_dq_kernel, rows: the visible columns of a 32-key half block as one
  unsigned range compare, and the warp-wide shortcut taken when every column is
  visible.
- bwd_dkdv_kernel, rows: the query columns of a key as one range, and the
  same shortcut.
- bwd_dq_kernel, epilogue: the lanes of one token share its 32 RoPE angles
  through a shared-memory slot per (warp, token).
- sinkattn_causal_kernel, epilogue: the output row written by each of the four
  stores of a lane quad, for any number G of query heads per KV head.
"""
import random

import pytest


def _visible(key, ti, window):
    """Key `key` is visible to the query at position ti (eq. (2) with the
    sliding window of §2.1: i - W < j <= i; W = 0 is global)."""
    lo = ti - window + 1 if window > 0 else 0
    return max(0, lo) <= key <= ti


def _dq_columns(ti, rvalid, window, kb):
    """The dq rows' test, as in backward_kernel.cuh: column c of the half block
    starting at key kb is visible iff (unsigned)(c - c_lo) <= span."""
    c_lo = (ti - window + 1 if window > 0 else 0) - kb
    span = (ti - kb - c_lo) & 0xFFFFFFFF if rvalid else 0
    vis = [((c - c_lo) & 0xFFFFFFFF) <= span and rvalid for c in range(32)]
    whole = rvalid and c_lo <= 0 and ti - kb >= 31
    return vis, whole


@pytest.mark.parametrize("window", [0, 1, 5, 64, 127, 128, 300])
def test_dq_column_range_matches_the_window(window):
    rng = random.Random(window)
    for _ in range(4000):
        ti = rng.randrange(0, 2000)
        kb = rng.randrange(0, 2000) // 32 * 32
        rvalid = rng.random() < 0.9
        vis, whole = _dq_columns(ti, rvalid, window, kb)
        want = [rvalid and _visible(kb + c, ti, window) for c in range(32)]
        assert vis == want, (ti, kb, window, rvalid)
        # the shortcut is taken exactly when every column is visible
        assert whole == all(want), (ti, kb, window, rvalid)


def _dkdv_columns(kj, kvalid, i0, L, window, G, half):
    """The dk/dv rows' test, as in backward_kernel.cuh: key kj, a sub-tile of
    64 packed rows starting at query token i0 (column c is token i0 + c // G),
    this thread's columns 32 half .. 32 half + 31 as c - 32 half."""
    d0 = kj - i0
    c_lo = (d0 * G if d0 > 0 else 0) - 32 * half
    c_hi = min(L - i0, 64) * G
    if window > 0:
        c_hi = min(c_hi, max(0, min(d0 + window, 64)) * G)
    c_hi = min(c_hi, 64) - 32 * half
    span = c_hi - c_lo if (kvalid and c_hi > c_lo) else 0
    return [((c - c_lo) & 0xFFFFFFFF) < span for c in range(32)], c_lo, span


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("window", [0, 1, 7, 128, 300])
def test_dkdv_column_range_matches_the_window(G, window):
    rng = random.Random(G * 1000 + window)
    TS = 64 // G
    for _ in range(1500):
        L = rng.randrange(1, 1500)
        kj = rng.randrange(0, L + 130)  # keys past the end too
        kvalid = kj < L
        i0 = rng.randrange(0, L) // TS * TS
        for half in (0, 1):
            vis, c_lo, span = _dkdv_columns(kj, kvalid, i0, L, window, G, half)
            for c in range(32):
                col = c + 32 * half
                i = i0 + col // G
                want = kvalid and i < L and _visible(kj, i, window)
                assert vis[c] == want, (G, window, L, kj, i0, half, c)
            whole = kvalid and c_lo <= 0 and span > 31 - c_lo
            assert whole == all(vis)


def test_dkdv_whole_shortcut():
    """bwd_dkdv_kernel, rows: column c is visible iff (unsigned)(c - c_lo) <
    span (span 0 for a key past the sequence); the shortcut is taken iff the
    key is valid, c_lo <= 0 and span > 31 - c_lo, which must mean all 32."""
    rng = random.Random(5)
    for _ in range(20000):
        c_lo = rng.randrange(-200, 200)
        kvalid = rng.random() < 0.9
        span = rng.randrange(0, 260) if kvalid else 0
        vis = [((c - c_lo) & 0xFFFFFFFF) < span for c in range(32)]
        whole = kvalid and c_lo <= 0 and span > 31 - c_lo
        assert whole == all(vis), (c_lo, span, kvalid)


@pytest.mark.parametrize("G", [8, 16, 32, 64])
def test_dq_epilogue_angle_slots(G):
    """Rows r = 32 w + lane of warps w = 0..3 hold token r // G of the tile.  A
    lane writes the angles of pairs lane % Gw, lane % Gw + Gw, ... into slot
    4 w + lane // Gw (Gw = min(G, 32)) and reads all 32 back from its slot."""
    Gw = min(G, 32)
    for w in range(4):
        written = {}
        for lane in range(32):
            row = 32 * w + lane
            slot = 4 * w + lane // Gw
            assert 0 <= slot < 16  # 4 warps x 4 tokens x 32 pairs of (cos, sin)
            for p in range(lane % Gw, 32, Gw):
                key = (slot, p)
                # one writer per (slot, pair), and the writer's token is the slot's
                assert key not in written
                written[key] = row // G
        for lane in range(32):
            slot = 4 * w + lane // Gw
            token = (32 * w + lane) // G
            # every pair of the reader's slot is written, by a lane of its own token
            assert all(written[(slot, p)] == token for p in range(32))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64, 128])
def test_causal_quad_store_rows(G):
    """Lane q of the quad holding rows 4k..4k+3 makes four stores; store pq
    writes sector q of tile row rq = 4k + pq at out row
    (s0 + t0 + X T + rq // G) Hq + kvh G + rq % G, skipped past the sequence.
    Over the tile's 128 rows every row of a token inside the sequence gets each
    of its four sectors exactly once and no other row is written; for G >= 4
    the quad's rows are consecutive out rows (four heads of one token)."""
    T = 128 // G
    Hq = max(64, G)
    rng = random.Random(G)
    for _ in range(100):
        kvh = rng.randrange(Hq // G)
        s0 = rng.randrange(0, 5000)
        t0 = rng.randrange(0, 4096) // (2 * T) * (2 * T)
        L = t0 + rng.randrange(1, 2 * T + 1)
        X = rng.randrange(2)
        writes = []
        for row in range(128):
            q = row & 3
            orow = (s0 + t0 + X * T + row // G) * Hq + kvh * G + row % G
            for pq in range(4):
                rq = (row & ~3) + pq
                pos_q = t0 + X * T + rq // G
                if pos_q >= L:
                    continue
                orq = (s0 + pos_q) * Hq + kvh * G + rq % G
                if G >= 4:
                    assert orq == orow - q + pq
                writes.append((orq, q))
        # the tile's rows: tokens t0 + X T + t (t < T) inside the sequence, heads g < G
        want = sorted(((s0 + t0 + X * T + t) * Hq + kvh * G + g, sec)
                      for t in range(T) for g in range(G) for sec in range(4)
                      if t0 + X * T + t < L)
        assert sorted(writes) == want
