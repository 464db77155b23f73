"""Pins for the oracle: checks against what the pages and the mathematics fix.

Each test here compares the oracle with something other than itself: a value
worked by hand from eqs. (2)-(3) of §2.2 of the MiMo-V2-Flash Technical Report
(tests/golden), a closed form, an invariant, a special case that reduces to a
library routine (torch's scaled_dot_product_attention / softmax in fp64), or a
brute-force enumeration written from the page's unshifted form of the sink
softmax (the blog post's "MiMo Softmax": exp(q.k) / (exp(sink) + sum exp(q.k))).
RoPE is pinned against a complex-number formulation (RoFormer), not against the
oracle's real-pair rotation.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_2h4t.txt")


# ---------------------------------------------------------------- helpers
def rope_complex(x: np.ndarray, pos: np.ndarray, base: float, drot: int, style: int):
    """RoPE via complex multiplication: pair t of x, viewed as a complex number,
    is multiplied by exp(i * pos * base^(-2t/drot)).  x [n, ..., d], pos [n]."""
    y = np.array(x, dtype=np.float64, copy=True)
    if drot == 0:
        return y
    half = drot // 2
    theta = base ** (-2.0 * np.arange(half, dtype=np.float64) / drot)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta[None, :]
    rot = np.exp(1j * ang).reshape((x.shape[0],) + (1,) * (x.ndim - 2) + (half,))
    if style == 0:
        z = (y[..., 0:drot:2] + 1j * y[..., 1:drot:2]) * rot
        y[..., 0:drot:2], y[..., 1:drot:2] = z.real, z.imag
    else:
        z = (y[..., :half] + 1j * y[..., half:drot]) * rot
        y[..., :half], y[..., half:drot] = z.real, z.imag
    return y


def bf16_tensor(shape, gen):
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def to64(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------- (i) golden
def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            case, head, row, out, else_, sw = line.split()
            rows.append((case, int(head), int(row), Fraction(out), int(else_), Fraction(sw)))
    return rows


def _hand_inputs():
    L = 4
    q = np.ones((L, 2, 1))
    k = np.array([j * math.log(2.0) for j in range(L)]).reshape(L, 1, 1)
    v = np.arange(L, dtype=np.float64).reshape(L, 1, 1)
    sink = np.array([0.0, -np.inf], dtype=np.float32)
    cu = np.array([0, L], dtype=np.int32)
    return q, k, v, sink, cu


def test_hand_worked_example(oracle_mod):
    q, k, v, sink, cu = _hand_inputs()
    got = {}
    for case, window in (("global", 0), ("window2", 2)):
        out, lse = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=0.0,
                                      scale=1.0, drot=0)
        got[case] = (out, lse)
    rows = _golden_rows()
    assert len(rows) == 12
    for case, head, row, o_exp, else_exp, sw_exp in rows:
        out, lse = got[case]
        assert abs(out[row, head, 0] - float(o_exp)) < 1e-12, (case, head, row)
        assert abs(lse[row, head] - math.log(else_exp)) < 1e-12, (case, head, row)
        sw = math.exp(float(sink[head]) - lse[row, head])
        assert abs(sw - float(sw_exp)) < 1e-12, (case, head, row)


# ------------------------------------------- (ii) sink -> -inf is plain SDPA
def _sdpa_reference(q, k, v, cu, window, base, drot, style, scale):
    """torch scaled_dot_product_attention (fp64) per sequence with GQA repeat,
    on q/k rotated by the complex-number RoPE."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    outs = []
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        L = s1 - s0
        if L == 0:
            continue
        pos = np.arange(L)
        qr = rope_complex(q[s0:s1], pos, base, drot, style)
        kr = rope_complex(k[s0:s1], pos, base, drot, style)
        qt = torch.from_numpy(qr).permute(1, 0, 2)  # [Hq, L, d]
        kt = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(G, dim=0)
        vt = torch.from_numpy(v[s0:s1]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        i = torch.arange(L)[:, None]
        j = torch.arange(L)[None, :]
        mask = j <= i
        if window > 0:
            mask &= j > i - window
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask, scale=scale)
        outs.append(o.permute(1, 0, 2).numpy())
    return np.concatenate(outs, axis=0)


@pytest.mark.parametrize("window", [0, 1, 3, 5, 40])
@pytest.mark.parametrize("style", [0, 1])
def test_sink_neg_inf_is_sdpa(oracle_mod, window, style):
    gen = torch.Generator().manual_seed(11 + window + 100 * style)
    lens = [7, 0, 13, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, Hq, Hkv = int(cu[-1]), 8, 2
    q, k, v = bf16_tensor((total, Hq, 192), gen), bf16_tensor((total, Hkv, 192), gen), \
        bf16_tensor((total, Hkv, 128), gen)
    sink = torch.full((Hq,), -math.inf)
    out, _ = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=1e4,
                                rope_style=style)
    ref = _sdpa_reference(to64(q), to64(k), to64(v), cu, window, 1e4, 64, style,
                          1.0 / math.sqrt(192))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ------------------------- (iii) the sink is an extra logit whose value is 0
@pytest.mark.parametrize("window", [0, 4])
def test_sink_is_extra_key_with_zero_value(oracle_mod, window):
    gen = torch.Generator().manual_seed(5)
    L, Hq, Hkv = 12, 4, 1
    q, k, v = bf16_tensor((L, Hq, 192), gen), bf16_tensor((L, Hkv, 192), gen), \
        bf16_tensor((L, Hkv, 128), gen)
    sink = torch.tensor([-1.5, 0.0, 0.7, 3.0])
    cu = np.array([0, L], dtype=np.int32)
    base = 640000.0
    out, lse = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=base)
    pos = np.arange(L)
    qr = rope_complex(to64(q), pos, base, 64, 0)
    kr = rope_complex(to64(k), pos, base, 64, 0)
    vv = to64(v)
    s = 1.0 / math.sqrt(192)
    for h in range(Hq):
        logits = torch.from_numpy(qr[:, h] @ kr[:, 0].T * s)  # [L, L]
        i = torch.arange(L)[:, None]
        j = torch.arange(L)[None, :]
        vis = (j <= i) & ((j > i - window) if window else torch.ones_like(j, dtype=torch.bool))
        logits = logits.masked_fill(~vis, -math.inf)
        ext = torch.cat([logits, torch.full((L, 1), float(sink[h]), dtype=torch.float64)], 1)
        w = torch.softmax(ext, dim=1)[:, :L]
        ref_o = w.numpy() @ vv[:, 0]
        ref_lse = torch.logsumexp(ext, dim=1).numpy()
        np.testing.assert_allclose(out[:, h], ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, h], ref_lse, rtol=0, atol=1e-12)


# ------------------------------------ (iv) weights plus sink weight sum to 1
def test_weights_plus_sink_sum_to_one(oracle_mod):
    gen = torch.Generator().manual_seed(9)
    lens = [1, 17, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, Hq, Hkv = int(cu[-1]), 8, 2
    q, k = bf16_tensor((total, Hq, 192), gen), bf16_tensor((total, Hkv, 192), gen)
    v = torch.ones(total, Hkv, 128, dtype=torch.bfloat16)
    sink = torch.randn(Hq, generator=gen) * 3
    for window in (0, 5):
        out, lse = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=1e4)
        sw = np.exp(sink.double().numpy()[None, :] - lse)
        np.testing.assert_allclose(out[:, :, 0] + sw, 1.0, rtol=0, atol=1e-13)
        assert np.all(out[:, :, 0] < 1.0)


# ------------------------------------------- (v) identical keys: closed form
@pytest.mark.parametrize("sink", [-2.0, 0.0, 1.25])
def test_identical_keys_closed_form(oracle_mod, sink):
    L, Hq, Hkv, a = 9, 2, 1, 0.8
    q = np.zeros((L, Hq, 4)); q[:, :, 0] = a
    k = np.zeros((L, Hkv, 4)); k[:, :, 0] = 1.0
    vrow = np.array([0.5, -1.0, 2.0])
    v = np.broadcast_to(vrow, (L, Hkv, 3)).copy()
    cu = np.array([0, L], dtype=np.int32)
    sk = np.full(Hq, sink, dtype=np.float32)
    for window in (0, 3):
        out, lse = oracle_mod.prefill(q, k, v, sk, cu, window=window, rope_base=0.0,
                                      scale=1.0, drot=0)
        for i in range(L):
            n = i + 1 if window == 0 else min(i + 1, window)
            sig = 1.0 / (1.0 + math.exp(-(a + math.log(n) - float(sk[0]))))
            np.testing.assert_allclose(out[i, 0], sig * vrow, rtol=0, atol=1e-13)
            assert abs(lse[i, 0] - math.log(math.exp(float(sk[0])) + n * math.exp(a))) < 1e-13


# ------------------------------------------------- (vi) shift invariance
def test_shift_invariance(oracle_mod):
    rng = np.random.default_rng(3)
    L, Hq, Hkv, d = 10, 2, 1, 6
    q = rng.standard_normal((L, Hq, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, 5))
    sink = np.array([0.25, -0.875], dtype=np.float32)  # sink + c exact in fp32
    cu = np.array([0, L], dtype=np.int32)
    c = 2.5
    # add c to every logit through an extra dim (q_extra = c, k_extra = 1) and to the sink
    q2 = np.concatenate([q, np.full((L, Hq, 1), c)], axis=2)
    k2 = np.concatenate([k, np.ones((L, Hkv, 1))], axis=2)
    o1, l1 = oracle_mod.prefill(np.concatenate([q, np.zeros((L, Hq, 1))], 2), k2, v, sink, cu,
                                window=0, rope_base=0.0, scale=1.0, drot=0)
    o2, l2 = oracle_mod.prefill(q2, k2, v, (sink + np.float32(c)), cu, window=0,
                                rope_base=0.0, scale=1.0, drot=0)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1 + c, rtol=0, atol=1e-12)


# ------------------------------------------- negative logit scale (sign flip)
@pytest.mark.parametrize("window", [0, 3])
def test_negative_scale_is_negated_query(oracle_mod, window):
    """a = scale * (rot(q) . rot(k)) and the rotation is linear, so a scale -s
    with q is the scale s with -q, bit for bit: the oracle's path for negative
    scales (the ones the general kernel takes) reduces to its positive one."""
    rng = np.random.default_rng(11)
    L, Hq, Hkv = 9, 4, 2
    q = rng.standard_normal((L, Hq, 192))
    k = rng.standard_normal((L, Hkv, 192))
    v = rng.standard_normal((L, Hkv, 128))
    sink = rng.standard_normal(Hq).astype(np.float32)
    cu = np.array([0, 5, L], dtype=np.int32)
    for s in (0.07, 1.0 / math.sqrt(192)):
        o1, l1 = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=1e4, scale=-s)
        o2, l2 = oracle_mod.prefill(-q, k, v, sink, cu, window=window, rope_base=1e4, scale=s)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)
        # and it is not the positive-scale result on q itself
        o3, _ = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=1e4, scale=s)
        assert np.max(np.abs(o3 - o1)) > 1e-3


# ------------------------------------------------------- (vii) large sink
def test_large_sink_suppresses_output(oracle_mod):
    gen = torch.Generator().manual_seed(1)
    L, Hq, Hkv = 20, 8, 1
    q, k, v = bf16_tensor((L, Hq, 192), gen), bf16_tensor((L, Hkv, 192), gen), \
        bf16_tensor((L, Hkv, 128), gen)
    sink = torch.full((Hq,), 40.0)
    cu = np.array([0, L], dtype=np.int32)
    out, lse = oracle_mod.prefill(q, k, v, sink, cu, window=0, rope_base=1e4)
    assert np.max(np.abs(out)) < 1e-9
    np.testing.assert_allclose(lse, 40.0, atol=1e-9)


# --------------------------------------------- (viii) W >= L is the global variant
def test_window_at_least_length_is_global(oracle_mod):
    gen = torch.Generator().manual_seed(2)
    lens = [5, 31, 16]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, Hq, Hkv = int(cu[-1]), 4, 2
    q, k, v = bf16_tensor((total, Hq, 192), gen), bf16_tensor((total, Hkv, 192), gen), \
        bf16_tensor((total, Hkv, 128), gen)
    sink = torch.randn(Hq, generator=gen)
    og, lg = oracle_mod.prefill(q, k, v, sink, cu, window=0, rope_base=1e4)
    for w in (31, 32, 1000):
        ow, lw = oracle_mod.prefill(q, k, v, sink, cu, window=w, rope_base=1e4)
        assert np.array_equal(ow, og) and np.array_equal(lw, lg)
    ow, _ = oracle_mod.prefill(q, k, v, sink, cu, window=30, rope_base=1e4)
    assert not np.array_equal(ow, og)


# ----------------------- (ix) brute force with the page's unshifted formula
def _brute_prefill(q, k, v, sink, lens, window, base, drot, style, scale):
    """Pure-Python loops: enumerate each row's visible set explicitly and use
    exp(a) / (exp(sink) + sum exp(a)) with no max subtraction."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    out = np.zeros((q.shape[0], Hq, v.shape[2]))
    lse = np.zeros((q.shape[0], Hq))
    s0 = 0
    for L in lens:
        pos = np.arange(L)
        qr = rope_complex(q[s0:s0 + L], pos, base, drot, style)
        kr = rope_complex(k[s0:s0 + L], pos, base, drot, style)
        for i in range(L):
            vis = [j for j in range(L) if j <= i and (window == 0 or i - window < j)]
            for h in range(Hq):
                g = h // G
                e = {j: math.exp(scale * float(np.dot(qr[i, h], kr[j, g]))) for j in vis}
                den = math.exp(float(sink[h])) + sum(e.values())
                out[s0 + i, h] = sum(e[j] * v[s0 + j, g] for j in vis) / den
                lse[s0 + i, h] = math.log(den)
        s0 += L
    return out, lse


def test_bruteforce_all_small_shapes(oracle_mod):
    rng = np.random.default_rng(7)
    d, dv = 6, 3
    n_cases = 0
    for L, G in itertools.product(range(1, 8), (1, 2, 4)):
        for window in range(0, L + 2):
            Hkv = 2 if G < 4 else 1
            Hq = G * Hkv
            q = rng.uniform(-1, 1, (L, Hq, d))
            k = rng.uniform(-1, 1, (L, Hkv, d))
            v = rng.uniform(-1, 1, (L, Hkv, dv))
            sink = rng.uniform(-1, 1, Hq).astype(np.float32)
            cu = np.array([0, L], dtype=np.int32)
            style = (L + window) % 2
            o, l = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=7.0,
                                      scale=0.7, drot=4, rope_style=style)
            ob, lb = _brute_prefill(q, k, v, sink, [L], window, 7.0, 4, style, 0.7)
            np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)
            n_cases += 1
    assert n_cases > 100


def test_bruteforce_varlen_batch(oracle_mod):
    rng = np.random.default_rng(8)
    lens = [3, 0, 6, 1, 5]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, Hq, Hkv = int(cu[-1]), 4, 2
    q = rng.uniform(-1, 1, (total, Hq, 8))
    k = rng.uniform(-1, 1, (total, Hkv, 8))
    v = rng.uniform(-1, 1, (total, Hkv, 4))
    sink = rng.uniform(-1, 1, Hq).astype(np.float32)
    for window in (0, 2):
        o, l = oracle_mod.prefill(q, k, v, sink, cu, window=window, rope_base=11.0,
                                  scale=0.5, drot=4)
        ob, lb = _brute_prefill(q, k, v, sink, lens, window, 11.0, 4, 0, 0.5)
        np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lb, rtol=0, atol=1e-12)


# ------------------------------------------------------------ (x)-(xiii) RoPE
def test_rope_closed_form_two_dims(oracle_mod):
    # drot = 2: theta_0 = base^0 = 1, so (1, 0) at position p is (cos p, sin p)
    for p in (0.0, 1.0, 2.5, 100.0, 131071.0):
        y = oracle_mod.rope(np.array([1.0, 0.0, 0.3]), p, base=1e4, drot=2)
        np.testing.assert_allclose(y, [math.cos(p), math.sin(p), 0.3], rtol=0, atol=1e-12)
    # so the logit between positions i and j is cos(i - j)
    for i, j in ((5, 2), (9, 9), (1000, 3)):
        a = np.dot(oracle_mod.rope(np.array([1.0, 0.0]), i, base=3.0, drot=2),
                   oracle_mod.rope(np.array([1.0, 0.0]), j, base=3.0, drot=2))
        assert abs(a - math.cos(i - j)) < 1e-12


@pytest.mark.parametrize("style", [0, 1])
@pytest.mark.parametrize("base", [1e4, 5e6])
def test_rope_matches_complex_form(oracle_mod, style, base):
    rng = np.random.default_rng(4)
    x = rng.standard_normal(192)
    for p in (0, 1, 77, 32767, 262143):
        y = oracle_mod.rope(x, p, base=base, drot=64, rope_style=style)
        ref = rope_complex(x[None, :], np.array([p]), base, 64, style)[0]
        np.testing.assert_allclose(y, ref, rtol=0, atol=1e-9)
        assert np.array_equal(y[64:], x[64:])                      # dims 64.. untouched
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12  # norm preserved
    assert np.array_equal(oracle_mod.rope(x, 0, base=base, rope_style=style), x)


def test_rope_relative_position(oracle_mod):
    rng = np.random.default_rng(6)
    qv, kv = rng.standard_normal(192), rng.standard_normal(192)
    for i, j, delta in ((10, 3, 1000), (200, 200, 7), (5, 0, 65536)):
        a0 = np.dot(oracle_mod.rope(qv, i, base=1e4), oracle_mod.rope(kv, j, base=1e4))
        a1 = np.dot(oracle_mod.rope(qv, i + delta, base=1e4),
                    oracle_mod.rope(kv, j + delta, base=1e4))
        assert abs(a0 - a1) < 1e-9


# ---------------------------------------------- (xiv) decode = prefill tail
@pytest.mark.parametrize("window", [0, 3, 128])
def test_decode_equals_prefill_tail(oracle_mod, window):
    gen = torch.Generator().manual_seed(21)
    B, T, S_cap, Hq, Hkv = 3, 4, 40, 8, 2
    seqlens = [4, 17, 40]
    kc = bf16_tensor((B, S_cap, Hkv, 192), gen)
    vc = bf16_tensor((B, S_cap, Hkv, 128), gen)
    qd = bf16_tensor((B, T, Hq, 192), gen)
    sink = torch.randn(Hq, generator=gen)
    od, ld = oracle_mod.decode(qd, kc, vc, torch.tensor(seqlens, dtype=torch.int32), sink,
                               window=window, rope_base=5e6)
    for b, L in enumerate(seqlens):
        # the same sequence as a prefill whose last T query rows are the drafts
        qp = bf16_tensor((L, Hq, 192), gen)
        qp[L - T:] = qd[b]
        cu = np.array([0, L], dtype=np.int32)
        op, lp = oracle_mod.prefill(qp, kc[b, :L], vc[b, :L], sink, cu, window=window,
                                    rope_base=5e6)
        np.testing.assert_allclose(od[b], op[L - T:], rtol=0, atol=1e-12)
        np.testing.assert_allclose(ld[b], lp[L - T:], rtol=0, atol=1e-12)


def test_decode_short_cache_rows_are_empty(oracle_mod):
    # seqlen < T: queries at negative positions see nothing -> o = 0, lse = sink
    gen = torch.Generator().manual_seed(22)
    B, T, S_cap, Hq, Hkv = 1, 4, 8, 2, 1
    kc, vc = bf16_tensor((B, S_cap, Hkv, 192), gen), bf16_tensor((B, S_cap, Hkv, 128), gen)
    qd = bf16_tensor((B, T, Hq, 192), gen)
    sink = torch.tensor([0.5, -math.inf])
    od, ld = oracle_mod.decode(qd, kc, vc, torch.tensor([2], dtype=torch.int32), sink,
                               window=0, rope_base=1e4)
    assert np.all(od[0, :2] == 0.0)
    assert ld[0, 0, 0] == pytest.approx(0.5) and ld[0, 0, 1] == -math.inf
    assert np.all(np.isfinite(ld[0, 2:]))


# ------------------- (xv) split-KV restatement: sink counted once in the merge
def test_split_merge_counts_sink_once(oracle_mod):
    """The merge of per-chunk partials (m_s, l_s, O_s) taken WITHOUT the sink,
    followed by one sink term, reproduces eq. (2) over the whole row -- for any
    partition of the keys."""
    gen = torch.Generator().manual_seed(31)
    B, T, S_cap, Hq, Hkv = 1, 4, 300, 4, 1
    seqlens = [300]
    kc, vc = bf16_tensor((B, S_cap, Hkv, 192), gen), bf16_tensor((B, S_cap, Hkv, 128), gen)
    qd = bf16_tensor((B, T, Hq, 192), gen)
    sink = torch.tensor([0.0, 1.0, -3.0, 2.0])
    ref_o, ref_l = oracle_mod.decode(qd, kc, vc, torch.tensor(seqlens, dtype=torch.int32),
                                     sink, window=0, rope_base=1e4)
    # logits from the oracle's own rope (fp64) and a plain dot product
    s = 1.0 / math.sqrt(192)
    kr = np.stack([oracle_mod.rope(to64(kc[0, j, 0]), j, base=1e4) for j in range(300)])
    vv = to64(vc[0, :, 0])
    for bounds in ([0, 300], [0, 128, 256, 300], [0, 1, 2, 299, 300], [0, 77, 150, 300]):
        for t in range(T):
            p = 300 - T + t
            for h in range(Hq):
                qr = oracle_mod.rope(to64(qd[0, t, h]), p, base=1e4)
                parts = []
                for c0, c1 in zip(bounds[:-1], bounds[1:]):
                    js = [j for j in range(c0, c1) if j <= p]
                    if not js:
                        continue
                    a = np.array([s * np.dot(qr, kr[j]) for j in js])
                    m = a.max()
                    e = np.exp(a - m)
                    parts.append((m, e.sum(), e @ vv[js]))
                sk = float(sink[h])
                M = max([sk] + [m for m, _, _ in parts])
                Ls = math.exp(sk - M) + sum(l * math.exp(m - M) for m, l, _ in parts)
                o = sum(math.exp(m - M) * O for m, _, O in parts) / Ls
                np.testing.assert_allclose(o, ref_o[0, t, h], rtol=0, atol=1e-12)
                assert abs(M + math.log(Ls) - ref_l[0, t, h]) < 1e-12


# --------------------------- rotated-cache decode (a cache holding rotated keys)
@pytest.mark.parametrize("style", [0, 1])
def test_rope_rows_matches_complex_form(oracle_mod, style):
    """The oracle's row-wise rotation (used to build rotated caches) against the
    complex-number form, one position per row."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((50, 3, 192))
    pos = rng.integers(0, 262144, size=50).astype(np.float64)
    y = oracle_mod.rope_rows(x, pos[:, None], base=5e6, rope_style=style)
    np.testing.assert_allclose(y, rope_complex(x, pos, 5e6, 64, style), rtol=0, atol=1e-9)


@pytest.mark.parametrize("window,style", [(0, 0), (3, 0), (128, 1)])
def test_decode_rotated_cache_equals_raw_cache(oracle_mod, window, style):
    """A cache that stores every key already rotated at its own position (rotated
    here by the complex-number form, independently of the oracle), decoded with
    k_rotated, gives the decode of the raw cache: the rotation of a key depends
    on its position only, so doing it when the key is stored or when it is read
    is the same arithmetic."""
    gen = torch.Generator().manual_seed(23)
    B, T, S_cap, Hq, Hkv, base = 3, 4, 300, 8, 2, 1e4
    seqlens = [4, 170, 300]
    kc = to64(bf16_tensor((B, S_cap, Hkv, 192), gen))
    vc = to64(bf16_tensor((B, S_cap, Hkv, 128), gen))
    qd = to64(bf16_tensor((B, T, Hq, 192), gen))
    sink = torch.randn(Hq, generator=gen)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    pos = np.arange(S_cap, dtype=np.float64)
    kr = np.stack([rope_complex(kc[b], pos, base, 64, style) for b in range(B)])
    o0, l0 = oracle_mod.decode(qd, kc, vc, sl, sink, window=window, rope_base=base,
                               rope_style=style)
    o1, l1 = oracle_mod.decode(qd, kr, vc, sl, sink, window=window, rope_base=base,
                               rope_style=style, k_rotated=True)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)
    # without the switch the keys would be rotated twice: a different result
    o2, _ = oracle_mod.decode(qd, kr, vc, sl, sink, window=window, rope_base=base,
                              rope_style=style)
    assert np.abs(o2 - o0).max() > 1e-3
