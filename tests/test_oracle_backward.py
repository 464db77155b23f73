"""Pins for the oracle's backward pass (oracle.prefill_backward).

The gradient of L = sum(dO * o) is checked against two things other than the
oracle's own chain rule: (1) torch fp64 autograd through an independent
restatement of eqs. (1)-(3) of §2.2 of the MiMo-V2-Flash Technical Report, the
sink written as one extra key column whose value vector is zero and RoPE in
complex form, and (2) central finite differences of the oracle's forward.
"""
import math

import numpy as np
import pytest
import torch


def _inputs(lens, hq, hkv, dqk, dv, seed):
    g = np.random.default_rng(seed)
    total = sum(lens)
    q = g.standard_normal((total, hq, dqk))
    k = g.standard_normal((total, hkv, dqk))
    v = g.standard_normal((total, hkv, dv))
    dout = g.standard_normal((total, hq, dv))
    sink = g.standard_normal(hq).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, dout, sink, cu


def _torch_rope(x, pos, base, drot, style):
    """RoPE as complex multiplication (RoFormer), differentiable."""
    if drot == 0:
        return x
    half = drot // 2
    theta = base ** (-2.0 * torch.arange(half, dtype=torch.float64) / drot)
    ang = pos[:, None].to(torch.float64) * theta[None, :]
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    if style == 0:
        a, b = x[..., 0:drot:2], x[..., 1:drot:2]
    else:
        a, b = x[..., :half], x[..., half:drot]
    ra, rb = a * c - b * s, a * s + b * c
    if style == 0:
        rot = torch.stack([ra, rb], dim=-1).reshape(x.shape[:-1] + (drot,))
    else:
        rot = torch.cat([ra, rb], dim=-1)
    return torch.cat([rot, x[..., drot:]], dim=-1)


def _torch_forward(q, k, v, sink, cu, window, base, drot, style, scale):
    """o for every (token, head): per sequence, logits plus one sink column,
    torch.softmax, the sink column dropped, times v."""
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    outs = []
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        L = s1 - s0
        if L == 0:
            continue
        pos = torch.arange(L)
        qr = _torch_rope(q[s0:s1], pos, base, drot, style)
        kr = _torch_rope(k[s0:s1], pos, base, drot, style)
        krep = kr.repeat_interleave(G, dim=1)           # [L, hq, dqk]
        vrep = v[s0:s1].repeat_interleave(G, dim=1)
        a = torch.einsum("ihd,jhd->hij", qr, krep) * scale  # [hq, L, L]
        i = torch.arange(L)[:, None]
        j = torch.arange(L)[None, :]
        vis = (j <= i) & ((window == 0) | (j > i - window))
        a = a.masked_fill(~vis, -math.inf)
        col = sink.to(torch.float64)[:, None, None].expand(hq, L, 1)
        w = torch.softmax(torch.cat([a, col], dim=-1), dim=-1)[..., :L]
        outs.append(torch.einsum("hij,jhd->ihd", w, vrep))
    return torch.cat(outs, dim=0)


@pytest.mark.parametrize("window,style,base", [(0, 0, 1e4), (2, 1, 1e4), (3, 0, 5e6), (0, 1, 0.0)])
def test_backward_matches_torch_autograd(oracle_mod, window, style, base):
    lens, hq, hkv, dqk, dv, drot = [5, 0, 7, 1], 4, 2, 8, 6, 4
    q, k, v, dout, sink, cu = _inputs(lens, hq, hkv, dqk, dv, seed=window + 10 * style)
    sink[1] = -np.inf                      # a head without sink: dsink = 0
    scale = 0.37
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ts = torch.tensor(sink.astype(np.float64), requires_grad=True)
    o = _torch_forward(tq, tk, tv, ts, cu, window, base, drot if base > 0 else 0, style, scale)
    (o * torch.tensor(dout)).sum().backward()
    dq, dk, dvv, ds = oracle_mod.prefill_backward(q, k, v, sink, cu, dout, window=window,
                                                  rope_base=base, scale=scale, drot=drot,
                                                  rope_style=style)
    assert np.max(np.abs(dq - tq.grad.numpy())) < 1e-11
    assert np.max(np.abs(dk - tk.grad.numpy())) < 1e-11
    assert np.max(np.abs(dvv - tv.grad.numpy())) < 1e-11
    want_ds = ts.grad.numpy().copy()
    want_ds[1] = 0.0
    assert np.max(np.abs(ds - want_ds)) < 1e-11
    assert ds[1] == 0.0


def test_backward_matches_finite_differences(oracle_mod):
    """Central differences of L(x) = sum(dO * o(x)) with the oracle's forward."""
    lens, hq, hkv, dqk, dv, drot = [4, 3], 2, 1, 6, 3, 4
    q, k, v, dout, sink, cu = _inputs(lens, hq, hkv, dqk, dv, seed=3)
    sink[:] = np.float32([0.25, -0.5])
    kw = dict(window=2, rope_base=100.0, scale=0.5, drot=drot, rope_style=0)

    def loss(q_, k_, v_, s_):
        o, _ = oracle_mod.prefill(q_, k_, v_, s_, cu, **kw)
        return float(np.sum(o * dout))

    dq, dk, dvv, ds = oracle_mod.prefill_backward(q, k, v, sink, cu, dout, **kw)
    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dvv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            ap = [xp if a is x else a for a in args]
            am = [xm if a is x else a for a in args]
            num = (loss(*ap, sink) - loss(*am, sink)) / (2 * h)
            assert abs(num - grad[idx]) < 1e-7, (name, idx, num, grad[idx])
    for hh in range(hq):
        sp, sm = sink.copy(), sink.copy()
        sp[hh] = np.float32(sink[hh] + np.float32(1e-3))
        sm[hh] = np.float32(sink[hh] - np.float32(1e-3))
        num = (loss(q, k, v, sp) - loss(q, k, v, sm)) / (float(sp[hh]) - float(sm[hh]))
        assert abs(num - ds[hh]) < 1e-6, (hh, num, ds[hh])
