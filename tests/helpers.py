"""Shared helpers for the parity tests (no attention arithmetic here)."""
import numpy as np
import torch

# Tolerances of the parity gate: max-abs error of out (bf16) and of lse (fp32)
# against the fp64 oracle.  out is delivered in bf16 (8 significant bits), and
# rounding an exact result to bf16 alone moves it by up to half a bf16 step,
# 2^(e-8) for |x| in [2^e, 2^(e+1)): 0.0078 at |x| in [2, 4), 0.0156 at [4, 8),
# more than the whole gate.  The out gate therefore bounds the error of the
# computation, beyond that final rounding: |out - oracle| <= OUT_TOL + half a
# bf16 step at that magnitude.
OUT_TOL = 1e-2
LSE_TOL = 2e-3


def bf16_half_step(x):
    """Half the spacing of bf16 numbers at magnitude |x| (the largest error of
    rounding x to the nearest bf16)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def out_err(gpu, ref):
    """Largest |gpu - ref| beyond half a bf16 step at max(|gpu|, |ref|): the
    error of the computation with the final rounding to the bf16 output taken
    out (NaN where one side is NaN counts as infinite)."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64).reshape(g.shape)
    both_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    d = np.abs(np.where(both_inf, 0.0, g - r))
    with np.errstate(invalid="ignore"):
        d = d - bf16_half_step(np.maximum(np.abs(np.where(np.isfinite(g), g, 0.0)),
                                          np.abs(np.where(np.isfinite(r), r, 0.0))))
    d = np.where(np.isnan(d), np.inf, np.maximum(d, 0.0))
    return float(d.max()) if d.size else 0.0


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    d = np.abs(np.where(both_inf, 0.0, a - b))
    return float(np.nanmax(np.where(np.isnan(d), np.inf, d))) if d.size else 0.0


def worst_element(a, b):
    """(flat index, a value, b value) of the largest |a - b|."""
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    d = np.abs(a - b)
    d = np.where(np.isnan(d), np.inf, d)
    i = int(np.argmax(d)) if d.size else 0
    return i, (float(a[i]) if d.size else 0.0), (float(b[i]) if d.size else 0.0)


def assert_parity(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    l = lse_gpu.detach().float().cpu().numpy().astype(np.float64)
    eo = out_err(o, out_ref)
    el = max_abs(l, lse_ref)
    if not (eo <= OUT_TOL and el <= LSE_TOL):
        i, g, r = worst_element(o, np.asarray(out_ref).reshape(o.shape))
        dv = o.shape[-1] if o.ndim else 1
        raise AssertionError(f"{what}: out err {eo:.3e} (beyond bf16 rounding; raw "
                             f"{max_abs(o, out_ref):.3e}), lse err {el:.3e}; worst out element "
                             f"row {i // dv} dim {i % dv}: gpu {g:.6g} oracle {r:.6g}")
    return eo, el


def sample_rows(n_tokens, hq, k, seed, must=()):
    """k token indices (sorted, unique) including `must`, every head of each."""
    rng = np.random.default_rng(seed)
    toks = set(int(t) for t in must if 0 <= t < n_tokens)
    while len(toks) < min(k, n_tokens):
        toks.add(int(rng.integers(0, n_tokens)))
    toks = np.array(sorted(toks), dtype=np.int64)
    rows = (toks[:, None] * hq + np.arange(hq)[None, :]).reshape(-1)
    return toks, rows
