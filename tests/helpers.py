"""Shared helpers for the parity tests (no attention arithmetic here)."""
import numpy as np
import torch

# Tolerances of the parity gate: max-abs error of out (bf16) and of lse (fp32)
# against the fp64 oracle.
OUT_TOL = 1e-2
LSE_TOL = 2e-3


def max_abs(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    d = np.abs(np.where(both_inf, 0.0, a - b))
    return float(np.nanmax(np.where(np.isnan(d), np.inf, d))) if d.size else 0.0


def assert_parity(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    l = lse_gpu.detach().float().cpu().numpy().astype(np.float64)
    eo = max_abs(o, out_ref)
    el = max_abs(l, lse_ref)
    assert eo <= OUT_TOL and el <= LSE_TOL, f"{what}: out err {eo:.3e}, lse err {el:.3e}"
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
