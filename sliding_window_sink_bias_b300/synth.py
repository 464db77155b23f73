"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and shapes only; it holds none of the
attention arithmetic.  Both the CUDA path and the oracle receive the very same
tensors made here.  Values follow the workloads of the MiMo-V2-Flash model
(§2.1 Table 1: 64 query heads, 8 KV heads for sliding-window layers and 4 for
global layers, QK head dim 192, V head dim 128): q, k, v ~ N(0, 1) rounded to
bf16, one sink per query head ~ N(0, 1) in fp32.

Generators are torch's own (CPU or CUDA Philox), seeded per tensor, so a given
(seed, device) always yields the same bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DQK = 192
DV = 128
DROT = 64

# tensor stream ids, so each tensor of a workload has its own seed
_STREAM = {"q": 1, "k": 2, "v": 3, "sink": 4, "lens": 5, "kcache": 6, "vcache": 7, "dout": 8}


def _gen(seed: int, stream: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + _STREAM[stream] * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def randn_bf16(shape, seed: int, stream: str, device="cpu") -> torch.Tensor:
    return torch.randn(*shape, generator=_gen(seed, stream, device), device=device,
                       dtype=torch.bfloat16)


def sink_vector(hq: int, seed: int, device="cpu") -> torch.Tensor:
    return torch.randn(hq, generator=_gen(seed, "sink", "cpu"), dtype=torch.float32).to(device)


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    sink: torch.Tensor
    cu_seqlens: torch.Tensor  # int32 [B+1], on the same device as q
    seqlens: list
    window: int
    rope_base: float

    @property
    def total(self) -> int:
        return int(sum(self.seqlens))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens)) if self.seqlens else 0


def prefill_inputs(seqlens, hq: int, hkv: int, *, window: int, rope_base: float,
                   seed: int = 0, device="cpu") -> PrefillInputs:
    seqlens = [int(x) for x in seqlens]
    total = sum(seqlens)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    return PrefillInputs(
        q=randn_bf16((total, hq, DQK), seed, "q", device),
        k=randn_bf16((total, hkv, DQK), seed, "k", device),
        v=randn_bf16((total, hkv, DV), seed, "v", device),
        sink=sink_vector(hq, seed, device),
        cu_seqlens=torch.from_numpy(cu).to(device),
        seqlens=seqlens, window=int(window), rope_base=float(rope_base))


@dataclass
class DecodeInputs:
    q: torch.Tensor        # [B, T, Hq, 192]
    kcache: torch.Tensor   # [B, S_cap, Hkv, 192]
    vcache: torch.Tensor   # [B, S_cap, Hkv, 128]
    seqlens: torch.Tensor  # int32 [B]
    sink: torch.Tensor
    window: int
    rope_base: float
    seqlens_host: list = field(default_factory=list)

    @property
    def max_seqlen(self) -> int:
        return int(max(self.seqlens_host)) if self.seqlens_host else 0


def decode_inputs(seqlens, t: int, s_cap: int, hq: int, hkv: int, *, window: int,
                  rope_base: float, seed: int = 0, device="cpu") -> DecodeInputs:
    seqlens = [int(x) for x in seqlens]
    b = len(seqlens)
    return DecodeInputs(
        q=randn_bf16((b, t, hq, DQK), seed, "q", device),
        kcache=randn_bf16((b, s_cap, hkv, DQK), seed, "kcache", device),
        vcache=randn_bf16((b, s_cap, hkv, DV), seed, "vcache", device),
        seqlens=torch.tensor(seqlens, dtype=torch.int32, device=device),
        sink=sink_vector(hq, seed, device),
        window=int(window), rope_base=float(rope_base), seqlens_host=seqlens)


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n integers uniform in [lo, hi] (decode cache lengths)."""
    rng = np.random.default_rng([int(seed), _STREAM["lens"]])
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def log_uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    """n lengths round(exp(U[ln lo, ln hi])) (the ragged hybrid-block batch)."""
    rng = np.random.default_rng([int(seed), _STREAM["lens"]])
    u = rng.uniform(math.log(lo), math.log(hi), size=n)
    return [int(min(hi, max(lo, round(math.exp(x))))) for x in u]


# The workloads, named by what they are (shapes from §2.1 Table 1, context
# lengths from §3.1/§3.2: 32K native, 256K extended; MTP verify = 1 + 3 drafts).
SWA = dict(hq=64, hkv=8, window=128, rope_base=1e4)
GA = dict(hq=64, hkv=4, window=0, rope_base=5e6)

WORKLOADS = {
    "swa_tiny_1x512": dict(kind="prefill", seqlens=[512], **SWA),
    "swa_prefill_4x32768": dict(kind="prefill", seqlens=[32768] * 4, **SWA),
    "ga_prefill_1x131072": dict(kind="prefill", seqlens=[131072], **GA),
    "mtp_decode_ga_b64_t4": dict(kind="decode", batch=64, t=4, s_cap=262144,
                                 len_lo=65536, len_hi=262144, **GA),
    "mtp_decode_swa_b64_t4": dict(kind="decode", batch=64, t=4, s_cap=262144,
                                  len_lo=65536, len_hi=262144, **SWA),
    # the GA decode batch over an FP8 (E4M3) cache, one scale per KV head
    "mtp_decode_ga_fp8_b64_t4": dict(kind="decode", batch=64, t=4, s_cap=262144, fp8=True,
                                     len_lo=65536, len_hi=262144, **GA),
    # the same FP8 batch with the keys stored after RoPE (an FP8 cache is
    # quantised when a key is stored, after its rotation): the kernel rotates q only
    "mtp_decode_ga_fp8_rot_b64_t4": dict(kind="decode", batch=64, t=4, s_cap=262144, fp8=True,
                                         k_rotated=True, len_lo=65536, len_hi=262144, **GA),
    # the same SWA layer with the KV cache an SWA layer needs: a ring of 144
    # slots (>= W + T - 1 = 131, a multiple of 16) per sequence
    "mtp_decode_swa_ring_b64_t4": dict(kind="decode", batch=64, t=4, s_cap=144, kv_ring=True,
                                       len_lo=65536, len_hi=262144, **SWA),
    # the same ring holding keys stored after RoPE: the kernel rotates q only
    "mtp_decode_swa_ring_rot_b64_t4": dict(kind="decode", batch=64, t=4, s_cap=144, kv_ring=True,
                                           k_rotated=True, len_lo=65536, len_hi=262144, **SWA),
    # one hybrid block of the model (§2.1: 5 SWA layers then 1 GA layer) over a
    # varlen batch of 8 sequences, lengths log-uniform in [4096, 131072]
    "hybrid_block_ragged_8seq": dict(kind="hybrid", n_seq=8, len_lo=4096, len_hi=131072,
                                     swa_layers=5, ga_layers=1, hq=64, swa_hkv=8, ga_hkv=4,
                                     window=128, swa_base=1e4, ga_base=5e6),
    # one SWA layer and one GA layer of the model timed on a single sequence at
    # 32K, 128K and 256K tokens: attention time of a hybrid block (5 SWA + 1 GA)
    # and of the 48-layer stack (39 SWA + 9 GA) against all-global attention
    "hybrid_vs_all_ga": dict(kind="ratio", lens=[32768, 131072, 262144], hq=64, swa_hkv=8,
                             ga_hkv=4, window=128, swa_base=1e4, ga_base=5e6,
                             block=(5, 1), model=(39, 9)),
    # backward pass (dq, dk, dv, dsink) of an SWA layer on the bulk batch and of
    # a GA layer at 32K tokens
    "swa_backward_4x32768": dict(kind="backward", seqlens=[32768] * 4, **SWA),
    "ga_backward_1x32768": dict(kind="backward", seqlens=[32768], **GA),
    # the same SWA layer with a 512-token window (outside the band kernel's
    # W <= 128): the causal kernel, visiting only the key blocks the window reaches
    "swa_w512_prefill_1x32768": dict(kind="prefill", seqlens=[32768], hq=64, hkv=8, window=512,
                                     rope_base=1e4),
    # a 128-token window over 64 query heads in pairs (2 per KV head, tiles of
    # 64 tokens): the causal kernel
    "swa_g2_prefill_1x32768": dict(kind="prefill", seqlens=[32768], hq=64, hkv=32, window=128,
                                   rope_base=1e4),
    # reduced shapes of the same kernels, for profiler captures (a few GB on the device)
    "swa_prefill_1x32768": dict(kind="prefill", seqlens=[32768], **SWA),
    # the SWA layer with a negative logit scale: the general prefill kernel
    "swa_negscale_prefill_1x32768": dict(kind="prefill", seqlens=[32768], scale=-0.0721,
                                         **SWA),
    "ga_prefill_1x16384": dict(kind="prefill", seqlens=[16384], **GA),
    "mtp_decode_ga_b8_t4": dict(kind="decode", batch=8, t=4, s_cap=131072,
                                len_lo=65536, len_hi=131072, **GA),
    "mtp_decode_ga_fp8_b8_t4": dict(kind="decode", batch=8, t=4, s_cap=131072, fp8=True,
                                    len_lo=65536, len_hi=131072, **GA),
    "mtp_decode_ga_fp8_rot_b8_t4": dict(kind="decode", batch=8, t=4, s_cap=131072, fp8=True,
                                        k_rotated=True, len_lo=65536, len_hi=131072, **GA),
    "swa_backward_1x32768": dict(kind="backward", seqlens=[32768], **SWA),
    "ga_backward_1x8192": dict(kind="backward", seqlens=[8192], **GA),
}


def algorithmic_pairs_prefill(seqlens, window: int) -> int:
    """Visible (query, key) pairs per query head: sum over sequences of
    L(L+1)/2 (global) or sum_p min(p+1, W) (window W)."""
    tot = 0
    for L in seqlens:
        if window <= 0 or window >= L:
            tot += L * (L + 1) // 2
        else:
            tot += window * (window + 1) // 2 + (L - window) * window
    return tot


def algorithmic_pairs_decode(seqlens, t: int, window: int) -> int:
    tot = 0
    for L in seqlens:
        for i in range(t):
            p = L - t + i
            if p < 0:
                continue
            lo = max(0, p - window + 1) if window > 0 else 0
            tot += p - lo + 1
    return tot
