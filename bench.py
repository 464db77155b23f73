"""Benchmark of the sink-bias GQA attention forward on B300.

Default (N = 1): the headline workload is SWA prefill, batch 4 x 32768 tokens,
64 query / 8 KV heads, window 128, RoPE base 1e4 (one SWA layer of the
MiMo-V2-Flash model at its 32K native context).  One step = one
sinkattn_prefill call over that batch.  The same JSON line also reports the
global-attention prefill (1 x 131072 tokens, 64/4 heads) and the MTP-verify
decode (batch 64, 4 query tokens, caches of 64K-256K tokens; GA and SWA layers),
each timed the same way.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference there is) on a
bounded sample of the same workload, on the host cores.
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: every rank
runs the whole workload on its own GPU; value = work of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sink-attn prefill TFLOP/s & decode KV GB/s on 1 B300; % of roofline"
MAIN = "swa_prefill_4x32768"
FLOP_PER_PAIR_HEAD = 2 * 192 + 2 * 128  # QK^T + PV per visible (query, key) pair and head


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--main-only", action="store_true", help="skip the GA prefill and decode lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=None,
                    help="time only this workload of synth.WORKLOADS (one line, no e2e, no "
                         "CPU baseline); used for the reduced profiler captures")
    return ap.parse_args()


# ------------------------------------------------------------------ environment
def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    """The largest of the ranks' values (the slowest rank's time)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of this
    process's GPU while the timed region runs: through NVML every 5 ms (pynvml,
    or the driver's NVML library by ctypes), else through `nvidia-smi -lms 50`
    in a subprocess."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._proc = None
        self.error = None
        self.source = None

    def _bus_id(self):
        import torch
        p = torch.cuda.get_device_properties(self.cuda_index)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"

    def _nvml(self):
        """(get_clock, get_reasons, max_clock) through pynvml if it imports, else
        through the driver's libnvidia-ml.so.1 by ctypes (same NVML calls)."""
        import torch
        uuid = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        try:
            import pynvml
            pynvml.nvmlInit()
            try:
                h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            except Exception:
                h = pynvml.nvmlDeviceGetHandleByPciBusId(self._bus_id())
            return (lambda: pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM),
                    lambda: pynvml.nvmlDeviceGetCurrentClocksEventReasons(h),
                    pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM), "nvml")
        except ImportError:
            pass
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0 and \
                nv.nvmlDeviceGetHandleByPciBusId_v2(self._bus_id().encode(), ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle for this GPU")
        sm = 1  # NVML_CLOCK_SM
        mx = ctypes.c_uint(0)
        nv.nvmlDeviceGetMaxClockInfo(h, sm, ctypes.byref(mx))
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons

        def clock():
            v = ctypes.c_uint(0)
            if nv.nvmlDeviceGetClockInfo(h, sm, ctypes.byref(v)) != 0:
                raise RuntimeError("nvmlDeviceGetClockInfo failed")
            return v.value

        def reasons():
            v = ctypes.c_ulonglong(0)
            if reasons_fn(h, ctypes.byref(v)) != 0:
                raise RuntimeError("clock event reasons query failed")
            return v.value

        return clock, reasons, mx.value, "nvml-ctypes"

    def _start_nvml(self):
        import threading
        clock, reasons, self.max_mhz, source = self._nvml()
        clock(), reasons()  # fail here, not in the sampling thread
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                try:
                    self.samples.append((clock(), reasons()))
                except Exception as e:
                    self.error = f"{type(e).__name__}: {e}"
                time.sleep(0.005)

        self._t = threading.Thread(target=loop, daemon=True)
        self._t.start()
        self.source = source

    def _start_smi(self):
        import subprocess
        import threading
        q = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"
        self._proc = subprocess.Popen(
            ["nvidia-smi", "-i", self._bus_id(), f"--query-gpu={q}",
             "--format=csv,noheader,nounits", "-lms", "50"],
            stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        first = threading.Event()

        def reader():
            for line in self._proc.stdout:
                parts = [x.strip() for x in line.split(",")]
                try:
                    mhz, mx, rs = float(parts[0]), float(parts[1]), int(parts[2], 16)
                except (ValueError, IndexError):
                    continue
                self.max_mhz = mx
                self.samples.append((mhz, rs))
                first.set()

        self._t = threading.Thread(target=reader, daemon=True)
        self._t.start()
        first.wait(timeout=5.0)
        self.source = "nvidia-smi"

    def __enter__(self):
        try:
            self._start_nvml()
        except Exception as e:
            self.error = f"nvml: {type(e).__name__}: {e}"
            try:
                self._start_smi()
            except Exception as e2:  # no sampler at all: the line says "unsampled" and why
                self.error += f"; nvidia-smi: {type(e2).__name__}: {e2}"
        return self

    def __exit__(self, *exc):
        if self._stop is not None:
            self._stop.set()
            self._t.join(timeout=2)
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
            self._t.join(timeout=2)
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0, "error": self.error}
        mhz = [s[0] for s in self.samples]
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items()
                          if r & bit})
        out = {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(mhz), "source": self.source}
        if self.source == "nvidia-smi" and self.error:
            out["nvml_error"] = self.error[:200]
        return out


# ------------------------------------------------------------------ workloads
def prefill_work(wl):
    from sliding_window_sink_bias_b300 import synth
    pairs = synth.algorithmic_pairs_prefill(wl["seqlens"], wl["window"])
    total = sum(wl["seqlens"])
    hq, hkv = wl["hq"], wl["hkv"]
    flops = pairs * hq * FLOP_PER_PAIR_HEAD
    bytes_ = total * (hq * 192 * 2 + hkv * 192 * 2 + hkv * 128 * 2 + hq * 128 * 2 + hq * 4)
    return flops, bytes_, total


def time_calls(fn, steps, warmup, ws):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(ws)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    ev[-1].synchronize()
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    barrier(ws)
    return max_over_ranks(total_ms, ws) / steps, per


def bench_prefill(name, steps, warmup, ws, local, with_e2e):
    import torch

    import sliding_window_sink_bias_b300 as sa
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[name]
    dev = f"cuda:{local}"
    inp = synth.prefill_inputs(wl["seqlens"], wl["hq"], wl["hkv"], window=wl["window"],
                               rope_base=wl["rope_base"], seed=0, device=dev)
    out = torch.empty(inp.total, wl["hq"], 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(inp.total, wl["hq"], dtype=torch.float32, device=dev)

    def call():
        sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, max_seqlen=inp.max_seqlen,
                   window=wl["window"], rope_base=wl["rope_base"], out=out, lse=lse,
                   scale=wl.get("scale"))

    with ClockSampler(local) as clk:
        ms, per = time_calls(call, steps, warmup, ws)
    st, word = sa.device_status()
    if st != sa.OK:
        raise RuntimeError(f"device status {st} word {word:#x} after {name}")
    flops, bytes_, total = prefill_work(wl)
    res = {"name": name, "ms": ms, "per_launch_ms": per, "flops": flops, "bytes": bytes_,
           "tokens": total, "clocks": clk.summary(), "launches": steps}
    if with_e2e:
        pin = lambda t: t.cpu().pin_memory()
        qh, kh, vh, sh, ch = pin(inp.q), pin(inp.k), pin(inp.v), pin(inp.sink), pin(inp.cu_seqlens)
        oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

        def e2e_call():
            inp.q.copy_(qh, non_blocking=True)
            inp.k.copy_(kh, non_blocking=True)
            inp.v.copy_(vh, non_blocking=True)
            inp.sink.copy_(sh, non_blocking=True)
            inp.cu_seqlens.copy_(ch, non_blocking=True)
            call()
            oh.copy_(out, non_blocking=True)
            lh.copy_(lse, non_blocking=True)

        e_ms, _ = time_calls(e2e_call, max(3, steps // 4), 1, ws)
        res["e2e_ms"] = e_ms
        res["h2d"] = sum(t.numel() * t.element_size() for t in (qh, kh, vh, sh, ch))
        res["d2h"] = sum(t.numel() * t.element_size() for t in (oh, lh))
        del qh, kh, vh, oh, lh
    del inp, out, lse
    torch.cuda.empty_cache()
    return res


def bench_hybrid(name, steps, warmup, ws, local):
    """One hybrid block (5 SWA layers, 1 GA layer) over a ragged batch: every
    step runs the six layer prefills back to back on the same stream."""
    import torch

    import sliding_window_sink_bias_b300 as sa
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[name]
    dev = f"cuda:{local}"
    lens = synth.log_uniform_lengths(wl["n_seq"], wl["len_lo"], wl["len_hi"], seed=0)
    hq = wl["hq"]
    swa = synth.prefill_inputs(lens, hq, wl["swa_hkv"], window=wl["window"],
                               rope_base=wl["swa_base"], seed=0, device=dev)
    ga = synth.prefill_inputs(lens, hq, wl["ga_hkv"], window=0, rope_base=wl["ga_base"], seed=1,
                              device=dev)
    n_layers = wl["swa_layers"] + wl["ga_layers"]
    sinks = [synth.sink_vector(hq, seed=10 + i, device=dev) for i in range(n_layers)]
    total = sum(lens)
    out = torch.empty(total, hq, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(total, hq, dtype=torch.float32, device=dev)

    def swa_layers():
        for i in range(wl["swa_layers"]):
            sa.prefill(swa.q, swa.k, swa.v, sinks[i], swa.cu_seqlens, max_seqlen=max(lens),
                       window=wl["window"], rope_base=wl["swa_base"], out=out, lse=lse)

    def ga_layers():
        for i in range(wl["ga_layers"]):
            sa.prefill(ga.q, ga.k, ga.v, sinks[wl["swa_layers"] + i], ga.cu_seqlens,
                       max_seqlen=max(lens), window=0, rope_base=wl["ga_base"], out=out, lse=lse)

    def call():
        swa_layers()
        ga_layers()

    # the SWA layers alone first, before any GA layer has run the GPU into its
    # power cap (the split below times them right after a GA layer)
    with ClockSampler(local) as clk_swa:
        swa_alone_ms, _ = time_calls(swa_layers, max(3, steps), warmup, ws)
    with ClockSampler(local) as clk:
        ms, _ = time_calls(call, steps, warmup, ws)
    # the split of one pass between the SWA layers and the GA layer (events
    # around each part on the launching stream, three passes averaged)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    swa_ms = ga_ms = 0.0
    for _ in range(3):
        ev[0].record()
        swa_layers()
        ev[1].record()
        ga_layers()
        ev[2].record()
        torch.cuda.synchronize()
        swa_ms += ev[0].elapsed_time(ev[1]) / (3 * wl["swa_layers"])
        ga_ms += ev[1].elapsed_time(ev[2]) / (3 * wl["ga_layers"])
    st, word = sa.device_status()
    if st != sa.OK:
        raise RuntimeError(f"device status {st} word {word:#x} after {name}")
    swa_pairs = synth.algorithmic_pairs_prefill(lens, wl["window"])
    ga_pairs = synth.algorithmic_pairs_prefill(lens, 0)
    flops = hq * FLOP_PER_PAIR_HEAD * (wl["swa_layers"] * swa_pairs + wl["ga_layers"] * ga_pairs)
    hkv = wl["swa_hkv"]
    per_layer = {"swa_ms": swa_ms, "ga_ms": ga_ms,
                 "swa_ms_alone": swa_alone_ms / wl["swa_layers"],
                 "swa_alone_clocks": clk_swa.summary(),
                 "swa_bytes": total * (hq * 192 * 2 + hkv * 192 * 2 + hkv * 128 * 2 + hq * 128 * 2
                                       + hq * 4),
                 "ga_flops": hq * FLOP_PER_PAIR_HEAD * ga_pairs}
    res = {"name": name, "ms": ms, "flops": flops, "tokens": total, "lens": lens,
           "clocks": clk.summary(), "launches": n_layers * steps, "per_layer": per_layer}
    del swa, ga, out, lse
    torch.cuda.empty_cache()
    return res


def per_layer_roofline(pl, peaks):
    """Time and roofline fraction of one SWA layer (HBM-bound) and one GA layer
    (tensor-bound) of a hybrid block pass."""
    swa_gbs = pl["swa_bytes"] / (pl["swa_ms"] / 1e3) / 1e9
    ga_tf = pl["ga_flops"] / (pl["ga_ms"] / 1e3) / 1e12
    out = {"swa_ms": pl["swa_ms"], "swa_gbs": swa_gbs, "swa_frac_hbm": swa_gbs / peaks["hbm_gbs"],
           "ga_ms": pl["ga_ms"], "ga_tflops": ga_tf, "ga_frac_tensor": ga_tf / peaks["bf16_tflops"]}
    if "swa_ms_alone" in pl:
        a_gbs = pl["swa_bytes"] / (pl["swa_ms_alone"] / 1e3) / 1e9
        out.update({"swa_ms_alone": pl["swa_ms_alone"], "swa_frac_hbm_alone": a_gbs / peaks["hbm_gbs"],
                    "swa_alone_sm_mhz": pl["swa_alone_clocks"].get("sm_mhz")})
    return out


def bench_ratio(name, warmup, ws, local):
    """Attention time of the hybrid design against all-global attention: one
    SWA layer and one GA layer timed on a single sequence per length; the
    block (5 SWA + 1 GA) and model (39 SWA + 9 GA) ratios are the all-GA time
    of the same layer count over the hybrid time.  The KV-cache ratio counts
    the keys a decode must keep: L per GA layer, the 128-key window per SWA
    layer."""
    import torch

    import sliding_window_sink_bias_b300 as sa
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[name]
    dev = f"cuda:{local}"
    hq = wl["hq"]
    (bs, bg), (ms_, mg) = wl["block"], wl["model"]
    rows = [{"seq_len": L} for L in wl["lens"]]
    # all SWA layers first: a GA layer leaves the GPU at its power cap for a while
    for tag, hkv, win, base in (("swa", wl["swa_hkv"], wl["window"], wl["swa_base"]),
                                ("ga", wl["ga_hkv"], 0, wl["ga_base"])):
        for res in rows:
            L = res["seq_len"]
            inp = synth.prefill_inputs([L], hq, hkv, window=win, rope_base=base, seed=0,
                                       device=dev)
            out = torch.empty(L, hq, 128, dtype=torch.bfloat16, device=dev)
            lse = torch.empty(L, hq, dtype=torch.float32, device=dev)

            def call():
                sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, max_seqlen=L,
                           window=win, rope_base=base, out=out, lse=lse)

            steps = 5 if (tag == "swa" or L <= 32768) else 2
            ms, _ = time_calls(call, steps, min(warmup, 2) if tag == "swa" else 1, ws)
            st, word = sa.device_status()
            if st != sa.OK:
                raise RuntimeError(f"device status {st} word {word:#x} after {name}")
            res[f"{tag}_ms"] = ms
            del inp, out, lse
            torch.cuda.empty_cache()
    for res in rows:
        L = res["seq_len"]
        s_, g_ = res["swa_ms"], res["ga_ms"]
        res["block_ratio"] = (bs + bg) * g_ / (bs * s_ + bg * g_)
        res["model_ratio"] = (ms_ + mg) * g_ / (ms_ * s_ + mg * g_)
        kv_ga, kv_swa = L * wl["ga_hkv"], min(L, wl["window"]) * wl["swa_hkv"]
        res["model_kv_ratio"] = (ms_ + mg) * kv_ga / (ms_ * kv_swa + mg * kv_ga)
    return rows


FLOP_PER_PAIR_HEAD_BWD = 2 * (3 * 192 + 2 * 128)  # S, dP, dV, dK, dQ per visible pair and head


def bench_backward(name, steps, warmup, ws, local):
    """sinkattn_prefill_backward on a workload: algorithmic FLOPs are the five
    products per visible (query, key) pair and head; algorithmic bytes read q,
    k, v, out, dout, lse once and write dq, dk, dv once."""
    import torch

    import sliding_window_sink_bias_b300 as sa
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[name]
    dev = f"cuda:{local}"
    hq, hkv, W, base = wl["hq"], wl["hkv"], wl["window"], wl["rope_base"]
    inp = synth.prefill_inputs(wl["seqlens"], hq, hkv, window=W, rope_base=base, seed=0,
                               device=dev)
    g = torch.Generator(device=dev).manual_seed(7)
    dout = torch.randn(inp.total, hq, 128, generator=g, device=dev).to(torch.bfloat16)
    out, lse = sa.prefill(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens,
                          max_seqlen=inp.max_seqlen, window=W, rope_base=base)
    work = torch.empty(sa.prefill_backward_workspace_size(inp.total, hq, hkv), dtype=torch.uint8,
                       device=dev)
    dq = torch.empty(inp.total, hq, 192, dtype=torch.bfloat16, device=dev)
    dk = torch.empty(inp.total, hkv, 192, dtype=torch.bfloat16, device=dev)
    dv = torch.empty(inp.total, hkv, 128, dtype=torch.bfloat16, device=dev)
    dsink = torch.empty(hq, dtype=torch.float32, device=dev)

    def call():
        sa.prefill_backward(inp.q, inp.k, inp.v, inp.sink, inp.cu_seqlens, out, lse, dout,
                            max_seqlen=inp.max_seqlen, window=W, rope_base=base, workspace=work,
                            dq=dq, dk=dk, dv=dv, dsink=dsink)

    with ClockSampler(local) as clk:
        ms, _ = time_calls(call, steps, warmup, ws)
    st, word = sa.device_status()
    if st != sa.OK:
        raise RuntimeError(f"device status {st} word {word:#x} after {name}")
    pairs = synth.algorithmic_pairs_prefill(wl["seqlens"], W)
    total = inp.total
    bytes_ = total * (hq * (192 + 128 + 128 + 192) * 2 + hq * 4 + hkv * (192 + 128) * 2 * 2)
    res = {"ms": ms, "flops": pairs * hq * FLOP_PER_PAIR_HEAD_BWD, "bytes": bytes_,
           "tokens": total, "clocks": clk.summary(), "launches": 4 * steps}
    del inp, out, lse, dout, work, dq, dk, dv
    torch.cuda.empty_cache()
    return res


def bench_decode(name, steps, warmup, ws, local):
    import torch

    import sliding_window_sink_bias_b300 as sa
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[name]
    dev = f"cuda:{local}"
    lens = synth.uniform_lengths(wl["batch"], wl["len_lo"], wl["len_hi"], seed=0)
    inp = synth.decode_inputs(lens, wl["t"], wl["s_cap"], wl["hq"], wl["hkv"],
                              window=wl["window"], rope_base=wl["rope_base"], seed=0, device=dev)
    fp8 = wl.get("fp8", False)
    if fp8:
        # E4M3 cache, one scale per KV head (largest magnitude -> 224)
        def quant(c):
            # sequence by sequence, so the fp32 temporaries stay small
            amax = torch.stack([c[b].abs().amax(dim=(0, 2)).float() for b in range(c.shape[0])])
            sc = (amax.amax(dim=0) / 224.0).clamp_min(1e-6)
            q8 = torch.empty(c.shape, dtype=torch.float8_e4m3fn, device=c.device)
            for b in range(c.shape[0]):
                q8[b] = (c[b].float() / sc[None, :, None]).to(torch.float8_e4m3fn)
            return q8, sc.float()
        k8, ks = quant(inp.kcache)
        inp.kcache = None
        v8, vs = quant(inp.vcache)
        inp.vcache = None
        torch.cuda.empty_cache()
    ws_bytes = sa.decode_workspace_size(wl["batch"], wl["t"], wl["hq"], wl["hkv"], max(lens),
                                        wl["window"])
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty(wl["batch"], wl["t"], wl["hq"], 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl["batch"], wl["t"], wl["hq"], dtype=torch.float32, device=dev)

    def call():
        if fp8:
            sa.decode_fp8(inp.q, k8, v8, ks, vs, inp.seqlens, inp.sink, max_seqlen=max(lens),
                          window=wl["window"], rope_base=wl["rope_base"], workspace=work, out=out,
                          lse=lse, k_rotated=wl.get("k_rotated", False))
        else:
            sa.decode(inp.q, inp.kcache, inp.vcache, inp.seqlens, inp.sink, max_seqlen=max(lens),
                      window=wl["window"], rope_base=wl["rope_base"], workspace=work, out=out,
                      lse=lse, kv_ring=wl.get("kv_ring", False),
                      k_rotated=wl.get("k_rotated", False))

    # the decode working set can sit in L2 for the SWA layer: flush between steps
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    import sliding_window_sink_bias_b300 as _sa  # noqa: F401
    times = []
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    barrier(ws)
    stream = torch.cuda.current_stream()
    # every step is enqueued without waiting for the previous one; a GPU sleep
    # ahead of the first step (outside the timed steps) lets the host enqueue
    # all of them before the GPU reaches them, so the host's per-call latency
    # never shows in a step's events
    with ClockSampler(local) as clk:
        torch.cuda._sleep(int(2e6) * max(20, steps))  # about 1 ms per step at 2 GHz
        evs = []
        for _ in range(steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            evs.append((e0, e1))
        evs[-1][1].synchronize()
        times = [a.elapsed_time(b) for a, b in evs]
    barrier(ws)
    ms = max_over_ranks(sum(times) / len(times), ws)
    st, word = sa.device_status()
    if st != sa.OK:
        raise RuntimeError(f"device status {st} word {word:#x} after {name}")
    hkv, t, hq, W = wl["hkv"], wl["t"], wl["hq"], wl["window"]
    keys = [min(L, t + W - 1) if W > 0 else L for L in lens]
    kv_bytes = sum(keys) * hkv * (192 + 128) * (1 if fp8 else 2)
    io_bytes = wl["batch"] * t * hq * (192 * 2 + 128 * 2 + 4)
    pairs = synth.algorithmic_pairs_decode(lens, t, W)
    res = {"name": name, "ms": ms, "kv_bytes": kv_bytes, "bytes": kv_bytes + io_bytes,
           "flops": pairs * hq * FLOP_PER_PAIR_HEAD, "clocks": clk.summary(),
           "launches": steps, "tokens": wl["batch"] * t, "vis_keys": sum(keys)}
    del inp, work, out, lse, flush
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ CPU oracle
def oracle_sample_prefill(wl, n_tokens, seed=0):
    """Run the oracle on the first n_tokens tokens of sequence 0 (every head);
    returns (seconds, flops, threads)."""
    import numpy as np

    import oracle
    from sliding_window_sink_bias_b300 import synth
    oracle.build()
    L = min(n_tokens, wl["seqlens"][0])
    inp = synth.prefill_inputs([L], wl["hq"], wl["hkv"], window=wl["window"],
                               rope_base=wl["rope_base"], seed=seed, device="cpu")
    t0 = time.perf_counter()
    oracle.prefill(inp.q, inp.k, inp.v, inp.sink, np.array([0, L], dtype=np.int32),
                   window=wl["window"], rope_base=wl["rope_base"])
    dt = time.perf_counter() - t0
    pairs = synth.algorithmic_pairs_prefill([L], wl["window"])
    return dt, pairs * wl["hq"] * FLOP_PER_PAIR_HEAD, oracle.max_threads()


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def cpu_baseline(target_s=12.0):
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[MAIN]
    dt, fl, thr = oracle_sample_prefill(wl, 256)
    n = int(min(32768, max(256, 256 * target_s / max(dt, 1e-3))))
    dt, fl, thr = oracle_sample_prefill(wl, n)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"first {n} tokens of sequence 0 of {MAIN}, all 64 heads "
                      f"({fl / 1e9:.1f} GFLOP, {dt:.1f} s)"}


def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[MAIN]
    n = 512
    for _ in range(args.warmup):
        oracle_sample_prefill(wl, n)
    times, flops = [], 0
    thr = 0
    for _ in range(args.steps):
        dt, fl, thr = oracle_sample_prefill(wl, n)
        times.append(dt)
        flops = fl
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": MAIN, "sample_tokens_per_step": n, "window": 128,
                   "heads": "64q/8kv", "head_dims": "192/128"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"first {n} tokens of sequence 0 of {MAIN}, all 64 heads, "
                                   "per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main
def single_workload(args, ws, rank, local, peaks):
    from sliding_window_sink_bias_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    if wl["kind"] == "backward":
        r = bench_backward(args.workload, args.steps, args.warmup, ws, local)
        tf = r["flops"] / (r["ms"] / 1e3) / 1e12
        gbs = r["bytes"] / (r["ms"] / 1e3) / 1e9
        line = {"workload": args.workload, "ms": r["ms"], "tflops": tf, "gbs": gbs,
                "frac_tensor": tf / peaks["bf16_tflops"], "frac_hbm": gbs / peaks["hbm_gbs"],
                "clocks": r["clocks"]}
    elif wl["kind"] == "ratio":
        line = {"workload": args.workload, "rows": bench_ratio(args.workload, args.warmup, ws, local)}
    elif wl["kind"] == "hybrid":
        r = bench_hybrid(args.workload, args.steps, args.warmup, ws, local)
        line = {"workload": args.workload, "ms": r["ms"], "tokens_per_s": r["tokens"] / (r["ms"] / 1e3),
                "tflops": r["flops"] / (r["ms"] / 1e3) / 1e12, "lens": r["lens"],
                "per_layer": per_layer_roofline(r["per_layer"], peaks), "clocks": r["clocks"]}
    elif wl["kind"] == "prefill":
        r = bench_prefill(args.workload, args.steps, args.warmup, ws, local, with_e2e=False)
        tf = r["flops"] / (r["ms"] / 1e3) / 1e12
        gbs = r["bytes"] / (r["ms"] / 1e3) / 1e9
        line = {"workload": args.workload, "ms": r["ms"], "tflops": tf, "gbs": gbs,
                "frac_tensor": tf / peaks["bf16_tflops"], "frac_hbm": gbs / peaks["hbm_gbs"],
                "clocks": r["clocks"]}
    else:
        r = bench_decode(args.workload, args.steps, args.warmup, ws, local)
        gbs = r["bytes"] / (r["ms"] / 1e3) / 1e9
        line = {"workload": args.workload, "ms": r["ms"], "gbs": gbs,
                "frac_hbm": gbs / peaks["hbm_gbs"], "clocks": r["clocks"]}
    if rank == 0:
        print(json.dumps(line), flush=True)


# DRAM bytes per launch measured by ncu (profiles/dram_traffic.json), keyed by
# kernel; each entry holds the sha256 of the kernel sources it was measured on
# and is ignored (traffic null) once those sources change.
KERNEL_SOURCES = {
    "band": ["band_kernel.cuh", "common.cuh", "ptx.cuh"],
    "causal": ["causal_kernel.cuh", "common.cuh", "ptx.cuh"],
    "decode": ["decode_kernel.cuh", "common.cuh", "ptx.cuh"],
}


def kernel_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sliding_window_sink_bias_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_for(key, tokens):
    """DRAM bytes of one launch of the benchmarked workload, or None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        tab = json.load(f)
    e = tab.get(key)
    if not e or e.get("sha256") != kernel_hash(e["kernel"]):
        return None
    b = e["dram_bytes_per_launch"]
    if tokens and e.get("tokens"):  # measured on a smaller case: scale by the units processed
        b = b * tokens / e["tokens"]
    return b


def roofline_obj(bound, achieved, peak, unit, traffic=None):
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak if peak else None, "traffic": traffic}


def _r(x, n=4):
    return None if x is None else round(float(x), n)


def summary_of(line):
    """One compact entry per workload (time per step, value, roofline fraction,
    median SM clock), placed last on the line so that a reader keeping only the
    end of the output still has every workload's numbers."""
    def entry(ms, value, unit, roof, clocks):
        e = {"ms": _r(ms, 4), "value": _r(value, 1), "unit": unit}
        if roof:
            e["frac"] = _r(roof.get("frac"), 4)
            e["bound"] = roof.get("bound")
        if clocks:
            e["sm_mhz"] = clocks.get("sm_mhz")
            e["clk_samples"] = clocks.get("samples")
        return e
    out = {line["config"]["workload"]: entry(line["ms_per_step"], line["value"], line["unit"],
                                             line.get("roofline"), line.get("clocks"))}
    for name, w in line.get("other_workloads", {}).items():
        if name == "hybrid_vs_all_ga":
            out[name] = {f"{r['seq_len']}": _r(r["block_ratio"], 3) for r in w["rows"]}
            continue
        e = entry(w.get("ms_per_step"), w.get("value"), w.get("unit"), w.get("roofline"),
                  w.get("clocks"))
        if "per_layer" in w:
            pl = w["per_layer"]
            e["swa_frac_hbm"] = _r(pl["swa_frac_hbm"])
            e["swa_frac_hbm_alone"] = _r(pl.get("swa_frac_hbm_alone"))
            e["ga_frac_tensor"] = _r(pl["ga_frac_tensor"])
        out[name] = e
    return out


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    ws, rank, local = dist_setup()
    from sliding_window_sink_bias_b300 import build
    if rank == 0:
        build.build()
    barrier(ws)
    peaks = load_peaks()
    if args.workload:
        single_workload(args, ws, rank, local, peaks)
        return
    m = bench_prefill(MAIN, args.steps, args.warmup, ws, local, with_e2e=True)
    tflops = ws * m["flops"] / (m["ms"] / 1e3) / 1e12
    gbs = m["bytes"] / (m["ms"] / 1e3) / 1e9  # per GPU, per launch (one launch per step)
    e2e_tflops = ws * m["flops"] / (m["e2e_ms"] / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": MAIN, "batch": 4, "seq_len": 32768, "heads": "64q/8kv",
                   "head_dims": "192/128", "window": 128, "rope_base": 1e4,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2 (6.07 GB per step), no flush"},
        "tokens_per_s": ws * m["tokens"] / (m["ms"] / 1e3),
        "roofline": roofline_obj("hbm", gbs, peaks["hbm_gbs"], "GB/s",
                                 traffic_for("band", m["tokens"])),
        "peaks_source": peaks["source"],
        "e2e": {"value": e2e_tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": m["d2h"], "ms_per_step": m["e2e_ms"]},
        "gpu_launches": m["launches"],
        "clocks": m["clocks"],
    }
    if not args.main_only:
        # the short workloads first, before the long GA runs bring the GPU to its
        # power limit (each line records the clocks it ran at)
        extra = {}
        w = bench_prefill("swa_w512_prefill_1x32768", args.steps, args.warmup, ws, local,
                          with_e2e=False)
        w_tf = w["flops"] / (w["ms"] / 1e3) / 1e12
        extra["swa_w512_prefill_1x32768"] = {
            "value": ws * w_tf, "unit": "TFLOP/s", "ms_per_step": w["ms"],
            "kernel": "causal prefill kernel with a window (512 > 128)",
            "roofline": roofline_obj("tensor", w_tf, peaks["bf16_tflops"], "TFLOP/s", None),
            "clocks": w["clocks"]}
        w = bench_prefill("swa_g2_prefill_1x32768", args.steps, args.warmup, ws, local,
                          with_e2e=False)
        w_tf = w["flops"] / (w["ms"] / 1e3) / 1e12
        w_gbs = w["bytes"] / (w["ms"] / 1e3) / 1e9
        extra["swa_g2_prefill_1x32768"] = {
            "value": ws * w_tf, "unit": "TFLOP/s", "ms_per_step": w["ms"],
            "kernel": "causal prefill kernel (2 query heads per KV head, W = 128)",
            "gbs": w_gbs,
            "roofline": roofline_obj("hbm", w_gbs, peaks["hbm_gbs"], "GB/s",
                                     traffic_for("causal_swa_g2_prefill_1x32768", w["tokens"])),
            "clocks": w["clocks"]}
        for name in ("mtp_decode_ga_b64_t4", "mtp_decode_ga_fp8_b64_t4",
                     "mtp_decode_ga_fp8_rot_b64_t4", "mtp_decode_swa_b64_t4",
                     "mtp_decode_swa_ring_b64_t4"):
            d = bench_decode(name, args.steps, args.warmup, ws, local)
            d_gbs = d["bytes"] / (d["ms"] / 1e3) / 1e9
            extra[name] = {"value": ws * d_gbs, "unit": "GB/s", "ms_per_step": d["ms"],
                           "kv_bytes": d["kv_bytes"],
                           "tflops": d["flops"] / (d["ms"] / 1e3) / 1e12,
                           "roofline": roofline_obj("hbm", d_gbs, peaks["hbm_gbs"], "GB/s",
                                                    traffic_for("decode_" + name, d["vis_keys"])),
                           "clocks": d["clocks"], "l2": "256 MB flush between steps"}
        r = bench_backward("swa_backward_4x32768", max(3, args.steps // 4), args.warmup, ws, local)
        tf = r["flops"] / (r["ms"] / 1e3) / 1e12
        gbs = r["bytes"] / (r["ms"] / 1e3) / 1e9
        extra["swa_backward_4x32768"] = {
            "value": ws * tf, "unit": "TFLOP/s", "ms_per_step": r["ms"], "gbs": gbs,
            "roofline": roofline_obj("hbm", gbs, peaks["hbm_gbs"], "GB/s", None),
            "clocks": r["clocks"], "outputs": "dq, dk, dv, dsink for sum(dout * out)"}
        g = bench_prefill("ga_prefill_1x131072", max(3, args.steps // 4), args.warmup, ws, local,
                          with_e2e=False)
        g_tf = g["flops"] / (g["ms"] / 1e3) / 1e12
        extra["ga_prefill_1x131072"] = {
            "value": ws * g_tf, "unit": "TFLOP/s", "ms_per_step": g["ms"],
            "roofline": roofline_obj("tensor", g_tf, peaks["bf16_tflops"], "TFLOP/s",
                                     traffic_for("causal", g["tokens"])),
            "frac_of_sustained_peak": (g_tf / peaks["bf16_tflops_sustained"]
                                       if peaks.get("bf16_tflops_sustained") else None),
            "clocks": g["clocks"]}
        h = bench_hybrid("hybrid_block_ragged_8seq", max(3, args.steps // 4), args.warmup, ws,
                         local)
        extra["hybrid_block_ragged_8seq"] = {
            "value": ws * h["tokens"] / (h["ms"] / 1e3), "unit": "tokens/s",
            "ms_per_step": h["ms"], "tflops": h["flops"] / (h["ms"] / 1e3) / 1e12,
            "seq_lens": h["lens"], "layers": "5 SWA (64/8, W=128) + 1 GA (64/4)",
            "per_layer": per_layer_roofline(h["per_layer"], peaks), "clocks": h["clocks"]}
        for name, bound in (("ga_backward_1x32768", "tensor"),):
            r = bench_backward(name, max(3, args.steps // 4), args.warmup, ws, local)
            tf = r["flops"] / (r["ms"] / 1e3) / 1e12
            gbs = r["bytes"] / (r["ms"] / 1e3) / 1e9
            roof = (roofline_obj("hbm", gbs, peaks["hbm_gbs"], "GB/s", None) if bound == "hbm"
                    else roofline_obj("tensor", tf, peaks["bf16_tflops"], "TFLOP/s", None))
            extra[name] = {"value": ws * tf, "unit": "TFLOP/s", "ms_per_step": r["ms"],
                           "gbs": gbs, "roofline": roof, "clocks": r["clocks"],
                           "outputs": "dq, dk, dv, dsink for sum(dout * out)"}
        extra["hybrid_vs_all_ga"] = {
            "rows": bench_ratio("hybrid_vs_all_ga", args.warmup, ws, local),
            "note": "ratio = all-GA attention time / hybrid attention time for the same layer "
                    "count; block = 5 SWA + 1 GA, model = 39 SWA + 9 GA; the pages claim "
                    "nearly 6x (context, not a target)"}
        line["other_workloads"] = extra
    if ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    line["summary"] = summary_of(line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
