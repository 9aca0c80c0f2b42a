#!/usr/bin/env python3
"""Benchmark of the Direct-P FP4 attention forward on GB300.

One step = the whole hot path on one batch of synthetic input already resident
in HBM: NVFP4-quantize Q and K, MXFP4-quantize V, and the Direct-P forward.
value = 4*B*H*N^2*D attention FLOPs per step / step time (TFLOP/s), summed
over ranks (each rank runs its own replica of the workload: weak scaling).

Default workload: B=1, H=40, N=32768, D=128 (video-DiT shape, token RMS
spread), the largest configuration and the one the throughput target is
quoted on.  Its inputs (1 GB bf16, 0.28 GB quantized) exceed the 129 MB L2, so
no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload I] [--causal] [--fp8pv] [--bwd]
                  [--no-variants] [--no-cpu-baseline]

"e2e" repeats the K steps from pinned host memory through the C ABI's
host-buffer call (fp4attn_fwd_host_batch): every step's upload of Q, K, V
and download of O and LSE run inside the timed region, pipelined across
steps.  --bwd prints the causal backward's line alone (FP8 operand
quantizers, prep pass and the two backward kernels per step).

--impl reference times the CPU oracle (the plain C restatement used by the
tests) on a bounded sample of the same workload; it is a reported baseline.
--causal times the causal forward instead (query i sees keys 0..i); its
FLOPs are counted over the unmasked (query, key) pairs, 4*D*N*(N+1)/2 per head.
--fp8pv times the FP8 P/V variant (MXFP8 V, E4M3 probability codes).

The roofline peak is measured on the same GPU before the timed region: a loop
of the block-scaled tcgen05 products the forward issues (QK^T: E2M1 with
16-element UE4M3 scales; PV: E2M1 with 32-element UE8M0 scales, or E4M3 for
the FP8 P/V variant), one CTA per SM (fp4attn_debug_mma_peak).  The forward
spends half its FLOPs in each product, so its peak is the FLOP-weighted
harmonic combination of the two rates.  The default run also times the
forward of the D=64 workload and the causal and FP8 P/V forwards on the
default workload and the causal backward, reported in "variants" of the
same JSON line (--no-variants skips them; --no-cpu-baseline skips the timed
oracle sample).

  python bench.py --mma-peak   prints the measured peaks and the clocks seen
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Direct-P FP4 attn fwd TFLOP/s (4BHN²D/t), % of GB300 dense FP4 peak"
METRIC_CAUSAL = "Causal Direct-P FP4 attn fwd TFLOP/s (4BHD·N(N+1)/2 / t), % of GB300 dense FP4 peak"


def metric_name(args):
    m = METRIC_CAUSAL if args.causal else METRIC
    return m.replace("FP4 attn", "FP4-QK/FP8-PV attn") if args.fp8pv else m
UNIT = "TFLOP/s"
# Context only (the roofline uses the measured block-scaled rates): nominal
# dense FP4 : BF16 = 13.5 : 2.25 PFLOP/s, FP8 : BF16 = 4.5 : 2.25.
FP4_OVER_BF16 = 13.5 / 2.25
FP8PV_OVER_BF16 = 1.0 / (0.5 / FP4_OVER_BF16 + 0.5 / (4.5 / 2.25))
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic of one forward launch, from an ncu capture (see profiles/), and
# the hash of the kernel sources it was taken on; reported only while the
# sources are unchanged.
TRAFFIC_RECORD = {"sources_sha": "9bfce670efca4f95", "shape": (1, 40, 32768, 128),
                  "bytes_per_launch": 278259968 + 291760896,
                  "note": "dram__bytes_read.sum + dram__bytes_write.sum of one launch on the 40-head "
                          "N=32768 D=128 workload (ncu capture of the same kernel sources)"}
TRAFFIC_RECORD_CAUSAL = {"sources_sha": TRAFFIC_RECORD["sources_sha"], "shape": TRAFFIC_RECORD["shape"],
                         "bytes_per_launch": 278377216 + 293730304,
                         "note": "the same capture of the causal forward"}
KERNEL_SOURCES = ["blackwell_nvfp4_quantize_gb300/csrc/fwd_directp.cu", "blackwell_nvfp4_quantize_gb300/csrc/ptx.cuh",
                  "blackwell_nvfp4_quantize_gb300/csrc/fp8.cuh"]


def sources_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling over the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def measure_mma_peaks(iters=1 << 20, launches=3, rounds=3):
    """Dense TFLOP/s of the block-scaled products the forward issues, best of
    `rounds` timings of `launches` launches each (CUDA events)."""
    import blackwell_nvfp4_quantize_gb300 as fa

    out = {}
    for kind in ("nvf4", "mxf4", "mxf8"):
        fa.debug_mma_peak(kind, iters=1 << 14, launches=1)  # warm-up
        out[kind] = max(fa.debug_mma_peak(kind, iters=iters, launches=launches) for _ in range(rounds))
    if fa.device_status() != fa.FP4ATTN_OK:
        raise RuntimeError("a bounded wait timed out in the MMA peak loop")
    return out


def forward_peak(peaks, fp8pv):
    """The forward spends half of its FLOPs in QK^T and half in PV, one after
    the other: its peak is the harmonic combination of the two rates."""
    pv = peaks["mxf8"] if fp8pv else peaks["mxf4"]
    return 1.0 / (0.5 / peaks["nvf4"] + 0.5 / pv)


def attn_flops(rows, N, D, causal):
    """4*D per (query, key) pair the rows attend to: N keys each, or i+1 for row i (causal)."""
    import numpy as np

    rows = np.asarray(rows, dtype=np.int64)
    keys = (rows % N + 1).sum() if causal else rows.size * N
    return 4.0 * D * float(keys)


def max_over_ranks(values, dist=None, device=None):
    """Each timing (ms) maximised over the ranks of the process group (the
    slowest replica sets the whole job's time); the values as they are for one
    process."""
    if dist is None:
        return [float(x) for x in values]
    import torch

    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_tflops(world, flops_per_replica, ms):
    """Throughput of the whole job: every rank runs one replica of the workload."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


def cpu_baseline(w, q, k, v, causal=False, fp8pv=False, budget_s=16.0):
    """The oracle as it stands, on host cores, on a bounded row sample of head 0."""
    import numpy as np

    import oracle
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    threads = oracle.default_threads()
    B, H, N, D = w.shape
    head = slice(0, 1)
    qb = wl.bf16_bits(q[:1, head].contiguous())
    kb = wl.bf16_bits(k[:1, head].contiguous())
    vb = wl.bf16_bits(v[:1, head].contiguous())
    shape1 = (1, 1, N, D)
    t0 = time.perf_counter()
    qq = oracle.quant_nvfp4(qb, threads)
    kq = oracle.quant_nvfp4(kb, threads)
    vq = oracle.quant_mxfp8_v(vb, threads) if fp8pv else oracle.quant_mxfp4_v(vb, threads)
    pv_fmt = oracle.PV_MXFP8 if fp8pv else oracle.PV_MXFP4
    t_quant = time.perf_counter() - t0
    # calibrate in two stages (a tiny probe overstates the per-row cost: the
    # thread pool's start-up dominates it), then time a sample sized to the budget
    def timed_rows(n):
        r = np.linspace(0, N - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        oracle.directp_rows(qq, kq, vq, shape1, w.softmax_scale, r, threads, causal=causal, pv_fmt=pv_fmt)
        return time.perf_counter() - t0

    n1 = min(N, 2 * threads)
    t1 = timed_rows(n1)
    n2 = int(max(n1, min(N, n1 * 1.5 / max(t1, 1e-6))))
    t2 = timed_rows(n2) if n2 > n1 else t1
    rows = int(max(n2, min(N, n2 * budget_s / max(t2, 1e-6))))
    sample = np.linspace(0, N - 1, rows).astype(np.int64)
    t0 = time.perf_counter()
    oracle.directp_rows(qq, kq, vq, shape1, w.softmax_scale, sample, threads, causal=causal, pv_fmt=pv_fmt)
    t = time.perf_counter() - t0
    flops = attn_flops(sample, N, D, causal)
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d of %d query rows of head 0 of %s (attention rows only; the oracle's quantization "
                      "of that head took %.1f s and is excluded), %.1f s" % (rows, N, w.name, t_quant, t)}


def run_reference(args, w):
    """--impl reference: the CPU oracle on a bounded sample, per step."""
    import numpy as np

    import oracle
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    q, k, v = wl.make_inputs(w)
    threads = oracle.default_threads()
    B, H, N, D = w.shape
    qb, kb, vb = (wl.bf16_bits(t[:1, :1].contiguous()) for t in (q, k, v))
    shape1 = (1, 1, N, D)
    qq, kq = oracle.quant_nvfp4(qb, threads), oracle.quant_nvfp4(kb, threads)
    vq = oracle.quant_mxfp8_v(vb, threads) if args.fp8pv else oracle.quant_mxfp4_v(vb, threads)
    pv_fmt = oracle.PV_MXFP8 if args.fp8pv else oracle.PV_MXFP4
    causal = args.causal
    rows_per_step = max(threads, 2 * threads)
    probe = np.linspace(0, N - 1, rows_per_step).astype(np.int64)
    t0 = time.perf_counter()
    oracle.directp_rows(qq, kq, vq, shape1, w.softmax_scale, probe, threads, causal=causal, pv_fmt=pv_fmt)
    t_probe = time.perf_counter() - t0
    per_step_budget = max(0.5, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    rows_per_step = int(max(threads, min(N, rows_per_step * per_step_budget / max(t_probe, 1e-6))))
    rng = np.random.default_rng(0)
    times = []
    flops = 0.0
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(N, size=rows_per_step, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.directp_rows(qq, kq, vq, shape1, w.softmax_scale, rows, threads, causal=causal, pv_fmt=pv_fmt)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            flops += attn_flops(rows, N, D, causal)
    t = sum(times)
    value = flops / t / 1e12
    sample = "%d query rows per step of head 0 of %s (attention rows; quantization excluded)" % (rows_per_step, w.name)
    line = {"metric": metric_name(args), "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "recipe": w.description,
                       "mask": "causal" if causal else "none", "pv": "fp8" if args.fp8pv else "fp4"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_variant(w, causal, fp8pv, mma_peaks, dev, local, steps=10, warmup=3):
    """Forward-only timing of one more configuration (CUDA events around each
    launch, inputs resident in HBM, no flush: every variant's inputs exceed
    the L2), with its own roofline and clocks."""
    import torch

    import blackwell_nvfp4_quantize_gb300 as fa
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    B, H, N, D = w.shape
    stream = torch.cuda.current_stream()
    q, k, v = (t.to(dev) for t in wl.make_inputs(w))
    qq, kq = fa.quant_qk_nvfp4(q, stream=stream), fa.quant_qk_nvfp4(k, stream=stream)
    vq = fa.quant_v_mxfp8(v, stream=stream) if fp8pv else fa.quant_v_mxfp4(v, stream=stream)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    del q, k, v

    def fwd():
        if fp8pv:
            fa.fwd_directp_fp8pv(qq, kq, vq, w.softmax_scale, causal=causal, o=o, lse=lse, stream=stream)
        else:
            (fa.fwd_directp_causal if causal else fa.fwd_directp)(qq, kq, vq, w.softmax_scale, o=o, lse=lse,
                                                                 stream=stream)

    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    times = []
    with ClockSampler(local) as clocks:
        for _ in range(steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fwd()
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
    if fa.device_status() != fa.FP4ATTN_OK:
        raise RuntimeError("device-side wait timed out in a variant")
    ms = sum(a.elapsed_time(b) for a, b in times) / steps
    flops = B * H * attn_flops(range(N), N, D, causal)
    achieved = flops / (ms * 1e-3) / 1e12
    peak = forward_peak(mma_peaks, fp8pv)
    del qq, kq, vq, o, lse
    torch.cuda.empty_cache()
    return {"workload": w.name, "B": B, "H": H, "N": N, "D": D, "mask": "causal" if causal else "none",
            "pv": "fp8" if fp8pv else "fp4", "steps": steps, "warmup": warmup, "fwd_ms": ms,
            "metric": "forward TFLOP/s (%s)" % ("4*D per unmasked (query, key) pair" if causal else "4BHN^2D/t"),
            "value": achieved,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "peak_source": "measured block-scaled MMA loop, FLOP-weighted (see the main line)"},
            "clocks": clocks.summary()}


def backward_peak(peaks):
    """The backward's five products: S on FP4 (kind::mxf4nvf4), dP, dV, dK, dQ
    on FP8 (kind::mxf8f6f4), equal FLOPs each: the harmonic combination."""
    return 1.0 / (0.2 / peaks["nvf4"] + 0.8 / peaks["mxf8"])


def time_backward(w, mma_peaks, dev, local, steps=5, warmup=3):
    """The causal backward at workload w: the training forward (quantize Q, K,
    V; causal Direct-P; its O, LSE and saved NVFP4 Q/K) once, outside the
    timed region, then per step the FP8 operand quantizers (E4M3 V rows,
    E5M2 dO rows and dO^T, E4M3 Q^T, K^T), the prep pass and the two
    backward kernels, with CUDA events around each step and around the
    kernels.  Inputs exceed the L2 (no flush)."""
    import torch

    import blackwell_nvfp4_quantize_gb300 as fa
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    B, H, N, D = w.shape
    stream = torch.cuda.current_stream()
    q, k, v = (t.to(dev) for t in wl.make_inputs(w))
    g = torch.Generator().manual_seed(5000 + w.index)
    dout = torch.randn((B, H, N, D), generator=g).to(torch.bfloat16).to(dev)
    o, lse, q_saved, k_saved, _ = fa.fwd_directp_causal_save(q, k, v, w.softmax_scale, stream=stream)
    bufs = {"v_rows": fa.empty_fp8(w.shape, "rows", fa.FP8_E4M3, dev),
            "do_rows": fa.empty_fp8(w.shape, "rows", fa.FP8_E5M2, dev),
            "do_t": fa.empty_fp8(w.shape, "t", fa.FP8_E5M2, dev),
            "q_t": fa.empty_fp8(w.shape, "t", fa.FP8_E4M3, dev),
            "k_t": fa.empty_fp8(w.shape, "t", fa.FP8_E4M3, dev)}
    npad = (N + 127) // 128 * 128
    nl2 = torch.empty((B, H, npad), dtype=torch.float32, device=dev)
    delta = torch.empty_like(nl2)
    grads = [torch.empty((B, H, N, D), dtype=torch.float32, device=dev) for _ in range(3)]

    def step(ev=None):
        fa.quant_mxfp8_rows(v, fa.FP8_E4M3, bufs["v_rows"], stream=stream)
        fa.quant_mxfp8_rows(dout, fa.FP8_E5M2, bufs["do_rows"], stream=stream)
        fa.quant_mxfp8_t(dout, fa.FP8_E5M2, bufs["do_t"], stream=stream)
        fa.quant_mxfp8_t(q, fa.FP8_E4M3, bufs["q_t"], stream=stream)
        fa.quant_mxfp8_t(k, fa.FP8_E4M3, bufs["k_t"], stream=stream)
        fa.bwd_prep(o, dout, lse, nl2, delta, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        fa.bwd_directp_causal(q_saved, k_saved, bufs["v_rows"], bufs["do_rows"], bufs["do_t"], bufs["q_t"],
                              bufs["k_t"], nl2, delta, w.softmax_scale, *grads, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    rec = []
    with ClockSampler(local) as clocks:
        for _ in range(steps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            ev[2].record(stream)
            step(ev)
            ev[3].record(stream)
            rec.append(ev)
        torch.cuda.synchronize()
    if fa.device_status() != fa.FP4ATTN_OK:
        raise RuntimeError("device-side wait timed out in the backward")
    step_ms = sum(e[2].elapsed_time(e[3]) for e in rec) / steps
    kern_ms = sum(e[0].elapsed_time(e[1]) for e in rec) / steps
    flops = 2.5 * B * H * attn_flops(range(N), N, D, True)  # 10*D per unmasked (query, key) pair
    achieved = flops / (kern_ms * 1e-3) / 1e12
    peak = backward_peak(mma_peaks)
    del q, k, v, dout, o, lse, q_saved, k_saved, bufs, nl2, delta, grads
    torch.cuda.empty_cache()
    return {"workload": w.name, "B": B, "H": H, "N": N, "D": D, "mask": "causal", "pass": "backward",
            "steps": steps, "warmup": warmup,
            "metric": "causal backward TFLOP/s (10*D per unmasked (query, key) pair: S, dP, dV, dK, dQ)",
            "value": flops / (step_ms * 1e-3) / 1e12, "step_ms": step_ms, "bwd_kernels_ms": kern_ms,
            "step": "E4M3 V rows, E5M2 dO rows and dO^T, E4M3 Q^T and K^T quantizers, prep (Delta, log2 LSE), "
                    "key-stationary dK/dV kernel, query-stationary dQ kernel",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "kernels": "bwd_kernel<%d, KV=true> + bwd_kernel<%d, KV=false>" % (D, D),
                         "peak_source": "measured block-scaled MMA loop: 1/5 of the FLOPs on kind::mxf4nvf4 "
                                        "(S), 4/5 on kind::mxf8f6f4 (dP, dV, dK, dQ), harmonic combination; "
                                        "S and dP are computed twice (once per kernel) but counted once"},
            "gpu_launches_per_step": 8,
            "clocks": clocks.summary()}


def run_mma_peak(args):
    """--mma-peak: the block-scaled tensor rates of this GPU and the clocks they ran at."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    with ClockSampler(dev.index) as clocks:
        peaks = measure_mma_peaks(iters=1 << 21, launches=5, rounds=5)
    line = {"mma_peak_tflops": peaks, "forward_peak_fp4": forward_peak(peaks, False),
            "forward_peak_fp8pv": forward_peak(peaks, True), "clocks": clocks.summary(),
            "shape": "M=128, N=128, K=128 per round (two K=64 E2M1 or four K=32 E4M3 products), one CTA per SM"}
    print(json.dumps(line), flush=True)
    return 0


def run_bwd(args, w):
    """--bwd: the causal backward line alone (measured peaks, then time_backward)."""
    import torch

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    with ClockSampler(dev.index) as clocks:
        peaks = measure_mma_peaks()
    line = time_backward(w, peaks, dev, dev.index, steps=args.steps, warmup=args.warmup)
    line["peak_clocks"] = clocks.summary()
    line["mma_peak_tflops"] = peaks
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch

    import blackwell_nvfp4_quantize_gb300 as fa
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    B, H, N, D = w.shape

    q_h, k_h, v_h = wl.make_inputs(w, seed=w.seed + rank)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    qq, kq = fa.empty_nvfp4(w.shape, dev), fa.empty_nvfp4(w.shape, dev)
    vq = fa.empty_mxfp8(w.shape, dev) if args.fp8pv else fa.empty_mxfp4(w.shape, dev)
    quant_v = fa.quant_v_mxfp8 if args.fp8pv else fa.quant_v_mxfp4
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    quant_bytes = sum(t.numel() * t.element_size() for t in (qq.payload, qq.sf, kq.payload, kq.sf, vq.payload_t, vq.sf))
    launches_per_step = 3 + 3 + 1 + 1  # amax, quant, finalize (x2), V quant, forward
    if args.fp8pv:
        def fwd(qq, kq, vq, scale, o, lse, stream):
            return fa.fwd_directp_fp8pv(qq, kq, vq, scale, causal=args.causal, o=o, lse=lse, stream=stream)
    else:
        fwd = fa.fwd_directp_causal if args.causal else fa.fwd_directp

    fwd_events = []

    def step(record=False):
        fa.quant_qk_nvfp4(q, out=qq, stream=stream)
        fa.quant_qk_nvfp4(k, out=kq, stream=stream)
        quant_v(v, out=vq, stream=stream)
        if record:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fwd(qq, kq, vq, w.softmax_scale, o=o, lse=lse, stream=stream)
            e1.record(stream)
            fwd_events.append((e0, e1))
        else:
            fwd(qq, kq, vq, w.softmax_scale, o=o, lse=lse, stream=stream)

    # roofline denominator: the block-scaled tensor rates of this GPU, measured
    # now (about half a second), with the clocks they ran at
    with ClockSampler(local) as peak_clocks:
        mma_peaks = measure_mma_peaks()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.device_status() != fa.FP4ATTN_OK:
        raise RuntimeError("device-side wait timed out during warm-up")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # Inputs larger than L2 need no flush between steps; otherwise each step
    # is timed by its own events and a write of twice the L2 size between
    # steps (outside those events) evicts the previous step's data.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    in_bytes = 3 * B * H * N * D * 2
    flush = None if in_bytes > l2_bytes else torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
    step_events = []
    with ClockSampler(local) as clocks:
        barrier()
        t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for _ in range(args.steps):
            if flush is None:
                step(record=True)
            else:
                flush.zero_()
                s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(stream)
                step(record=True)
                s1.record(stream)
                step_events.append((s0, s1))
        t_stop.record(stream)
        barrier()
    if flush is None:
        ms_total = t_start.elapsed_time(t_stop)
    else:
        ms_total = sum(a.elapsed_time(b) for a, b in step_events)
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_events]
    if fa.device_status() != fa.FP4ATTN_OK:
        raise RuntimeError("device-side wait timed out in the timed region")

    # End to end through the C ABI with host buffers (pinned): one
    # fp4attn_fwd_host_batch call runs the K steps, each uploading its Q, K, V
    # and downloading its O and LSE inside the timed region.  The call
    # pipelines them the way a serving loop runs them back to back: step i+1's
    # upload and step i-1's download overlap step i's kernels (its own upload
    # and download streams beside the compute stream, two device slots).
    q_p, k_p, v_p = (t.pin_memory() for t in (q_h, k_h, v_h))
    o_p = [torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_p = [torch.empty((B, H, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    ws = fa.empty_host_batch_workspace((B, H, N, D), dev, causal=args.causal, fp8pv=args.fp8pv)

    def e2e_run(nsteps):
        fa.fwd_host_batch([q_p] * nsteps, [k_p] * nsteps, [v_p] * nsteps, [o_p[i % 2] for i in range(nsteps)],
                          [lse_p[i % 2] for i in range(nsteps)], w.softmax_scale, causal=args.causal,
                          fp8pv=args.fp8pv, workspace=ws, stream=stream)

    e2e_steps = max(4, args.steps)  # the same K steps as the device-timed region, fill and drain included
    e2e_run(2)
    barrier()
    # the host link as this run sees it (the GPU's neighbours on the machine
    # share its host memory): one pinned upload and one download of Q's bytes
    link = {}
    for name, dst, src in (("h2d", q, q_p), ("d2h", q_p, q)):
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        dst.copy_(src, non_blocking=True)
        l1.record(stream)
        l1.synchronize()
        link[name] = round(q.numel() * 2 / (l0.elapsed_time(l1) * 1e-3) / 1e9, 1)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if fa.device_status() != fa.FP4ATTN_OK:
        raise RuntimeError("device-side wait timed out in the end-to-end leg")

    ms_total, e2e_ms = max_over_ranks([ms_total, e2e_ms], dist, dev)

    flops = B * H * attn_flops(range(N), N, D, args.causal)
    ms_step = ms_total / args.steps
    value = whole_job_tflops(world, flops, ms_step)
    fwd_avg = sum(fwd_ms) / len(fwd_ms)
    achieved = flops / (fwd_avg * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    ratio = FP8PV_OVER_BF16 if args.fp8pv else FP4_OVER_BF16
    peak_nominal = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS)) * ratio
    peak = forward_peak(mma_peaks, args.fp8pv)
    record = TRAFFIC_RECORD_CAUSAL if args.causal else TRAFFIC_RECORD
    traffic = (record["bytes_per_launch"]
               if (record["sources_sha"] == sources_sha() and not args.fp8pv and w.shape == record["shape"])
               else None)
    line = {
        "metric": metric_name(args), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1+e4m3" if args.fp8pv else "e2m1", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "D": D, "recipe": w.description,
                   "step": "NVFP4 quantize Q and K, %s quantize V, %sDirect-P forward"
                           % ("MXFP8" if args.fp8pv else "MXFP4", "causal " if args.causal else ""),
                   "mask": "causal" if args.causal else "none", "pv": "fp8" if args.fp8pv else "fp4",
                   "l2": (("inputs larger than L2 (%.2f GB bf16 in, %.2f GB quantized); no flush"
                           % (in_bytes / 1e9, quant_bytes / 1e9)) if flush is None else
                          ("inputs (%.3f GB bf16) fit in L2 (%d MB): a %d MB write between steps, "
                           "outside each step's events" % (in_bytes / 1e9, l2_bytes >> 20, (2 * l2_bytes) >> 20))),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "fwd_ms": fwd_avg,
        "fwd_frac_of_fp4_peak": achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": ("measured block-scaled tcgen05 MMA loop on this GPU (M=N=128, one CTA per "
                                     "SM): QK^T kind::mxf4nvf4 %.0f, PV kind::%s %.0f TFLOP/s, FLOP-weighted "
                                     "harmonic combination; burst"
                                     % (mma_peaks["nvf4"], "mxf8f6f4" if args.fp8pv else "mxf4",
                                        mma_peaks["mxf8" if args.fp8pv else "mxf4"])),
                     "peak_clocks": peak_clocks.summary(),
                     "frac_of_nominal_bf16_ratio": achieved / peak_nominal,
                     "nominal_bf16_ratio_peak": peak_nominal,
                     "kernel": "fwd_directp_kernel<%d, causal=%s, fp8pv=%s>"
                               % (D, str(bool(args.causal)).lower(), str(bool(args.fp8pv)).lower())},
        "e2e": {"value": whole_job_tflops(world, flops, e2e_ms), "unit": UNIT,
                "api": "fp4attn_fwd_host_batch (C ABI, pinned host buffers in and out)",
                "pipelining": "upload of step i+1 and download of step i-1 overlap step i's kernels",
                "steps": e2e_steps, "timed": "first upload to last download (pipeline fill and drain included)",
                "h2d_bytes_per_step": 3 * B * H * N * D * 2, "d2h_bytes_per_step": B * H * N * D * 2 + B * H * N * 4,
                "host_link_gbs": link},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_variants and args.workload == 4 and not args.causal \
            and not args.fp8pv:
        del q, k, v, qq, kq, vq, o, lse, ws, flush
        torch.cuda.empty_cache()
        line["variants"] = [time_variant(wl.WORKLOADS[5], False, False, mma_peaks, dev, local),
                            time_variant(w, True, False, mma_peaks, dev, local),
                            time_variant(w, False, True, mma_peaks, dev, local),
                            time_backward(w, mma_peaks, dev, local)]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q_h, k_h, v_h, causal=args.causal, fp8pv=args.fp8pv)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, help="workload index 1-5 (default 4)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--causal", action="store_true", help="time the causal forward (query i sees keys 0..i)")
    ap.add_argument("--fp8pv", action="store_true", help="time the FP8 P/V variant (MXFP8 V, E4M3 codes)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the D=64, causal and FP8 P/V forward timings of the default run")
    ap.add_argument("--mma-peak", action="store_true", help="print the measured block-scaled tensor rates and exit")
    ap.add_argument("--bwd", action="store_true",
                    help="time only the causal backward of the workload and print its line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    w = wl.WORKLOADS[args.workload]
    if args.mma_peak:
        return run_mma_peak(args)
    if args.bwd:
        return run_bwd(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
