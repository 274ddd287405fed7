"""Benchmark of the fused MX attention forward on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
MX quantisation of Q, K and V (fsa_mx_quantize_qkv, one launch) and the fused
attention forward (fsa_attention_fwd_ex).  The metric is attention forward TFLOP/s
(4*B*H*Sq*Sk*D per layer, halved for causal).  Inputs are resident in HBM when
the timed region starts; L2 is flushed (a 512 MB write) between timed steps.
The quantisation launch of a step is captured once as a CUDA graph and
replayed (--no-graph: launched eagerly); the attention launch is bracketed by
CUDA events of its own.  The end-to-end figure makes every call eagerly.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
(the forward needs no exchange between GPUs): value = all ranks' FLOPs / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, Workload, generate  # noqa: E402

# the largest single-GPU workload: long-context causal attention at 128K keys, MXFP4
# QK^T with EFQ probability codes
DEFAULT_WORKLOAD = "long_efq_128k"
# further workloads reported in the same line (kernel throughput, fraction of the
# measured peak, speedup over the BF16 kernel, fallback rate)
EXTRA_WORKLOADS = ["long_fp8_16k", "long_fp8_128k", "long_efq_16k", "long_nvfp4_128k", "video_dit", "adversarial"]
FMT = {"E4M3": 0, "E2M3": 1, "E2M1": 2, "E2M1_EFQ": 3, "E3M2": 4, "NVFP4": 5}
# tensor-core kind of each operand format: 0 kind::f16, 1 kind::mxf8f6f4, 2 kind::mxf4
KIND = {"E4M3": 1, "E2M3": 1, "E3M2": 1, "E2M1": 2, "E2M1_EFQ": 2, "NVFP4": 3}
# nominal dense ratio of each kind to BF16 on GB300 (2.25 / 4.5 / 13.5 PFLOP/s): used
# only when the probe could not run
KIND_RATIO = {0: 1.0, 1: 2.0, 2: 6.0, 3: 6.0}
# DRAM bytes (read + write) of one attention launch of the current kernel build, from
# an ncu capture, by workload; absent: not captured for this build
TRAFFIC = {"long_efq_128k": 439.05e6 + 2.09e9, "long_efq_16k": 53.57e6 + 207.16e6,
           "long_fp8_16k": 103.88e6 + 210.56e6, "video_dit": 1.01e9 + 1.51e9}


def metric_name():
    return "attention fwd TFLOP/s (MXFP8/MXFP4) and % of block-scaled tensor-core peak"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    return 1900.0, 1700.0, "fallback"


def peak_for(w: Workload, measured=None):
    """Dense peak for the workload's formats: the harmonic mix of its QK^T and PV kinds
    (each GEMM is half the FLOPs).  measured: {kind: TFLOP/s} from the probe; else the
    MEASURED_PEAKS bf16 figure times the nominal ratio."""
    bf16, _, src = peaks()
    kq, kp = KIND[w.fmt_qk], KIND[w.fmt_pv]
    if measured and kq in measured and kp in measured:
        pq, pp, src = measured[kq], measured[kp], "measured on this GPU by the tcgen05 probe (fsa_mma_peak)"
    else:
        pq, pp = bf16 * KIND_RATIO[kq], bf16 * KIND_RATIO[kp]
        src = f"{src} bf16 GEMM burst (MEASURED_PEAKS.json) x nominal block-scaled/bf16 ratio"
    return 1.0 / (0.5 / pq + 0.5 / pp), src


def measure_mma_peaks(dev, seconds=0.03, sustained_s=0.0):
    """Dense tensor-core TFLOP/s per kind (0 bf16, 1 MXFP8, 2 MXFP4 kind::mxf4, 3 MXFP4
    through kind::mxf4nvf4) from the library's
    probe: one CTA per SM, operands resident on chip, timed with CUDA events.  Burst: one
    launch of about `seconds`; sustained: back-to-back launches for `sustained_s`."""
    import torch
    import softmax_mx_block_gb300 as fsa
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {}
    for kind in (0, 1, 2, 3):
        out[kind] = {}
        for nn in (128, 256):
            fsa.fsa_mma_peak(kind, n_sm, 2000, status, n=nn)           # warm-up and a first rate
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f = fsa.fsa_mma_peak(kind, n_sm, 20000, status, n=nn)
            e1.record()
            torch.cuda.synchronize()
            rate = f / (e0.elapsed_time(e1) * 1e-3)
            iters = max(1000, int(seconds * rate / (f / 20000)))
            best = 0.0
            for _ in range(3):
                e0.record()
                f = fsa.fsa_mma_peak(kind, n_sm, iters, status, n=nn)
                e1.record()
                torch.cuda.synchronize()
                best = max(best, f / (e0.elapsed_time(e1) * 1e-3) / 1e12)
            out[kind][f"burst_n{nn}"] = best
            if sustained_s > 0:
                reps = max(1, int(sustained_s / seconds))
                e0.record()
                tot = sum(fsa.fsa_mma_peak(kind, n_sm, iters, status, n=nn) for _ in range(reps))
                e1.record()
                torch.cuda.synchronize()
                out[kind][f"sustained_n{nn}"] = tot / (e0.elapsed_time(e1) * 1e-3) / 1e12
        # the dense peak of the kind: the better of the two shapes
        out[kind]["burst"] = max(out[kind]["burst_n128"], out[kind]["burst_n256"])
    if int(status.item()) != 0:
        raise RuntimeError("tensor-core probe timed out")
    return out


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and clock-event reasons sampled every millisecond through NVML
    (libnvidia-ml, read-only queries) while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id=None):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self._stop = threading.Event()
        self._thread = None
        self.nvml = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            ok = False
            if pci_bus_id:
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h)) == 0
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0
            if ok:
                self.nvml, self.h, self.ct = nv, h, ctypes
                mx = ctypes.c_uint()
                if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                    self.max_mhz = float(mx.value)
        except OSError:
            self.nvml = None

    def _poll(self):
        ct, nv, h = self.ct, self.nvml, self.h
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if get_reasons(h, ct.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(0.001)

    def start(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        reasons = sorted(n for b, n in self.REASONS.items() if self.reasons & b)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples)}


# ----------------------------------------------------------------------------- GPU arm
def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks of the default process group
    (the values themselves when there is none): the slowest replica sets the time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def run_gpu(args, w: Workload, world):
    import torch
    import softmax_mx_block_gb300 as fsa
    from softmax_mx_block_gb300._binding import empty_mx

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    layers = [w.layer(l) for l in range(w.layers)] if w.layers > 1 else [w]
    host, inputs, bufs = [], [], []
    for wl in layers:
        q, k, v = generate(wl)
        hs = tuple(torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory() for a in (q, k, v))
        host.append(hs)
        inputs.append(tuple(t.to(dev) for t in hs))
        fq, fp = FMT[wl.fmt_qk], FMT[wl.fmt_pv]
        fv = 2 if fp == 3 else fp
        bufs.append((empty_mx(wl.B, wl.H, wl.Sq, wl.D, 0, fq, dev), empty_mx(wl.B, wl.Hkv, wl.Sk, wl.D, 0, fq, dev),
                     empty_mx(wl.B, wl.Hkv, wl.Sk, wl.D, 1, fv, dev),
                     torch.empty((wl.B, wl.H, wl.Sq, wl.D), dtype=torch.float32, device=dev)))
    stream = torch.cuda.current_stream()
    stats = fsa.new_stats(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    attn_ev = []

    def quantise(i):
        wl, (qd, kd, vd), (mq, mk, mv, _) = layers[i], inputs[i], bufs[i]
        fq, fp = FMT[wl.fmt_qk], FMT[wl.fmt_pv]
        fsa.fsa_mx_quantize_qkv(qd, kd, vd, fq, 2 if fp == 3 else fp, out=(mq, mk, mv))

    qgraphs = []          # per layer: the quantisation launch captured as a CUDA graph

    def step(record=False):
        for i, (wl, (mq, mk, mv, out)) in enumerate(zip(layers, bufs)):
            fq, fp = FMT[wl.fmt_qk], FMT[wl.fmt_pv]
            if qgraphs:
                qgraphs[i].replay()
            else:
                quantise(i)
            if record:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            fsa.fsa_attention_fwd(mq, mk, mv, out, causal=wl.causal, scale=wl.scale, fmt_qk=fq, fmt_pv=fp,
                                  stats=stats, exp_mode=args.exp_mode)
            if record:
                e1.record(stream)
                attn_ev.append((e0, e1))

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launch_mode = "eager"
    if not args.no_graph:
        # the same library calls, captured once and replayed: no host launch overhead
        try:
            for i in range(len(layers)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, capture_error_mode="relaxed"):
                    quantise(i)
                qgraphs.append(g)
            step()
            torch.cuda.synchronize()
            launch_mode = "quantisation from a CUDA graph, attention eager"
        except Exception as e:  # capture unsupported: stay eager and say so
            qgraphs.clear()
            torch.cuda.synchronize()
            launch_mode = f"eager (graph capture failed: {type(e).__name__})"
    stats.zero_()
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
        bus = f"{torch.cuda.get_device_properties(dev).pci_domain_id:08x}:{bus:02x}:{torch.cuda.get_device_properties(dev).pci_device_id:02x}.0"
    except Exception:
        bus = None
    clk = ClockSampler(bus)
    clk.start()
    barrier()
    total_ms = 0.0
    for _ in range(args.steps):
        flush.fill_(1.0)                      # evict L2 between timed steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(record=True)
        e1.record(stream)
        e1.synchronize()
        total_ms += e0.elapsed_time(e1)
    barrier()
    clocks = clk.stop()
    st = fsa.read_stats(stats)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in attn_ev)

    # end to end through the public API from pinned host memory: one fsa_attention_fwd_host
    # call per layer copies Q, K, V in, quantises, attends and copies O back, by groups of
    # kv heads whose copies overlap the other groups' compute
    out_host = [torch.empty(b[3].shape, dtype=torch.float32).pin_memory() for b in bufs]
    hbufs = [fsa.HostCallBuffers.from_tensors(*ds, b[:3], b[3]) for ds, b in zip(inputs, bufs)]
    n_e2e = max(1, min(args.steps, 5))
    e2e_ms = 0.0
    for _ in range(n_e2e):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for wl, hs, oh, hb in zip(layers, host, out_host, hbufs):
            fsa.fsa_attention_fwd_host(*hs, oh, buffers=hb, fmt_qk=FMT[wl.fmt_qk], fmt_pv=FMT[wl.fmt_pv],
                                       causal=wl.causal, scale=wl.scale, stats=stats, exp_mode=args.exp_mode)
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= n_e2e
    h2d = sum(t.numel() * 2 for hs in host for t in hs)
    d2h = sum(b[3].numel() * 4 for b in bufs)

    # the in-house BF16 exact-softmax kernel on the same inputs (speedup reference)
    vts = [fsa.fsa_bf16_transpose_v(ds[2]) for ds in inputs]
    out_bf = [torch.empty_like(b[3]) for b in bufs]
    bf_ms = []
    for it in range(args.warmup + max(3, min(args.steps, 10))):
        for wl, (qd, kd, _), vt, ob in zip(layers, inputs, vts, out_bf):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fsa.fsa_attention_fwd_bf16(qd, kd, vt, ob, causal=wl.causal, scale=wl.scale)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                bf_ms.append(e0.elapsed_time(e1))

    ms, e2e_ms = max_over_ranks([total_ms / args.steps, e2e_ms], dev)
    return dict(ms=ms, attn_ms=attn_ms, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, clocks=clocks, stats=st, launch_mode=launch_mode,
                launches=args.steps * 2 * len(layers), bf16_ms=statistics.mean(bf_ms))


def time_workload(name, dev, steps, exp_mode, measured_peaks):
    """Attention-kernel throughput of one further workload (inputs resident, L2 flushed
    between launches), the BF16 kernel on the same inputs, and the fallback rate at the
    library's default margin (and at margin 0 for the adversarial workload)."""
    import torch
    import softmax_mx_block_gb300 as fsa
    w = WORKLOADS[name]
    layers = [w.layer(l) for l in range(w.layers)] if w.layers > 1 else [w]
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    attn_ms, bf_ms = [], []
    st8, st0 = fsa.new_stats(dev), fsa.new_stats(dev)
    for wl in layers:
        q, k, v = (torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16) for a in generate(wl))
        fq, fp = FMT[wl.fmt_qk], FMT[wl.fmt_pv]
        mq, mk, mv = fsa.fsa_mx_quantize_qkv(q, k, v, fq, 2 if fp == 3 else fp)
        out = torch.empty((wl.B, wl.H, wl.Sq, wl.D), dtype=torch.float32, device=dev)
        call = dict(causal=wl.causal, scale=wl.scale, fmt_qk=fq, fmt_pv=fp, exp_mode=exp_mode)
        n = steps if len(layers) == 1 else 2
        for it in range(3 + n):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fsa.fsa_attention_fwd(mq, mk, mv, out, stats=st8 if it == 3 else None, **call)
            e1.record(stream)
            e1.synchronize()
            if it >= 3:
                attn_ms.append(e0.elapsed_time(e1))
        if wl.kind == "planted":
            fsa.fsa_attention_fwd(mq, mk, mv, out, stats=st0, delta=0.0, **call)
        del mq, mk, mv
        vt = fsa.fsa_bf16_transpose_v(v)
        for it in range(2 + max(1, n // 2)):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fsa.fsa_attention_fwd_bf16(q, k, vt, out, causal=wl.causal, scale=wl.scale)
            e1.record(stream)
            e1.synchronize()
            if it >= 2:
                bf_ms.append(e0.elapsed_time(e1))
        del q, k, v, vt, out
    torch.cuda.synchronize()
    r8, r0 = fsa.read_stats(st8), fsa.read_stats(st0)
    # per layer: the mean launch time; per workload: FLOPs of all layers over their summed means
    per_layer = len(attn_ms) // len(layers)
    a_ms = sum(statistics.mean(attn_ms[i * per_layer:(i + 1) * per_layer]) for i in range(len(layers)))
    per_layer_bf = len(bf_ms) // len(layers)
    b_ms = sum(statistics.mean(bf_ms[i * per_layer_bf:(i + 1) * per_layer_bf]) for i in range(len(layers)))
    tf = w.flops / (a_ms * 1e-3) / 1e12
    peak, _ = peak_for(w if w.layers == 1 else layers[0], measured_peaks)
    if w.layers > 1:   # alternating kinds: the harmonic mix over the layers
        peak = len(layers) / sum(1.0 / peak_for(wl, measured_peaks)[0] for wl in layers)
    res = {"tflops": tf, "frac_of_peak": tf / peak, "peak_tflops": peak,
           "bf16_tflops": w.flops / (b_ms * 1e-3) / 1e12, "speedup_vs_bf16": b_ms / a_ms,
           "fallback_rate": r8["fallback_events"] / r8["row_tiles"] if r8["row_tiles"] else None,
           "delta": 8.0}
    if w.kind == "planted":
        res["fallback_rate_delta0"] = r0["fallback_events"] / r0["row_tiles"] if r0["row_tiles"] else None
    del flush
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- CPU oracle arm
# which key positions of a 32-key block the oracle takes through ex2 (bit set) for
# each exp mode: 0 the cubic everywhere, 1 ex2 everywhere, 2 the cubic at 4k+3
MUFU_MASK = {0: 0x00000000, 1: 0xFFFFFFFF, 2: 0x77777777}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def run_oracle_sample(w: Workload, budget_s=15.0, exp_mode=1):
    """The oracle's step-by-step emulation on a bounded sample of query rows, timed on
    the host cores; returns (TFLOP/s-equivalent, description, threads)."""
    import oracle
    wl = w.layer(0) if w.layers > 1 else w
    q, k, v = generate(wl)
    fp = FMT[wl.fmt_pv]
    mx = oracle.MxInputs.from_bf16(q, k, v, FMT[wl.fmt_qk], 2 if fp == 3 else fp)
    # every query row of the workload in a seeded random order, taken in growing
    # chunks until the time budget is spent or the rows run out
    rows_all = np.random.default_rng(0).permutation(wl.B * wl.H * wl.Sq).astype(np.int64)
    threads = oracle.nthreads_default()
    n, t_used, flops, done = 32, 0.0, 0.0, 0
    while done < len(rows_all):
        rows = np.sort(rows_all[done:done + n])
        t0 = time.perf_counter()
        oracle.fsa_emulate(mx, wl.Sk, wl.causal, wl.scale, fp, rows, delta=8.0, mufu_mask=MUFU_MASK[exp_mode])
        dt = time.perf_counter() - t0
        i = rows % wl.Sq
        vis = np.minimum(wl.Sk, i + 1 + wl.Sk - wl.Sq) if wl.causal else np.full(len(rows), wl.Sk)
        flops += float(np.sum(4.0 * vis * wl.D))
        t_used += dt
        done += len(rows)
        if t_used > budget_s:
            break
        n = min(4096, n * 2)
    which = "all" if done == len(rows_all) else f"{done} randomly sampled of the {len(rows_all)}"
    desc = (f"oracle emulation (fsa_emulate, fp64 accumulation) of {which} query rows of {wl.name} "
            f"({wl.fmt_qk}/{wl.fmt_pv}) in {t_used:.1f} s on {threads} threads ({cpu_model()}, "
            f"{os.cpu_count()} logical CPUs); FLOPs = 4*D*visible keys per row")
    return flops / t_used / 1e12, desc, threads


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="fsa", choices=["fsa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the quantisation eagerly (no CUDA graph)")
    ap.add_argument("--no-extra", action="store_true", help="skip the further workloads of the line")
    ap.add_argument("--no-peak-probe", action="store_true", help="skip the tensor-core probe (nominal ratios)")
    ap.add_argument("--exp-mode", type=int, default=1, choices=[0, 1, 2],
                    help="0 cubic, 1 ex2.approx (default, the library's), 2 split 3:1")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    flops_per_step = w.flops

    config = {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
              "causal": w.causal, "fmt_qk": w.fmt_qk, "fmt_pv": w.fmt_pv, "layers": w.layers,
              "l2": "flushed between timed steps (512 MB write)", "exp_mode": args.exp_mode, "parallelism": f"replicas x{max(world, 1)}"}

    if args.impl == "reference":
        if rank != 0:
            return
        v, desc, threads = run_oracle_sample(w, budget_s=20.0, exp_mode=args.exp_mode)
        line = {"metric": metric_name(), "value": v, "unit": "TFLOP/s", "impl": "reference", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, workloads.py)", "config": config,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    import torch
    import softmax_mx_block_gb300 as fsa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    fsa.load()
    measured = None
    peak_info = None
    if not args.no_peak_probe:
        mp = measure_mma_peaks(dev, sustained_s=0.5)
        measured = {k: v["burst"] for k, v in mp.items()}
        peak_info = {{0: "bf16", 1: "mxf8f6f4_e4m3", 2: "mxf4_e2m1", 3: "mxf4nvf4_2x_e2m1"}[k]: v
                     for k, v in mp.items()}
        # MXFP4 operands run through either instruction kind: the peak is the faster one
        measured[2] = max(measured[2], measured[3])
    r = run_gpu(args, w, world)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    config["launch"] = r["launch_mode"]
    value = flops_per_step * world / (r["ms"] * 1e-3) / 1e12
    attn_tflops = flops_per_step / w.layers / (r["attn_ms"] * 1e-3) / 1e12
    peak, src = peak_for(w, measured)
    peak_nominal, src_nominal = peak_for(w, None)
    if w.layers > 1:
        peak = w.layers / sum(1.0 / peak_for(w.layer(l), measured)[0] for l in range(w.layers))
        peak_nominal = w.layers / sum(1.0 / peak_for(w.layer(l), None)[0] for l in range(w.layers))
    rt = r["stats"]["row_tiles"]
    line = {
        "metric": metric_name(), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": f"mx-{w.fmt_qk.lower()}/{w.fmt_pv.lower()}",
        "data": "synthetic (seeded, workloads.py)", "config": config,
        "attention_kernel": {"tflops": attn_tflops, "ms_per_launch": r["attn_ms"],
                             "frac_of_block_scaled_peak": attn_tflops / peak},
        "bf16_kernel": {"tflops": flops_per_step / w.layers / (r["bf16_ms"] * 1e-3) / 1e12,
                        "ms_per_launch": r["bf16_ms"]},
        "speedup_vs_bf16": r["bf16_ms"] / r["attn_ms"],
        "fallback_rate": (r["stats"]["fallback_events"] / rt) if rt else None,
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak, "traffic": TRAFFIC.get(w.name),
                     "peak_source": src + " (burst, the better of M=128 N=128 and N=256 dense MMAs; harmonic "
                                          "mix of the QK^T and PV kinds)",
                     # the same fraction against the other denominator: the bf16 GEMM
                     # figure of MEASURED_PEAKS.json (or the fallback) times the nominal
                     # block-scaled/bf16 ratio of each kind
                     "vs_bf16_gemm_x_nominal": {"peak": peak_nominal, "frac": attn_tflops / peak_nominal,
                                                "source": src_nominal}},
        "tensor_peaks_tflops": peak_info,
        "e2e": {"value": flops_per_step * world / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if not args.no_extra and world == 1:
        line["workloads"] = {}
        for name in EXTRA_WORKLOADS:
            if name != w.name:
                line["workloads"][name] = time_workload(name, torch.device("cuda", 0), min(args.steps, 5),
                                                        args.exp_mode, measured)
    if not args.no_cpu_baseline and world == 1:
        v, desc, threads = run_oracle_sample(w, budget_s=15.0, exp_mode=args.exp_mode)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
