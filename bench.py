#!/usr/bin/env python
"""Benchmark: the fp16 TN GEMM shape sweep (343 shapes, M, N, K in {64..4096}) on one GPU.

One step = one gemm_run for every shape of the sweep, each on its own
device-resident A, B, C (2.77 GB of distinct operands per step, more than the
129 MB L2, so no step finds the previous step's data in L2).  `value` is the
throughput sum(2*M*N*K) / step time in TFLOP/s.

  python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `roofline` is the step's roofline: per shape the largest
of tensor time, compulsory-byte HBM time and the launch floor, summed over the
343 shapes and divided by the timed step (also per class of shapes).  Also on
the line (measured outside the timed region): `e2e` (the same sweep through the
C ABI with operands copied from pinned host memory and C copied back inside the
timed region), `named` (µs/call and TFLOP/s of the named workloads: 64x4096x64
and 128x2048x128 fp16, 8192^3 fp16, the 4096x14336x4096 bf16 FFN shape,
4096^3 int8->int32), GPU clocks sampled during the timed region, and the CPU
oracle timed on bounded samples (`cpu_baseline`).

The library runs on one GPU: with --gpus > 1 (or WORLD_SIZE > 1) the GEMM arm
prints one "unavailable" line and does no work.

--impl reference times the CPU oracle (the only reference this method has) on a
bounded sample of the same sweep, on the host cores, and prints the same line
with "impl": "reference" (rank 0 only under torchrun).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from dense_gemm_hgemm_gb300 import inputs, workloads  # noqa: E402

METRIC = "GEMM TFLOPS and % of roofline per (M,N,K,dtype); µs/call at 64x4096x64 fp16"
UNIT = "TFLOP/s"
WORKLOAD = "hgemm_tn_fp16_sweep_343_shapes_M_N_K_in_64..4096"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------- helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--skip-extras", action="store_true",
                    help="only the timed sweep (no e2e, named workloads or CPU baseline)")
    ap.add_argument("--ncu-steps", type=int, default=0,
                    help="run this many untimed steps and exit (for profiler launch lists)")
    ap.add_argument("--tma-sweep", action="store_true",
                    help="run the TMA load-mode x FMA-intensity experiment and print its table")
    ap.add_argument("--shape", default=None,
                    help="with --ncu-steps: run only this workload, 'M,N,K,dtype' (profiling)")
    ap.add_argument("--config", default=None,
                    help="with --shape: a JSON kernel configuration instead of the table's")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def one_gpu_only(args) -> bool:
    """The library runs on one GPU; a multi-GPU launch of the GEMM arm prints one
    'unavailable' line (rank 0) and does no work on any rank.  True if so."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus <= 1 and world <= 1:
        return False
    if int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps({"metric": METRIC, "impl": "ours", "n_gpus": max(args.gpus, world),
                          "unavailable": "one-GPU library: the GEMM runs on a single GPU and "
                                         "has no multi-GPU path"}), flush=True)
    return True


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# Sources that build no kernel a sweep launch runs (the int8 widening / fill /
# empty kernels, the TMA intensity sweep, the CPython entry points, the MMA
# rate probe, the allocation-free entry point): left out of the digest.
_DIGEST_SKIP = ("gemm_aux.cu", "tma_intensity.cu", "gemm_pycall.c", "gemm_probe.cu",
                "gemm_noalloc.cu")


def source_digest() -> str:
    """Hash of the GEMM kernels' sources (kernels, launch code, config table), to
    tell whether stored ncu counters of the sweep still apply."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_hgemm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in _DIGEST_SKIP:
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic():
    """Per-launch DRAM bytes of the sweep from the committed ncu summary, if current."""
    path = os.path.join(ROOT, "profiles", "sweep_f16_dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, "no committed ncu capture"
    if d.get("source_digest") != source_digest():
        return None, "kernel changed since the ncu capture"
    return d.get("dram_bytes_per_launch"), "ncu capture %s" % d.get("when", "?")


# --------------------------------------------------------------------------- our arm

def make_sweep(device):
    """Per-shape seeded operands on the device (own buffers per shape) and plans."""
    import dense_gemm_hgemm_gb300 as g
    shapes = workloads.sweep_shapes()
    items = []
    gen = torch.Generator(device=device)
    for w in shapes:
        gen.manual_seed(inputs.shape_seed(w.M, w.N, w.K, w.dtype))
        A = torch.randn(w.M, w.K, generator=gen, device=device, dtype=torch.float32).half()
        B = torch.randn(w.N, w.K, generator=gen, device=device, dtype=torch.float32).half()
        C = torch.empty(w.M, w.N, device=device, dtype=torch.float16)
        items.append((w, g.Plan(w.M, w.N, w.K, "f16"), A, B, C))
    return items


def run_step(items, stream):
    for _, plan, A, B, C in items:
        plan.run(A, B, C, stream)


def time_sweep(items, steps, warmup, stream, sampler=None):
    """Eager steps: one gemm_run per shape, timed with CUDA events on `stream`."""
    for _ in range(warmup):
        run_step(items, stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(steps):
        run_step(items, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    return e0.elapsed_time(e1), wall, clocks


def capture_step(items, stream):
    """One sweep step (all of `items`' gemm_run launches) captured as a CUDA graph:
    the same kernels, parameters and buffers, replayed without per-launch host work."""
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run_step(items, stream)
    torch.cuda.synchronize()
    return graph


def time_graph(graph, steps, warmup, stream, sampler=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = sampler.stop() if sampler else None
    return e0.elapsed_time(e1), wall, clocks


def per_shape_times(items, stream, reps=3):
    """Device time of every launch of one step (events around each launch), median of reps."""
    res = {}
    for _ in range(reps):
        evs = []
        for w, plan, A, B, C in items:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.run(A, B, C, stream)
            b.record(stream)
            evs.append((w, a, b))
        torch.cuda.synchronize()
        for w, a, b in evs:
            res.setdefault(w.name, []).append(a.elapsed_time(b))
    return {k: statistics.median(v) for k, v in res.items()}


def e2e_sweep(items, stream, steps, groups=32):
    """The sweep through the public API with host operands, end to end: every step
    copies all A, B from pinned host memory to the device, runs gemm_run per shape
    and copies every C back.  Operands are packed in one pinned buffer per
    direction and the step is pipelined over groups of shapes on three streams
    (host-to-device copy of group g+1 and device-to-host copy of group g-1 overlap
    the GEMMs of group g), as a user feeding the GPU from host memory would.  Groups
    are consecutive shapes of about equal bytes (in + out), so that neither the
    first copy in nor the last copy back is a large exposed share of the step."""
    align = 256
    in_off, out_off, n_in, n_out = [], [], 0, 0
    for w, plan, A, B, C in items:
        a_b, b_b, c_b = A.numel() * 2, B.numel() * 2, C.numel() * 2
        in_off.append((n_in, n_in + -(-a_b // align) * align))
        n_in += -(-a_b // align) * align + -(-b_b // align) * align
        out_off.append(n_out)
        n_out += -(-c_b // align) * align
    h_in = torch.empty(n_in, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(n_out, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(n_in, dtype=torch.uint8, device="cuda")
    d_out = torch.empty(n_out, dtype=torch.uint8, device="cuda")
    views = []
    h2d = d2h = 0
    for (w, plan, A, B, C), (oa, ob), oc in zip(items, in_off, out_off):
        a_b, b_b, c_b = A.numel() * 2, B.numel() * 2, C.numel() * 2
        h_in[oa:oa + a_b].copy_(A.view(-1).view(torch.uint8).cpu())
        h_in[ob:ob + b_b].copy_(B.view(-1).view(torch.uint8).cpu())
        dA = d_in[oa:oa + a_b].view(torch.float16).view(A.shape)
        dB = d_in[ob:ob + b_b].view(torch.float16).view(B.shape)
        dC = d_out[oc:oc + c_b].view(torch.float16).view(C.shape)
        views.append((plan, dA, dB, dC))
        h2d += a_b + b_b
        d2h += c_b
    # groups of consecutive shapes (contiguous byte ranges) of about equal bytes
    n = len(items)
    sizes = [A.numel() * 2 + B.numel() * 2 + C.numel() * 2 for _, _, A, B, C in items]
    total = float(sum(sizes))
    bounds, acc = [0], 0
    for i, sz in enumerate(sizes):
        acc += sz
        if acc >= total * len(bounds) / groups and i + 1 < n and len(bounds) < groups:
            bounds.append(i + 1)
    bounds.append(n)
    groups = len(bounds) - 1
    rng_in = [(in_off[bounds[g]][0], in_off[bounds[g + 1]][0] if bounds[g + 1] < n else n_in)
              for g in range(groups)]
    rng_out = [(out_off[bounds[g]], out_off[bounds[g + 1]] if bounds[g + 1] < n else n_out)
               for g in range(groups)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(groups)]
    ev_mm = [torch.cuda.Event() for _ in range(groups)]
    ev_out = [torch.cuda.Event() for _ in range(groups)]
    torch.cuda.synchronize()

    def timed_copy(st, dst, src, marks):
        # one copy on stream `st`; with `marks`, bracketed by timing events
        if marks is None:
            dst.copy_(src, non_blocking=True)
            return
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        dst.copy_(src, non_blocking=True)
        b.record(st)
        marks.append((a, b))

    def one(busy_in=None, busy_out=None):
        for g in range(groups):
            lo, hi = rng_in[g]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_mm[g])          # the previous step's GEMMs read this range
                timed_copy(s_in, d_in[lo:hi], h_in[lo:hi], busy_in)
                ev_in[g].record(s_in)
            stream.wait_event(ev_in[g])
            stream.wait_event(ev_out[g])           # the previous step's copy-out of this range
            for plan, dA, dB, dC in views[bounds[g]:bounds[g + 1]]:
                plan.run(dA, dB, dC, stream)
            ev_mm[g].record(stream)
            lo, hi = rng_out[g]
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_mm[g])
                timed_copy(s_out, h_out[lo:hi], d_out[lo:hi], busy_out)
                ev_out[g].record(s_out)

    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    # How long the host link is busy in the step: the summed durations of the
    # step's copies in each direction, timed on the copy streams in untimed
    # steps run the same way (median of three)
    busy = []
    for _ in range(3):
        m_in, m_out = [], []
        one(m_in, m_out)
        torch.cuda.synchronize()
        busy.append((sum(a.elapsed_time(b) for a, b in m_in),
                     sum(a.elapsed_time(b) for a, b in m_out)))
    busy_ms = (statistics.median(x[0] for x in busy), statistics.median(x[1] for x in busy))
    # results came back: spot-check one C against the device copy of the eager run
    mid = len(items) // 2
    w, plan, A, B, C = items[mid]
    oc = out_off[mid]
    got = h_out[oc:oc + C.numel() * 2].view(torch.float16).view(C.shape)
    one()   # leave every result in place for the check below
    torch.cuda.synchronize()
    if not torch.equal(got.view(torch.int16), C.cpu().view(torch.int16)):
        raise RuntimeError("e2e: copied-back result differs from the device result")
    return wall * 1e3 / steps, h2d, d2h, busy_ms


def launch_floor_us(stream, sms, n=2000, graph=False):
    """Back-to-back period of an empty kernel launched like the GEMM (PDL, one CTA
    per SM): eagerly one call at a time, or replayed from a captured graph."""
    import dense_gemm_hgemm_gb300 as g
    for _ in range(100):
        g.gemm_launch_empty(sms, stream.cuda_stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if graph:
        per = 500
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            for _ in range(per):
                g.gemm_launch_empty(sms, stream.cuda_stream)
        with torch.cuda.stream(stream):
            cg.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(n // per):
                cg.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (per * (n // per))
    e0.record(stream)
    for _ in range(n):
        g.gemm_launch_empty(sms, stream.cuda_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / n


def named_workloads(stream, peaks, p_tensor, floor_us, sms, sm_max_mhz):
    """Warm µs/call (back-to-back on the same buffers, median of 5 repeats of a
    >= 20 ms loop; >= 200 ms for the large shapes, with SM clocks sampled) and
    TFLOP/s with the roofline fraction for each named shape; cold µs/call (L2
    flushed before every call) for the two skinny shapes.  Large shapes also
    report the throughput scaled to the maximum SM clock (x max / median sampled
    clock), which separates a box's power-capped clock from the kernel."""
    import dense_gemm_hgemm_gb300 as g
    out = {}
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for w in workloads.NAMED:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(inputs.shape_seed(w.M, w.N, w.K, w.dtype))
        if w.dtype == "i8":
            A = torch.randint(-128, 128, (w.M, w.K), generator=gen, device="cuda", dtype=torch.int8)
            B = torch.randint(-128, 128, (w.N, w.K), generator=gen, device="cuda", dtype=torch.int8)
        else:
            td = inputs.TORCH_DTYPE[w.dtype]
            A = (torch.randn(w.M, w.K, generator=gen, device="cuda") * w.a_scale).to(td)
            B = (torch.randn(w.N, w.K, generator=gen, device="cuda") * w.b_scale).to(td)
        C = torch.empty(w.M, w.N, device="cuda", dtype=inputs.OUT_DTYPE[w.dtype])
        large = w.flops >= 1e11
        with g.Plan(w.M, w.N, w.K, w.dtype) as plan:
            for _ in range(20):
                plan.run(A, B, C, stream)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plan.run(A, B, C, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            one = max(e0.elapsed_time(e1), 1e-3)
            reps = max(10, min(5000, int((200.0 if large else 20.0) / one)))
            sampler = ClockSampler(0) if large else None
            if sampler:
                sampler.start()
            samples = []
            for _ in range(5):
                e0.record(stream)
                for _ in range(reps):
                    plan.run(A, B, C, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                samples.append(e0.elapsed_time(e1) * 1e3 / reps)
            clk = sampler.stop() if sampler else None
            us = statistics.median(samples)
            cold = None
            if w.flops < 1e9:
                cs = []
                for _ in range(30):
                    with torch.cuda.stream(stream):
                        flush.add_(1)      # 512 MB write evicts A, B, C from the 129 MB L2
                    e0.record(stream)
                    plan.run(A, B, C, stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    cs.append(e0.elapsed_time(e1) * 1e3)
                cold = statistics.median(cs)
            plan.check(stream)
            cfg = plan.config
        tflops = w.flops / (us * 1e-6) / 1e12
        t_tensor = w.flops / (p_tensor * 1e12) * 1e6
        t_hbm = w.compulsory_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        t_roof = max(t_tensor, t_hbm, floor_us)
        bound = "tensor" if t_roof == t_tensor else ("hbm" if t_roof == t_hbm else "launch")
        key = "TOPS" if w.dtype == "i8" else "TFLOPS"
        out[w.name] = {
            "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype, "us_per_call": round(us, 3),
            "us_per_call_cold_l2": round(cold, 3) if cold is not None else None,
            key: round(tflops, 2),
            "roofline_bound": bound, "roofline_us": round(t_roof, 3),
            "roofline_frac": round(t_roof / us, 4),
            "frac_of_measured_burst_peak": round(tflops / peaks["bf16_tflops"], 4),
            "config": cfg,
        }
        if clk and clk.get("sm_mhz"):
            out[w.name]["clocks"] = clk
            out[w.name][key + "_at_max_clock"] = round(tflops * sm_max_mhz / clk["sm_mhz"], 2)
        if w.dtype == "i8":
            out[w.name]["note"] = ("int8 runs on the fp16 tensor path (sm_103a has no tcgen05 "
                                   "kind::i8); peak is the fp16/bf16 rate")
        if w is workloads.FFN_BF16:
            # The same shape with the linear-layer epilogue fused: C = GELU(A B^T + bias).
            bias = torch.randn(w.N, generator=gen, device="cuda").float()
            with g.Plan(w.M, w.N, w.K, w.dtype) as plan:
                for _ in range(5):
                    plan.run(A, B, C, stream, bias=bias, act=g.ACT_GELU)
                samples = []
                for _ in range(5):
                    e0.record(stream)
                    for _ in range(reps):
                        plan.run(A, B, C, stream, bias=bias, act=g.ACT_GELU)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    samples.append(e0.elapsed_time(e1) * 1e3 / reps)
                plan.check(stream)
            us2 = statistics.median(samples)
            out[w.name + "_bias_gelu"] = {
                "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype, "epilogue": "bias + GELU fused",
                "us_per_call": round(us2, 3), "TFLOPS": round(w.flops / (us2 * 1e-6) / 1e12, 2),
                "overhead_vs_plain": round(us2 / us - 1.0, 4)}
        del A, B, C
    del flush
    torch.cuda.empty_cache()
    return out


def server_mode(stream, calls=2000):
    """Back-to-back 64x4096x64 fp16 GEMMs (the pages' inference-server shape):
    calls/s issued one gemm_run at a time, and replayed from a captured CUDA graph."""
    import dense_gemm_hgemm_gb300 as g
    w = workloads.SKINNY
    gen = torch.Generator(device="cuda")
    gen.manual_seed(inputs.shape_seed(w.M, w.N, w.K, w.dtype))
    A = torch.randn(w.M, w.K, generator=gen, device="cuda").half()
    B = torch.randn(w.N, w.K, generator=gen, device="cuda").half()
    C = torch.empty(w.M, w.N, device="cuda", dtype=torch.float16)
    out = {}
    with g.Plan(w.M, w.N, w.K, w.dtype) as plan:
        for _ in range(50):
            plan.run(A, B, C, stream)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(calls):
            plan.run(A, B, C, stream)
        torch.cuda.synchronize()
        out["eager_calls_per_s"] = round(calls / (time.perf_counter() - t0), 1)
        per_graph = 100
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(per_graph):
                plan.run(A, B, C, torch.cuda.current_stream())
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        reps = max(1, calls // per_graph)
        t0 = time.perf_counter()
        for _ in range(reps):
            graph.replay()
        torch.cuda.synchronize()
        out["graph_calls_per_s"] = round(reps * per_graph / (time.perf_counter() - t0), 1)
        plan.check(stream)
    out["shape"] = [w.M, w.N, w.K, w.dtype]
    out["note"] = ("host wall clock over %d calls; eager = one Plan.run -> gemm_run per call "
                   "(the package's vectorcall entry point), graph = %d captured calls per "
                   "replay" % (calls, per_graph))
    return out


def cpu_oracle_sample(budget_s: float = 10.0, rows: int = 64):
    """Time the CPU oracle on rows [0, rows) of the sweep's shapes, in seeded
    random shape order, until `budget_s` seconds of work; TFLOP/s achieved."""
    import numpy as np

    import oracle
    oracle.build()
    shapes = workloads.sweep_shapes()
    order = torch.randperm(len(shapes), generator=torch.Generator().manual_seed(7)).tolist()
    flops = 0
    elapsed = 0.0
    done = 0
    threads = oracle.max_threads()
    for i in order:
        w = shapes[i]
        A, B = inputs.make_operands(min(rows, w.M), w.N, w.K, "f16")
        a = A.view(torch.int16).numpy().view(np.uint16)
        b = B.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        oracle.gemm_tn_half(a, b, 0, threads)
        elapsed += time.perf_counter() - t0
        flops += 2 * A.shape[0] * w.N * w.K
        done += 1
        if elapsed >= budget_s:
            break
    return {"value": flops / elapsed / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "rows [0,%d) of %d of the 343 sweep shapes (seeded order), %.3g FLOP, "
                      "%.1f s" % (rows, done, flops, elapsed)}


def _oracle_time(w, rows, threads):
    """Seconds the oracle takes for rows [0, rows) of workload w (all of B)."""
    import numpy as np

    import oracle
    A, B = inputs.make_operands(rows, w.N, w.K, w.dtype, w.a_scale, w.b_scale,
                                seed=inputs.shape_seed(w.M, w.N, w.K, w.dtype))
    if w.dtype == "i8":
        a, b = A.numpy(), B.numpy()
        t0 = time.perf_counter()
        oracle.gemm_tn_i8(a, b, threads)
    else:
        a = A.view(torch.int16).numpy().view(np.uint16)
        b = B.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        oracle.gemm_tn_half(a, b, oracle.FMT_BF16 if w.dtype == "bf16" else oracle.FMT_F16,
                            threads)
    return time.perf_counter() - t0


def cpu_oracle_named(full_limit_s: float = 2.0, block_rows: int = 64):
    """The oracle per named workload on the host cores: the full problem when a
    64-row block predicts it under `full_limit_s`, else that row block timed and
    extrapolated linearly in M (marked).  Plus one single-thread figure on the
    sweep's headline shape 128x2048x128."""
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    out = {}
    for w in workloads.NAMED:
        rows = min(block_rows, w.M)
        t_blk = _oracle_time(w, rows, threads)
        est = t_blk * w.M / rows
        if rows < w.M and est <= full_limit_s:
            rows, t_full, extrapolated = w.M, _oracle_time(w, w.M, threads), False
        elif rows < w.M:
            t_full, extrapolated = est, True
        else:
            t_full, extrapolated = t_blk, False
        out[w.name] = {"seconds": round(t_full, 4), "extrapolated": extrapolated,
                       "timed_rows": rows,
                       ("TOPS" if w.dtype == "i8" else "TFLOPS"): round(w.flops / t_full / 1e12, 5)}
    w = workloads.HEADLINE_SWEEP
    t1 = _oracle_time(w, w.M, 1)
    single = {"shape": [w.M, w.N, w.K, w.dtype], "cores": 1, "seconds": round(t1, 4),
              "TFLOPS": round(w.flops / t1 / 1e12, 6)}
    return out, single, threads


def profile_one(spec, calls, stream, config=None):
    """`calls` launches of one shape with the table's configuration, or `config`
    (a JSON object of gemm_config_t fields), for ncu."""
    import dense_gemm_hgemm_gb300 as g
    M, N, K, dtype = spec.split(",")
    M, N, K = int(M), int(N), int(K)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(inputs.shape_seed(M, N, K, dtype))
    if dtype == "i8":
        A = torch.randint(-128, 128, (M, K), generator=gen, device="cuda", dtype=torch.int8)
        B = torch.randint(-128, 128, (N, K), generator=gen, device="cuda", dtype=torch.int8)
    else:
        A = torch.randn(M, K, generator=gen, device="cuda").to(inputs.TORCH_DTYPE[dtype])
        B = torch.randn(N, K, generator=gen, device="cuda").to(inputs.TORCH_DTYPE[dtype])
    C = torch.empty(M, N, device="cuda", dtype=inputs.OUT_DTYPE[dtype])
    with g.Plan(M, N, K, dtype, json.loads(config) if config else None) as plan:
        for _ in range(calls):
            plan.run(A, B, C, stream)
        plan.check(stream)
        print(json.dumps({"shape": [M, N, K, dtype], "config": plan.config, "calls": calls}))


def mma_probe(sms, stream, iters=4096):
    """tcgen05.mma issue rate (gemm_probe_mma_rate): dense FLOP per clock per SM
    from one CTA alone and from one CTA on every SM (median over CTAs)."""
    import dense_gemm_hgemm_gb300 as g
    out = {}
    for grid in (1, sms):
        cyc = torch.zeros(grid, dtype=torch.int64, device="cuda")
        ns = torch.zeros(grid, dtype=torch.int64, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            g.gemm_probe_mma_rate(grid, iters, cyc, ns, err, stream)
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise RuntimeError("gemm_probe_mma_rate: a completion wait ran out")
        c = sorted(cyc.cpu().tolist())
        t = sorted(ns.cpu().tolist())
        med_c, med_t = c[len(c) // 2], t[len(t) // 2]
        out["grid_%d" % grid] = {"flop_per_clk_per_sm": round(iters * 1048576 / med_c, 1),
                                 "clock_mhz_seen": round(med_c / med_t * 1e3, 1)}
    return out


def ours(args):
    if one_gpu_only(args):
        return
    torch.cuda.set_device(0)
    import dense_gemm_hgemm_gb300 as g
    g.build_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if args.ncu_steps and args.shape:
        profile_one(args.shape, args.ncu_steps, stream, args.config)
        return
    items = make_sweep("cuda")
    flops_step = sum(w.flops for w, *_ in items)
    bytes_step = sum(w.compulsory_bytes for w, *_ in items)
    torch.cuda.synchronize()

    if args.ncu_steps:
        for _ in range(args.ncu_steps):
            run_step(items, stream)
        torch.cuda.synchronize()
        for _, plan, *_ in items:
            plan.check(stream)
        return

    # Eager: one Plan.run -> gemm_run per shape.
    ms_e, _, _ = time_sweep(items, args.steps, args.warmup, stream)
    for _, plan, *_ in items:
        plan.check(stream)     # raises if any kernel gave up on a wait
    ms_step_eager = ms_e / args.steps
    # Headline: the same step launched from a captured CUDA graph (the launch
    # overhead of 343 mostly tiny GEMMs is host work, not GEMM work).
    graph = capture_step(items, stream)
    sampler = ClockSampler(0)
    ms, wall, clocks = time_graph(graph, args.steps, args.warmup, stream, sampler)
    for _, plan, *_ in items:
        plan.check(stream)
    ms_step = ms / args.steps
    value = flops_step / (ms_step * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) fp16 operands per shape, generated on the device)",
        "config": {"workload": WORKLOAD, "shapes": 343, "flop_per_step": flops_step,
                   "compulsory_bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2: each shape has its own A, B, C "
                         "(%.2f GB per step vs 129 MB L2); no explicit flush" % (bytes_step / 1e9),
                   "layout": "TN", "accumulate": "fp32",
                   "launch": "one step = the 343 gemm_run launches captured once as a CUDA "
                             "graph and replayed; eager = one gemm_run call per shape"},
        "eager": {"value": round(flops_step / (ms_step_eager * 1e-3) / 1e12, 3),
                  "unit": UNIT, "ms_per_step": round(ms_step_eager, 4)},
        "gpu_launches": len(items) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }

    # ---- roofline of the step: per shape max(tensor, HBM, launch floor), summed.
    probe = mma_probe(sms, stream)
    per_clk = probe["grid_%d" % sms]["flop_per_clk_per_sm"]
    sm_max = (clocks or {}).get("sm_max_mhz") or 2070.0
    theo = sms * sm_max * 1e6 * per_clk / 1e12
    p_tensor = max(theo, peaks["bf16_tflops"])          # the stricter denominator
    floor_graph = launch_floor_us(stream, sms, graph=True)
    classes = {}
    t_roof = 0.0
    t_roof_meas = 0.0
    for item in items:
        w = item[0]
        tt = w.flops / (p_tensor * 1e12) * 1e6
        th = w.compulsory_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        tr = max(tt, th, floor_graph)
        t_roof += tr
        t_roof_meas += max(w.flops / (peaks["bf16_tflops"] * 1e12) * 1e6, th, floor_graph)
        kind = "tensor" if tr == tt else ("hbm" if tr == th else "launch")
        c = classes.setdefault(kind, {"shapes": 0, "t_roof_us": 0.0, "items": []})
        c["shapes"] += 1
        c["t_roof_us"] += tr
        c["items"].append(item)
    for kind, c in classes.items():
        # each class's shapes alone, in sweep order, as one graph (same launch regime)
        sub = capture_step(c.pop("items"), stream)
        ms_c, _, _ = time_graph(sub, max(5, args.steps), 3, stream)
        c["t_graph_us"] = round(ms_c * 1e3 / max(5, args.steps), 1)
        c["frac"] = round(c["t_roof_us"] / c["t_graph_us"], 4)
        c["t_roof_us"] = round(c["t_roof_us"], 1)
        del sub
    traffic, traffic_note = stored_traffic()
    line["roofline"] = {
        "bound": "mixed",
        "achieved": round(value, 2),
        "peak": round(flops_step / (t_roof * 1e-6) / 1e12, 2),
        "unit": "TFLOP/s",
        "frac": round(t_roof / (ms_step * 1e3), 4),
        "traffic": traffic,
        "rule": "per shape t_roof = max(2MNK / tensor peak, compulsory bytes / HBM, launch "
                "floor); peak = step FLOP / sum t_roof (the throughput the 343-shape mix "
                "allows), frac = sum t_roof / timed step = achieved / peak",
        "tensor_peak_tflops": round(p_tensor, 1),
        "tensor_peak_source": "stricter of measured bf16 burst (%s, %.1f) and theoretical "
                              "%d SMs x %.0f MHz x %.1f FLOP/clk/SM (tcgen05 issue-rate probe, "
                              "%.1f)" % (peak_src, peaks["bf16_tflops"], sms, sm_max, per_clk, theo),
        "hbm_gbs": peaks["hbm_gbs"],
        "launch_floor_graph_us": round(floor_graph, 3),
        "frac_with_measured_tensor_peak": round(t_roof_meas / (ms_step * 1e3), 4),
        "frac_of_tensor_peak": round(value / p_tensor, 4),
        "by_class": classes,
        "traffic_note": traffic_note,
        "mma_probe": probe,
    }

    if not args.skip_extras:
        floor = launch_floor_us(stream, sms)
        times = per_shape_times(items, stream)
        line["sweep_isolated"] = {
            "launch_floor_eager_us": round(floor, 3),
            "t_meas_us_sum": round(sum(times.values()) * 1e3, 1),
            "headline_128x2048x128_us": round(times.get("sweep_128x2048x128_f16", 0) * 1e3, 3),
            "skinny_64x4096x64_us": round(times.get("sweep_64x4096x64_f16", 0) * 1e3, 3),
            "note": "each launch alone between CUDA events (no launch overlap)",
        }
        e2e_ms, h2d, d2h, busy_ms = e2e_sweep(items, stream, steps=max(3, min(20, args.steps)))
        line["e2e"] = {"value": round(flops_step / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_ms, 3),
                       "h2d_busy_ms_per_step": round(busy_ms[0], 3),
                       "d2h_busy_ms_per_step": round(busy_ms[1], 3),
                       "link_busy_frac": round(max(busy_ms) / e2e_ms, 4),
                       "note": "busy: the summed durations of the step's host-to-device and "
                               "device-to-host copies, timed on their streams in three "
                               "untimed steps run the same way (median); link_busy_frac = "
                               "the busier direction / the timed step (two separate "
                               "measurements: near 1, within a percent or so either way, "
                               "means the step is bound by the host link)"}
        del graph
        for _, plan, *_ in items:
            plan.close()
        del items
        torch.cuda.empty_cache()
        line["named"] = named_workloads(stream, peaks, p_tensor, floor, sms,
                                        (clocks or {}).get("sm_max_mhz") or 2070.0)
        line["server_mode"] = server_mode(stream)
        cpu = cpu_oracle_sample()
        named_cpu, single, threads = cpu_oracle_named()
        cpu["single_thread_headline"] = single
        cpu["named"] = named_cpu
        cpu["note"] = ("the oracle as it stands (fp64, plain i-j-k loop, rows over %d host "
                       "threads); named: full problem where it takes under 2 s, else a 64-row "
                       "block extrapolated linearly in M" % threads)
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- reference arm

def reference(args):
    """The CPU oracle, as it stands, on a bounded sample of the sweep per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    import oracle
    oracle.build()
    threads = oracle.max_threads()
    shapes = workloads.sweep_shapes()
    order = torch.randperm(len(shapes), generator=torch.Generator().manual_seed(7)).tolist()
    rows = 16
    cache = {}

    def operands(i):
        if i not in cache:
            w = shapes[i]
            A, B = inputs.make_operands(min(rows, w.M), w.N, w.K, "f16")
            cache[i] = (w, A.view(torch.int16).numpy().view(np.uint16),
                        B.view(torch.int16).numpy().view(np.uint16))
        return cache[i]

    def step(n):
        w, a, b = operands(order[n % len(order)])
        t0 = time.perf_counter()
        oracle.gemm_tn_half(a, b, 0, threads)
        return time.perf_counter() - t0, 2 * a.shape[0] * w.N * w.K

    for n in range(args.warmup):
        step(n)
    el = 0.0
    flops = 0
    for n in range(args.warmup, args.warmup + args.steps):
        dt, f = step(n)
        el += dt
        flops += f
    value = flops / el / 1e12
    sample = ("one sweep shape per step (seeded rotation over the 343), rows [0,%d) of A "
              "against all of B; %.3g FLOP over %d steps" % (rows, flops, args.steps))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "shapes": 343, "sample_rows_per_shape": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def tma_sweep():
    """The tutorial page's experiment on this GPU: n = 4 Mi floats, 4 KiB tiles, 64 tiles per
    256-thread block; CUDA-event median of 25 launches per (mode, fma_iters)."""
    import dense_gemm_hgemm_gb300 as g
    g.build_library()
    n = 4_194_304
    x = torch.randn(n, device="cuda")
    y = torch.empty_like(x)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    modes = ("sync", "bulk1d", "tensor2d", "pipe2")
    rows = []
    for iters in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        rec = {"fma_iters": iters}
        for m in modes:
            for _ in range(3):
                g.tma_intensity_run(m, iters, 0.999, 0.001, x, y, 2048, err, stream)
            ts = []
            for _ in range(25):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.tma_intensity_run(m, iters, 0.999, 0.001, x, y, 2048, err, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            rec[m + "_ms"] = round(statistics.median(ts), 5)
        for m in modes[1:]:
            rec["speedup_" + m] = round(rec["sync_ms"] / rec[m + "_ms"], 3)
        rows.append(rec)
    assert int(err.item()) == 0
    print(json.dumps({"experiment": "tma_intensity", "gpu": torch.cuda.get_device_name(0),
                      "n": n, "tile_bytes": 4096, "tiles_per_block": 64, "block": 256,
                      "blocks": n // 65536, "timing": "CUDA-event median of 25", "rows": rows}))


def main(argv=None):
    args = parse_args(argv)
    if args.tma_sweep:
        tma_sweep()
        return
    if args.warmup < 3 and not args.ncu_steps:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
