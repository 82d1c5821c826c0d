#!/usr/bin/env python
"""Benchmark: the fp16 TN GEMM shape sweep (343 shapes, M, N, K in {64..4096}).

One step = one gemm_run for every shape of the sweep, each on its own
device-resident A, B, C (2.77 GB of distinct operands per step, more than the
129 MB L2, so no step finds the previous step's data in L2).  `value` is the
whole-job throughput sum(2*M*N*K) / step time in TFLOP/s, over all ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Also reported on that line (measured outside
the timed region): `e2e` (the same sweep through the C ABI with operands copied
from pinned host memory and C copied back inside the timed region), `named`
(µs/call and TFLOP/s of the named workloads: 64x4096x64 and 128x2048x128 fp16,
8192^3 fp16, the 4096x14336x4096 bf16 FFN shape, 4096^3 int8->int32), the
roofline of the sweep, GPU clocks sampled during the timed region, and the CPU
oracle timed on a bounded sample (`cpu_baseline`).

--impl reference times the CPU oracle (the only reference this method has) on a
bounded sample of the same sweep, on the host cores, and prints the same line
with "impl": "reference".
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
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class Dist:
    """Rank bookkeeping; torch.distributed only when launched with WORLD_SIZE > 1."""

    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.pg = dist
            self.backend = backend

    def barrier(self):
        if self.pg is not None:
            if self.backend == "nccl":
                self.pg.barrier(device_ids=[self.local_rank])
            else:
                self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


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


# Sources that build no kernel a GEMM launch runs (the int8 widening / fill /
# empty kernels, the TMA intensity sweep, the CPython entry points): left out
# of the digest.
_DIGEST_SKIP = ("gemm_aux.cu", "tma_intensity.cu", "gemm_pycall.c")


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


def time_sweep(items, dist, steps, warmup, stream, sampler=None):
    for _ in range(warmup):
        run_step(items, stream)
    torch.cuda.synchronize()
    dist.barrier()
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
    dist.barrier()
    ms = e0.elapsed_time(e1)
    return ms, wall, clocks


def capture_step(items, stream):
    """One sweep step (all 343 gemm_run launches) captured as a CUDA graph: the
    same kernels, parameters and buffers, replayed without per-launch host work."""
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run_step(items, stream)
    torch.cuda.synchronize()
    return graph


def time_graph(graph, dist, steps, warmup, stream, sampler=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    dist.barrier()
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
    dist.barrier()
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

    def one(compute=True, copy_out=True):
        for g in range(groups):
            lo, hi = rng_in[g]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_mm[g])          # the previous step's GEMMs read this range
                d_in[lo:hi].copy_(h_in[lo:hi], non_blocking=True)
                ev_in[g].record(s_in)
            stream.wait_event(ev_in[g])
            stream.wait_event(ev_out[g])           # the previous step's copy-out of this range
            if compute:
                for plan, dA, dB, dC in views[bounds[g]:bounds[g + 1]]:
                    plan.run(dA, dB, dC, stream)
            ev_mm[g].record(stream)
            if not copy_out:
                continue
            lo, hi = rng_out[g]
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_mm[g])
                h_out[lo:hi].copy_(d_out[lo:hi], non_blocking=True)
                ev_out[g].record(s_out)

    one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    # the step's host-to-device copies alone (the larger direction; the results
    # travel back concurrently): the floor the host link sets for this step
    one(compute=False, copy_out=False)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one(compute=False, copy_out=False)
    torch.cuda.synchronize()
    copy_ms = (time.perf_counter() - t0) * 1e3 / steps
    # results came back: spot-check one C against the device copy of the eager run
    mid = len(items) // 2
    w, plan, A, B, C = items[mid]
    oc = out_off[mid]
    got = h_out[oc:oc + C.numel() * 2].view(torch.float16).view(C.shape)
    one()   # leave every result in place for the check below
    torch.cuda.synchronize()
    if not torch.equal(got.view(torch.int16), C.cpu().view(torch.int16)):
        raise RuntimeError("e2e: copied-back result differs from the device result")
    return wall * 1e3 / steps, h2d, d2h, copy_ms


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


def named_workloads(stream, peaks, floor_us, sms):
    """Warm µs/call (back-to-back on the same buffers, median of 5 repeats of a
    >= 20 ms loop) and TFLOP/s with the roofline fraction for each named shape;
    cold µs/call (L2 flushed before every call) for the two skinny shapes."""
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
            reps = max(10, min(5000, int(20.0 / one)))
            samples = []
            for _ in range(5):
                e0.record(stream)
                for _ in range(reps):
                    plan.run(A, B, C, stream)
                e1.record(stream)
                torch.cuda.synchronize()
                samples.append(e0.elapsed_time(e1) * 1e3 / reps)
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
        t_tensor = w.flops / (peaks["bf16_tflops"] * 1e12) * 1e6
        t_hbm = w.compulsory_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        t_roof = max(t_tensor, t_hbm, floor_us)
        bound = "tensor" if t_roof == t_tensor else ("hbm" if t_roof == t_hbm else "launch")
        out[w.name] = {
            "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype, "us_per_call": round(us, 3),
            "us_per_call_cold_l2": round(cold, 3) if cold is not None else None,
            ("TOPS" if w.dtype == "i8" else "TFLOPS"): round(tflops, 2),
            "roofline_bound": bound, "roofline_us": round(t_roof, 3),
            "roofline_frac": round(t_roof / us, 4),
            "tensor_frac_of_measured_peak": round(tflops / peaks["bf16_tflops"], 4),
            "config": cfg,
        }
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


def cpu_oracle_sample(budget_s: float = 15.0, rows: int = 64):
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


def profile_one(spec, calls, stream):
    """`calls` launches of one shape with the table's configuration (for ncu)."""
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
    with g.Plan(M, N, K, dtype) as plan:
        for _ in range(calls):
            plan.run(A, B, C, stream)
        plan.check(stream)
        print(json.dumps({"shape": [M, N, K, dtype], "config": plan.config, "calls": calls}))


def ours(args):
    dist = Dist()
    torch.cuda.set_device(dist.local_rank)
    import dense_gemm_hgemm_gb300 as g
    g.build_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    sms = torch.cuda.get_device_properties(dist.local_rank).multi_processor_count
    if args.ncu_steps and args.shape:
        profile_one(args.shape, args.ncu_steps, stream)
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

    # Eager: one gemm_run (ctypes -> C ABI -> cudaLaunchKernelEx) per shape.
    ms_e, wall_e, _ = time_sweep(items, dist, args.steps, args.warmup, stream)
    for _, plan, *_ in items:
        plan.check(stream)     # raises if any kernel gave up on a wait
    ms_step_eager = dist.max(ms_e) / args.steps
    # Headline: the same step launched from a captured CUDA graph (the launch
    # overhead of 343 mostly tiny GEMMs is host work, not GEMM work).
    graph = capture_step(items, stream)
    sampler = ClockSampler(dist.local_rank)
    ms, wall, clocks = time_graph(graph, dist, args.steps, args.warmup, stream, sampler)
    for _, plan, *_ in items:
        plan.check(stream)
    ms_max = dist.max(ms)
    ms_step = ms_max / args.steps
    value = dist.world * flops_step / (ms_step * 1e-3) / 1e12
    per_gpu = flops_step / (ms_step * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded N(0,1) fp16 operands per shape, generated on the device)",
        "config": {"workload": WORKLOAD, "shapes": 343, "flop_per_step": flops_step,
                   "compulsory_bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2: each shape has its own A, B, C "
                         "(%.2f GB per step vs 129 MB L2); no explicit flush" % (bytes_step / 1e9),
                   "replicas": dist.world, "layout": "TN", "accumulate": "fp32",
                   "launch": "one step = the 343 gemm_run launches captured once as a CUDA "
                             "graph and replayed; eager = one gemm_run call per shape"},
        "eager": {"value": round(dist.world * flops_step / (ms_step_eager * 1e-3) / 1e12, 3),
                  "unit": UNIT, "ms_per_step": round(ms_step_eager, 4)},
        "gpu_launches": len(items) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    traffic, traffic_note = stored_traffic()
    line["roofline"] = {
        "bound": "tensor", "achieved": round(per_gpu, 2),
        "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
        "frac": round(per_gpu / peaks["bf16_tflops_sustained"], 4),
        "traffic": traffic,
        "peak_source": "bf16_tflops_sustained of %s (fp16 dense rate equals bf16)" % peak_src,
        "frac_of_burst_peak": round(per_gpu / peaks["bf16_tflops"], 4),
        "kernel": "gemm_tn_kernel (all sweep launches; average launch = step/343)",
        "traffic_note": traffic_note,
    }

    if not args.skip_extras and dist.rank == 0:
        floor = launch_floor_us(stream, sms)
        floor_graph = launch_floor_us(stream, sms, graph=True)
        times = per_shape_times(items, stream)
        t_meas = t_roof = t_roof_graph = 0.0
        classes = {}
        for w, *_ in items:
            us = times[w.name] * 1e3
            tt = w.flops / (peaks["bf16_tflops"] * 1e12) * 1e6
            th = w.compulsory_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6
            tr = max(tt, th, floor)
            t_roof_graph += max(tt, th, floor_graph)
            kind = "tensor" if tr == tt else ("hbm" if tr == th else "launch")
            c = classes.setdefault(kind, {"shapes": 0, "t_meas_us": 0.0, "t_roof_us": 0.0})
            c["shapes"] += 1
            c["t_meas_us"] += us
            c["t_roof_us"] += tr
            t_meas += us
            t_roof += tr
        for c in classes.values():
            c["frac"] = round(c["t_roof_us"] / c["t_meas_us"], 4)
            c["t_meas_us"] = round(c["t_meas_us"], 1)
            c["t_roof_us"] = round(c["t_roof_us"], 1)
        head = workloads.HEADLINE_SWEEP.name.replace("hgemm_tn_", "sweep_").replace("_f16", "_f16")
        line["sweep_roofline"] = {
            "launch_floor_us": round(floor, 3),
            "launch_floor_graph_us": round(floor_graph, 3),
            "t_roof_us_sum": round(t_roof_graph, 1),
            "frac_of_timed_step": round(t_roof_graph / (ms_step * 1e3), 4),
            "t_roof_us_sum_eager_floor": round(t_roof, 1),
            "frac_of_eager_step": round(t_roof / (ms_step_eager * 1e3), 4),
            "t_meas_us_sum_isolated": round(t_meas, 1),
            "frac_isolated": round(t_roof / t_meas, 4), "by_bound_isolated": classes,
            "rule": "per shape t_roof = max(2MNK/bf16 burst peak, compulsory bytes/HBM, "
                    "launch floor of an empty kernel launched like the GEMM: from a graph "
                    "for the timed (graph) step, one call at a time for the eager step and "
                    "the isolated times); frac_of_timed_step = sum t_roof / timed "
                    "ms_per_step; *_isolated = each launch timed alone between events (no "
                    "launch overlap)",
            "headline_128x2048x128_us_in_sweep": round(times.get("sweep_128x2048x128_f16", 0) * 1e3, 3),
        }
        e2e_ms, h2d, d2h, copy_ms = e2e_sweep(items, stream, steps=max(3, min(20, args.steps)))
        line["e2e"] = {"value": round(flops_step / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_ms, 3),
                       "h2d_only_ms_per_step": round(copy_ms, 3),
                       "frac_of_h2d_floor": round(copy_ms / e2e_ms, 4),
                       "note": "h2d_only: the step's host-to-device copies alone (no GEMM, no "
                               "copy back); the step is bound by the host link when the "
                               "fraction is near 1"}
        del graph
        for _, plan, *_ in items:
            plan.close()
        del items
        torch.cuda.empty_cache()
        line["named"] = named_workloads(stream, peaks, floor, sms)
        line["server_mode"] = server_mode(stream)
        line["cpu_baseline"] = cpu_oracle_sample()
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


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
