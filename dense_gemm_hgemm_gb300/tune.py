"""Measured per-shape configuration sweep -> csrc/gemm_config_table.inc.

The pages pick tile shape, pipeline depth and swizzle with an RL agent; this
library picks (tile width, split-K, raster band) per shape by timing every
candidate on the target GPU and keeping the fastest.

  python -m dense_gemm_hgemm_gb300.tune --out tuned.json      # on the GPU
  python -m dense_gemm_hgemm_gb300.tune --emit tuned.json     # writes the .inc

Timing regime: each call with L2 flushed first (a 256 MB write on the same
stream), CUDA events around the call, median of repeats -- the situation of a
shape inside the 343-shape benchmark step, where every shape's operands come
from HBM.  Warm back-to-back µs/call is recorded alongside.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

PKG = os.path.dirname(os.path.abspath(__file__))
TABLE = os.path.join(PKG, "csrc", "gemm_config_table.inc")
TUNED_JSON = os.path.join(PKG, "tuned_configs.json")


def candidates(M, N, K, dtype, sms):
    bns = (64, 128) if dtype == "i8" else (64, 128, 256)
    num_kb = -(-K // 64)
    out = []
    for bn in bns:
        tiles = -(-M // 128) * -(-N // bn)
        for s in (1, 2, 3, 4, 6, 8, 12, 16):
            if s > 1 and (num_kb < 2 * s or tiles * s > 4 * sms or tiles >= sms):
                continue
            groups = (16,)
            if tiles >= 4 * sms and s == 1:
                groups = (4, 8, 16, 32)
            for g in groups:
                out.append({"block_n": bn, "split_k": s, "raster_group": g, "split_mode": 0})
            per = -(-num_kb // s) if s > 1 else 0
            if s in (2, 4, 8) and -(-num_kb // per) == s:
                out.append({"block_n": bn, "split_k": s, "raster_group": 16, "split_mode": 1})
        if dtype != "i8" and bn >= 128 and M > 128:
            # SM pair: 256-row tiles (raster bands count 256-row blocks)
            pair_tiles = -(-M // 256) * -(-N // bn)
            groups = (4, 8, 16) if pair_tiles >= 2 * sms else (8,)
            for g in groups:
                out.append({"block_n": bn, "split_k": 1, "raster_group": g, "split_mode": 0,
                            "cta_pair": 1})
    return out


def _time(plan, A, B, C, stream, flush, reps_cold=7, reps_warm=20):
    import torch
    for _ in range(3):
        plan.run(A, B, C, stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    cold = []
    for _ in range(reps_cold):
        with torch.cuda.stream(stream):
            flush.add_(1)
        e0.record(stream)
        plan.run(A, B, C, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        cold.append(e0.elapsed_time(e1) * 1e3)
    e0.record(stream)
    for _ in range(reps_warm):
        plan.run(A, B, C, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    plan.check(stream)
    return statistics.median(cold), e0.elapsed_time(e1) * 1e3 / reps_warm


def sweep(out_path, only=None):
    import torch

    import dense_gemm_hgemm_gb300 as g
    from dense_gemm_hgemm_gb300 import inputs, workloads
    g.build_library()
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    stream = torch.cuda.Stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    shapes = [(w.M, w.N, w.K, w.dtype) for w in workloads.sweep_shapes()]
    shapes += [(w.M, w.N, w.K, w.dtype) for w in workloads.NAMED
               if (w.M, w.N, w.K, w.dtype) not in shapes]
    if only:
        shapes = [s for s in shapes if s in only]
    results = []
    t_start = time.time()
    for M, N, K, dtype in shapes:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(inputs.shape_seed(M, N, K, dtype))
        if dtype == "i8":
            A = torch.randint(-128, 128, (M, K), generator=gen, device="cuda", dtype=torch.int8)
            B = torch.randint(-128, 128, (N, K), generator=gen, device="cuda", dtype=torch.int8)
        else:
            A = torch.randn(M, K, generator=gen, device="cuda").to(inputs.TORCH_DTYPE[dtype])
            B = torch.randn(N, K, generator=gen, device="cuda").to(inputs.TORCH_DTYPE[dtype])
        C = torch.empty(M, N, device="cuda", dtype=inputs.OUT_DTYPE[dtype])
        rec = {"M": M, "N": N, "K": K, "dtype": dtype, "candidates": []}
        for cfg in candidates(M, N, K, dtype, sms):
            with g.Plan(M, N, K, dtype, cfg) as plan:
                cold, warm = _time(plan, A, B, C, stream, flush)
            rec["candidates"].append({**cfg, "cold_us": round(cold, 3), "warm_us": round(warm, 3)})
        best = min(rec["candidates"], key=lambda c: (c["cold_us"], c["warm_us"]))
        rec["best"] = {k: best.get(k, 0) for k in ("block_n", "split_k", "raster_group",
                                                   "split_mode", "cta_pair")}
        rec["model"] = g.gemm_select_config(M, N, K, dtype, sms)
        results.append(rec)
        del A, B, C
    doc = {"gpu": props.name, "sms": sms, "when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()),
           "seconds": round(time.time() - t_start, 1),
           "regime": "L2 flushed before each call; median of 7; warm = back-to-back mean of 20",
           "shapes": results}
    with open(out_path, "w") as f:
        json.dump(doc, f, indent=1)
    print("tuned %d shapes in %.1f s -> %s" % (len(results), doc["seconds"], out_path))


def emit(json_path, table_path=TABLE):
    """Write the C table of best configurations from a sweep's JSON."""
    with open(json_path) as f:
        doc = json.load(f)
    code = {"f16": 0, "bf16": 1, "i8": 2}
    lines = [
        "// gemm_config_table.inc -- measured per-shape configurations.",
        "// Written by dense_gemm_hgemm_gb300/tune.py from %s" % os.path.basename(json_path),
        "// (%s, %d SMs, %s; %s)." % (doc["gpu"], doc["sms"], doc["when"], doc["regime"]),
        "// Fields: M, N, K, dtype (0 f16, 1 bf16, 2 i8), block_n, split_k, raster_group,",
        "// split_mode (0 workspace, 1 cluster), cta_pair (0 one SM, 1 SM pair).",
        "static const TableEntry kTunedTable[] = {",
    ]
    n = 0
    for r in doc["shapes"]:
        b = r["best"]
        lines.append("    {%d, %d, %d, %d, %d, %d, %d, %d, %d}," % (
            r["M"], r["N"], r["K"], code[r["dtype"]], b["block_n"], b["split_k"],
            b["raster_group"], b.get("split_mode", 0), b.get("cta_pair", 0)))
        n += 1
    lines.append("};")
    lines.append("static const int kTunedCount = %d;" % n)
    with open(table_path, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote %d entries to %s" % (n, table_path))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=None, help="run the sweep on the GPU and write this JSON")
    ap.add_argument("--emit", default=None, help="write the C table from this JSON")
    args = ap.parse_args(argv)
    if args.out:
        sweep(args.out)
    if args.emit:
        emit(args.emit)
    if not args.out and not args.emit:
        ap.print_help()
        return 2
    return 0


if __name__ == "__main__":
    sys.exit(main())
