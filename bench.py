"""Benchmark harness: AWQ W4A16 decode GEMV sweep (Llama-2-7B linear shapes) on GB300.

One step = one pass of the hot path over the decode workload: 16 GEMV calls,
M in {1, 2, 4, 8} x (K, N) in {(4096, 12288) qkv, (4096, 4096) o_proj,
(4096, 22016) gate_up, (11008, 4096) down}, group size 128, each call with its own
weight buffers (405 MB of packed weights per step, more than 3x the 126 MB L2, so
every step streams its weights from HBM).

Timed region (device value): the step captured as one CUDA graph, replayed K times
between CUDA events on the launching stream, barrier + synchronize on both sides,
max over ranks.  e2e: the same step through the public Python API (one call per
layer call), with all of the step's activations copied in from pinned host memory and
all of its outputs copied back, every step: calls grouped into runs of at least 8 MB
of copies, each run's copies on their own streams so that they overlap the
neighbouring runs' compute (the decode step is one run: one copy in, one out).  The CPU baseline and `--impl reference` time the numpy oracle on a
bounded sample of the same workload.

Other workloads (`--workload prefill|crossover|w4a8`) print the same line for the
other sweeps; the default is the decode sweep.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_weight_only_awq_gb300 import synth  # noqa: E402

WORKLOAD_FILTER = {"only": None, "ms": None}
METRIC = "W4A16 group-quant GEMM TFLOP/s & HBM GB/s vs M; % of roofline on 1 GB300"


# ------------------------------------------------------------------ workloads
def w4a16_bytes(M, K, N):
    return K * N / 2 + 2 * N * K / 128 + 4 * (K / 128) * (N / 8) + 2 * M * K + 2 * M * N


def w4a8_bytes(M, K, N):
    return K * N / 2 + 2 * N + M * K + 4 * M + 2 * M * N


def awq_linear_gemv_max():
    """Largest token count the library's dispatch (awq_linear) sends to the GEMV kernel."""
    return 16


def workload_calls(workload, only=None, ms=None):
    """List of (kind, name, M, K, N) for one step (optionally filtered by shape name / M)."""
    calls = _workload_calls(workload)
    if only:
        calls = [c for c in calls if c[1] in only.split(",")]
    if ms:
        calls = [c for c in calls if c[2] in ms]
    if not calls:
        raise ValueError("the filters leave no call")
    return calls


def _workload_calls(workload):
    if workload == "decode":
        return [("gemv", n, m, k, nn) for n, k, nn in synth.LLAMA2_7B_DECODE for m in synth.DECODE_M]
    if workload == "prefill":
        return [("gemm", n, m, k, nn) for n, k, nn in synth.MISTRAL_7B_PREFILL for m in synth.PREFILL_M]
    if workload == "crossover":
        out = []
        for n, k, nn in synth.LLAMA31_8B_STACK:
            for m in synth.CROSSOVER_M:
                out.append(("gemv" if m <= awq_linear_gemv_max() else "gemm", n, m, k, nn))
        return out
    if workload == "w4a8":
        k, nn = synth.W4A8_SHAPE
        return [("w4a8", "w4a8", m, k, nn) for m in synth.W4A8_M]
    raise ValueError(workload)


def call_bytes(kind, M, K, N):
    return w4a8_bytes(M, K, N) if kind == "w4a8" else w4a16_bytes(M, K, N)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[1].isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [int(r[1]) for r in rows]
        reasons = set()
        for r in rows:
            for name, val in (("hw_slowdown", r[5]), ("hw_thermal_slowdown", r[6]),
                              ("sw_thermal_slowdown", r[7]), ("sw_power_cap", r[8])):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][2]), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None,
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)
def oracle_sample(workload, budget_s, seed=7):
    """Time the oracle on a bounded, seeded sample of the workload; returns (bytes/s, description).

    The sample: every call of one step, restricted to 256 output columns, repeated
    until about `budget_s` seconds of oracle work have been spent (at least one pass).
    """
    import oracle

    calls = workload_calls(workload)
    cols = 256
    problems = []
    for i, (kind, name, M, K, N) in enumerate(calls):
        if kind == "w4a8":
            problems.append((kind, M, K, synth.w4a8_problem(M, K, cols, seed=seed + i)))
        else:
            problems.append((kind, M, K, synth.awq_problem(M, K, cols, seed=seed + i)))
    done_bytes = 0.0
    spent = 0.0
    passes = 0
    while passes == 0 or spent < budget_s:
        for kind, M, K, p in problems:
            t0 = time.perf_counter()
            if kind == "w4a8":
                xq, s = oracle.quant_act(p["x"])
                oracle.w4a8_linear(xq, s, p["wq"], p["s_ch"])
                done_bytes += w4a8_bytes(M, K, cols)
            else:
                oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
                done_bytes += w4a16_bytes(M, K, cols)
            spent += time.perf_counter() - t0
        passes += 1
    desc = (f"{passes} pass(es) over all {len(calls)} calls of one step, each restricted to {cols} seeded "
            f"output columns; numpy oracle, one thread, {spent:.1f} s")
    return done_bytes / spent, desc


def run_oracle_subprocess(workload, budget_s):
    """Run the oracle sample in a child process pinned to one BLAS / OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench; v, d = bench.oracle_sample(%r, %r); print(json.dumps({'v': v, 'd': d}))"
            % (workload, budget_s))
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    res = json.loads(out.stdout.strip().splitlines()[-1])
    return res["v"], res["d"], 1


# ------------------------------------------------------------------ GPU arm
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def build_inputs(torch, workload, device):
    """Per-call device buffers (weights distinct per call).  The activations and outputs of all calls
    are views into one device buffer each, mirrored by one pinned host buffer each, so that the e2e
    step moves them with one host-to-device and one device-to-host copy."""
    bufs = []
    for i, (kind, name, M, K, N) in enumerate(workload_calls(workload, **WORKLOAD_FILTER)):
        seed = 10_000 + i
        if kind == "w4a8":
            p = synth.w4a8_problem(M, K, N, seed=seed)
            b = {"x": torch.from_numpy(p["x"]).to(device), "wq": torch.from_numpy(p["wq"]).to(device),
                 "s_ch": torch.from_numpy(p["s_ch"]).to(device)}
            b["xq"] = torch.empty((M, K), dtype=torch.int8, device=device)
            b["s_tok"] = torch.empty((M,), dtype=torch.float32, device=device)
        else:
            p = synth.awq_problem(M, K, N, seed=seed)
            b = {k: torch.from_numpy(p[k]).to(device) for k in ("x", "qweight", "qzeros", "scales")}
        b["x_np"] = p["x"]
        b["meta"] = (kind, name, M, K, N)
        bufs.append(b)
    # every view starts on a 16-byte boundary: M * K and M * N are multiples of 8 halves
    nx = sum(b["meta"][2] * b["meta"][3] for b in bufs)
    ny = sum(b["meta"][2] * b["meta"][4] for b in bufs)
    packed = {"x": torch.empty(nx, dtype=torch.float16, device=device),
              "x_host": torch.empty(nx, dtype=torch.float16).pin_memory(),
              "y": torch.empty(ny, dtype=torch.float16, device=device),
              "y_host": torch.empty(ny, dtype=torch.float16).pin_memory()}
    ox = oy = 0
    for b in bufs:
        _, _, M, K, N = b["meta"]
        b["x"] = packed["x"][ox:ox + M * K].view(M, K)
        b["x"].copy_(torch.from_numpy(b.pop("x_np")))
        packed["x_host"][ox:ox + M * K].copy_(b["x"].view(-1).cpu())
        b["y"] = packed["y"][oy:oy + M * N].view(M, N)
        ox += M * K
        oy += M * N
    bufs[0]["packed"] = packed
    return bufs


def e2e_segments(torch, bufs, min_bytes):
    """Runs of consecutive calls whose activations and outputs span at least `min_bytes`; each run is
    one contiguous range of the packed buffers, so it moves with one copy in and one copy out."""
    packed = bufs[0]["packed"]
    segs, start, ox, oy, nbytes = [], 0, 0, 0, 0
    x0, y0 = 0, 0
    for i, b in enumerate(bufs):
        _, _, M, K, N = b["meta"]
        ox += M * K
        oy += M * N
        nbytes += 2 * (M * K + M * N)
        if nbytes >= min_bytes or i == len(bufs) - 1:
            segs.append({"bufs": bufs[start:i + 1],
                         "x": packed["x"][x0:ox], "x_host": packed["x_host"][x0:ox],
                         "y": packed["y"][y0:oy], "y_host": packed["y_host"][y0:oy],
                         "ev_in": torch.cuda.Event(), "ev_out": torch.cuda.Event()})
            start, x0, y0, nbytes = i + 1, ox, oy, 0
    return segs


def issue_step(awq, bufs, stream):
    """All calls of one step on `stream`; returns the number of kernels launched."""
    launches = 0
    for b in bufs:
        kind, _, M, K, N = b["meta"]
        if kind == "gemv":
            awq.awq_gemv(b["x"], b["qweight"], b["qzeros"], b["scales"], out=b["y"], stream=stream)
            launches += 1
        elif kind == "gemm":
            awq.awq_gemm(b["x"], b["qweight"], b["qzeros"], b["scales"], out=b["y"], stream=stream)
            launches += 1
        else:
            awq.w4a8_linear(b["x"], b["wq"], b["s_ch"], out=b["y"], s_tok=b["s_tok"], stream=stream)
            launches += 2  # quantize (fp16 codes into the workspace), then the GEMV or the tensor-core GEMM
    return launches


def max_over_ranks(values, torch, dist, device):
    """Element-wise maximum of `values` (times) over all ranks of `dist` (None: one rank)."""
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_rate(units_per_rank_step, world, step_s):
    """Weak scaling: every rank processes `units_per_rank_step` per step; the job's rate is all ranks'
    units over the slowest rank's step time."""
    return units_per_rank_step * world / step_s


def gpu_arm(args, rank, world, torch, dist):
    from bit_weight_only_awq_gb300 import build as awq_build
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq

    device = torch.device("cuda", torch.cuda.current_device())
    bufs = build_inputs(torch, args.workload, device)
    calls = [b["meta"] for b in bufs]
    step_bytes = sum(call_bytes(k, M, K, N) for k, _, M, K, N in calls)
    step_flops = sum(2.0 * M * K * N for _, _, M, K, N in calls)

    stream = torch.cuda.Stream(device=device)
    # pre-size the shared workspace for the largest call, then warm every code path once
    for b in bufs:
        kind, _, M, K, N = b["meta"]
        op = {"gemv": awq.OP_GEMV, "gemm": awq.OP_GEMM, "w4a8": awq.OP_W4A8_GEMM}[kind]
        awq.device_workspace(awq.awq_workspace_bytes(op, M, K, N, 0), device)
    with torch.cuda.stream(stream):
        launches_per_step = issue_step(awq, bufs, stream)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        issue_step(awq, bufs, stream)
    torch.cuda.synchronize()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        graph.replay()
    barrier()

    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index) as clk:
        barrier()
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(args.steps):
                graph.replay()
            stop.record(stream)
        barrier()
    ms = start.elapsed_time(stop)
    clocks = clk.summary()

    # e2e through the public API: every step copies all activations in from pinned host memory and all
    # outputs back.  Consecutive calls are grouped into segments of at least 8 MB of copies; each
    # segment's input copy (copy-in stream), its calls (compute stream) and its output copy (copy-out
    # stream) are chained by events, so that one segment's copies overlap the neighbours' compute.
    segs = e2e_segments(torch, bufs, min_bytes=8 << 20)
    h2d = torch.cuda.Stream(device=device)
    d2h = torch.cuda.Stream(device=device)

    def e2e_step():
        for seg in segs:
            with torch.cuda.stream(h2d):
                seg["x"].copy_(seg["x_host"], non_blocking=True)
                seg["ev_in"].record(h2d)
            stream.wait_event(seg["ev_in"])
            with torch.cuda.stream(stream):
                issue_step(awq, seg["bufs"], stream)
                seg["ev_out"].record(stream)
            d2h.wait_event(seg["ev_out"])
            with torch.cuda.stream(d2h):
                seg["y_host"].copy_(seg["y"], non_blocking=True)
        d2h.synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_step()
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    barrier()
    e2e_s = time.perf_counter() - t0

    ms, e2e_s = max_over_ranks([ms, e2e_s], torch, dist, device)
    return {
        "awq": awq, "calls": calls, "step_bytes": step_bytes, "step_flops": step_flops, "ms": ms,
        "e2e_s": e2e_s, "clocks": clocks, "launches_per_step": launches_per_step,
        "h2d": sum(2 * M * K for _, _, M, K, _ in calls), "d2h": sum(2 * M * N for _, _, M, _, N in calls),
    }


def dominant_kernel(workload):
    return {"decode": ("awq_gemv (gemv_kernel)", "hbm"), "prefill": ("awq_gemm (gemm_kernel)", "tensor"),
            "crossover": ("awq_gemv + awq_gemm", "hbm"), "w4a8": ("w4a8_linear (gemm_kernel<W4A8>)", "tensor")}[workload]


def load_traffic(workload, algorithmic_bytes_per_launch):
    """Per-launch DRAM traffic of the dominant kernel from the committed ncu summary.

    Returns None when there is no summary or the kernel source changed since it was taken.
    """
    import hashlib
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    src = os.path.join(ROOT, rec["kernel_source"])
    if not os.path.exists(src):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if not digest.startswith(rec["sha256_prefix"]):
        return None
    return round(rec["traffic_over_algorithmic"] * algorithmic_bytes_per_launch)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "crossover", "w4a8"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, help="comma-separated shape names to keep (profiling small cases)")
    ap.add_argument("--m", type=int, nargs="*", default=None, help="token counts to keep (profiling small cases)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    calls = workload_calls(args.workload, args.only, args.m)
    WORKLOAD_FILTER.update(only=args.only, ms=args.m)
    kinds = sorted({c[0] for c in calls})
    config = {"workload": f"{args.workload}: " + ", ".join(sorted({f'{n} K={k} N={nn}' for _, n, _, k, nn in calls})),
              "M": sorted({c[2] for c in calls}), "group_size": 128, "kernels": kinds,
              "calls_per_step": len(calls),
              "l2": "inputs larger than L2: every call of a step has its own weights "
                    f"({sum(c[3] * c[4] / 2 for c in calls) / 1e6:.0f} MB packed per step)"}
    unit = "GB/s" if args.workload in ("decode", "crossover") else "TFLOP/s"

    if args.impl == "reference":
        if rank != 0:
            return
        v, desc, cores = run_oracle_subprocess(args.workload, args.cpu_budget)
        value = v / 1e9 if unit == "GB/s" else None
        if unit == "TFLOP/s":
            # convert the oracle's byte rate to flop rate with the workload's flop/byte ratio
            fb = sum(2.0 * M * K * N for _, _, M, K, N in calls) / sum(call_bytes(k, M, K, N) for k, _, M, K, N in calls)
            value = v * fb / 1e12
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                          "dtype": "f64 (oracle)", "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                                           "sample": desc},
                          "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                          "vs_baseline": None}))
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)

    r = gpu_arm(args, rank, world, torch, dist)
    step_s = r["ms"] / 1e3 / args.steps
    gbs = whole_job_rate(r["step_bytes"], world, step_s) / 1e9
    tfs = whole_job_rate(r["step_flops"], world, step_s) / 1e12
    value = gbs if unit == "GB/s" else tfs
    e2e_step_s = r["e2e_s"] / args.steps
    e2e_value = (r["step_bytes"] * world / e2e_step_s / 1e9) if unit == "GB/s" else \
        (r["step_flops"] * world / e2e_step_s / 1e12)

    hbm, bf16, bf16_sus, src = load_peaks()
    kname, bound = dominant_kernel(args.workload)
    per_launch_s = step_s / max(1, len(r["calls"]))
    if bound == "hbm":
        achieved = r["step_bytes"] / len(r["calls"]) / per_launch_s / 1e9
        peak, punit = hbm, "GB/s"
    else:
        achieved = r["step_flops"] / len(r["calls"]) / per_launch_s / 1e12
        peak, punit = bf16, "TFLOP/s"   # fp16 dense rate equals the bf16 rate
    roofline = {"kernel": kname, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": punit,
                "frac": round(achieved / peak, 4), "peak_source": f"{src} (MEASURED_PEAKS.json)",
                "traffic": load_traffic(args.workload, r["step_bytes"] / len(r["calls"]))}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        try:
            v, desc, cores = run_oracle_subprocess(args.workload, args.cpu_budget)
            cv = v / 1e9 if unit == "GB/s" else v * (r["step_flops"] / r["step_bytes"]) / 1e12
            cpu = {"value": cv, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc}
        except Exception as exc:  # the baseline is reported, never required
            cpu = {"value": None, "unit": unit, "cores": 0, "kind": "oracle", "sample": f"failed: {exc}"[:200]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16 in, fp32 accumulate (int4 weights)",
            "data": "synthetic", "config": config,
            "throughput": {"GB/s": round(gbs, 1), "TFLOP/s": round(tfs, 3)},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": unit, "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"], "path": "python binding, one API call per layer call; pinned copies in and out every step, overlapped with compute in runs of >= 8 MB"},
            "gpu_launches": r["launches_per_step"] * args.steps,
            "clocks": r["clocks"],
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
