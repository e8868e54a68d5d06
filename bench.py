"""Benchmark harness: AWQ W4A16 / W4A8 quantized linear layer on GB300.

Headline (`value`): the decode GEMV sweep at Llama-2-7B linear shapes.  One step =
16 GEMV calls, M in {1, 2, 4, 8} x (K, N) in {(4096, 12288) qkv, (4096, 4096) o_proj,
(4096, 22016) gate_up, (11008, 4096) down}, group size 128, each call with its own
weight buffers (405 MB of packed weights per step, more than 3x the 126 MB L2, so
every step streams its weights from HBM).

The default run (`--workload all`) also times, in the same process, the other sweeps
of the metric "TFLOP/s & HBM GB/s vs M" and reports each as a record under
`workloads`: the prefill GEMM (Mistral-7B shapes, M in {256 .. 8192}), the GEMV/GEMM
crossover on the Llama-3.1-8B layer stack (M in {1 .. 1024}) with zero-point weights
and with symmetric weights (zero fixed at 8), and W4A8 (N=8192, K=21760,
M in {1 .. 4096}).  Every record has its own value, roofline, cpu_baseline, e2e,
clocks and per-M rates.

Timed region (device value): the step captured as one CUDA graph; windows of K graph
replays are timed between CUDA events on the launching stream, back to back, until at
least `--min-seconds` of device time (and at least 5 windows) have run; barrier +
synchronize on both sides; the median window gives ms_per_step; max over ranks.
Per-M rates: a graph of one M's calls, each replay timed between events with an L2
flush (a write of twice the L2 size) between replays, median over replays.
e2e: the same step through the public Python API (one call per layer call), with all of
the step's activations copied in from pinned host memory and all of its outputs copied
back, every step: calls grouped into runs of at least 8 MB of copies, each run's copies
on their own streams so that they overlap the neighbouring runs' compute.  The CPU
baseline and `--impl reference` time the numpy oracle on a bounded sample of the same
workload, on one core and on all host cores (one process per core).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_weight_only_awq_gb300 import synth  # noqa: E402

WORKLOAD_FILTER = {"only": None, "ms": None}
METRIC = "W4A16 group-quant GEMM TFLOP/s & HBM GB/s vs M; % of roofline on 1 GB300"
WORKLOADS = ("decode", "decode_awq", "prefill", "crossover", "crossover_sym", "w4a8", "w4a8_grouped",
             "decode_bf16", "prefill_bf16")
HEADLINE = "decode"
L2_BYTES = 126 * 1024 * 1024  # GB300 L2 (the flush writes twice this)


# ------------------------------------------------------------------ workloads
def w4a16_bytes(M, K, N):
    return K * N / 2 + 2 * N * K / 128 + 4 * (K / 128) * (N / 8) + 2 * M * K + 2 * M * N


def w4a16_sym_bytes(M, K, N):
    """Symmetric weights have no packed zero points."""
    return K * N / 2 + 2 * N * K / 128 + 2 * M * K + 2 * M * N


def w4a8_bytes(M, K, N):
    return K * N / 2 + 2 * N + M * K + 4 * M + 2 * M * N


def w4a8_grouped_bytes(M, K, N):
    """Per-group W4A8: the per-channel bytes plus the fp16 group factors s3 [K/128, N]."""
    return w4a8_bytes(M, K, N) + 2 * (K / 128) * N


def awq_linear_gemv_max():
    """Largest token count the library's dispatch (awq_linear) sends to the GEMV kernel."""
    return 16


def is_symmetric(workload):
    return workload.endswith("_sym")


def is_bf16(workload):
    return workload.endswith("_bf16")


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
        # the production decode path: weights prepared once at load time (awq_prepack_gemv)
        return [("gemv_pp", n, m, k, nn) for n, k, nn in synth.LLAMA2_7B_DECODE for m in synth.DECODE_M]
    if workload == "decode_awq":
        # the same sweep on the AWQ-format words (awq_gemv), no preparation
        return [("gemv", n, m, k, nn) for n, k, nn in synth.LLAMA2_7B_DECODE for m in synth.DECODE_M]
    if workload == "prefill":
        return [("gemm", n, m, k, nn) for n, k, nn in synth.MISTRAL_7B_PREFILL for m in synth.PREFILL_M]
    if workload == "decode_bf16":
        return [("gemv_bf16", n, m, k, nn) for n, k, nn in synth.LLAMA2_7B_DECODE for m in synth.DECODE_M]
    if workload == "prefill_bf16":
        return [("gemm_bf16", n, m, k, nn) for n, k, nn in synth.MISTRAL_7B_PREFILL for m in synth.PREFILL_M]
    if workload in ("crossover", "crossover_sym"):
        out = []
        for n, k, nn in synth.LLAMA31_8B_STACK:
            for m in synth.CROSSOVER_M:
                out.append(("gemv" if m <= awq_linear_gemv_max() else "gemm", n, m, k, nn))
        return out
    if workload == "w4a8":
        k, nn = synth.W4A8_SHAPE
        return [("w4a8", "w4a8", m, k, nn) for m in synth.W4A8_M]
    if workload == "w4a8_grouped":
        k, nn = synth.W4A8_SHAPE
        return [("w4a8g", "w4a8_grouped", m, k, nn) for m in synth.W4A8_M]
    raise ValueError(workload)


def call_bytes(kind, M, K, N, symmetric=False):
    if kind == "w4a8":
        return w4a8_bytes(M, K, N)
    if kind == "w4a8g":
        return w4a8_grouped_bytes(M, K, N)
    return w4a16_sym_bytes(M, K, N) if symmetric else w4a16_bytes(M, K, N)


def workload_unit(workload):
    """The sweep's own rate: GB/s where HBM bounds it (decode, crossover), TFLOP/s on the tensor cores."""
    return "GB/s" if workload in ("decode", "decode_awq", "decode_bf16", "crossover", "crossover_sym") else "TFLOP/s"


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
def _oracle_problems(workload, cols, seed):
    sym = is_symmetric(workload)
    problems = []
    for i, (kind, name, M, K, N) in enumerate(workload_calls(workload)):
        if kind == "w4a8":
            problems.append((kind, M, K, synth.w4a8_problem(M, K, cols, seed=seed + i)))
        elif kind == "w4a8g":
            problems.append((kind, M, K, synth.w4a8_group_problem(M, K, cols, seed=seed + i)))
        elif is_bf16(workload):
            problems.append((kind, M, K, synth.awq_problem_bf16(M, K, cols, seed=seed + i)))
        else:
            problems.append((kind, M, K, synth.awq_problem(M, K, cols, seed=seed + i, symmetric=sym)))
    return problems


def oracle_sample(workload, budget_s, seed=7):
    """Time the oracle on a bounded, seeded sample of the workload; returns (bytes/s, description).

    The sample: every call of one step, restricted to 256 output columns, repeated
    until about `budget_s` seconds of oracle work have been spent (at least one pass).
    """
    done, spent, passes, ncalls = _oracle_passes(workload, budget_s, seed)
    desc = (f"{passes} pass(es) over all {ncalls} calls of one step, each restricted to 256 seeded "
            f"output columns; numpy oracle, one thread, {spent:.1f} s")
    return done / spent, desc


def _oracle_passes(workload, budget_s, seed):
    import oracle

    cols = 256
    problems = _oracle_problems(workload, cols, seed)
    sym = is_symmetric(workload)
    done_bytes = 0.0
    spent = 0.0
    passes = 0
    while passes == 0 or spent < budget_s:
        for kind, M, K, p in problems:
            t0 = time.perf_counter()
            if kind == "w4a8":
                xq, s = oracle.quant_act(p["x"])
                oracle.w4a8_linear(xq, s, p["wq"], p["s_ch"])
            elif kind == "w4a8g":
                xq, s = oracle.quant_act(p["x"])
                oracle.w4a8_group_linear(xq, s, p["wq"], p["s3"], p["s2"], 128)
            elif kind.endswith("_bf16"):
                oracle.awq_linear_bf16(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
            else:
                oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
            spent += time.perf_counter() - t0
            done_bytes += call_bytes(kind, M, K, cols, sym)
        passes += 1
    return done_bytes, spent, passes, len(problems)


def _oracle_worker(args):
    workload, budget_s, seed = args
    done, spent, passes, _ = _oracle_passes(workload, budget_s, seed)
    return done, spent, passes


def oracle_sample_all_cores(workload, budget_s, procs):
    """The same sample on `procs` single-threaded processes at once (distinct seeds); returns
    (bytes/s over the wall time, description)."""
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(procs) as pool:
        res = pool.map(_oracle_worker, [(workload, budget_s, 7 + 1000 * i) for i in range(procs)])
    wall = time.perf_counter() - t0
    done = sum(r[0] for r in res)
    passes = sum(r[2] for r in res)
    desc = (f"{procs} processes x >= {budget_s:.0f} s, {passes} passes in all over the calls of one step, each "
            f"restricted to 256 seeded output columns; numpy oracle, one thread per process, {wall:.1f} s wall")
    return done / wall, desc


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle_subprocess(workload, budget_s, all_cores=False):
    """Run the oracle sample in a child process (every process pinned to one BLAS / OpenMP thread).
    Returns (bytes/s, description, cores used)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs = host_cores() if all_cores else 1
    if all_cores:
        code = ("import json, bench; v, d = bench.oracle_sample_all_cores(%r, %r, %d); "
                "print(json.dumps({'v': v, 'd': d}))" % (workload, budget_s, procs))
    else:
        code = ("import json, bench; v, d = bench.oracle_sample(%r, %r); print(json.dumps({'v': v, 'd': d}))"
                % (workload, budget_s))
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=900)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    res = json.loads(out.stdout.strip().splitlines()[-1])
    return res["v"], res["d"], procs


def oracle_rate_in_unit(v_bytes, unit, calls, symmetric=False):
    """An oracle byte rate in the workload's unit (TFLOP/s through the workload's flop/byte ratio)."""
    if unit == "GB/s":
        return v_bytes / 1e9
    fb = sum(2.0 * M * K * N for _, _, M, K, N in calls) / \
        sum(call_bytes(k, M, K, N, symmetric) for k, _, M, K, N in calls)
    return v_bytes * fb / 1e12


def cpu_baseline(workload, budget_s, unit, all_cores_too=True):
    calls = workload_calls(workload)
    sym = is_symmetric(workload)
    out = {}
    for label, all_cores in (("one_core", False), ("all_cores", True)):
        if all_cores and not all_cores_too:
            continue
        try:
            v, desc, cores = run_oracle_subprocess(workload, budget_s, all_cores=all_cores)
            out[label] = {"value": oracle_rate_in_unit(v, unit, calls, sym), "unit": unit, "cores": cores,
                          "kind": "oracle", "sample": desc}
        except Exception as exc:  # the baseline is reported, never required
            out[label] = {"value": None, "unit": unit, "cores": 0, "kind": "oracle", "sample": f"failed: {exc}"[:200]}
    rec = dict(out["one_core"])
    if "all_cores" in out:
        rec["all_cores"] = out["all_cores"]
    rec["nproc"] = host_cores()
    return rec


# ------------------------------------------------------------------ GPU arm
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def build_inputs(torch, workload, device, only=None, ms=None):
    """Per-call device buffers (weights distinct per call).  The activations and outputs of all calls
    are views into one device buffer each, mirrored by one pinned host buffer each, so that the e2e
    step moves them with one host-to-device and one device-to-host copy.

    Weights, zero points and scales come from the seeded generators of `synth`; the activations,
    N(0, 1) rounded to the layer's 16-bit format, are drawn on the device from a CUDA generator seeded
    per workload (the host-side normal generator takes tens of seconds for the prefill sweeps)."""
    sym = is_symmetric(workload)
    bufs = []
    for i, (kind, name, M, K, N) in enumerate(workload_calls(workload, only, ms)):
        seed = 10_000 + i
        if kind == "w4a8":
            p = synth.w4a8_problem(M, K, N, seed=seed, with_x=False)
            b = {"wq": torch.from_numpy(p["wq"]).to(device), "s_ch": torch.from_numpy(p["s_ch"]).to(device)}
            b["s_tok"] = torch.empty((M,), dtype=torch.float32, device=device)
        elif kind == "w4a8g":
            p = synth.w4a8_group_problem(M, K, N, seed=seed, with_x=False)
            b = {k: torch.from_numpy(p[k]).to(device) for k in ("wq", "s3", "s2")}
            b["s_tok"] = torch.empty((M,), dtype=torch.float32, device=device)
        elif kind.endswith("_bf16"):
            p = synth.awq_problem_bf16(M, K, N, seed=seed, with_x=False)
            b = {k: torch.from_numpy(p[k]).to(device) for k in ("qweight", "qzeros")}
            b["scales"] = torch.from_numpy(p["scales"].view(np.int16)).to(device).view(torch.bfloat16)
        else:
            p = synth.awq_problem(M, K, N, seed=seed, symmetric=sym, with_x=False)
            b = {k: (None if p[k] is None else torch.from_numpy(p[k]).to(device))
                 for k in ("qweight", "qzeros", "scales")}
            if kind == "gemv_pp":  # prepared once, as at model load; the AWQ words are not kept
                b["pp"] = awq_module().awq_prepack_gemv(b["qweight"], b["qzeros"], b["scales"])
                b.update(qweight=None, qzeros=None, scales=None)
        b["meta"] = (kind, name, M, K, N)
        bufs.append(b)
    # every view starts on a 16-byte boundary: M * K and M * N are multiples of 8 halves
    nx = sum(b["meta"][2] * b["meta"][3] for b in bufs)
    ny = sum(b["meta"][2] * b["meta"][4] for b in bufs)
    dt = torch.bfloat16 if is_bf16(workload) else torch.float16
    packed = {"x": torch.empty(nx, dtype=dt, device=device),
              "x_host": torch.empty(nx, dtype=dt).pin_memory(),
              "y": torch.empty(ny, dtype=dt, device=device),
              "y_host": torch.empty(ny, dtype=dt).pin_memory()}
    gen = torch.Generator(device=device)
    gen.manual_seed(20_000 + WORKLOADS.index(workload))
    packed["x"].copy_(torch.randn(nx, generator=gen, device=device, dtype=torch.float32))
    packed["x_host"].copy_(packed["x"])
    ox = oy = 0
    for b in bufs:
        _, _, M, K, N = b["meta"]
        b["x"] = packed["x"][ox:ox + M * K].view(M, K)
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


def awq_module():
    from bit_weight_only_awq_gb300 import awq
    return awq


def issue_step(awq, bufs, stream):
    """All calls of one step on `stream`; returns the number of kernels launched."""
    launches = 0
    for b in bufs:
        kind, _, M, K, N = b["meta"]
        if kind == "gemv_pp":
            awq.awq_gemv_prepacked(b["x"], b["pp"], out=b["y"], stream=stream)
            launches += 1
        elif kind == "gemv_bf16":
            awq.awq_gemv_bf16(b["x"], b["qweight"], b["qzeros"], b["scales"], out=b["y"], stream=stream)
            launches += 1
        elif kind == "gemm_bf16":
            awq.awq_gemm_bf16(b["x"], b["qweight"], b["qzeros"], b["scales"], out=b["y"], stream=stream)
            launches += 1
        elif kind == "gemv":
            awq.awq_gemv(b["x"], b["qweight"], b["qzeros"], b["scales"], out=b["y"], stream=stream)
            launches += 1
        elif kind == "gemm":
            awq.awq_gemm(b["x"], b["qweight"], b["qzeros"], b["scales"], out=b["y"], stream=stream)
            launches += 1
        elif kind == "w4a8g":
            awq.w4a8_linear_grouped(b["x"], b["wq"], b["s3"], b["s2"], out=b["y"], s_tok=b["s_tok"], stream=stream)
            launches += 2  # quantize (fp16 codes into the workspace), then the tensor-core GEMM
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


def windows_needed(probe_ms, min_seconds, min_windows=5):
    """Windows of one probe's length that cover at least `min_seconds` (and `min_windows`)."""
    return max(min_windows, int(math.ceil(min_seconds * 1e3 / max(probe_ms, 1e-3))))


def capture(torch, awq, bufs, stream):
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        launches = issue_step(awq, bufs, stream)
    torch.cuda.synchronize()
    return graph, launches


def time_windows(torch, graph, stream, steps, n_windows):
    """n_windows windows of `steps` replays, back to back on `stream`; returns each window's ms."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_windows + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for w in range(n_windows):
            for _ in range(steps):
                graph.replay()
            evs[w + 1].record(stream)
    stream.synchronize()
    return [evs[w].elapsed_time(evs[w + 1]) for w in range(n_windows)]


def time_flushed(torch, graph, stream, flush, reps):
    """`reps` replays of `graph`, each between its own events, with an L2 flush (outside the events)
    before each one; returns each replay's ms."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush.add_(1)
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def gpu_workload(args, workload, world, torch, dist, awq, device, flush):
    """Times one workload; returns the raw measurements (times already max-reduced over ranks)."""
    sym = is_symmetric(workload)
    bufs = build_inputs(torch, workload, device, **WORKLOAD_FILTER)
    calls = [b["meta"] for b in bufs]

    stream = torch.cuda.Stream(device=device)
    # pre-size the shared workspace for the largest call, then warm every code path once
    for b in bufs:
        kind, _, M, K, N = b["meta"]
        op = {"gemv": awq.OP_GEMV, "gemm": awq.OP_GEMM, "w4a8": awq.OP_W4A8_GEMM,
              "gemv_pp": awq.OP_GEMV_PREPACKED, "gemv_bf16": awq.OP_GEMV_BF16, "gemm_bf16": awq.OP_GEMM_BF16,
              "w4a8g": awq.OP_W4A8_GROUPED}[kind]
        awq.device_workspace(awq.awq_workspace_bytes(op, M, K, N, 0), device)
    with torch.cuda.stream(stream):
        issue_step(awq, bufs, stream)
    torch.cuda.synchronize()
    graph, launches_per_step = capture(torch, awq, bufs, stream)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        graph.replay()
    barrier()
    probe = time_windows(torch, graph, stream, args.steps, 1)[0]
    n_windows = int(max_over_ranks([windows_needed(probe, args.min_seconds)], torch, dist, device)[0])
    barrier()
    with ClockSampler(device.index) as clk:
        barrier()
        win_ms = time_windows(torch, graph, stream, args.steps, n_windows)
        barrier()
    clocks = clk.summary()
    med_ms = statistics.median(win_ms)

    # per-M rates: one graph per token count, each replay timed alone after an L2 flush
    per_m = []
    for m in sorted({c[2] for c in calls}):
        sub = [b for b in bufs if b["meta"][2] == m]
        g, _ = capture(torch, awq, sub, stream)
        for _ in range(3):
            g.replay()
        reps = time_flushed(torch, g, stream, flush, args.per_m_reps)
        per_m.append((m, sub, statistics.median(reps)))

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

    reduced = max_over_ranks([med_ms, e2e_s] + [t for _, _, t in per_m], torch, dist, device)
    med_ms, e2e_s, per_m_ms = reduced[0], reduced[1], reduced[2:]
    res = {
        "calls": calls, "symmetric": sym, "win_ms": win_ms, "n_windows": n_windows, "ms": med_ms,
        "e2e_s": e2e_s, "clocks": clocks, "launches_per_step": launches_per_step,
        "h2d": sum(2 * M * K for _, _, M, K, _ in calls), "d2h": sum(2 * M * N for _, _, M, _, N in calls),
        "per_m": [(m, [b["meta"] for b in sub], t) for (m, sub, _), t in zip(per_m, per_m_ms)],
    }
    del graph, bufs, segs
    torch.cuda.synchronize()
    return res


def dominant_kernel(workload):
    return {"decode": ("awq_gemv_prepacked (gemv_pp_kernel)", "hbm"),
            "decode_awq": ("awq_gemv (gemv_kernel)", "hbm"), "prefill": ("awq_gemm (gemm_kernel)", "tensor"),
            "crossover": ("awq_gemv + awq_gemm", "hbm"), "crossover_sym": ("awq_gemv + awq_gemm", "hbm"),
            "w4a8": ("w4a8_linear (gemm_kernel<W4A8>)", "tensor"),
            "w4a8_grouped": ("w4a8_linear_grouped (gemm_kernel<W4A8, group factors>)", "tensor"),
            "decode_bf16": ("awq_gemv_bf16 (gemv_kernel<8, bf16>)", "hbm"),
            "prefill_bf16": ("awq_gemm_bf16 (gemm_kernel<bf16>)", "tensor")}[workload]


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


def workload_record(workload, r, args, world):
    """The JSON record of one timed workload (value, roofline, e2e, per-M rates, clocks)."""
    unit = workload_unit(workload)
    sym = r["symmetric"]
    calls = r["calls"]
    step_bytes = sum(call_bytes(k, M, K, N, sym) for k, _, M, K, N in calls)
    step_flops = sum(2.0 * M * K * N for _, _, M, K, N in calls)
    step_s = r["ms"] / 1e3 / args.steps
    gbs = whole_job_rate(step_bytes, world, step_s) / 1e9
    tfs = whole_job_rate(step_flops, world, step_s) / 1e12
    value = gbs if unit == "GB/s" else tfs
    e2e_step_s = r["e2e_s"] / args.steps
    e2e_value = (step_bytes * world / e2e_step_s / 1e9) if unit == "GB/s" else (step_flops * world / e2e_step_s / 1e12)

    hbm, bf16, bf16_sus, src = load_peaks()
    kname, bound = dominant_kernel(workload)
    per_launch_s = step_s / max(1, len(calls))
    if bound == "hbm":
        achieved = step_bytes / len(calls) / per_launch_s / 1e9
        peak, punit, pnote = hbm, "GB/s", f"{src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
        extra = {}
    else:
        # timed inside >= 1 s of back-to-back tensor work: the sustained peak; the burst one beside it
        achieved = step_flops / len(calls) / per_launch_s / 1e12
        peak, punit = bf16_sus, "TFLOP/s"
        pnote = f"{src} bf16 cuBLAS, sustained (MEASURED_PEAKS.json bf16_tflops_sustained); fp16 has the same dense rate"
        extra = {"peak_burst": bf16, "frac_of_burst": round(achieved / bf16, 4)}
    roofline = {"kernel": kname, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": punit,
                "frac": round(achieved / peak, 4), "peak_source": pnote, **extra,
                "traffic": load_traffic(workload, step_bytes / len(calls))}

    vs_m = []
    for m, mcalls, ms in r["per_m"]:
        b = sum(call_bytes(k, M, K, N, sym) for k, _, M, K, N in mcalls)
        f = sum(2.0 * M * K * N for _, _, M, K, N in mcalls)
        g = b / (ms / 1e3) / 1e9
        t = f / (ms / 1e3) / 1e12
        vs_m.append({"M": m, "kernels": sorted({c[0] for c in mcalls}), "calls": len(mcalls),
                     "us_per_call": round(ms * 1e3 / len(mcalls), 2), "GB/s": round(g, 1),
                     "TFLOP/s": round(t, 2), "frac_hbm": round(g / hbm, 4), "frac_tensor": round(t / bf16, 4)})
    config = {"workload": f"{workload}: " + ", ".join(sorted({f'{n} K={k} N={nn}' for _, n, _, k, nn in calls})),
              "M": sorted({c[2] for c in calls}), "group_size": 128,
              "weights": "symmetric (zero 8, no qzeros)" if sym else (
                  "per-channel int4, u = q + 8" if workload == "w4a8" else
                  "int4 u = q + 8 with integer group factors s3 (g=128) and channel scales s2" if workload == "w4a8_grouped"
                  else "zero-point (packed qzeros)"),
              "activations": "bf16 (bf16 scales and output)" if is_bf16(workload) else "fp16",
              "kernels": sorted({c[0] for c in calls}), "calls_per_step": len(calls),
              "l2": "inputs larger than L2: every call of a step has its own weights "
                    f"({sum(c[3] * c[4] / 2 for c in calls) / 1e6:.0f} MB packed per step); per-M rates flush L2 "
                    "(a write of 252 MB) before each timed replay",
              "timing": f"{r['n_windows']} windows of {args.steps} CUDA-graph replays back to back "
                        f"({sum(r['win_ms']) / 1e3:.2f} s of device time), median window"}
    return {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "ms_per_step": round(step_s * 1e3, 4),
        "config": config, "throughput": {"GB/s": round(gbs, 1), "TFLOP/s": round(tfs, 3)},
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 2), "unit": unit, "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "path": "python binding, one API call per layer call; pinned copies in and out every step, "
                        "overlapped with compute in runs of >= 8 MB"},
        "gpu_launches": r["launches_per_step"] * args.steps * r["n_windows"],
        "clocks": r["clocks"], "vs_M": vs_m,
        "window_ms": {"min": round(min(r["win_ms"]), 4), "median": round(statistics.median(r["win_ms"]), 4),
                      "max": round(max(r["win_ms"]), 4)},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", choices=("all",) + WORKLOADS)
    ap.add_argument("--min-seconds", type=float, default=1.0, help="device time each workload is timed for")
    ap.add_argument("--per-m-reps", type=int, default=15, help="L2-flushed replays per token count")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work per CPU-baseline run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, help="comma-separated shape names to keep (profiling small cases)")
    ap.add_argument("--m", type=int, nargs="*", default=None, help="token counts to keep (profiling small cases)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    head = HEADLINE if args.workload == "all" else args.workload
    others = [w for w in WORKLOADS if w != HEADLINE] if args.workload == "all" else []
    workload_calls(head, args.only, args.m)  # the filters must leave a call
    WORKLOAD_FILTER.update(only=args.only, ms=args.m)
    unit = workload_unit(head)

    if args.impl == "reference":
        if rank != 0:
            return
        calls = workload_calls(head, args.only, args.m)
        v, desc, cores = run_oracle_subprocess(head, args.cpu_budget, all_cores=True)
        value = oracle_rate_in_unit(v, unit, calls, is_symmetric(head))
        config = {"workload": f"{head}: " + ", ".join(sorted({f'{n} K={k} N={nn}' for _, n, _, k, nn in calls})),
                  "M": sorted({c[2] for c in calls}), "group_size": 128, "kernels": sorted({c[0] for c in calls}),
                  "calls_per_step": len(calls)}
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

    from bit_weight_only_awq_gb300 import build as awq_build
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq

    device = torch.device("cuda", torch.cuda.current_device())
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    records = {}
    for w in [head] + others:
        r = gpu_workload(args, w, world, torch, dist, awq, device, flush)
        records[w] = workload_record(w, r, args, world)
    if rank == 0 and not args.no_cpu_baseline:
        # one core and all host cores for the headline and the prefill sweep (the two halves of the metric);
        # one core for the other sweeps, on a shorter sample
        for i, w in enumerate([head] + others):
            budget = args.cpu_budget if i == 0 else max(1.0, args.cpu_budget / 4)
            records[w]["cpu_baseline"] = cpu_baseline(w, budget, records[w]["unit"],
                                                      all_cores_too=w in (head, "prefill"))

    if rank == 0:
        top = records[head]
        line = {
            "metric": METRIC, "value": top["value"], "unit": top["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": top["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16 in, fp32 accumulate (int4 weights)",
            "data": "synthetic", "config": top["config"], "throughput": top["throughput"],
            "roofline": top["roofline"], "cpu_baseline": top.get("cpu_baseline"), "e2e": top["e2e"],
            "gpu_launches": top["gpu_launches"],
            "gpu_launches_all_workloads": sum(rec["gpu_launches"] for rec in records.values()),
            "clocks": top["clocks"], "vs_M": top["vs_M"], "window_ms": top["window_ms"],
            "workloads": {w: rec for w, rec in records.items() if w != head},
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
