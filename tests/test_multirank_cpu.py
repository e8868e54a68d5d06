"""The N > 1 paths of bench.py on CPU: two gloo ranks for the max-over-ranks timing and the
whole-job rate, and the reference arm under torchrun (rank 0 prints the line, the others exit 0)."""

import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
dist = pytest.importorskip("torch.distributed")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took (r + 1) ms per step and 10 (r + 1) s end to end
    ms, e2e = bench.max_over_ranks([rank + 1.0, 10.0 * (rank + 1)], torch, dist, torch.device("cpu"))
    rate = bench.whole_job_rate(100.0, world, ms / 1e3)
    out.put((rank, ms, e2e, rate))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_two_gloo_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, e2e, rate in res:
        assert ms == 2.0 and e2e == 20.0          # every rank sees the slowest rank's times
        assert rate == pytest.approx(100.0 * 2 / 2e-3)  # both ranks' units over the slowest step


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 4.0], torch, None, torch.device("cpu")) == [3.0, 4.0]


def test_reference_arm_under_torchrun_prints_once():
    port = 29600 + (os.getpid() % 1000)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-budget", "1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["e2e"]["value"] == rec["value"]
    # the same metric, unit and workload as the GPU arm's line, with the oracle described as the baseline
    assert rec["metric"].startswith("W4A16 group-quant GEMM") and rec["unit"] == "GB/s"
    assert rec["higher_is_better"] is True and rec["config"]["workload"].startswith("decode:")
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["cpu_baseline"]["cores"] >= 1 and rec["cpu_baseline"]["sample"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
