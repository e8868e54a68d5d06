"""Host-side checks of the measurement definitions in bench.py (no GPU).

The workloads are the configurations of the problem statement, and the algorithmic byte counts are
the ones the rates divide by. Where a figure is pinned against a number, the number is worked out
by hand from the formula's terms.
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_decode_workload_is_the_llama2_sweep():
    calls = bench.workload_calls("decode")
    assert len(calls) == 16
    assert {c[0] for c in calls} == {"gemv_pp"}        # the prepared-weight decode GEMV
    awq_layout = bench.workload_calls("decode_awq")   # the same calls on the AWQ words
    assert [c[1:] for c in awq_layout] == [c[1:] for c in calls] and {c[0] for c in awq_layout} == {"gemv"}
    shapes = {(c[1], c[3], c[4]) for c in calls}
    assert shapes == {("qkv", 4096, 12288), ("o_proj", 4096, 4096), ("gate_up", 4096, 22016),
                      ("down", 11008, 4096)}
    assert sorted({c[2] for c in calls}) == [1, 2, 4, 8]


def test_prefill_and_w4a8_workloads():
    pre = bench.workload_calls("prefill")
    assert len(pre) == 16 and {c[0] for c in pre} == {"gemm"}
    assert sorted({c[2] for c in pre}) == [256, 1024, 4096, 8192]
    assert {(c[3], c[4]) for c in pre} == {(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)}
    w = bench.workload_calls("w4a8")
    assert [c[2] for c in w] == [1, 16, 64, 256, 1024, 4096]
    assert {(c[3], c[4]) for c in w} == {(21760, 8192)} and {c[0] for c in w} == {"w4a8"}


def test_crossover_routes_by_token_count():
    calls = bench.workload_calls("crossover")
    assert len(calls) == 24
    for kind, _, M, _, _ in calls:
        assert kind == ("gemv" if M <= 16 else "gemm")


def test_filters():
    calls = bench.workload_calls("decode", only="qkv", ms=[8])
    assert calls == [("gemv_pp", "qkv", 8, 4096, 12288)]
    with pytest.raises(ValueError):
        bench.workload_calls("decode", only="nope")


def test_algorithmic_bytes():
    # W4A16 at M = 1, qkv: packed weights 4096*12288/2 = 25165824, fp16 scales 2*12288*32 = 786432,
    # packed zeros 4*32*1536 = 196608, x 2*4096 = 8192, y 2*12288 = 24576
    assert bench.w4a16_bytes(1, 4096, 12288) == 25165824 + 786432 + 196608 + 8192 + 24576
    # the 0.5195 bytes per weight of the weight side: 1/2 + 2/128 + 1/2/128
    per_weight = (bench.w4a16_bytes(0, 4096, 4096)) / (4096 * 4096)
    assert per_weight == pytest.approx(0.5 + 2 / 128 + 0.5 / 128)
    # W4A8 at M = 1, K = 21760, N = 8192: weights 89128960, channel scales 16384, int8 x 21760,
    # token scale 4, y 16384
    assert bench.w4a8_bytes(1, 21760, 8192) == 89128960 + 16384 + 21760 + 4 + 16384
    assert bench.call_bytes("w4a8", 1, 21760, 8192) == bench.w4a8_bytes(1, 21760, 8192)
    assert bench.call_bytes("gemm", 256, 4096, 4096) == bench.w4a16_bytes(256, 4096, 4096)


def test_decode_step_sizes():
    calls = bench.workload_calls("decode")
    # 405 MB of packed weights per step (each M of each shape has its own weights), 422 MB in all
    packed = sum(K * N / 2 for _, _, _, K, N in calls)
    assert packed == 4 * (4096 * 12288 + 4096 * 4096 + 4096 * 22016 + 11008 * 4096) / 2 == 404750336
    total = sum(bench.call_bytes(k, M, K, N) for k, _, M, K, N in calls)
    assert 422e6 < total < 423e6


def test_crossover_symmetric_workload_and_bytes():
    calls = bench.workload_calls("crossover_sym")
    assert calls == bench.workload_calls("crossover") and bench.is_symmetric("crossover_sym")
    # symmetric weights carry no packed zero points: 4 * (K/128) * (N/8) bytes fewer
    assert bench.w4a16_bytes(1, 4096, 6144) - bench.w4a16_sym_bytes(1, 4096, 6144) == 4 * 32 * 768
    assert bench.call_bytes("gemv", 1, 4096, 6144, symmetric=True) == bench.w4a16_sym_bytes(1, 4096, 6144)
    assert bench.workload_unit("crossover_sym") == "GB/s" and bench.workload_unit("prefill") == "TFLOP/s"


def test_windows_cover_the_minimum_time():
    assert bench.windows_needed(3.6, 1.0) == 278          # 278 windows of 3.6 ms >= 1 s
    assert bench.windows_needed(400.0, 1.0) == 5          # never fewer than 5 windows
    assert bench.windows_needed(250.0, 1.0) == 5 and bench.windows_needed(150.0, 1.0) == 7


def test_workload_record_from_fabricated_timings():
    # a decode step of 16 calls timed at 0.2 ms per step over 20-step windows: value = bytes / time
    args = type("A", (), {"steps": 20})()
    calls = bench.workload_calls("decode")
    r = {"calls": calls, "symmetric": False, "win_ms": [4.0, 4.0, 4.2], "n_windows": 3, "ms": 4.0, "e2e_s": 0.008,
         "clocks": {"sm_mhz": 2070}, "launches_per_step": 16, "h2d": 1, "d2h": 2,
         "per_m": [(m, [c for c in calls if c[2] == m], 0.05) for m in (1, 2, 4, 8)]}
    rec = bench.workload_record("decode", r, args, world=1)
    step_bytes = sum(bench.call_bytes(k, M, K, N) for k, _, M, K, N in calls)
    assert rec["value"] == pytest.approx(step_bytes / 0.2e-3 / 1e9, rel=1e-4)
    assert rec["roofline"]["bound"] == "hbm" and rec["roofline"]["frac"] == pytest.approx(
        rec["roofline"]["achieved"] / rec["roofline"]["peak"], rel=1e-3)
    assert rec["e2e"]["value"] == pytest.approx(step_bytes / 0.4e-3 / 1e9, rel=1e-4)
    assert rec["gpu_launches"] == 16 * 20 * 3
    assert [row["M"] for row in rec["vs_M"]] == [1, 2, 4, 8]
    m1 = rec["vs_M"][0]
    b1 = sum(bench.call_bytes(k, M, K, N) for k, _, M, K, N in calls if M == 1)
    assert m1["GB/s"] == pytest.approx(b1 / 0.05e-3 / 1e9, rel=1e-3) and m1["us_per_call"] == 12.5
    # a tensor-bound sweep reports TFLOP/s against the sustained peak, with the burst fraction beside it
    pcalls = bench.workload_calls("prefill")
    r2 = dict(r, calls=pcalls, per_m=[(256, [c for c in pcalls if c[2] == 256], 1.0)])
    rec2 = bench.workload_record("prefill", r2, args, world=1)
    flops = sum(2.0 * M * K * N for _, _, M, K, N in pcalls)
    assert rec2["unit"] == "TFLOP/s" and rec2["value"] == pytest.approx(flops / 0.2e-3 / 1e12, rel=1e-4)
    assert rec2["roofline"]["bound"] == "tensor" and "frac_of_burst" in rec2["roofline"]


def test_w4a8_grouped_workload_and_bytes():
    calls = bench.workload_calls("w4a8_grouped")
    assert [c[2] for c in calls] == [1, 16, 64, 256, 1024, 4096] and {c[0] for c in calls} == {"w4a8g"}
    # the per-channel bytes plus fp16 group factors: 2 * 170 groups * 8192 columns
    assert bench.call_bytes("w4a8g", 1, 21760, 8192) == bench.w4a8_bytes(1, 21760, 8192) + 2 * 170 * 8192
