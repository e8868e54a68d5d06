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
    assert {c[0] for c in calls} == {"gemv"}
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
    assert calls == [("gemv", "qkv", 8, 4096, 12288)]
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
