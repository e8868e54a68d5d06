"""GPU parity of the bf16 variant (through the C ABI) against the CPU oracle.

Bars:
* awq_dequant_bf16: bit-exact (W = bf16_RN((q - z) s));
* awq_gemv_bf16 / awq_gemm_bf16 bf16 outputs: |y - y_oracle| <= 2e-3 rms(y_oracle) + 2^-8 |y_oracle|
  element by element, y_oracle the unrounded float64 product of the oracle's bf16 weights and the bf16
  activations.  The 2e-3 rms budget is the computation's (as for fp16); the bf16 output format adds its
  own rounding of at most half an ulp, which for 8 significant bits is 2^-8 of |y| (fp16: 11 bits,
  2^-11).  Both kernels make every weight exactly as the oracle does and add in fp32, so the computation
  itself stays far inside the budget.
"""

import numpy as np
import pytest

import oracle
from bit_weight_only_awq_gb300 import synth
from tests.test_gpu_parity import sample_word_cols

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3
BF16_HALF_ULP = 2.0 ** -8  # half an ulp of an 8-significant-bit output, relative


@pytest.fixture(scope="module")
def awq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_awq_gb300 import build as awq_build
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq as mod
    return mod


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host_bits(t):
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bf16_within_tol(y_bits, ref64, what):
    y = oracle.bf16_to_float(y_bits)
    rms = np.sqrt(np.mean(ref64 ** 2))
    err = np.max(np.abs(y - ref64) - BF16_HALF_ULP * np.abs(ref64))
    assert np.all(np.isfinite(y)), what
    assert err <= TOL * rms, f"{what}: max err beyond the output rounding {err:.3e} > {TOL} * rms {rms:.3e}"


def run(awq, fn, p, split_k=0):
    qz = None if p["qzeros"] is None else dev(p["qzeros"])
    y = fn(dev_bf16(p["x"]), dev(p["qweight"]), qz, dev_bf16(p["scales"]), 128, split_k=split_k)
    return host_bits(y)


def oracle_cols(p, wc):
    qw = p["qweight"][:, wc]
    qz = None if p["qzeros"] is None else p["qzeros"][:, wc]
    cols = (8 * np.asarray(wc)[:, None] + np.arange(8)[None, :]).ravel()
    return oracle.awq_linear_bf16(p["x"], qw, qz, p["scales"][:, cols], 128), cols


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("K,N,g", [(512, 512, 128), (384, 264, 128), (256, 64, 64)])
def test_dequant_bf16_bitexact(awq, K, N, g, symmetric):
    p = synth.awq_problem_bf16(1, K, N, seed=8000 + K + N, group_size=g, symmetric=symmetric)
    qz = None if symmetric else dev(p["qzeros"])
    w = awq.awq_dequant_bf16(dev(p["qweight"]), qz, dev_bf16(p["scales"]), g)
    want = oracle.dequant_bf16(p["qweight"], p["qzeros"], p["scales"], g)
    assert np.array_equal(host_bits(w), want)


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("split_k", [1, 3, 0])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
def test_gemv_bf16_small_ragged(awq, M, split_k, symmetric):
    p = synth.awq_problem_bf16(M, 1280, 416, seed=8100 + M, symmetric=symmetric)
    y = run(awq, awq.awq_gemv_bf16, p, split_k)
    ref = oracle.awq_linear_bf16(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert_bf16_within_tol(y, ref, f"gemv bf16 M={M} split={split_k} sym={symmetric}")


@pytest.mark.parametrize("M", [1, 8, 16])
@pytest.mark.parametrize("name,K,N", synth.LLAMA31_8B_STACK)
def test_gemv_bf16_llama31_shapes_sampled(awq, name, K, N, M):
    p = synth.awq_problem_bf16(M, K, N, seed=8200 + K + N + M)
    y = run(awq, awq.awq_gemv_bf16, p)
    ref, cols = oracle_cols(p, sample_word_cols(N // 8, seed=K + N + 4, count=24))
    assert_bf16_within_tol(y[:, cols], ref, f"gemv bf16 {name} M={M}")


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("M", [1, 9, 40, 64, 100, 128, 256, 300])
def test_gemm_bf16_small_ragged(awq, M, symmetric):
    p = synth.awq_problem_bf16(M, 640, 416, seed=8300 + M, symmetric=symmetric)
    y = run(awq, awq.awq_gemm_bf16, p, 1)
    ref = oracle.awq_linear_bf16(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert_bf16_within_tol(y, ref, f"gemm bf16 M={M} sym={symmetric}")


@pytest.mark.parametrize("split_k", [2, 3, 0])
def test_gemm_bf16_split_k(awq, split_k):
    p = synth.awq_problem_bf16(70, 1024, 256, seed=8400 + split_k)
    y = run(awq, awq.awq_gemm_bf16, p, split_k)
    ref = oracle.awq_linear_bf16(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert_bf16_within_tol(y, ref, f"gemm bf16 split={split_k}")


@pytest.mark.parametrize("M", [256, 1024])
@pytest.mark.parametrize("name,K,N", synth.MISTRAL_7B_PREFILL)
def test_gemm_bf16_mistral_shapes_sampled(awq, name, K, N, M):
    p = synth.awq_problem_bf16(M, K, N, seed=8500 + K + N + M)
    y = run(awq, awq.awq_gemm_bf16, p)
    ref, cols = oracle_cols(p, sample_word_cols(N // 8, seed=K + N + 5, count=16))
    assert_bf16_within_tol(y[:, cols], ref, f"gemm bf16 {name} M={M}")


def test_gemm_bf16_two_mblock_tiles_sampled_rows(awq):
    # 4096 tokens: 256-token tiles with two 128-column M-blocks per CTA
    K, N, M = 4096, 28672, 4096
    p = synth.awq_problem_bf16(M, K, N, seed=8600)
    y = run(awq, awq.awq_gemm_bf16, p)
    rows = np.array(sorted(set(np.random.default_rng(2).choice(M, 24, replace=False).tolist()) | {0, M - 1}))
    ref, cols = oracle_cols(dict(p, x=p["x"][rows]), sample_word_cols(N // 8, seed=6, count=12))
    assert_bf16_within_tol(y[np.ix_(rows, cols)], ref, "gemm bf16 gate_up M=4096")


def test_no_device_timeouts_recorded_bf16(awq):
    torch.cuda.synchronize()
    assert awq.awq_last_device_error() == 0
