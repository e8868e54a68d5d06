"""awq_gemv_noalloc: the decode GEMV for callers that cannot allocate device memory.

Such callers (a plugin inside a runtime that owns all device memory, a serving loop that
forbids allocation after start-up) cannot hand awq_gemv a workspace; awq_gemv_noalloc keeps
the split-K scratch in a fixed array inside the library instead.  This test calls it through
the C ABI and checks its output against awq_gemv's on two calls in a row (the second call
finds the array holding the first call's leftovers), within the tolerance the parity tests
use.  The file sorts last so that a run stopping at the first failure has run every other test.
"""

import numpy as np
import pytest

import oracle
from bit_weight_only_awq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3
EWORKSPACE = -6


@pytest.fixture(scope="module")
def awq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_awq_gb300 import build as awq_build
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq as mod
    return mod


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _noalloc_via_abi(awq, x, qw, qz, sc, y, split_k):
    M, K = x.shape
    N = qw.shape[1] * 8
    stream = torch.cuda.current_stream().cuda_stream
    return awq.lib.awq_gemv_noalloc(x.data_ptr(), qw.data_ptr(), None if qz is None else qz.data_ptr(),
                                    sc.data_ptr(), y.data_ptr(), M, K, N, 128, split_k, stream)


@pytest.mark.parametrize("M,K,N,split_k,symmetric", [
    (8, 4096, 12288, 0, False),   # automatic split: the fixed scratch array is used
    (3, 1280, 416, 3, True),      # explicit split, ragged column tile, symmetric
    (1, 11008, 4096, 0, False),
    (16, 4096, 22016, 0, False),  # two 8-token halves: twice the partial rows per contributor
])
def test_noalloc_matches_gemv_on_two_calls_in_a_row(awq, M, K, N, split_k, symmetric):
    p = synth.awq_problem(M, K, N, seed=900 + M + K, symmetric=symmetric)
    x, qw, sc = _dev(p["x"]), _dev(p["qweight"]), _dev(p["scales"])
    qz = None if symmetric else _dev(p["qzeros"])
    y_ref = awq.awq_gemv(x, qw, qz, sc, 128, split_k=split_k)
    torch.cuda.synchronize()
    ref = y_ref.cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc_via_abi(awq, x, qw, qz, sc, y, split_k) == 0
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        # both outputs are fp16: each carries its own output rounding (half an ulp, 2^-11 relative)
        assert np.max(np.abs(got - ref) - 2 * 2.0 ** -11 * np.abs(ref)) <= TOL * rms
        # no bounded device wait of either call gave up
        assert awq.awq_last_device_error() == 0


@pytest.mark.parametrize("M,K,N,split_k", [(3, 1280, 416, 3), (9, 1280, 416, 0)])
def test_noalloc_matches_the_oracle(awq, M, K, N, split_k):
    # the same check straight against the CPU oracle (unrounded float64 product of its fp16 weights):
    # |y - ref| <= 2e-3 * rms(ref) + 2^-11 |ref|, the bar of the GEMV parity tests
    p = synth.awq_problem(M, K, N, seed=950 + M)
    x, qw, qz, sc = _dev(p["x"]), _dev(p["qweight"]), _dev(p["qzeros"]), _dev(p["scales"])
    ref = oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    rms = np.sqrt(np.mean(ref ** 2))
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc_via_abi(awq, x, qw, qz, sc, y, split_k) == 0
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref) - 2.0 ** -11 * np.abs(ref)) <= TOL * rms
        assert awq.awq_last_device_error() == 0


def test_noalloc_rejects_a_split_whose_scratch_exceeds_the_array(awq):
    # N = 153600 is 300 tiles of 512 columns.  split_k = 2 asks for 600 CTAs, clamped to one per SM;
    # with K = 256 (4 row blocks per tile) the tiles then straddle CTAs, two contributors each:
    # 300 tiles * 2 * (8 tokens * 512 columns * 4 bytes) = 9.8 MB of partials > 8 MiB.
    M, K, N = 8, 256, 153600
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    qw = torch.zeros((K, N // 8), dtype=torch.int32, device="cuda")
    sc = torch.zeros((K // 128, N), dtype=torch.float16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert _noalloc_via_abi(awq, x, qw, None, sc, y, 2) == EWORKSPACE
    # the automatic split falls back to one CTA per tile, which needs no scratch
    assert _noalloc_via_abi(awq, x, qw, None, sc, y, 0) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 0)
