"""GPU parity of the decode GEMV's prepared weight layout (through the C ABI) against the CPU oracle.

* awq_prepack_gemv: the prepared bytes equal the oracle's restatement of the layout, bit for bit,
  including ragged last tiles and the symmetric variant; awq_unprepack_gemv gives back the AWQ words,
  zero points and scales exactly;
* awq_gemv_prepacked: |y - y_oracle| <= 2e-3 rms(y_oracle) + 2^-11 |y_oracle| element by element (the
  bar of the other fp16 GEMV/GEMM outputs; y_oracle is the unrounded float64 product of the oracle's
  fp16 weights) on small ragged cases over several tiles and split choices, and on the decode shapes
  with sampled columns.
"""

import numpy as np
import pytest

import oracle
from bit_weight_only_awq_gb300 import synth
from tests.test_gpu_parity import assert_within_tol, dev, host, oracle_columns, sample_word_cols

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def awq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_awq_gb300 import build as awq_build
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq as mod
    return mod


def _prepack(awq, p):
    qz = None if p["qzeros"] is None else dev(p["qzeros"])
    return awq.awq_prepack_gemv(dev(p["qweight"]), qz, dev(p["scales"]))


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("K,N", [(128, 256), (256, 416), (384, 1056), (1280, 4096)])
def test_prepack_bitexact_and_round_trip(awq, K, N, symmetric):
    p = synth.awq_problem(1, K, N, seed=7000 + K + N, symmetric=symmetric)
    pk = _prepack(awq, p)
    want = oracle.prepack_gemv(p["qweight"], p["qzeros"], p["scales"])
    assert np.array_equal(host(pk.data), want)
    qw, qz, sc = awq.awq_unprepack_gemv(pk, with_zeros=not symmetric)
    assert np.array_equal(host(qw), p["qweight"])
    assert np.array_equal(host(sc).view(np.uint16), p["scales"].view(np.uint16))
    if not symmetric:
        assert np.array_equal(host(qz), p["qzeros"])


@pytest.mark.parametrize("symmetric", [False, True])
@pytest.mark.parametrize("split_k", [1, 3, 0])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_gemv_prepacked_small_ragged(awq, M, split_k, symmetric):
    # N = 416: two 256-column tiles, the second one 160 columns wide; K = 1280: 10 groups
    p = synth.awq_problem(M, 1280, 416, seed=7100 + M, symmetric=symmetric)
    pk = _prepack(awq, p)
    y = host(awq.awq_gemv_prepacked(dev(p["x"]), pk, split_k=split_k))
    ref = oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert_within_tol(y, ref, f"gemv prepacked M={M} split={split_k} sym={symmetric}")


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("name,K,N", synth.LLAMA2_7B_DECODE + (("down_l31", 14336, 4096),))
def test_gemv_prepacked_decode_shapes_sampled(awq, name, K, N, M):
    p = synth.awq_problem(M, K, N, seed=7200 + K + N + M)
    pk = _prepack(awq, p)
    y = host(awq.awq_gemv_prepacked(dev(p["x"]), pk))
    wc = sample_word_cols(N // 8, seed=K + N + 3, count=40)
    ref, cols = oracle_columns(p, wc)
    assert_within_tol(y[:, cols], ref, f"gemv prepacked {name} M={M}")


@pytest.mark.parametrize("xkind", ["common_mode", "outliers"])
def test_gemv_prepacked_activation_offsets(awq, xkind):
    M, K, N = 8, 14336, 1024
    p = synth.awq_problem(M, K, N, seed=7300)
    rng = np.random.default_rng(7301)
    z = rng.standard_normal((M, K))
    x = 20.0 + 0.1 * z if xkind == "common_mode" else z * np.where(rng.random((M, K)) < 0.01, 100.0, 1.0)
    p["x"] = x.astype(np.float16)
    pk = _prepack(awq, p)
    y = host(awq.awq_gemv_prepacked(dev(p["x"]), pk))
    ref = oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert_within_tol(y, ref, f"gemv prepacked {xkind} K={K}")


def test_gemv_prepacked_repeatable_and_back_to_back(awq):
    # the same call twice gives the same bits (fixed reduction order); calls issued back to back on one
    # stream (the next call's CTAs start while the previous one finishes) give the same results as
    # calls separated by a synchronize
    shapes = [(4096, 4096), (4096, 12288), (11008, 4096)]
    probs = [synth.awq_problem(8, K, N, seed=7400 + i) for i, (K, N) in enumerate(shapes)]
    packs = [_prepack(awq, p) for p in probs]
    xs = [dev(p["x"]) for p in probs]
    alone = []
    for x, pk in zip(xs, packs):
        alone.append(host(awq.awq_gemv_prepacked(x, pk)))
    outs = [awq.awq_gemv_prepacked(x, pk) for _ in range(3) for x, pk in zip(xs, packs)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert np.array_equal(host(o).view(np.uint16), alone[i % 3].view(np.uint16))
    assert awq.awq_last_device_error() == 0
