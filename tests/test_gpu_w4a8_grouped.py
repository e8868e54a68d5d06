"""GPU parity of W4A8 with per-group weight factors (through the C ABI) against the CPU oracle.

acc[m, n] = sum_k xq[m, k] (u[k, n] - 8) s3[k / 128, n] is an exact integer and y =
fp16((fp32(acc) s_tok[m]) s2[n]): both are compared bit for bit (the oracle's
w4a8_group_linear), on small ragged shapes spanning several 1024-row chunks and K slices, on
128-token tiles whose chunks are drained into int32 sums during the main loop (0 to 2 chunks
drained there, the rest in the epilogue), on the W4A8 configuration's shape with sampled
columns, and on extreme codes where every chunk's sum reaches 2^24.
"""

import numpy as np
import pytest

import oracle
from bit_weight_only_awq_gb300 import synth
from tests.test_gpu_parity import sample_word_cols

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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def run(awq, p, split_k=0, xq=None):
    """The library's quantization + grouped product; returns (xq, s_tok, y, acc)."""
    M, K = p["x"].shape
    N = p["wq"].shape[1] * 8
    if xq is None:
        xq_t, s_t = awq.w4a8_quant_act(dev(p["x"]))
    else:
        xq_t, s_t = dev(xq), dev(np.ones(M, np.float32))
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = awq.w4a8_gemm_grouped(xq_t, s_t, dev(p["wq"]), dev(p["s3"]), dev(p["s2"]), split_k=split_k, acc_out=acc)
    return host(xq_t), host(s_t), host(y), host(acc)


@pytest.mark.parametrize("split_k", [1, 2, 0])
@pytest.mark.parametrize("M", [1, 5, 16, 40, 64, 100])
def test_w4a8_grouped_small_bitexact(awq, M, split_k):
    # K = 2560: 20 groups, 2.5 chunks of 1024 rows; N = 288: a ragged last 128-column tile
    p = synth.w4a8_group_problem(M, 2560, 288, seed=9000 + M + 10 * split_k)
    xq, s, y, acc = run(awq, p, split_k)
    want_y, want_acc = oracle.w4a8_group_linear(xq, s, p["wq"], p["s3"], p["s2"], 128)
    assert np.array_equal(acc, want_acc)
    assert np.array_equal(y.view(np.uint16), want_y.view(np.uint16))


@pytest.mark.parametrize("M", [1, 16, 64, 256, 1000])
def test_w4a8_grouped_config_shape_sampled(awq, M):
    K, N = synth.W4A8_SHAPE
    p = synth.w4a8_group_problem(M, K, N, seed=9100 + M)
    xq, s, y, acc = run(awq, p)
    wc = sample_word_cols(N // 8, seed=M + 9, count=6)
    cols = (8 * wc[:, None] + np.arange(8)[None, :]).ravel()
    want_y, want_acc = oracle.w4a8_group_linear(xq, s, p["wq"][:, wc], p["s3"][:, cols], p["s2"][cols], 128)
    assert np.array_equal(acc[:, cols], want_acc)
    assert np.array_equal(y[:, cols].view(np.uint16), want_y.view(np.uint16))


@pytest.mark.parametrize("split_k", [0, 1])
def test_w4a8_grouped_extreme_chunks(awq, split_k):
    # codes -128 against weights (0 - 8) * 16 = -128: every product is 2^14 and every 1024-row chunk sums
    # to exactly 2^24; across K = 21760 the accumulator reaches 356 million (int32, exact)
    M, K, N = 2, 21760, 256
    xq = np.full((M, K), -128, dtype=np.int8)
    xq[1, 1::2] = 127
    wq = np.zeros((K, N // 8), dtype=np.int32)            # every nibble 0: u - 8 = -8
    p = {"x": np.zeros((M, K), np.float16), "wq": wq, "s3": np.full((K // 128, N), 16, np.float16),
         "s2": np.full(N, 1e-6, np.float16)}
    _, s, y, acc = run(awq, p, split_k, xq=xq)
    want_y, want_acc = oracle.w4a8_group_linear(xq, s, wq, p["s3"], p["s2"], 128)
    assert want_acc[0, 0] == K * 16384
    assert np.array_equal(acc, want_acc)
    assert np.array_equal(y.view(np.uint16), want_y.view(np.uint16))


@pytest.mark.parametrize("split_k", [0, 2])
@pytest.mark.parametrize("K", [1280, 1408, 2304, 2432, 3200])
def test_w4a8_grouped_drained_chunks_sampled(awq, K, split_k):
    # 1000 tokens over 1952 columns take 128-token tiles (the last one 104 tokens, the last column tile 32
    # columns), whose 1024-row chunks alternate between two accumulators; every chunk but a slice's last
    # is drained into int32 sums once the next chunk is four k-steps in, or after the loop when the slice
    # ends first (K = 1280: 20 k-steps).  K = 1280 .. 3200 gives 2 to 4 chunks per slice; split 2 halves
    # every slice.
    M, N = 1000, 1952
    p = synth.w4a8_group_problem(M, K, N, seed=9400 + K + split_k)
    xq, s, y, acc = run(awq, p, split_k)
    wc = sample_word_cols(N // 8, seed=K + split_k, count=6)
    cols = (8 * wc[:, None] + np.arange(8)[None, :]).ravel()
    want_y, want_acc = oracle.w4a8_group_linear(xq, s, p["wq"][:, wc], p["s3"][:, cols], p["s2"][cols], 128)
    assert np.array_equal(acc[:, cols], want_acc)
    assert np.array_equal(y[:, cols].view(np.uint16), want_y.view(np.uint16))
    assert awq.awq_last_device_error() == 0


@pytest.mark.parametrize("split_k", [0, 2])
@pytest.mark.parametrize("K", [1024, 1152, 2176, 3200])
def test_w4a8_grouped_drained_chunks_256_token_tiles_sampled(awq, K, split_k):
    # 2000 tokens over 1952 columns take 256-token tiles (the last one 208 tokens) with one chunk
    # accumulator: the mmas of a chunk wait until the dequant warps have drained the one before, at the
    # first two k-steps of the new chunk.  K = 1024 (one chunk, nothing drained), 1152 (a last chunk of
    # two k-steps), 2176, 3200; with split 2 the 2176 slices end in a one-k-step chunk whose predecessor
    # one dequant group drains after its loop.
    M, N = 2000, 1952
    p = synth.w4a8_group_problem(M, K, N, seed=9450 + K + split_k)
    xq, s, y, acc = run(awq, p, split_k)
    wc = sample_word_cols(N // 8, seed=K + split_k + 1, count=5)
    cols = (8 * wc[:, None] + np.arange(8)[None, :]).ravel()
    want_y, want_acc = oracle.w4a8_group_linear(xq, s, p["wq"][:, wc], p["s3"][:, cols], p["s2"][cols], 128)
    assert np.array_equal(acc[:, cols], want_acc)
    assert np.array_equal(y[:, cols].view(np.uint16), want_y.view(np.uint16))
    assert awq.awq_last_device_error() == 0


@pytest.mark.parametrize("M,split_k", [(256, 1), (256, 0), (512, 1)])
def test_w4a8_grouped_drained_extreme_chunks(awq, M, split_k):
    # every 1024-row chunk sums to exactly 2^24 in its fp32 accumulator (codes -128 against weights
    # (0 - 8) * 16), and the drained int32 sums reach 21760 * 2^14 = 356 million: over 7424 columns, 256
    # tokens without a split take 128-token tiles (two accumulators), with the automatic plan 256-token
    # tiles and a K split of two; 512 tokens 256-token tiles (one accumulator)
    K, N = 21760, 7424
    xq = np.full((M, K), -128, dtype=np.int8)
    xq[1::3, 1::2] = 127
    wq = np.zeros((K, N // 8), dtype=np.int32)
    p = {"x": np.zeros((M, K), np.float16), "wq": wq, "s3": np.full((K // 128, N), 16, np.float16),
         "s2": np.full(N, 1e-6, np.float16)}
    _, s, y, acc = run(awq, p, split_k, xq=xq)
    wc = np.array([0, 17, N // 8 - 1])
    cols = (8 * wc[:, None] + np.arange(8)[None, :]).ravel()
    want_y, want_acc = oracle.w4a8_group_linear(xq, s, wq[:, wc], p["s3"][:, cols], p["s2"][cols], 128)
    assert want_acc[0, 0] == K * 16384
    assert np.array_equal(acc[:, cols], want_acc)
    assert np.array_equal(y[:, cols].view(np.uint16), want_y.view(np.uint16))


@pytest.mark.parametrize("M,K,N", [(1, 21760, 8192), (300, 4096, 1024)])
def test_w4a8_linear_grouped_matches_two_calls(awq, M, K, N):
    p = synth.w4a8_group_problem(M, K, N, seed=9200 + M)
    xq, s, y2, acc2 = run(awq, p)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    xq_out = torch.empty((M, K), dtype=torch.int8, device="cuda")
    y, s_tok = awq.w4a8_linear_grouped(dev(p["x"]), dev(p["wq"]), dev(p["s3"]), dev(p["s2"]), acc_out=acc,
                                       xq_out=xq_out)
    assert np.array_equal(host(xq_out), xq)
    assert np.array_equal(host(s_tok).view(np.uint32), s.view(np.uint32))
    assert np.array_equal(host(acc), acc2)
    assert np.array_equal(host(y).view(np.uint16), y2.view(np.uint16))


def test_w4a8_grouped_factor_16_is_the_per_channel_kernel(awq):
    # s3 = 16 everywhere with s2 = s_ch / 16 (exact) gives the per-channel kernel's outputs bit for bit
    M, K, N = 40, 4096, 512
    p = synth.w4a8_problem(M, K, N, seed=9300)
    xq_t, s_t = awq.w4a8_quant_act(dev(p["x"]))
    y_c = awq.w4a8_gemm(xq_t, s_t, dev(p["wq"]), dev(p["s_ch"]))
    s3 = np.full((K // 128, N), 16, np.float16)
    s2 = (p["s_ch"].astype(np.float32) / 16).astype(np.float16)
    y_g = awq.w4a8_gemm_grouped(xq_t, s_t, dev(p["wq"]), dev(s3), dev(s2))
    assert np.array_equal(host(y_g).view(np.uint16), host(y_c).view(np.uint16))
    assert awq.awq_last_device_error() == 0
