"""Host-side checks of the C ABI (no GPU needed, no compute call is made).

* the library builds and exports every function include/awq.h declares;
* argument checks reject bad shapes, NULL and misaligned pointers and short
  workspaces before anything touches the GPU;
* workspace sizing follows the documented layout.
"""

import ctypes
import re
import subprocess

import pytest

from bit_weight_only_awq_gb300 import build as awq_build


@pytest.fixture(scope="module")
def awq():
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq as mod
    return mod


EINVAL, EALIGN, EWORKSPACE, ENULL = -1, -2, -6, -7
FAKE = 1 << 40          # an aligned address that is never dereferenced (checks run first)
FAKE_MISALIGNED = FAKE + 4


def test_header_declares_the_boundary(awq):
    names = awq.header_functions()
    for want in ("awq_pack", "awq_unpack", "awq_dequant", "awq_gemv", "awq_gemm", "awq_workspace_bytes",
                 "w4a8_quant_act", "w4a8_gemm", "w4a8_linear", "awq_status_string", "awq_last_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(awq):
    out = subprocess.run(["nm", "-D", "--defined-only", awq._LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    for name in awq.header_functions():
        assert name in exported, name
        assert getattr(awq.lib, name) is not None


def test_status_strings(awq):
    for code, name in awq.STATUS.items():
        assert awq.lib.awq_status_string(code).decode().startswith(name)


def _gemv(awq, M=1, K=4096, N=4096, g=128, split=0, x=FAKE, qw=FAKE, qz=FAKE, sc=FAKE, y=FAKE, ws=None, wsb=0):
    return awq.lib.awq_gemv(x, qw, qz, sc, y, M, K, N, g, split, ws, wsb, None)


def test_gemv_rejects_bad_shapes_before_launch(awq):
    assert _gemv(awq, M=17) == EINVAL          # the decode kernel takes up to 16 tokens
    assert _gemv(awq, M=-1) == EINVAL
    assert _gemv(awq, K=100) == EINVAL
    assert _gemv(awq, N=24) == EINVAL
    assert _gemv(awq, N=48) == EINVAL           # the TMA row stride needs N % 32 == 0
    assert _gemv(awq, g=64) == EINVAL
    assert _gemv(awq, split=-2) == EINVAL


def test_gemv_rejects_null_and_misaligned(awq):
    assert _gemv(awq, x=None) == ENULL
    assert _gemv(awq, y=None) == ENULL
    assert _gemv(awq, qw=FAKE_MISALIGNED) == EALIGN
    assert _gemv(awq, sc=FAKE_MISALIGNED) == EALIGN


def test_gemv_requires_workspace_when_split(awq):
    need = awq.awq_workspace_bytes(awq.OP_GEMV, 4, 4096, 4096, 4)
    assert need > 0
    assert _gemv(awq, M=4, split=4) == EWORKSPACE
    assert _gemv(awq, M=4, split=4, ws=FAKE, wsb=need - 1) == EWORKSPACE
    assert _gemv(awq, M=4, split=4, ws=FAKE + 16, wsb=need) == EALIGN   # workspace wants 256-byte alignment


def test_empty_batch_is_a_noop(awq):
    assert _gemv(awq, M=0, x=None, y=None) == 0
    assert awq.lib.awq_gemm(None, None, None, None, None, 0, 4096, 4096, 128, 0, None, 0, None) == 0
    assert awq.lib.awq_pack(None, 0, 64, None, None) == 0


def test_gemm_and_w4a8_argument_checks(awq):
    f = awq.lib.awq_gemm
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 256, 4096, 4112, 128, 0, None, 0, None) == EINVAL   # N % 32
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 256, 4000, 4096, 128, 0, None, 0, None) == EINVAL   # K % 128
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 256, 4096, 4096, 32, 0, None, 0, None) == EINVAL    # group size
    g = awq.lib.w4a8_gemm
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 21760, 8192, 0, None, 0, None) == EWORKSPACE
    assert g(None, FAKE, FAKE, FAKE, FAKE, None, 4, 21760, 8192, 0, None, 0, None) == ENULL
    lin = awq.lib.w4a8_linear  # x, wq, s_ch, y, acc_out, xq_out, s_tok, M, K, N, split_k, ws, bytes, stream
    assert lin(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 4, 21760, 8192, 0, None, 0, None) == EWORKSPACE
    assert lin(FAKE, FAKE, FAKE, FAKE, None, None, None, 4, 21760, 8192, 0, None, 0, None) == ENULL  # s_tok
    assert lin(FAKE, FAKE, FAKE, FAKE, None, FAKE_MISALIGNED, FAKE, 4, 21760, 8192, 0, None, 0, None) == EALIGN
    assert lin(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 4, 21700, 8192, 0, None, 0, None) == EINVAL   # K % 128
    assert lin(None, FAKE, FAKE, FAKE, None, None, FAKE, 0, 21760, 8192, 0, None, 0, None) == 0       # M = 0
    q = awq.lib.w4a8_quant_act
    assert q(FAKE, FAKE, FAKE, 4, 100, None) == EINVAL
    assert q(FAKE, FAKE_MISALIGNED, FAKE, 4, 128, None) == EALIGN
    assert awq.lib.awq_dequant(FAKE, None, FAKE, 128, 64, 96, FAKE, None) == EINVAL
    assert awq.lib.awq_unpack(FAKE, 4, 12, FAKE, None) == EINVAL


def align256(n):
    return (n + 255) // 256 * 256


def test_workspace_layout(awq):
    counters = 65536
    # GEMV: counters block + split x M x N fp32 partials (256-byte rounded)
    assert awq.awq_workspace_bytes(awq.OP_GEMV, 8, 4096, 4096, 1) == 0
    assert awq.awq_workspace_bytes(awq.OP_GEMV, 8, 4096, 4096, 4) == counters + 4 * 8 * 4096 * 4
    # 9..16 tokens: partials carry 16 token rows
    assert awq.awq_workspace_bytes(awq.OP_GEMV, 12, 4096, 4096, 4) == counters + 4 * 16 * 4096 * 4
    # W4A8 at K = 21760 and 4096 tokens: two M-blocks per CTA (one exact accumulator each) with a K split
    # of two (slices of 10880 rows), which the plan's cost model rates faster than one M-block covering
    # K with its two accumulators
    x16 = 4096 * 21760 * 2
    assert awq.awq_workspace_bytes(awq.OP_W4A8_GEMM, 4096, 21760, 8192, 0) == counters + x16 + 2 * 4096 * 8192 * 4
    assert awq.awq_workspace_bytes(awq.OP_W4A8_GEMM, 16, 21760, 8192, 1) == counters + 16 * 21760 * 2
    # 256 tokens: 256-token tiles with two M-blocks and a K split of four (128 CTAs, slices of 5440 rows)
    # are rated faster by the plan's cost model than 128-token tiles running all 21760 rows
    assert awq.awq_workspace_bytes(awq.OP_W4A8_GEMM, 256, 21760, 8192, 0) == \
        counters + 256 * 21760 * 2 + 4 * 256 * 8192 * 4
    # K beyond 2 x 16384 rows forces a K split across CTAs with int32 partials
    assert awq.awq_workspace_bytes(awq.OP_W4A8_GEMM, 4096, 40960, 8192, 1) == \
        counters + 4096 * 40960 * 2 + 2 * 4096 * 8192 * 4
    # small-K W4A8 without split still needs the fp16 copy of the codes
    assert awq.awq_workspace_bytes(awq.OP_W4A8_GEMM, 4096, 4096, 8192, 1) == counters + 4096 * 4096 * 2
    # W4A8 with group factors: 64-token tiles keep at most 8 chunks of 1024 rows per K slice, so
    # K = 21760 splits in three (int32 partials); 128- and 256-token tiles drain their chunks during the
    # main loop and need no split
    g = awq.OP_W4A8_GROUPED
    assert awq.awq_workspace_bytes(g, 64, 21760, 8192, 0) == counters + 64 * 21760 * 2 + 3 * 64 * 8192 * 4
    assert awq.awq_workspace_bytes(g, 1000, 21760, 8192, 0) == counters + align256(1000 * 21760 * 2)
    assert awq.awq_workspace_bytes(g, 4096, 21760, 8192, 0) == counters + 4096 * 21760 * 2
    # 256 tokens: 256-token tiles with a K split of two (int32 partials) are rated faster by the plan's
    # cost model than 128-token tiles running all 21760 rows
    assert awq.awq_workspace_bytes(g, 256, 21760, 8192, 0) == counters + 256 * 21760 * 2 + 2 * 256 * 8192 * 4
    # invalid shapes need nothing (the compute call reports the error)
    assert awq.awq_workspace_bytes(awq.OP_GEMM, 16, 100, 4096, 0) == 0


def test_gemm_plan_split_choices(awq):
    # The automatic GEMM plan shows in the workspace it asks for: the counters block plus
    # split x M x N fp32 partials when it splits K, nothing otherwise.
    counters = 65536
    ws = lambda M, K, N: awq.awq_workspace_bytes(awq.OP_GEMM, M, K, N, 0)
    # one M-block fits one wave (128 CTAs of 64 tokens): no split
    assert ws(256, 4096, 4096) == 0
    # above 64 tokens the measured cost model may replace that plan: 256 tokens over 6144 columns take
    # one M-block of 128-token tiles in one wave (96 CTAs) instead of two M-blocks with a split of three
    assert ws(256, 4096, 6144) == 0
    # two M-blocks fill the wave with slices of 56 k-steps: split of four (the model's best differs by
    # less than 5 %, so the plan stays)
    assert ws(256, 14336, 4096) == counters + 4 * 256 * 4096 * 4
    # 1024 tokens at K = 14336: two M-blocks of 256 tokens with a split of two (128 CTAs) instead of 128
    # CTAs of 128-token tiles running 224 k-steps each
    assert ws(1024, 14336, 4096) == counters + 2 * 1024 * 4096 * 4
    # under a wave with one M-block: the largest split that stays within one wave (32 x 4 CTAs)
    assert ws(64, 4096, 4096) == counters + 4 * 64 * 4096 * 4
    # a full wave without splitting
    assert ws(64, 4096, 28672) == 0
    assert ws(1024, 4096, 6144) == 0


def test_w4a8_route_by_token_count(awq):
    # W4A8 with at most 16 tokens runs on the GEMV when every CTA's rows of a tile stay within 16384; its
    # workspace is counters | fp16 codes | the GEMV's partial slots, sized for 16 token rows.
    counters = 65536
    a256 = lambda b: (b + 255) // 256 * 256
    ws = lambda M, K, N, sp: awq.awq_workspace_bytes(awq.OP_W4A8_GEMM, M, K, N, sp)
    gemv_partials = awq.awq_workspace_bytes(awq.OP_GEMV, 16, 21760, 8192, 0) - counters
    assert gemv_partials > 0
    for M in (1, 16):
        assert ws(M, 21760, 8192, 0) == counters + a256(M * 21760 * 2) + gemv_partials
    # split_k = 1: one CTA per tile would cover all 21760 rows, so the GEMM takes the call
    assert ws(16, 21760, 8192, 1) == counters + 16 * 21760 * 2
    # 17 tokens: the GEMM (one M-block, two exact accumulators, K split of two to fill the SMs)
    assert ws(17, 21760, 8192, 0) == counters + a256(17 * 21760 * 2) + 2 * 17 * 8192 * 4
    # K = 4096 with one CTA per tile: the GEMV without partials
    assert ws(8, 4096, 4096, 1) == counters + 8 * 4096 * 2


def test_selftest_rejects_bad_limits_before_launch(awq):
    assert awq.lib.awq_selftest_wait_timeout(0, None) == EINVAL
    assert awq.lib.awq_selftest_wait_timeout(-5, None) == EINVAL
    assert awq.lib.awq_selftest_wait_timeout(3_000_000_000, None) == EINVAL


def test_binding_has_no_fallback(awq):
    src = open(awq.__file__).read()
    assert "oracle" not in src
    assert "numpy" not in src


def test_prepared_layout_entry_points_check_arguments(awq):
    lib = awq.lib
    # size of the prepared copy: ceil(N / 256) tiles x K / 128 groups x 17024 bytes
    assert lib.awq_prepacked_bytes(4096, 4096) == 16 * 32 * 17024
    assert lib.awq_prepacked_bytes(4096, 4128) == 17 * 32 * 17024
    assert lib.awq_prepacked_bytes(100, 4096) == 0 and lib.awq_prepacked_bytes(4096, 40) == 0
    need = lib.awq_prepacked_bytes(256, 512)
    assert lib.awq_prepack_gemv(FAKE, FAKE, FAKE, 256, 512, 128, FAKE, need - 16, None) == EINVAL
    assert lib.awq_prepack_gemv(FAKE, FAKE, FAKE, 256, 512, 64, FAKE, need, None) == EINVAL
    assert lib.awq_prepack_gemv(None, FAKE, FAKE, 256, 512, 128, FAKE, need, None) == ENULL
    assert lib.awq_prepack_gemv(FAKE, FAKE, FAKE, 256, 512, 128, FAKE_MISALIGNED, need, None) == EALIGN
    assert lib.awq_unprepack_gemv(FAKE, 256, 500, FAKE, FAKE, FAKE, None) == EINVAL
    gp = lib.awq_gemv_prepacked
    assert gp(FAKE, FAKE, FAKE, 9, 4096, 4096, 0, None, 0, None) == EINVAL      # up to 8 tokens
    assert gp(FAKE, FAKE, FAKE, 0, 4096, 4096, 0, None, 0, None) == 0           # empty batch: no-op
    assert gp(FAKE, None, FAKE, 4, 4096, 4096, 0, None, 0, None) == ENULL
    assert gp(FAKE_MISALIGNED, FAKE, FAKE, 4, 4096, 4096, 0, None, 0, None) == EALIGN
    # shared tiles need a workspace; split 1 (one CTA per tile) needs none
    ws = awq.awq_workspace_bytes(awq.OP_GEMV_PREPACKED, 4, 4096, 4096, 0)
    assert ws > 65536 and gp(FAKE, FAKE, FAKE, 4, 4096, 4096, 0, None, 0, None) == EWORKSPACE
    assert awq.awq_workspace_bytes(awq.OP_GEMV_PREPACKED, 4, 4096, 4096, 1) == 0
    assert awq.awq_workspace_bytes(awq.OP_GEMV_PREPACKED, 9, 4096, 4096, 0) == 0


def test_order_map_entry_points_check_arguments(awq):
    lib = awq.lib
    assert lib.awq_pack_order(FAKE, 4, 16, 2, FAKE, None) == EINVAL     # no third order map
    assert lib.awq_unpack_order(FAKE, 4, 12, 1, FAKE, None) == EINVAL   # n % 8
    assert lib.awq_pack_order(None, 4, 16, 1, FAKE, None) == ENULL
    assert lib.awq_unpack_order(FAKE, 4, 16, 0, FAKE_MISALIGNED, None) == EALIGN
    assert lib.awq_pack_order(FAKE, 0, 16, 1, FAKE, None) == 0          # nothing to pack
