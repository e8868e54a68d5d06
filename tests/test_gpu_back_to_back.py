"""Calls issued back to back on one stream give the results of the same calls separated by
synchronizes.

The GEMV and GEMM kernels are launched with programmatic dependent launch: a call's set-up and weight
stream overlap the previous kernel, and only its activation copies and its writes (outputs, split-K
partials and tile counters in the shared workspace) wait for it.  The W4A8 quantization kernels let
the GEMM after them launch early.  A chain of different entry points in which every call reads the
previous call's output, with split-K workspaces shared between the calls, goes through each of those
waits; before every chained run the outputs are overwritten with a NaN pattern, so that a read or a
write ahead of the previous kernel shows as a difference.
"""

import numpy as np
import pytest

from bit_weight_only_awq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

K = 4096  # every layer is 4096 -> 4096, so each output feeds the next call


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


def _layers(awq):
    w16 = [synth.awq_problem(1, K, K, seed=9600 + i, with_x=False) for i in range(4)]
    w16 = [(dev(p["qweight"]), dev(p["qzeros"]), dev(p["scales"])) for p in w16]
    w8 = synth.w4a8_problem(1, K, K, seed=9610, with_x=False)
    g8 = synth.w4a8_group_problem(1, K, K, seed=9611, with_x=False)
    return {
        "w16": w16,
        "pp": awq.awq_prepack_gemv(*w16[2]),
        "w8": (dev(w8["wq"]), dev(w8["s_ch"])),
        "g8": (dev(g8["wq"]), dev(g8["s3"]), dev(g8["s2"])),
    }


def _chain(awq, L, x0, outs):
    """256 tokens through the tensor-core GEMM (split K) and W4A8, then 8 tokens through the prepared
    GEMV, the GEMM's 16-token tiles, per-group W4A8 and the AWQ-layout GEMV."""
    w16 = L["w16"]
    awq.awq_gemm(x0, *w16[0], out=outs[0])
    awq.w4a8_linear(outs[0], *L["w8"], out=outs[1])
    awq.awq_gemv_prepacked(outs[1][:8], L["pp"], out=outs[2])
    awq.awq_gemm(outs[2], *w16[1], out=outs[3])
    awq.w4a8_linear_grouped(outs[3], *L["g8"], out=outs[4])
    awq.awq_gemv(outs[4], *w16[3], out=outs[5])


def _outputs(M=256):
    rows = [M, M, 8, 8, 8, 8]
    return [torch.empty((r, K), dtype=torch.float16, device="cuda") for r in rows]


def test_chain_back_to_back_matches_synchronized_calls(awq):
    L = _layers(awq)
    x0 = dev((np.random.default_rng(9620).standard_normal((256, K)) * 0.05).astype(np.float16))
    # reference: every call alone, with a synchronize before and after it
    ref = _outputs()
    w16 = L["w16"]
    steps = [
        lambda o: awq.awq_gemm(x0, *w16[0], out=o[0]),
        lambda o: awq.w4a8_linear(o[0], *L["w8"], out=o[1]),
        lambda o: awq.awq_gemv_prepacked(o[1][:8], L["pp"], out=o[2]),
        lambda o: awq.awq_gemm(o[2], *w16[1], out=o[3]),
        lambda o: awq.w4a8_linear_grouped(o[3], *L["g8"], out=o[4]),
        lambda o: awq.awq_gemv(o[4], *w16[3], out=o[5]),
    ]
    for s in steps:
        torch.cuda.synchronize()
        s(ref)
        torch.cuda.synchronize()
    ref_bits = [r.view(torch.int16).cpu().numpy() for r in ref]
    assert all(np.isfinite(r.float().cpu().numpy()).all() for r in ref)
    # the same chain issued back to back, three times, into outputs filled with NaN before each run
    outs = _outputs()
    for _ in range(3):
        for o in outs:
            o.view(torch.int16).fill_(0x7E01)
        torch.cuda.synchronize()
        _chain(awq, L, x0, outs)
        torch.cuda.synchronize()
        for i, (o, r) in enumerate(zip(outs, ref_bits)):
            assert np.array_equal(o.view(torch.int16).cpu().numpy(), r), f"call {i} differs back to back"
    assert awq.awq_last_device_error() == 0
