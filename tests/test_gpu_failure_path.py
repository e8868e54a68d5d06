"""The failure path of the kernels' bounded waits, exercised without a GPU fault.

Every mbarrier wait in the library's kernels gives up after a time limit, records the wait's id in
a per-device error word and lets the kernel return; awq_last_device_error reports it.  Here the
same wait runs on a barrier that nothing arrives on, with a 1 ms limit: the call must report
AWQ_ETIMEOUT with the self-test's id, clear the word, and leave the context usable for a normal
GEMV whose result still matches the oracle.
"""

import numpy as np
import pytest

import oracle
from bit_weight_only_awq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SELFTEST_ID = 901


@pytest.fixture(scope="module")
def awq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_weight_only_awq_gb300 import build as awq_build
    awq_build.build()
    from bit_weight_only_awq_gb300 import awq as mod
    return mod


def test_expired_wait_is_reported_and_the_context_stays_usable(awq):
    torch.cuda.synchronize()
    assert awq.awq_last_device_error() == 0
    awq.awq_selftest_wait_timeout(1_000_000)
    assert awq.awq_last_device_error() == SELFTEST_ID
    assert awq.awq_last_device_error() == 0          # reading clears the word
    p = synth.awq_problem(2, 1280, 416, seed=77)
    y = awq.awq_gemv(torch.from_numpy(p["x"]).cuda(), torch.from_numpy(p["qweight"]).cuda(),
                     torch.from_numpy(p["qzeros"]).cuda(), torch.from_numpy(p["scales"]).cuda(), 128)
    got = y.cpu().numpy().astype(np.float64)
    ref = oracle.awq_linear(p["x"], p["qweight"], p["qzeros"], p["scales"], 128)
    assert np.max(np.abs(got - ref) - 2.0 ** -11 * np.abs(ref)) <= 2e-3 * np.sqrt(np.mean(ref ** 2))
    assert awq.awq_last_device_error() == 0


def test_selftest_rejects_limits_outside_the_range(awq):
    for bad in (0, -1, 3_000_000_000):
        with pytest.raises(awq.AwqError):
            awq.awq_selftest_wait_timeout(bad)
