"""Failure detection on the device, without a fault.

Every wait in the kernels is bounded: past its limit the waiting thread records a site code in
the device error word and the kernel winds down, so the host learns of the stall from
fa_last_device_error and the CUDA context stays usable. The self-test kernel waits through the
same routine on a barrier that nothing arrives on, which makes the wait run out on purpose.
"""
import pytest

import oracle
from tests import parity
from tiled_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SITE_SELFTEST = 30
FA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_gb300 import fa as fa_mod

    fa_mod.lib()
    return fa_mod


def _forward_matches_oracle(fa, w):
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    assert fa.last_device_error() == (0, 0)
    ref = oracle.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), w.scale,
                           w.causal)
    parity.assert_parity(parity.compare(inputs.from_torch(o), ref, w.dtype), True, w.name)


@pytest.mark.parametrize("timeout_ms", [2, 50])
def test_wait_runs_out_and_is_reported(fa, timeout_ms):
    fa.last_device_error()  # start from a clear error word
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    fa.wait_selftest(timeout_ms * 1_000_000, stream)
    t1.record(stream)
    status, site = fa.last_device_error(stream)
    assert (status, site) == (FA_ERR_TIMEOUT, SITE_SELFTEST)
    elapsed = t0.elapsed_time(t1)
    assert timeout_ms <= elapsed < timeout_ms + 500
    # The word was cleared by the read, and the context still runs kernels correctly.
    assert fa.last_device_error() == (0, 0)
    _forward_matches_oracle(fa, inputs.WORKLOADS["single_head"])


def test_first_report_wins(fa):
    fa.last_device_error()
    fa.wait_selftest(1_000_000)
    w = inputs.WORKLOADS["ragged"]
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    fa.forward(q, k, v, scale=w.scale)  # completes normally after the self-test's report
    assert fa.last_device_error() == (FA_ERR_TIMEOUT, SITE_SELFTEST)
    assert fa.last_device_error() == (0, 0)
