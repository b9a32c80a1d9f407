"""fa_fwd_noalloc, the entry point for callers that cannot allocate device memory (code inside an
allocator or memory-pool callback, processes whose device memory a framework pool reserved up
front, fixed-footprint serving paths). Its kernel's scratch is a static device array instead of
cudaMalloc'd memory; the output must match fa_fwd's on every call.

Collected last on purpose: if it fails, a run that stops at the first failure has already run
every other test. It passes alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest

from tests import parity
from tiled_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_gb300 import fa as fa_mod

    fa_mod.lib()
    return fa_mod


def _call(fn, w, q, k, v, o, stream):
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), w.B, w.H, w.Nq, w.Nk, w.D,
              w.scale, int(w.causal), w.dtype_code, stream.cuda_stream)


@pytest.mark.parametrize("w", [
    inputs.Workload("noalloc_ragged_causal", 2, 3, 300, 300, 128, "bf16", True, seed=31),
    inputs.Workload("noalloc_f16", 1, 4, 257, 190, 64, "f16", False, seed=32),
], ids=lambda w: w.name)
def test_noalloc_matches_fa_fwd_on_two_calls(fa, w):
    stream = torch.cuda.current_stream()
    for call in range(2):  # two calls in a row: the shared scratch keeps the last call's contents
        bits = inputs.draw(w.with_(seed=w.seed + call))
        q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
        o_ref = torch.empty_like(q)
        o_new = torch.full_like(q, 3.0)
        # fa_fwd as one launch, the form fa_fwd_noalloc always takes (fa_fwd may otherwise split
        # some shapes over keys, which changes the rounding of those rows).
        try:
            fa.set_tail_split(False)
            assert _call(fa.fa_fwd, w, q, k, v, o_ref, stream) == 0
        finally:
            fa.set_tail_split(True)
        st = _call(fa.fa_fwd_noalloc, w, q, k, v, o_new, stream)
        assert st == 0, fa.lib().fa_last_error_message().decode()
        torch.cuda.synchronize()
        ref = inputs.bits_to_f64(inputs.from_torch(o_ref), w.dtype)
        stats = parity.compare(inputs.from_torch(o_new), ref, w.dtype)
        assert stats["finite"]
        assert stats["max_err"] <= parity.MAX_ERR and stats["mean_err"] <= parity.MEAN_ERR
        # Same kernel, same single launch, same inputs: in fact identical bits.
        assert np.array_equal(inputs.from_torch(o_new), inputs.from_torch(o_ref))
        assert fa.last_device_error(stream) == (0, 0)  # the static record stayed clear


def test_noalloc_rejects_like_fa_fwd(fa):
    assert fa.lib().fa_wait_selftest_noalloc(0, None) == 1
    q = torch.zeros(1, 1, 128, 96, dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    assert fa.fa_fwd_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 1, 1, 128,
                             128, 96, 0.1, 0, 0, 0) == 2


def test_noalloc_record_reports_a_timeout(fa):
    """A bounded wait that runs out while the static record is its target (the self-test's wait
    on a barrier nothing arrives on) is reported by fa_last_device_error, which clears it; the
    next allocation-free call then runs clean."""
    stream = torch.cuda.current_stream()
    assert fa.last_device_error(stream) == (0, 0)
    fa.wait_selftest_noalloc(2_000_000, stream)  # 2 ms
    assert fa.last_device_error(stream) == (5, 30)  # FA_ERR_TIMEOUT at the self-test's site
    assert fa.last_device_error(stream) == (0, 0)   # read and cleared
    w = inputs.Workload("noalloc_after_timeout", 1, 2, 200, 300, 128, "bf16", False, seed=33)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o = torch.empty_like(q)
    assert _call(fa.fa_fwd_noalloc, w, q, k, v, o, stream) == 0
    assert fa.last_device_error(stream) == (0, 0)
    want = fa.forward(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    diff = np.abs(inputs.bits_to_f64(inputs.from_torch(o), w.dtype)
                  - inputs.bits_to_f64(inputs.from_torch(want), w.dtype))
    assert diff.max() <= 2e-2
