"""fa_fwd_lse: O and the per-row log-sum-exp against the fp64 oracle.

The kernel's LSE is log of the denominator that O is divided by: m + log sum_j P_j over the
16-bit-rounded weights P the PV product uses. Each rounded weight is within 2^-9 (bf16) of its
exact value, so l and exp(LSE) are within that relative error of the exact sum, i.e.
|LSE - LSE_ref| <= 2^-9 plus fp32 rounding. The test allows 4e-3.
"""
import numpy as np
import pytest

import oracle
from tests import parity
from tiled_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
LSE_TOL = 4e-3


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_gb300 import fa as fa_mod

    fa_mod.lib()
    return fa_mod


CASES = [
    inputs.WORKLOADS["single_head"],
    inputs.WORKLOADS["ragged"].with_(causal=True),
    inputs.Workload("lse_ragged_bf16", 2, 3, 300, 700, 128, "bf16", False, seed=41),
    inputs.WORKLOADS["causal_prefill"].with_(H=4),
    inputs.WORKLOADS["rescale_stress"].with_(B=1, H=2, Nq=1024, Nk=1024),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_lse_matches_oracle(fa, w):
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o, lse = fa.forward_lse(q, k, v, causal=w.causal, scale=w.scale)
    o_plain = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    ref_o, ref_lse = oracle.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"),
                                      w.scale, w.causal, with_lse=True)
    got_lse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_lse))
    assert np.max(np.abs(got_lse - ref_lse)) <= LSE_TOL
    # The LSE path writes the same O as fa_fwd.
    assert torch.equal(o.view(torch.int16), o_plain.view(torch.int16))
    stats = parity.compare(inputs.from_torch(o), ref_o, w.dtype)
    parity.describe(w)
    if w.sigma_q == 1.0:
        parity.assert_parity(stats, True, w.name)
    else:  # the large-magnitude distribution: max beyond output rounding, literal mean
        parity.assert_parity(stats, False, w.name, mean="literal")


def test_lse_rejects_bad_pointer(fa):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(2, dtype=torch.float32, device="cuda")
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr())
    assert fa.lib().fa_fwd_lse(*args, 0, 1, 1, 128, 128, 64, 0.1, 0, 0, None) == 1
    assert fa.lib().fa_fwd_lse(*args, lse.data_ptr() + 2, 1, 1, 128, 128, 64, 0.1, 0, 0, None) == 3
