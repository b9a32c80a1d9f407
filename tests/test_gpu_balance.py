"""fa_fwd's work balancing on seeded random shapes in each of its regimes, taken from the device's
own SM count S:

  few    at most S/2 units: every unit split over keys, so one wave covers (nearly) all SMs;
  tail   S to 2S units plus a partial last wave of at most S/2: that wave's units split 2-4 ways;
  whole  more than S/2 and at most S units: one launch, nothing split.

For each, fa_fwd_plan reports the regime's plan, and O and the log-sum-exp from fa_fwd_lse (the
same division into launches) match the fp64 oracle on every element. The LSE bound is the one
of the LSE tests: the kernel's denominator sums the 16-bit-rounded weights, each within 2^-9
relative of its exact value (bf16), so |LSE - LSE_ref| stays within 2^-9 plus fp32 rounding."""
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


def draw_shape(regime: str, S: int, rng) -> tuple[int, int, int, int]:
    """(B * H, Nq, Nk, units) for the regime on S SMs."""
    if regime == "few":
        per = int(rng.integers(1, 3))  # units per slice
        units = int(rng.integers(1, S // 2 + 1))
        bh = max(1, units // per)
        Nq = int(rng.integers(256 * (per - 1) + 1, 256 * per + 1))
        Nk = int(rng.integers(4 * 128, 24 * 128 + 1))  # at least 4 key tiles: 2 ranges of 2
    elif regime == "tail":
        bh = S * int(rng.integers(1, 3)) + int(rng.integers(1, S // 2 + 1))
        Nq = int(rng.integers(1, 257))  # one unit per slice
        Nk = int(rng.integers(8 * 128 + 1, 12 * 128 + 1))  # enough tiles for 4 ranges of 2
    else:
        bh = int(rng.integers(S // 2 + 1, S + 1))
        Nq = int(rng.integers(1, 257))
        Nk = int(rng.integers(1, 1025))
    units = bh * ((Nq + 255) // 256)
    return bh, Nq, Nk, units


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("regime", ["few", "tail", "whole"])
def test_balanced_launches_match_oracle(fa, regime, seed):
    S = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(5000 + 10 * seed + ["few", "tail", "whole"].index(regime))
    bh, Nq, Nk, units = draw_shape(regime, S, rng)
    B = 2 if bh % 2 == 0 else 1
    H = bh // B
    D = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["f16", "bf16"]))
    w = inputs.Workload(f"balance_{regime}_{seed}", B, H, Nq, Nk, D, dtype, False,
                        seed=500 + 10 * seed + len(regime))

    plan = fa.plan(B, H, Nq, Nk, D, causal=False)
    assert plan["units"] == units
    if regime == "few":
        assert plan["launches"] == 2 and plan["split_begin"] == 0 and plan["split_units"] == units
        assert plan["num_splits"] >= 2 and plan["ctas"] <= S
    elif regime == "tail":
        tail = units % S
        assert plan["launches"] == 2 and plan["split_units"] == tail
        assert plan["split_begin"] == units - tail and 2 <= plan["num_splits"] <= 4
        assert plan["ctas"] == units - tail + tail * plan["num_splits"]
    else:
        assert plan["launches"] == 1 and plan["ctas"] == units

    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o, lse = fa.forward_lse(q, k, v, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error() == (0, 0)
    ref_o, ref_lse = oracle.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"),
                                      w.scale, False, with_lse=True)
    got_lse = lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got_lse))
    assert np.max(np.abs(got_lse - ref_lse)) <= LSE_TOL
    parity.describe(w)
    parity.assert_parity(parity.compare(inputs.from_torch(o), ref_o, w.dtype), False, w.name,
                         mean="auto")
