"""The fp64 oracle against its pins (values the pages print, closed forms, invariants,
library special cases and brute force). CPU only."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_empty_and_bad_arguments(orc):
    import numpy as np

    with pytest.raises(RuntimeError):
        orc.online_state(np.zeros(2), np.zeros((3, 2)), np.zeros((3, 2)), 0, 3, 1.0, block=0)
    with pytest.raises(RuntimeError):
        orc.attention_online(np.zeros((1, 2)), np.zeros((3, 2)), np.zeros((3, 2)), 1.0, block=0)


def test_two_oracles_agree_on_every_workload(orc):
    """The two-pass definition and the online recurrence (one key at a time and 37 keys at a
    time) agree to 1e-12 on the actual seeded inputs of every named workload: the small ones
    whole, the large ones on slice (0, 0) (the first 512 query rows against every key when
    non-causal; the first 4096 rows, so keys 0..4095, for long causal)."""
    import math

    import numpy as np

    from tiled_online_softmax_gb300 import inputs

    for w in inputs.WORKLOADS.values():
        if w.name == "long_context_chunk":
            continue  # the same distribution as the headline, 8 heads of 128 rows
        small = w.B * w.H * w.Nq * w.Nk * w.D <= 2 ** 31
        bits = inputs.draw(w.with_(B=1, H=1)) if not small else inputs.draw(w)
        q, k, v = (inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv")
        if not small:
            rows = 4096 if w.causal else 512
            q = q[..., :rows, :]
            if w.causal:
                k, v = k[..., :rows, :], v[..., :rows, :]
        o2, l2 = orc.attention(q, k, v, w.scale, w.causal, with_lse=True)
        for block in (1, 37):
            o1, l1 = orc.attention_online(q, k, v, w.scale, w.causal, block=block, with_lse=True)
            scale = max(1.0, float(np.max(np.abs(o2))))
            assert np.max(np.abs(o1 - o2)) <= 1e-12 * scale, (w.name, block)
            assert np.max(np.abs(l1 - l2)) <= 1e-12 * max(1.0, float(np.max(np.abs(l2)))), (w.name, block)
        assert math.isfinite(float(o2.sum()))
