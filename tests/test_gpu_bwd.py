"""Backward pass on the GPU against the fp64 oracle's exact gradients.

The GPU runs its own forward (O, LSE) and then fa_bwd, as a training step would; the oracle
differentiates the definition exactly on the same Q, K, V, dO. Tolerance, from the arithmetic:
P and dS enter the MMAs rounded to 16 bits (relative 2^-9 for bf16, 2^-11 for fp16) and O, the
outputs and the forward's O/LSE are 16-bit too, so elementwise relative accuracy is not
meaningful where dS cancels (dP - D); each gradient is checked normwise,
||g - g_ref|| <= 2e-2 ||g_ref||, and elementwise against 5e-2 of its largest magnitude."""
import numpy as np
import pytest

import oracle
from tiled_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
NORM_TOL, MAX_TOL = 2e-2, 5e-2


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_gb300 import fa as fa_mod

    fa_mod.lib()
    return fa_mod


CASES = [
    inputs.Workload("bwd_small_f16", 1, 2, 128, 128, 64, "f16", False, seed=81),
    inputs.Workload("bwd_ragged_bf16", 1, 3, 300, 257, 128, "bf16", False, seed=82),
    inputs.Workload("bwd_causal_bf16", 2, 2, 384, 384, 128, "bf16", True, seed=83),
    inputs.Workload("bwd_causal_ragged_f16", 1, 2, 200, 333, 64, "f16", True, seed=84),
    inputs.Workload("bwd_long_bf16", 1, 2, 1024, 1024, 128, "bf16", True, seed=85),
    # A negative scale: hidden scores then hold +inf, so that 2^(s*c - L) is still 0.
    inputs.Workload("bwd_neg_scale_causal_f16", 1, 2, 300, 300, 64, "f16", True, scale=-0.125,
                    seed=88),
    inputs.Workload("bwd_neg_scale_ragged_bf16", 1, 2, 200, 333, 128, "bf16", False,
                    scale=-0.0883883, seed=89),
]


def rel(g, ref):
    return np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_oracle(fa, w):
    bits = inputs.draw(w)
    dout_bits = inputs.draw(w.with_(seed=w.seed + 1000))["q"]
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    do = inputs.to_torch(dout_bits, w.dtype).cuda()
    o, lse = fa.forward_lse(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    f = lambda x: inputs.bits_to_f64(x, w.dtype)
    ref = oracle.attention_backward(f(bits["q"]), f(bits["k"]), f(bits["v"]), f(dout_bits),
                                    w.scale, w.causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = f(inputs.from_torch(got))
        assert np.all(np.isfinite(g)), name
        assert rel(g, r) <= NORM_TOL, f"{name}: relative error {rel(g, r):.3g}"
        assert np.max(np.abs(g - r)) <= MAX_TOL * np.max(np.abs(r)), name


def test_backward_is_deterministic(fa):
    w = CASES[2]
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    do = inputs.to_torch(inputs.draw(w.with_(seed=9))["q"], w.dtype).cuda()
    o, lse = fa.forward_lse(q, k, v, causal=True, scale=w.scale)
    a = fa.backward(q, k, v, o, lse, do, causal=True, scale=w.scale)
    b = fa.backward(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_backward_keys_past_all_queries_get_zero(fa):
    """Causal, Nk > Nq: keys after the last query are seen by no query, so dK = dV = 0 there."""
    w = inputs.Workload("bwd_wide", 1, 1, 130, 400, 64, "bf16", True, seed=86)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    do = inputs.to_torch(inputs.draw(w.with_(seed=10))["q"], w.dtype).cuda()
    o, lse = fa.forward_lse(q, k, v, causal=True, scale=w.scale)
    _, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert bool((dk[:, :, 130:] == 0).all()) and bool((dv[:, :, 130:] == 0).all())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_results_are_ordered_in_the_stream(fa, causal):
    """The backward's kernels overlap one another (programmatic dependent launches), yet work
    queued after fa_bwd on the same stream sees every gradient complete: copies taken there, with
    no synchronisation in between, equal the gradients read after the device is idle."""
    w = inputs.Workload("bwd_order", 1, 16, 2048, 2048, 128, "bf16", causal, seed=86)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    do = inputs.to_torch(inputs.draw(w.with_(seed=w.seed + 1000))["q"], w.dtype).cuda()
    o, lse = fa.forward_lse(q, k, v, causal=causal, scale=w.scale)
    for _ in range(3):
        grads = fa.backward(q, k, v, o, lse, do, causal=causal, scale=w.scale)
        copies = [g.clone() for g in grads]
        torch.cuda.synchronize()
        assert fa.last_device_error()[0] == 0
        for name, g, c in zip(("dq", "dk", "dv"), grads, copies):
            assert torch.equal(g.view(torch.int16), c.view(torch.int16)), name
