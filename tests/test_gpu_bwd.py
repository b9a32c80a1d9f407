"""Backward pass on the GPU against the fp64 oracle's exact gradients.

The GPU runs its own forward (O, LSE) and then fa_bwd, as a training step would; the oracle
differentiates the definition exactly on the same Q, K, V, dO.

Tolerance, from the arithmetic, per 16-bit type with unit roundoff u = 2^-p (p significand bits:
u = 2^-8 for bf16, 2^-11 for fp16). Four roundings to the type enter each gradient, each of
relative size at most u/2: P and dS as MMA operands, the forward's O (from which D_i = dO_i . O_i
is formed), and the gradient's own output rounding; fp32 accumulation adds far less. The errors
of the many terms of each sum are independent, so normwise they add in quadrature, to about u;
each gradient must satisfy ||g - g_ref|| <= 2u ||g_ref||. Elementwise, where dS cancels
(dP - D small) a relative bound means nothing, so each element is held to 4u of the gradient's
largest magnitude. Measured: about 0.6u normwise and at most 1.5u elementwise, for both types."""
import json
import os

import numpy as np
import pytest

import oracle
from tiled_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
UNIT_ROUNDOFF = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


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


def check_grads(w, grads, ref, what):
    """Normwise and elementwise checks of (dQ, dK, dV) against the oracle; with FA_PARITY_REPORT
    set, one JSON line per gradient with the errors found."""
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        assert np.all(np.isfinite(g)), f"{what} {name}"
        e_norm = rel(g, r)
        e_max = np.max(np.abs(g - r)) / max(np.max(np.abs(r)), 1e-30)
        path = os.environ.get("FA_PARITY_REPORT")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps(dict(what=f"bwd {what} {name}", shape=f"B={w.B} H={w.H} "
                                        f"Nq={w.Nq} Nk={w.Nk} D={w.D} {w.dtype}"
                                        f"{' causal' if w.causal else ''}", elements=int(g.size),
                                        rel_norm_err=float(e_norm), rel_max_err=float(e_max))) + "\n")
        u = UNIT_ROUNDOFF[w.dtype]
        assert e_norm <= 2 * u, f"{what} {name}: relative error {e_norm:.3g} > 2u = {2 * u:.3g}"
        assert e_max <= 4 * u, f"{what} {name}: max error {e_max:.3g} of max |g| > 4u = {4 * u:.3g}"


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
    check_grads(w, [f(inputs.from_torch(g)) for g in (dq, dk, dv)], ref, w.name)


@pytest.mark.parametrize("name", ["headline", "causal_prefill"])
def test_backward_full_size(fa, name):
    """The backward at the shapes it is benchmarked on (the headline, 32 heads x 4096 tokens, and
    causal prefill, 32 heads x 2048 tokens, D = 128, bf16), run whole on the GPU in the bench's
    launch configuration; four whole (batch, head) slices (every gradient element of them)
    compared with the oracle's exact gradients. Slices are independent, so the other slices'
    work does not enter these."""
    w = inputs.WORKLOADS[name]
    bits = inputs.draw(w)
    dout_bits = inputs.draw(w.with_(seed=w.seed + 1000))["q"]
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    do = inputs.to_torch(dout_bits, w.dtype).cuda()
    o, lse = fa.forward_lse(q, k, v, causal=w.causal, scale=w.scale)
    grads = fa.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    heads = [0, 11, 22, w.H - 1]
    f = lambda x: inputs.bits_to_f64(x, w.dtype)
    ref = oracle.attention_backward(*(f(bits[n][0, heads]) for n in "qkv"), f(dout_bits[0, heads]),
                                    w.scale, w.causal)
    got = [f(inputs.from_torch(g)[0, heads]) for g in grads]
    check_grads(w, got, ref, f"{name} heads {heads}")


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


@pytest.mark.parametrize("seed", range(3))
def test_backward_random_shapes(fa, seed):
    """Seeded random problems (B, H in 1..3, Nq and Nk in 1..400, either D and 16-bit type, causal
    or not, scale of either sign): the GPU's forward and backward against the oracle's exact
    gradients, to the same per-dtype bound."""
    rng = np.random.default_rng(2000 + seed)
    for case in range(4):
        D = int(rng.choice([64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        causal = bool(rng.integers(2))
        B, H = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        Nq, Nk = int(rng.integers(1, 401)), int(rng.integers(1, 401))
        scale = float(np.float32(rng.choice([-1.0, 1.0]) * rng.uniform(0.3, 1.5) / np.sqrt(D)))
        w = inputs.Workload(f"bwd_random_{seed}_{case}", B, H, Nq, Nk, D, dtype, causal,
                            seed=500 + seed * 10 + case, scale=scale)
        bits = inputs.draw(w)
        dout_bits = inputs.draw(w.with_(seed=w.seed + 1000))["q"]
        q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
        do = inputs.to_torch(dout_bits, w.dtype).cuda()
        o, lse = fa.forward_lse(q, k, v, causal=w.causal, scale=w.scale)
        grads = fa.backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        assert fa.last_device_error()[0] == 0
        f = lambda x: inputs.bits_to_f64(x, w.dtype)
        ref = oracle.attention_backward(f(bits["q"]), f(bits["k"]), f(bits["v"]), f(dout_bits),
                                        w.scale, w.causal)
        check_grads(w, [f(inputs.from_torch(g)) for g in grads], ref, w.name)
