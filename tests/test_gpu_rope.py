"""Rotary position embedding on the GPU against the fp64 oracle, alone and in front of attention.

fa_rope computes in fp32 and rounds once to the 16-bit type, so each output is within one unit
in the last place of the exactly rotated value (half an ulp of rounding plus fp32 error, which
can tip a near-tie)."""
import numpy as np
import pytest

import oracle
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


def tables(n, d, offset=0, base=10000.0):
    pos = np.arange(offset, offset + n, dtype=np.float64)[:, None]
    ang = pos * base ** (-np.arange(d // 2, dtype=np.float64) / (d // 2))
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
def test_rope_matches_oracle(fa, form, dtype, D):
    w = inputs.Workload("rope", 2, 3, 257, 257, D, dtype, False, seed=61 + D + form)
    x = inputs.draw(w)["q"]
    c, s = tables(w.Nq, D, offset=5)
    xt = inputs.to_torch(x, dtype).cuda()
    ct, st = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    y = fa.rope(xt, ct, st, form=form)
    inplace = xt.clone()
    fa.rope(inplace, ct, st, form=form, out=inplace)
    torch.cuda.synchronize()
    ref = oracle.rope(inputs.bits_to_f64(x, dtype), c.astype(np.float64), s.astype(np.float64),
                      form)
    got = inputs.bits_to_f64(inputs.from_torch(y), dtype)
    assert np.all(np.abs(got - ref) <= parity.ulp(ref, dtype) + 1e-30)
    assert torch.equal(y.view(torch.int16), inplace.view(torch.int16))


@pytest.mark.parametrize("form", [0, 1])
def test_attention_on_rotated_inputs(fa, form):
    w = inputs.Workload("rope_attn", 1, 4, 300, 300, 128, "bf16", True, seed=71 + form)
    bits = inputs.draw(w)
    c, s = tables(w.Nq, w.D)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    ct, st = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
    q_before = q.clone()
    o = fa.forward_rope(q, k, v, ct, st, ct, st, form=form, causal=True, scale=w.scale, lse=lse)
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    assert torch.equal(q.view(torch.int16), q_before.view(torch.int16))  # inputs untouched
    c64, s64 = c.astype(np.float64), s.astype(np.float64)
    rot = {n: inputs.bits_to_f64(inputs.round_to_bits(
        oracle.rope(inputs.bits_to_f64(bits[n], "bf16"), c64, s64, form).astype(np.float32), "bf16"),
        "bf16") for n in "qk"}
    ref, ref_lse = oracle.attention(rot["q"], rot["k"], inputs.bits_to_f64(bits["v"], "bf16"),
                                    w.scale, True, with_lse=True)
    parity.assert_parity(parity.compare(inputs.from_torch(o), ref, "bf16"), False, "rope attention")
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= 4e-3


@pytest.mark.parametrize("w,form", [
    (inputs.Workload("rope_fused_causal", 1, 4, 300, 300, 128, "bf16", True, seed=81), 0),
    (inputs.Workload("rope_fused_split", 1, 2, 200, 3000, 128, "bf16", False, seed=82), 1),
    (inputs.Workload("rope_fused_d64_f16", 2, 3, 257, 1000, 64, "f16", False, seed=83), 0),
    (inputs.Workload("rope_fused_d64_pairs", 1, 5, 513, 513, 64, "bf16", True, seed=84), 1),
], ids=lambda x: getattr(x, "name", str(x)))
def test_fused_q_rotation_equals_the_two_pass_form(fa, w, form):
    """fa_fwd_rope rotates Q inside the attention kernel (in shared memory, after each tile's
    load) and K in a pass of its own. The result equals rotating both with fa_rope and then
    running the attention, bit for bit (same fp32 rotation, same launches), for both pair forms,
    both head dims and dtypes, causal or split over keys, with ragged query tiles; and it matches
    the oracle on the rotated inputs."""
    bits = inputs.draw(w)
    c, s = tables(max(w.Nq, w.Nk), w.D, offset=3)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    cq, sq = torch.from_numpy(c[:w.Nq]).cuda(), torch.from_numpy(s[:w.Nq]).cuda()
    ck, sk = torch.from_numpy(c[:w.Nk]).cuda(), torch.from_numpy(s[:w.Nk]).cuda()
    lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
    fused = fa.forward_rope(q, k, v, cq, sq, ck, sk, form=form, causal=w.causal, scale=w.scale,
                            lse=lse)
    qr, kr = fa.rope(q, cq, sq, form=form), fa.rope(k, ck, sk, form=form)
    lse2 = torch.empty_like(lse)
    two_pass, _ = fa.forward_lse(qr, kr, v, causal=w.causal, scale=w.scale, lse=lse2)
    torch.cuda.synchronize()
    assert fa.last_device_error() == (0, 0)
    assert torch.equal(fused.view(torch.int16), two_pass.view(torch.int16))
    assert torch.equal(lse, lse2)
    rot = {n: inputs.bits_to_f64(inputs.round_to_bits(
        oracle.rope(inputs.bits_to_f64(bits[n], w.dtype), c[:getattr(w, "N" + n)].astype(np.float64),
                    s[:getattr(w, "N" + n)].astype(np.float64), form).astype(np.float32), w.dtype),
        w.dtype) for n in "qk"}
    ref = oracle.attention(rot["q"], rot["k"], inputs.bits_to_f64(bits["v"], w.dtype), w.scale,
                           w.causal)
    parity.describe(w)
    parity.assert_parity(parity.compare(inputs.from_torch(fused), ref, w.dtype), False, w.name)


@pytest.mark.parametrize("seed", range(2))
def test_fused_rotation_random_shapes(fa, seed):
    """Seeded random problems through fa_fwd_rope (Q rotated in the attention kernel, K by its
    pass): equal bit for bit to the three-pass form, both pair forms, ragged shapes."""
    rng = np.random.default_rng(3000 + seed)
    for case in range(4):
        D = int(rng.choice([64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        causal = bool(rng.integers(2))
        form = int(rng.integers(2))
        B, H = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        Nq, Nk = int(rng.integers(1, 701)), int(rng.integers(1, 701))
        w = inputs.Workload(f"rope_random_{seed}_{case}", B, H, Nq, Nk, D, dtype, causal,
                            seed=700 + seed * 10 + case)
        bits = inputs.draw(w)
        c, s = tables(max(Nq, Nk), D, offset=int(rng.integers(0, 1000)))
        q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
        cq, sq = torch.from_numpy(c[:Nq]).cuda(), torch.from_numpy(s[:Nq]).cuda()
        ck, sk = torch.from_numpy(c[:Nk]).cuda(), torch.from_numpy(s[:Nk]).cuda()
        fused = fa.forward_rope(q, k, v, cq, sq, ck, sk, form=form, causal=causal, scale=w.scale)
        two_pass = fa.forward(fa.rope(q, cq, sq, form=form), fa.rope(k, ck, sk, form=form), v,
                              causal=causal, scale=w.scale)
        torch.cuda.synchronize()
        assert fa.last_device_error() == (0, 0)
        assert torch.equal(fused.view(torch.int16), two_pass.view(torch.int16)), w.name
