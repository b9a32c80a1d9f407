"""Split over keys (flash-decoding): partial states per key range, merged by the state-merge
rule, against the fp64 oracle and against the unsplit path."""
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
    (inputs.Workload("decode_1row", 1, 8, 1, 4096, 128, "bf16", False, seed=51), 16),
    (inputs.Workload("decode_7rows_f16", 2, 4, 7, 3000, 64, "f16", False, seed=52), 5),
    (inputs.Workload("chunk_ragged", 1, 2, 300, 1000, 128, "bf16", False, seed=53), 3),
    (inputs.Workload("chunk_auto", 1, 4, 130, 777, 64, "bf16", False, seed=54), 0),
    (inputs.Workload("more_splits_than_tiles", 1, 1, 64, 200, 128, "bf16", False, seed=55), 9),
]


@pytest.mark.parametrize("w,splits", CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_splitkv_matches_oracle(fa, w, splits):
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
    o = fa.forward_splitkv(q, k, v, num_splits=splits, scale=w.scale, lse=lse)
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    ref_o, ref_lse = oracle.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"),
                                      w.scale, False, with_lse=True)
    stats = parity.compare(inputs.from_torch(o), ref_o, w.dtype)
    parity.assert_parity(stats, False, w.name)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_TOL
    # Close to the unsplit path (different summation order, same arithmetic).
    o1 = inputs.bits_to_f64(inputs.from_torch(fa.forward(q, k, v, scale=w.scale)), w.dtype)
    assert np.max(np.abs(inputs.bits_to_f64(inputs.from_torch(o), w.dtype) - o1)) <= 2e-2


def test_long_context_chunk_full_size(fa):
    w = inputs.WORKLOADS["long_context_chunk"]
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o = inputs.from_torch(fa.forward_splitkv(q, k, v, num_splits=0, scale=w.scale))
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    for h in (0, 7):
        ref = oracle.attention_rows(inputs.bits_to_f64(bits["q"][0, h], w.dtype), np.arange(w.Nq),
                                    inputs.bits_to_f64(bits["k"][0, h], w.dtype),
                                    inputs.bits_to_f64(bits["v"][0, h], w.dtype), w.scale, False)
        parity.assert_parity(parity.compare(o[0, h], ref, w.dtype), True, f"head {h}")


def test_one_split_is_fa_fwd(fa):
    """One key range is fa_fwd's single launch (work balancing off), bit for bit."""
    w = inputs.Workload("one_split", 1, 2, 200, 500, 128, "bf16", False, seed=56)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    a = fa.forward_splitkv(q, k, v, num_splits=1, scale=w.scale)
    try:
        fa.set_tail_split(False)
        b = fa.forward(q, k, v, scale=w.scale)
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_workspace_checks(fa):
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 1024, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    need = fa.splitkv_workspace_bytes(1, 1, 16, 1024, 64, 4)
    assert need > 0 and fa.splitkv_workspace_bytes(1, 1, 16, 1024, 64, 1) == 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    call = lambda ptr, size: fa.lib().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), k.data_ptr(),
                                                     o.data_ptr(), None, 1, 1, 16, 1024, 64, 0.1,
                                                     4, 1, ptr, size, None)
    assert call(ws.data_ptr(), need - 1) == 1      # too small
    assert call(None, need) == 1                    # missing
    assert call(ws.data_ptr() + 16, need - 16) in (1, 3)  # misaligned or too small
    assert call(ws.data_ptr(), need) == 0
    torch.cuda.synchronize()


def test_last_wave_split_matches_oracle_and_unsplit(fa):
    """40 heads x 8 units = 320 units: the last 16 (two heads) run split over keys."""
    w = inputs.Workload("tail", 1, 40, 2048, 1024, 64, "bf16", False, seed=57)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
    o, _ = fa.forward_lse(q, k, v, scale=w.scale, lse=lse)
    try:
        fa.set_tail_split(False)
        o_plain = fa.forward(q, k, v, scale=w.scale)
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    assert fa.last_device_error()[0] == 0
    got = inputs.from_torch(o)
    for h in (37, 38, 39):  # 37 runs whole, 38 and 39 split
        ref, ref_lse = oracle.attention(*(inputs.bits_to_f64(bits[n][0, h], w.dtype) for n in "qkv"),
                                        w.scale, False, with_lse=True)
        parity.assert_parity(parity.compare(got[0, h], ref, w.dtype), True, f"head {h}")
        assert np.max(np.abs(lse[0, h].cpu().numpy() - ref_lse)) <= LSE_TOL
    diff = np.abs(inputs.bits_to_f64(got, "bf16") - inputs.bits_to_f64(inputs.from_torch(o_plain), "bf16"))
    assert diff[0, :38].max() == 0.0  # whole units: identical bits
    assert diff.max() <= 2e-2


@pytest.mark.parametrize("w,splits", [
    # 4 units, 24 key tiles: each unit split into min(152 // 4, 24 // 2) = 12 ranges.
    (inputs.Workload("few_units", 1, 2, 300, 3000, 128, "bf16", False, seed=60), 12),
    # 2 units, 3 key tiles: ranges would be shorter than 2 tiles, so one launch.
    (inputs.Workload("few_keys", 1, 2, 200, 380, 64, "f16", False, seed=61), 1),
], ids=lambda x: getattr(x, "name", str(x)))
def test_few_units_split_over_keys(fa, w, splits):
    """When the units cannot fill half the SMs, the default entry splits every unit over keys
    (one attention launch and one merge launch) unless the key ranges would be too short. Either
    way the result matches the oracle, and the unsplit launch up to rounding."""
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
    fa.forward_lse(q, k, v, scale=w.scale, lse=lse)
    torch.cuda.synchronize()
    fa.timer_start()
    o, _ = fa.forward_lse(q, k, v, scale=w.scale, lse=lse)
    kernels = fa.timer_stop()
    assert kernels["fwd"][1] == 1
    assert kernels.get("merge", (0.0, 0))[1] == (1 if splits > 1 else 0)
    try:
        fa.set_tail_split(False)
        o_plain = fa.forward(q, k, v, scale=w.scale)
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == (0, 0)
    got = inputs.from_torch(o)
    for h in range(w.H):
        ref, ref_lse = oracle.attention(*(inputs.bits_to_f64(bits[n][0, h], w.dtype) for n in "qkv"),
                                        w.scale, False, with_lse=True)
        parity.assert_parity(parity.compare(got[0, h], ref, w.dtype), True, f"head {h}")
        assert np.max(np.abs(lse[0, h].cpu().numpy() - ref_lse)) <= LSE_TOL
    diff = np.abs(inputs.bits_to_f64(got, w.dtype) - inputs.bits_to_f64(inputs.from_torch(o_plain), w.dtype))
    if splits == 1:
        assert diff.max() == 0.0
    else:
        assert diff.max() <= 2e-2


def test_last_wave_split_workspace_is_reused_across_calls(fa):
    """The split last wave's partial states live in a workspace shared by every call: calls of
    two shapes interleaved (ragged rows, both head dims, both dtypes) give the same bits every
    time and match the unsplit launch and the oracle."""
    shapes = [inputs.Workload("tail_a", 1, 40, 2048, 1024, 64, "bf16", False, seed=58),
              inputs.Workload("tail_b", 1, 10, 4000, 2000, 128, "f16", False, seed=59)]
    data = []
    for w in shapes:
        bits = inputs.draw(w)
        q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
        try:
            fa.set_tail_split(False)
            plain = inputs.from_torch(fa.forward(q, k, v, scale=w.scale))
        finally:
            fa.set_tail_split(True)
        data.append((w, bits, (q, k, v), plain))
    first = {}
    for rep in range(3):
        for w, bits, (q, k, v), plain in data:
            got = inputs.from_torch(fa.forward(q, k, v, scale=w.scale))
            assert fa.last_device_error() == (0, 0)
            if w.name in first:
                assert np.array_equal(got, first[w.name]), f"{w.name} changed on call {rep}"
                continue
            first[w.name] = got
            diff = np.abs(inputs.bits_to_f64(got, w.dtype) - inputs.bits_to_f64(plain, w.dtype))
            assert diff.max() <= 2e-2
            h = w.H - 1  # the last head's units are in the split wave
            ref = oracle.attention(*(inputs.bits_to_f64(bits[n][0, h], w.dtype) for n in "qkv"),
                                   w.scale, False)
            parity.assert_parity(parity.compare(got[0, h], ref, w.dtype), True, f"{w.name} head {h}")


@pytest.mark.parametrize("shape", [
    (1, 32, 4096, 4096, 128, False),   # last wave split
    (1, 8, 128, 65536, 128, False),    # few units, every unit split
    (2, 4, 1000, 1000, 64, False),     # ragged, split in 4
    (1, 32, 2048, 2048, 128, True),    # causal: one launch
    (1, 2, 200, 380, 64, False),       # too few key tiles to split
    (64, 32, 128, 1024, 64, False),    # 2048 units, last wave of 72 split
], ids=str)
def test_plan_matches_the_launches(fa, shape):
    """fa_fwd_plan on the current device (its SM count read from the device) describes the
    launches fa_fwd then makes: one attention launch, plus a merge launch when it splits."""
    B, H, Nq, Nk, D, causal = shape
    props = torch.cuda.get_device_properties(0)
    plan = fa.plan(B, H, Nq, Nk, D, causal)
    assert plan == fa.plan(B, H, Nq, Nk, D, causal, num_sms=props.multi_processor_count)
    q = torch.zeros(B, H, Nq, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, H, Nk, D, dtype=torch.bfloat16, device="cuda")
    fa.forward(q, k, k, causal=causal)
    torch.cuda.synchronize()
    fa.timer_start()
    fa.forward(q, k, k, causal=causal)
    kernels = fa.timer_stop()
    assert kernels["fwd"][1] == 1
    assert kernels.get("merge", (0.0, 0))[1] == plan["launches"] - 1
    assert fa.last_device_error() == (0, 0)
