"""Parity of the CUDA path (called through the C interface) with the fp64 oracle.

Every workload, the largest included, runs at full size in the launch configuration the bench
times and is compared with the oracle element by element on every output. The large workloads
are compared a few (batch, head) slices at a time, so that the oracle's fp64 copies stay small.
"""
import math
import time

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


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def run_gpu(fa, bits, w: inputs.Workload, out=None):
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o = fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=out)
    torch.cuda.synchronize()
    st, site = fa.last_device_error()
    assert st == 0, f"device error word set (site {site})"
    return o


def full_check(fa, orc, w: inputs.Workload, literal=True, mean=None, slices_per_chunk=8):
    """Run w at full size once; compare every output element with the oracle, `slices_per_chunk`
    (batch, head) slices at a time; return the statistics over all of them."""
    parity.describe(w)
    bits = inputs.draw(w)
    o = inputs.from_torch(run_gpu(fa, bits, w)).reshape(w.B * w.H, w.Nq, w.D)
    q, k, v = (bits[n].reshape(w.B * w.H, -1, w.D) for n in "qkv")
    parts = []
    oracle_s = 0.0
    for c0 in range(0, w.B * w.H, slices_per_chunk):
        c1 = min(c0 + slices_per_chunk, w.B * w.H)
        args = [inputs.bits_to_f64(x[c0:c1], w.dtype) for x in (q, k, v)]
        t0 = time.perf_counter()
        ref = orc.attention(*args, w.scale, w.causal)
        oracle_s += time.perf_counter() - t0
        parts.append(parity.compare(o[c0:c1], ref, w.dtype))
    stats = parity.merge(parts)
    parity.assert_parity(stats, literal, w.name, mean,
                         extra=dict(oracle_seconds=oracle_s, oracle_threads=orc.num_threads(),
                                    gflop=w.flops / 1e9))
    return stats


# --- the workloads ---------------------------------------------------------------------------
# The five named workloads, the headline shape and its D = 64 variant, all at full size and
# every element: the literal bar (max 1e-2, mean 1e-3) on every N(0, 1) workload; on the
# large-magnitude one the max beyond output rounding (1e-2 + ulp/2) and the literal mean.

def test_single_head(fa, orc):
    full_check(fa, orc, inputs.WORKLOADS["single_head"])


def test_ragged(fa, orc):
    full_check(fa, orc, inputs.WORKLOADS["ragged"])


def test_causal_prefill(fa, orc):
    full_check(fa, orc, inputs.WORKLOADS["causal_prefill"])


def test_rescale_stress_full_size(fa, orc):
    full_check(fa, orc, inputs.WORKLOADS["rescale_stress"], literal=False, mean="literal")


def test_long_causal_full_size(fa, orc):
    full_check(fa, orc, inputs.WORKLOADS["long_causal"], slices_per_chunk=2)


def test_headline_full_size(fa, orc):
    full_check(fa, orc, inputs.WORKLOADS["headline"])


def test_headline_d64_full_size(fa, orc):
    """The headline shape at D = 64 in fp16 (4-stage K/V ring, split last wave)."""
    full_check(fa, orc, inputs.WORKLOADS["headline_d64"])


# --- edge cases ------------------------------------------------------------------------------

EDGE_SIZES = [1, 2, 63, 64, 65, 127, 128, 129, 255, 257]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_shapes(fa, orc, D, dtype, causal):
    """Ragged query and key counts around the 128-row tile, including Nq != Nk under causal."""
    seed = 100 + D + (dtype == "bf16") * 7 + causal * 13
    for i, nq in enumerate(EDGE_SIZES):
        nk = EDGE_SIZES[(i * 3 + 1) % len(EDGE_SIZES)]
        for nq_, nk_ in ((nq, nq), (nq, nk)):
            w = inputs.Workload(f"edge_{nq_}x{nk_}", 1, 2, nq_, nk_, D, dtype, causal,
                                seed=seed + nq_ * 1000 + nk_)
            full_check(fa, orc, w, literal=False, mean="auto")


def test_late_maximum(fa, orc):
    """Scores that grow along the row (the running max moves at every key tile): a kernel that
    forgets to rescale O fails here."""
    D, n = 64, 1024
    q = np.zeros((1, 1, n, D), np.float32)
    k = np.zeros((1, 1, n, D), np.float32)
    q[..., 0] = 1.0
    k[0, 0, :, 0] = np.linspace(0, 24, n)  # score rises with the key index
    v = np.random.default_rng(7).standard_normal((1, 1, n, D)).astype(np.float32)
    w = inputs.Workload("late_max", 1, 1, n, n, D, "f16", False, seed=0, scale=1.0)
    bits = {"q": inputs.round_to_bits(q, "f16"), "k": inputs.round_to_bits(k, "f16"),
            "v": inputs.round_to_bits(v, "f16")}
    o = run_gpu(fa, bits, w)
    ref = orc.attention(*(inputs.bits_to_f64(bits[x], "f16") for x in "qkv"), 1.0)
    parity.describe(w)
    parity.assert_parity(parity.compare(inputs.from_torch(o), ref, "f16"), True, "late max")


@pytest.mark.parametrize("w", [
    inputs.Workload("neg_scale", 1, 3, 300, 333, 128, "bf16", False, scale=-0.0883883, seed=19),
    inputs.Workload("neg_scale_causal", 2, 2, 257, 257, 64, "f16", True, scale=-0.125, seed=20),
    inputs.Workload("neg_scale_split", 1, 2, 200, 2000, 64, "bf16", False, scale=-0.5, seed=21),
], ids=lambda w: w.name)
def test_negative_scale(fa, orc, w):
    """A negative scale (the largest weights go to the most negative scores) matches the oracle,
    through the single launch, the causal mask and the key split with its merge."""
    full_check(fa, orc, w, literal=False, mean="auto")


def test_all_equal_scores_give_mean(fa):
    """Q = 0: every visible key weighs the same, O is the (prefix) mean of V."""
    for causal in (False, True):
        w = inputs.Workload("zero_q", 1, 2, 200, 300, 128, "bf16", causal, seed=9)
        bits = inputs.draw(w)
        bits["q"][:] = 0
        o = inputs.bits_to_f64(inputs.from_torch(run_gpu(fa, bits, w)), "bf16")
        v = inputs.bits_to_f64(bits["v"], "bf16")
        if causal:
            want = np.cumsum(v, axis=2)[:, :, :200] / np.arange(1, 201)[None, None, :, None]
        else:
            want = np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape)
        assert np.max(np.abs(o - want)) < 1e-2


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_gives_mean(fa, orc, causal):
    """scale = 0 (the softmax temperature's special case): every visible key weighs 1 whatever Q
    is, so O is the (prefix) mean of V. The kernel maps a zero scale to a tiny positive one so
    that hidden keys keep weight 0; checked against the oracle and the closed form, with the key
    split (non-causal) and across a ragged tail."""
    w = inputs.Workload("zero_scale", 1, 3, 333, 1000 if not causal else 333, 64, "f16", causal,
                        seed=22, scale=0.0)
    bits = inputs.draw(w)
    o = inputs.from_torch(run_gpu(fa, bits, w))
    ref = orc.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), 0.0, causal)
    parity.describe(w)
    parity.assert_parity(parity.compare(o, ref, w.dtype), True, "scale 0")
    v = inputs.bits_to_f64(bits["v"], w.dtype)
    if causal:
        want = np.cumsum(v, axis=2) / np.arange(1, w.Nk + 1)[None, None, :, None]
    else:
        want = np.broadcast_to(v.mean(axis=2, keepdims=True), ref.shape)
    assert np.max(np.abs(ref - want)) < 1e-12


def test_single_key_gives_v(fa):
    w = inputs.Workload("one_key", 2, 3, 130, 1, 64, "f16", False, seed=10)
    bits = inputs.draw(w)
    o = inputs.from_torch(run_gpu(fa, bits, w))
    assert np.array_equal(o, np.broadcast_to(bits["v"], o.shape))


def test_deterministic_and_no_stray_writes(fa):
    """Two runs give identical bits; bytes around O stay untouched."""
    w = inputs.Workload("canary", 1, 3, 300, 400, 128, "bf16", True, seed=11)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    n = q.numel()
    pad = 4096
    buf = torch.full((n + 2 * pad,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + n].view(q.shape)
    fa.forward(q, k, v, causal=True, scale=w.scale, out=out)
    first = out.clone()
    fa.forward(q, k, v, causal=True, scale=w.scale, out=out)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))
    assert bool((buf[:pad] == -7.0).all()) and bool((buf[pad + n:] == -7.0).all())


def test_rejections_on_device(fa):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda")
    flat = torch.zeros(128 * 64 + 8, dtype=torch.float16, device="cuda")
    mis = flat[1:1 + 128 * 64]  # 2-byte offset
    assert fa.fa_fwd(mis.data_ptr(), q.data_ptr(), q.data_ptr(), torch.empty_like(q).data_ptr(),
                     1, 1, 128, 128, 64, 0.125, 0, 0, 0) == 3
    q96 = torch.zeros(1, 1, 128, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FaError):
        fa.forward(q96, q96, q96)
    assert fa.last_device_error()[0] == 0


def test_host_buffer_entry_matches_device_entry(fa):
    w = inputs.Workload("host", 1, 4, 257, 300, 128, "bf16", False, seed=12)
    bits = inputs.draw(w)
    dev = inputs.from_torch(run_gpu(fa, bits, w))
    qh, kh, vh = (inputs.to_torch(bits[n], w.dtype).pin_memory() for n in "qkv")
    oh = torch.empty_like(qh).pin_memory()
    fa.forward_host(qh, kh, vh, oh, causal=False, scale=w.scale)
    assert np.array_equal(inputs.from_torch(oh), dev)


@pytest.mark.parametrize("dtype,taus", [("bf16", (0.0, 8.0, 32.0, 64.0)), ("f16", (0.0, 8.0, 15.0, 64.0))])
def test_rescale_threshold_choices_agree(fa, orc, dtype, taus):
    """Rescaling on every rise of the maximum (threshold 0) and lazily (thresholds up to 64; fp16
    launches cap it at 15) are the same computation up to rounding; every choice meets the bar on
    the large-magnitude distribution, whose row maxima move by tens of log2 units."""
    w = inputs.WORKLOADS["rescale_stress"].with_(B=1, H=2, Nq=2048, Nk=2048, dtype=dtype)
    bits = inputs.draw(w)
    ref = orc.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), w.scale, w.causal)
    parity.describe(w)
    old = fa.get_rescale_threshold()
    try:
        outs = {}
        for tau in taus:
            fa.set_rescale_threshold(tau)
            outs[tau] = inputs.from_torch(run_gpu(fa, bits, w))
            parity.assert_parity(parity.compare(outs[tau], ref, w.dtype), False, f"tau={tau}",
                                 mean="literal")
        for tau in taus[1:]:
            diff = np.abs(inputs.bits_to_f64(outs[0.0], w.dtype) - inputs.bits_to_f64(outs[tau], w.dtype))
            assert diff.max() <= 2e-2, tau
    finally:
        fa.set_rescale_threshold(old)


@pytest.mark.parametrize("causal", [False, True])
def test_rescale_on_every_rise_at_d64(fa, orc, causal):
    """D = 64, where the S products of the two query tiles rotate through three TMEM buffers and a
    tile's softmax runs ahead of the PV products: a rescale of O must first wait for the previous
    PV product. Threshold 0 rescales on every rise of the maximum (on the large-magnitude
    distribution, at most key steps), 15 lazily; both meet the bar, causal (one more key tile
    for the second query tile) and not."""
    w = inputs.WORKLOADS["rescale_stress"].with_(name="d64_rescale", B=1, H=2, Nq=1100, Nk=1100,
                                                 D=64, dtype="f16", causal=causal, scale=0.125,
                                                 seed=30 + causal)
    bits = inputs.draw(w)
    ref = orc.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), w.scale, w.causal)
    parity.describe(w)
    old = fa.get_rescale_threshold()
    try:
        for tau in (0.0, 15.0):
            fa.set_rescale_threshold(tau)
            o = inputs.from_torch(run_gpu(fa, bits, w))
            parity.assert_parity(parity.compare(o, ref, w.dtype), True, f"d64 tau={tau}")
    finally:
        fa.set_rescale_threshold(old)


def test_rescale_threshold_setter_validates(fa):
    old = fa.get_rescale_threshold()
    for bad in (-1.0, 64.5, float("inf"), float("nan")):
        with pytest.raises(fa.FaError):
            fa.set_rescale_threshold(bad)
    assert fa.get_rescale_threshold() == old


def test_host_buffer_pipeline_uneven_chunks(fa):
    """The host entry copies and computes in chunks of slices on several streams: 37 slices make
    chunks of 7 and a last one of 2. The result equals the device entry's bit for bit."""
    w = inputs.Workload("host_chunks", 1, 37, 300, 500, 64, "f16", True, seed=13)
    bits = inputs.draw(w)
    dev = inputs.from_torch(run_gpu(fa, bits, w))
    qh, kh, vh = (inputs.to_torch(bits[n], w.dtype).pin_memory() for n in "qkv")
    oh = torch.full_like(qh, 5.0).pin_memory()
    fa.forward_host(qh, kh, vh, oh, causal=True, scale=w.scale)
    assert np.array_equal(inputs.from_torch(oh), dev)


def test_host_buffer_entry_from_two_threads(fa):
    """fa_fwd_host from two host threads at once, with shapes that make the shared staging buffer
    grow between calls: the calls run one after another, and each result equals the device
    entry's bit for bit."""
    import threading

    ws = [inputs.Workload("host_t0", 1, 6, 700, 900, 128, "bf16", False, seed=14),
          inputs.Workload("host_t1", 2, 5, 1500, 1300, 64, "f16", True, seed=15)]
    cases = []
    try:
        fa.set_tail_split(False)  # the host entry runs each chunk as one launch, unsplit
        for w in ws:
            bits = inputs.draw(w)
            dev = inputs.from_torch(run_gpu(fa, bits, w))
            host = [inputs.to_torch(bits[n], w.dtype).pin_memory() for n in "qkv"]
            cases.append((w, dev, host))
    finally:
        fa.set_tail_split(True)
    fa.release_host_buffers()
    errors, outs = [], {}

    def worker(i):
        w, _, (qh, kh, vh) = cases[i]
        try:
            for r in range(3):
                oh = torch.empty_like(qh).pin_memory()
                fa.forward_host(qh, kh, vh, oh, causal=w.causal, scale=w.scale)
                outs[(i, r)] = inputs.from_torch(oh)
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for (i, r), o in outs.items():
        assert np.array_equal(o, cases[i][1]), (i, r)
    assert len(outs) == 6


def test_long_context_chunk_full_size(fa, orc):
    """128 queries against 65536 keys: sampled rows of two heads against the oracle, from the
    split-KV entry, from the default entry (which splits the 8 units over keys by itself) and
    from one unsplit launch."""
    w = inputs.WORKLOADS["long_context_chunk"]
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    outs = {"split": fa.forward_splitkv(q, k, v, scale=w.scale),
            "balanced": fa.forward(q, k, v, scale=w.scale)}
    try:
        fa.set_tail_split(False)
        outs["single"] = fa.forward(q, k, v, scale=w.scale)
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == (0, 0)
    rows = np.array([0, 1, 63, 64, 127])
    parity.describe(w)
    for h in (0, w.H - 1):
        ref = orc.attention_rows(inputs.bits_to_f64(bits["q"][0, h, rows], w.dtype), rows,
                                 inputs.bits_to_f64(bits["k"][0, h], w.dtype),
                                 inputs.bits_to_f64(bits["v"][0, h], w.dtype), w.scale, False)
        for name, o in outs.items():
            got = inputs.from_torch(o)[0, h, rows]
            parity.assert_parity(parity.compare(got, ref, w.dtype), True, f"{name} head {h}")


def test_many_slices_with_split_last_wave(fa, orc):
    """2048 slices of 128 queries against 1024 keys: 2048 units leave a last wave of 72, whose
    keys are split in two (slices 1976 and up). Whole-unit slices and split ones both match
    the oracle."""
    w = inputs.Workload("many_slices", 64, 32, 128, 1024, 64, "bf16", False, seed=14)
    bits = inputs.draw(w)
    o = inputs.from_torch(run_gpu(fa, bits, w))
    parity.describe(w)
    for b, h in ((0, 0), (31, 7), (62, 31), (63, 30), (63, 31)):
        ref = orc.attention(*(inputs.bits_to_f64(bits[n][b, h], w.dtype) for n in "qkv"),
                            w.scale, False)
        parity.assert_parity(parity.compare(o[b, h], ref, w.dtype), True, f"slice ({b},{h})")


@pytest.mark.parametrize("w", [
    # 16 units, split over keys in 4 when run eagerly; one launch under capture.
    inputs.Workload("graph_split", 1, 4, 1024, 1024, 128, "bf16", False, seed=15),
    inputs.Workload("graph_causal", 1, 8, 700, 700, 64, "f16", True, seed=16),
], ids=lambda w: w.name)
def test_cuda_graph_replay_matches_eager(fa, w):
    """Each attention launch is a programmatic dependent of the stream's previous kernel. Two
    forward calls captured back to back in a CUDA graph (the second reading the first's output as
    its Q) replay to the same bits as the eager calls, replay after replay. Under capture the
    default entry never splits over keys (a graph may replay concurrently with anything, so it
    must not share a workspace): the replays equal the eager single launch."""
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    try:
        fa.set_tail_split(False)
        fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=o1)
        fa.forward(o1, k, v, causal=w.causal, scale=w.scale, out=o2)
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    want1, want2 = o1.clone(), o2.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=o1)
            fa.forward(o1, k, v, causal=w.causal, scale=w.scale, out=o2)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        o1.zero_()
        o2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert fa.last_device_error() == (0, 0)
        assert torch.equal(o1.view(torch.int16), want1.view(torch.int16))
        assert torch.equal(o2.view(torch.int16), want2.view(torch.int16))


def test_more_streams_than_workspace_slots(fa, orc):
    """Eight non-blocking streams (the pool has four workspace slots) enqueue split shapes with no
    ordering. A call that finds every slot in use by other streams' unfinished work runs as one
    unsplit launch: with the streams held back while the calls are enqueued, four streams split
    and four run unsplit, every output equals the split or the unsplit result bit for bit, and
    both match the oracle."""
    w = inputs.Workload("slots_few", 1, 2, 300, 3000, 128, "bf16", False, seed=43)
    assert fa.plan(w.B, w.H, w.Nq, w.Nk, w.D, w.causal)["launches"] == 2
    bits = inputs.draw(w)
    qkv = tuple(inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    split_ref = inputs.from_torch(fa.forward(*qkv, scale=w.scale))
    try:
        fa.set_tail_split(False)
        whole_ref = inputs.from_torch(fa.forward(*qkv, scale=w.scale))
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(8)]
    # Hold every stream behind a fixed-length spin (about 10 ms) while the calls are enqueued, so
    # that no slot's last use has finished: the first four streams take the four slots (and keep
    # them: a stream's own slot needs no wait), the other four run unsplit.
    torch.cuda._sleep(20_000_000)
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    reps = 6
    outs = [[torch.empty_like(qkv[0]) for _ in range(reps)] for _ in streams]
    fa.timer_start()
    for r in range(reps):
        for i, s in enumerate(streams):
            fa.forward(*qkv, scale=w.scale, out=outs[i][r], stream=s)
    torch.cuda.synchronize()
    kernels = fa.timer_stop()
    assert fa.last_device_error() == (0, 0)
    n_split = n_whole = 0
    for i in range(len(streams)):
        for r in range(reps):
            got = inputs.from_torch(outs[i][r])
            if np.array_equal(got, split_ref):
                n_split += 1
            else:
                assert np.array_equal(got, whole_ref), f"stream {i} call {r}"
                n_whole += 1
    assert kernels["merge"][1] == n_split
    assert n_split == 4 * reps and n_whole == 4 * reps, (n_split, n_whole)
    ref = orc.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), w.scale)
    for got in (split_ref, whole_ref):
        parity.assert_parity(parity.compare(got, ref, w.dtype), True, "slots_few")


def test_unordered_streams_never_share_a_workspace(fa, orc):
    """Two non-blocking streams run split shapes back to back with no ordering between them: a
    shape whose last wave is split (40 heads x 8 units = 320 units, last wave of 16) and a shape
    whose few units are split 12 ways. Every call's output equals the same call run alone, bit
    for bit, and matches the oracle: the streams' partial states never mix."""
    ws = [inputs.Workload("streams_tail", 1, 40, 2048, 1024, 64, "bf16", False, seed=41),
          inputs.Workload("streams_few", 1, 2, 300, 3000, 128, "bf16", False, seed=42)]
    data = []
    for w in ws:
        plan = fa.plan(w.B, w.H, w.Nq, w.Nk, w.D, w.causal)
        assert plan["launches"] == 2, w.name
        bits = inputs.draw(w)
        qkv = tuple(inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
        alone = inputs.from_torch(fa.forward(*qkv, scale=w.scale))
        torch.cuda.synchronize()
        data.append((w, bits, qkv, alone))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    reps = 6
    outs = [[torch.empty_like(data[(i + r) % 2][2][0]) for r in range(reps)] for i in range(2)]
    fa.timer_start()
    for r in range(reps):
        for i, s in enumerate(streams):
            w, _, qkv, _ = data[(i + r) % 2]
            fa.forward(*qkv, scale=w.scale, out=outs[i][r], stream=s)
    torch.cuda.synchronize()
    kernels = fa.timer_stop()
    assert kernels["merge"][1] == 2 * reps  # every call split and merged
    assert fa.last_device_error() == (0, 0)
    for i in range(2):
        for r in range(reps):
            w, _, _, alone = data[(i + r) % 2]
            got = inputs.from_torch(outs[i][r])
            assert np.array_equal(got, alone), f"stream {i} call {r} ({w.name})"
    for w, bits, _, alone in data:
        h = w.H - 1  # in the split units
        ref = orc.attention(*(inputs.bits_to_f64(bits[n][0, h], w.dtype) for n in "qkv"), w.scale)
        parity.assert_parity(parity.compare(alone[0, h], ref, w.dtype), True, f"{w.name} head {h}")


@pytest.mark.parametrize("w", [
    inputs.Workload("order_split", 1, 4, 1024, 1024, 128, "bf16", False, seed=17),  # fwd + merge
    inputs.Workload("order_causal", 1, 16, 2048, 2048, 128, "bf16", True, seed=18),
], ids=lambda w: w.name)
def test_results_are_ordered_in_the_stream(fa, w):
    """Work queued right after a forward call on the same stream (here a copy of O, and a second
    call that reads O as its Q) sees the call's complete result, with no synchronisation between
    them: the copies equal O read once the device is idle, and the chained call equals the same
    call run on its own."""
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    for _ in range(3):
        fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=o1)
        copy = o1.clone()
        fa.forward(o1, k, v, causal=w.causal, scale=w.scale, out=o2)
        torch.cuda.synchronize()
        assert fa.last_device_error() == (0, 0)
        assert torch.equal(copy.view(torch.int16), o1.view(torch.int16))
        alone = fa.forward(copy, k, v, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(alone.view(torch.int16), o2.view(torch.int16))


def test_million_keys(fa, orc):
    """128 queries against 2^20 keys (256 MB each of K and V): the default entry splits the one
    unit across every SM (ranges of 54-55 key tiles) and merges; the first, middle and last rows
    of the slice are compared with the oracle, which computes them one by one."""
    w = inputs.Workload("million_keys", 1, 1, 128, 1 << 20, 128, "bf16", False, seed=23)
    bits = inputs.draw(w)
    plan = fa.plan(w.B, w.H, w.Nq, w.Nk, w.D, w.causal)
    assert plan["launches"] == 2 and plan["split_units"] * plan["num_splits"] > 100
    o = inputs.from_torch(run_gpu(fa, bits, w))
    rows = np.array([0, 1, 63, 64, 126, 127])
    ref = orc.attention_rows(inputs.bits_to_f64(bits["q"][0, 0, rows], w.dtype), rows,
                             inputs.bits_to_f64(bits["k"][0, 0], w.dtype),
                             inputs.bits_to_f64(bits["v"][0, 0], w.dtype), w.scale, False)
    parity.describe(w)
    parity.assert_parity(parity.compare(o[0, 0, rows], ref, w.dtype), True, w.name)


def test_many_tiny_slices(fa, orc):
    """65 536 (batch, head) slices of 3 queries and 5 keys (65 536 CTAs, each one partial tile):
    every output compared, causal and not."""
    for causal in (False, True):
        w = inputs.Workload("tiny_slices", 64, 1024, 3, 5, 64, "f16", causal, seed=24 + causal)
        full_check(fa, orc, w, literal=False, mean="auto", slices_per_chunk=65536)


def test_rescale_stress_fp32_output_meets_the_literal_bar(fa, orc):
    """The large-magnitude workload at full size with O written in fp32 before any rounding: every
    element within the literal 1e-2 of the exact result and the mean within 1e-3, which the
    16-bit output cannot meet only because rounding |O| >= 4 to bf16 costs up to 0.0156. Rounding
    this fp32 output to bf16 gives fa_fwd's single-launch output bit for bit, so it is the same
    arithmetic."""
    w = inputs.WORKLOADS["rescale_stress"]
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    o32 = fa.forward_f32(q, k, v, causal=w.causal, scale=w.scale)
    try:
        fa.set_tail_split(False)
        o16 = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
    finally:
        fa.set_tail_split(True)
    torch.cuda.synchronize()
    assert fa.last_device_error() == (0, 0)
    got = o32.cpu().numpy().reshape(w.B * w.H, w.Nq, w.D)
    assert np.array_equal(inputs.round_to_bits(got, "bf16").reshape(-1),
                          inputs.from_torch(o16).reshape(-1))
    qq, kk, vv = (bits[n].reshape(w.B * w.H, -1, w.D) for n in "qkv")
    max_err, sum_err, n = 0.0, 0.0, 0
    for c0 in range(0, w.B * w.H, 8):
        ref = orc.attention(*(inputs.bits_to_f64(x[c0:c0 + 8], w.dtype) for x in (qq, kk, vv)),
                            w.scale, w.causal)
        err = np.abs(got[c0:c0 + 8].astype(np.float64) - ref)
        max_err = max(max_err, float(err.max()))
        sum_err += float(err.sum())
        n += err.size
    parity.describe(w)
    stats = dict(max_err=max_err, mean_err=sum_err / n, rounding_floor=0.0, mean_floor=0.0, n=n,
                 finite=bool(np.all(np.isfinite(got))), worst_excess=max_err - parity.MAX_ERR)
    parity.assert_parity(stats, True, "rescale_stress fp32 output")


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes(fa, orc, seed):
    """Seeded random problems: B, H in 1..5, Nq and Nk in 1..700, either head dimension and
    16-bit type, causal or not, scale of either sign and size 0.02-2 / sqrt(D). Every output
    element compared with the oracle, through the default entry (which may split over keys) and,
    non-causal, through the split-KV entry with a random number of ranges."""
    rng = np.random.default_rng(1000 + seed)
    for case in range(5):
        D = int(rng.choice([64, 128]))
        dtype = str(rng.choice(["f16", "bf16"]))
        causal = bool(rng.integers(2))
        B, H = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        Nq, Nk = int(rng.integers(1, 701)), int(rng.integers(1, 701))
        scale = float(np.float32(rng.choice([-1.0, 1.0]) * rng.uniform(0.02, 2.0) / math.sqrt(D)))
        w = inputs.Workload(f"random_{seed}_{case}", B, H, Nq, Nk, D, dtype, causal,
                            seed=seed * 100 + case, scale=scale)
        full_check(fa, orc, w, literal=False, mean="auto")
        if not causal:
            bits = inputs.draw(w)
            q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
            o = fa.forward_splitkv(q, k, v, num_splits=int(rng.integers(1, 9)), scale=w.scale)
            torch.cuda.synchronize()
            assert fa.last_device_error() == (0, 0)
            ref = orc.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), w.scale)
            parity.assert_parity(parity.compare(inputs.from_torch(o), ref, w.dtype), False,
                                 f"{w.name} split-KV", mean="auto")


def test_tensor_map_cache_eviction_and_reuse(fa, orc):
    """The library keeps the last 64 tensor maps, keyed by (address, shape, dtype). Forty problems
    on distinct buffers (160 maps, so entries are evicted and encoded again) run twice more in
    other orders and give the same bits; one set of buffers used with two shapes in turn (same
    addresses, other extents) gives each shape's own result, equal to a run on buffers of its
    own."""
    rng = np.random.default_rng(77)
    ws = [inputs.Workload(f"cache_{i}", 1, 2, int(rng.integers(1, 300)), int(rng.integers(1, 300)),
                          int(rng.choice([64, 128])), "f16", bool(i % 2), seed=700 + i)
          for i in range(40)]
    tensors = []
    for w in ws:
        bits = inputs.draw(w)
        tensors.append(tuple(inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv"))
    first = [fa.forward(q, k, v, causal=w.causal, scale=w.scale) for w, (q, k, v) in zip(ws, tensors)]
    for order in (list(range(39, -1, -1)), list(rng.permutation(40))):
        for i in order:
            w, (q, k, v) = ws[i], tensors[i]
            o = fa.forward(q, k, v, causal=w.causal, scale=w.scale)
            assert torch.equal(o.view(torch.int16), first[i].view(torch.int16)), i
    torch.cuda.synchronize()
    assert fa.last_device_error() == (0, 0)

    # Same base addresses, two shapes.
    D, Nk = 64, 300
    big = {n: torch.zeros(1 * 2 * 512 * D, dtype=torch.float16, device="cuda") for n in "qkvo"}
    results = {}
    for Nq in (512, 128, 512):
        w = inputs.Workload(f"cache_shape_{Nq}", 1, 2, Nq, Nk, D, "f16", False, seed=790 + Nq)
        bits = inputs.draw(w)
        own = [inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv"]
        q = big["q"][:2 * Nq * D].view(1, 2, Nq, D)
        k = big["k"][:2 * Nk * D].view(1, 2, Nk, D)
        v = big["v"][:2 * Nk * D].view(1, 2, Nk, D)
        o = big["o"][:2 * Nq * D].view(1, 2, Nq, D)
        q.copy_(own[0]); k.copy_(own[1]); v.copy_(own[2])
        fa.forward(q, k, v, scale=w.scale, out=o)
        ref = fa.forward(*own, scale=w.scale)
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), Nq
        results[Nq] = inputs.from_torch(o.clone())
        exact = orc.attention(*(inputs.bits_to_f64(bits[n], w.dtype) for n in "qkv"), w.scale)
        parity.assert_parity(parity.compare(results[Nq], exact, w.dtype), False, w.name, mean="auto")
    assert fa.last_device_error() == (0, 0)


def test_splitkv_in_cuda_graph(fa):
    """fa_fwd_splitkv (attention over key ranges, then the merge, which signals the next launch
    early) followed by a forward that reads its output, captured in a CUDA graph: the replays give
    the eager bits, replay after replay."""
    w = inputs.Workload("graph_splitkv", 1, 4, 130, 2048, 128, "bf16", False, seed=17)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    ws = torch.empty(fa.lib().fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.D, 6),
                     dtype=torch.uint8, device="cuda")
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    try:
        fa.set_tail_split(False)  # the second call as one launch, eager and captured alike
        fa.forward_splitkv(q, k, v, num_splits=6, scale=w.scale, out=o1, workspace=ws)
        fa.forward(o1, k, v, scale=w.scale, out=o2)
        torch.cuda.synchronize()
        eager1, eager2 = o1.clone(), o2.clone()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fa.forward_splitkv(q, k, v, num_splits=6, scale=w.scale, out=o1, workspace=ws,
                               stream=s)
            fa.forward(o1, k, v, scale=w.scale, out=o2, stream=s)
        for _ in range(3):
            o1.zero_()
            o2.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(o1.view(torch.int16), eager1.view(torch.int16))
            assert torch.equal(o2.view(torch.int16), eager2.view(torch.int16))
    finally:
        fa.set_tail_split(True)
    assert fa.last_device_error() == (0, 0)
