"""Work planning of the default forward entry (fa_fwd_plan), on the CPU: how a shape is divided
into launches for a given SM count. No GPU is touched (the SM count is passed in)."""
import pytest

from tiled_online_softmax_gb300 import inputs


@pytest.fixture(scope="module")
def fa():
    from tiled_online_softmax_gb300 import build, fa

    if not fa.LIB_PATH.exists():
        build.build()
    fa.lib()
    return fa


def plan(fa, w, sms):
    return fa.plan(w.B, w.H, w.Nq, w.Nk, w.D, w.causal, num_sms=sms)


def test_headline_splits_its_last_wave_on_152_sms(fa):
    # 32 heads x 16 units of 256 rows = 512 units: 3 full waves of 152 and a last wave of 56,
    # whose units are split into floor(152 / 56) = 2 key ranges of 16 tiles.
    p = plan(fa, inputs.WORKLOADS["headline"], 152)
    assert p["units"] == 512 and p["launches"] == 2
    assert (p["split_begin"], p["split_units"], p["num_splits"], p["tiles_per_split"]) == (456, 56, 2, 16)
    assert p["ctas"] == 456 + 112
    assert p["workspace_bytes"] == (2 * 56 * 256 * 128 * 4) + 2 * 56 * 256 * 8


def test_plan_follows_the_sm_count(fa):
    w = inputs.WORKLOADS["headline"]
    # 132 SMs: 512 = 3 x 132 + 116; a last wave of 116 > 66 is not split.
    assert plan(fa, w, 132)["launches"] == 1
    # 148 SMs: last wave of 68 <= 74 -> 2 ranges.
    p = plan(fa, w, 148)
    assert (p["split_begin"], p["split_units"], p["num_splits"]) == (444, 68, 2)
    # 512 SMs: one wave, nothing to split (512 units > 256 = half the SMs).
    assert plan(fa, w, 512)["launches"] == 1


def test_few_units_cover_the_sms(fa):
    # 8 units of 128 rows against 512 key tiles: each split into floor(S / 8) ranges.
    w = inputs.WORKLOADS["long_context_chunk"]
    for sms, splits in ((152, 19), (64, 8), (16, 2)):
        p = plan(fa, w, sms)
        assert p["split_units"] == 8 and p["num_splits"] == splits, sms
        assert p["ctas"] == 8 * splits
    assert plan(fa, w, 8)["launches"] == 1  # 8 units fill 8 SMs already


@pytest.mark.parametrize("sms", [1, 2, 3, 16, 76, 132, 148, 152, 160, 264])
def test_split_ctas_never_exceed_the_sm_count(fa, sms):
    """The split units times their ranges stay within the SM count, so the partial state always
    fits the fixed-size workspace of S * 256 rows of D = 128."""
    bound = sms * 256 * (128 * 4 + 8) + 256
    for B, H, Nq, Nk, D in [(1, 32, 4096, 4096, 128), (1, 8, 128, 65536, 128), (2, 4, 1000, 1000, 64),
                            (64, 32, 128, 1024, 64), (1, 1, 1, 100000, 64), (3, 7, 300, 5000, 128),
                            (1, 40, 2048, 1024, 64), (4, 32, 4096, 4096, 128)]:
        p = fa.plan(B, H, Nq, Nk, D, False, num_sms=sms)
        assert p["split_units"] * p["num_splits"] <= max(sms, 0) or p["launches"] == 1
        assert p["workspace_bytes"] <= bound
        if p["launches"] == 2:
            nkt = -(-Nk // 128)
            assert p["num_splits"] >= 2 and p["tiles_per_split"] * (p["num_splits"] - 1) < nkt
            assert p["ctas"] == p["split_begin"] + p["split_units"] * p["num_splits"]


def test_causal_and_short_key_ranges_run_as_one_launch(fa):
    assert plan(fa, inputs.WORKLOADS["causal_prefill"], 152)["launches"] == 1
    assert plan(fa, inputs.WORKLOADS["long_causal"], 152)["launches"] == 1
    # 2 units, 3 key tiles: ranges would be shorter than 2 tiles.
    assert fa.plan(1, 2, 200, 380, 64, False, num_sms=152)["launches"] == 1


def test_tail_split_switch(fa):
    w = inputs.WORKLOADS["headline"]
    try:
        fa.set_tail_split(False)
        assert plan(fa, w, 152)["launches"] == 1
    finally:
        fa.set_tail_split(True)
    assert plan(fa, w, 152)["launches"] == 2


def test_plan_rejects_bad_arguments(fa):
    for args, status in [((0, 1, 8, 8, 64, 0, 152), 1), ((1, 1, 8, 8, 96, 0, 152), 2),
                         ((1, 1, 8, 8, 64, 2, 152), 1), ((1, 1, 8, 8, 64, 0, -1), 1)]:
        p = fa.Plan()
        assert fa.lib().fa_fwd_plan(*args, fa.ctypes.byref(p)) == status
    assert fa.lib().fa_fwd_plan(1, 1, 8, 8, 64, 0, 152, None) == 1
