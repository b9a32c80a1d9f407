"""Host-side logic of bench.py that needs no GPU: which profile summary's DRAM traffic the
roofline line may quote."""
import importlib.util
import pathlib
import sys

ROOT = pathlib.Path(__file__).resolve().parents[1]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_kernel_code_ignores_comments_and_blank_lines():
    b = _bench()
    src = "int a = 1;  // first\n\n// a whole comment line\n  int b = a;   \n"
    assert b.kernel_code(src) == "int a = 1;\n  int b = a;"
    assert b.kernel_code(src + "// another note\n") == b.kernel_code(src)
    assert b.kernel_code(src.replace("a = 1", "a = 2")) != b.kernel_code(src)


def test_committed_headline_profile_matches_the_kernel_code():
    """When the committed ncu summary was taken on the current forward kernel code, the bench
    line quotes its traffic, and the figure is plausible. (After a code change the bench reports
    null until the summary is re-taken; the test then skips and says so.)"""
    import pytest

    b = _bench()
    traffic = b.profiled_traffic("headline")
    if traffic is None:
        pytest.skip("profiles/fa_fwd_kernel_headline.md predates the kernel code: re-take it")
    # Q, K, V read once and O written once at the headline shape: 134.2 MB; the summary's DRAM
    # bytes lie between the reads alone and that.
    assert 100e6 < traffic <= 135e6


def test_profile_summary_with_another_hash_is_ignored(tmp_path, monkeypatch):
    b = _bench()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "fa_fwd_kernel_headline.md").write_text(
        "- kernel_source_sha256_16: `0000000000000000`\n- dram_bytes_per_launch: `1`\n")
    src = tmp_path / "tiled_online_softmax_gb300" / "csrc"
    src.mkdir(parents=True)
    for s in b.KERNEL_SOURCES:
        (tmp_path / s).write_text((ROOT / s).read_text())
    monkeypatch.setattr(b, "ROOT", tmp_path)
    assert b.profiled_traffic("headline") is None
