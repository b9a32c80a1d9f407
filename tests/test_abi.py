"""The C interface without a GPU: libfa.so loads, exports every function include/fa.h declares,
and rejects bad arguments before touching CUDA. CPU only (no compute call is made)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = (ROOT / "include" / "fa.h").read_text()


@pytest.fixture(scope="module")
def fa():
    from tiled_online_softmax_gb300 import build, fa

    if not fa.LIB_PATH.exists():
        build.build()
    fa.lib()
    return fa


def declared_functions():
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(fa_\w+)\s*\(", HEADER, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "fa_fwd" in names and "fa_fwd_host" in names and "fa_last_device_error" in names


def test_every_declared_symbol_is_exported(fa):
    lib = ctypes.CDLL(str(fa.LIB_PATH))
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(fa.EXPORTS) <= set(declared_functions())


def test_status_strings(fa):
    for code, name in fa.STATUS.items():
        assert fa.status_string(code) == name


A = 1 << 20  # a fake, 16-byte aligned address: never dereferenced (validation fails first)


def call(fa, **kw):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, B=1, H=1, Nq=128, Nk=128, D=64, scale=0.125,
                causal=0, dtype=0)
    args.update(kw)
    return fa.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["B"], args["H"], args["Nq"],
                     args["Nk"], args["D"], args["scale"], args["causal"], args["dtype"], 0)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(Nq=0), 1), (dict(Nk=0), 1), (dict(D=0), 1),
    (dict(D=96), 2), (dict(D=256), 2), (dict(D=32), 2),
    (dict(causal=2), 1), (dict(dtype=7), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(q=A + 2), 3), (dict(o=4 * A + 8), 3),
    (dict(o=A), 1),  # output overlaps Q
    (dict(o=2 * A + 64), 1),  # output overlaps K
])
def test_rejects_bad_arguments(fa, kw, status):
    assert call(fa, **kw) == status
    assert fa.lib().fa_last_error_message().decode()


def test_lse_entry_rejects_bad_arguments(fa):
    lse = fa.lib().fa_fwd_lse
    assert lse(A, 2 * A, 3 * A, 4 * A, 0, 1, 1, 8, 8, 64, 0.1, 0, 0, 0) == 1          # null LSE
    assert lse(A, 2 * A, 3 * A, 4 * A, 5 * A + 2, 1, 1, 8, 8, 64, 0.1, 0, 0, 0) == 3  # misaligned
    assert lse(A, 2 * A, 3 * A, 4 * A, 4 * A, 1, 1, 8, 8, 64, 0.1, 0, 0, 0) == 1      # overlaps O
    assert lse(A, 2 * A, 3 * A, 4 * A, 5 * A, 1, 1, 8, 8, 96, 0.1, 0, 0, 0) == 2      # D


def test_host_entry_rejects_bad_arguments(fa):
    assert fa.fa_fwd_host(0, A, A, A, 1, 1, 8, 8, 64, 0.1, 0, 0, 0) == 1
    assert fa.fa_fwd_host(A, A, A, 4 * A, 1, 1, 8, 8, 80, 0.1, 0, 0, 0) == 2


def test_binding_refuses_cpu_tensors(fa):
    import torch

    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.forward(q, q, q)
    with pytest.raises(TypeError):
        fa.forward(q.float(), q.float(), q.float())


def test_wait_selftest_rejects_bad_timeout(fa):
    assert fa.lib().fa_wait_selftest(0, None) == 1
    assert fa.lib().fa_wait_selftest(2_000_000_000, None) == 1


def test_kernel_timer_host_checks(fa):
    import ctypes

    assert fa.lib().fa_timer_stop() == 1  # not running
    ms, n = ctypes.c_double(), ctypes.c_int()
    assert fa.lib().fa_timer_read(6, ctypes.byref(ms), ctypes.byref(n)) == 1
    assert fa.lib().fa_timer_read(-1, ctypes.byref(ms), ctypes.byref(n)) == 1
    assert fa.lib().fa_timer_read(0, None, ctypes.byref(n)) == 1


def test_checked_build_exports_the_same_interface(fa):
    """libfa_debug.so (every global store bounds-checked) exports everything fa.h declares and says
    it checks; the release build says it does not and refuses the bounds self-test."""
    dbg = fa.debug_lib()
    rel = fa._load(fa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(dbg, n)]
    assert not missing, missing
    assert dbg.fa_debug_bounds_enabled() == 1
    assert rel.fa_debug_bounds_enabled() == 0
    assert rel.fa_debug_bounds_selftest(A, None) == 2  # FA_ERR_UNSUPPORTED
    assert dbg.fa_debug_bounds_selftest(None, None) == 1    # null buffer
    assert dbg.fa_debug_bounds_selftest(A + 2, None) == 3   # misaligned
    assert rel.fa_debug_bounds_report(None, None) == 1


def test_workspaces_must_not_overlap_tensors(fa):
    """Caller-owned workspaces of the split-KV, rotary and backward entries are rejected when they
    overlap any tensor of the call (checked before any CUDA call, on fake addresses)."""
    L = fa.lib()
    B, H, N, D = 1, 2, 256, 128
    t = B * H * N * D * 2  # bytes of one 16-bit tensor
    q, k, v, o = A, A + t, A + 2 * t, A + 3 * t
    ws_bad = A + t + 256  # starts inside K
    need = L.fa_splitkv_workspace_bytes(B, H, N, N, D, 2)
    assert L.fa_fwd_splitkv(q, k, v, o, None, B, H, N, N, D, 0.1, 2, 1, ws_bad, need, None) == 1
    assert b"overlaps" in L.fa_last_error_message()
    need = L.fa_rope_workspace_bytes(B, H, N, N, D)
    tab = A + 16 * t
    assert L.fa_fwd_rope(q, k, v, o, None, tab, tab, tab, tab, 0, B, H, N, N, D, 0.1, 0, 1,
                         o + 256, need, None) == 1
    need = L.fa_bwd_workspace_bytes(B, H, N)
    lse, do, dq, dk, dv = A + 4 * t, A + 5 * t, A + 6 * t, A + 7 * t, A + 9 * t
    assert L.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, B, H, N, N, D, 0.1, 0, 1, dq + 512, need,
                    None) == 1
    assert b"overlaps" in L.fa_last_error_message()
