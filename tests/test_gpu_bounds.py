"""The bounds-checked build (libfa_debug.so) on the GPU: a planted out-of-bounds index is caught
and its store skipped, and every entry point run through the checked build gives the release
build's bits with no violation recorded. The checks stand in for a memory sanitizer: each global
store is compared with the extent of the tensor it writes before it is made."""
import ctypes

import numpy as np
import pytest

from tiled_online_softmax_gb300 import inputs

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_gb300 import fa as fa_mod

    fa_mod.lib()
    fa_mod.debug_lib()
    return fa_mod


def test_planted_violation_is_recorded_and_skipped(fa):
    dbg = fa.debug_lib()
    assert fa.bounds_report(dbg) == (0, 0)
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    assert dbg.fa_debug_bounds_selftest(buf.data_ptr(), None) == 0
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    assert got[8] == 1 and got[40] == 0 and got.sum() == 1  # in-bounds store made, the other not
    assert fa.bounds_report(dbg) == (49, 40)
    assert fa.bounds_report(dbg) == (0, 0)  # read and cleared


def _bits(t):
    return inputs.from_torch(t)


def _fwd(L, w, q, k, v, o, lse=None):
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr())
    tail = (w.B, w.H, w.Nq, w.Nk, w.D, w.scale, int(w.causal), w.dtype_code, None)
    st = L.fa_fwd_lse(*args, lse.data_ptr(), *tail) if lse is not None else L.fa_fwd(*args, *tail)
    assert st == 0, L.fa_last_error_message().decode()


@pytest.mark.parametrize("w", [
    inputs.Workload("chk_split", 1, 4, 1024, 1024, 128, "bf16", False, seed=91),      # key split + merge
    inputs.Workload("chk_causal_ragged", 2, 3, 300, 300, 128, "bf16", True, seed=92),
    inputs.Workload("chk_d64_wide", 1, 3, 257, 700, 64, "f16", False, seed=93),
    inputs.Workload("chk_decode", 1, 8, 1, 4096, 128, "bf16", False, seed=94),         # 8 units split
    inputs.Workload("chk_causal_wide", 1, 2, 130, 400, 64, "bf16", True, seed=95),
], ids=lambda w: w.name)
def test_checked_forward_equals_release(fa, w):
    rel, dbg = fa.lib(), fa.debug_lib()
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    outs = {}
    for name, L in (("release", rel), ("checked", dbg)):
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
        _fwd(L, w, q, k, v, o, lse)
        o2 = torch.empty_like(q)
        _fwd(L, w, q, k, v, o2)
        outs[name] = (o, lse, o2)
    torch.cuda.synchronize()
    assert fa.bounds_report(dbg) == (0, 0)
    for a, b in zip(outs["release"], outs["checked"]):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                           b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))


def test_checked_rope_splitkv_and_backward_equal_release(fa):
    rel, dbg = fa.lib(), fa.debug_lib()
    w = inputs.Workload("chk_all", 1, 3, 300, 900, 128, "bf16", False, seed=96)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    do = inputs.to_torch(inputs.draw(w.with_(seed=97))["q"], w.dtype).cuda()
    half = w.D // 2
    ang = np.arange(max(w.Nq, w.Nk))[:, None] * 10000.0 ** (-np.arange(half) / half)
    ct = torch.from_numpy(np.cos(ang).astype(np.float32)).cuda()
    sn = torch.from_numpy(np.sin(ang).astype(np.float32)).cuda()
    res = {}
    for name, L in (("release", rel), ("checked", dbg)):
        r = {}
        # rotary pass alone, then attention with rotary Q (in the kernel) and K (its pass)
        r["rope"] = torch.empty_like(k)
        assert L.fa_rope(k.data_ptr(), r["rope"].data_ptr(), ct.data_ptr(), sn.data_ptr(), w.B, w.H,
                         w.Nk, w.D, 1, w.dtype_code, None) == 0
        ws = torch.empty(L.fa_rope_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.D), dtype=torch.uint8,
                         device="cuda")
        r["fwd_rope"] = torch.empty_like(q)
        assert L.fa_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), r["fwd_rope"].data_ptr(), None,
                             ct.data_ptr(), sn.data_ptr(), ct.data_ptr(), sn.data_ptr(), 0, w.B, w.H,
                             w.Nq, w.Nk, w.D, w.scale, 0, w.dtype_code, ws.data_ptr(), ws.numel(),
                             None) == 0
        # split over keys with the caller's workspace
        n_ws = L.fa_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.D, 5)
        wsk = torch.empty(n_ws, dtype=torch.uint8, device="cuda")
        r["splitkv"] = torch.empty_like(q)
        assert L.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), r["splitkv"].data_ptr(),
                                None, w.B, w.H, w.Nq, w.Nk, w.D, w.scale, 5, w.dtype_code,
                                wsk.data_ptr(), n_ws, None) == 0
        # backward, causal and ragged
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device="cuda")
        assert L.fa_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            w.B, w.H, w.Nq, w.Nk, w.D, w.scale, 1, w.dtype_code, None) == 0
        wsb = torch.empty(L.fa_bwd_workspace_bytes(w.B, w.H, w.Nq), dtype=torch.uint8, device="cuda")
        r["dq"], r["dk"], r["dv"] = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        assert L.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                        lse.data_ptr(), r["dq"].data_ptr(), r["dk"].data_ptr(), r["dv"].data_ptr(),
                        w.B, w.H, w.Nq, w.Nk, w.D, w.scale, 1, w.dtype_code, wsb.data_ptr(),
                        wsb.numel(), None) == 0
        res[name] = r
    torch.cuda.synchronize()
    assert fa.bounds_report(dbg) == (0, 0)
    for key in res["release"]:
        assert np.array_equal(_bits(res["release"][key]), _bits(res["checked"][key])), key
