"""The library's kernel timer: it counts and times every launch by kernel kind."""
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
    return fa_mod


def test_timer_counts_launches_by_kind(fa):
    # A decoding shape split over keys: each call is an attention launch and a merge launch.
    w = inputs.Workload("timer", 1, 4, 64, 4096, 64, "bf16", False, seed=91)
    bits = inputs.draw(w)
    q, k, v = (inputs.to_torch(bits[n], w.dtype).cuda() for n in "qkv")
    ws = torch.empty(fa.splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.D, 8), dtype=torch.uint8,
                     device="cuda")
    run = lambda: fa.forward_splitkv(q, k, v, num_splits=8, scale=w.scale, workspace=ws)
    run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.timer_start()
    e0.record(stream)
    for _ in range(5):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    kernels = fa.timer_stop()
    assert set(kernels) == {"fwd", "merge"}
    assert kernels["fwd"][1] == 5 and kernels["merge"][1] == 5
    total = e0.elapsed_time(e1)
    timed = kernels["fwd"][0] + kernels["merge"][0]
    assert 0 < timed <= total * 1.001
    assert kernels["fwd"][0] > kernels["merge"][0]
    # Stopped: further launches are not counted, and a second stop is an error.
    run()
    with pytest.raises(fa.FaError):
        fa.timer_stop()
    assert fa.last_device_error() == (0, 0)
