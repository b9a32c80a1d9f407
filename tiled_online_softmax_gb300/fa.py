"""ctypes binding of libfa (include/fa.h). Argument marshalling only: every step of the attention
forward runs in the library's CUDA kernels. There is no fallback: without a built libfa.so or a
GPU, every call raises."""
from __future__ import annotations

import ctypes
import math
import os
from pathlib import Path

LIB_PATH = Path(__file__).resolve().with_name("libfa.so")
DEBUG_LIB_PATH = Path(__file__).resolve().with_name("libfa_debug.so")

FA_F16, FA_BF16 = 0, 1
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARGUMENT", 2: "FA_ERR_UNSUPPORTED",
          3: "FA_ERR_MISALIGNED", 4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT"}
EXPORTS = ("fa_fwd", "fa_fwd_host", "fa_release_host_buffers", "fa_last_device_error",
           "fa_status_string", "fa_last_error_message", "fa_fwd_noalloc",
           "fa_set_rescale_threshold", "fa_get_rescale_threshold", "fa_fwd_lse",
           "fa_splitkv_workspace_bytes", "fa_fwd_splitkv", "fa_set_tail_split", "fa_rope",
           "fa_rope_workspace_bytes", "fa_fwd_rope", "fa_bwd_workspace_bytes", "fa_bwd",
           "fa_wait_selftest", "fa_wait_selftest_noalloc", "fa_timer_start", "fa_timer_stop",
           "fa_timer_read", "fa_fwd_plan", "fa_debug_bounds_enabled", "fa_debug_bounds_report",
           "fa_debug_bounds_selftest", "fa_fwd_f32out")


class Plan(ctypes.Structure):
    """struct fa_plan: how fa_fwd divides a shape into launches."""
    _fields_ = [("units", ctypes.c_int64), ("split_begin", ctypes.c_int64),
                ("split_units", ctypes.c_int64), ("num_splits", ctypes.c_int),
                ("tiles_per_split", ctypes.c_int), ("ctas", ctypes.c_int64),
                ("launches", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]


class FaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib: ctypes.CDLL | None = None
_debug_lib: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    """The loaded libfa.so with its signatures declared; libfa_debug.so, the bounds-checked
    build, instead when the environment sets FA_CHECKED_BUILD=1."""
    global _lib
    if _lib is None:
        _lib = debug_lib() if os.environ.get("FA_CHECKED_BUILD") == "1" else _load(LIB_PATH)
    return _lib


def debug_lib() -> ctypes.CDLL:
    """The bounds-checked build, libfa_debug.so (same functions, same results; every global store
    checked against its tensor's extent)."""
    global _debug_lib
    if _debug_lib is None:
        _debug_lib = _load(DEBUG_LIB_PATH)
    return _debug_lib


def _load(path: Path) -> ctypes.CDLL:
    if not path.exists():
        raise RuntimeError(f"{path} is not built: run tiled_online_softmax_gb300.build.build()")
    L = ctypes.CDLL(str(path))
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    sig = [vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, ctypes.c_int, vp]
    L.fa_fwd.argtypes = sig
    L.fa_fwd.restype = ctypes.c_int
    L.fa_fwd_host.argtypes = sig
    L.fa_fwd_host.restype = ctypes.c_int
    L.fa_fwd_noalloc.argtypes = sig
    L.fa_fwd_noalloc.restype = ctypes.c_int
    L.fa_fwd_lse.argtypes = sig[:4] + [vp] + sig[4:]
    L.fa_fwd_lse.restype = ctypes.c_int
    L.fa_fwd_f32out.argtypes = sig[:4] + [vp] + sig[4:]
    L.fa_fwd_f32out.restype = ctypes.c_int
    L.fa_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int]
    L.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
    L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_float,
                                 ctypes.c_int, ctypes.c_int, vp, ctypes.c_size_t, vp]
    L.fa_fwd_splitkv.restype = ctypes.c_int
    L.fa_set_tail_split.argtypes = [ctypes.c_int]
    L.fa_set_tail_split.restype = ctypes.c_int
    L.fa_rope.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int, vp]
    L.fa_rope.restype = ctypes.c_int
    L.fa_rope_workspace_bytes.argtypes = [i64, i64, i64, i64, i64]
    L.fa_rope_workspace_bytes.restype = ctypes.c_size_t
    L.fa_fwd_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, i64, i64, i64,
                              i64, i64, ctypes.c_float, ctypes.c_int, ctypes.c_int, vp,
                              ctypes.c_size_t, vp]
    L.fa_fwd_rope.restype = ctypes.c_int
    L.fa_bwd_workspace_bytes.argtypes = [i64, i64, i64]
    L.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    L.fa_bwd.argtypes = [vp] * 9 + [i64] * 5 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, vp,
                                                 ctypes.c_size_t, vp]
    L.fa_bwd.restype = ctypes.c_int
    L.fa_release_host_buffers.argtypes = []
    L.fa_release_host_buffers.restype = ctypes.c_int
    L.fa_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    L.fa_last_device_error.restype = ctypes.c_int
    L.fa_wait_selftest.argtypes = [ctypes.c_ulonglong, vp]
    L.fa_wait_selftest.restype = ctypes.c_int
    L.fa_wait_selftest_noalloc.argtypes = [ctypes.c_ulonglong, vp]
    L.fa_wait_selftest_noalloc.restype = ctypes.c_int
    L.fa_fwd_plan.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                              ctypes.POINTER(Plan)]
    L.fa_fwd_plan.restype = ctypes.c_int
    L.fa_timer_start.argtypes = []
    L.fa_timer_start.restype = ctypes.c_int
    L.fa_timer_stop.argtypes = []
    L.fa_timer_stop.restype = ctypes.c_int
    L.fa_timer_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                ctypes.POINTER(ctypes.c_int)]
    L.fa_timer_read.restype = ctypes.c_int
    L.fa_status_string.argtypes = [ctypes.c_int]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_last_error_message.argtypes = []
    L.fa_last_error_message.restype = ctypes.c_char_p
    L.fa_set_rescale_threshold.argtypes = [ctypes.c_float]
    L.fa_set_rescale_threshold.restype = ctypes.c_int
    L.fa_get_rescale_threshold.argtypes = []
    L.fa_get_rescale_threshold.restype = ctypes.c_float
    L.fa_debug_bounds_enabled.argtypes = []
    L.fa_debug_bounds_enabled.restype = ctypes.c_int
    L.fa_debug_bounds_report.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_longlong)]
    L.fa_debug_bounds_report.restype = ctypes.c_int
    L.fa_debug_bounds_selftest.argtypes = [vp, vp]
    L.fa_debug_bounds_selftest.restype = ctypes.c_int
    return L


def _raise_if(status: int) -> None:
    if status != 0:
        raise FaError(status, lib().fa_last_error_message().decode())


def fa_fwd(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, B: int, H: int, Nq: int, Nk: int,
           D: int, scale: float, causal: int, dtype: int, stream: int = 0) -> int:
    """The raw C call on device pointers; returns the fa_status code."""
    return lib().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, B, H, Nq, Nk, D, scale, causal, dtype, stream)


def fa_fwd_host(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, B: int, H: int, Nq: int,
                Nk: int, D: int, scale: float, causal: int, dtype: int, stream: int = 0) -> int:
    """The raw C call on host pointers (synchronous); returns the fa_status code."""
    return lib().fa_fwd_host(q_ptr, k_ptr, v_ptr, o_ptr, B, H, Nq, Nk, D, scale, causal, dtype,
                             stream)


def fa_fwd_noalloc(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, B: int, H: int, Nq: int,
                   Nk: int, D: int, scale: float, causal: int, dtype: int, stream: int = 0) -> int:
    """The raw allocation-free C call on device pointers; returns the fa_status code."""
    return lib().fa_fwd_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, B, H, Nq, Nk, D, scale, causal, dtype,
                                stream)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float16:
        return FA_F16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"attention inputs must be float16 or bfloat16, got {t.dtype}")


def _shape(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, H, Nq, D = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != D or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    return B, H, Nq, k.shape[2], D


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, stream=None):
    """O = softmax(scale * q k^T) v for CUDA tensors q [B,H,Nq,D], k, v [B,H,Nk,D].

    Launches on `stream` (default: torch's current stream) and returns `out` without waiting.
    """
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    code = _dtype_code(q)
    if not q.is_cuda:
        raise ValueError("forward() takes CUDA tensors; use forward_host() for host buffers")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _raise_if(fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, Nq, Nk,
                         D, float(scale), int(bool(causal)), code, stream.cuda_stream))
    return out


def forward_lse(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                stream=None):
    """(O, LSE) for CUDA tensors; LSE[b, h, i] = log sum_j exp(scale * q_i . k_j), fp32."""
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    code = _dtype_code(q)
    if not q.is_cuda:
        raise ValueError("forward_lse() takes CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, Nq]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _raise_if(lib().fa_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse.data_ptr(), B, H, Nq, Nk, D, float(scale),
                                   int(bool(causal)), code, stream.cuda_stream))
    return out, lse


def forward_f32(q, k, v, causal: bool = False, scale: float | None = None, lse=None, stream=None):
    """O in fp32, unrounded (a checking aid: the arithmetic without the 16-bit output rounding),
    for CUDA tensors; one launch."""
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    if not q.is_cuda:
        raise ValueError("forward_f32() takes CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = torch.empty(B, H, Nq, D, dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _raise_if(lib().fa_fwd_f32out(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                      lse.data_ptr() if lse is not None else None, B, H, Nq, Nk,
                                      D, float(scale), int(bool(causal)), _dtype_code(q),
                                      stream.cuda_stream))
    return out


def splitkv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, D: int, num_splits: int = 0) -> int:
    return int(lib().fa_splitkv_workspace_bytes(B, H, Nq, Nk, D, num_splits))


def forward_splitkv(q, k, v, num_splits: int = 0, scale: float | None = None, out=None,
                    lse=None, workspace=None, stream=None):
    """Non-causal attention with the keys split into ranges and the partial states merged.
    `workspace` (a CUDA tensor of at least splitkv_workspace_bytes bytes) is allocated here
    when not given."""
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    code = _dtype_code(q)
    if not q.is_cuda:
        raise ValueError("forward_splitkv() takes CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    need = splitkv_workspace_bytes(B, H, Nq, Nk, D, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _raise_if(lib().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse.data_ptr() if lse is not None else None, B, H, Nq, Nk,
                                       D, float(scale), int(num_splits), code,
                                       workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                       stream.cuda_stream))
    return out


def rope(x, cos_t, sin_t, form: int = 0, out=None, stream=None):
    """Rotary embedding of x [B, H, N, D] (CUDA, 16-bit) with fp32 tables [N, D/2]; returns out
    (pass out=x to rotate in place)."""
    import torch

    if x.dim() != 4 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [B, H, N, D]")
    B, H, N, D = x.shape
    for t in (cos_t, sin_t):
        if t.dtype != torch.float32 or tuple(t.shape) != (N, D // 2) or not t.is_contiguous():
            raise ValueError("cos/sin tables must be contiguous float32 [N, D/2]")
    if out is None:
        out = torch.empty_like(x)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        _raise_if(lib().fa_rope(x.data_ptr(), out.data_ptr(), cos_t.data_ptr(), sin_t.data_ptr(),
                                B, H, N, D, int(form), _dtype_code(x), stream.cuda_stream))
    return out


def forward_rope(q, k, v, cos_q, sin_q, cos_k, sin_k, form: int = 0, causal: bool = False,
                 scale: float | None = None, out=None, lse=None, workspace=None, stream=None):
    """Attention on rotary-embedded q and k (the rotation runs on device copies)."""
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    need = int(lib().fa_rope_workspace_bytes(B, H, Nq, Nk, D))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        _raise_if(lib().fa_fwd_rope(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr() if lse is not None else None,
                                    cos_q.data_ptr(), sin_q.data_ptr(), cos_k.data_ptr(),
                                    sin_k.data_ptr(), int(form), B, H, Nq, Nk, D, float(scale),
                                    int(bool(causal)), code, workspace.data_ptr(),
                                    workspace.numel(), stream.cuda_stream))
    return out


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             workspace=None, stream=None):
    """(dQ, dK, dV) for CUDA tensors, from the forward's inputs, its O and LSE (forward_lse)
    and the upstream gradient dout."""
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = int(lib().fa_bwd_workspace_bytes(B, H, Nq))
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    for t in (o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("o and dout must be contiguous and shaped like q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, Nq]")
    with torch.cuda.device(q.device):
        _raise_if(lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                               dv.data_ptr(), B, H, Nq, Nk, D, float(scale), int(bool(causal)),
                               code, workspace.data_ptr(), workspace.numel(), stream.cuda_stream))
    return dq, dk, dv


def forward_host(q, k, v, out, causal: bool = False, scale: float | None = None, stream=None,
                 device: int = 0):
    """The same on host (CPU, ideally pinned) tensors: copies in, runs, copies out, waits."""
    import torch

    B, H, Nq, Nk, D = _shape(q, k, v)
    if q.is_cuda or out.is_cuda:
        raise ValueError("forward_host() takes host tensors")
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor shaped and typed like q")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(device):
        if stream is None:
            stream = torch.cuda.current_stream(device)
        _raise_if(fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                              Nq, Nk, D, float(scale), int(bool(causal)), _dtype_code(q),
                              stream.cuda_stream))
    return out


def release_host_buffers(device: int = 0) -> None:
    """Free the device staging buffers forward_host() keeps on `device`."""
    import torch

    with torch.cuda.device(device):
        _raise_if(lib().fa_release_host_buffers())


def last_device_error(stream=None) -> tuple[int, int]:
    """Synchronise `stream` and return (status, wait-site code) of the device error word."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    site = ctypes.c_int(0)
    st = lib().fa_last_device_error(stream.cuda_stream, ctypes.byref(site))
    return st, site.value


KERNEL_KINDS = ("fwd", "merge", "rope", "bwd_prep", "bwd_dkdv", "bwd_dq")  # fa_kernel_kind order


def timer_start() -> None:
    """Start the library's kernel timer: each launch from now on is bracketed by CUDA events."""
    _raise_if(lib().fa_timer_start())


def timer_stop() -> dict:
    """Stop the kernel timer; {kind: (total device ms, launches)} for every kind that ran."""
    _raise_if(lib().fa_timer_stop())
    out = {}
    for i, name in enumerate(KERNEL_KINDS):
        ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
        _raise_if(lib().fa_timer_read(i, ctypes.byref(ms), ctypes.byref(n)))
        if n.value:
            out[name] = (ms.value, n.value)
    return out


def wait_selftest(timeout_ns: int, stream=None) -> None:
    """Launch the bounded-wait self-test on `stream`: a wait that runs out after timeout_ns and
    leaves its site code in the device error word (read it with last_device_error)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    _raise_if(lib().fa_wait_selftest(int(timeout_ns), stream.cuda_stream))


def wait_selftest_noalloc(timeout_ns: int, stream=None) -> None:
    """The same self-test aimed at fa_fwd_noalloc's static record (allocates nothing)."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    _raise_if(lib().fa_wait_selftest_noalloc(int(timeout_ns), stream.cuda_stream))


def plan(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool = False, num_sms: int = 0) -> dict:
    """How forward() divides a shape into launches on `num_sms` SMs (0: the current device)."""
    p = Plan()
    _raise_if(lib().fa_fwd_plan(B, H, Nq, Nk, D, int(bool(causal)), int(num_sms), ctypes.byref(p)))
    return {name: getattr(p, name) for name, _ in Plan._fields_}


def set_rescale_threshold(log2_threshold: float) -> None:
    """Process-wide lazy-rescale threshold (log2 units, [0, 64]; 0 = rescale on every rise;
    fp16 launches use at most 15)."""
    _raise_if(lib().fa_set_rescale_threshold(float(log2_threshold)))


def set_tail_split(enable: bool) -> None:
    """Turn forward()'s work balancing (key splits of some units, then a merge) on or off
    (process-wide)."""
    _raise_if(lib().fa_set_tail_split(int(bool(enable))))


def get_rescale_threshold() -> float:
    return float(lib().fa_get_rescale_threshold())


def bounds_report(L: ctypes.CDLL | None = None) -> tuple[int, int]:
    """(site, index) of the first bounds violation the checked build recorded since the last
    report, (0, 0) if none; read and cleared. Synchronise the device first."""
    L = L or debug_lib()
    site, index = ctypes.c_int(0), ctypes.c_longlong(0)
    st = L.fa_debug_bounds_report(ctypes.byref(site), ctypes.byref(index))
    if st != 0:
        raise FaError(st, L.fa_last_error_message().decode())
    return site.value, index.value


def status_string(status: int) -> str:
    return lib().fa_status_string(status).decode()
