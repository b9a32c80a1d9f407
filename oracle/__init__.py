"""fp64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. The product path (``tiled_online_softmax_gb300``) never imports it, and the two
share no code: this package wraps the plain C file ``oracle.c`` (float64, libm ``exp``/``log``)
through ctypes and adds nothing to its arithmetic.

Functions and the passages they follow (page title, section):

* ``attention``        -- "11. Fusion, recompute, and flash attention" section 11.2 (definition of
  S, P, O) with the stable softmax of ithelp article 10405336 ("先回顧 Stable Softmax").
* ``attention_rows``   -- the same definition for selected query rows of one (batch, head) slice.
* ``softmax``          -- the P matrix of that definition.
* ``attention_online`` -- section 11.6 "Online softmax", taken b keys at a time as in
  "Flash Attention 2", "Overview of the algorithm".
* ``online_state``     -- the unnormalised running state (m, l, o) of that recurrence.
* ``merge_state``      -- section 11.6, merge of two partial states (exercise 3).
* ``attention_backward`` -- dQ, dK, dV of the definition (section 11.9, "Backward"; the pages
  print no formulas, so this is the plain derivative of section 11.2's definition).
* ``rope``             -- "Attention" (phobos stdlib docs), "Rotary position embeddings":
  `rope` (rotate-half) and `rope_pairs` (interleaved pairs).

Every function is pinned by ``tests/test_oracle.py`` against values the pages print, closed
forms, invariants and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_LIB = _HERE / "liboracle.so"

# -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts give bit-identical results.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(src: Path = _SRC, out: Path = _LIB, extra_flags: list[str] | None = None) -> Path:
    """Compile ``oracle.c`` (or another C file with the same exports) into a shared library."""
    cmd = ["gcc", *CFLAGS, *(extra_flags or []), "-o", str(out), str(src), "-lm"]
    subprocess.run(cmd, check=True)
    return out


_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)
_i64 = ctypes.c_int64


def load(path: Path | None = None) -> ctypes.CDLL:
    """Load a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(str(path or _LIB))
    lib.oracle_attention.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64, ctypes.c_double,
                                     ctypes.c_int, _dp, _dp]
    lib.oracle_attention_rows.argtypes = [_dp, _ip, _i64, _dp, _dp, _i64, _i64, ctypes.c_double,
                                          ctypes.c_int, _dp, _dp]
    lib.oracle_softmax.argtypes = [_dp, _dp, _i64, _i64, _i64, ctypes.c_double, ctypes.c_int, _dp]
    lib.oracle_online_state.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, ctypes.c_double, _i64,
                                        _dp, _dp, _dp]
    lib.oracle_merge_state.argtypes = [ctypes.c_double, ctypes.c_double, _dp, ctypes.c_double,
                                       ctypes.c_double, _dp, _i64, _dp, _dp, _dp]
    lib.oracle_attention_online.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                            ctypes.c_double, ctypes.c_int, _i64, _dp, _dp]
    lib.oracle_rope.argtypes = [_dp, _dp, _dp, _i64, _i64, ctypes.c_int]
    lib.oracle_attention_backward.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                              ctypes.c_double, ctypes.c_int, _dp, _dp, _dp]
    lib.oracle_num_threads.argtypes = []
    for name in ("oracle_attention", "oracle_attention_rows", "oracle_softmax",
                 "oracle_online_state", "oracle_merge_state", "oracle_attention_online",
                 "oracle_rope", "oracle_attention_backward", "oracle_num_threads"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib: ctypes.CDLL | None = None


def _get() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not _LIB.exists() or _LIB.stat().st_mtime < _SRC.stat().st_mtime:
            build()
        _lib = load()
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


class Oracle:
    """The oracle entry points bound to one compiled library (the default one, or a test build)."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    def attention(self, q, k, v, scale: float, causal: bool = False, with_lse: bool = False):
        """O (and LSE) for q: [..., Nq, D], k, v: [..., Nk, D]; leading dims are independent."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        *lead, nq, d = q.shape
        nk = k.shape[-2]
        bh = int(np.prod(lead)) if lead else 1
        out = np.empty(q.shape, np.float64)
        lse = np.empty((*lead, nq), np.float64)
        _check(self.lib.oracle_attention(_ptr(q), _ptr(k), _ptr(v), bh, nq, nk, d, float(scale),
                                         int(bool(causal)), _ptr(out), _ptr(lse)), "attention")
        return (out, lse) if with_lse else out

    def attention_rows(self, q_rows, row_pos, k, v, scale: float, causal: bool = False,
                       with_lse: bool = False):
        """O for selected query rows of ONE slice: q_rows [R, D] at positions row_pos [R]."""
        q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
        pos = np.ascontiguousarray(row_pos, dtype=np.int64)
        n_rows, d = q_rows.shape
        out = np.empty((n_rows, d), np.float64)
        lse = np.empty(n_rows, np.float64)
        _check(self.lib.oracle_attention_rows(_ptr(q_rows), pos.ctypes.data_as(_ip), n_rows,
                                              _ptr(k), _ptr(v), k.shape[0], d, float(scale),
                                              int(bool(causal)), _ptr(out), _ptr(lse)),
               "attention_rows")
        return (out, lse) if with_lse else out

    def softmax(self, q, k, scale: float, causal: bool = False) -> np.ndarray:
        """P = softmax(scale * q k^T) of one slice, zeros on hidden keys: [Nq, Nk]."""
        q, k = _f64(q), _f64(k)
        nq, d = q.shape
        nk = k.shape[0]
        p = np.empty((nq, nk), np.float64)
        _check(self.lib.oracle_softmax(_ptr(q), _ptr(k), nq, nk, d, float(scale),
                                       int(bool(causal)), _ptr(p)), "softmax")
        return p

    def attention_online(self, q, k, v, scale: float, causal: bool = False, block: int = 1,
                         with_lse: bool = False):
        """O by the online recurrence, ``block`` keys at a time."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        *lead, nq, d = q.shape
        nk = k.shape[-2]
        bh = int(np.prod(lead)) if lead else 1
        out = np.empty(q.shape, np.float64)
        lse = np.empty((*lead, nq), np.float64)
        _check(self.lib.oracle_attention_online(_ptr(q), _ptr(k), _ptr(v), bh, nq, nk, d,
                                                float(scale), int(bool(causal)), int(block),
                                                _ptr(out), _ptr(lse)), "attention_online")
        return (out, lse) if with_lse else out

    def online_state(self, q_row, k, v, j0: int, j1: int, scale: float, block: int = 1):
        """Unnormalised state (m, l, o) of one query row over keys [j0, j1) of one slice."""
        q_row, k, v = _f64(q_row), _f64(k), _f64(v)
        d = q_row.shape[-1]
        m, l = ctypes.c_double(), ctypes.c_double()
        o = np.empty(d, np.float64)
        _check(self.lib.oracle_online_state(_ptr(q_row), _ptr(k), _ptr(v), j0, j1, d,
                                            float(scale), int(block), ctypes.byref(m),
                                            ctypes.byref(l), _ptr(o)), "online_state")
        return m.value, l.value, o

    def merge_state(self, s1, s2):
        """Merge two states (m, l, o) over disjoint key sets."""
        (m1, l1, o1), (m2, l2, o2) = s1, s2
        o1, o2 = _f64(o1), _f64(o2)
        d = o1.shape[0]
        m, l = ctypes.c_double(), ctypes.c_double()
        o = np.empty(d, np.float64)
        _check(self.lib.oracle_merge_state(float(m1), float(l1), _ptr(o1), float(m2), float(l2),
                                           _ptr(o2), d, ctypes.byref(m), ctypes.byref(l),
                                           _ptr(o)), "merge_state")
        return m.value, l.value, o

    def attention_backward(self, q, k, v, dout, scale: float, causal: bool = False):
        """(dQ, dK, dV) of O = softmax(scale q k^T) v for the upstream gradient dout."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        *lead, nq, d = q.shape
        nk = k.shape[-2]
        bh = int(np.prod(lead)) if lead else 1
        dq, dk, dv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
        _check(self.lib.oracle_attention_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), bh, nq,
                                                  nk, d, float(scale), int(bool(causal)),
                                                  _ptr(dq), _ptr(dk), _ptr(dv)),
               "attention_backward")
        return dq, dk, dv

    def rope(self, x, cos_t, sin_t, form: int = 0) -> np.ndarray:
        """Rotary embedding of x [..., rows, d] with per-row angle tables cos/sin [rows, d/2]
        (form 0: rotate-half, 1: interleaved pairs). Returns a new array."""
        x = np.array(x, dtype=np.float64, order="C", copy=True)
        c, s_ = _f64(cos_t), _f64(sin_t)
        *lead, rows, d = x.shape
        flat = x.reshape(-1, rows, d)
        for sl in flat:  # the same table for every leading index
            _check(self.lib.oracle_rope(_ptr(sl), _ptr(c), _ptr(s_), rows, d, int(form)), "rope")
        return flat.reshape(x.shape)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())


def default() -> Oracle:
    """The oracle built from ``oracle.c`` in this directory (compiled on first use)."""
    return Oracle(_get())


def attention(*a, **kw):
    return default().attention(*a, **kw)


def attention_rows(*a, **kw):
    return default().attention_rows(*a, **kw)


def softmax(*a, **kw):
    return default().softmax(*a, **kw)


def attention_online(*a, **kw):
    return default().attention_online(*a, **kw)


def online_state(*a, **kw):
    return default().online_state(*a, **kw)


def merge_state(*a, **kw):
    return default().merge_state(*a, **kw)


def rope(*a, **kw):
    return default().rope(*a, **kw)


def attention_backward(*a, **kw):
    return default().attention_backward(*a, **kw)


def num_threads() -> int:
    return default().num_threads()

