"""CPU oracle for HyTopK exact top-k selection, its threshold filter and
selection replay.

TEST INFRASTRUCTURE ONLY: the plain, slow definition that the GPU library is
checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. It shares no code with
``exact_top_token_gb300`` and never imports it.

The arithmetic lives in ``hytopk_oracle.c`` (plain C, OpenMP over queries,
compiled with ``-ffp-contract=off`` so x86 and Arm hosts give the same bits);
this module only marshals numpy arrays. Each function cites the passage of
the HyScale pages it follows in the C source.

Inputs are a dict as built by ``synthetic_inputs``::

    q [n,H,d] uint16 (bf16 bits) or uint8 (e4m3 codes), q_scale [n,H] f32|None,
    k [L,d] same dtype, k_scale [L] f32|None, w [n,H] f32, positions [n] i32,
    dtype "bf16"|"e4m3", k_top int
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hytopk_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libhytopk_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]

_DTYPES = {"bf16": 0, "e4m3": 1, "e4m3_bf16": 2}
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, seconds)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_bf16_value.restype = ctypes.c_float
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_e4m3_value.restype = ctypes.c_float
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_table.argtypes = [P]
    lib.oracle_sample_count.restype = I64
    lib.oracle_sample_count.argtypes = [I64]
    lib.oracle_threshold_rank.restype = I64
    lib.oracle_threshold_rank.argtypes = [I64, I64]
    lib.oracle_sample_position.restype = I64
    lib.oracle_sample_position.argtypes = [I64, I64, I64]
    lib.oracle_sample_positions.argtypes = [I64, P]
    common = [P, P, P, P, P]
    lib.oracle_row_scores.restype = I32
    lib.oracle_row_scores.argtypes = common + [P, I64, I64, I32, I32, I32, I64, P, I32]
    lib.oracle_select.restype = I32
    lib.oracle_select.argtypes = common + [P, P, I64, I64, I64, I32, I32, I32, I64, P, P, I32]
    lib.oracle_replay.restype = I32
    lib.oracle_replay.argtypes = common + [P, I64, I64, I32, I32, I32, I64, P, P, I32]
    lib.oracle_backward.restype = I32
    lib.oracle_backward.argtypes = common + [P, P, I64, I64, I32, I32, I32, I64,
                                             ctypes.c_double] + [P] * 10 + [I32]
    lib.oracle_filter_sim.restype = I32
    lib.oracle_filter_sim.argtypes = common + [
        P, P, I64, I64, I64, I32, I32, I32, I64, I64, P, P, P, P, P, I32]
    _lib = lib
    return lib


class _use_library:
    """Context manager that points this module at another build of the oracle
    (used by the tests that plant mistakes in a copy of the C source)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _load()
        _lib = None
        real_build = globals()["build"]
        globals()["build"] = lambda force=False: self.path
        try:
            _load()
        finally:
            globals()["build"] = real_build
        return _lib

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(inp):
    q = np.ascontiguousarray(inp["q"])
    k = np.ascontiguousarray(inp["k"])
    n, H, d = q.shape
    L = k.shape[0]
    dt = _DTYPES[inp["dtype"]]
    qs = inp.get("q_scale")
    ks = inp.get("k_scale")
    qs = None if qs is None else np.ascontiguousarray(qs, dtype=np.float32)
    ks = None if ks is None else np.ascontiguousarray(ks, dtype=np.float32)
    w = np.ascontiguousarray(inp["w"], dtype=np.float32)
    pos = np.ascontiguousarray(inp["positions"], dtype=np.int32)
    keep = (q, k, qs, ks, w, pos)
    args = [_ptr(q), _ptr(qs), _ptr(k), _ptr(ks), _ptr(w)]
    return keep, args, pos, n, L, H, d, dt


def _rows(rows):
    if rows is None:
        return None
    return np.ascontiguousarray(rows, dtype=np.int32)


def _check(st, what):
    if st != 0:
        raise ValueError(f"oracle {what} failed with status {st}")


# ---- parameter functions (HyTopK paragraph and worked example) -------------

def sample_count(ctx: int) -> int:
    return int(_load().oracle_sample_count(int(ctx)))


def threshold_rank(ctx: int, k_top: int) -> int:
    return int(_load().oracle_threshold_rank(int(ctx), int(k_top)))


def sample_position(ctx: int, m: int, j: int) -> int:
    return int(_load().oracle_sample_position(int(ctx), int(m), int(j)))


def sample_positions(ctx: int) -> np.ndarray:
    out = np.empty(sample_count(ctx), dtype=np.int64)
    _load().oracle_sample_positions(int(ctx), _ptr(out))
    return out


def e4m3_table() -> np.ndarray:
    out = np.empty(256, dtype=np.float32)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def bf16_value(bits: int) -> float:
    return float(_load().oracle_bf16_value(int(bits)))


# ---- the method -------------------------------------------------------------

def row_scores(inp, t: int, nthreads: int = 0) -> np.ndarray:
    """Every score I[t,s] of query t over its causal prefix, s < ctx(t)."""
    keep, args, pos, n, L, H, d, dt = _prep(inp)
    out = np.empty(int(pos[t]) + 1, dtype=np.float32)
    st = _load().oracle_row_scores(*args, _ptr(pos), n, L, H, d, dt, int(t), _ptr(out), nthreads)
    _check(st, "row_scores")
    return out


def select(inp, rows=None, nthreads: int = 0):
    """Exact top-k (idx int32, scores f32) of the listed queries (default all)."""
    keep, args, pos, n, L, H, d, dt = _prep(inp)
    rows = _rows(rows)
    n_rows = n if rows is None else len(rows)
    k_top = int(inp["k_top"])
    idx = np.empty((n_rows, k_top), dtype=np.int32)
    sc = np.empty((n_rows, k_top), dtype=np.float32)
    st = _load().oracle_select(*args, _ptr(pos), _ptr(rows), n_rows, n, L, H, d, dt, k_top,
                               _ptr(idx), _ptr(sc), nthreads)
    _check(st, "select")
    return idx, sc


def replay(inp, idx, nthreads: int = 0):
    """Selection replay: (scores f32 [n,k], number of out-of-range indices)."""
    keep, args, pos, n, L, H, d, dt = _prep(inp)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k_top = idx.shape[1]
    out = np.empty(idx.shape, dtype=np.float32)
    bad = np.zeros(1, dtype=np.int64)
    st = _load().oracle_replay(*args, _ptr(idx), n, L, H, d, dt, k_top, _ptr(out), _ptr(bad),
                               nthreads)
    _check(st, "replay")
    return out, int(bad[0])


def backward(inp, idx, grad, eps: float = 0.0, nthreads: int = 0):
    """Gradients of sum_{t,j} grad[t,j] * I[t, idx[t,j]] (fp64): a dict with
    dq [n,H,d], dk [L,d], dw [n,H], the matching *_abs (sum of |terms|) and
    *_amb (|terms| whose head dot is within eps*|q||k| of zero), and bad (the
    number of indices outside [0, L) other than -1)."""
    keep, args, pos, n, L, H, d, dt = _prep(inp)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    grad = np.ascontiguousarray(grad, dtype=np.float32)
    k_top = idx.shape[1]
    out = {name: np.zeros(shape, dtype=np.float64) for name, shape in (
        ("dq", (n, H, d)), ("dk", (L, d)), ("dw", (n, H)), ("dq_abs", (n, H, d)),
        ("dk_abs", (L, d)), ("dw_abs", (n, H)), ("dq_amb", (n, H, d)), ("dk_amb", (L, d)),
        ("dw_amb", (n, H)))}
    bad = np.zeros(1, dtype=np.int64)
    st = _load().oracle_backward(
        *args, _ptr(idx), _ptr(grad), n, L, H, d, dt, k_top, float(eps),
        *[_ptr(out[k]) for k in ("dq", "dk", "dw", "dq_abs", "dk_abs", "dw_abs", "dq_amb",
                                 "dk_amb", "dw_amb")], _ptr(bad), nthreads)
    _check(st, "backward")
    out["bad"] = int(bad[0])
    return out


def filter_sim(inp, capacity: int, rows=None, nthreads: int = 0):
    """The HyTopK threshold filter simulated per listed query."""
    keep, args, pos, n, L, H, d, dt = _prep(inp)
    rows = _rows(rows)
    n_rows = n if rows is None else len(rows)
    k_top = int(inp["k_top"])
    T = np.empty(n_rows, dtype=np.float32)
    cnt = np.empty(n_rows, dtype=np.int64)
    M = np.empty(n_rows, dtype=np.int64)
    r = np.empty(n_rows, dtype=np.int64)
    failed = np.empty(n_rows, dtype=np.uint8)
    st = _load().oracle_filter_sim(*args, _ptr(pos), _ptr(rows), n_rows, n, L, H, d, dt, k_top,
                                   int(capacity), _ptr(T), _ptr(cnt), _ptr(M), _ptr(r),
                                   _ptr(failed), nthreads)
    _check(st, "filter_sim")
    return {"T": T, "cnt": cnt, "M": M, "r": r, "failed": failed.astype(bool)}
