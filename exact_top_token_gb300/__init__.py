"""exact_top_token_gb300 -- exact top-k indexer selection without a score
table (HyTopK), selection replay and the two-pass comparison path, for one
NVIDIA GB300 (sm_103a).

This module is a thin ctypes binding over the C ABI declared in
``include/hytopk.h`` (``_build/libhytopk.so``): it checks dtypes, allocates
outputs and workspace with torch on the tensors' device and passes raw
pointers and the current CUDA stream. Every step of the computation runs in
the library's kernels; there is no CPU path. If the compiled library is
missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = ["build", "load", "select", "select_twopass", "replay", "select_workspace_size",
           "select_fallback_chunks",
           "select_sharded", "select_varlen", "replay_varlen", "replay_backward",
           "replay_backward_varlen",
           "twopass_workspace_size", "sample_plan", "HytopkError", "STATUS", "PHASES", "Stats",
           "symbols"]

MAX_RECOVERY_ROWS = 64
PHASES = ("prep", "threshold", "filter", "check", "select", "recover")
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or dtype",
          3: "workspace too small", 4: "CUDA error", 5: "device pointer misaligned"}
DEV_REPLAY_BAD_INDEX = 0x1
DEV_BAD_SCALE = 0x2
DEV_BAD_POSITION = 0x4
DEV_WAIT_TIMEOUT = 0x80000000  # a bounded wait gave up: the call's outputs are undefined
BF16, E4M3, E4M3_BF16 = 0, 1, 2  # E4M3_BF16: e4m3 q (with q_scale), bf16 k

# the C-ABI symbols declared in include/hytopk.h
symbols = ("hytopk_select_workspace_size", "hytopk_select_fallback_chunks", "hytopk_select",
           "hytopk_select_ex", "hytopk_replay",
           "hytopk_twopass_workspace_size", "hytopk_select_twopass", "hytopk_select_noalloc",
           "hytopk_select_sharded_workspace_size", "hytopk_select_sharded",
           "hytopk_replay_backward", "hytopk_select_varlen_workspace_size",
           "hytopk_select_varlen", "hytopk_replay_varlen", "hytopk_replay_grouped",
           "hytopk_replay_backward_varlen", "hytopk_sample_plan",
           "hytopk_status_string", "hytopk_version")


class HytopkError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {STATUS.get(status, status)} (status {status})")
        self.status = status


class Stats(ctypes.Structure):
    _fields_ = [("n_failed", ctypes.c_int32), ("n_overflow", ctypes.c_int32),
                ("n_under_k", ctypes.c_int32), ("fallback_used", ctypes.c_int32),
                ("total_candidates", ctypes.c_int64), ("device_status", ctypes.c_uint32),
                ("n_queries", ctypes.c_int32)]


class SelectOptions(ctypes.Structure):
    _fields_ = [("threshold_override", ctypes.c_void_p), ("phase_events", ctypes.c_void_p),
                ("reverse_schedule", ctypes.c_int), ("reserved", ctypes.c_int)]


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree)."""
    return _build.build(force=force, verbose=verbose)


def load(path: str | None = None):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"the HyTopK CUDA library is not built ({path}); "
                           "call exact_top_token_gb300.build() first")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.hytopk_select_workspace_size.restype = Z
    lib.hytopk_select_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.hytopk_select_fallback_chunks.restype = ctypes.c_int32
    lib.hytopk_select_fallback_chunks.argtypes = [I, I, I, I, I, I, I]
    sel = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, I, P, Z, P]
    lib.hytopk_select.restype = I
    lib.hytopk_select.argtypes = sel + [P]
    lib.hytopk_select_ex.restype = I
    lib.hytopk_select_ex.argtypes = sel + [P, P]
    lib.hytopk_replay.restype = I
    lib.hytopk_replay.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]
    lib.hytopk_replay_grouped.restype = I
    lib.hytopk_replay_grouped.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P]
    lib.hytopk_twopass_workspace_size.restype = Z
    lib.hytopk_twopass_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.hytopk_select_twopass.restype = I
    lib.hytopk_select_twopass.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, Z, P, P]
    lib.hytopk_select_sharded_workspace_size.restype = Z
    lib.hytopk_select_sharded_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
    lib.hytopk_select_sharded.restype = I
    lib.hytopk_select_sharded.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, I, P, Z, P,
                                          P]
    lib.hytopk_replay_backward.restype = I
    lib.hytopk_replay_backward.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, P]
    lib.hytopk_select_varlen_workspace_size.restype = Z
    lib.hytopk_select_varlen_workspace_size.argtypes = [P, P, I, I, I, I, I, I]
    lib.hytopk_select_varlen.restype = I
    lib.hytopk_select_varlen.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, I, P, Z, P,
                                         P]
    lib.hytopk_replay_varlen.restype = I
    lib.hytopk_replay_varlen.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, P]
    lib.hytopk_replay_backward_varlen.restype = I
    lib.hytopk_replay_backward_varlen.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, P, P, P,
                                                  P, P]
    lib.hytopk_sample_plan.restype = ctypes.c_int32
    lib.hytopk_sample_plan.argtypes = [ctypes.c_int64, ctypes.c_int32, P, P]
    lib.hytopk_status_string.restype = ctypes.c_char_p
    lib.hytopk_status_string.argtypes = [I]
    lib.hytopk_version.restype = I
    lib.hytopk_version.argtypes = []
    if path == _build.LIB:
        _lib = lib
    return lib


# ---- argument marshalling -----------------------------------------------------------

def _dtype_code(q, k):
    import torch

    kinds = {torch.bfloat16: BF16, torch.int16: BF16, torch.uint16: BF16,
             torch.float8_e4m3fn: E4M3, torch.uint8: E4M3}
    if q.dtype not in kinds or k.dtype not in kinds:
        raise TypeError("q and k must be bfloat16 (or its 16-bit patterns) or float8_e4m3fn "
                        "(or its 8-bit codes)")
    dq, dk = kinds[q.dtype], kinds[k.dtype]
    if dq == dk:
        return dq
    if dq == E4M3 and dk == BF16:
        return E4M3_BF16
    raise TypeError("bf16 q with e4m3 k is not supported (e4m3 q with bf16 k is)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    import torch

    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensor(name, t, device, dtype=None, shape=None):
    if t is None:
        return
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _common(q, q_scale, k, k_scale, w):
    import torch

    dt = _dtype_code(q, k)
    n, H, d = q.shape
    L = k.shape[0]
    dev = k.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    _check_tensor("q", q, dev)
    _check_tensor("k", k, dev, shape=(L, d))
    _check_tensor("w", w, dev, torch.float32, (n, H))
    _check_tensor("q_scale", q_scale, dev, torch.float32, (n, H))
    _check_tensor("k_scale", k_scale, dev, torch.float32, (L,))
    return dt, n, L, H, d, dev


def sample_plan(ctx: int, k_top: int):
    """(positions, r): the sample positions of a query with ctx visible keys
    and the rank of its threshold among them (host computation in the library)."""
    import numpy as np

    lib = load()
    out = np.zeros(8192, dtype=np.int32)
    r = ctypes.c_int32(0)
    m = lib.hytopk_sample_plan(int(ctx), int(k_top), out.ctypes.data_as(ctypes.c_void_p),
                               ctypes.byref(r))
    return out[:m].copy(), int(r.value)


def select_workspace_size(n, L, H, d, k_top, capacity=0, dtype=BF16) -> int:
    return int(load().hytopk_select_workspace_size(n, L, H, d, k_top, capacity, dtype))


def select_fallback_chunks(n, L, H, d, k_top, capacity=0, dtype=BF16) -> int:
    """Score-table chunks (table writer + read-back launch pairs) of
    hytopk_select's fallback; -1 for invalid arguments."""
    return int(load().hytopk_select_fallback_chunks(n, L, H, d, k_top, capacity, dtype))


def twopass_workspace_size(n, L, H, d, k_top, dtype=BF16, rows_per_chunk=0) -> int:
    return int(load().hytopk_twopass_workspace_size(n, L, H, d, k_top, dtype, rows_per_chunk))


def _workspace(nbytes, device, workspace):
    import torch

    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise HytopkError(3, "workspace")
        return workspace
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if ws.data_ptr() % 256:
        raise RuntimeError("allocator returned a workspace that is not 256-byte aligned")
    return ws


def select(q, k, w, positions, k_top, *, q_scale=None, k_scale=None, capacity=0,
           scores=True, stats=False, workspace=None, threshold_override=None,
           phase_events=None, reverse_schedule=False, out=None, stream=None):
    """Exact top-k key positions per query (HyTopK).

    Returns ``(idx [n,k] int32, scores [n,k] f32 or None, stats or None)``.
    ``stats`` (when requested) is a device int32 tensor holding the
    ``hytopk_stats`` struct; read it with :func:`read_stats`.
    """
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    _check_tensor("positions", positions, dev, torch.int32, (n,))
    if out is not None:
        idx, sc = out
    else:
        idx = torch.empty((n, k_top), dtype=torch.int32, device=dev)
        sc = torch.empty((n, k_top), dtype=torch.float32, device=dev) if scores else None
    need = lib.hytopk_select_workspace_size(n, L, H, d, k_top, capacity, dt)
    if need == 0:
        raise HytopkError(2, "hytopk_select_workspace_size")
    ws = _workspace(need, dev, workspace)
    st = torch.zeros(8, dtype=torch.int32, device=dev) if stats else None
    opts = None
    ev_array = None
    if threshold_override is not None or phase_events is not None or reverse_schedule:
        opts = SelectOptions()
        if threshold_override is not None:
            _check_tensor("threshold_override", threshold_override, dev, torch.float32, (n,))
            opts.threshold_override = threshold_override.data_ptr()
        if phase_events is not None:
            if len(phase_events) != len(PHASES) + 1:
                raise ValueError(f"phase_events needs {len(PHASES) + 1} events")
            ev_array = (ctypes.c_void_p * len(phase_events))(
                *[e.cuda_event for e in phase_events])
            opts.phase_events = ctypes.cast(ev_array, ctypes.c_void_p).value
        opts.reverse_schedule = int(bool(reverse_schedule))
    status = lib.hytopk_select_ex(
        _ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(positions), n, L, H, d,
        k_top, dt, _ptr(idx), _ptr(sc), capacity, _ptr(ws), ws.numel(), _ptr(st),
        ctypes.byref(opts) if opts is not None else None, _stream(dev, stream))
    if status != 0:
        raise HytopkError(status, "hytopk_select")
    return idx, sc, st


def select_sharded_workspace_size(n, L, H, d, k_top, num_shards, capacity=0, dtype=BF16) -> int:
    return int(load().hytopk_select_sharded_workspace_size(n, L, H, d, k_top, capacity, dtype,
                                                           num_shards))


def select_sharded(q, k, w, positions, k_top, num_shards, *, q_scale=None, k_scale=None,
                   capacity=0, scores=True, stats=False, workspace=None, stream=None):
    """Key-sharded exact selection: one HyTopK selection per key range, then a
    merge per query. Same outputs as :func:`select`."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    _check_tensor("positions", positions, dev, torch.int32, (n,))
    idx = torch.empty((n, k_top), dtype=torch.int32, device=dev)
    sc = torch.empty((n, k_top), dtype=torch.float32, device=dev) if scores else None
    need = lib.hytopk_select_sharded_workspace_size(n, L, H, d, k_top, capacity, dt, num_shards)
    if need == 0:
        raise HytopkError(2, "hytopk_select_sharded_workspace_size")
    ws = _workspace(need, dev, workspace)
    st = torch.zeros(8, dtype=torch.int32, device=dev) if stats else None
    status = lib.hytopk_select_sharded(
        _ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(positions), n, L, H, d,
        k_top, dt, num_shards, _ptr(idx), _ptr(sc), capacity, _ptr(ws), ws.numel(), _ptr(st),
        _stream(dev, stream))
    if status != 0:
        raise HytopkError(status, "hytopk_select_sharded")
    return idx, sc, st


def _offsets(cu, name):
    """Host int32 copy of a B+1 offset array (list, numpy or tensor)."""
    import numpy as np

    if hasattr(cu, "cpu"):
        cu = cu.cpu().numpy()
    a = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
    if a.ndim != 1 or a.size < 2:
        raise ValueError(f"{name} must hold B+1 offsets")
    return a


def _cu_ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def select_varlen_workspace_size(cu_q, cu_k, H, d, k_top, capacity=0, dtype=BF16) -> int:
    cq, ck = _offsets(cu_q, "cu_q"), _offsets(cu_k, "cu_k")
    if cq.size != ck.size:
        raise ValueError("cu_q and cu_k must have the same length")
    return int(load().hytopk_select_varlen_workspace_size(_cu_ptr(cq), _cu_ptr(ck), cq.size - 1, H,
                                                          d, k_top, capacity, dtype))


def select_varlen(q, k, w, positions, cu_q, cu_k, k_top, *, q_scale=None, k_scale=None,
                  capacity=0, scores=True, stats=False, workspace=None, stream=None):
    """Packed variable-length batch: sequence b owns queries cu_q[b]:cu_q[b+1]
    and keys cu_k[b]:cu_k[b+1]; positions and returned indices are relative to
    the sequence. Same outputs as :func:`select` over the concatenated rows."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    _check_tensor("positions", positions, dev, torch.int32, (n,))
    cq, ck = _offsets(cu_q, "cu_q"), _offsets(cu_k, "cu_k")
    if cq.size != ck.size or cq[-1] != n or ck[-1] != L:
        raise ValueError("cu_q / cu_k do not match the query and key counts")
    B = cq.size - 1
    idx = torch.empty((n, k_top), dtype=torch.int32, device=dev)
    sc = torch.empty((n, k_top), dtype=torch.float32, device=dev) if scores else None
    need = lib.hytopk_select_varlen_workspace_size(_cu_ptr(cq), _cu_ptr(ck), B, H, d, k_top,
                                                   capacity, dt)
    if need == 0:
        raise HytopkError(2, "hytopk_select_varlen_workspace_size")
    ws = _workspace(need, dev, workspace)
    st = torch.zeros(8, dtype=torch.int32, device=dev) if stats else None
    status = lib.hytopk_select_varlen(
        _ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(positions), _cu_ptr(cq),
        _cu_ptr(ck), B, H, d, k_top, dt, _ptr(idx), _ptr(sc), capacity, _ptr(ws), ws.numel(),
        _ptr(st), _stream(dev, stream))
    if status != 0:
        raise HytopkError(status, "hytopk_select_varlen")
    return idx, sc, st


def replay_varlen(q, k, w, idx, cu_q, cu_k, *, q_scale=None, k_scale=None, status=None,
                  stream=None):
    """Selection replay over a packed variable-length batch (indices relative
    to each query's sequence)."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    k_top = idx.shape[1]
    _check_tensor("idx", idx, dev, torch.int32, (n, k_top))
    cq, ck = _offsets(cu_q, "cu_q"), _offsets(cu_k, "cu_k")
    if cq.size != ck.size or cq[-1] != n or ck[-1] != L:
        raise ValueError("cu_q / cu_k do not match the query and key counts")
    res = torch.empty((n, k_top), dtype=torch.float32, device=dev)
    st = lib.hytopk_replay_varlen(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w),
                                  _ptr(idx), _cu_ptr(cq), _cu_ptr(ck), cq.size - 1, H, d, k_top,
                                  dt, _ptr(res), _ptr(status), _stream(dev, stream))
    if st != 0:
        raise HytopkError(st, "hytopk_replay_varlen")
    return res


def replay_backward_varlen(q, k, w, idx, grad, cu_q, cu_k, *, q_scale=None, k_scale=None,
                           dk=None, status=None, stream=None):
    """Gradients at the selected entries of a packed variable-length batch
    (indices relative to each query's sequence): (dq, dk, dw) as
    :func:`replay_backward`; dk covers all sequences' keys and is added to."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    k_top = idx.shape[1]
    _check_tensor("idx", idx, dev, torch.int32, (n, k_top))
    _check_tensor("grad", grad, dev, torch.float32, (n, k_top))
    cq, ck = _offsets(cu_q, "cu_q"), _offsets(cu_k, "cu_k")
    if cq.size != ck.size or cq[-1] != n or ck[-1] != L:
        raise ValueError("cu_q / cu_k do not match the query and key counts")
    dq = torch.empty((n, H, d), dtype=torch.float32, device=dev)
    dw = torch.empty((n, H), dtype=torch.float32, device=dev)
    if dk is None:
        dk = torch.zeros((L, d), dtype=torch.float32, device=dev)
    else:
        _check_tensor("dk", dk, dev, torch.float32, (L, d))
    st = lib.hytopk_replay_backward_varlen(
        _ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(idx), _ptr(grad),
        _cu_ptr(cq), _cu_ptr(ck), cq.size - 1, H, d, k_top, dt, _ptr(dq), _ptr(dk), _ptr(dw),
        _ptr(status), _stream(dev, stream))
    if st != 0:
        raise HytopkError(st, "hytopk_replay_backward_varlen")
    return dq, dk, dw


def read_stats(st) -> dict:
    """Decode a stats tensor returned by :func:`select` (synchronises)."""
    raw = st.cpu().numpy().tobytes()
    s = Stats.from_buffer_copy(raw[:ctypes.sizeof(Stats)])
    return {name: getattr(s, name) for name, _ in Stats._fields_}


def replay(q, k, w, idx, *, q_scale=None, k_scale=None, status=None, out=None, group=1,
           stream=None):
    """Selection replay: scores [n,k] of the stored indices idx [n,k].
    ``group=2`` replays adjacent query pairs over the union of their indices
    (same result)."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    k_top = idx.shape[1]
    _check_tensor("idx", idx, dev, torch.int32, (n, k_top))
    res = out if out is not None else torch.empty((n, k_top), dtype=torch.float32, device=dev)
    if group == 1:
        st = lib.hytopk_replay(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w), _ptr(idx),
                               n, L, H, d, k_top, dt, _ptr(res), _ptr(status),
                               _stream(dev, stream))
    else:
        st = lib.hytopk_replay_grouped(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w),
                                       _ptr(idx), n, L, H, d, k_top, dt, group, _ptr(res),
                                       _ptr(status), _stream(dev, stream))
    if st != 0:
        raise HytopkError(st, "hytopk_replay")
    return res


def replay_backward(q, k, w, idx, grad, *, q_scale=None, k_scale=None, dk=None, status=None,
                    stream=None):
    """Gradients at the selected entries: returns (dq [n,H,d], dk [L,d], dw [n,H]),
    fp32. ``dk`` is added to when given (else a zeroed tensor is used)."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    k_top = idx.shape[1]
    _check_tensor("idx", idx, dev, torch.int32, (n, k_top))
    _check_tensor("grad", grad, dev, torch.float32, (n, k_top))
    dq = torch.empty((n, H, d), dtype=torch.float32, device=dev)
    dw = torch.empty((n, H), dtype=torch.float32, device=dev)
    if dk is None:
        dk = torch.zeros((L, d), dtype=torch.float32, device=dev)
    else:
        _check_tensor("dk", dk, dev, torch.float32, (L, d))
    st = lib.hytopk_replay_backward(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w),
                                    _ptr(idx), _ptr(grad), n, L, H, d, k_top, dt, _ptr(dq),
                                    _ptr(dk), _ptr(dw), _ptr(status), _stream(dev, stream))
    if st != 0:
        raise HytopkError(st, "hytopk_replay_backward")
    return dq, dk, dw


def select_twopass(q, k, w, positions, k_top, *, q_scale=None, k_scale=None, rows_per_chunk=0,
                   scores=True, workspace=None, status=None, stream=None):
    """The conventional materialise-then-top-k path (same outputs as select)."""
    import torch

    lib = load()
    dt, n, L, H, d, dev = _common(q, q_scale, k, k_scale, w)
    _check_tensor("positions", positions, dev, torch.int32, (n,))
    idx = torch.empty((n, k_top), dtype=torch.int32, device=dev)
    sc = torch.empty((n, k_top), dtype=torch.float32, device=dev) if scores else None
    # with a caller workspace the library picks the largest chunk that fits
    need = lib.hytopk_twopass_workspace_size(n, L, H, d, k_top, dt,
                                             1 if workspace is not None else rows_per_chunk)
    if need == 0:
        raise HytopkError(2, "hytopk_twopass_workspace_size")
    ws = _workspace(need, dev, workspace)
    st = lib.hytopk_select_twopass(_ptr(q), _ptr(q_scale), _ptr(k), _ptr(k_scale), _ptr(w),
                                   _ptr(positions), n, L, H, d, k_top, dt, _ptr(idx), _ptr(sc),
                                   _ptr(ws), ws.numel(), _ptr(status), _stream(dev, stream))
    if st != 0:
        raise HytopkError(st, "hytopk_select_twopass")
    return idx, sc
