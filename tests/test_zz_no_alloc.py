"""hytopk_select_noalloc through the C ABI: the selection for callers that
cannot allocate device memory (a host framework that owns the whole device
memory budget, or a latency-critical path that must not allocate). It runs on
a fixed scratch array the library holds on the device, and must return the
same results as hytopk_select with a caller workspace, call after call.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest

import synthetic_inputs as si

pytestmark = pytest.mark.gpu

REL_TOL = 1e-3  # the score tolerance of the parity tests


def noalloc_fn():
    import exact_top_token_gb300 as hk

    hk.build()
    lib = hk.load()
    f = lib.hytopk_select_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.restype = I
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, I, P, P]
    return hk, f


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(f, t, case, dev):
    import torch

    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    k_top = case["k_top"]
    idx = torch.full((n, k_top), -7, dtype=torch.int32, device=dev)
    sc = torch.full((n, k_top), float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros(8, dtype=torch.int32, device=dev)
    dt = 0 if case["dtype"] == "bf16" else 1
    status = f(ptr(t["q"]), ptr(t["q_scale"]), ptr(t["k"]), ptr(t["k_scale"]), ptr(t["w"]),
               ptr(t["positions"]), n, L, H, d, k_top, dt, ptr(idx), ptr(sc), 0, ptr(st),
               ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    torch.cuda.synchronize()
    return status, idx, sc, st


def test_noalloc_matches_select_on_consecutive_calls():
    import torch

    hk, f = noalloc_fn()
    dev = torch.device("cuda", 0)
    cases = [si.random_case(5000, 100, 32, 128, 300, "bf16", seed=51, positions="random"),
             si.random_case(9000, 70, 64, 128, 256, "e4m3", seed=52, positions="random")]
    for case in cases:  # two calls in a row; the second reuses the first call's array
        t = si.to_torch(case, dev)
        ref_idx, ref_sc, ref_st = hk.select(t["q"], t["k"], t["w"], t["positions"],
                                            case["k_top"], q_scale=t["q_scale"],
                                            k_scale=t["k_scale"], stats=True)
        status, idx, sc, st = call_noalloc(f, t, case, dev)
        assert status == 0, hk.STATUS.get(status, status)
        assert torch.equal(idx, ref_idx)
        a, b = sc.cpu().numpy(), ref_sc.cpu().numpy()
        ok = np.isfinite(b)
        assert np.array_equal(np.isneginf(a), np.isneginf(b))
        s_k = np.abs(np.where(ok, b, 0)).max(axis=1, keepdims=True)
        tol = REL_TOL * np.maximum(np.abs(b), s_k)
        assert np.all(np.abs(a[ok] - b[ok]) <= tol[ok])
        assert hk.read_stats(st) == hk.read_stats(ref_st)


def test_noalloc_rejects_problems_beyond_the_array():
    import torch

    hk, f = noalloc_fn()
    dev = torch.device("cuda", 0)
    n, L, H, d, k_top = 8192, 1 << 20, 64, 128, 2048
    assert hk.select_workspace_size(n, L, H, d, k_top, 0, hk.E4M3) > (32 << 20)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    status = f(fake, fake, fake, fake, fake, fake, n, L, H, d, k_top, 1, fake, None, 0, None,
               ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert status == 3  # HYTOPK_WORKSPACE_TOO_SMALL
