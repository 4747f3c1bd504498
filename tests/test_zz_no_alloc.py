"""hytopk_select_noalloc through the C ABI: the selection for callers that
cannot allocate device memory (a host framework that owns the whole device
memory budget, or a latency-critical path that must not allocate). It runs on
a fixed scratch array the library holds on the device, and must return the
same results as hytopk_select with a caller workspace, call after call.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import pytest

import synthetic_inputs as si

pytestmark = pytest.mark.gpu

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


def small_recovery_case():
    """Integer data with failing queries that fits the 32 MiB array: 4 mass-tie
    rows overflow their buffers and 4 decoy rows fall short of k, 8 failed
    queries in all, repaired one by one (no fallback). The recovery rows of the
    array carry these rows' state, which the next call must not see."""
    import oracle

    c = si.recovery_stress(oracle.sample_positions, seed=5, L=16384, n=128, H=16, d=64,
                           k_top=256, n_tie_rows=4, tie_values=2, group_rows=32,
                           n_decoy_rows=4, n_decoys=200, decoy_every=13)
    c["name"] = "recovery_noalloc"
    return c


def test_noalloc_matches_select_on_consecutive_calls():
    import torch

    hk, f = noalloc_fn()
    dev = torch.device("cuda", 0)
    clean_bf16 = si.random_case(5000, 100, 32, 128, 300, "bf16", seed=51, positions="random")
    clean_e4m3 = si.random_case(9000, 70, 64, 128, 256, "e4m3", seed=52, positions="random")
    failing = small_recovery_case()
    # calls in a row on the one array: a clean call, one with failed queries, a
    # clean call after it, then the failing one again
    for case in (clean_bf16, failing, clean_e4m3, failing):
        t = si.to_torch(case, dev)
        ref_idx, ref_sc, ref_st = hk.select(t["q"], t["k"], t["w"], t["positions"],
                                            case["k_top"], q_scale=t["q_scale"],
                                            k_scale=t["k_scale"], stats=True)
        status, idx, sc, st = call_noalloc(f, t, case, dev)
        assert status == 0, hk.STATUS.get(status, status)
        # the same kernels on the same inputs: indices and scores bit for bit
        assert torch.equal(idx, ref_idx)
        assert torch.equal(sc.view(torch.int32), ref_sc.view(torch.int32))
        stats = hk.read_stats(st)
        assert stats == hk.read_stats(ref_st)
        if case is failing:
            assert stats["n_failed"] == 8 and stats["fallback_used"] == 0
            assert stats["n_overflow"] == 4 and stats["n_under_k"] == 4
        else:
            assert stats["n_failed"] == 0


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
