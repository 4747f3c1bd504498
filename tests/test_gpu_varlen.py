"""GPU parity of packed variable-length batches through the C ABI: every
sequence's rows equal hytopk_select run on that sequence alone (bit for bit)
and the oracle's result; replay over the packed batch returns the selected
scores."""
import numpy as np
import pytest

import synthetic_inputs as si
from parity import compare, run_select

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    import exact_top_token_gb300 as hk

    hk.build()
    hk.load()
    return hk


@pytest.fixture(scope="module")
def dev():
    import torch

    return torch.device("cuda", 0)


def sequences(specs, H, d, k_top, dt, kind="normal"):
    """specs: (L_b, n_b, positions) per sequence."""
    return [si.random_case(L, n, H, d, k_top, dt, seed=1000 + 7 * b + L, positions=pos, kind=kind)
            for b, (L, n, pos) in enumerate(specs)]


def check_varlen(hk, dev, cases, exact=False):
    packed, cu_q, cu_k = si.pack_varlen(cases)
    t = si.to_torch(packed, dev)
    idx, sc, st = hk.select_varlen(t["q"], t["k"], t["w"], t["positions"], cu_q, cu_k,
                                   packed["k_top"], q_scale=t["q_scale"], k_scale=t["k_scale"],
                                   stats=True)
    idx_h, sc_h = idx.cpu().numpy(), sc.cpu().numpy()
    n_fail = 0
    for b, c in enumerate(cases):
        lo, hi = cu_q[b], cu_q[b + 1]
        if hi == lo:
            continue
        ref_i, ref_s, st_b, _ = run_select(hk, c, dev, stats=True)
        assert np.array_equal(idx_h[lo:hi], ref_i.cpu().numpy()), f"sequence {b}"
        assert np.array_equal(sc_h[lo:hi], ref_s.cpu().numpy()), f"sequence {b}"
        n_fail += hk.read_stats(st_b)["n_failed"]
        rows = si.sampled_rows(hi - lo, 24)
        compare(c, rows, idx_h[lo:hi][rows], sc_h[lo:hi][rows], exact=exact)
    stats = hk.read_stats(st)
    assert stats["n_queries"] == cu_q[-1] and stats["device_status"] == 0
    assert stats["n_failed"] == n_fail
    # replay of the packed selection gives back its scores
    rep = hk.replay_varlen(t["q"], t["k"], t["w"], idx, cu_q, cu_k, q_scale=t["q_scale"],
                           k_scale=t["k_scale"])
    r = rep.cpu().numpy()
    keep = idx_h >= 0
    assert np.array_equal(r[keep], sc_h[keep])
    assert np.all(np.isneginf(r[~keep]))
    return idx_h, sc_h


def test_varlen_exact_mixed_lengths(hk, dev):
    # an empty sequence, one shorter than k_top, one spanning many key tiles
    cases = sequences([(3000, 40, "spaced"), (500, 0, "last"), (100, 9, "last"),
                       (9000, 70, "random")], H=4, d=64, k_top=256, dt="bf16", kind="int")
    check_varlen(hk, dev, cases, exact=True)


@pytest.mark.parametrize("dt,H,d", [("bf16", 32, 128), ("e4m3", 64, 128), ("e4m3_bf16", 16, 64),
                                    ("bf16", 1, 32), ("e4m3", 2, 256)])
def test_varlen_random(hk, dev, dt, H, d):
    # odd key counts and H < 4 put k_scale and w at offsets that are not 16-byte aligned
    cases = sequences([(5001, 33, "random"), (777, 13, "last"), (20003, 65, "spaced")],
                      H=H, d=d, k_top=512, dt=dt)
    check_varlen(hk, dev, cases)


def test_varlen_single_sequence_is_select(hk, dev):
    case = si.tiny_exact()
    check_varlen(hk, dev, [case], exact=True)


def test_varlen_all_empty(hk, dev):
    import torch

    cases = sequences([(300, 0, "last"), (200, 0, "last")], H=4, d=64, k_top=16, dt="bf16")
    packed, cu_q, cu_k = si.pack_varlen(cases)
    t = si.to_torch(packed, dev)
    idx, sc, st = hk.select_varlen(t["q"], t["k"], t["w"], t["positions"], cu_q, cu_k, 16,
                                   stats=True)
    assert idx.shape == (0, 16)
    assert hk.read_stats(st)["n_queries"] == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("dt,H,d", [("bf16", 16, 64), ("e4m3", 4, 128)])
def test_backward_varlen_exact(hk, dev, dt, H, d):
    """Gradients of a packed batch on integer data: each sequence's dq, dw and
    its rows of dk equal the oracle's for that sequence."""
    import oracle
    import torch

    specs = [(2000, 20, "spaced"), (600, 0, "last"), (3000, 31, "random")]
    cases = [si.random_case(L, n, H, d, 128, "bf16", seed=300 + b, positions=pos, kind="int")
             for b, (L, n, pos) in enumerate(specs)]
    if dt == "e4m3":  # the same integer values as e4m3 codes with power-of-two scales
        cases = [dict(c, dtype="e4m3",
                      q=torch.from_numpy(si.bf16_bits_to_f32(c["q"])).to(torch.float8_e4m3fn)
                      .view(torch.uint8).numpy(),
                      k=torch.from_numpy(si.bf16_bits_to_f32(c["k"])).to(torch.float8_e4m3fn)
                      .view(torch.uint8).numpy(),
                      q_scale=np.full(c["w"].shape, 0.5, np.float32),
                      k_scale=np.full(c["k"].shape[0], 2.0, np.float32)) for c in cases]
    g = si.rng_for(77)
    idxs, grads = [], []
    for c in cases:
        n, L = len(c["positions"]), c["k"].shape[0]
        rows = [g.choice(L, size=128, replace=False) for _ in range(n)]
        idxs.append(np.array(rows, dtype=np.int32).reshape(n, 128))
        grads.append(g.integers(-3, 4, size=(n, 128)).astype(np.float32))
    packed, cu_q, cu_k = si.pack_varlen(cases)
    t = si.to_torch(packed, dev)
    idx = torch.from_numpy(np.concatenate(idxs)).to(dev)
    grad = torch.from_numpy(np.concatenate(grads)).to(dev)
    dq, dk, dw = hk.replay_backward_varlen(t["q"], t["k"], t["w"], idx, grad, cu_q, cu_k,
                                           q_scale=t["q_scale"], k_scale=t["k_scale"])
    dq, dk, dw = dq.cpu().numpy(), dk.cpu().numpy(), dw.cpu().numpy()
    for b, c in enumerate(cases):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 > q0:
            ref = oracle.backward(c, idxs[b], grads[b])
            assert np.array_equal(dq[q0:q1], ref["dq"].astype(np.float32)), f"dq {b}"
            assert np.array_equal(dw[q0:q1], ref["dw"].astype(np.float32)), f"dw {b}"
            assert np.array_equal(dk[k0:k1], ref["dk"].astype(np.float32)), f"dk {b}"
        else:
            assert (dk[k0:k1] == 0).all()
