"""GPU parity of the grouped replay (adjacent queries 2i, 2i+1 replayed over
the union of their index lists): bit for bit the scores, -inf / NaN entries
and status bits of the single-query replay, and the oracle's scores, through
the C ABI."""
import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from parity import replay_tolerance

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


def overlapping_indices(L, n, k_top, share, seed):
    """Row 2i: k distinct keys; row 2i+1: a fraction `share` of row 2i's keys
    (in another order) plus fresh keys."""
    g = si.rng_for(seed)
    idx = np.empty((n, k_top), np.int32)
    for t in range(0, n, 2):
        a = g.choice(L, size=k_top, replace=False)
        idx[t] = a
        if t + 1 < n:
            keep = g.permutation(a)[: int(share * k_top)]
            fresh = np.setdiff1d(g.choice(L, size=min(L, 3 * k_top), replace=False), keep)
            b = np.concatenate([keep, fresh[: k_top - len(keep)]])
            idx[t + 1] = g.permutation(b)
    return idx


def both(hk, dev, case, idx):
    import torch

    t = si.to_torch(case, dev)
    it = torch.from_numpy(np.ascontiguousarray(idx)).to(dev)
    s1 = torch.zeros(1, dtype=torch.int32, device=dev)
    s2 = torch.zeros(1, dtype=torch.int32, device=dev)
    r1 = hk.replay(t["q"], t["k"], t["w"], it, q_scale=t["q_scale"], k_scale=t["k_scale"],
                   status=s1)
    r2 = hk.replay(t["q"], t["k"], t["w"], it, q_scale=t["q_scale"], k_scale=t["k_scale"],
                   status=s2, group=2)
    a, b = r1.cpu().numpy(), r2.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))  # NaN payloads included
    assert int(s1.item()) == int(s2.item())
    return b, int(s2.item())


@pytest.mark.parametrize("H,d,dt", [(1, 64, "bf16"), (2, 128, "e4m3"), (4, 64, "bf16"),
                                    (8, 32, "bf16"), (16, 128, "bf16"), (32, 64, "e4m3"),
                                    (64, 128, "e4m3"), (64, 256, "e4m3"), (16, 64, "e4m3_bf16"),
                                    (128, 64, "bf16")])
def test_grouped_equals_single(hk, dev, H, d, dt):
    L, n, k_top = 3000, 37, 300  # odd n: the last query is alone
    case = si.random_case(L, n, H, d, k_top, dt, seed=H + d, positions="last")
    idx = overlapping_indices(L, n, k_top, 0.7, seed=5 + H)
    sc, st = both(hk, dev, case, idx)
    assert st == 0
    ref, bad = oracle.replay(case, idx)
    assert bad == 0
    assert (np.abs(sc.astype(np.float64) - ref) <= replay_tolerance(case, idx, ref)).all()


def test_grouped_exact_integer_data(hk, dev):
    case = si.tiny_exact()
    idx = overlapping_indices(4096, 64, 256, 0.9, seed=3)
    sc, st = both(hk, dev, case, idx)
    ref, bad = oracle.replay(case, idx)
    assert st == 0 and bad == 0
    assert np.array_equal(sc, ref)


@pytest.mark.parametrize("share", [0.0, 1.0])
def test_grouped_disjoint_and_identical_lists(hk, dev, share):
    case = si.random_case(20000, 16, 64, 128, 2048, "e4m3", seed=7)
    idx = overlapping_indices(20000, 16, 2048, share, seed=8)
    both(hk, dev, case, idx)


def test_grouped_empty_bad_and_repeated_entries(hk, dev):
    """-1 entries give -inf, other out-of-range entries NaN and a status bit; a
    key listed twice in one row is scored at both entries."""
    case = si.random_case(1000, 10, 16, 64, 64, "bf16", seed=9)
    idx = overlapping_indices(1000, 10, 64, 0.5, seed=10)
    idx[0, 3] = -1
    idx[1, :5] = -1
    idx[2, 7] = 1000
    idx[3, 0] = -9
    idx[4, 10] = idx[4, 11] = idx[4, 12]     # the same key three times in one row
    idx[5, 1] = idx[4, 12]                    # and in the neighbour
    idx[9, :] = -1                            # a row with nothing to gather
    sc, st = both(hk, dev, case, idx)
    assert st == 1  # HYTOPK_DEV_REPLAY_BAD_INDEX
    assert np.isneginf(sc[0, 3]) and np.isneginf(sc[1, :5]).all() and np.isneginf(sc[9]).all()
    assert np.isnan(sc[2, 7]) and np.isnan(sc[3, 0])
    assert sc[4, 10] == sc[4, 11] == sc[4, 12]
    ref, bad = oracle.replay(case, idx)
    assert bad == 2
    ok = (idx >= 0) & (idx < 1000)
    tol = replay_tolerance(case, idx, ref)
    assert (np.abs(sc[ok].astype(np.float64) - ref[ok]) <= tol[ok]).all()


def test_grouped_k_above_pairing_limit_runs_single(hk, dev):
    case = si.random_case(9000, 6, 16, 64, 4096, "bf16", seed=11)
    idx = overlapping_indices(9000, 6, 4096, 0.8, seed=12)
    both(hk, dev, case, idx)


def test_grouped_on_the_selection(hk, dev):
    """Replay of the selection's own indices, grouped, returns its scores."""
    case = si.mixed_contexts()
    case = si.subset(case, np.arange(512, 768))
    t = si.to_torch(case, dev)
    idx, sc, _ = hk.select(t["q"], t["k"], t["w"], t["positions"], case["k_top"],
                           q_scale=t["q_scale"], k_scale=t["k_scale"])
    rs = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"],
                   group=2)
    a, b = rs.cpu().numpy(), sc.cpu().numpy()
    keep = idx.cpu().numpy() >= 0
    assert np.array_equal(a[keep], b[keep]) and np.isneginf(a[~keep]).all()
