"""GPU parity of the key-sharded selection (one HyTopK selection per key range,
then a merge per query): the same indices and scores as hytopk_select, bit for
bit, and the oracle's result, through the C ABI."""
import numpy as np
import pytest

import oracle
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


def run_sharded(hk, case, dev, P, **kw):
    t = si.to_torch(case, dev)
    return hk.select_sharded(t["q"], t["k"], t["w"], t["positions"], case["k_top"], P,
                             q_scale=t["q_scale"], k_scale=t["k_scale"], **kw)


def same_as_select(hk, case, dev, P):
    ref_i, ref_s, _, _ = run_select(hk, case, dev)
    idx, sc, st = run_sharded(hk, case, dev, P, stats=True)
    assert np.array_equal(idx.cpu().numpy(), ref_i.cpu().numpy())
    assert np.array_equal(sc.cpu().numpy(), ref_s.cpu().numpy())
    return idx, sc, hk.read_stats(st)


@pytest.mark.parametrize("P", [1, 2, 3, 7])
def test_tiny_exact_sharded(hk, dev, P):
    case = si.tiny_exact()
    idx, sc, stats = same_as_select(hk, case, dev, P)
    compare(case, np.arange(64), idx.cpu().numpy(), sc.cpu().numpy(), exact=True)
    assert stats["device_status"] == 0 and stats["n_queries"] == 64


@pytest.mark.parametrize("L,n,H,d,k_top,dt,pos,P", [
    (5000, 100, 32, 128, 300, "bf16", "random", 4),   # many queries below a range start
    (20000, 70, 64, 128, 512, "e4m3", "random", 5),
    (3000, 129, 4, 64, 100, "e4m3", "spaced", 2),
    (9001, 33, 16, 64, 256, "bf16", "last", 64),      # ranges of 256 keys, last one short
    (130, 7, 2, 128, 200, "e4m3", "random", 3),       # L < P ranges of a tile: one range
])
def test_random_sharded(hk, dev, L, n, H, d, k_top, dt, pos, P):
    case = si.random_case(L, n, H, d, k_top, dt, seed=L + n + P, positions=pos)
    idx, sc, stats = same_as_select(hk, case, dev, P)
    compare(case, np.arange(n), idx.cpu().numpy(), sc.cpu().numpy())
    assert stats["device_status"] == 0


def test_recovery_small_sharded(hk, dev):
    """The ranges fail and recover on their own; the merged result is exact."""
    case = si.recovery_small(oracle.sample_positions)
    idx, sc, stats = same_as_select(hk, case, dev, 2)
    compare(case, np.arange(len(case["positions"])), idx.cpu().numpy(), sc.cpu().numpy(),
            exact=True)
    assert stats["device_status"] == 0


def test_bad_position_reported_once(hk, dev):
    import torch

    case = si.tiny_exact()
    t = si.to_torch(case, dev)
    pos = t["positions"].clone()
    pos[3] = -5
    pos[10] = case["k"].shape[0]
    idx, sc, st = hk.select_sharded(t["q"], t["k"], t["w"], pos, case["k_top"], 4, stats=True)
    i = idx.cpu().numpy()
    assert (i[3] == -1).all() and (i[10] == -1).all()
    ref, _, _ = hk.select(t["q"], t["k"], t["w"], pos, case["k_top"])
    assert torch.equal(idx, ref)
    assert hk.read_stats(st)["device_status"] == hk.DEV_BAD_POSITION


@pytest.mark.slow
def test_glm_1m_slice_sharded(hk, dev):
    case = si.glm_1m()
    case = si.subset(case, np.arange(len(case["positions"]) - 256, len(case["positions"])))
    idx, sc, stats = same_as_select(hk, case, dev, 4)
    rows = si.sampled_rows(256, 8)
    compare(case, rows, idx.cpu().numpy()[rows], sc.cpu().numpy()[rows])
    assert stats["n_failed"] == 0 and stats["device_status"] == 0
