"""Pins for the CPU oracle: checks against what the HyScale pages and plain
mathematics fix, not against the oracle's own formula.

* closed forms printed in the explainer's worked GLM-5.1 example (golden file);
* the e4m3 / bf16 decoders against torch's format conversions on every code;
* exact brute force in Python integers on tiny integer-valued problems;
* textbook special cases (H=1, w=1, d=1 reduces to a sort of ReLU(q*k));
* invariants: key permutation, all-equal scores, ctx <= k padding, the
  threshold certificate (cnt >= k implies the true top-k are all candidates);
* fp64 recomputation bounds the oracle's fp32 rounding on random inputs.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def int_case(L, n, H, d, k_top, seed, positions=None, lo=-3, hi=3, wlo=1, whi=2, dtype="bf16",
             pow2_scales=False):
    """Integer-valued problem plus its exact integer arrays for brute force."""
    g = np.random.Generator(np.random.PCG64(1000 + seed))
    qi = g.integers(lo, hi + 1, size=(n, H, d))
    ki = g.integers(lo, hi + 1, size=(L, d))
    wi = g.integers(wlo, whi + 1, size=(n, H))
    pos = (g.integers(0, L, size=n) if positions is None else np.asarray(positions)).astype(np.int32)
    case = {"w": wi.astype(np.float32), "positions": pos, "k_top": k_top, "dtype": dtype,
            "name": "int"}
    exact = {"q": [[[Fraction(int(v)) for v in row] for row in head] for head in qi],
             "k": [[Fraction(int(v)) for v in row] for row in ki], "w": wi}
    if dtype == "bf16":
        case.update(q=si.f32_to_bf16_bits(qi.astype(np.float32)), q_scale=None,
                    k=si.f32_to_bf16_bits(ki.astype(np.float32)), k_scale=None)
    else:
        import torch

        def codes(x):
            return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(
                torch.uint8).numpy().copy()

        qs = np.ones((n, H), np.float32)
        ks = np.ones(L, np.float32)
        if pow2_scales:
            qs = np.ldexp(1.0, g.integers(-3, 4, size=(n, H))).astype(np.float32)
            ks = np.ldexp(1.0, g.integers(-3, 4, size=L)).astype(np.float32)
        case.update(q=codes(qi), q_scale=qs, k=codes(ki), k_scale=ks)
        exact["q"] = [[[Fraction(int(v)) * Fraction(float(qs[t, h])) for v in qi[t, h]]
                       for h in range(H)] for t in range(n)]
        exact["k"] = [[Fraction(int(v)) * Fraction(float(ks[s])) for v in ki[s]] for s in range(L)]
    return case, exact


def brute(exact, case):
    """Exact scores and (score desc, position asc) order, in rationals."""
    out = []
    q, k, w = exact["q"], exact["k"], exact["w"]
    H = len(q[0])
    for t, p in enumerate(case["positions"]):
        ctx = int(p) + 1
        sc = []
        for s in range(ctx):
            tot = Fraction(0)
            for h in range(H):
                dot = sum(a * b for a, b in zip(q[t][h], k[s]))
                tot += int(w[t, h]) * max(Fraction(0), dot)
            sc.append(tot)
        order = sorted(range(ctx), key=lambda s: (-sc[s], s))
        out.append((sc, order))
    return out


# ---- closed forms of the worked example -------------------------------------

def test_worked_example_closed_forms():
    g = json.load(open(os.path.join(GOLDEN, "glm51_worked_example.json")))
    pr = g["printed"]
    L, n, k = g["L"], g["n"], g["k_top"]
    M = oracle.sample_count(L)
    r = oracle.threshold_rank(L, k)
    assert M == pr["sample_count_M"]
    assert L // M == pr["keys_per_sample"]
    assert r == pr["threshold_rank_r"]
    assert r * (L // M) == pr["keys_represented_by_threshold"]
    assert r * (L // M) == pr["threshold_keys_over_k"] * k
    table = n * L * g["score_bytes"]
    idx = n * k * g["index_bytes"]
    assert table == pr["score_table_GiB"] * 2**30
    assert idx == pr["indices_MiB"] * 2**20
    assert table // idx == pr["table_over_indices"]
    assert round(100 * k / L, 1) == pr["kept_percent_rounded"]
    assert L // k == pr["replay_fewer_scoring_ops"]
    # the sample spacing at the 1M setting is exactly 128 keys, starting at key 0
    sp = oracle.sample_positions(L)
    assert sp[0] == 0 and np.all(np.diff(sp) == 128)


@pytest.mark.parametrize("ctx", [4097, 65536, 200000, 524288, 600000, 1048576, 1 << 24])
def test_sample_count_within_printed_bounds(ctx):
    g = json.load(open(os.path.join(GOLDEN, "glm51_worked_example.json")))["sample_count_bounds"]
    M = oracle.sample_count(ctx)
    assert g["low"] <= M <= g["high"]
    sp = oracle.sample_positions(ctx)
    assert len(sp) == M and sp[0] == 0 and sp[-1] < ctx
    assert np.all(np.diff(sp) >= 1)  # distinct, increasing
    gaps = np.diff(np.append(sp, ctx))
    assert gaps.max() - gaps.min() <= 1  # evenly spaced
    if 4096 < M < 8192:
        # each sample stands for at least the worked example's 128 keys
        assert ctx / M >= 128 and ctx / (M + 1) < 128
    r = oracle.threshold_rank(ctx, 2048)
    if ctx >= 3 * 2048:
        # the threshold sample stands for about 3k keys: r*ctx/M in [3k, 3k + ctx/M)
        assert 3 * 2048 <= r * ctx / M < 3 * 2048 + ctx / M
    else:
        assert r == M  # fewer than 3k keys: the rank clamps to the sample count


def test_sample_count_small_contexts():
    for ctx in [1, 2, 100, 2048, 4095, 4096]:
        assert oracle.sample_count(ctx) == ctx  # every key is a sample
        assert list(oracle.sample_positions(ctx)) == list(range(ctx))
    # between k and 3k keys the rank clamps to M: the threshold is the smallest sample
    assert oracle.threshold_rank(3000, 2048) == 3000
    assert oracle.threshold_rank(4096, 256) == 768


# ---- element decoding --------------------------------------------------------

def test_e4m3_decode_every_code():
    import torch

    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = oracle.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0**-9 and got[0x08] == 2.0**-6


def test_bf16_decode():
    import torch

    g = np.random.Generator(np.random.PCG64(5))
    bits = g.integers(0, 1 << 16, size=4000, dtype=np.int64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits], dtype=np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])


# ---- exact brute force ---------------------------------------------------------

@pytest.mark.parametrize("L,n,H,d,k_top,seed", [
    (16, 6, 1, 1, 4, 0), (40, 8, 2, 3, 7, 1), (64, 10, 4, 8, 16, 2), (33, 5, 3, 5, 40, 3),
    (64, 12, 8, 16, 5, 4), (50, 6, 16, 4, 50, 5)])
def test_select_matches_exact_bruteforce(L, n, H, d, k_top, seed):
    case, exact = int_case(L, n, H, d, k_top, seed)
    idx, sc = oracle.select(case)
    for t, (scores, order) in enumerate(brute(exact, case)):
        want = order[:k_top] + [-1] * max(0, k_top - len(order))
        assert list(idx[t]) == want
        for j, s in enumerate(want):
            if s < 0:
                assert sc[t, j] == -np.inf
            else:
                assert Fraction(float(sc[t, j])) == scores[s]


def test_select_e4m3_scales_exact():
    # power-of-two scales keep every product exact; a dropped or misplaced scale fails
    case, exact = int_case(48, 8, 4, 6, 9, 7, dtype="e4m3", pow2_scales=True)
    idx, sc = oracle.select(case)
    for t, (scores, order) in enumerate(brute(exact, case)):
        want = order[:9] + [-1] * max(0, 9 - len(order))
        assert list(idx[t]) == want
        for j, s in enumerate(want):
            if s >= 0:
                assert Fraction(float(sc[t, j])) == scores[s]


def test_negative_weights_and_relu():
    # weights of both signs: ReLU must clip each head before the weighted sum
    case, exact = int_case(30, 6, 3, 4, 10, 8, wlo=-2, whi=2)
    idx, sc = oracle.select(case)
    for t, (scores, order) in enumerate(brute(exact, case)):
        want = order[:10] + [-1] * max(0, 10 - len(order))
        assert list(idx[t]) == want


def test_scalar_textbook_case():
    # H=1, w=1, d=1: the score is ReLU(q*k); top-k is Python's sort of it
    g = np.random.Generator(np.random.PCG64(9))
    L = 64
    kv = g.integers(-20, 21, size=L)
    for qv in (3, -2, 0):
        case = {"q": si.f32_to_bf16_bits(np.full((1, 1, 1), qv, np.float32)), "q_scale": None,
                "k": si.f32_to_bf16_bits(kv.reshape(L, 1).astype(np.float32)), "k_scale": None,
                "w": np.ones((1, 1), np.float32), "positions": np.array([L - 1], np.int32),
                "k_top": 10, "dtype": "bf16"}
        idx, sc = oracle.select(case)
        relu = [max(0, qv * int(x)) for x in kv]
        assert list(idx[0]) == sorted(range(L), key=lambda s: (-relu[s], s))[:10]


def test_all_equal_scores_and_short_context():
    n, L, H, d = 3, 20, 2, 4
    case = {"q": si.f32_to_bf16_bits(np.ones((n, H, d), np.float32)), "q_scale": None,
            "k": si.f32_to_bf16_bits(np.ones((L, d), np.float32)), "k_scale": None,
            "w": np.ones((n, H), np.float32), "positions": np.array([19, 5, 0], np.int32),
            "k_top": 8, "dtype": "bf16"}
    idx, sc = oracle.select(case)
    assert list(idx[0]) == list(range(8))
    assert list(idx[1]) == list(range(6)) + [-1, -1]
    assert list(idx[2]) == [0] + [-1] * 7
    assert np.all(sc[1, :6] == 8.0) and np.all(sc[1, 6:] == -np.inf)


def test_key_permutation_permutes_output():
    case = si.random_case(300, 4, 4, 16, 20, "bf16", seed=11, positions=np.full(4, 299))
    idx, sc = oracle.select(case)
    perm = np.random.Generator(np.random.PCG64(12)).permutation(300)
    moved = dict(case)
    moved["k"] = case["k"][perm]  # new key j is old key perm[j]
    idx2, sc2 = oracle.select(moved)
    inv = np.argsort(perm)
    # distinct scores (checked) -> the same keys, renamed
    assert all(len(set(row)) == len(row) for row in sc.tolist())
    assert np.array_equal(perm[idx2], idx)
    assert np.array_equal(sc2, sc)
    assert np.array_equal(inv[idx], idx2)


def test_fp32_rounding_within_bound_of_fp64():
    import torch

    case = si.random_case(2000, 6, 8, 64, 50, "bf16", seed=13, positions="random")
    q = torch.from_numpy(case["q"].view(np.int16)).view(torch.bfloat16).double().numpy()
    k = torch.from_numpy(case["k"].view(np.int16)).view(torch.bfloat16).double().numpy()
    w = case["w"].astype(np.float64)
    for t in range(6):
        got = oracle.row_scores(case, t).astype(np.float64)
        ctx = int(case["positions"][t]) + 1
        dots = q[t] @ k[:ctx].T  # [H, ctx]
        ref = (w[t][:, None] * np.maximum(dots, 0)).sum(0)
        bound = 1e-5 * (np.abs(w[t])[:, None] * np.abs(q[t]) @ np.abs(k[:ctx]).T).sum(0) + 1e-30
        assert np.all(np.abs(got - ref) <= bound)


def test_e4m3_fp32_rounding_within_bound_of_fp64():
    case = si.random_case(1500, 4, 8, 128, 30, "e4m3", seed=14, positions="random")
    tab = oracle.e4m3_table().astype(np.float64)
    q = tab[case["q"]] * case["q_scale"][..., None].astype(np.float64)
    k = tab[case["k"]] * case["k_scale"][:, None].astype(np.float64)
    w = case["w"].astype(np.float64)
    for t in range(4):
        got = oracle.row_scores(case, t).astype(np.float64)
        ctx = int(case["positions"][t]) + 1
        ref = (w[t][:, None] * np.maximum(q[t] @ k[:ctx].T, 0)).sum(0)
        bound = 1e-5 * (np.abs(w[t])[:, None] * (np.abs(q[t]) @ np.abs(k[:ctx]).T)).sum(0)
        assert np.all(np.abs(got - ref) <= bound + 1e-30)


# ---- threshold filter ----------------------------------------------------------

def test_filter_full_sampling_threshold_is_exact_rank():
    # tiny_exact: ctx <= 4096, so every key is a sample and T is the exact r-th best
    case = si.tiny_exact()
    fs = oracle.filter_sim(case, capacity=8 * 256)
    for t in range(0, 64, 9):
        row = oracle.row_scores(case, t)
        ctx = len(row)
        assert fs["M"][t] == ctx and fs["r"][t] == 768
        T = np.sort(row)[::-1][767]
        assert fs["T"][t] == T
        assert fs["cnt"][t] == int((row >= T).sum())
        assert not fs["failed"][t]


def test_filter_threshold_rank_on_distinct_scores():
    # ctx <= 4096: all keys are samples, scores are distinct, so T must be exactly the
    # r-th best score and exactly r keys (r = 3k here) pass the filter
    case = si.random_case(3000, 8, 16, 32, 100, "bf16", seed=17,
                          positions=np.array([2999, 2500, 1800, 900, 400, 301, 150, 99]))
    fs = oracle.filter_sim(case, capacity=10**6)
    for t in range(8):
        row = oracle.row_scores(case, t)
        ctx = len(row)
        if ctx <= 100:
            assert fs["T"][t] == -np.inf and fs["cnt"][t] == ctx and not fs["failed"][t]
            continue
        r = min(ctx, 300)
        desc = np.sort(row)[::-1]
        if r < ctx:
            assert desc[r - 1] > desc[r]  # the rank is unambiguous for this seed
        assert fs["r"][t] == r and fs["M"][t] == ctx
        assert fs["T"][t] == desc[r - 1]
        assert fs["cnt"][t] == r


def test_filter_certificate_holds():
    # whenever cnt >= k (and no overflow), every true top-k key passes the threshold
    case = si.random_case(9000, 12, 4, 32, 40, "bf16", seed=15, positions="random")
    fs = oracle.filter_sim(case, capacity=10**9)
    idx, sc = oracle.select(case)
    for t in range(12):
        ctx = int(case["positions"][t]) + 1
        if ctx <= 40:
            continue
        if fs["cnt"][t] >= 40:
            assert np.all(sc[t] >= fs["T"][t])
            assert not fs["failed"][t]
        else:
            assert fs["failed"][t]


def test_recovery_small_flags_exact_rows():
    case = si.recovery_small(oracle.sample_positions)
    C = 8 * case["k_top"]
    fs = oracle.filter_sim(case, capacity=C)
    failed = set(np.flatnonzero(fs["failed"]).tolist())
    ties = set(case["tie_rows"].tolist())
    decoys = set(case["decoy_rows"].tolist())
    assert failed == ties | decoys
    assert all(fs["cnt"][t] > C for t in ties)
    assert all(fs["cnt"][t] < case["k_top"] for t in decoys)
    assert len(failed) <= 64
    # a spike row's exact top-k is its group's k spikes (all above background)
    t = max(ties) + 1
    idx, sc = oracle.select(case, rows=[t])
    assert np.all(sc[0] >= 256) and len(set(idx[0].tolist())) == case["k_top"]


# ---- replay -------------------------------------------------------------------

def test_replay_equals_selected_scores_and_flags_bad_indices():
    case = si.random_case(700, 9, 4, 32, 64, "e4m3", seed=16, positions="random")
    idx, sc = oracle.select(case)
    rs, bad = oracle.replay(case, idx)
    assert bad == 0
    assert np.array_equal(rs, sc)  # bitwise: same score function
    idx2 = idx.copy()
    idx2[0, 0] = 700
    idx2[1, 1] = -5
    rs2, bad2 = oracle.replay(case, idx2)
    assert bad2 == 2 and math.isnan(rs2[0, 0]) and math.isnan(rs2[1, 1])


def test_mixed_e4m3_q_bf16_k_reduces_to_bf16():
    """e4m3 q (power-of-two q_scale) with bf16 k equals the bf16 problem whose q
    is those values, exactly (every such value is a bf16 value): selection,
    replay and backward."""
    import torch

    g = si.rng_for(31)
    n, H, d, L, k_top = 6, 4, 16, 300, 20
    codes = g.choice([0x38, 0x40, 0xB8, 0x44, 0xC0, 0x30, 0x00], size=(n, H, d)).astype(np.uint8)
    qs = np.exp2(g.integers(-2, 3, size=(n, H))).astype(np.float32)
    qf = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy() * qs[:, :, None]
    kf = g.integers(-3, 4, size=(L, d)).astype(np.float32)
    base = {"k": si.f32_to_bf16_bits(kf), "k_scale": None,
            "w": g.integers(1, 3, size=(n, H)).astype(np.float32),
            "positions": np.array([299, 250, 120, 40, 10, 299], np.int32), "k_top": k_top,
            "name": "mixed"}
    mixed = dict(base, q=codes, q_scale=qs, dtype="e4m3_bf16")
    plain = dict(base, q=si.f32_to_bf16_bits(qf), q_scale=None, dtype="bf16")
    i1, s1 = oracle.select(mixed)
    i2, s2 = oracle.select(plain)
    assert np.array_equal(i1, i2) and np.array_equal(s1, s2)
    idx = i1.copy()
    r1, _ = oracle.replay(mixed, idx)
    r2, _ = oracle.replay(plain, idx)
    assert np.array_equal(r1, r2)
    grad = g.integers(-2, 3, size=idx.shape).astype(np.float32)
    b1, b2 = oracle.backward(mixed, idx, grad), oracle.backward(plain, idx, grad)
    for key in ("dq", "dk", "dw"):
        assert np.array_equal(b1[key], b2[key])
