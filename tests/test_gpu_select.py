"""GPU parity: hytopk_select, hytopk_replay and the two-pass path against the
CPU oracle, through the C ABI, on the named workloads and edge cases."""
import numpy as np
import pytest

import oracle
import synthetic_inputs as si
from parity import check_structure, compare, replay_tolerance, run_select

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


def host(*ts):
    return [None if t is None else t.cpu().numpy() for t in ts]


# ---- exact (integer-valued) workloads --------------------------------------------

def test_tiny_exact_bit_exact(hk, dev):
    case = si.tiny_exact()
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(64), gi, gs, exact=True)
    stats = hk.read_stats(st)
    fs = oracle.filter_sim(case, capacity=8 * 256)
    assert stats["n_failed"] == int(fs["failed"].sum()) == 0
    assert stats["total_candidates"] == int(fs["cnt"].sum())
    assert stats["device_status"] == 0 and stats["n_queries"] == 64


def _desc32_upper(scores):
    """Upper halves of the selection keys: an unsigned order that is descending score."""
    u = np.asarray(scores, np.float32).copy()
    u[u == 0.0] = 0.0
    u = u.view(np.uint32).astype(np.uint64)
    asc = np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)
    return (~asc) & 0xFFFFFFFF


def test_sort_ties_inside_buckets(hk, dev):
    """Integer scores over a wide range: the kept scores of a query are mostly
    distinct with some exact ties, so the final ordering takes its bucket pass
    (no bucket above 32 keys) and must order tied scores by position."""
    case = si.random_case(32768, 32, 16, 64, 2048, dtype="bf16", seed=11, kind="int",
                          name="int_wide")
    # weights 1..64: |partial sums| <= 576 * 64 * 16 < 2^24, so scores stay exact
    case["w"] = si.rng_for(12).integers(1, 65, size=case["w"].shape).astype(np.float32)
    rows = np.arange(32)
    ref_idx, ref_sc = oracle.select(case, rows=rows)
    ties = 0
    for r in rows:
        s = ref_sc[r]
        ties += int(np.sum(s[1:] == s[:-1]))
        up = _desc32_upper(s)
        rng = int(up.max() - up.min())
        sh = max(0, rng.bit_length() - 12)
        buckets = np.bincount(((up - up.min()) >> np.uint64(sh)).astype(np.int64))
        assert buckets.max() <= 32  # the bucket pass, not the bitonic fallback
    assert ties > 100  # tied scores inside buckets, ordered by position
    idx, sc, _, _ = run_select(hk, case, dev)
    gi, gs = host(idx, sc)
    compare(case, rows, gi, gs, exact=True)
    t = si.to_torch(case, dev)
    ti, ts = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], case["k_top"],
                               q_scale=t["q_scale"], k_scale=t["k_scale"])
    assert np.array_equal(ti.cpu().numpy(), gi)
    assert np.array_equal(ts.cpu().numpy().view(np.uint32), gs.view(np.uint32))


def test_recovery_small_per_row_recovery(hk, dev):
    case = si.recovery_small(oracle.sample_positions)
    C = 8 * case["k_top"]
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(len(case["positions"])), gi, gs, exact=True)
    stats = hk.read_stats(st)
    fs = oracle.filter_sim(case, capacity=C)
    assert stats["n_failed"] == int(fs["failed"].sum()) > 0
    assert stats["n_overflow"] == int((fs["cnt"] > C).sum())
    assert stats["n_under_k"] == int((fs["cnt"] < case["k_top"]).sum())
    assert stats["fallback_used"] == 0
    assert stats["total_candidates"] == int(fs["cnt"].sum())


@pytest.mark.slow
def test_recovery_stress_full_fallback(hk, dev):
    """The recovery-stress workload (1024 mass-tie rows that overflow, spiked
    rows, decoy rows that fall short of k): more than 64 failed queries, so
    every query is rescored. All 2048 rows bit-exact against the oracle."""
    case = si.recovery_stress(oracle.sample_positions)
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    rows = np.arange(len(case["positions"]))
    compare(case, rows, gi, gs, exact=True)
    stats = hk.read_stats(st)
    assert stats["fallback_used"] == 1 and stats["n_failed"] > 64
    fs = oracle.filter_sim(case, capacity=8 * case["k_top"])
    assert stats["n_failed"] == int(fs["failed"].sum())
    assert stats["n_overflow"] == int((fs["cnt"] > 8 * case["k_top"]).sum())
    assert stats["n_under_k"] == int((fs["cnt"] < case["k_top"]).sum())
    assert stats["total_candidates"] == int(fs["cnt"].sum())
    assert set(np.flatnonzero(fs["failed"]).tolist()) >= set(case["decoy_rows"].tolist())


@pytest.mark.parametrize("dt,kind,mode", [("bf16", "int", "pos_inf"), ("e4m3", "normal", "neg_inf")])
def test_fallback_table_in_chunks(hk, dev, dt, kind, mode):
    """More than 64 failed queries with a small candidate buffer: every query
    is rescored through score-table rows that fill the candidate and
    recovery-row buffers chunk by chunk (several chunks here)."""
    import torch

    n, L, k_top = 300, 16384, 64
    case = si.random_case(L, n, 8, 64, k_top, dt, seed=61, positions="random", kind=kind)
    thr = torch.full((n,), float("inf") if mode == "pos_inf" else -float("inf"), device=dev)
    idx, sc, st, t = run_select(hk, case, dev, threshold_override=thr, stats=True,
                                capacity=k_top)
    stats = hk.read_stats(st)
    ctx = case["positions"] + 1
    assert stats["fallback_used"] == 1 and stats["n_failed"] == int((ctx > k_top).sum()) > 64
    gi, gs = host(idx, sc)
    compare(case, np.arange(n), gi, gs, exact=(kind == "int"))
    # the same selection without the fallback, bit for bit
    i2, s2, _, _ = run_select(hk, case, dev)
    assert np.array_equal(i2.cpu().numpy(), gi)
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), gs.view(np.uint32))


def test_sampled_threshold_every_sample_count(hk, dev):
    """Integer data at contexts that give every kind of sample count: M = ctx
    (ctx <= 4096), M = 4096, M = ctx/128 between 4096 and 8192 (a ragged last
    tile of samples) and M = 8192 (ctx >= 2^20). The thresholds decide the
    candidate counts and the failed queries, which must equal the oracle's
    filter simulation exactly; the selection is bit-exact."""
    L = (1 << 20) + 5000
    pos = np.array([L - 1, L - 2, (1 << 20) - 1, 1 << 20, 700001, 600000, 524287, 524288,
                    524289, 300000, 5000, 4097, 3000, 900], np.int32)
    case = si.random_case(L, len(pos), 16, 64, 512, "bf16", seed=71, positions=pos, kind="int")
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    rows = np.arange(len(pos))
    compare(case, rows, gi, gs, exact=True)
    stats = hk.read_stats(st)
    fs = oracle.filter_sim(case, capacity=8 * 512)
    assert stats["total_candidates"] == int(fs["cnt"].sum())
    assert stats["n_failed"] == int(fs["failed"].sum())
    assert stats["device_status"] == 0
    counts = {oracle.sample_count(int(p) + 1) for p in pos}
    assert {8192, 5468, 4687, 4096, 3001, 901} <= counts


# ---- random workloads ---------------------------------------------------------------

@pytest.mark.parametrize("L,n,H,d,k_top,dt,pos", [
    (5000, 100, 32, 128, 300, "bf16", "random"),
    (20000, 70, 64, 128, 512, "e4m3", "random"),
    (9001, 33, 16, 64, 256, "bf16", "last"),
    (3000, 129, 4, 64, 100, "e4m3", "spaced"),
    (700, 5, 128, 128, 64, "bf16", "random"),
    (4500, 40, 8, 64, 1, "bf16", "random"),
    (130, 7, 2, 128, 200, "e4m3", "random"),
    (4000, 50, 16, 32, 256, "bf16", "random"),     # 64-byte bf16 rows
    (6000, 40, 64, 256, 300, "e4m3", "random"),    # 256-byte e4m3 rows
    (300, 9, 8, 256, 500, "e4m3", "last"),         # ctx < k
    (5000, 40, 32, 128, 256, "e4m3_bf16", "random"),  # e4m3 q, bf16 k
    (3000, 30, 16, 64, 200, "e4m3_bf16", "last"),
    (9000, 20, 1, 64, 100, "bf16", "random"),      # one head
    (12000, 24, 4, 128, 300, "e4m3", "random"),    # four heads, 128-byte rows
    (20000, 20, 128, 128, 256, "e4m3", "random"),  # 128 heads, 4096 samples
    (15000, 16, 128, 128, 512, "bf16", "random"),  # 128 heads, 256-byte rows
])
def test_random_small(hk, dev, L, n, H, d, k_top, dt, pos):
    case = si.random_case(L, n, H, d, k_top, dt, seed=L + n, positions=pos)
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(n), gi, gs)
    assert hk.read_stats(st)["device_status"] == 0


@pytest.mark.slow
def test_mixed_contexts_full(hk, dev):
    case = si.mixed_contexts()
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(len(case["positions"])), gi, gs)
    assert int((case["positions"] + 1 <= case["k_top"]).sum()) > 0  # some select-all rows



@pytest.mark.slow
def test_large_batch_64bit_offsets(hk, dev):
    """131072 queries with room for 32768 candidates each: slot x capacity
    passes 2^31 (and the candidate buffer's byte offsets 2^32) for half of the
    slots. 32 sampled rows against the oracle, structure on 4096 sampled rows,
    no device status."""
    n, L, H, d, k_top, cap = 131072, 32768, 8, 64, 256, 32768
    case = si.random_case(L, n, H, d, k_top, "bf16", seed=13, positions="random")
    idx, sc, st, _ = run_select(hk, case, dev, stats=True, capacity=cap)
    gi, gs = host(idx, sc)
    stats = hk.read_stats(st)
    assert stats["device_status"] == 0 and stats["n_queries"] == n
    rows = si.sampled_rows(n, 32)
    compare(case, rows, gi[rows], gs[rows])
    many = si.sampled_rows(n, 4096)
    check_structure(gi[many], gs[many], case["positions"][many], k_top)


@pytest.mark.slow
def test_long_work_items_ragged_context(hk, dev):
    """2048 queries at random positions over 700,001 keys with H = 64: enough
    work items for the long (256-tile) key chunks of the filter and of the
    two-pass table writer, a last chunk cut short by L and blocks cut short
    by their positions. 64 sampled rows against the oracle, structure on
    every row, and the two-pass path bit for bit the selection."""
    n, L, H, d, k_top = 2048, 700001, 64, 128, 1024
    case = si.random_case(L, n, H, d, k_top, "e4m3", seed=21, positions="random")
    idx, sc, st, t = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    stats = hk.read_stats(st)
    assert stats["device_status"] == 0 and stats["n_queries"] == n
    rows = si.sampled_rows(n, 64)
    compare(case, rows, gi[rows], gs[rows])
    check_structure(gi, gs, case["positions"], k_top)
    # the two-pass path's table writer takes the long chunks here too
    i2, s2 = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], k_top,
                               q_scale=t["q_scale"], k_scale=t["k_scale"])
    assert np.array_equal(i2.cpu().numpy(), gi)
    assert np.array_equal(s2.cpu().numpy().view(np.uint32), gs.view(np.uint32))

@pytest.fixture(scope="module")
def glm_run(hk, dev):
    """The 1M-key workload selected once and its indices replayed once."""
    case = si.glm_1m()
    idx, sc, st, t = run_select(hk, case, dev, stats=True)
    rs = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"])
    gi, gs, gr = host(idx, sc, rs)
    stats = hk.read_stats(st)
    del t, idx, sc, rs
    return case, gi, gs, gr, stats


@pytest.mark.slow
def test_glm_1m_sampled_rows(glm_run):
    """Selection on the 1M-key workload: 64 rows (the first 16, the last 16, 32
    evenly spaced) against the oracle, structure on all 8192 rows."""
    case, gi, gs, _, stats = glm_run
    rows = si.sampled_rows(len(case["positions"]), 64)
    assert len(rows) == 64
    compare(case, rows, gi[rows], gs[rows])
    check_structure(gi, gs, case["positions"], case["k_top"])
    assert stats["device_status"] == 0 and stats["fallback_used"] == 0


@pytest.mark.slow
def test_glm_1m_replay_every_entry(glm_run):
    """Selection replay on the 1M-key shapes: every one of the 8192 x 2048
    stored entries rescored, each within 1e-3 relative of the oracle's score
    of that (query, key) (no floor: all are top-k scores), and bit for bit the
    score the selection returned."""
    case, gi, gs, gr, _ = glm_run
    assert np.array_equal(gr.view(np.uint32), gs.view(np.uint32))
    assert np.all(gi >= 0)
    ref, bad = oracle.replay(case, gi)
    assert bad == 0
    err = np.abs(gr.astype(np.float64) - ref)
    assert np.all(err <= 1e-3 * np.abs(ref.astype(np.float64))), \
        f"max relative error {np.max(err / np.abs(ref))}"


# ---- the threshold does not change the result (metamorphic) -----------------------------

@pytest.mark.parametrize("mode", ["neg_inf", "pos_inf", "random"])
def test_threshold_override_same_result(hk, dev, mode):
    import torch

    case = si.random_case(6000, 90, 16, 64, 128, "bf16", seed=21, positions="random",
                          kind="int")
    base, bsc, _, t = run_select(hk, case, dev)
    n = len(case["positions"])
    if mode == "neg_inf":
        thr = torch.full((n,), -float("inf"), device=dev)
    elif mode == "pos_inf":
        thr = torch.full((n,), float("inf"), device=dev)
    else:
        thr = torch.from_numpy(np.random.Generator(np.random.PCG64(3)).uniform(
            0, 80, n).astype(np.float32)).to(dev)
    idx, sc, st, _ = run_select(hk, case, dev, threshold_override=thr, stats=True, capacity=300)
    gi, gs = host(idx, sc)
    compare(case, np.arange(n), gi, gs, exact=True)
    stats = hk.read_stats(st)
    ctx = case["positions"] + 1
    expect = {"neg_inf": int((ctx > 300).sum()), "pos_inf": int((ctx > 128).sum())}
    if mode in expect:
        assert stats["n_failed"] == expect[mode]
        assert stats["fallback_used"] == (expect[mode] > 64)


def test_determinism_and_reverse_schedule(hk, dev):
    case = si.random_case(12000, 64, 32, 128, 512, "e4m3", seed=22, positions="random")
    runs = [run_select(hk, case, dev, reverse_schedule=(i % 2 == 1)) for i in range(4)]
    first = host(runs[0][0], runs[0][1])
    for r in runs[1:]:
        other = host(r[0], r[1])
        assert np.array_equal(first[0], other[0]) and np.array_equal(first[1], other[1])


def test_power_of_two_weight_scaling(hk, dev):
    case = si.random_case(3000, 20, 16, 64, 100, "bf16", seed=23, positions="random")
    idx, sc, _, _ = run_select(hk, case, dev)
    scaled = dict(case, w=case["w"] * np.float32(8.0))
    idx2, sc2, _, _ = run_select(hk, scaled, dev)
    gi, gs = host(idx, sc)
    gi2, gs2 = host(idx2, sc2)
    assert np.array_equal(gi, gi2)
    valid = gi >= 0
    assert np.array_equal(gs2[valid], gs[valid] * np.float32(8.0))


def test_all_equal_scores_and_edge_rows(hk, dev):
    import torch

    n, L, H, d, k_top = 6, 300, 4, 64, 50
    case = {"q": si.f32_to_bf16_bits(np.ones((n, H, d), np.float32)), "q_scale": None,
            "k": si.f32_to_bf16_bits(np.ones((L, d), np.float32)), "k_scale": None,
            "w": np.ones((n, H), np.float32),
            "positions": np.array([299, 49, 0, 120, 10, 200], np.int32), "k_top": k_top,
            "dtype": "bf16", "name": "equal"}
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(n), gi, gs, exact=True)
    assert list(gi[0]) == list(range(50))
    assert list(gi[2]) == [0] + [-1] * 49
    # positions outside [0, L) give an all -1 row and the status bit
    bad = dict(case, positions=np.array([299, -3, 300, 5, 1000, 7], np.int32))
    idx, sc, st, _ = run_select(hk, bad, dev, stats=True)
    gi, gs = host(idx, sc)
    for r in (1, 2, 4):
        assert np.all(gi[r] == -1) and np.all(np.isneginf(gs[r]))
    assert list(gi[0]) == list(range(50)) and list(gi[3]) == list(range(6)) + [-1] * 44
    assert hk.read_stats(st)["device_status"] & hk.DEV_BAD_POSITION
    # an empty problem is a no-op
    t = si.to_torch(case, dev)
    e_idx, _, e_st = hk.select(t["q"][:0], t["k"], t["w"][:0], t["positions"][:0], k_top,
                               stats=True)
    assert e_idx.shape == (0, k_top) and hk.read_stats(e_st)["n_queries"] == 0


# ---- replay ---------------------------------------------------------------------------

@pytest.mark.parametrize("which,bad", [("k", 0.0), ("k", -1.0), ("q", 0.0), ("q", -1.0)])
def test_bad_scale_sets_status(hk, dev, which, bad):
    """A key or query scale that is not > 0 sets the bad-scale status bit; with
    valid scales the bit stays clear. The key scales of 1M keys are checked by
    a grid of many blocks, so the bad one sits near the end."""
    L = 300000 if which == "k" else 4000
    case = si.random_case(L, 8, 8, 64, 64, "e4m3", seed=7, positions="random")
    idx, sc, st, _ = run_select(hk, case, dev, stats=True)
    assert hk.read_stats(st)["device_status"] == 0
    if which == "k":
        ks = case["k_scale"].copy()
        ks[L - 3] = bad
        bad_case = dict(case, k_scale=ks)
    else:
        qs = case["q_scale"].copy()
        qs[5, 3] = bad
        bad_case = dict(case, q_scale=qs)
    idx, sc, st, _ = run_select(hk, bad_case, dev, stats=True)
    assert hk.read_stats(st)["device_status"] & hk.DEV_BAD_SCALE


def test_replay_parity_and_bad_indices(hk, dev):
    import torch

    case = si.random_case(8000, 50, 64, 128, 256, "e4m3", seed=24, positions="random")
    idx, sc, _, t = run_select(hk, case, dev)
    rs = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"])
    gi, gs, gr = host(idx, sc, rs)
    assert np.array_equal(gr, gs)
    ref, bad = oracle.replay(case, gi)
    assert bad == 0
    ok = gi >= 0
    assert np.all(np.isneginf(gr[~ok]))
    tol = replay_tolerance(case, gi, ref)
    assert np.all(np.abs(gr[ok].astype(np.float64) - ref[ok]) <= tol[ok])
    idx2 = idx.clone()
    idx2[0, 0] = 8000
    idx2[3, 5] = -7
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rs2 = hk.replay(t["q"], t["k"], t["w"], idx2, q_scale=t["q_scale"], k_scale=t["k_scale"],
                    status=status)
    r2 = rs2.cpu().numpy()
    assert np.isnan(r2[0, 0]) and np.isnan(r2[3, 5])
    assert int(status.item()) & hk.DEV_REPLAY_BAD_INDEX


@pytest.mark.parametrize("d,dt", [(64, "bf16"), (32, "bf16"), (256, "e4m3")])
def test_replay_random_indices_vs_oracle(hk, dev, d, dt):
    import torch

    case = si.random_case(4000, 37, 16, d, 333, dt, seed=25, positions="last")
    g = np.random.Generator(np.random.PCG64(26))
    idx = g.integers(-1, 4000, size=(37, 333)).astype(np.int32)
    t = si.to_torch(case, dev)
    rs = hk.replay(t["q"], t["k"], t["w"], torch.from_numpy(idx).to(dev), q_scale=t["q_scale"],
                   k_scale=t["k_scale"])
    ref, bad = oracle.replay(case, idx)
    got = rs.cpu().numpy()
    assert bad == 0
    assert np.array_equal(np.isneginf(got), idx == -1)
    ok = idx >= 0
    tol = replay_tolerance(case, idx, ref)
    assert np.all(np.abs(got[ok].astype(np.float64) - ref[ok]) <= tol[ok])


# ---- two-pass comparison path ------------------------------------------------------------

@pytest.mark.parametrize("chunk", [0, 7])
def test_twopass_matches_select(hk, dev, chunk):
    case = si.random_case(7000, 45, 32, 128, 400, "bf16", seed=27, positions="random")
    idx, sc, _, t = run_select(hk, case, dev)
    ws = None
    if chunk:
        import torch

        nbytes = hk.twopass_workspace_size(45, 7000, 32, 128, 400, hk.BF16, chunk)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    i2, s2 = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], 400, workspace=ws)
    assert np.array_equal(i2.cpu().numpy(), idx.cpu().numpy())
    assert np.array_equal(s2.cpu().numpy(), sc.cpu().numpy())


@pytest.mark.parametrize("d,dt", [(32, "bf16"), (256, "e4m3")])
def test_new_row_shapes_exact_and_consistent(hk, dev, d, dt):
    """Integer data with the new row shapes: exact against the oracle, and the
    two-pass path and replay agree with the selection bit for bit."""
    case = si.random_case(3000, 30, 8, d, 200, "bf16", seed=d, positions="spaced", kind="int")
    if dt == "e4m3":
        import torch

        qf = si.bf16_bits_to_f32(case["q"])
        kf = si.bf16_bits_to_f32(case["k"])
        case = dict(case, dtype="e4m3",
                    q=torch.from_numpy(qf).to(torch.float8_e4m3fn).view(torch.uint8).numpy(),
                    k=torch.from_numpy(kf).to(torch.float8_e4m3fn).view(torch.uint8).numpy(),
                    q_scale=np.ones(qf.shape[:2], np.float32),
                    k_scale=np.ones(kf.shape[0], np.float32))
    idx, sc, _, t = run_select(hk, case, dev)
    gi, gs = host(idx, sc)
    compare(case, np.arange(30), gi, gs, exact=True)
    i2, s2 = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], case["k_top"],
                               q_scale=t["q_scale"], k_scale=t["k_scale"])
    assert np.array_equal(i2.cpu().numpy(), gi) and np.array_equal(s2.cpu().numpy(), gs)
    rs = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"])
    assert np.array_equal(rs.cpu().numpy(), gs)


def test_twopass_exact_on_integer_data(hk, dev):
    case = si.tiny_exact()
    t = si.to_torch(case, dev)
    i2, s2 = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], case["k_top"])
    compare(case, np.arange(64), i2.cpu().numpy(), s2.cpu().numpy(), exact=True)


def test_mixed_q_e4m3_k_bf16_paths_agree(hk, dev):
    """e4m3 q with bf16 k: the selection matches the oracle, and replay, the
    two-pass path and the key-sharded selection return its scores bit for bit."""
    case = si.random_case(6000, 48, 64, 128, 300, "e4m3_bf16", seed=41, positions="random")
    idx, sc, st, t = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(48), gi, gs)
    assert hk.read_stats(st)["device_status"] == 0
    rs = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"])
    assert np.array_equal(rs.cpu().numpy(), gs)
    i2, s2 = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], 300, q_scale=t["q_scale"])
    assert np.array_equal(i2.cpu().numpy(), gi) and np.array_equal(s2.cpu().numpy(), gs)
    i3, s3, _ = hk.select_sharded(t["q"], t["k"], t["w"], t["positions"], 300, 3,
                                  q_scale=t["q_scale"])
    assert np.array_equal(i3.cpu().numpy(), gi) and np.array_equal(s3.cpu().numpy(), gs)


# ---- the largest k the library takes ------------------------------------------------------

@pytest.mark.parametrize("dt,kind", [("bf16", "int"), ("e4m3", "normal")])
def test_maximum_k(hk, dev, dt, kind):
    """k = 16384 (the largest supported): queries with more and with fewer keys
    than k; the selection against the oracle (exact on integer data), replay
    and the two-pass path bit for bit."""
    k_top = 16384
    L, n = 40000, 12
    pos = np.array([100, 16383, 16384, 16385, 20000, 25000, 30000, 33333, 36000, 38000,
                    39000, 39999], np.int32)
    case = si.random_case(L, n, 16, 64, k_top, dt, seed=44, positions=pos, kind=kind)
    idx, sc, st, t = run_select(hk, case, dev, stats=True)
    gi, gs = host(idx, sc)
    compare(case, np.arange(n), gi, gs, exact=(kind == "int"))
    assert hk.read_stats(st)["device_status"] == 0
    rs = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"])
    r = rs.cpu().numpy()
    keep = gi >= 0
    assert np.array_equal(r[keep], gs[keep]) and np.isneginf(r[~keep]).all()
    i2, s2 = hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], k_top,
                               q_scale=t["q_scale"], k_scale=t["k_scale"])
    assert np.array_equal(i2.cpu().numpy(), gi) and np.array_equal(s2.cpu().numpy(), gs)
