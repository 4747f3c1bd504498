"""Comparison of the GPU selection with the CPU oracle.

Integer-valued inputs: indices and scores must match bit for bit.
Random inputs (several results can be correct when fp32 scores nearly tie):
with s_k the oracle's k-th best score of the row and
tol(x) = 1e-3 * max(|x|, |s_k|, 1e-30),
  * each GPU score is within tol of the oracle's score of the same key;
  * a key the GPU kept but the oracle did not has oracle score >= s_k - tol;
  * a key the oracle kept but the GPU did not has oracle score <= s_k + tol;
  * the GPU row lists distinct causal keys, in non-increasing GPU score, with
    ascending position among exactly equal scores, then -1 padding.
"""
import numpy as np

import oracle
import synthetic_inputs as si

REL_TOL = 1e-3
# A score smaller than 2^-10 of the sum of the magnitudes of its terms has lost
# ten bits or more to cancellation; there "1e-3 relative" is taken relative to
# that sum / 1024 instead (see replay_tolerance).
CANCEL_FLOOR = 2.0 ** -10


def decoded(case):
    """q [n,H,d] and k [L,d] as fp64 values (element code times its row scale)."""
    qdt, kdt = si.element_types(case["dtype"])
    table = oracle.e4m3_table().astype(np.float64)

    def dec(a, dt, scale):
        v = (si.bf16_bits_to_f32(a).astype(np.float64) if dt == "bf16" else table[a])
        if scale is not None:
            v = v * np.asarray(scale, np.float64)[..., None]
        return v

    return dec(case["q"], qdt, case["q_scale"]), dec(case["k"], kdt, case["k_scale"])


def abs_term_sum(case, idx):
    """B[t,j] = sum_h |w[t,h]| * sum_i |q[t,h,i]| |k[idx[t,j],i]| (fp64): the sum
    of the magnitudes of every product that enters the score of entry (t, j).
    Entries with idx outside [0, L) get 0."""
    q, k = decoded(case)
    L = k.shape[0]
    idx = np.asarray(idx)
    out = np.zeros(idx.shape, np.float64)
    aq, ak, aw = np.abs(q), np.abs(k), np.abs(np.asarray(case["w"], np.float64))
    for t in range(idx.shape[0]):
        ok = (idx[t] >= 0) & (idx[t] < L)
        if ok.any():
            out[t, ok] = aw[t] @ (aq[t] @ ak[idx[t, ok]].T)
    return out


def replay_tolerance(case, idx, ref):
    """Per-entry tolerance of a replayed score: 1e-3 relative to
    max(|ref|, CANCEL_FLOOR * B) with B = abs_term_sum. Both sides evaluate the
    score in fp32 (a dot of d products, then a weighted sum of H terms); their
    rounding errors scale with B, not with the possibly cancelled result
    (about sqrt(d + H) * 2^-24 * B each, i.e. < 1e-6 B at d + H = 192), so
    below B / 1024 the relative error of a correct fp32 evaluation is not
    bounded by 1e-3. Selected (top-k) entries sit far above the floor."""
    B = abs_term_sum(case, idx)
    return REL_TOL * np.maximum(np.abs(ref).astype(np.float64), CANCEL_FLOOR * B)


def check_structure(idx, scores, positions, k_top):
    """Validity of a GPU selection that does not need the oracle."""
    for r in range(idx.shape[0]):
        ctx = int(positions[r]) + 1 if positions[r] >= 0 else 0
        k_eff = min(k_top, ctx)
        row = idx[r]
        assert np.all(row[k_eff:] == -1), f"row {r}: padding"
        kept = row[:k_eff]
        assert np.all((kept >= 0) & (kept < ctx)), f"row {r}: non-causal index"
        assert len(np.unique(kept)) == k_eff, f"row {r}: duplicate index"
        if scores is not None:
            sc = scores[r, :k_eff]
            assert np.all(np.isneginf(scores[r, k_eff:])), f"row {r}: score padding"
            assert np.all(sc[:-1] >= sc[1:]), f"row {r}: scores not descending"
            tie = sc[:-1] == sc[1:]
            assert np.all(kept[:-1][tie] < kept[1:][tie]), f"row {r}: tie order"


def compare(case, rows, gpu_idx, gpu_scores, exact=False):
    """Compare GPU rows (arrays indexed like `rows`) with the oracle."""
    rows = np.asarray(rows)
    k_top = case["k_top"]
    ref_idx, ref_sc = oracle.select(case, rows=rows)
    pos = case["positions"][rows]
    check_structure(gpu_idx, gpu_scores, pos, k_top)
    if exact:
        bad = np.flatnonzero(np.any(gpu_idx != ref_idx, axis=1))
        assert len(bad) == 0, (f"{len(bad)} rows differ, first row {rows[bad[0]]}: gpu "
                               f"{gpu_idx[bad[0], :8]} oracle {ref_idx[bad[0], :8]}")
        if gpu_scores is not None:
            assert np.array_equal(gpu_scores, ref_sc)
        return
    sub = si.subset(case, rows)
    safe = np.where(gpu_idx >= 0, gpu_idx, -1)
    ref_at_gpu, bad = oracle.replay(sub, safe)
    assert bad == 0
    for r in range(len(rows)):
        ctx = int(pos[r]) + 1
        k_eff = min(k_top, ctx)
        if k_eff == 0:
            continue
        s_k = float(ref_sc[r, k_eff - 1])

        def tol(x):
            return REL_TOL * np.maximum(np.maximum(np.abs(x), abs(s_k)), 1e-30)

        g = gpu_idx[r, :k_eff]
        o = ref_idx[r, :k_eff]
        if gpu_scores is not None:
            d = np.abs(gpu_scores[r, :k_eff] - ref_at_gpu[r, :k_eff])
            assert np.all(d <= tol(ref_at_gpu[r, :k_eff])), \
                f"row {rows[r]}: score error {d.max()} (s_k {s_k})"
        extra = np.setdiff1d(g, o)
        if len(extra):
            ex_sc = ref_at_gpu[r, :k_eff][np.isin(g, extra)]
            assert np.all(ex_sc >= s_k - tol(ex_sc)), f"row {rows[r]}: wrongly kept keys"
        missing = np.setdiff1d(o, g)
        if len(missing):
            ms = ref_sc[r, :k_eff][np.isin(o, missing)]
            assert np.all(ms <= s_k + tol(ms)), f"row {rows[r]}: dropped keys {missing[:4]}"


def run_select(hk, case, dev, **kw):
    t = si.to_torch(case, dev)
    idx, sc, st = hk.select(t["q"], t["k"], t["w"], t["positions"], case["k_top"],
                            q_scale=t["q_scale"], k_scale=t["k_scale"], **kw)
    return idx, sc, st, t
