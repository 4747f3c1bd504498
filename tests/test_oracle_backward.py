"""Pins of the oracle's backward at the selected entries (CPU).

The expected values come from the forward oracle, not from the backward's
formulas: on integer data the indexer score is exactly piecewise linear and
every score is exact in fp32, so a unit step of one input changes
L = sum_{t,j} G[t,j] * I[t, idx[t,j]] by exactly that input's derivative
whenever no head dot changes sign. Special cases fix what differences cannot:
the derivative of max(0, x) at x = 0 (taken as 0), idx = -1, bad indices."""
import numpy as np

import oracle
import synthetic_inputs as si


def int_case(L, n, H, d, seed, k_top, dtype="bf16"):
    g = si.rng_for(seed)
    qf = g.integers(-3, 4, size=(n, H, d)).astype(np.float32)
    kf = g.integers(-3, 4, size=(L, d)).astype(np.float32)
    w = g.integers(-2, 3, size=(n, H)).astype(np.float32)  # both signs and zero
    case = {"q": si.f32_to_bf16_bits(qf), "q_scale": None, "k": si.f32_to_bf16_bits(kf),
            "k_scale": None, "w": w, "positions": np.full(n, L - 1, dtype=np.int32),
            "dtype": dtype, "k_top": k_top, "name": "int"}
    idx = np.stack([g.choice(L, size=k_top, replace=False) for _ in range(n)]).astype(np.int32)
    grad = g.integers(-3, 4, size=(n, k_top)).astype(np.float32)
    return case, qf, kf, idx, grad


def loss(case, idx, grad):
    sc, bad = oracle.replay(case, idx)
    assert bad == 0
    sc = np.where(np.isfinite(sc), sc, 0.0)
    return float((sc.astype(np.float64) * grad).sum())


def head_dots(qf, kf):
    """Exact integer head dots [n, H, L] (only to pick steps that keep every sign)."""
    return np.einsum("thi,si->ths", qf.astype(np.int64), kf.astype(np.int64))


def with_q(case, qf):
    return dict(case, q=si.f32_to_bf16_bits(qf))


def with_k(case, kf):
    return dict(case, k=si.f32_to_bf16_bits(kf))


def test_dw_is_the_difference_in_w():
    case, qf, kf, idx, grad = int_case(L=48, n=4, H=4, d=8, seed=11, k_top=12)
    r = oracle.backward(case, idx, grad)
    base = loss(case, idx, grad)
    for t in range(4):
        for h in range(4):
            w2 = case["w"].copy()
            w2[t, h] += 1.0
            assert loss(dict(case, w=w2), idx, grad) - base == r["dw"][t, h]
    assert r["bad"] == 0


def test_dq_is_the_difference_in_q():
    case, qf, kf, idx, grad = int_case(L=40, n=3, H=4, d=6, seed=12, k_top=10)
    r = oracle.backward(case, idx, grad)
    base = loss(case, idx, grad)
    x = head_dots(qf, kf)
    checked = 0
    for t in range(3):
        for h in range(4):
            xs = x[t, h, idx[t]]
            for i in range(6):
                step = xs + kf[idx[t], i].astype(np.int64)
                if (xs == 0).any() or (np.sign(step) != np.sign(xs)).any():
                    continue  # a sign would change: not a derivative
                q2 = qf.copy()
                q2[t, h, i] += 1.0
                assert loss(with_q(case, q2), idx, grad) - base == r["dq"][t, h, i]
                checked += 1
    assert checked >= 20


def test_dk_is_the_difference_in_k():
    case, qf, kf, idx, grad = int_case(L=24, n=3, H=3, d=5, seed=13, k_top=8)
    r = oracle.backward(case, idx, grad)
    base = loss(case, idx, grad)
    x = head_dots(qf, kf)
    checked = 0
    for s in range(24):
        users = [(t, j) for t in range(3) for j in range(8) if idx[t, j] == s]
        for i in range(5):
            safe = True
            for t, _ in users:
                xs = x[t, :, s]
                step = xs + qf[t, :, i].astype(np.int64)
                if (xs == 0).any() or (np.sign(step) != np.sign(xs)).any():
                    safe = False
            if not safe:
                continue
            k2 = kf.copy()
            k2[s, i] += 1.0
            assert loss(with_k(case, k2), idx, grad) - base == r["dk"][s, i]
            checked += 1
    assert checked >= 20
    # keys nobody selected get no gradient
    unused = np.setdiff1d(np.arange(24), idx.ravel())
    assert (r["dk"][unused] == 0).all()


def test_relu_kink_derivative_is_zero():
    """x = 0 exactly: reading, d max(0, x) / dx = 0 there (no term at all)."""
    qf = np.zeros((1, 2, 4), np.float32)
    qf[0, 0] = [1, -1, 0, 0]   # head 0: dot with k = (1, 1, .) is 0
    qf[0, 1] = [1, 1, 0, 0]    # head 1: dot 2
    kf = np.zeros((3, 4), np.float32)
    kf[1] = [1, 1, 2, 0]
    case = {"q": si.f32_to_bf16_bits(qf), "q_scale": None, "k": si.f32_to_bf16_bits(kf),
            "k_scale": None, "w": np.array([[3.0, 5.0]], np.float32),
            "positions": np.array([2], np.int32), "dtype": "bf16", "k_top": 1, "name": "kink"}
    r = oracle.backward(case, np.array([[1]], np.int32), np.array([[2.0]], np.float32))
    assert (r["dq"][0, 0] == 0).all() and r["dw"][0, 0] == 0
    assert np.array_equal(r["dq"][0, 1], 2 * 5 * kf[1])
    assert np.array_equal(r["dk"][1], 2 * 5 * qf[0, 1])
    assert r["dw"][0, 1] == 2 * 2


def test_empty_and_bad_indices():
    case, qf, kf, idx, grad = int_case(L=32, n=2, H=2, d=4, seed=14, k_top=6)
    idx2 = idx.copy()
    idx2[0, 1] = -1
    idx2[1, 3] = 99
    idx2[1, 4] = -7
    g0 = grad.copy()
    g0[0, 1] = g0[1, 3] = g0[1, 4] = 0
    a = oracle.backward(case, idx2, grad)
    b = oracle.backward(case, idx, g0)
    assert a["bad"] == 2 and b["bad"] == 0
    for key in ("dq", "dk", "dw"):
        assert np.array_equal(a[key], b[key])


def test_e4m3_scales_enter_the_gradient():
    """Power-of-two scales keep the data exact: dw from differences in w."""
    g = si.rng_for(15)
    n, H, d, L, k_top = 2, 3, 4, 20, 5
    codes_q = g.choice([0x38, 0x40, 0xB8, 0x44, 0xC0], size=(n, H, d)).astype(np.uint8)
    codes_k = g.choice([0x38, 0x40, 0xB8, 0x30, 0xC4], size=(L, d)).astype(np.uint8)
    case = {"q": codes_q, "q_scale": np.exp2(g.integers(-2, 3, size=(n, H))).astype(np.float32),
            "k": codes_k, "k_scale": np.exp2(g.integers(-2, 3, size=L)).astype(np.float32),
            "w": g.integers(-2, 3, size=(n, H)).astype(np.float32),
            "positions": np.full(n, L - 1, np.int32), "dtype": "e4m3", "k_top": k_top,
            "name": "e4m3"}
    idx = np.stack([g.choice(L, size=k_top, replace=False) for _ in range(n)]).astype(np.int32)
    grad = g.integers(-2, 3, size=(n, k_top)).astype(np.float32)
    r = oracle.backward(case, idx, grad)
    base = loss(case, idx, grad)
    for t in range(n):
        for h in range(H):
            w2 = case["w"].copy()
            w2[t, h] += 1.0
            assert loss(dict(case, w=w2), idx, grad) - base == r["dw"][t, h]
    assert np.abs(r["dw"]).sum() > 0


def test_abs_and_ambiguity_bounds():
    case, qf, kf, idx, grad = int_case(L=30, n=2, H=3, d=4, seed=16, k_top=7)
    r = oracle.backward(case, idx, grad, eps=0.0)
    assert (np.abs(r["dq"]) <= r["dq_abs"]).all() and (np.abs(r["dk"]) <= r["dk_abs"]).all()
    assert (np.abs(r["dw"]) <= r["dw_abs"]).all()
    # a huge eps marks every term ambiguous, positive dot or not
    big = oracle.backward(case, idx, grad, eps=1e9)
    assert (big["dq_amb"] >= big["dq_abs"]).all() and (big["dk_amb"] >= big["dk_abs"]).all()
    assert (big["dq_amb"] > r["dq_amb"]).any()
