"""GPU parity of hytopk_replay_backward (gradients at the selected entries)
against the oracle's fp64 backward, through the C ABI: bit-exact on integer
data, within a tolerance derived from the arithmetic on random data."""
import numpy as np
import pytest

import oracle
import synthetic_inputs as si

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


def random_entries(g, n, L, k_top, pos=None):
    """k_top distinct stored indices per query (causal when positions are given),
    with a few -1 entries."""
    idx = np.full((n, k_top), -1, dtype=np.int32)
    for t in range(n):
        hi = L if pos is None else int(pos[t]) + 1
        m = min(k_top, hi)
        idx[t, :m] = g.choice(hi, size=m, replace=False)
    idx[g.random((n, k_top)) < 0.03] = -1
    return idx


def run(hk, case, dev, idx, grad, **kw):
    import torch

    t = si.to_torch(case, dev)
    ti = torch.from_numpy(idx).to(dev)
    tg = torch.from_numpy(grad).to(dev)
    dq, dk, dw = hk.replay_backward(t["q"], t["k"], t["w"], ti, tg, q_scale=t["q_scale"],
                                    k_scale=t["k_scale"], **kw)
    return dq.cpu().numpy(), dk.cpu().numpy(), dw.cpu().numpy()


def int_case(L, n, H, d, k_top, dtype, seed):
    g = si.rng_for(seed)
    case = si.random_case(L, n, H, d, k_top, "bf16", seed, "last", "int")
    case["w"] = g.integers(-2, 3, size=(n, H)).astype(np.float32)
    if dtype in ("e4m3", "e4m3_bf16"):
        # integer codes 1..3 in e4m3 with power-of-two scales: exact everywhere
        import torch

        qf = g.integers(-3, 4, size=(n, H, d)).astype(np.float32)
        case["q"] = torch.from_numpy(qf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        case["q_scale"] = np.exp2(g.integers(-2, 2, size=(n, H))).astype(np.float32)
        if dtype == "e4m3":
            kf = g.integers(-3, 4, size=(L, d)).astype(np.float32)
            case["k"] = torch.from_numpy(kf).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            case["k_scale"] = np.exp2(g.integers(-2, 2, size=L)).astype(np.float32)
        case["dtype"] = dtype
    return case, g


@pytest.mark.parametrize("L,n,H,d,k_top,dtype", [
    (4096, 64, 16, 64, 256, "bf16"),
    (3000, 40, 32, 128, 300, "bf16"),
    (2048, 33, 64, 128, 200, "e4m3"),
    (1500, 20, 16, 64, 129, "e4m3"),
    (1800, 24, 32, 128, 160, "e4m3_bf16"),
    # fewer than 16 heads (padded to 16 inside the engine)
    (4096, 64, 4, 64, 256, "bf16"),
    (2500, 30, 1, 128, 140, "e4m3"),
    (2200, 26, 2, 64, 170, "bf16"),
    (1900, 21, 8, 128, 150, "e4m3_bf16"),
])
def test_integer_data_bit_exact(hk, dev, L, n, H, d, k_top, dtype):
    case, g = int_case(L, n, H, d, k_top, dtype, seed=L + n + H)
    idx = random_entries(g, n, L, k_top, case["positions"])
    grad = g.integers(-3, 4, size=(n, k_top)).astype(np.float32)
    dq, dk, dw = run(hk, case, dev, idx, grad)
    ref = oracle.backward(case, idx, grad)
    assert np.array_equal(dq, ref["dq"].astype(np.float32))
    assert np.array_equal(dw, ref["dw"].astype(np.float32))
    assert np.array_equal(dk, ref["dk"].astype(np.float32))
    assert np.abs(ref["dq"]).sum() > 0 and np.abs(ref["dk"]).sum() > 0


def within(gpu, ref, name, rtol=2e-4, eps_amb=True):
    tol = rtol * ref[name + "_abs"] + (ref[name + "_amb"] if eps_amb else 0) + 1e-30
    bad = np.abs(gpu - ref[name]) > tol
    assert not bad.any(), (name, int(bad.sum()), float(np.abs(gpu - ref[name]).max()))


@pytest.mark.parametrize("L,n,H,d,k_top,dtype", [
    (5000, 48, 32, 128, 512, "bf16"),
    (8192, 40, 64, 128, 1024, "e4m3"),
    (3000, 70, 16, 64, 300, "e4m3"),
    (4000, 30, 64, 128, 400, "e4m3_bf16"),
    (3500, 45, 4, 64, 256, "bf16"),
    (3000, 33, 8, 128, 300, "e4m3"),
])
def test_random_data_within_tolerance(hk, dev, L, n, H, d, k_top, dtype):
    case = si.random_case(L, n, H, d, k_top, dtype, seed=7 + n, positions="random")
    g = si.rng_for(100 + n)
    idx = random_entries(g, n, L, k_top, case["positions"])
    grad = g.standard_normal((n, k_top)).astype(np.float32)
    dq, dk, dw = run(hk, case, dev, idx, grad)
    ref = oracle.backward(case, idx, grad, eps=1e-5)
    within(dq, ref, "dq")
    within(dw, ref, "dw")
    within(dk, ref, "dk")


def test_dk_accumulates_and_bad_indices(hk, dev):
    import torch

    case, g = int_case(2000, 16, 16, 64, 64, "bf16", seed=5)
    idx = random_entries(g, 16, 2000, 64, case["positions"])
    grad = g.integers(-3, 4, size=(16, 64)).astype(np.float32)
    idx_bad = idx.copy()
    idx_bad[2, 5] = 5000
    idx_bad[7, 0] = -9
    grad0 = grad.copy()
    grad0[2, 5] = grad0[7, 0] = 0
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    base = torch.full((2000, 64), 1.0, dtype=torch.float32, device=dev)
    t = si.to_torch(case, dev)
    dq, dk, dw = hk.replay_backward(t["q"], t["k"], t["w"], torch.from_numpy(idx_bad).to(dev),
                                    torch.from_numpy(grad).to(dev), dk=base, status=st)
    ref = oracle.backward(case, idx, grad0)
    assert np.array_equal(dk.cpu().numpy(), (ref["dk"] + 1.0).astype(np.float32))
    assert np.array_equal(dq.cpu().numpy(), ref["dq"].astype(np.float32))
    assert st.item() == hk.DEV_REPLAY_BAD_INDEX


@pytest.mark.slow
def test_glm_1m_slice(hk, dev):
    """The 1M-key workload: 64 of its queries with the indices the selection
    returns and a random upstream gradient."""
    import torch

    case = si.glm_1m()
    case = si.subset(case, np.arange(len(case["positions"]) - 64, len(case["positions"])))
    t = si.to_torch(case, dev)
    idx, _, _ = hk.select(t["q"], t["k"], t["w"], t["positions"], case["k_top"],
                          q_scale=t["q_scale"], k_scale=t["k_scale"])
    g = si.rng_for(77)
    grad = g.standard_normal(idx.shape).astype(np.float32)
    dq, dk, dw = hk.replay_backward(t["q"], t["k"], t["w"], idx, torch.from_numpy(grad).to(dev),
                                    q_scale=t["q_scale"], k_scale=t["k_scale"])
    ref = oracle.backward(case, idx.cpu().numpy(), grad, eps=1e-5)
    within(dq.cpu().numpy(), ref, "dq")
    within(dw.cpu().numpy(), ref, "dw")
    within(dk.cpu().numpy(), ref, "dk")
