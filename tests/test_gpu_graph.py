"""The selection and the replay captured in a CUDA graph: the library never
synchronises and allocates nothing, so one capture of hytopk_select +
hytopk_replay (caller-owned outputs and workspace) replays to the eager
results bit for bit."""
import numpy as np
import pytest

import synthetic_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    import exact_top_token_gb300 as hk

    hk.build()
    hk.load()
    return hk


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
def test_select_and_replay_in_a_cuda_graph(hk, dt):
    import torch

    dev = torch.device("cuda", 0)
    case = si.random_case(20000, 96, 32, 128, 512, dt, seed=61, positions="random")
    t = si.to_torch(case, dev)
    n, k_top = 96, 512
    code = hk.E4M3 if dt == "e4m3" else hk.BF16
    ws = torch.empty(hk.select_workspace_size(n, 20000, 32, 128, k_top, 0, code),
                     dtype=torch.uint8, device=dev)
    idx = torch.empty((n, k_top), dtype=torch.int32, device=dev)
    sc = torch.empty((n, k_top), dtype=torch.float32, device=dev)
    rs = torch.empty((n, k_top), dtype=torch.float32, device=dev)

    def step():
        hk.select(t["q"], t["k"], t["w"], t["positions"], k_top, q_scale=t["q_scale"],
                  k_scale=t["k_scale"], workspace=ws, out=(idx, sc))
        hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"],
                  out=rs)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()  # eager, on the capture stream
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    ref = [x.clone() for x in (idx, sc, rs)]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for x in (idx, sc, rs):
        x.fill_(7)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip((idx, sc, rs), ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    keep = idx.cpu().numpy() >= 0
    assert np.array_equal(rs.cpu().numpy()[keep], sc.cpu().numpy()[keep])
