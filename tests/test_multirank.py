"""The bench's N > 1 path on the CPU: two gloo ranks under
torch.distributed.run (127.0.0.1), no GPU.

Queries shard across ranks (weak scaling, keys replicated, no collective on the
data path); the only collectives are the bench's timing reductions."""
import json
import os
import socket
import subprocess
import sys

import numpy as np

import bench
import synthetic_inputs as si

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def torchrun(script_args, nproc=2, timeout=240):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={nproc}", "--master-addr=127.0.0.1",
           f"--master-port={free_port()}", *script_args]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout,
                          env=env)


def test_shard_case_partitions_the_last_positions():
    case = si.tiny_exact()
    n, L = len(case["positions"]), case["k"].shape[0]
    for world in (2, 4, 8):
        shards = [bench.shard_case(case, world, r)["positions"] for r in range(world)]
        allpos = np.concatenate(shards)
        assert len(np.unique(allpos)) == world * n
        assert np.array_equal(np.sort(allpos), np.arange(L - world * n, L))
        assert all(len(s) == n for s in shards)
    assert bench.shard_case(case, 1, 0) is case


def test_shard_case_keeps_other_workloads():
    case = si.random_case(512, 16, 4, 64, 8, positions="spaced", seed=5)
    for r in range(2):
        assert np.array_equal(bench.shard_case(case, 2, r)["positions"], case["positions"])


def test_two_gloo_ranks_reduce_times_and_pairs(tmp_path):
    r = torchrun([os.path.join("tests", "dist_worker.py"), str(tmp_path)])
    assert r.returncode == 0, r.stderr[-3000:]
    res = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert sorted(x["rank"] for x in res) == [0, 1]
    by_rank = {x["rank"]: x for x in res}
    total = by_rank[0]["pairs"] + by_rank[1]["pairs"]
    for x in res:
        assert x["world"] == 2
        assert x["ms_max"] == 11.0          # the slowest rank's time
        assert x["pairs_all"] == total      # every rank's pairs counted once
    p0, p1 = set(by_rank[0]["positions"]), set(by_rank[1]["positions"])
    assert not (p0 & p1)


def test_reference_arm_prints_once_under_two_ranks():
    r = torchrun(["bench.py", "--impl", "reference", "--workload", "tiny_exact", "--steps", "1",
                  "--warmup", "1", "--gpus", "2"])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
