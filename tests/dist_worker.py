"""One rank of the multi-process host-logic test (run under torch.distributed.run
on the CPU with the gloo backend): the bench's process-group setup, its query
sharding, and the max / sum reductions that turn per-rank times and pair counts
into the one JSON line rank 0 prints."""
import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
import synthetic_inputs as si  # noqa: E402


def main():
    args = argparse.Namespace(impl="reference")  # selects the gloo backend
    world, rank, local = bench.dist_setup(args)
    cpu = torch.device("cpu")
    case = bench.shard_case(si.tiny_exact(), world, rank)
    pairs = bench.pairs_of(case)
    fake_ms = 10.0 + rank  # a per-rank time; the bench keeps the slowest
    out = {"rank": rank, "world": world, "local": local,
           "positions": case["positions"].tolist(),
           "pairs": pairs,
           "pairs_all": bench.sum_over_ranks(pairs, world, cpu),
           "ms_max": bench.max_over_ranks(fake_ms, world, cpu)}
    bench.barrier(world)
    # one file per rank (the ranks share one stdout, where lines can interleave)
    with open(os.path.join(sys.argv[1], f"rank{rank}.json"), "w") as f:
        json.dump(out, f)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
