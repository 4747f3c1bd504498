#!/usr/bin/env python
"""Benchmark of the HyTopK hot path on one GB300 (or N independent GPUs).

One step = hytopk_select over the workload (sampled threshold, fused
score + filter, check, exact select/sort, recovery) followed by
hytopk_replay of the selected indices. The default workload is the
GLM-5.1-like slice of the HyScale explainer's worked example: L = 2^20 keys,
n = 8192 queries at the last positions, H = 64, d = 128, k = 2048, fp8 e4m3
inputs with fp32 scales (synthetic, seeded).

Prints ONE JSON line (rank 0). `value` is scored causal query-key pairs per
second over the whole step (select + replay), summed over ranks.

Timing: W warm-up steps, then exactly K steps between a barrier +
synchronize on both sides, CUDA events on the launching stream, max over
ranks. At the default workload a step touches more than the 129 MB L2
(K 128 MiB + Q 64 MiB + ~384 MiB of candidates), so no flush is added; for a
workload whose step would fit in L2 the L2 is flushed before every timed
step and the steps are timed one by one, without the flushes.

--impl reference times the CPU oracle (test infrastructure, the baseline
arm) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = ("indexer q-k pairs/s + exact top-k at 1M ctx (% TC peak); "
          "replay entries/s (% HBM)")
REPLAY_BYTES_PER_ENTRY = {  # idx 4 + key row d*esize + key scale + out 4 + q/w share
    "e4m3": 4 + 128 + 4 + 4 + 4.25, "bf16": 4 + 256 + 4 + 4.25}


def recovery_stress():
    """The recovery-stress workload, its sample positions taken from the
    library's own sample plan (the same formulas its kernels use)."""
    import exact_top_token_gb300 as hk

    hk.build()
    hk.load()
    return si.recovery_stress(lambda ctx: hk.sample_plan(ctx, 1)[0])


WORKLOADS = {"glm_1m": si.glm_1m, "glm_1m_adjacent": si.glm_1m_adjacent,
             "glm_1m_bf16": si.glm_1m_bf16,
             "mixed_contexts": si.mixed_contexts,
             "recovery_stress": recovery_stress,
             "tiny_exact": si.tiny_exact}
# DRAM bytes (read + write) of one full-size filter launch, from one ncu
# capture of the filter kernel (dram__bytes_read.sum + dram__bytes_write.sum,
# a single pass) at the build named beside it by the digest of its source
# files (profiles/glm_1m_slices_filter_k_stream_ncu.txt gives the command).
# Reported as roofline.traffic only while the running library is that build;
# otherwise the traffic is reported as null.
FILTER_TRAFFIC = {"glm_1m": {"bytes": 1196557312 + 397560832, "build": "a16bbb981209"}}
FILTER_SOURCES = ("stream_engine.cuh", "stream_launch.cu", "stream_d128_e4m3.cu", "tc.cuh",
                  "common.cuh")


def filter_source_digest():
    """sha256 (first 12 hex digits) of the filter kernel's source files."""
    import hashlib

    h = hashlib.sha256()
    for name in FILTER_SOURCES:
        with open(os.path.join(ROOT, "exact_top_token_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def filter_traffic(workload):
    rec = FILTER_TRAFFIC.get(workload)
    if rec is None or rec["build"] != filter_source_digest():
        return None
    return rec["bytes"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="hytopk", choices=["hytopk", "reference"])
    ap.add_argument("--workload", default="glm_1m", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-twopass", action="store_true")
    ap.add_argument("--no-sharded", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-grouped", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the mixed-context and recovery-stress sections")
    ap.add_argument("--replay-group", type=int, default=1, choices=[1, 2],
                    help="replay of the step: 1 = per query, 2 = adjacent pairs")
    ap.add_argument("--shards", type=int, default=4, help="key ranges of the sharded selection")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=64,
                    help="oracle sample size (queries): the first 16, the last 16, 32 evenly spaced")
    ap.add_argument("--queries", type=int, default=0,
                    help="keep only the last N queries of the workload (profiling captures)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "hytopk" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def pairs_of(case):
    return int((case["positions"].astype(np.int64) + 1).sum())


def shard_case(case, world, rank):
    """Rank `rank`'s shard of a global batch of world x n queries over the same
    keys (weak scaling: every rank keeps n queries, no data-path collective).
    For workloads whose queries sit at the last n positions, the global batch is
    the last world x n positions and rank r takes the r-th block of n counted
    from the end; other workloads give every rank the same positions."""
    if world == 1:
        return case
    n = len(case["positions"])
    L = int(case["k"].shape[0])
    last = np.arange(L - n, L, dtype=np.int32)
    if world * n <= L and np.array_equal(case["positions"], last):
        out = dict(case)
        out["positions"] = (last - rank * n).astype(np.int32)
        return out
    return case


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---- clocks during the timed region ---------------------------------------------------

class ClockSampler:
    """nvidia-smi every 50 ms, started before the warm-up steps; stop(window)
    keeps the samples whose timestamps fall in the timed region's wall-clock
    window (host time.time() bounds), when there are any."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    @staticmethod
    def _when(stamp):
        import datetime

        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        """End sampling; the samples, for summary() over one window or more."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        for line in open(self.file.name):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 11:
                continue
            try:
                rows.append({"t": self._when(parts[0]), "sm": float(parts[2]),
                             "max": float(parts[3]), "util": float(parts[5]), "hw": parts[7],
                             "hwt": parts[8], "swt": parts[9], "pcap": parts[10],
                             "watts": float(parts[4]) if parts[4] not in ("", "[N/A]") else None})
            except ValueError:
                continue
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summary(rows, window=None):
        """Median SM clock under load, the maximum clock and the throttle
        reasons seen inside window (host time.time() bounds)."""
        if rows is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        if window is not None:
            inside = [r for r in rows if r["t"] is not None and window[0] <= r["t"] <= window[1]]
            rows = inside or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if r["util"] >= 50] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if any(r[key] == "Active" for r in busy):
                reasons.append(name)
        watts = [r["watts"] for r in busy if r["watts"] is not None]
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in busy), "reasons": reasons,
                "samples": len(busy),
                # nvidia-smi's power.draw: the board's mean power over the last second
                "power_w_1s_mean": statistics.median(watts) if watts else None}


# ---- the CPU oracle (baseline arm and cpu_baseline) -------------------------------------

def oracle_sample(case, rows):
    import oracle

    sub_pairs = int((case["positions"][rows].astype(np.int64) + 1).sum())
    t0 = time.perf_counter()
    oracle.select(case, rows=rows)
    dt = time.perf_counter() - t0
    return sub_pairs, dt


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(case, n_rows):
    rows = si.sampled_rows(len(case["positions"]), n_rows)
    pairs, dt = oracle_sample(case, rows)
    return {"value": pairs / dt, "unit": "pairs/s", "cores": os.cpu_count(), "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"oracle select of {len(rows)} of {len(case['positions'])} queries "
                      f"({pairs} causal pairs) of {case['name']}, {dt:.1f} s, OpenMP over "
                      "queries on all host cores"}


def reference_arm(args, world, rank):
    if rank != 0:
        return
    case = WORKLOADS[args.workload]()
    rows = si.sampled_rows(len(case["positions"]), min(16, len(case["positions"])))
    for _ in range(args.warmup):
        oracle_sample(case, rows)
    tot_pairs, tot_t = 0, 0.0
    for _ in range(args.steps):
        p, dt = oracle_sample(case, rows)
        tot_pairs += p
        tot_t += dt
    value = tot_pairs / tot_t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "pairs/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": case["dtype"],
            "data": "synthetic", "config": workload_config(case),
            "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": os.cpu_count(),
                             "kind": "oracle", "cpu": cpu_model(),
                             "sample": f"each step: oracle select of {len(rows)} queries"},
            "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 2**20       # GB300 L2
FLUSH_BYTES = 512 * 2**20    # written between timed steps when a step's data could stay in L2


def step_bytes(case):
    """Bytes one step touches at least: keys, queries and ~3k candidates (8 B) per query."""
    n, H, d = case["q"].shape
    return (case["k"].nbytes + case["q"].nbytes + n * 3 * case["k_top"] * 8)


def needs_flush(case):
    return step_bytes(case) < 2 * L2_BYTES


def workload_config(case, world=1):
    n, H, d = case["q"].shape
    mib = step_bytes(case) / 2**20
    l2 = (f"inputs larger than L2: keys {case['k'].nbytes / 2**20:.0f} MiB + queries "
          f"{case['q'].nbytes / 2**20:.0f} MiB + candidates, {mib:.0f} MiB per step"
          if not needs_flush(case) else
          f"L2 flushed before every timed step ({FLUSH_BYTES // 2**20} MiB write, not timed): "
          f"{mib:.0f} MiB per step would fit in the {L2_BYTES // 2**20} MiB L2")
    cfg = {"workload": case["name"], "L": int(case["k"].shape[0]), "n": int(n), "H": int(H),
           "d": int(d), "k_top": int(case["k_top"]), "capacity": 8 * int(case["k_top"]),
           "positions": ("last n" if case["name"] in ("glm_1m", "glm_1m_bf16", "glm_1m_adjacent")
                         else "see synthetic_inputs"),
           "l2": l2}
    if world > 1:
        cfg["parallelism"] = (f"dp{world}: query shards of n per GPU (rank r: the r-th block of n "
                              "positions from the end), keys replicated, no collective")
    return cfg


# ---- the GPU arm -------------------------------------------------------------------------

def launches_per_step(hk, case):
    """Kernels of one step: select (rank, pack, [key-scale check], threshold,
    plan, filter, check, select, recovery, then per fallback chunk the table
    writer and the read-back, which return at once without a fallback) and
    one replay launch. The chunk count is the library's own."""
    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    dt_code = hk.E4M3 if case["dtype"] == "e4m3" else hk.BF16
    chunks = hk.select_fallback_chunks(n, L, H, d, case["k_top"], 0, dt_code)
    if chunks < 0:
        raise ValueError("unsupported shape")
    base = 9 if case["dtype"] == "e4m3" else 8
    return base + 2 * chunks + 1


def gpu_arm(args, world, rank, local):
    import torch

    import exact_top_token_gb300 as hk

    hk.build()
    hk.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = WORKLOADS[args.workload]()
    if args.queries:
        case = si.subset(case, np.arange(len(case["positions"]) - args.queries,
                                         len(case["positions"])))
    case = shard_case(case, world, rank)
    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    k_top = case["k_top"]
    pairs = pairs_of(case)
    pairs_all = sum_over_ranks(pairs, world, dev)
    t = si.to_torch(case, dev)
    dt_code = hk.E4M3 if case["dtype"] == "e4m3" else hk.BF16
    ws = torch.empty(hk.select_workspace_size(n, L, H, d, k_top, 0, dt_code), dtype=torch.uint8,
                     device=dev)
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    tm = time_steps(hk, case, t, ws, dev, args.steps, args.warmup, args.replay_group, world)
    idx, sc = tm["idx"], tm["scores"]
    ms_step = tm["ms_step"]
    phase_ms, replay_ms, select_ms = tm["phases_ms"], tm["replay_ms"], tm["select_ms"]

    pk = peaks()
    flops_per_pair = 2 * H * d
    filter_s = phase_ms["filter"] / 1e3
    achieved_tflops = pairs * flops_per_pair / filter_s / 1e12
    # dense tensor peak of the input dtype: fp8 = 2 x the measured bf16 GEMM peak
    # (the nominal fp8/bf16 ratio); bf16 = the measured bf16 peak
    peak = pk["bf16_tflops"] * (2.0 if case["dtype"] == "e4m3" else 1.0)
    roofline = {"kernel": "k_stream filter (fused score + threshold filter)", "bound": "tensor",
                "achieved": achieved_tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved_tflops / peak,
                "traffic": (None if args.queries else filter_traffic(args.workload)),
                "traffic_unit": ("bytes per launch (ncu dram read + write of the filter "
                                 "build with source digest " + filter_source_digest() + ")"),
                "algorithmic_flops_per_launch": pairs * flops_per_pair,
                "peak_source": (f"{'2 x ' if case['dtype'] == 'e4m3' else ''}measured bf16 burst "
                                f"{pk['bf16_tflops']} TFLOP/s ({pk['source']})")}
    replay_bytes = n * k_top * REPLAY_BYTES_PER_ENTRY[case["dtype"]]
    replay = {"entries_per_s": n * k_top / (replay_ms / 1e3), "ms": replay_ms,
              "achieved_gbs": replay_bytes / (replay_ms / 1e3) / 1e9,
              "frac_hbm_of_measured": replay_bytes / (replay_ms / 1e3) / 1e9 / pk["hbm_gbs"]}

    line = {"metric": METRIC, "value": pairs_all / (ms_step / 1e3), "unit": "pairs/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": case["dtype"], "data": "synthetic", "config": workload_config(case, world),
            "clocks": None, "gpu_launches": launches_per_step(hk, case) * args.steps,
            "roofline": roofline, "select_ms": select_ms, "phases_ms": phase_ms,
            "replay": replay, "peaks": pk}

    if not args.no_e2e:
        line["e2e"] = e2e(args, hk, case, dev, ws, world)
    # clocks of the main timed region (and of the e2e loop, which runs next)
    rows = clocks.stop() if rank == 0 else None
    if rank == 0:
        line["clocks"] = ClockSampler.summary(rows, tm["wall"])
        if "e2e" in line:
            line["e2e"]["clocks"] = ClockSampler.summary(rows, line["e2e"].pop("wall"))
    if not args.no_twopass:
        line["twopass"] = twopass(hk, case, t, dev, idx, pairs)
    if not args.no_sharded:
        line["sharded"] = sharded(hk, case, t, dev, idx, pairs, args.shards)
    if not args.no_grouped and world == 1:
        line["grouped_replay"] = grouped(hk, case, t, dev, idx, ws, args, pk)
    if not args.no_backward and H in (16, 32, 64):
        line["backward"] = backward(hk, case, t, dev, idx, pk)
    if (not args.no_workloads and world == 1 and args.workload == "glm_1m"
            and not args.queries):
        del t, ws, idx, sc, tm
        torch.cuda.empty_cache()
        line["workloads"] = {name: side_workload(hk, name, dev, pk)
                             for name in ("mixed_contexts", "recovery_stress")}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_steps(hk, case, t, ws, dev, steps, warmup, replay_group=1, world=1, stats=False):
    """`warmup` untimed steps, then `steps` timed ones (select + replay), with
    the library's phase events around each phase. When a step's data would fit
    in the L2, the L2 is flushed before every timed step and the steps are
    timed one by one (first phase event to the event after the replay), so
    the flushes are not counted; otherwise the whole run is timed between
    barrier + synchronize. Returns the mean times, the last step's outputs
    and, on request, its statistics."""
    import torch

    n, H, d = case["q"].shape
    k_top = case["k_top"]
    idx = torch.empty((n, k_top), dtype=torch.int32, device=dev)
    sc = torch.empty((n, k_top), dtype=torch.float32, device=dev)
    rs = torch.empty((n, k_top), dtype=torch.float32, device=dev)
    st = torch.zeros(8, dtype=torch.int32, device=dev) if stats else None
    stream = torch.cuda.current_stream(dev)
    nph = len(hk.PHASES) + 1
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)]
                   for _ in range(steps)]
    # torch creates CUDA events lazily: record each once so that the handles
    # exist before the library records them on the stream
    for evs in step_events:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()

    def step(events=None):
        _, _, st_out = hk.select(t["q"], t["k"], t["w"], t["positions"], k_top,
                                 q_scale=t["q_scale"], k_scale=t["k_scale"], workspace=ws,
                                 out=(idx, sc), stats=False,
                                 phase_events=None if events is None else events[:nph])
        hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"],
                  group=replay_group, out=rs)
        if events is not None:
            events[nph].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    flush = needs_flush(case)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    start.record(stream)
    for i in range(steps):
        if flush:
            flush_buf.fill_(i & 0xFF)  # evicts the previous step's data from L2
        step(step_events[i])
    stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    mine = (sum(ev[0].elapsed_time(ev[nph]) for ev in step_events) if flush
            else start.elapsed_time(stop))
    ms_total = max_over_ranks(mine, world, dev)
    out = {"ms_step": ms_total / steps, "flushed": flush, "wall": (wall0, wall1),
           "phases_ms": {name: statistics.mean(ev[j].elapsed_time(ev[j + 1])
                                               for ev in step_events)
                         for j, name in enumerate(hk.PHASES)},
           "replay_ms": statistics.mean(ev[nph - 1].elapsed_time(ev[nph]) for ev in step_events),
           "select_ms": statistics.mean(ev[0].elapsed_time(ev[nph - 1]) for ev in step_events),
           "idx": idx, "scores": sc}
    # correctness guard: replay reproduces the selected scores bit for bit
    if not torch.equal(rs.view(torch.int32), sc.view(torch.int32)):
        raise RuntimeError("replayed scores differ from the selected scores")
    if stats:
        _, _, st = hk.select(t["q"], t["k"], t["w"], t["positions"], k_top,
                             q_scale=t["q_scale"], k_scale=t["k_scale"], workspace=ws,
                             out=(idx, sc), stats=True)
        out["stats"] = hk.read_stats(st)
    del flush_buf
    return out


def side_workload(hk, name, dev, pk, steps=10, warmup=3):
    """One of the other workloads timed like the headline one (select + replay
    per step, phase events): mixed contexts (64K keys, queries at evenly
    spaced positions, some with fewer keys than k) and recovery stress (256K
    keys, more than 64 failed queries, so every query is rescored over its
    whole context). The in-library two-pass path is timed beside them."""
    import torch

    case = WORKLOADS[name]()
    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    k_top = case["k_top"]
    t = si.to_torch(case, dev)
    dt_code = hk.E4M3 if case["dtype"] == "e4m3" else hk.BF16
    ws = torch.empty(hk.select_workspace_size(n, L, H, d, k_top, 0, dt_code), dtype=torch.uint8,
                     device=dev)
    tm = time_steps(hk, case, t, ws, dev, steps, warmup, stats=True)
    pairs = pairs_of(case)
    flops = pairs * 2 * H * d
    peak = pk["bf16_tflops"] * (2.0 if case["dtype"] == "e4m3" else 1.0)
    filt = tm["phases_ms"]["filter"]
    res = {"config": workload_config(case), "dtype": case["dtype"], "steps": steps,
           "warmup": warmup, "ms_per_step": tm["ms_step"],
           "pairs_per_s": pairs / (tm["ms_step"] / 1e3), "select_ms": tm["select_ms"],
           "replay_ms": tm["replay_ms"], "phases_ms": tm["phases_ms"],
           "filter": {"tflops": flops / (filt / 1e3) / 1e12, "peak_tflops": peak,
                      "frac": flops / (filt / 1e3) / 1e12 / peak},
           "stats": tm["stats"],
           "replay_entries_per_s": n * k_top / (tm["replay_ms"] / 1e3)}
    if name == "recovery_stress":
        st = tm["stats"]
        res["recovery"] = {"ms": tm["phases_ms"]["recover"], "n_failed": st["n_failed"],
                           "fallback_used": st["fallback_used"],
                           "rescored_pairs_per_s": (pairs / (tm["phases_ms"]["recover"] / 1e3)
                                                    if st["fallback_used"] else None)}
    tp = twopass(hk, case, t, dev, tm["idx"], pairs)
    res["twopass"] = {"select_ms": tp["ms"], "same_idx_as_hytopk": tp["same_idx_as_hytopk"],
                      "hytopk_select_ms": tm["select_ms"]}
    del t, ws, tm
    torch.cuda.empty_cache()
    return res


def e2e(args, hk, case, dev, ws, world):
    """Same step through the public API with pinned host inputs: every step
    copies all of its inputs host-to-device and reads idx and the replay
    scores back device-to-host, inside the timed region. The copies run on
    their own streams, double-buffered, so that step i+1's inputs go up and
    step i's results come down while step i+1 / step i compute (as a loader
    that prefetches the next batch would)."""
    import torch

    host = {}
    for key in ("q", "k", "q_scale", "k_scale", "w", "positions"):
        a = case[key]
        host[key] = None if a is None else torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    n, H, d = case["q"].shape
    k_top = case["k_top"]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = 2 * n * k_top * 4
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    dev_in = [{k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in host.items()}
              for _ in range(2)]
    dev_idx = [torch.empty((n, k_top), dtype=torch.int32, device=dev) for _ in range(2)]
    dev_rs = [torch.empty((n, k_top), dtype=torch.float32, device=dev) for _ in range(2)]
    out_idx = [torch.empty((n, k_top), dtype=torch.int32).pin_memory() for _ in range(2)]
    out_rs = [torch.empty((n, k_top), dtype=torch.float32).pin_memory() for _ in range(2)]
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]

    def upload(b):
        with torch.cuda.stream(up):
            up.wait_event(computed[b])  # the step that last read buffer b is done
            for key, v in host.items():
                if v is not None:
                    dev_in[b][key].copy_(v, non_blocking=True)
            uploaded[b].record(up)

    def compute(b):
        comp.wait_event(uploaded[b])
        comp.wait_event(downloaded[b])  # the results last in buffer b have left
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ev[0].record(comp)
        dv = dev_in[b]
        if case["dtype"] == "bf16":
            q = dv["q"].view(torch.int16).view(torch.bfloat16)
            k = dv["k"].view(torch.int16).view(torch.bfloat16)
        else:
            q = dv["q"].view(torch.float8_e4m3fn)
            k = dv["k"].view(torch.float8_e4m3fn)
        hk.select(q, k, dv["w"], dv["positions"], k_top, q_scale=dv["q_scale"],
                  k_scale=dv["k_scale"], scores=False, workspace=ws, out=(dev_idx[b], None))
        hk.replay(q, k, dv["w"], dev_idx[b], q_scale=dv["q_scale"], k_scale=dv["k_scale"],
                  out=dev_rs[b])
        ev[1].record(comp)
        compute_events.append(ev)
        computed[b].record(comp)

    def download(b):
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            out_idx[b].copy_(dev_idx[b], non_blocking=True)
            out_rs[b].copy_(dev_rs[b], non_blocking=True)
            downloaded[b].record(down)

    def run(steps):
        upload(0)
        for i in range(steps):
            b = i & 1
            compute(b)
            if i + 1 < steps:
                upload(b ^ 1)
            download(b)
        torch.cuda.synchronize()

    compute_events = []  # device time of each step's select + replay
    for e in computed + downloaded:
        e.record(comp)
    run(2)  # warm-up
    steps = max(10, min(args.steps, 20))  # pipeline fill and drain spread over 10+ steps
    barrier(world)
    gc.disable()  # no collector pause while the host issues the steps
    compute_events.clear()
    wall0 = time.time()
    t0 = time.perf_counter()
    run(steps)
    elapsed = time.perf_counter() - t0
    wall1 = time.time()
    gc.enable()
    dt = max_over_ranks(elapsed / steps, world, dev)
    # the last step's results arrived whole
    if not torch.equal(out_idx[(steps - 1) & 1], dev_idx[(steps - 1) & 1].cpu()):
        raise RuntimeError("e2e: downloaded indices differ from the device result")
    return {"value": sum_over_ranks(pairs_of(case), world, dev) / dt, "unit": "pairs/s",
            "ms_per_step": dt * 1e3,
            # device time of the step's select + replay inside this loop (CUDA
            # events on the compute stream, after its waits for the copies)
            "compute_ms_per_step": statistics.mean(a.elapsed_time(b) for a, b in compute_events),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "copies": "own streams, double-buffered: next step's inputs up and this step's "
                      "results down while a step computes", "wall": (wall0, wall1)}


def twopass(hk, case, t, dev, idx_ref, pairs):
    """The in-library materialise-then-top-k path: the median of three timed runs
    after a warm-up."""
    import torch

    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    dt_code = hk.E4M3 if case["dtype"] == "e4m3" else hk.BF16
    free, _ = torch.cuda.mem_get_info(dev)
    full = hk.twopass_workspace_size(n, L, H, d, case["k_top"], dt_code, 0)
    rows = n if full < 0.8 * free else max(1, int(0.6 * free) // (L * 4))
    wsz = hk.twopass_workspace_size(n, L, H, d, case["k_top"], dt_code, rows)
    ws2 = torch.empty(wsz, dtype=torch.uint8, device=dev)

    def run():
        return hk.select_twopass(t["q"], t["k"], t["w"], t["positions"], case["k_top"],
                                 q_scale=t["q_scale"], k_scale=t["k_scale"], workspace=ws2)

    run()
    torch.cuda.synchronize()
    times = []
    for _ in range(3):  # median of three timed runs
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        i2, _ = run()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    same = bool(torch.equal(i2, idx_ref))
    del ws2
    return {"value": pairs / (ms / 1e3), "unit": "pairs/s", "ms": ms, "runs": 3,
            "rows_per_chunk": rows, "table_bytes_written": n * L * 4,
            "same_idx_as_hytopk": same}


def sharded(hk, case, t, dev, idx_ref, pairs, P):
    """The key-sharded selection (one selection per key range + merge), timed
    once after a warm-up, with its result checked against hytopk_select."""
    import torch

    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    dt_code = hk.E4M3 if case["dtype"] == "e4m3" else hk.BF16
    ws3 = torch.empty(hk.select_sharded_workspace_size(n, L, H, d, case["k_top"], P, 0, dt_code),
                      dtype=torch.uint8, device=dev)

    def run():
        return hk.select_sharded(t["q"], t["k"], t["w"], t["positions"], case["k_top"], P,
                                 q_scale=t["q_scale"], k_scale=t["k_scale"], workspace=ws3)

    run()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    i3, _, _ = run()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    same = bool(torch.equal(i3, idx_ref))
    del ws3
    return {"value": pairs / (ms / 1e3), "unit": "pairs/s", "ms": ms, "shards": P,
            "same_idx_as_hytopk": same}


def adjacent_share(idx):
    """Mean fraction of query 2i's selected keys that query 2i+1 also selected."""
    a = idx.cpu().numpy()
    m = a.shape[0] // 2
    k = a.shape[1]
    shared = [np.intersect1d(a[2 * i][a[2 * i] >= 0], a[2 * i + 1][a[2 * i + 1] >= 0]).size
              for i in range(m)]
    return float(np.mean(shared)) / k if m else 0.0


def time_replays(hk, t, idx, group, reps=5):
    """Median CUDA-event time of `reps` replays (after one warm-up) and the result."""
    import torch

    times = []
    out = None
    for rep in range(reps + 1):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        out = hk.replay(t["q"], t["k"], t["w"], idx, q_scale=t["q_scale"], k_scale=t["k_scale"],
                        group=group)
        b.record()
        torch.cuda.synchronize()
        if rep:
            times.append(a.elapsed_time(b))
    return statistics.median(times), out


def grouped(hk, case, t, dev, idx, ws, args, pk):
    """Replay with adjacent queries grouped in pairs (group 2: the union of the
    two index lists is gathered once) against the per-query replay: on this
    workload's own selection, and for the 1M-key workload also on the same
    shapes with neighbouring queries alike (glm_1m_adjacent, whose selection is
    run once here). Both replays must agree bit for bit."""
    import torch

    def compare(tt, ii):
        n, k_top = ii.shape
        ms1, r1 = time_replays(hk, tt, ii, 1)
        ms2, r2 = time_replays(hk, tt, ii, 2)
        same = bool(torch.equal(r1.view(torch.int32), r2.view(torch.int32)))
        if not same:
            raise RuntimeError("grouped replay differs from the per-query replay")
        share = adjacent_share(ii)
        nbytes = n * k_top * REPLAY_BYTES_PER_ENTRY[case["dtype"]]
        return {"adjacent_share": share, "single_ms": ms1, "grouped_ms": ms2,
                "speedup": ms1 / ms2, "grouped_entries_per_s": n * k_top / (ms2 / 1e3),
                "grouped_frac_hbm_of_measured": nbytes / (ms2 / 1e3) / 1e9 / pk["hbm_gbs"],
                "gathered_rows_vs_single": 1.0 - share / 2, "same_scores": same}

    res = {args.workload: compare(t, idx)}
    if args.workload == "glm_1m" and not args.queries:
        adj = si.glm_1m_adjacent()
        ta = si.to_torch(adj, dev)
        n, H, d = adj["q"].shape
        ia, _, _ = hk.select(ta["q"], ta["k"], ta["w"], ta["positions"], adj["k_top"],
                             q_scale=ta["q_scale"], k_scale=ta["k_scale"], workspace=ws)
        r = compare(ta, ia)
        r["rho"] = 0.98
        res["glm_1m_adjacent"] = r
        del ta, ia
    return res


def backward(hk, case, t, dev, idx, pk):
    """Gradients at the selected entries (hytopk_replay_backward) for the indices
    of the last step and a seeded upstream gradient: 3 timed calls after one
    warm-up, CUDA events around each call."""
    import torch

    n, H, d = case["q"].shape
    L = case["k"].shape[0]
    k_top = idx.shape[1]
    es = 1 if case["dtype"] == "e4m3" else 2
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    grad = torch.randn(idx.shape, generator=gen, device=dev, dtype=torch.float32)
    dk = torch.zeros((L, d), dtype=torch.float32, device=dev)
    times = []
    for rep in range(4):
        dk.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        hk.replay_backward(t["q"], t["k"], t["w"], idx, grad, q_scale=t["q_scale"],
                           k_scale=t["k_scale"], dk=dk)
        b.record()
        torch.cuda.synchronize()
        if rep:
            times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    entries = n * k_top
    # DRAM bytes a perfect implementation moves: per entry idx, grad, key row and
    # key scale; per query q, w, q_scale, dq and dw; dk read and written once
    nbytes = (entries * (4 + 4 + d * es + (4 if es == 1 else 0)) +
              n * (H * d * es + 4 * H * (2 if es == 1 else 1) + 4 * H * d + 4 * H) + 2 * L * d * 4)
    flops = entries * 3 * 2 * H * d  # rescoring, dq and dk contractions
    return {"ms": ms, "entries_per_s": entries / (ms / 1e3),
            "algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (ms / 1e3) / 1e9,
            "frac_hbm_of_measured": nbytes / (ms / 1e3) / 1e9 / pk["hbm_gbs"],
            "algorithmic_flops": flops, "achieved_tflops": flops / (ms / 1e3) / 1e12,
            "frac_bf16_tensor_of_measured": flops / (ms / 1e3) / 1e12 / pk["bf16_tflops"]}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        reference_arm(args, world, rank)
    else:
        gpu_arm(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
