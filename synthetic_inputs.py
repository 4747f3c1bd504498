"""Seeded synthetic inputs for HyTopK selection and selection replay.

This module only draws and encodes input data; it holds none of the method's
arithmetic. Both the GPU library's tests and the CPU oracle receive the very
same arrays from here. Nothing here reads files or the network.

Every case is a dict of numpy arrays::

    q         [n,H,d] uint16 (bf16 bits) or uint8 (OCP FP8 E4M3 codes)
    q_scale   [n,H] float32 (e4m3 only, else None)  one scale per 128-element row
    k         [L,d] same element type as q           one shared key head
    k_scale   [L]   float32 (e4m3 only, else None)
    w         [n,H] float32
    positions [n]   int32, 0 <= pos < L  (query t sees keys s <= pos)
    dtype     "bf16" | "e4m3";  k_top int;  name str

Random draws use numpy's PCG64 with the stated seed, in the order q, k, w.
bf16 encoding is round-to-nearest-even from fp32; e4m3 encoding divides each
row by amax(row)/448 and rounds to nearest even (torch's float8_e4m3fn cast).

The named workloads are the HyScale GLM-5.1 setting of the explainer page's
worked example and the surrounding test cases:

* ``tiny_exact``       L=4096, n=64 at 4032..4095, H=4, d=64, k=256, integer data
* ``mixed_contexts``   L=65536, n=1024 spaced positions, H=32, d=128, k=2048, bf16
* ``glm_1m``           L=2^20, n=8192 last positions, H=64, d=128, k=2048, e4m3
* ``recovery_stress``  L=262144, n=2048 last, H=16, d=64, k=2048: mass ties and
                       spiked / decoy rows that force the recovery paths
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def rng_for(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def e4m3_encode_rows(x):
    """Per-row scaled e4m3: returns (codes uint8 [..., d], scale f32 [...])."""
    import torch

    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = np.clip(x / scale[..., None], -E4M3_MAX, E4M3_MAX).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, scale


def element_types(dtype):
    """(q element type, k element type) of a case dtype: "bf16", "e4m3", or
    "e4m3_bf16" (e4m3 q with a per-row scale, bf16 k without one)."""
    if dtype == "e4m3_bf16":
        return "e4m3", "bf16"
    return dtype, dtype


def _encode(x, dtype):
    if dtype == "bf16":
        return f32_to_bf16_bits(x), None
    if dtype == "e4m3":
        return e4m3_encode_rows(x)
    raise ValueError(dtype)


def last_positions(L: int, n: int) -> np.ndarray:
    return np.arange(L - n, L, dtype=np.int32)


def spaced_positions(L: int, n: int) -> np.ndarray:
    """n positions spread evenly over 1..L-1: 1 + floor(i*(L-2)/(n-1))."""
    i = np.arange(n, dtype=np.int64)
    return (1 + (i * (L - 2)) // max(n - 1, 1)).astype(np.int32)


def random_case(L, n, H, d, k_top, dtype="bf16", seed=0, positions="last", kind="normal",
                name=None, pair_rho=None):
    """A general case. kind="normal": q,k ~ N(0,1)/sqrt(d), w ~ N(0,1)/sqrt(H);
    kind="int": q,k integers in [-3,3], w integers in {1,2} (scores exact in fp32).
    positions: "last", "spaced", "random" or an int32 array.
    pair_rho (normal data): query 2i+1 becomes rho * query 2i + sqrt(1 - rho^2)
    * its own draw, with the weights of query 2i, so that neighbouring queries
    select mostly the same keys, as adjacent tokens do."""
    g = rng_for(seed)
    if kind == "normal":
        qf = g.standard_normal((n, H, d), dtype=np.float32) / np.float32(np.sqrt(d))
        kf = g.standard_normal((L, d), dtype=np.float32) / np.float32(np.sqrt(d))
        w = g.standard_normal((n, H), dtype=np.float32) / np.float32(np.sqrt(H))
    elif kind == "int":
        qf = g.integers(-3, 4, size=(n, H, d)).astype(np.float32)
        kf = g.integers(-3, 4, size=(L, d)).astype(np.float32)
        w = g.integers(1, 3, size=(n, H)).astype(np.float32)
    else:
        raise ValueError(kind)
    if pair_rho is not None:
        m = n // 2
        rho = np.float32(pair_rho)
        qf[1:2 * m:2] = rho * qf[0:2 * m:2] + np.float32(np.sqrt(1.0 - pair_rho ** 2)) * qf[1:2 * m:2]
        w[1:2 * m:2] = w[0:2 * m:2]
    if isinstance(positions, str):
        if positions == "last":
            pos = last_positions(L, n)
        elif positions == "spaced":
            pos = spaced_positions(L, n)
        elif positions == "random":
            pos = g.integers(0, L, size=n).astype(np.int32)
        else:
            raise ValueError(positions)
    else:
        pos = np.ascontiguousarray(positions, dtype=np.int32)
    qdt, kdt = element_types(dtype)
    q, q_scale = _encode(qf, qdt)
    k, k_scale = _encode(kf, kdt)
    return {"q": q, "q_scale": q_scale, "k": k, "k_scale": k_scale, "w": w.astype(np.float32),
            "positions": pos, "dtype": dtype, "k_top": int(k_top),
            "name": name or f"random_{kind}_{dtype}_L{L}_n{n}_H{H}_d{d}_k{k_top}"}


def tiny_exact(seed: int = 0):
    """L=4096 keys, 64 queries at 4032..4095, H=4, d=64, k=256; integer data."""
    return random_case(4096, 64, 4, 64, 256, "bf16", seed, "last", "int", name="tiny_exact")


def mixed_contexts(seed: int = 1, L=65536, n=1024, H=32, d=128, k_top=2048):
    """Evenly spaced causal positions 1..L-1, so some queries see fewer than k keys."""
    return random_case(L, n, H, d, k_top, "bf16", seed, "spaced", "normal",
                       name="mixed_contexts")


def glm_1m(seed: int = 2, L=1 << 20, n=8192, H=64, d=128, k_top=2048):
    """The GLM-5.1-like one-GPU slice at 1M keys: n last queries, fp8 e4m3 with
    per-token (key) and per-token-head (query) fp32 scales."""
    return random_case(L, n, H, d, k_top, "e4m3", seed, "last", "normal", name="glm_1m")


def glm_1m_bf16(seed: int = 2, L=1 << 20, n=8192, H=64, d=128, k_top=2048):
    """The glm_1m shapes with bf16 inputs (no scales): the filter's bf16 MMA
    path at full scale."""
    return random_case(L, n, H, d, k_top, "bf16", seed, "last", "normal", name="glm_1m_bf16")


def glm_1m_adjacent(seed: int = 2, rho: float = 0.98, L=1 << 20, n=8192, H=64, d=128,
                    k_top=2048):
    """glm_1m with neighbouring queries alike (pair_rho = rho): the workload of
    the grouped replay, where queries 2i and 2i+1 share most selected keys."""
    return random_case(L, n, H, d, k_top, "e4m3", seed, "last", "normal",
                       name="glm_1m_adjacent", pair_rho=rho)


def recovery_stress(sampler, seed: int = 3, L=262144, n=2048, H=16, d=64, k_top=2048,
                    n_tie_rows=1024, tie_values=8, group_rows=32, n_decoy_rows=8,
                    n_decoys=200, decoy_every=20):
    """Queries built to defeat the sampled threshold. All values are small
    integers, so every score is exact in fp32 and indices must match bit for bit.

    Key features: k[s,0] = u(s) in [0, tie_values); k[s,1], k[s,2] in [0,16) give
    a background score 16*k1 + k2; k[s,3+g] = 1 marks key s as one of group g's
    k spikes; k[s,3+G+i] = 1 marks key s as one of decoy row i's decoys.
    Rows t < n_tie_rows score u(s) only (mass ties: the buffer overflows).
    Other rows score background + 256*spike (+1024*decoy). Spikes avoid the
    sample points of every row in their group. Decoy rows get n_decoys decoys on
    every decoy_every-th of their own sample points, scored above the spikes,
    so that fewer than k keys pass their threshold.

    ``sampler(ctx)`` returns the sample positions of a query with ctx keys; it
    is passed in so that this module holds none of the method's arithmetic.
    """
    g = rng_for(seed)
    pos = last_positions(L, n)
    spike_rows = n - n_tie_rows
    n_groups = -(-spike_rows // group_rows)
    if d < 3 + n_groups + n_decoy_rows:
        raise ValueError("d too small for the requested groups")
    kf = np.zeros((L, d), dtype=np.float32)
    kf[:, 0] = g.integers(0, tie_values, size=L)
    kf[:, 1] = g.integers(0, 16, size=L)
    kf[:, 2] = g.integers(0, 16, size=L)
    qf = np.zeros((n, H, d), dtype=np.float32)
    w = np.zeros((n, H), dtype=np.float32)
    # every row: heads >= 2 read only zero features; their weights are random
    w[:, 2:] = g.integers(1, 4, size=(n, H - 2))
    qf[:, 2:, 3 + n_groups + n_decoy_rows:] = g.integers(-3, 4, size=(n, H - 2,
                                                          d - 3 - n_groups - n_decoy_rows))
    # mass-tie rows: head 0 reads u(s); head 1 reads -u(s) (always clipped by ReLU)
    qf[:n_tie_rows, 0, 0] = 1.0
    qf[:n_tie_rows, 1, 0] = -1.0
    w[:n_tie_rows, 0] = 1.0
    w[:n_tie_rows, 1] = 5.0
    min_ctx = int(pos[n_tie_rows:].min()) + 1 if spike_rows else L
    for gi in range(n_groups):
        rows = np.arange(n_tie_rows + gi * group_rows, min(n, n_tie_rows + (gi + 1) * group_rows))
        sampled = np.zeros(L, dtype=bool)
        for t in rows:
            sampled[np.asarray(sampler(int(pos[t]) + 1), dtype=np.int64)] = True
        free = np.flatnonzero(~sampled[:min_ctx])
        spikes = g.choice(free, size=k_top, replace=False)
        kf[spikes, 3 + gi] = 1.0
        qf[rows, 0, 1] = 16.0
        qf[rows, 0, 2] = 1.0
        qf[rows, 0, 3 + gi] = 256.0
        w[rows, 0] = 1.0
        w[rows, 1] = 0.0
    decoy_rows = []
    if spike_rows and n_decoy_rows:
        decoy_rows = np.linspace(n_tie_rows, n - 1, n_decoy_rows).astype(np.int64)
        for i, t in enumerate(decoy_rows):
            sp = np.asarray(sampler(int(pos[t]) + 1), dtype=np.int64)
            chosen = sp[::decoy_every][:n_decoys]
            kf[chosen, 3 + n_groups + i] = 1.0
            qf[t, 0, 3 + n_groups + i] = 1024.0
    q, _ = _encode(qf, "bf16")
    k, _ = _encode(kf, "bf16")
    return {"q": q, "q_scale": None, "k": k, "k_scale": None, "w": w, "positions": pos,
            "dtype": "bf16", "k_top": int(k_top), "name": "recovery_stress",
            "tie_rows": np.arange(n_tie_rows), "decoy_rows": np.asarray(decoy_rows)}


def recovery_small(sampler, seed: int = 3):
    """A small recovery case with fewer than 64 failing queries (per-row recovery)."""
    c = recovery_stress(sampler, seed, L=32768, n=256, H=16, d=64, k_top=512, n_tie_rows=8,
                        tie_values=2, group_rows=32, n_decoy_rows=4, n_decoys=300,
                        decoy_every=13)
    c["name"] = "recovery_small"
    return c


def subset(case, rows):
    """The same problem restricted to some queries (keys unchanged)."""
    rows = np.asarray(rows, dtype=np.int64)
    out = dict(case)
    for key in ("q", "w", "positions"):
        out[key] = np.ascontiguousarray(case[key][rows])
    if case["q_scale"] is not None:
        out["q_scale"] = np.ascontiguousarray(case["q_scale"][rows])
    out["name"] = case["name"] + f"_sub{len(rows)}"
    return out


def pack_varlen(cases):
    """Concatenate independent cases (same H, d, dtype, k_top) into one packed
    variable-length batch: returns (packed case, cu_q, cu_k), the offset arrays
    holding B+1 entries. Positions stay relative to each sequence."""
    first = cases[0]
    cu_q = np.zeros(len(cases) + 1, np.int32)
    cu_k = np.zeros(len(cases) + 1, np.int32)
    for b, c in enumerate(cases):
        assert c["dtype"] == first["dtype"] and c["k_top"] == first["k_top"]
        cu_q[b + 1] = cu_q[b] + len(c["positions"])
        cu_k[b + 1] = cu_k[b] + c["k"].shape[0]

    def cat(key):
        if first[key] is None:
            return None
        return np.ascontiguousarray(np.concatenate([c[key] for c in cases]))

    out = {key: cat(key) for key in ("q", "q_scale", "k", "k_scale", "w", "positions")}
    out.update(dtype=first["dtype"], k_top=first["k_top"], name=f"varlen_B{len(cases)}")
    return out, cu_q, cu_k


def sampled_rows(n: int, count: int = 64) -> np.ndarray:
    """A fixed subset of query rows: the first 16, the last 16 and the rest evenly spaced."""
    if n <= count:
        return np.arange(n)
    edge = count // 4
    mid = np.linspace(edge, n - edge - 1, count - 2 * edge).astype(np.int64)
    return np.unique(np.concatenate([np.arange(edge), mid, np.arange(n - edge, n)]))


WORKLOADS = {
    "tiny_exact": {"L": 4096, "n": 64, "H": 4, "d": 64, "k_top": 256, "dtype": "bf16"},
    "mixed_contexts": {"L": 65536, "n": 1024, "H": 32, "d": 128, "k_top": 2048, "dtype": "bf16"},
    "glm_1m": {"L": 1 << 20, "n": 8192, "H": 64, "d": 128, "k_top": 2048, "dtype": "e4m3"},
    "recovery_stress": {"L": 262144, "n": 2048, "H": 16, "d": 64, "k_top": 2048, "dtype": "bf16"},
}


def to_torch(case, device="cuda"):
    """The case's arrays as torch tensors on `device` (bf16 / float8_e4m3fn
    element types), in the layouts the library takes."""
    import torch

    def t(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(device)

    qdt, kdt = element_types(case["dtype"])
    q = (t(case["q"].view(np.int16)).view(torch.bfloat16) if qdt == "bf16"
         else t(case["q"]).view(torch.float8_e4m3fn))
    k = (t(case["k"].view(np.int16)).view(torch.bfloat16) if kdt == "bf16"
         else t(case["k"]).view(torch.float8_e4m3fn))
    return {"q": q, "k": k, "q_scale": t(case["q_scale"]), "k_scale": t(case["k_scale"]),
            "w": t(case["w"]), "positions": t(case["positions"]), "k_top": case["k_top"]}
