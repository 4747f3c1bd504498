"""The C-ABI library without a GPU: it builds, loads, exports every symbol
that include/hytopk.h declares, and its host-side argument checks return the
documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

import exact_top_token_gb300 as hk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    hk.build()
    return hk.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hytopk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hytopk_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(hk.symbols)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code, text in hk.STATUS.items():
        assert lib.hytopk_status_string(code).decode() == text
    assert lib.hytopk_version() >= 100


def test_supported_row_shapes(lib):
    """Rows of 64, 128 or 256 bytes: bf16 d = 32, 64, 128; e4m3 d = 64, 128, 256."""
    ws = lib.hytopk_select_workspace_size
    for d, dt, ok in [(32, 0, True), (64, 0, True), (128, 0, True), (256, 0, False),
                      (32, 1, False), (64, 1, True), (128, 1, True), (256, 1, True),
                      (96, 0, False), (16, 0, False)]:
        assert (ws(64, 4096, 4, d, 256, 0, dt) > 0) == ok, (d, dt)


def test_workspace_size_rules(lib):
    ws = lib.hytopk_select_workspace_size
    assert ws(64, 4096, 4, 64, 256, 0, 0) > 0
    assert ws(64, 4096, 4, 64, 256, 100, 0) == 0  # capacity below k
    assert ws(64, 4096, 3, 64, 256, 0, 0) == 0  # H not a power of two
    assert ws(64, 4096, 4, 96, 256, 0, 0) == 0  # d unsupported
    assert ws(64, 4096, 4, 64, 0, 0, 0) == 0
    assert ws(64, 4096, 4, 64, 256, 0, 7) == 0  # bad dtype
    # candidate buffer dominates at the 1M setting: 8192 x 8k x 8 bytes
    big = ws(8192, 1 << 20, 64, 128, 2048, 0, 1)
    assert big >= 8192 * 16384 * 8
    assert lib.hytopk_twopass_workspace_size(8192, 1 << 20, 64, 128, 2048, 1, 0) >= 32 * 2**30


def test_host_checks_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: every case fails a host check first
    args = dict(q=fake, qs=None, k=fake, ks=None, w=fake, pos=fake, n=4, L=100, H=4, d=64,
                k_top=8, dt=0, idx=fake, sc=None, cap=0, ws=fake, wsb=1 << 30, st=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.hytopk_select(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["pos"], a["n"], a["L"],
                                 a["H"], a["d"], a["k_top"], a["dt"], a["idx"], a["sc"], a["cap"],
                                 a["ws"], a["wsb"], a["st"], None)

    assert call(k=None) == 1
    assert call(n=-1) == 1
    assert call(H=6) == 2
    assert call(d=48) == 2
    assert call(d=256) == 2  # bf16 rows of 512 bytes
    assert call(k_top=20000) == 2
    assert call(dt=1) == 1  # e4m3 needs scales
    assert call(dt=2) == 1  # e4m3 q needs q_scale
    assert call(dt=2, qs=fake, ks=fake) == 1  # bf16 k takes no k_scale
    assert call(dt=2, qs=fake, wsb=16) == 3  # accepted up to the workspace check
    assert call(dt=3) == 1
    assert call(qs=fake) == 1  # bf16 takes no scales
    assert call(cap=4) == 1  # capacity < k
    assert call(wsb=16) == 3
    assert call(q=P((1 << 20) + 4)) == 5
    assert call(ws=P((1 << 20) + 128)) == 5
    r = lib.hytopk_replay(fake, None, fake, None, fake, None, 4, 100, 4, 64, 8, 0, fake, None, None)
    assert r == 1  # idx missing
    assert lib.hytopk_select_twopass(fake, None, fake, None, fake, fake, 4, 100, 4, 64, 8, 0, fake,
                                     None, fake, 16, None, None) == 3


def test_sharded_host_checks(lib):
    ws = lib.hytopk_select_sharded_workspace_size
    one = lib.hytopk_select_workspace_size(64, 4096, 4, 64, 256, 0, 0)
    assert ws(64, 4096, 4, 64, 256, 0, 0, 1) > one  # + local lists and merge keys
    assert ws(64, 4096, 4, 64, 256, 0, 0, 0) == 0  # no shard
    assert ws(64, 4096, 4, 64, 256, 0, 0, 65) == 0  # more than 64 shards
    assert ws(64, 4096, 3, 64, 256, 0, 0, 2) == 0  # H not a power of two
    # one range's selection workspace (512 keys) + the merge keys, n x P x k x 8 bytes
    assert ws(64, 4096, 4, 64, 256, 0, 0, 8) >= \
        lib.hytopk_select_workspace_size(64, 512, 4, 64, 256, 0, 0) + 64 * 8 * 256 * 8
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def call(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, pos=fake, n=4, L=100, H=4, d=64,
                 k_top=8, dt=0, P=2, idx=fake, sc=None, cap=0, ws=fake, wsb=1 << 30, st=None)
        a.update(kw)
        return lib.hytopk_select_sharded(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["pos"],
                                         a["n"], a["L"], a["H"], a["d"], a["k_top"], a["dt"],
                                         a["P"], a["idx"], a["sc"], a["cap"], a["ws"], a["wsb"],
                                         a["st"], None)

    assert call(P=0) == 1
    assert call(P=100) == 1
    assert call(H=6) == 2
    assert call(k=None) == 1
    assert call(wsb=16) == 3
    assert call(ws=P((1 << 20) + 128)) == 5
    assert call(pos=None) == 1


def test_backward_host_checks(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def call(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, idx=fake, g=fake, n=4, L=100, H=16,
                 d=64, k_top=8, dt=0, dq=fake, dk=fake, dw=fake, st=None)
        a.update(kw)
        return lib.hytopk_replay_backward(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["idx"],
                                          a["g"], a["n"], a["L"], a["H"], a["d"], a["k_top"],
                                          a["dt"], a["dq"], a["dk"], a["dw"], a["st"], None)

    assert call(H=128) == 2  # more than 64 heads
    assert call(H=3) == 2  # not a power of two (the selection's shape rule)
    assert call(d=32) == 2
    assert call(g=None) == 1 and call(idx=None) == 1 and call(dk=None) == 1
    assert call(dt=1) == 1  # e4m3 needs scales
    assert call(dq=P((1 << 20) + 4)) == 5
    assert call(n=0, idx=None) == 0  # nothing to do


def test_varlen_host_checks(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def arr(*v):
        return (ctypes.c_int32 * len(v))(*v)

    ws = lib.hytopk_select_varlen_workspace_size
    cq, ck = arr(0, 10, 10, 30), arr(0, 1000, 1500, 5000)
    per = max(lib.hytopk_select_workspace_size(10, 1000, 4, 64, 64, 0, 0),
              lib.hytopk_select_workspace_size(20, 3500, 4, 64, 64, 0, 0))
    assert ws(cq, ck, 3, 4, 64, 64, 0, 0) >= per  # the largest sequence's workspace
    assert ws(arr(0, 5, 3), arr(0, 10, 20), 2, 4, 64, 64, 0, 0) == 0  # decreasing offsets
    assert ws(arr(1, 5), arr(0, 10), 1, 4, 64, 64, 0, 0) == 0  # not starting at 0
    assert ws(arr(0, 5), arr(0, 0), 1, 4, 64, 64, 0, 0) == 0  # queries without keys
    assert ws(cq, ck, 0, 4, 64, 64, 0, 0) == 0  # no sequence
    assert ws(cq, ck, 3, 3, 64, 64, 0, 0) == 0  # H not a power of two

    def call(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, pos=fake, cq=cq, ck=ck, B=3, H=4, d=64,
                 k_top=64, dt=0, idx=fake, sc=None, cap=0, ws=fake, wsb=1 << 34, st=None)
        a.update(kw)
        return lib.hytopk_select_varlen(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["pos"],
                                        a["cq"], a["ck"], a["B"], a["H"], a["d"], a["k_top"],
                                        a["dt"], a["idx"], a["sc"], a["cap"], a["ws"], a["wsb"],
                                        a["st"], None)

    assert call(cq=arr(0, 10, 5, 30)) == 1
    assert call(B=0) == 1
    assert call(cq=None) == 1
    assert call(H=6) == 2 and call(d=96) == 2
    assert call(k=None) == 1 and call(pos=None) == 1
    assert call(wsb=16) == 3
    assert call(ws=P((1 << 20) + 128)) == 5
    assert call(k=P((1 << 20) + 8)) == 5  # key rows must start 16-byte aligned
    assert call(w=P((1 << 20) + 2)) == 5  # floats 4-byte aligned
    assert call(dt=1) == 1  # e4m3 needs both scales
    # a scale offset by one key passes the alignment check (then meets the small workspace)
    assert call(dt=1, qs=fake, ks=P((1 << 20) + 4), wsb=16) == 3

    def replay(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, idx=fake, cq=cq, ck=ck, B=3, H=4,
                 d=64, k_top=64, dt=0, sc=fake, st=None)
        a.update(kw)
        return lib.hytopk_replay_varlen(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["idx"],
                                        a["cq"], a["ck"], a["B"], a["H"], a["d"], a["k_top"],
                                        a["dt"], a["sc"], a["st"], None)

    assert replay(ck=arr(0, 1000, 900, 5000)) == 1
    assert replay(idx=None) == 1 and replay(sc=None) == 1
    assert replay(cq=arr(0, 0, 0, 0), ck=arr(0, 1, 2, 3)) == 0  # no query: nothing to do


def test_replay_grouped_host_checks(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def call(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, idx=fake, n=4, L=100, H=4, d=64,
                 k_top=8, dt=0, g=2, sc=fake, st=None)
        a.update(kw)
        return lib.hytopk_replay_grouped(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["idx"],
                                         a["n"], a["L"], a["H"], a["d"], a["k_top"], a["dt"],
                                         a["g"], a["sc"], a["st"], None)

    assert call(g=0) == 1 and call(g=3) == 1
    assert call(idx=None) == 1 and call(sc=None) == 1
    assert call(H=3) == 2 and call(d=48) == 2
    assert call(k=P((1 << 20) + 8)) == 5
    assert call(n=0, idx=None) == 0  # nothing to do


def test_backward_varlen_host_checks(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)

    def arr(*v):
        return (ctypes.c_int32 * len(v))(*v)

    def call(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, idx=fake, g=fake, cq=arr(0, 3, 7),
                 ck=arr(0, 100, 250), B=2, H=16, d=64, k_top=8, dt=0, dq=fake, dk=fake, dw=fake,
                 st=None)
        a.update(kw)
        return lib.hytopk_replay_backward_varlen(a["q"], a["qs"], a["k"], a["ks"], a["w"],
                                                 a["idx"], a["g"], a["cq"], a["ck"], a["B"],
                                                 a["H"], a["d"], a["k_top"], a["dt"], a["dq"],
                                                 a["dk"], a["dw"], a["st"], None)

    assert call(cq=arr(0, 5, 3)) == 1  # decreasing offsets
    assert call(ck=arr(0, 0, 250)) == 1  # a sequence with queries and no keys
    assert call(g=None) == 1 and call(dk=None) == 1
    assert call(H=6) == 2
    assert call(cq=arr(0, 0, 0)) == 0  # no query: nothing to do


def test_wait_timeout_bit_matches_the_header():
    text = open(os.path.join(ROOT, "include", "hytopk.h")).read()
    m = re.search(r"#define HYTOPK_DEV_WAIT_TIMEOUT (0x[0-9a-fA-F]+)u", text)
    assert m and int(m.group(1), 16) == hk.DEV_WAIT_TIMEOUT


def test_sample_plan_equals_the_oracle(lib):
    """The library's host-side sample plan (sample count M, positions p_j and
    threshold rank r of a query with ctx keys) against the oracle's, at the
    clamp boundaries of M and at the 1M-key setting."""
    import numpy as np

    import oracle

    ctxs = [1, 2, 3, 100, 255, 256, 257, 2047, 2048, 2049, 4095, 4096, 4097, 6000, 65535,
            524287, 524288, 524289, 1000003, 1 << 20, (1 << 20) + 1, 1 << 24, (1 << 30) - 1]
    for k_top in (1, 256, 2048, 16384):
        for ctx in ctxs:
            pos, r = hk.sample_plan(ctx, k_top)
            m = oracle.sample_count(ctx)
            assert len(pos) == m
            assert r == oracle.threshold_rank(ctx, k_top)
            assert np.array_equal(pos, oracle.sample_positions(ctx).astype(np.int32)), ctx
    # the worked example at 1M keys: 8192 samples, 128 keys apart, the 48th best
    pos, r = hk.sample_plan(1 << 20, 2048)
    assert len(pos) == 8192 and r == 48 and np.all(np.diff(pos) == 128)
    assert lib.hytopk_sample_plan(0, 2048, None, None) == 0
    assert lib.hytopk_sample_plan(5000, 0, None, None) == 0


def test_noalloc_host_checks(lib):
    """hytopk_select_noalloc reports argument errors as hytopk_select does,
    before its scratch-size check, without touching the device."""
    P, I = ctypes.c_void_p, ctypes.c_int
    f = lib.hytopk_select_noalloc
    f.restype = I
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, I, P, P]
    fake = P(1 << 20)  # never dereferenced: every case fails a host check first

    def call(**kw):
        a = dict(q=fake, qs=None, k=fake, ks=None, w=fake, pos=fake, n=4, L=100, H=4, d=64,
                 k_top=8, dt=0, idx=fake, sc=None, cap=0, st=None)
        a.update(kw)
        return f(a["q"], a["qs"], a["k"], a["ks"], a["w"], a["pos"], a["n"], a["L"], a["H"],
                 a["d"], a["k_top"], a["dt"], a["idx"], a["sc"], a["cap"], a["st"], None)

    assert call(H=6) == 2 and call(d=48) == 2 and call(k_top=20000) == 2
    assert call(n=-1) == 1 and call(dt=7) == 1
    assert call(k=None) == 1 and call(pos=None) == 1 and call(idx=None) == 1
    assert call(dt=1) == 1  # e4m3 needs scales
    assert call(cap=4) == 1  # capacity below k
    assert call(q=P((1 << 20) + 4)) == 5
    # a problem beyond the 32 MiB array, with null and misaligned pointers:
    # the pointer errors are reported first
    big = dict(n=8192, L=1 << 20, H=64, d=128, k_top=2048, dt=1, qs=fake, ks=fake)
    assert call(**dict(big, pos=None)) == 1
    assert call(**dict(big, k=P((1 << 20) + 8))) == 5
    assert call(**big) == 3


def fallback_chunks_restated(n, L, k_top, capacity=0):
    """The fallback's score-table chunks from the workspace layout: whole rows
    of L fp32 scores in the candidate buffer (n padded to 512 queries x C
    slots x 8 bytes) and the 64 recovery rows (64 x L x 4 bytes), each buffer
    1 KiB aligned; rounded down to whole waves of the read-back's 304 CTAs
    when that takes no more chunks."""
    def al(x):
        return (x + 1023) // 1024 * 1024
    if n == 0:
        return 0
    n_pad = (n + 511) // 512 * 512
    C = capacity or 8 * k_top
    rows = (al(n_pad * C * 8) + al(64 * L * 4)) // (L * 4)
    if rows > 304:
        waves = rows - rows % 304
        if -(-n // waves) == -(-n // rows):
            rows = waves
    rows = min(rows, n)
    return -(-n // rows)


def test_fallback_chunk_count(lib):
    fc = lib.hytopk_select_fallback_chunks
    # the workloads: 1M keys (26 chunks of 320 rows), 262,144 keys with
    # 2048 queries (7 chunks of 304: one read-back wave each), 64K keys
    assert fc(8192, 1 << 20, 64, 128, 2048, 0, 1) == 26
    assert fc(2048, 1 << 18, 16, 64, 2048, 0, 0) == 7
    assert fc(1024, 1 << 16, 32, 128, 2048, 0, 0) == 2
    assert fc(0, 4096, 4, 64, 256, 0, 0) == 0
    assert fc(64, 4096, 4, 64, 256, 100, 0) == -1  # capacity below k
    assert fc(64, 4096, 3, 64, 256, 0, 0) == -1    # H unsupported
    for n in (1, 63, 512, 700, 4097, 8192):
        for L in (4096, 65537, 1 << 20):
            for k_top, cap in ((256, 0), (2048, 0), (2048, 4096), (16384, 0)):
                for H, d, dt in ((64, 128, 1), (16, 64, 0)):
                    got = fc(n, L, H, d, k_top, cap, dt)
                    assert got == fallback_chunks_restated(n, L, k_top, cap), (n, L, k_top, cap)


def test_bench_launch_count_per_step(lib):
    """The bench's gpu_launches claim per step: 9 select kernels with e4m3
    (8 with bf16: no key-scale check), 2 per fallback chunk, 1 replay."""
    import numpy as np

    import bench
    glm = {"q": np.empty((8192, 64, 128), np.uint8), "k": np.empty((1 << 20, 128), np.uint8),
           "k_top": 2048, "dtype": "e4m3"}
    assert bench.launches_per_step(hk, glm) == 9 + 2 * 26 + 1
    mixed = {"q": np.empty((1024, 32, 128), np.uint16), "k": np.empty((1 << 16, 128), np.uint16),
             "k_top": 2048, "dtype": "bf16"}
    assert bench.launches_per_step(hk, mixed) == 8 + 2 * 2 + 1
