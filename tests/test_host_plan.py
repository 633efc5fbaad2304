"""The host planner on the CPU: tile cost model, cluster shape, stream-K schedule and cut table,
operand extents and tensor-map eligibility.

``host_plan_harness.cu`` compiles the library's host source into a test library
(linked against libgemm_gb300.so for the kernel launchers, which no test here
calls), so the planner runs with a GPU's resource counts given as numbers.
The GB300 figures: 152 SMs; the fp16 pair kernel keeps 76 one-pair clusters or
36 two-pair clusters resident.  Its launch at fp16 4096^3 ran 144 CTAs in
four-CTA clusters with stream-K over 56 of 128 units (the launch record of the
bench and the ncu capture of that kernel).
"""
import ctypes
import os
import random
import subprocess

import pytest

from conftest import REPO

GB300_SMS, PAIRS, QUADS = 152, 76, 36
TILE_AUTO, TILE_1SM_256, TILE_1SM_128, TILE_PAIR = 0, 1, 2, 3
SCHED_AUTO, SCHED_TILES, SCHED_STREAM_K = 0, 1, 2
MCAST_AUTO, MCAST_OFF, MCAST_ON = 0, 1, 2


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    import __graft_entry__
    __graft_entry__.build()
    bm = __graft_entry__.build_module()
    lib_dir = os.path.dirname(bm.LIB_PATH)
    out = str(tmp_path_factory.mktemp("host_plan") / "libhost_plan.so")
    cmd = [bm._nvcc()] + bm.ARCH_FLAGS + [
        "-O1", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-I", bm.INCLUDE, "-I", bm.CSRC,
        os.path.join(REPO, "tests", "host_plan_harness.cu"), "-o", out,
        "-L", lib_dir, "-lgemm_gb300", "-cudart", "shared",
        "-Xlinker", f"-rpath,{lib_dir}:/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    lib = ctypes.CDLL(out)
    i64, i32, ll = ctypes.c_int64, ctypes.c_int, ctypes.c_longlong
    u32p, i32p, llp = ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_longlong)
    lib.plan_choose_tile.argtypes = [i64, i64, i32, i32, i32, i32, i32p]
    lib.plan_choose_cluster.argtypes = [i64, i64, i32, i32, i32, i32]
    lib.plan_choose_schedule.argtypes = [i64, i32, i32, i32, i32, i32, i32p, llp, u32p, i32p]
    lib.plan_stream_k_cuts.argtypes = [ll, i32, i32, i32, ll, u32p]
    lib.plan_stream_k_feasible.argtypes = [ll, i32, i32, i32, ll, ll, u32p]
    lib.plan_span_bytes.restype = ctypes.c_ulonglong
    lib.plan_span_bytes.argtypes = [i64, i64, i64, i64, i32]
    lib.plan_operand_kind.argtypes = [ctypes.c_ulonglong, i64, i64, i64, i64, i32]
    return lib


def tile(lib, M, N, sms=GB300_SMS, pairs=PAIRS, policy=TILE_AUTO, bn=0):
    out = ctypes.c_int()
    kind = lib.plan_choose_tile(M, N, sms, pairs, policy, bn, ctypes.byref(out))
    return kind, out.value


def schedule(lib, tiles, num_kb, max_clusters, have_ws=True, mode=SCHED_AUTO, bn=256):
    dp, sk, cl = ctypes.c_int(), ctypes.c_longlong(), ctypes.c_int()
    cuts = (ctypes.c_uint * (lib.plan_max_sk_clusters() + 1))()
    lib.plan_choose_schedule(tiles, num_kb, max_clusters, int(have_ws), mode, bn, ctypes.byref(dp),
                             ctypes.byref(sk), cuts, ctypes.byref(cl))
    return dp.value, sk.value, cl.value, list(cuts[:cl.value + 1]) if sk.value else []


def cuts_of(lib, units, num_kb, clusters, dp_tiles, e_kb):
    cuts = (ctypes.c_uint * (clusters + 1))()
    lib.plan_stream_k_cuts(units, num_kb, clusters, dp_tiles, e_kb, cuts)
    return list(cuts)


def feasible(lib, units, num_kb, clusters, dp_tiles, e_kb, limit):
    cuts = (ctypes.c_uint * (clusters + 1))()
    return bool(lib.plan_stream_k_feasible(units, num_kb, clusters, dp_tiles, e_kb, limit, cuts))


def test_headline_plan_is_the_recorded_launch(plan):
    """fp16 4096^3 (run as C^T = B^T A^T, the same 4096 x 4096 grid): SM-pair 256 x 256 tiles, two-pair
    clusters, 128 units of two tiles side by side, 72 whole units and 56 split by stream-K over the
    36 clusters (144 CTAs) -- the launch recorded on GB300."""
    assert tile(plan, 4096, 4096) == (2, 256)
    tiles_m = tiles_n = 4096 // 256
    cl = plan.plan_choose_cluster(tiles_m * tiles_n, tiles_n, PAIRS, QUADS, 1, MCAST_AUTO)
    assert cl == 4
    units = tiles_m * (tiles_n // 2)
    num_kb = 4096 // 64  # 128 bytes of K per k-block
    dp, sk, clusters, cuts = schedule(plan, units, num_kb, QUADS)
    assert (dp, clusters, units - dp) == (72, 36, 56) and sk == 56 * num_kb
    assert cl * clusters == 144
    assert cuts[0] == 0 and cuts[-1] == sk


def test_cut_table_by_hand(plan):
    """Three tiles of 10 k-blocks over two clusters, whole tiles following: pieces of 15 end with
    5 k-blocks of a tile.  With an epilogue of 4 k-blocks that ending is not short; with 6 it is,
    costs 10 + 6 = 16 > 15, and the smallest limit that covers the range is 16 (pieces 16, 14).
    Without whole tiles after the pieces nothing waits on the ending: 15, 15 again."""
    assert cuts_of(plan, 30, 10, 2, 2, 4) == [0, 15, 30]
    assert cuts_of(plan, 30, 10, 2, 2, 6) == [0, 16, 30]
    assert cuts_of(plan, 30, 10, 2, 0, 6) == [0, 15, 30]
    assert not feasible(plan, 30, 10, 2, 2, 6, 15) and feasible(plan, 30, 10, 2, 2, 6, 16)


def test_cut_tables_cover_the_range_in_balanced_pieces(plan):
    """Over many schedules: the cuts run from 0 to the range's end without going back, no piece
    exceeds the even share by more than one epilogue's k-blocks, a short tile ending kept in front
    of whole tiles fits the same limit, and the limit is the smallest the feasibility test accepts."""
    rng = random.Random(7)
    for _ in range(400):
        clusters = rng.choice([1, 2, 3, 16, 36, 76, rng.randint(1, 128)])
        num_kb = rng.choice([8, 16, 48, 64, 100, rng.randint(8, 300)])
        tiles = rng.randint(1, 3 * clusters + 2)
        units = tiles * num_kb
        if units < clusters:
            continue
        dp_tiles = rng.choice([0, clusters, rng.randint(0, 2 * clusters)])
        e_kb = rng.choice([4, 8, 16, 32])
        cuts = cuts_of(plan, units, num_kb, clusters, dp_tiles, e_kb)
        assert cuts[0] == 0 and cuts[-1] == units, (units, num_kb, clusters, dp_tiles, e_kb, cuts)
        assert all(b >= a for a, b in zip(cuts, cuts[1:]))
        share = -(-units // clusters)
        pieces = [b - a for a, b in zip(cuts, cuts[1:])]
        limit = max(pieces)
        assert limit <= share + e_kb
        for c, (x, y) in enumerate(zip(cuts, cuts[1:])):
            b = y % num_kb
            ts = y - b
            if 0 < b < e_kb and ts > x and c < dp_tiles:
                assert (ts - x) + e_kb <= share + e_kb
        # the search returns the smallest covering limit: every piece fits it, one less fails
        charged = max([limit] + [(y - y % num_kb - x) + e_kb
                                 for c, (x, y) in enumerate(zip(cuts, cuts[1:]))
                                 if 0 < y % num_kb < e_kb and y - y % num_kb > x and c < dp_tiles])
        assert feasible(plan, units, num_kb, clusters, dp_tiles, e_kb, charged)
        if charged > share:
            assert not feasible(plan, units, num_kb, clusters, dp_tiles, e_kb, charged - 1)


def test_schedule_rules(plan):
    # no workspace, or whole tiles asked for: every tile whole, at most one wave of clusters
    assert schedule(plan, 100, 64, 76, have_ws=False)[:3] == (100, 0, 76)
    assert schedule(plan, 100, 64, 76, mode=SCHED_TILES)[:3] == (100, 0, 76)
    assert schedule(plan, 40, 64, 76, mode=SCHED_TILES)[:3] == (40, 0, 40)
    # AUTO keeps whole tiles when the tiles divide evenly, with fewer than two waves, with short
    # tiles (fp8 4096^3: 32 k-blocks of 128 bytes), or when the last wave idles under 10 %
    assert schedule(plan, 152, 64, 76)[1] == 0
    assert schedule(plan, 100, 64, 76)[1] == 0
    assert schedule(plan, 256, 32, 76)[1] == 0
    assert schedule(plan, 300, 64, 76)[1] == 0        # 1 - 300 / 304 idle
    # ... and splits the last two waves' tiles otherwise: 4096^3 with one-pair clusters
    dp, sk, cl, cuts = schedule(plan, 256, 64, 76)     # 3 waves + 28 tiles: 1 - 256 / 304 idle
    assert (dp, sk, cl) == (2 * 76, (256 - 152) * 64, 76)
    assert cuts[0] == 0 and cuts[-1] == sk and len(cuts) == 77
    # STREAM_K: every tile in the split range, given enough k-blocks per cluster
    dp, sk, cl, cuts = schedule(plan, 64, 16, 76, mode=SCHED_STREAM_K)
    assert (dp, sk, cl) == (0, 64 * 16, 76)
    assert schedule(plan, 1, 8, 76, mode=SCHED_STREAM_K)[1] == 0   # 8 k-blocks < 8 per cluster
    # more clusters than the cut table holds: whole tiles
    big = plan.plan_max_sk_clusters() + 1
    assert schedule(plan, 3 * big + 1, 64, big)[1] == 0


def test_cluster_rules(plan):
    assert plan.plan_choose_cluster(256, 16, PAIRS, QUADS, 1, MCAST_OFF) == 2
    assert plan.plan_choose_cluster(256, 16, PAIRS, QUADS, 0, MCAST_ON) == 2   # A's rows do not split
    assert plan.plan_choose_cluster(256, 16, PAIRS, 0, 1, MCAST_ON) == 2       # no two-pair cluster fits
    assert plan.plan_choose_cluster(256, 15, PAIRS, QUADS, 1, MCAST_ON) == 4
    assert plan.plan_choose_cluster(256, 15, PAIRS, QUADS, 1, MCAST_AUTO) == 2  # odd tile columns
    # AUTO: up to 4 waves of pair tiles take two-pair clusters (144 of 152 SMs), beyond that one-pair
    assert plan.plan_choose_cluster(8 * 16, 16, PAIRS, QUADS, 1, MCAST_AUTO) == 4    # M = 2048, N = 4096
    assert plan.plan_choose_cluster(4 * PAIRS, 16, PAIRS, QUADS, 1, MCAST_AUTO) == 4
    assert plan.plan_choose_cluster(4 * PAIRS + 2, 16, PAIRS, QUADS, 1, MCAST_AUTO) == 2
    assert plan.plan_choose_cluster(32 * 32, 32, PAIRS, QUADS, 1, MCAST_AUTO) == 2   # 8192^3
    # ... and always when they lose no SM pair
    assert plan.plan_choose_cluster(32 * 32, 32, PAIRS, PAIRS // 2, 1, MCAST_AUTO) == 4


def test_tile_choice(plan):
    # forced policies
    assert tile(plan, 4096, 4096, policy=TILE_1SM_256) == (1, 256)
    assert tile(plan, 4096, 4096, policy=TILE_1SM_128) == (1, 128)
    assert tile(plan, 4096, 4096, policy=TILE_PAIR, bn=192) == (2, 192)
    assert tile(plan, 4096, 4096, policy=TILE_PAIR) == (2, 256)
    # no resident pair cluster: one SM per tile, whatever the policy
    assert tile(plan, 4096, 4096, pairs=0)[0] == 1
    assert tile(plan, 4096, 4096, pairs=0, policy=TILE_PAIR)[0] == 1
    # the cost model: large square problems take 256 x 256 pair tiles
    for n in (2048, 4096, 8192):
        assert tile(plan, n, n) == (2, 256)
    # worked by hand from the model: time = ceil(tiles / concurrent tiles) * bn / eff, with eff =
    # min(1, 128 / shared-memory bytes per clock), 4 (4096 + 16 bn) / bn of them for a pair tile and
    # 4 (4096 + 32 bn) / bn for a one-SM tile; the first cheapest of pair 256, pair 128, one-SM 256,
    # one-SM 128 wins.  One wave either way: pair 128 (192) beats pair 256 and one-SM 128 (256).
    assert tile(plan, 128, 4096) == (2, 128)
    assert tile(plan, 512, 512) == (2, 128)
    assert tile(plan, 8192, 256) == (2, 128)
    # with only 8 resident pairs, 1024^3: pair 256 needs 2 waves (512), pair 128 4 (768),
    # one-SM 256 one wave (384), one-SM 128 one wave (256)
    assert tile(plan, 1024, 1024, pairs=8) == (1, 128)


def test_span_bytes_is_the_last_element_plus_one(plan):
    """The byte extent checked against an operand's allocation, against brute force over every
    element's offset (row-major, column-major, padded and broadcast strides)."""
    rng = random.Random(11)
    for _ in range(300):
        rows, cols = rng.randint(0, 9), rng.randint(0, 9)
        s_rows, s_cols = rng.choice([0, 1, cols, cols + 3, 17]), rng.choice([0, 1, rows, rows + 5, 13])
        es = rng.choice([1, 2, 4])
        want = 0 if rows == 0 or cols == 0 else \
            (max(i * s_rows + j * s_cols for i in range(rows) for j in range(cols)) + 1) * es
        assert plan.plan_span_bytes(rows, cols, s_rows, s_cols, es) == want, (rows, cols, s_rows, s_cols, es)
    assert plan.plan_span_bytes(4096, 4096, 4096, 1, 2) == 4096 * 4096 * 2


def test_operand_read_by_tensor_map_when_the_rules_allow(plan):
    """A tensor map needs a 16-byte aligned base, a contiguous inner dimension and an outer pitch
    that is a multiple of 16 bytes (below 2^40); K-contiguous is taken first, then MN-contiguous,
    else the operand goes to the CUDA-core path."""
    base = 1 << 20
    # fp16 A, M x K = 64 x 1000: row-major (K-contiguous, pitch 2000 B), its transpose, a padded pitch
    assert plan.plan_operand_kind(base, 64, 1000, 1000, 1, 2) == 1
    assert plan.plan_operand_kind(base, 64, 1000, 1, 64, 2) == 2
    assert plan.plan_operand_kind(base, 64, 1000, 1008, 1, 2) == 1
    # pitches that are not a multiple of 16 bytes: 1001 fp16, 1002 e4m3, 66 fp16 (MN-contiguous)
    assert plan.plan_operand_kind(base, 64, 1001, 1001, 1, 2) == 0
    assert plan.plan_operand_kind(base, 64, 1002, 1002, 1, 1) == 0
    assert plan.plan_operand_kind(base, 64, 1000, 1, 66, 2) == 0
    # e4m3 needs a 16-element pitch, fp16 an 8-element one
    assert plan.plan_operand_kind(base, 64, 1008, 1008, 1, 1) == 1
    assert plan.plan_operand_kind(base, 64, 1000, 1000, 1, 1) == 0
    # misaligned base (8 bytes off), or neither dimension contiguous
    assert plan.plan_operand_kind(base + 8, 64, 1000, 1000, 1, 2) == 0
    assert plan.plan_operand_kind(base, 64, 1000, 2000, 2, 2) == 0
    # one row: the outer pitch is never used, so any pitch is fine
    assert plan.plan_operand_kind(base, 1, 1000, 7, 1, 2) == 1
    # a pitch of 2^40 bytes is beyond a tensor map's range
    assert plan.plan_operand_kind(base, 64, 8, 1 << 39, 1, 2) == 0
    # when both would do (a square block with both strides legal) the K-contiguous map wins
    assert plan.plan_operand_kind(base, 1, 1, 8, 1, 2) == 1
