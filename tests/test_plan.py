"""Host model of the work decomposition (no GPU).

For every configuration and mode the units the library would run must cover
each (tile, k-block) of the problem exactly once; the split-K zero slices must
cover every tile row exactly once; and the stream-K / split-K flag protocol,
simulated worker by worker with each worker taking its units in order, must
finish without a worker waiting forever ("SASS-Level Kernel Generation for
Blackwell", paragraph "Stream-K and split-K, added in the L2").
"""
import ctypes
import re
from collections import defaultdict

import numpy as np
import pytest

from dense_fp16_gemm_02_gb300 import build, wgemm

KIND_STORE, KIND_RAISE, KIND_ADD_OWNER, KIND_ADD_ZERO, KIND_ADD_ZEROED = 0, 1, 2, 3, 4
DP, SPLIT, STREAM, HYBRID, ZERO_FIRST = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    build.build()
    return wgemm.load()


def plan(lib, M, N, K, cfg, mode, splits, workers):
    tr, tc = ctypes.c_int(), ctypes.c_int()
    n = lib.wgemm_debug_plan(M, N, K, cfg, mode, splits, workers, None, 0, ctypes.byref(tr),
                             ctypes.byref(tc))
    assert n >= 0, n
    buf = np.zeros(7 * max(n, 1), dtype=np.int32)
    n2 = lib.wgemm_debug_plan(M, N, K, cfg, mode, splits, workers, buf.ctypes.data, n,
                              ctypes.byref(tr), ctypes.byref(tc))
    assert n2 == n
    return buf[:7 * n].reshape(n, 7), tr.value, tc.value




SHAPES = [(1, 1, 1), (300, 520, 200), (1024, 1024, 1024), (1000, 3000, 65),
          (2048, 2048, 16384), (1024, 1024, 65536), (4096, 4096, 1024), (257, 513, 4097)]


def tile_grid(M, N, tr, tc):
    return -(-M // tr), -(-N // tc)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("workers", [1, 7, 76, 152])
def test_data_parallel_covers_each_tile_once(lib, M, N, K, workers):
    for cfg in range(lib.wgemm_num_configs()):
        units, tr, tc = plan(lib, M, N, K, cfg, DP, 1, workers)
        tm, tn = tile_grid(M, N, tr, tc)
        kb = -(-K // 64)
        assert len(units) == tm * tn
        seen = {(int(u[1]), int(u[2])) for u in units}
        assert seen == {(i, j) for i in range(tm) for j in range(tn)}
        assert np.all(units[:, 3] == 0) and np.all(units[:, 4] == kb)
        assert np.all(units[:, 5] == KIND_STORE)


def tma_configs(lib):
    """Configurations that run split-K and stream-K (TMA epilogue, no column
    multicast; a row-multicast cluster is one worker)."""
    return [i for i, n in enumerate(wgemm.config_names())
            if n.endswith("_tma") and not re.match(r"g\dm2_", n)]


def direct_configs(lib):
    return [i for i, n in enumerate(wgemm.config_names()) if n.endswith("_direct")]


def multicast_configs(lib):
    """Column-multicast clusters (groups side by side sharing A): data parallel only."""
    return [i for i, n in enumerate(wgemm.config_names()) if re.match(r"g\dm2_", n)]


def coverage(units, tm, tn, kb):
    hits = defaultdict(int)
    for u in units:
        assert 0 <= u[1] < tm and 0 <= u[2] < tn and u[0] == u[0]
        assert 0 <= u[3] < u[4] <= kb
        for k in range(int(u[3]), int(u[4])):
            hits[(int(u[1]), int(u[2]), k)] += 1
    return hits


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("splits", [1, 2, 3, 9, 64])
def test_split_k_covers_each_kblock_once(lib, M, N, K, splits):
    for cfg in tma_configs(lib):
        units, tr, tc = plan(lib, M, N, K, cfg, SPLIT, splits, 76)
        tm, tn = tile_grid(M, N, tr, tc)
        kb = -(-K // 64)
        s_eff = min(splits, kb)
        hits = coverage(units, tm, tn, kb)
        assert len(hits) == tm * tn * kb and set(hits.values()) == {1}
        assert np.all(units[:, 5] == KIND_ADD_ZERO)
        sizes = units[:, 4] - units[:, 3]
        assert sizes.max() - sizes.min() <= 1  # near-equal contiguous ranges
        # Each tile's splits are 0..S-1 once each.
        per_tile = defaultdict(list)
        for u in units:
            per_tile[int(u[0])].append(int(u[6]))
        assert all(sorted(v) == list(range(s_eff)) for v in per_tile.values())


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("workers", [1, 5, 76, 300])
def test_stream_k_covers_each_kblock_once(lib, M, N, K, workers):
    for cfg in tma_configs(lib):
        units, tr, tc = plan(lib, M, N, K, cfg, STREAM, 1, workers)
        tm, tn = tile_grid(M, N, tr, tc)
        kb = -(-K // 64)
        hits = coverage(units, tm, tn, kb)
        assert len(hits) == tm * tn * kb and set(hits.values()) == {1}
        # Exactly one unit per tile starts at k-block 0, and it stores.
        starts = defaultdict(int)
        for u in units:
            if u[3] == 0:
                starts[int(u[0])] += 1
                assert u[5] in (KIND_STORE, KIND_RAISE)
            else:
                assert u[5] == KIND_ADD_OWNER
        assert len(starts) == tm * tn and set(starts.values()) == {1}




@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("workers", [1, 5, 76, 300])
def test_stream_k_zero_first(lib, M, N, K, workers):
    """Stream-K with zeroing first: the same units as stream-K (each
    (tile, k-block) once, the same ranges), but the unit holding a tile's
    first k-block zeroes the tile (kind 3, split 0) and every other part of a
    split tile adds after the zeroing (kind 4); a whole tile is stored. Every
    zeroing unit's flag is raised at kernel start, so no unit waits on
    another's main loop."""
    for cfg in tma_configs(lib):
        units, tr, tc = plan(lib, M, N, K, cfg, ZERO_FIRST, 1, workers)
        plain, _, _ = plan(lib, M, N, K, cfg, STREAM, 1, workers)
        assert np.array_equal(units[:, [0, 1, 2, 3, 4, 6]], plain[:, [0, 1, 2, 3, 4, 6]])
        tm, tn = tile_grid(M, N, tr, tc)
        kb = -(-K // 64)
        hits = coverage(units, tm, tn, kb)
        assert len(hits) == tm * tn * kb and set(hits.values()) == {1}
        for u in units:
            whole = u[3] == 0 and u[4] == kb
            if whole:
                assert u[5] == KIND_STORE
            elif u[3] == 0:
                assert u[5] == KIND_ADD_ZERO and u[6] == 0
            else:
                assert u[5] == KIND_ADD_ZEROED
        # Every split tile has exactly one zeroing unit.
        split_tiles = {int(u[0]) for u in units if u[5] in (KIND_ADD_ZERO, KIND_ADD_ZEROED)}
        zeroers = [int(u[0]) for u in units if u[5] == KIND_ADD_ZERO]
        assert sorted(zeroers) == sorted(split_tiles)


def simulate_stream_k(per_worker):
    """Each worker runs its units in order; an add-after-owner unit can finish
    only after its tile's owner unit finished. Returns True if every worker
    finishes (no deadlock)."""
    pos = [0] * len(per_worker)
    owner_done = set()
    progress = True
    while progress:
        progress = False
        for w, units in enumerate(per_worker):
            while pos[w] < len(units):
                u = units[pos[w]]
                if u[5] == KIND_ADD_OWNER and int(u[0]) not in owner_done:
                    break
                if u[5] in (KIND_RAISE, KIND_STORE):
                    owner_done.add(int(u[0]))
                pos[w] += 1
                progress = True
    return all(p == len(u) for p, u in zip(pos, per_worker))


def split_by_worker(lib, M, N, K, cfg, mode, splits, workers):
    """Per-worker lists: ask the library for each single worker count prefix.
    The worker-major listing is cut where the worker id changes, which we
    recover from the data-independent rule: stream-K ranges are contiguous in
    (tile, k) order and each worker walks its range downwards."""
    units, tr, tc = plan(lib, M, N, K, cfg, mode, splits, workers)
    kb = -(-K // 64)
    lists, cur, last_key = [], [], None
    for u in units:
        key = int(u[0]) * kb + int(u[3])
        # Within one worker the global iteration index strictly decreases.
        if cur and key > last_key:
            lists.append(cur)
            cur = []
        cur.append(u)
        last_key = key
    if cur:
        lists.append(cur)
    return lists


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 16384), (257, 513, 4097), (1024, 1024, 65536),
                                   (300, 520, 200)])
@pytest.mark.parametrize("workers", [3, 76, 74])
def test_stream_k_protocol_finishes(lib, M, N, K, workers):
    for cfg in tma_configs(lib):
        lists = split_by_worker(lib, M, N, K, cfg, STREAM, 1, workers)
        # A worker's first unit waits only when it is the worker's only unit
        # (a range inside one tile); every owner unit is its worker's first.
        for lst in lists:
            assert lst[0][5] != KIND_ADD_OWNER or len(lst) == 1
            assert all(u[5] != KIND_RAISE for u in lst[1:])
        assert simulate_stream_k(lists)


def hybrid_lists(units, workers, dp_waves, tail_tiles, kb):
    """Per-worker unit lists of a data-parallel + stream-K-tail plan, cut from
    the worker-major listing by the plan's definition: dp_waves whole tiles
    per worker, then one unit per tail tile that the worker's near-equal range
    [⌊T·w/P⌋, ⌊T·(w+1)/P⌋) of the T = tail_tiles·kb tail iterations touches."""
    T, lists, pos = tail_tiles * kb, [], 0
    for w in range(workers):
        b, e = T * w // workers, T * (w + 1) // workers
        n_tail = 0 if e <= b else (e - 1) // kb - b // kb + 1
        lists.append(units[pos:pos + dp_waves + n_tail])
        pos += dp_waves + n_tail
    assert pos == len(units)
    return lists


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (8192, 2048, 4096), (4096, 4096, 1024),
                                   (2600, 3000, 700), (257, 513, 4097), (300, 520, 200)])
@pytest.mark.parametrize("workers", [3, 74, 76, 152])
@pytest.mark.parametrize("held", [1, 2, 5])
def test_hybrid_waves_and_stream_k_tail(lib, M, N, K, workers, held):
    # Whole waves of tiles run data parallel, one tile per worker per wave in
    # tile order; the partial last wave (and held − 1 full waves before it)
    # goes to stream-K. Every (tile, k-block) once, one owner per tail tile,
    # and the flag protocol finishes.
    for cfg in tma_configs(lib):
        units, tr, tc = plan(lib, M, N, K, cfg, HYBRID, held, workers)
        tm, tn = tile_grid(M, N, tr, tc)
        tiles, kb = tm * tn, -(-K // 64)
        hits = coverage(units, tm, tn, kb)
        assert len(hits) == tiles * kb and set(hits.values()) == {1}
        if tiles < workers:
            continue  # no whole wave: plain stream-K, covered above
        dp_waves = max(0, tiles // workers - (held - 1))
        dp_tiles = dp_waves * workers
        lists = hybrid_lists(units, workers, dp_waves, tiles - dp_tiles, kb)
        for w, lst in enumerate(lists):
            for i in range(dp_waves):
                u = lst[i]
                assert u[0] == w + i * workers and u[3] == 0 and u[4] == kb
                assert u[5] == KIND_STORE
            tail = lst[dp_waves:]
            assert all(u[0] >= dp_tiles for u in tail)
            # The tail walks its range downwards: an owner unit comes first.
            assert all(u[5] != KIND_RAISE for u in tail[1:])
            assert len(tail) == 0 or tail[0][5] != KIND_ADD_OWNER or len(tail) == 1
        starts = defaultdict(int)
        for u in units:
            if u[3] == 0:
                starts[int(u[0])] += 1
        assert len(starts) == tiles and set(starts.values()) == {1}
        assert simulate_stream_k(lists)


def test_hybrid_rejects_bad_arguments(lib):
    cfg = tma_configs(lib)[0]
    assert lib.wgemm_debug_plan(4096, 4096, 4096, cfg, HYBRID, 0, 76, None, 0, None, None) == -6
    for c in direct_configs(lib) + multicast_configs(lib):
        assert lib.wgemm_debug_plan(4096, 4096, 4096, c, HYBRID, 1, 76, None, 0, None,
                                    None) == -6


@pytest.mark.parametrize("M,N,K,S", [(1024, 1024, 65536, 9), (300, 520, 200, 3),
                                     (257, 513, 4097, 5)])
def test_split_k_zero_slices_partition_rows(lib, M, N, K, S):
    # plan_zero_rows: the S slices of a tile's rows are disjoint and cover it.
    for tile_rows in (64, 128, 256):
        for s_eff in range(1, S + 1):
            per = -(-tile_rows // s_eff)
            covered = []
            for s in range(s_eff):
                r0, r1 = min(s * per, tile_rows), min((s + 1) * per, tile_rows)
                covered += list(range(r0, r1))
            assert covered == list(range(tile_rows))


def test_multicast_configs_are_data_parallel_only(lib):
    for cfg in multicast_configs(lib):
        for mode, s in ((SPLIT, 4), (STREAM, 1)):
            assert lib.wgemm_debug_plan(1024, 1024, 4096, cfg, mode, s, 38, None, 0, None,
                                        None) == -6


def test_direct_epilogue_configs_reject_split_modes(lib):
    for cfg in direct_configs(lib):
        n = lib.wgemm_debug_plan(1024, 1024, 4096, cfg, SPLIT, 4, 76, None, 0, None, None)
        assert n == -6
        n = lib.wgemm_debug_plan(1024, 1024, 4096, cfg, STREAM, 1, 76, None, 0, None, None)
        assert n == -6


def test_16bit_output_and_fused_configs_are_data_parallel_only(lib):
    for cfg, name in enumerate(wgemm.config_names()):
        if not name.endswith("_h") and "_ab" not in name:
            continue
        assert lib.wgemm_debug_plan(1024, 1024, 4096, cfg, DP, 1, 76, None, 0, None, None) > 0
        for mode, sp in ((SPLIT, 4), (STREAM, 1), (HYBRID, 1)):
            assert lib.wgemm_debug_plan(1024, 1024, 4096, cfg, mode, sp, 76, None, 0, None,
                                        None) == -6
