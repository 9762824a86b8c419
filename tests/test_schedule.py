"""The kernels' work schedule (csrc/schedule.h), checked on the CPU: every
(tile, k-block) is computed exactly once, split tiles know all their
contributions in k order, partial slots never collide, and stream-K shares
are balanced.  schedule.h is compiled here with g++ exactly as the kernels
include it."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from dense_gemm_10_gb300 import build as gbuild
from dense_gemm_10_gb300 import gemm as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def shim(repo_tmp_module):
    out = repo_tmp_module / "libsched.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
                    "-I" + os.path.join(ROOT, "dense_gemm_10_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "sched_shim.cpp"), "-o", str(out)], check=True)
    lib = ctypes.CDLL(str(out))
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.sched_units.restype = ctypes.c_int
    lib.sched_units.argtypes = [vp, i32, i32, vp, i32]
    lib.sched_contrib_slot.restype = i32
    lib.sched_contrib_slot.argtypes = [vp, vp, i32]
    lib.sched_partial_slots.restype = ctypes.c_int64
    lib.sched_partial_slots.argtypes = [vp]
    lib.sched_set_groups.restype = None
    lib.sched_set_groups.argtypes = [vp, i32]
    return lib


def params(plan_or_tuple):
    """tiles_i tiles_j num_kb raster_group mode split_k dp_tiles sk_slots sk_iters batch."""
    p = plan_or_tuple
    if isinstance(p, tuple):
        return np.array(p + (1,) if len(p) == 9 else p, dtype=np.int64)
    sk_iters = (p.tiles - p.dp_tiles) * p.num_kb if p.schedule == 1 else 0
    return np.array([p.tiles_i, p.tiles_j, p.num_kb, p.raster_group, p.schedule, p.split_k, p.dp_tiles,
                     p.sk_slots, sk_iters, p.batch], dtype=np.int64)


def enumerate_units(lib, prm, slots):
    units = []
    cap = 1 << 16
    buf = np.zeros(12 * cap, dtype=np.int32)
    for s in range(slots):
        n = lib.sched_units(prm.ctypes.data, s, slots, buf.ctypes.data, cap)
        assert n <= cap
        for k in range(n):
            units.append((s, tuple(int(x) for x in buf[12 * k:12 * k + 12])))
    return units


def check_schedule(lib, prm, slots, group_rows=None):
    """group_rows: tile rows of each group of a grouped schedule (else None)."""
    tiles_i, tiles_j, num_kb, _, mode = (int(x) for x in prm[:5])
    batch = int(prm[9])
    tiles = tiles_i * tiles_j * batch if group_rows is None else sum(group_rows) * tiles_j
    units = enumerate_units(lib, prm, slots)
    by_tile = {}
    for s, u in units:
        by_tile.setdefault(u[2], []).append((s, u))
    assert sorted(by_tile) == list(range(tiles)), "every tile exactly once in the schedule"
    pos = {(u[11], u[0], u[1]) for _, u in units}
    if group_rows is None:
        assert len(pos) == tiles and all(0 <= c < batch and 0 <= a < tiles_i and 0 <= b < tiles_j for c, a, b in pos)
        for _, u in units:   # the tile index is batch-major
            assert u[11] == u[2] // (tiles_i * tiles_j)
    else:
        assert len(pos) == tiles and all(0 <= a < group_rows[c] and 0 <= b < tiles_j for c, a, b in pos)
        start = np.concatenate([[0], np.cumsum(group_rows) * tiles_j])
        for _, u in units:   # group-major, every group's tiles in its own range
            assert start[u[11]] <= u[2] < start[u[11] + 1]
    n_pslots = lib.sched_partial_slots(prm.ctypes.data)
    used_pslots = set()
    counters = set()
    for t, lst in by_tile.items():
        lst.sort(key=lambda su: su[1][3])
        assert lst[0][1][3] == 0 and lst[-1][1][4] == num_kb
        for (_, a), (_, b) in zip(lst, lst[1:]):
            assert a[4] == b[3], "k-ranges of a tile are contiguous and disjoint"
        assert all(u[4] > u[3] for _, u in lst)
        if len(lst) == 1:
            assert lst[0][1][5] == 0, "a tile computed in one piece is not partial"
            continue
        ctr = lst[0][1][7]
        assert ctr not in counters
        counters.add(ctr)
        for k, (_, u) in enumerate(lst):
            assert u[5] == 1 and u[8] == len(lst) and u[7] == ctr
            assert 0 <= u[6] < n_pslots and u[6] not in used_pslots
            used_pslots.add(u[6])
        # every contribution enumerates the tile's partial slots in k order
        actual = [u[6] for _, u in lst]
        for _, u in lst:
            arr = np.array(u, dtype=np.int32)
            assert [lib.sched_contrib_slot(prm.ctypes.data, arr.ctypes.data, k) for k in range(len(lst))] == actual
    if mode == 1:
        dp_tiles, sk_slots = int(prm[6]), int(prm[7])
        share = [0] * slots
        for s, u in units:
            if u[2] >= dp_tiles:
                share[s] += u[4] - u[3]
        sk = share[:sk_slots]
        assert max(sk) - min(sk) <= 1, "stream-K shares differ by at most one k-block"
        assert all(x == 0 for x in share[sk_slots:])
    return units


@pytest.mark.parametrize("shape", [(4096, 4096, 4096, 0, 1), (64, 32000, 4096, 0, 1), (8192, 12288, 4096, 0, 0),
                                   (8192, 4096, 16384, 0, 0), (256, 256, 8192, 0, 1), (300, 520, 200, 0, 0),
                                   (1000, 3000, 777, 1, 0), (129, 70000, 64, 0, 1)])
@pytest.mark.parametrize("sm", [148, 152, 160])
def test_planned_schedules(shim, shape, sm):
    gbuild.build()
    M, N, K, ta, tb = shape
    p = G.plan(M, N, K, ta, tb, sm_count=sm)
    check_schedule(shim, params(p), p.grid // p.cluster)


@pytest.mark.parametrize("tiles_i,tiles_j,num_kb,slots,dp_tiles,sk_slots", [
    (3, 5, 7, 4, 12, 4), (1, 1, 64, 64, 0, 64), (1, 1, 5, 5, 0, 5), (2, 3, 64, 7, 0, 7), (16, 16, 64, 76, 228, 75),
    (10, 25, 64, 152, 152, 150), (5, 5, 3, 30, 0, 30), (7, 11, 9, 13, 65, 13)])
def test_stream_k_edge_cases(shim, tiles_i, tiles_j, num_kb, slots, dp_tiles, sk_slots):
    sk_iters = (tiles_i * tiles_j - dp_tiles) * num_kb
    assert sk_slots <= sk_iters
    check_schedule(shim, params((tiles_i, tiles_j, num_kb, 3, 1, 1, dp_tiles, sk_slots, sk_iters)), slots)


@pytest.mark.parametrize("split", [1, 2, 3, 7, 64])
def test_split_k_schedule(shim, split):
    check_schedule(shim, params((4, 6, 64, 5, 0, split, 0, 0, 0)), 9)


@pytest.mark.parametrize("mode", ["tiles", "split", "stream_k"])
def test_grouped_schedules(shim, mode):
    """Groups with different tile-row counts (one empty): every (group, tile,
    k-block) exactly once, found by the group search."""
    rows = [3, 0, 1, 5, 2, 1]
    tj, kb, slots = 4, 7, 9
    table = np.concatenate([[0], np.cumsum(rows) * tj]).astype(np.int32)
    tiles = int(table[-1])
    if mode == "tiles":
        prm = (sum(rows), tj, kb, 2, 0, 1, 0, 0, 0, 1)
    elif mode == "split":
        prm = (sum(rows), tj, kb, 2, 0, 2, 0, 0, 0, 1)
    else:
        dp = (tiles // slots) * slots
        prm = (sum(rows), tj, kb, 2, 1, 1, dp, slots, (tiles - dp) * kb, 1)
    shim.sched_set_groups(table.ctypes.data, len(rows))
    try:
        check_schedule(shim, params(prm), slots, group_rows=rows)
    finally:
        shim.sched_set_groups(None, 0)


@pytest.mark.parametrize("batch", [2, 7, 32])
@pytest.mark.parametrize("mode", ["tiles", "split", "stream_k"])
def test_batched_schedules(shim, batch, mode):
    """A batch extends the tile grid: every (batch, tile, k-block) exactly once."""
    ti, tj, kb, slots = 3, 5, 9, 13
    tiles = ti * tj * batch
    if mode == "tiles":
        prm = (ti, tj, kb, 2, 0, 1, 0, 0, 0, batch)
    elif mode == "split":
        prm = (ti, tj, kb, 2, 0, 3, 0, 0, 0, batch)
    else:
        dp = (tiles // slots) * slots
        iters = (tiles - dp) * kb
        prm = (ti, tj, kb, 2, 1, 1, dp, min(slots, iters), iters, batch)
    check_schedule(shim, params(prm), slots)
