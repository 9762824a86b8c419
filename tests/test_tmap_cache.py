"""The per-handle tensor-map cache (csrc/tmap_cache.h), checked on the CPU with a
stand-in encoder: an identical description is a hit and returns the map made
for it; a change in any field (base address, an extent, a stride, the box, the
type, the swizzle, the L2 promotion) is a miss; a failed encoding is not kept;
and a full set replaces its least recently used entry."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def shim(repo_tmp_module):
    out = repo_tmp_module / "libtmap.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-fPIC", "-shared",
                    "-I" + os.path.join(ROOT, "dense_gemm_10_gb300", "csrc"), "-I/usr/local/cuda/include",
                    os.path.join(ROOT, "tests", "tmap_shim.cpp"), "-o", str(out)], check=True)
    lib = ctypes.CDLL(str(out))
    vp = ctypes.c_void_p
    lib.tmap_get.restype = ctypes.c_int
    lib.tmap_get.argtypes = [ctypes.c_uint64, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
    lib.tmap_stats.argtypes = [vp, vp, vp]
    lib.tmap_fail_next.argtypes = [ctypes.c_int]
    return lib


BASE = dict(base=0x7f0000001000, dims=(4096, 4096, 1), strides=(8192, 8192 * 4096), box=(64, 128, 1),
            dtype=10, swizzle=3, promo=2)


def get(lib, **kw):
    d = dict(BASE, **kw)
    dims = np.array(d["dims"], dtype=np.uint64)
    strides = np.array(d["strides"], dtype=np.uint64)
    box = np.array(d["box"], dtype=np.uint32)
    out = np.zeros(2, dtype=np.uint64)
    ok = lib.tmap_get(d["base"], dims.ctypes.data, strides.ctypes.data, box.ctypes.data, d["dtype"],
                      d["swizzle"], d["promo"], out.ctypes.data)
    return ok, int(out[0]), int(out[1])


def stats(lib):
    h, m, e = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_int()
    lib.tmap_stats(ctypes.byref(h), ctypes.byref(m), ctypes.byref(e))
    return h.value, m.value, e.value


def test_identical_description_hits(shim):
    shim.tmap_reset()
    ok, base, serial = get(shim)
    assert ok and base == BASE["base"] and serial == 1
    for _ in range(5):
        assert get(shim) == (1, BASE["base"], 1)     # the map made the first time
    assert stats(shim) == (5, 1, 1)


@pytest.mark.parametrize("field,value", [("base", 0x7f0000002000), ("dims", (4096, 4097, 1)),
                                         ("dims", (4096, 4096, 2)), ("strides", (8208, 8208 * 4096)),
                                         ("strides", (8192, 8192 * 4097)), ("box", (64, 256, 1)),
                                         ("dtype", 9), ("swizzle", 0), ("promo", 0)])
def test_any_changed_field_misses(shim, field, value):
    shim.tmap_reset()
    get(shim)
    ok, _, serial = get(shim, **{field: value})
    assert ok and serial == 2
    assert stats(shim) == (0, 2, 2)
    assert get(shim)[2] == 1 and get(shim, **{field: value})[2] == 2   # both kept
    assert stats(shim)[:2] == (2, 2)


def test_failed_encoding_is_not_kept(shim):
    shim.tmap_reset()
    shim.tmap_fail_next(1)
    assert get(shim)[0] == 0
    shim.tmap_fail_next(0)
    ok, _, serial = get(shim)
    assert ok and serial == 1 and stats(shim) == (0, 2, 1)


def test_many_buffers_keep_the_recent_ones(shim):
    """More descriptions than the cache holds (256 = 64 sets of 4): every set
    keeps its four most recent entries, so the last four descriptions are
    always there, and the cache never answers with a map made for another
    description."""
    shim.tmap_reset()
    bases = [0x7f0000000000 + 0x100000 * i for i in range(600)]
    for b in bases:
        ok, got, _ = get(shim, base=b)
        assert ok and got == b
    assert stats(shim) == (0, 600, 600)
    for b in reversed(bases[-4:]):
        assert get(shim, base=b)[1] == b
    assert stats(shim)[0] == 4
    held = 0
    for b in reversed(bases[-256:]):   # most recent first: a lookup refreshes only its own entry
        h0 = stats(shim)[0]
        assert get(shim, base=b)[1] == b
        held += stats(shim)[0] - h0
    assert 64 <= held <= 256
