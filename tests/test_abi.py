"""The C ABI, without a GPU: the library loads, exports every entry point the
header declares, refuses bad arguments, and plans calls as designed."""
import ctypes
import os
import re

import pytest
import torch

from dense_gemm_10_gb300 import build as gbuild
from dense_gemm_10_gb300 import gemm as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_gb300.h")


@pytest.fixture(scope="module", autouse=True)
def built_library():
    gbuild.build()
    return G.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(gemm_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("gemm_create", "gemm_run", "gemm_destroy", "gemm_get_status", "gemm_plan"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(G.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding's signature table covers the header exactly
    assert sorted(G.SIGNATURES) == declared_functions()


def test_status_strings():
    for code in range(8):
        s = G.lib().gemm_status_string(code)
        assert s and s != b"unknown status"
    assert G.lib().gemm_status_string(99) == b"unknown status"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_create_without_gpu_reports_no_device():
    h = ctypes.c_void_p()
    assert G.lib().gemm_create(ctypes.byref(h), 0) == G.ERR_NO_DEVICE
    assert h.value is None
    assert G.lib().gemm_create(None, 0) == G.ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_noalloc_status_without_gpu_reports_no_device():
    word = ctypes.c_int32(-1)
    assert G.lib().gemm_noalloc_get_status(None, ctypes.byref(word)) == G.ERR_NO_DEVICE


def test_noalloc_options_are_checked():
    """Only the wait limit and the test hook are options of the no-allocation
    path; out-of-range values and other options are refused on the host."""
    L = G.lib()
    assert L.gemm_noalloc_set_option(G.OPT_WAIT_LIMIT_NS, 999_999) == G.ERR_INVALID_ARG
    assert L.gemm_noalloc_set_option(G.OPT_TEST_DROP_LOAD, -1) == G.ERR_INVALID_ARG
    for opt in (G.OPT_FORCE_PATH, G.OPT_SPLIT_K, G.OPT_PDL, 99):
        assert L.gemm_noalloc_set_option(opt, 0) == G.ERR_INVALID_ARG
    assert L.gemm_noalloc_set_option(G.OPT_WAIT_LIMIT_NS, 2_000_000_000) == G.OK
    assert L.gemm_noalloc_set_option(G.OPT_TEST_DROP_LOAD, 0) == G.OK


def test_null_handle_is_rejected():
    assert G.lib().gemm_run(None, 0, 0, 4, 4, 4, 1.0, 0x1000, 4, 0x1000, 4, 0.0, 0x1000, 4, 0, None) \
        == G.ERR_INVALID_ARG
    assert G.lib().gemm_destroy(None) == G.OK
    assert G.lib().gemm_set_option(None, 0, 10**9) == G.ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(G, "_lib", None)
    monkeypatch.setattr(G, "LIB_PATH", "/nonexistent/libgemm_gb300.so")
    with pytest.raises(RuntimeError, match="not built"):
        G.lib()


def test_product_code_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "dense_gemm_10_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b|liboracle|oracle_gemm", text, flags=re.M), \
                    os.path.join(dirpath, f)


# ----------------------------------------------------------------- planner --

def test_plan_square_nt():
    """4096^3: 256 x 256 tiles on CTA pairs; the tiles of an incomplete last
    wave are shared by stream-K."""
    p = G.plan(4096, 4096, 4096, 0, 1)
    assert p.path == G.PATH_TC_2CTA and p.swap_ab == 0
    assert p.cluster == 2
    assert p.a_kmajor == 1 and p.b_kmajor == 1
    assert p.bm == 256 and p.bk == 64 and p.bn == 256 and p.num_kb == 64
    assert p.tiles_i == 16 and p.tiles_j == 16 and p.tiles == p.tiles_i * p.tiles_j
    slots = 152 // p.cluster
    assert p.schedule == G.SCHED_STREAM_K and p.dp_tiles == (p.tiles // slots) * slots and 0 < p.sk_slots <= slots
    assert p.grid == 152 and p.repack_a == 0 and p.repack_b == 0
    assert p.vector_store == 1 and p.launches == 1
    assert p.workspace_bytes >= p.sk_slots * 2 * p.cluster * 256 * 128 * 4   # partial slots x CTAs


@pytest.mark.parametrize("ta,tb,ak,bk", [(0, 0, 1, 0), (0, 1, 1, 1), (1, 0, 0, 0), (1, 1, 0, 1)])
def test_plan_major_modes(ta, tb, ak, bk):
    p = G.plan(4096, 4096, 4096, ta, tb, G.F16_F32, beta=0.5)
    assert (p.a_kmajor, p.b_kmajor) == (ak, bk)


def test_plan_lm_head_swaps():
    """M = 64: the vocabulary rides on the MMA's M (swap-AB), 128 vocabulary rows
    against the 64 activation rows per tile.  The GEMM is bound by HBM: whole
    tiles would stream from only 125 of the 152 SMs (two waves), so the 98
    tiles past the first full wave are shared out by stream-K and every SM
    streams."""
    p = G.plan(64, 32000, 4096, 0, 1)
    assert p.swap_ab == 1 and p.path == G.PATH_TC_1CTA and p.cluster == 1
    assert p.a_kmajor == 1 and p.b_kmajor == 1   # MMA A = weights (N x K), MMA B = activations (M x K)
    assert p.bm == 128 and p.bn == 64 and p.tiles == 250
    assert p.schedule == G.SCHED_STREAM_K and p.grid == 152 and p.dp_tiles == 152


def test_plan_hbm_bound_full_waves_keep_whole_tiles():
    """An HBM-bound GEMM whose whole tiles keep at least nine tenths of the
    slots busy gets no stream-K tail (it would add only partial-sum traffic)."""
    p = G.plan(64, 38912, 4096, 0, 1)   # 304 tiles of 128 rows: two full waves on 152 SMs
    assert p.swap_ab == 1 and p.schedule == G.SCHED_TILES and p.grid == 152


def test_plan_compute_bound_keeps_stream_k():
    """Above the machine balance the last partial wave is shared out (stream-K)."""
    p = G.plan(4096, 4096, 4096, 0, 1)
    assert p.schedule == G.SCHED_STREAM_K and p.path == G.PATH_TC_2CTA and p.grid == 152


def test_plan_bulk_store_paths():
    """C leaves through bulk tensor stores of rows (beta != 0 too: the old C
    arrives by tensor loads into the same staging), of transposed blocks for a
    swapped problem with beta == 0, by per-row bulk copies (misaligned rows or
    a partial 16-byte piece at the right edge, beta == 0), or directly (the
    same with beta != 0, or a swapped problem with beta != 0)."""
    assert G.plan(4096, 4096, 4096, 0, 1).bulk_store == G.BULK_ROWS
    assert G.plan(64, 32000, 4096, 0, 1).bulk_store == G.BULK_TRANSPOSED
    assert G.plan(64, 32000, 4096, 0, 1, G.BF16_BF16).bulk_store == G.BULK_TRANSPOSED
    for ta, tb in ((0, 0), (0, 1), (1, 0), (1, 1)):
        assert G.plan(4096, 4096, 4096, ta, tb, G.F16_F32, beta=0.5).bulk_store == G.BULK_ROWS
    assert G.plan(4096, 4096, 4096, 0, 1, G.BF16_BF16, beta=0.5).bulk_store == G.BULK_ROWS
    assert G.plan(64, 32000, 4096, 0, 1, beta=1.0).bulk_store == G.BULK_NONE
    assert G.plan(512, 1002, 256, 0, 1).bulk_store == G.BULK_ROW_CLASSES   # 4008-byte rows
    assert G.plan(512, 1002, 256, 0, 1, G.BF16_BF16).bulk_store == G.BULK_ROW_COPIES
    assert G.plan(512, 1002, 256, 0, 1, beta=0.5).bulk_store == G.BULK_NONE
    assert G.plan(512, 1004, 256, 0, 1, ldc=1008).bulk_store == G.BULK_ROWS
    assert G.plan(512, 1004, 256, 0, 1, C=0x1004, ldc=1008).bulk_store == G.BULK_ROW_CLASSES
    assert G.plan(40, 1001, 256, 0, 1, G.BF16_BF16, ldc=1008).bulk_store == G.BULK_NONE


def test_plan_misaligned_c():
    """C that bulk tensor stores cannot write (misaligned rows, or rows ending
    inside a 16-byte piece), beta == 0, unswapped.  fp32 C of one GEMM: the
    rows fall into 1, 2 or 4 classes of one misalignment each, one tensor store
    per class and block.  Otherwise a large C of one GEMM with a short K
    (epilogue-bound) goes through an aligned copy in the workspace and a copy
    kernel (one more launch), and the rest leaves through per-row bulk copies.
    beta != 0, 8-bit C and swapped problems keep direct stores."""
    p = G.plan(4095, 4097, 1000, 0, 0, ldb=4097, ldc=4097)       # the ragged 4095 x 4097 x 1000 workload
    assert p.bulk_store == G.BULK_ROW_CLASSES and p.launches == 2 and p.repack_b == 1
    assert p.workspace_bytes < 1000 * 4104 * 2 + (1 << 20)        # the repacked B only
    assert G.plan(4096, 4097, 4096, 0, 1, ldc=4097).bulk_store == G.BULK_ROW_CLASSES
    p = G.plan(2048, 1001, 512, 0, 1, ldc=1008)                 # aligned rows ending inside a piece: one class
    assert p.bulk_store == G.BULK_ROW_CLASSES and p.launches == 1
    p = G.plan(2048, 1001, 512, 0, 1, G.BF16_BF16, ldc=1008)    # 16-bit C, short K: the workspace copy
    assert p.bulk_store == G.BULK_STAGED and p.launches == 2
    p = G.plan(2048, 1024, 2048, 0, 1, G.BF16_BF16, C=0x1002)   # 16-bit C, misaligned base, K = 2048
    assert p.bulk_store == G.BULK_ROW_COPIES
    assert G.plan(1000, 1001, 512, 0, 1, G.BF16_BF16, ldc=1008).bulk_store == G.BULK_ROW_COPIES   # small C
    assert G.plan(3, 2, 512, 0, 1, ldc=3).bulk_store == G.BULK_ROW_COPIES   # fewer rows than classes
    assert G.plan(2048, 1001, 512, 0, 1, ldc=1008, beta=0.5).bulk_store == G.BULK_NONE
    assert G.plan(2048, 1001, 512, 0, 1, G.fp8_dtype("e4m3", "e4m3", "e4m3"), ldc=1008).bulk_store == G.BULK_NONE
    assert G.plan(64, 32001, 4096, 0, 1, ldc=32008).swap_ab == 1
    assert G.plan(64, 32001, 4096, 0, 1, ldc=32008).bulk_store == G.BULK_NONE  # swapped
    pb = G.plan_batched(1000, 1001, 256, 3, ldc=1001)           # strided batches: per-row copies
    assert pb.bulk_store == G.BULK_ROW_COPIES


def test_plan_epilogue_warps():
    """The 256-wide CTA-pair tile has a kernel with eight epilogue warps, taken
    where C leaves through row classes, per-row copies or direct stores; with
    bulk tensor stores (and for other tiles) the four-warp kernel stays."""
    p = G.plan(4095, 4097, 1000, 0, 0, ldb=4097, ldc=4097)       # row classes
    assert p.bulk_store == G.BULK_ROW_CLASSES and p.bm == 256 and p.bn == 256 and p.epilogue_warps == 8
    p = G.plan(4095, 4097, 1000, 0, 0, ldb=4104, ldc=4100)       # aligned rows ending inside a piece
    assert p.bulk_store == G.BULK_ROW_CLASSES and p.epilogue_warps == 8
    p = G.plan(4096, 4096, 4096, 0, 0, G.F16_F16, ldc=4100, beta=0.5)   # beta != 0, 16-bit C: direct stores
    assert p.bulk_store == G.BULK_NONE and p.epilogue_warps == 8
    for args, kw in (((4096, 4096, 4096, 0, 1), {}),                       # bulk rows
                     ((4096, 4096, 4096, 1, 0, G.F16_F16), {"beta": 0.5}),  # bulk rows with the blend
                     ((64, 32000, 4096, 0, 1), {}),                        # swapped, 64-wide tiles
                     ((2048, 1001, 512, 0, 1, G.BF16_BF16), {"ldc": 1008})):  # the aligned workspace copy
        q = G.plan(*args, **kw)
        assert q.epilogue_warps == 4, (args, q.as_dict())
    # a 256-wide CTA-pair tile with eight warps keeps at least two ring stages
    assert 2 <= p.stages < G.plan(4096, 4096, 4096, 0, 1).stages


def test_plan_fp8():
    """8-bit inputs: 128-element k-slices (one 128-byte swizzle row), the 8-bit
    tile configurations, rows aligned to 16 elements, and K-major operands only."""
    p = G.plan(4096, 4096, 4096, 0, 1, G.E4M3_F32)
    assert p.path == G.PATH_TC_2CTA and p.bn == 256 and p.bk == 128 and p.num_kb == 32
    s = G.plan(64, 32000, 4096, 0, 1, G.fp8_dtype("e4m3", "e5m2", "bf16"))
    assert s.swap_ab == 1 and s.bn == 64 and s.kdepth == 2 and s.bk == 256 and s.bulk_store == G.BULK_TRANSPOSED
    assert G.plan(300, 520, 301, 0, 1, G.E5M2_F32, lda=304, ldb=320).repack_a == 0
    r = G.plan(300, 520, 301, 0, 1, G.E5M2_F32, lda=305, ldb=320)
    assert r.repack_a == 1 and r.repack_b == 0 and r.workspace_bytes >= 300 * 304   # rows padded to 16 bytes
    for ta, tb in [(0, 0), (1, 0), (1, 1)]:
        with pytest.raises(G.GemmError) as e:
            G.plan(256, 256, 256, ta, tb, G.E4M3_F32)
        assert e.value.status == G.ERR_UNSUPPORTED
    for bad in (8, 15, 32):
        with pytest.raises(G.GemmError) as e:
            G.plan(256, 256, 256, 0, 1, bad)
        assert e.value.status == G.ERR_INVALID_ARG
    assert [G.fp8_dtype(a, b, c) for c in ("f32", "bf16", "f16", "e4m3") for b in ("e4m3", "e5m2")
            for a in ("e4m3", "e5m2")] == list(range(16, 32))


def test_plan_block_scaled():
    """Block-scaled operands are written as bf16 first (two more launches), then
    the bf16 GEMM plans as usual; block-scaled types need their entry point."""
    p = G.plan_block_scaled(4096, 4096, 4096, G.mxfp8_dtype())
    assert p.repack_a == 1 and p.repack_b == 1 and p.launches == 3 and p.bk == 64 and p.bn == 256
    assert p.workspace_bytes >= 2 * 4096 * 4096 * 2
    # M <= 64: the weights B stay in their codes and the GEMM converts them (the
    # pass only for A); misaligned code or scale rows keep the pass for both
    q = G.plan_block_scaled(64, 32000, 4096, G.NVFP4_BF16)
    assert q.swap_ab == 1 and q.launches == 2 and q.repack_b == 0 and q.repack_a == 1
    assert q.bn == 64 and q.bm == 128 and q.kdepth == 1 and q.path == G.PATH_TC_1CTA
    assert q.workspace_bytes < 32000 * 4096                       # no 16-bit copy of B (2 x 131 MB)
    assert G.plan_block_scaled(64, 32000, 4096, G.mxfp8_dtype()).launches == 2
    assert G.plan_block_scaled(64, 32000, 4096, G.NVFP4_BF16, ldb=4128).launches == 2    # 2064-byte code rows
    assert G.plan_block_scaled(64, 32000, 4096, G.NVFP4_BF16, ldb=4104).launches == 3   # 2052-byte code rows
    assert G.plan_block_scaled(64, 32000, 4096, G.NVFP4_BF16, ld_sfb=264).launches == 3  # scale rows
    assert G.plan_block_scaled(64, 32000, 4096, G.NVFP4_BF16, SFB=0x1008).launches == 3
    assert G.plan_block_scaled(64, 32000, 4096, G.mxfp8_dtype(), ldb=4100).launches == 3
    r = G.plan_block_scaled(300, 264, 37, G.NVFP4_F32, lda=38, ldb=38)
    assert r.workspace_bytes >= (300 + 264) * 48 * 2          # 37 values padded to 48 bf16
    for kw in (dict(ld_sfa=1), dict(lda=39)):                  # scale rows too short; odd FP4 pitch
        with pytest.raises(G.GemmError) as e:
            G.plan_block_scaled(64, 64, 64, G.NVFP4_F32, **kw)
        assert e.value.status == G.ERR_INVALID_ARG
    with pytest.raises(G.GemmError) as e:
        G.plan(64, 64, 64, 0, 1, G.NVFP4_F32)
    assert e.value.status == G.ERR_INVALID_ARG
    assert [G.mxfp8_dtype(a, b, c) for c in ("f32", "bf16", "f16") for b in ("e4m3", "e5m2")
            for a in ("e4m3", "e5m2")] == list(range(32, 44))


def test_plan_fp32():
    """fp32 inputs: 32-element (128-byte) k-slices of the TF32 kind, K-major only.
    The fp32 GEMM writes both operands as two TF32 segments (K rounded up to a
    whole k-slice each) and runs one GEMM over three segments; one-pass TF32
    reads aligned K-major operands as they are and writes only the others."""
    p = G.plan(4096, 4096, 4096, 0, 1, G.F32_F32)
    assert p.path == G.PATH_TC_2CTA and p.bn == 256 and p.bk == 32 and p.num_kb == 3 * 4096 // 32
    assert p.repack_a == 1 and p.repack_b == 1 and p.launches == 3 and p.a_kmajor == 1 and p.b_kmajor == 1
    assert 2 * 4096 * 2 * 4096 * 4 <= p.workspace_bytes < 2 * 4096 * 3 * 4096 * 4
    t = G.plan(4096, 4096, 4096, 0, 1, G.TF32_F32)
    assert t.bk == 32 and t.num_kb == 128 and t.repack_a == 0 and t.repack_b == 0 and t.launches == 1
    for ta, tb in [(0, 0), (1, 0), (1, 1)]:   # MN-major operands are written K-major first
        u = G.plan(256, 264, 300, ta, tb, G.TF32_F32)
        assert (u.repack_a, u.repack_b) == (ta, 1 - tb) and u.a_kmajor == 1 and u.b_kmajor == 1
        assert u.launches == 1 + ta + (1 - tb)
    r = G.plan(300, 520, 301, 0, 1, G.F32_F32, lda=301, ldb=301)
    assert r.bk == 32 * r.kdepth and r.num_kb == -(-3 * 320 // r.bk)   # segments of 301 -> 320
    assert r.workspace_bytes >= (300 + 520) * 640 * 4          # two segments of 320 values a row
    v = G.plan(300, 520, 301, 0, 1, G.TF32_F32, lda=301, ldb=304)
    assert v.repack_a == 1 and v.repack_b == 0                 # 1204-byte rows: not 16-byte aligned
    s = G.plan(16, 4096, 4096, 0, 1, G.F32_F32)
    assert s.swap_ab == 1 and s.bn == 64



def test_plan_e4m3_output():
    """E4M3 C (quantised output): written only, by the direct-store epilogue."""
    for dt in (G.BF16_E4M3, G.F16_E4M3, G.fp8_dtype("e4m3", "e4m3", "e4m3")):
        p = G.plan(4096, 4096, 4096, 0, 1, dt)
        assert p.bulk_store == G.BULK_NONE and p.vector_store == 1
        with pytest.raises(G.GemmError) as e:
            G.plan(256, 256, 256, 0, 1, dt, beta=0.5)
        assert e.value.status == G.ERR_UNSUPPORTED
    assert G.plan(256, 256, 256, 0, 1, G.BF16_E4M3, ldc=260).vector_store == 0   # 260-byte rows


def test_plan_strided_batched():
    """A batch extends the tile grid; a stride of 0 shares one operand; C
    batches may not overlap; misaligned batch strides repack every batch."""
    p = G.plan_batched(2048, 2048, 128, 32, 0, 1, G.BF16_BF16)      # attention scores, 32 heads
    assert p.batch == 32 and p.tiles == p.tiles_i * p.tiles_j * 32 and p.num_kb == 2
    one = G.plan(2048, 2048, 128, 0, 1, G.BF16_BF16)
    assert one.batch == 1 and one.tiles == one.tiles_i * one.tiles_j
    s = G.plan_batched(64, 4096, 1024, 8, 0, 1, strideB=0)           # B shared, skinny M
    assert s.swap_ab == 1 and s.batch == 8 and s.repack_a == 0 and s.repack_b == 0
    r = G.plan_batched(100, 96, 64, 3, 0, 1, strideA=100 * 64 + 4)   # 8-byte gap: not 16-byte aligned
    assert r.repack_a == 1 and r.workspace_bytes >= 3 * 100 * 64 * 2
    assert G.plan_batched(100, 96, 64, 3, 0, 1, strideC=100 * 96 + 2).vector_store == 0   # 8-byte gap (fp32)
    assert G.plan_batched(4, 4, 4, 0).path == G.PATH_NOOP
    for bad in (dict(strideC=4 * 4 - 1), dict(strideA=-1)):
        with pytest.raises(G.GemmError) as e:
            G.plan_batched(4, 4, 4, 2, **bad)
        assert e.value.status == G.ERR_INVALID_ARG
    with pytest.raises(G.GemmError) as e:
        G.plan_batched(65536, 65536, 64, 4096)        # 2^31 tiles in all
    assert e.value.status == G.ERR_UNSUPPORTED


def test_plan_grouped():
    """Grouped calls: tiles counted per group (padded to whole tiles), direct
    stores; sizes must be non-negative."""
    sizes = [5, 0, 130, 1, 257, 64]
    p = G.plan_grouped(sizes, 300, 200, 1)
    cg = p.bm // 128
    rows = sum(-(-m // (128 * cg)) for m in sizes)
    assert p.tiles == rows * p.tiles_j and p.bulk_store == G.BULK_NONE
    assert p.swap_ab == 0 and p.workspace_bytes >= (len(sizes) + 1) * 4
    assert G.plan_grouped([], 8, 8).path == G.PATH_NOOP
    assert G.plan_grouped([4, 0], 8, 0).path == G.PATH_SCALE_C
    with pytest.raises(G.GemmError) as e:
        G.plan_grouped([3, -1], 8, 8)
    assert e.value.status == G.ERR_INVALID_ARG
    with pytest.raises(G.GemmError) as e:
        G.plan_grouped([3, 4], 8, 32, 0, G.E4M3_F32)       # 8-bit weights must be N x K
    assert e.value.status == G.ERR_UNSUPPORTED


def test_plan_half_atom_pairs_need_k_major_q():
    """A CTA pair with 64-wide tiles loads 32-row halves of the MMA's B operand,
    which only the K-major layout allows."""
    p = G.plan(64, 32000, 4096, 1, 1)     # A stored K x M: the activations are M-major
    assert not (p.cluster == 2 and p.bn == 64)
    assert p.vector_store == 0 and p.grid == 152   # (HBM-bound: stream-K keeps every SM streaming)


def test_plan_few_tiles_stream_k():
    """Far fewer tiles than SMs with a deep K: every tile's k-blocks are shared out."""
    p = G.plan(256, 256, 8192, 0, 1)
    assert p.schedule == G.SCHED_STREAM_K and p.dp_tiles == 0 and p.sk_slots > p.tiles
    assert p.units > p.tiles and p.workspace_bytes > 0


def test_plan_full_waves_need_no_stream_k():
    p = G.plan(128 * 152, 64, 512, 0, 1)   # exactly one wave of 128 x 64 tiles
    assert p.schedule == G.SCHED_TILES and p.units == p.tiles


def test_plan_ragged_repacks_misaligned_b():
    p = G.plan(4095, 4097, 1000, 0, 0, lda=1000, ldb=4097, ldc=4097)
    assert p.repack_a == 0 and p.repack_b == 1
    # 4097 fp32 = 16388-byte rows: four row classes, one tensor store each per block (repack, GEMM)
    assert p.launches == 2 and p.bulk_store == G.BULK_ROW_CLASSES
    assert p.workspace_bytes >= 1000 * 4104 * 2
    with_direct = G.plan(4095, 4097, 1000, 0, 0, lda=1000, ldb=4097, ldc=4097, beta=1.0)
    assert with_direct.launches == 2 and with_direct.vector_store == 0 and with_direct.bulk_store == G.BULK_NONE


def test_plan_misaligned_pointer_repacks():
    p = G.plan(512, 512, 512, 0, 1, A=0x1002)
    assert p.repack_a == 1 and p.repack_b == 0


def test_plan_degenerate_sizes():
    assert G.plan(0, 10, 10).path == G.PATH_NOOP
    assert G.plan(10, 0, 10).path == G.PATH_NOOP
    p = G.plan(10, 10, 0, lda=1)
    assert p.path == G.PATH_SCALE_C and p.launches == 1


@pytest.mark.parametrize("kw", [dict(M=-1, N=4, K=4), dict(M=4, N=4, K=8, lda=7), dict(M=4, N=4, K=8, ldb=3),
                                dict(M=4, N=8, K=4, ldc=7), dict(M=4, N=4, K=4, dtype=9),
                                dict(M=4, N=4, K=4, transA=2), dict(M=4, N=4, K=4, A=0)])
def test_plan_rejects_bad_arguments(kw):
    with pytest.raises(G.GemmError) as e:
        G.plan(**kw)
    assert e.value.status == G.ERR_INVALID_ARG


def test_plan_rejects_oversized_extent():
    with pytest.raises(G.GemmError) as e:
        G.plan(1 << 31, 8, 8)
    assert e.value.status == G.ERR_UNSUPPORTED


@pytest.mark.parametrize("shape", [(256, 256, 256), (1, 1, 1), (300, 520, 200), (8192, 12288, 4096),
                                   (8192, 4096, 16384), (33, 4000, 70), (4095, 4097, 1000)])
def test_plan_invariants(shape):
    M, N, K = shape
    for sm in (148, 152, 160):
        p = G.plan(M, N, K, 0, 0, sm_count=sm)
        I, J = (N, M) if p.swap_ab else (M, N)
        cg = p.bm // 128
        assert cg == p.cluster == {G.PATH_TC_1CTA: 1, G.PATH_TC_2CTA: 2}[p.path]
        assert p.tiles == -(-I // p.bm) * -(-J // p.bn) == p.tiles_i * p.tiles_j
        assert p.kdepth in (1, 2) and p.bk == 64 * p.kdepth and 2 <= p.stages and p.stages * p.kdepth <= 8
        assert p.num_kb == -(-K // p.bk)
        slots = sm // p.cluster
        if p.schedule == G.SCHED_TILES:
            assert p.units == p.tiles * p.split_k and p.dp_tiles == p.tiles
            waves = -(-p.units // slots)           # the units spread evenly over the waves
            assert p.grid == -(-p.units // waves) * p.cluster
        else:
            assert p.split_k == 1 and p.dp_tiles % (p.grid // p.cluster) == 0 and p.units >= p.tiles
            assert p.grid == min(p.units, slots) * p.cluster
        assert 1 <= p.split_k <= max(1, p.num_kb)
        assert 1 <= p.raster_group <= max(1, -(-I // p.bm))


def test_probe_tma_tile_rejects_bad_arguments():
    """The swizzle probe checks its arguments before any CUDA call."""
    L = G.lib()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: every call below fails its checks
    assert L.gemm_probe_tma_tile(None, 0x1000, 64, 64, 8, 0x2000, None) == G.ERR_INVALID_ARG
    assert L.gemm_probe_tma_tile(fake, 0x1000, 64, 64, 0, 0x2000, None) == G.ERR_INVALID_ARG    # rows < 1
    assert L.gemm_probe_tma_tile(fake, 0x1000, 64, 64, 257, 0x2000, None) == G.ERR_INVALID_ARG  # rows > 256
    assert L.gemm_probe_tma_tile(fake, 0x1002, 64, 64, 8, 0x2000, None) == G.ERR_INVALID_ARG   # misaligned
    assert L.gemm_probe_tma_tile(fake, 0x1000, 60, 60, 8, 0x2000, None) == G.ERR_INVALID_ARG    # 120-byte rows
    assert L.gemm_probe_tma_tile(fake, 0x1000, 32, 64, 8, 0x2000, None) == G.ERR_INVALID_ARG    # ld < cols
    assert L.gemm_probe_tma_tile(fake, 0x1000, 64, 64, 8, None, None) == G.ERR_INVALID_ARG


@pytest.mark.parametrize("argv", [
    ["square_4096_nt_f32", "--option", "OPT_BOGUS=1"],       # no such option
    ["square_4096_nt_f32", "--option", "OPT_STREAM_K=x"],    # not an integer
    ["square_4096_nt_f32", "--option", "STREAM_K=1"],        # not a binding option name
    ["square_4096_nt_f32", "--raster-group", "-1"],
    ["no_such_case"],
])
def test_profile_case_rejects_bad_arguments(argv, capsys):
    """The profiling entry point checks its arguments before any GPU call."""
    from dense_gemm_10_gb300 import profile_case
    with pytest.raises(SystemExit) as e:
        profile_case.main(argv)
    assert e.value.code == 2
