"""GPU parity against the CPU oracle, element by element, at sizes the oracle
finishes in seconds: several tiles, ragged tails, every layout, both input
types, every output type, alpha / beta, the swapped and split-K paths, and the
degenerate sizes.  Every call goes through the C ABI."""
import contextlib

import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, assert_close, device_problem, dtype_code, launch, oracle_full, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


# (CTAs per schedule slot, tile width): one CTA or a CTA pair
CONFIGS = [(1, 64), (1, 128), (1, 256), (2, 64), (2, 128), (2, 256)]
PATHS = {1: G.PATH_TC_1CTA, 2: G.PATH_TC_2CTA}


def skip_half_atom(cg, bn, q_kmajor):
    """A CTA pair with 64-wide tiles needs a K-major MMA B operand."""
    if cg == 2 and bn == 64 and not q_kmajor:
        pytest.skip("64-wide CTA-pair tiles take K-major B only")


@contextlib.contextmanager
def options(h, **kw):
    """Force planner options on the handle for the duration of a check."""
    codes = {"path": G.OPT_FORCE_PATH, "bn": G.OPT_FORCE_BN, "split": G.OPT_SPLIT_K, "raster": G.OPT_RASTER_GROUP,
             "grid": G.OPT_MAX_GRID, "stream_k": G.OPT_STREAM_K, "kdepth": G.OPT_KDEPTH}
    try:
        for k, v in kw.items():
            h.set_option(codes[k], v)
        yield
    finally:
        for k in kw:
            h.set_option(codes[k], 0)


def _check(p, h, guard=True):
    out, full = run(p, h, guard_rows=3 if guard else 0, guard_cols=5 if guard else 0)
    R, Mag = oracle_full(p)
    assert_close(out, R, Mag, p.out_dtype == "f32", p.name)
    if guard:
        # nothing outside the logical M x N block was written
        pad = full.clone().to(torch.float64)
        pad[:p.M, :p.N] = SENTINEL
        assert torch.all(pad == SENTINEL), "C written outside the M x N block"
    return out


def test_tiny_256(h):
    """M = N = K = 256, bf16 U[-1, 1], NN, fp32 C."""
    _check(inputs.tiny_256(), h)


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("in_dtype,out_dtype", [("bf16", "f32"), ("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
def test_layouts_and_types(h, transA, transB, in_dtype, out_dtype, cg):
    """Ragged in every dimension: partial last tiles, K not a multiple of 64; one
    CTA per tile and CTA pairs."""
    p = inputs.make_problem("lay", 300, 520, 200, transA, transB, in_dtype, out_dtype, ("uniform", -1, 1),
                            ("uniform", -1, 1), alpha=1.5, beta=0.5, seed=31)
    with options(h, path=PATHS[cg]):
        _check(p, h)


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 1, 70), (127, 129, 63), (128, 256, 64), (129, 257, 65),
                                   (7, 300, 1000), (1000, 7, 130), (513, 1031, 16)])
def test_ragged_shapes(h, shape):
    M, N, K = shape
    p = inputs.make_problem("rag", M, N, K, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1), seed=M + N + K)
    _check(p, h)


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("kdepth", [1, 2])
def test_small_integers_bit_exact(h, transA, transB, cg, kdepth):
    """Integers in {-4..4}: the fp32 result is exact whatever the order of the
    sum, so the GPU must equal the oracle bit for bit."""
    p = inputs.make_problem("ints", 384, 640, 1024, transA, transB, "bf16", "f32", ("ints", -4, 4), ("ints", -4, 4),
                            alpha=1.5, beta=0.5, dist_c=("ints", -9, 9), seed=5)
    with options(h, path=PATHS[cg], kdepth=kdepth):
        out, _ = run(p, h)
    R, _ = oracle_full(p)
    assert np.array_equal(out, R)


@pytest.mark.parametrize("M,N,K", [(64, 2000, 4096), (16, 3000, 512), (64, 640, 130), (40, 1000, 1000)])
def test_skinny_swapped_split(h, M, N, K):
    """Short M: the planner swaps operands (C^T = B^T A^T) and splits K."""
    p = inputs.make_problem("skinny", M, N, K, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 0.02), seed=N)
    plan = G.plan(M, N, K, 0, 1, sm_count=152)
    assert plan.swap_ab == 1
    _check(p, h)


@pytest.mark.parametrize("kdepth", [1, 2])
@pytest.mark.parametrize("split", [2, 3, 7])
@pytest.mark.parametrize("cg,bn", CONFIGS)
def test_forced_split_k(h, split, cg, bn, kdepth):
    """K = 960: 15 k-slices of 64, or 8 stages of two (the last holding one)."""
    p = inputs.make_problem("split", 300, 520, 960, 0, 1, "f16", "f32", ("uniform", -1, 1), ("uniform", -1, 1),
                            alpha=-0.75, beta=1.25, seed=split * bn + cg)
    with options(h, path=PATHS[cg], bn=bn, split=split, kdepth=kdepth):
        plan = G.plan(p.M, p.N, p.K, 0, 1, G.F16_F32, handle=h, beta=p.beta)
        assert plan.split_k == split and plan.bn == bn and plan.path == PATHS[cg]
        assert plan.kdepth == kdepth and plan.num_kb == -(-15 // kdepth)
        _check(p, h)


@pytest.mark.parametrize("kdepth", [1, 2])
@pytest.mark.parametrize("cg,bn", CONFIGS)
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_every_tile_configuration(h, cg, bn, transA, transB, kdepth):
    """K = 300: five k-slices, the last one partial; with two slices per stage the
    last stage holds that partial slice alone."""
    skip_half_atom(cg, bn, transB == 1)
    p = inputs.make_problem("cfg", 600, 900, 300, transA, transB, "bf16", "bf16", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.5, beta=-1.0, seed=bn + transA + 2 * transB + 7 * cg)
    with options(h, path=PATHS[cg], bn=bn, kdepth=kdepth):
        assert G.plan(p.M, p.N, p.K, transA, transB, G.BF16_BF16, handle=h, beta=p.beta).kdepth == kdepth
        _check(p, h)


@pytest.mark.parametrize("kdepth", [1, 2])
@pytest.mark.parametrize("gi", [0, 1, 2])
@pytest.mark.parametrize("cg,bn", CONFIGS)
def test_stream_k(h, cg, bn, gi, kdepth):
    """Stream-K tail forced on small grids: tiles cut into several pieces whose
    partials are summed by the last piece to finish.  The grids leave an
    incomplete last wave for every configuration (90, 48, 24, 24, 12 and 6 schedule tiles)."""
    grid = {1: (7, 13, 29), 2: (10, 14, 30), 4: (16, 20, 28)}[cg][gi]
    if (cg, bn) == (2, 64):
        grid = (8, 12, 16)[gi]   # 3 x 15 = 45 tiles: 45 % 4, 45 % 6, 45 % 8 all non-zero
    p = inputs.make_problem("sk", 700, 900, 1000, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=1.25, beta=-0.5, seed=grid + bn + cg)
    with options(h, path=PATHS[cg], bn=bn, grid=grid, stream_k=2, kdepth=kdepth):
        plan = G.plan(p.M, p.N, p.K, 0, 1, handle=h, beta=p.beta)
        assert plan.schedule == G.SCHED_STREAM_K and plan.path == PATHS[cg] and plan.grid <= grid
        assert plan.kdepth == kdepth
        _check(p, h)


@pytest.mark.parametrize("kdepth", [1, 2])
@pytest.mark.parametrize("cg,bn", CONFIGS)
def test_stream_k_all_tiles_shared(h, cg, bn, kdepth):
    """Fewer tiles than CTAs and a deep K (63 k-slices, the last partial): no
    whole tiles, every tile is shared."""
    skip_half_atom(cg, bn, False)
    p = inputs.make_problem("skdeep", 250, 250, 4000, 1, 0, "f16", "f16", ("uniform", -1, 1), ("uniform", -1, 1),
                            seed=bn * cg)
    with options(h, path=PATHS[cg], bn=bn, stream_k=2, kdepth=kdepth):
        plan = G.plan(p.M, p.N, p.K, 1, 0, G.F16_F16, handle=h)
        assert plan.schedule == G.SCHED_STREAM_K and plan.dp_tiles == 0
        _check(p, h)


@pytest.mark.parametrize("cg,bn", CONFIGS)
def test_many_tiles_per_cta(h, cg, bn):
    """More tiles than CTAs: every CTA runs several tiles through both TMEM buffers."""
    p = inputs.make_problem("persist", 1100, 1500, 192, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            seed=3 * bn + cg)
    with options(h, path=PATHS[cg], bn=bn, raster=3, grid=6, stream_k=1):
        plan = G.plan(p.M, p.N, p.K, 0, 1, handle=h)
        assert plan.grid <= 6 and plan.units >= 3 * plan.grid // cg
        _check(p, h)


def _check_bulk(p, h, expect_bulk):
    """Like _check, with 8 guard columns, which keep C's rows 16-byte aligned so
    that the epilogue can use bulk tensor stores; the guard region must survive
    the clipped edge boxes."""
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, dtype_code(p), handle=h, ldc=p.ldc + 8, beta=p.beta)
    assert plan.bulk_store == expect_bulk, plan.as_dict()
    out, full = run(p, h, guard_rows=3, guard_cols=8)
    R, Mag = oracle_full(p)
    assert_close(out, R, Mag, p.out_dtype == "f32", p.name)
    pad = full.clone().to(torch.float64)
    pad[:p.M, :p.N] = SENTINEL
    assert torch.all(pad == SENTINEL), "C written outside the M x N block"


OUT_TYPES = [("bf16", "f32"), ("bf16", "bf16"), ("f16", "f16")]


def _expected_misaligned_path(M, N, K, mode, out_dtype):
    """The planner's choice for C that bulk tensor stores cannot write (beta == 0,
    one unswapped GEMM): fp32 C in row classes (auto mode, at least 4 rows and
    8 columns); else the workspace copy for a large C with K < 2048, else
    per-row copies.  GEMM_OPT_EPILOGUE = 3 asks for the copy where allowed, 4
    for per-row copies."""
    staged_ok = M * N >= 1 << 20
    if mode == 3:
        return G.BULK_STAGED if staged_ok else G.BULK_ROW_COPIES
    if mode == 4:
        return G.BULK_ROW_COPIES
    if out_dtype == "f32" and M >= 4 and N >= 8:
        return G.BULK_ROW_CLASSES
    return G.BULK_STAGED if staged_ok and K < 2048 else G.BULK_ROW_COPIES


@pytest.mark.parametrize("mode", [0, 3, 4])
@pytest.mark.parametrize("in_dtype,out_dtype", OUT_TYPES)
@pytest.mark.parametrize("M,N,K,transB,guard_cols", [
    (1100, 1001, 300, 1, 5),    # misaligned rows (ldc = 1006), ragged N
    (1030, 1024, 200, 0, 3),    # misaligned rows, N whole pieces
    (1500, 1003, 96, 1, 13),    # rows aligned for 16-bit C only (ldc = 1016), N ends inside a piece
    (300, 77, 130, 1, 1),       # small C, a single partial tile column (ldc = 78)
    (600, 2003, 2100, 1, 2),    # long K
])
def test_misaligned_c(h, M, N, K, transB, guard_cols, in_dtype, out_dtype, mode):
    """C that bulk tensor stores cannot write: each row of a block leaves
    through one 1-D bulk copy of its whole 16-byte pieces (plain stores for the
    partial pieces at a tile's edges), or bulk stores write an aligned copy in
    the workspace that a copy kernel moves into C.  Exact values where they
    belong, nothing written in C's padding columns or the guard rows below it."""
    p = inputs.make_problem("misaligned", M, N, K, 0, transB, in_dtype, out_dtype, ("normal", 0, 1),
                            ("normal", 0, 1), alpha=0.5, seed=M + N + guard_cols)
    aligned = ((p.ldc + guard_cols) * (4 if out_dtype == "f32" else 2)) % 16 == 0
    whole = (N * (4 if out_dtype == "f32" else 2)) % 16 == 0
    h.set_option(G.OPT_EPILOGUE, mode)
    try:
        plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, dtype_code(p), handle=h, ldc=p.ldc + guard_cols)
        expect = G.BULK_ROWS if aligned and whole else _expected_misaligned_path(M, N, K, mode, out_dtype)
        assert plan.bulk_store == expect, plan.as_dict()
        out, full = run(p, h, guard_rows=3, guard_cols=guard_cols)
    finally:
        h.set_option(G.OPT_EPILOGUE, 0)
    R, Mag = oracle_full(p)
    assert_close(out, R, Mag, p.out_dtype == "f32", p.name)
    pad = full.clone().to(torch.float64)
    pad[:p.M, :p.N] = SENTINEL
    assert torch.all(pad == SENTINEL), "C written outside the M x N block"


@pytest.mark.parametrize("mode", [0, 4])
@pytest.mark.parametrize("cg,bn", CONFIGS)
@pytest.mark.parametrize("ldc_extra", [0, 1, 2])
def test_misaligned_fp32_every_tile_config(h, cg, bn, ldc_extra, mode):
    """Row classes (mode 0) and per-row bulk copies (mode 4) in every tile
    configuration, several tiles per CTA (grid 6) and every misalignment a row
    of fp32 C can have: with the 5 guard columns, ldc = 909, 910, 911 makes
    consecutive rows start 4, 8 or 12 bytes further off a 16-byte boundary
    (four, two and four row classes)."""
    p = inputs.make_problem("rowcopy", 700, 904, 2100, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.75, seed=bn + cg + ldc_extra, ldc=904 + ldc_extra)
    h.set_option(G.OPT_EPILOGUE, mode)
    try:
        with options(h, path=PATHS[cg], bn=bn, grid=6, stream_k=1):
            plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, handle=h, ldc=p.ldc + 5)   # _check adds 5 guard columns
            assert plan.bulk_store == (G.BULK_ROW_CLASSES if mode == 0 else G.BULK_ROW_COPIES), plan.as_dict()
            _check(p, h)
    finally:
        h.set_option(G.OPT_EPILOGUE, 0)


@pytest.mark.parametrize("M,N,K,ldc", [(4095, 4097, 1000, 4097), (300, 77, 130, 78), (129, 1001, 64, 1001),
                                       (70, 8, 16, 9), (1000, 1003, 300, 1006), (260, 36, 70, 39)])
def test_row_classes_shapes(h, M, N, K, ldc):
    """fp32 C in row classes at ragged sizes: tiles narrower than a block, a
    right edge inside a 16-byte piece (the values past the class tensor's last
    whole piece go out by plain stores), a single tile column, fewer rows than
    a tile, and C's rows packed end to end (ldc = N), where any write past
    column N would land in the next row."""
    p = inputs.make_problem("rowclass", M, N, K, 0, 0, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=1.25, seed=M + N + K, ldc=ldc)
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, handle=h, ldc=ldc)
    assert plan.bulk_store == G.BULK_ROW_CLASSES, plan.as_dict()
    Ad, Bd = p.A.cuda(), p.B.cuda()
    C = torch.full((p.M + 2, ldc), SENTINEL, dtype=torch.float32, device="cuda")
    C[:p.M, :p.N] = float("nan")
    launch(p, h, Ad, Bd, C, ldc)
    assert h.status()[0] == G.OK
    full = C.cpu()
    R, Mag = oracle_full(p)
    assert_close(full[:p.M, :p.N].double().numpy(), R, Mag, True, p.name)
    pad = full.clone().to(torch.float64)
    pad[:p.M, :p.N] = SENTINEL
    assert torch.all(pad == SENTINEL), "C written outside the M x N block"


def test_misaligned_c_in_sequence(h):
    """Misaligned calls of different sizes in a row on one stream, with per-row
    copies and with the workspace copy of C: each one's C is complete when the
    stream is."""
    for mode in (3, 4):
        h.set_option(G.OPT_EPILOGUE, mode)
        outs = []
        try:
            for i, (M, N, K) in enumerate([(1200, 1001, 128), (2100, 999, 64), (1100, 1001, 256)]):
                p = inputs.make_problem("misaligned_seq%d" % i, M, N, K, 0, 1, "bf16", "f32", ("normal", 0, 1),
                                        ("normal", 0, 1), seed=40 + i)
                Ad, Bd, Cd, ldc = device_problem(p, guard_rows=1, guard_cols=1)
                launch(p, h, Ad, Bd, Cd, ldc)
                outs.append((p, Cd))
            assert h.status()[0] == G.OK
        finally:
            h.set_option(G.OPT_EPILOGUE, 0)
        for p, Cd in outs:
            R, Mag = oracle_full(p)
            assert_close(Cd[:p.M, :p.N].double().cpu().numpy(), R, Mag, True, p.name)


@pytest.mark.parametrize("in_dtype,out_dtype", OUT_TYPES)
@pytest.mark.parametrize("grid", [0, 6])
@pytest.mark.parametrize("cg,bn", CONFIGS)
def test_bulk_store_rows(h, cg, bn, grid, in_dtype, out_dtype):
    """Staged bulk tensor stores of C rows, ragged in M and N (N = 904 keeps
    whole 16-byte pieces).  grid = 6: each CTA stores several tiles through its
    two staging buffers and its last one through the idle operand ring."""
    p = inputs.make_problem("bulk", 600, 904, 300, 0, 1, in_dtype, out_dtype, ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.75, seed=bn + cg + grid)
    with options(h, path=PATHS[cg], bn=bn, grid=grid, stream_k=1):
        _check_bulk(p, h, G.BULK_ROWS)


@pytest.mark.parametrize("in_dtype,out_dtype", OUT_TYPES)
@pytest.mark.parametrize("M,N,K", [(64, 2000, 1000), (40, 1000, 700), (1, 1032, 256), (64, 904, 130)])
def test_bulk_store_transposed(h, M, N, K, in_dtype, out_dtype):
    """Swapped problems (short M): C is stored J x I from the kernel's point of
    view, and each warp writes its 32 x 32 block transposed into staging."""
    p = inputs.make_problem("bulkT", M, N, K, 0, 1, in_dtype, out_dtype, ("normal", 0, 1), ("normal", 0, 0.5),
                            alpha=1.5, seed=M + N)
    _check_bulk(p, h, G.BULK_TRANSPOSED)


@pytest.mark.parametrize("grid", [0, 7])
@pytest.mark.parametrize("cg,bn", [(1, 64), (1, 128), (1, 256), (2, 64), (2, 128), (2, 256)])
def test_bulk_store_transposed_configs(h, cg, bn, grid):
    """Every configuration a swapped problem can take, forced, on full and small grids."""
    p = inputs.make_problem("bulkTc", 48, 3000, 520, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            seed=bn * cg + grid)
    with options(h, path=PATHS[cg], bn=bn, grid=grid, stream_k=1):
        _check_bulk(p, h, G.BULK_TRANSPOSED)


@pytest.mark.parametrize("kdepth", [1, 2])
@pytest.mark.parametrize("cg,bn", CONFIGS)
def test_bulk_store_after_stream_k(h, cg, bn, kdepth):
    """Stream-K fix-ups leave through bulk stores as well (the last arriving
    piece sums the partials and stores the tile)."""
    grid = {1: 13, 2: 14, 4: 20}[cg] if (cg, bn) != (2, 64) else 12
    p = inputs.make_problem("bulksk", 700, 904, 1000, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            seed=grid + bn + cg)
    with options(h, path=PATHS[cg], bn=bn, grid=grid, stream_k=2, kdepth=kdepth):
        _check_bulk(p, h, G.BULK_ROWS)


def test_misaligned_leading_dimensions(h):
    """Row pitches that are not multiples of 16 bytes go through the repack and
    scalar-store paths."""
    p = inputs.make_problem("mis", 333, 517, 301, 0, 0, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=1.0, beta=0.5, seed=77, lda=301, ldb=519, ldc=517)
    plan = G.plan(p.M, p.N, p.K, 0, 0, lda=p.lda, ldb=p.ldb, ldc=p.ldc)
    assert plan.repack_a == 1 and plan.repack_b == 1 and plan.vector_store == 0
    _check(p, h)


def test_misaligned_base_pointer(h):
    p = inputs.make_problem("misptr", 200, 264, 136, 0, 1, "f16", "f32", ("normal", 0, 1), ("normal", 0, 1), seed=8)
    Ad, Bd, Cd, ldc = device_problem(p)
    # shift A by one element inside a larger buffer: base no longer 16-byte aligned
    big = torch.empty(Ad.numel() + 8, dtype=Ad.dtype, device="cuda")
    big[1:1 + Ad.numel()] = Ad.reshape(-1)
    A_shift = big[1:1 + Ad.numel()]
    st = h.run_raw(0, 1, p.M, p.N, p.K, 1.0, A_shift.data_ptr(), p.lda, Bd.data_ptr(), p.ldb, 0.0, Cd.data_ptr(),
                   ldc, G.F16_F32, None)
    assert st == G.OK
    assert h.status()[0] == G.OK
    R, Mag = oracle_full(p)
    assert_close(Cd[:p.M, :p.N].double().cpu().numpy(), R, Mag, True, "misaligned base")


def test_beta_zero_ignores_nan_c(h):
    p = inputs.make_problem("nanc", 256, 384, 128, 0, 0, "bf16", "f32", seed=3)
    out, _ = run(p, h)   # C starts as NaN
    assert np.isfinite(out).all()


def test_k_zero_scales_c(h):
    M, N = 100, 77
    for beta in (0.0, -2.0):
        C = torch.randn(M, N, device="cuda")
        ref = (beta * C).cpu() if beta != 0.0 else torch.zeros(M, N)
        A = torch.empty(M, 1, dtype=torch.bfloat16, device="cuda")
        B = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
        assert h.run_raw(0, 0, M, N, 0, 1.0, A.data_ptr(), 1, B.data_ptr(), N, beta, C.data_ptr(), N,
                         G.BF16_F32, None) == G.OK
        assert h.status()[0] == G.OK
        assert torch.equal(C.cpu(), ref)


def test_empty_m_or_n_is_noop(h):
    C = torch.full((4, 4), 7.0, device="cuda")
    A = torch.zeros(4, 4, dtype=torch.bfloat16, device="cuda")
    before = h.launch_count()
    assert h.run_raw(0, 0, 0, 4, 4, 1.0, A.data_ptr(), 4, A.data_ptr(), 4, 0.0, C.data_ptr(), 4, G.BF16_F32, None) == G.OK
    assert h.run_raw(0, 0, 4, 0, 4, 1.0, A.data_ptr(), 4, A.data_ptr(), 4, 0.0, C.data_ptr(), 4, G.BF16_F32, None) == G.OK
    assert h.launch_count() == before
    assert torch.all(C == 7.0)


def test_bad_arguments_return_errors(h):
    A = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(8, 8, device="cuda")
    assert h.run_raw(0, 0, 8, 8, 8, 1.0, A.data_ptr(), 7, A.data_ptr(), 8, 0.0, C.data_ptr(), 8, 0, None) \
        == G.ERR_INVALID_ARG
    assert h.run_raw(0, 0, 8, 8, 8, 1.0, 0, 8, A.data_ptr(), 8, 0.0, C.data_ptr(), 8, 0, None) == G.ERR_INVALID_ARG
    assert h.run_raw(0, 0, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0, C.data_ptr(), 8, 8, None) \
        == G.ERR_INVALID_ARG


@pytest.mark.parametrize("pdl", [1, 0])
def test_chained_gemms_read_each_others_output(h, pdl):
    """C1 = A B, then C2 = C1 D and C3 = C2 E back to back on one stream: each
    kernel starts its set-up while the previous one runs (programmatic
    dependent launch) but must read the finished C of the one before.  The
    middle GEMM's operand needs a repack (odd pitch), so a copy kernel sits
    between two of them.  Checked against the oracle applied step by step."""
    import oracle
    g = torch.Generator().manual_seed(3)
    A = torch.randn(520, 384, generator=g).to(torch.bfloat16)
    B = torch.randn(384, 776, generator=g).to(torch.bfloat16)
    D = (torch.randn(776, 264, generator=g) / 16).to(torch.bfloat16)
    E = (torch.randn(264, 300, generator=g) / 8).to(torch.bfloat16)
    h.set_option(G.OPT_PDL, pdl)
    try:
        Ad, Bd, Dd, Ed = A.cuda(), B.cuda(), D.cuda(), E.cuda()
        C1 = torch.full((520, 777), float("nan"), dtype=torch.bfloat16, device="cuda")  # ldc 777: C2's A repacked
        C2 = torch.full((520, 264), float("nan"), dtype=torch.bfloat16, device="cuda")
        C3 = torch.full((520, 300), float("nan"), dtype=torch.float32, device="cuda")
        for _ in range(3):
            assert h.run_raw(0, 0, 520, 776, 384, 1.0, Ad.data_ptr(), 384, Bd.data_ptr(), 776, 0.0, C1.data_ptr(),
                             777, G.BF16_BF16, None) == G.OK
            assert h.run_raw(0, 0, 520, 264, 776, 1.0, C1.data_ptr(), 777, Dd.data_ptr(), 264, 0.0, C2.data_ptr(),
                             264, G.BF16_BF16, None) == G.OK
            assert h.run_raw(0, 0, 520, 300, 264, 1.0, C2.data_ptr(), 264, Ed.data_ptr(), 300, 0.0, C3.data_ptr(),
                             300, G.BF16_F32, None) == G.OK
        assert h.status()[0] == G.OK
    finally:
        h.set_option(G.OPT_PDL, 1)
    bits = lambda t: t.contiguous().view(torch.uint16).numpy()
    c1 = C1.cpu()
    R1, M1 = oracle.gemm(0, 0, 520, 776, 384, 1.0, bits(A), 384, bits(B), 776, 0.0, None, 776, oracle.IN_BF16)
    assert_close(c1[:, :776].double().numpy(), R1, M1, False, "C1")
    c2 = C2.cpu()
    R2, M2 = oracle.gemm(0, 0, 520, 264, 776, 1.0, bits(c1), 777, bits(D), 264, 0.0, None, 264, oracle.IN_BF16)
    assert_close(c2.double().numpy(), R2, M2, False, "C2 from the C1 the GPU wrote")
    R3, M3 = oracle.gemm(0, 0, 520, 300, 264, 1.0, bits(c2), 264, bits(E), 300, 0.0, None, 300, oracle.IN_BF16)
    assert_close(C3.cpu().double().numpy(), R3, M3, True, "C3 from the C2 the GPU wrote")


def test_run_to_run_determinism(h):
    """Same inputs, same bits, including the split-K fix-up (fixed summation order)."""
    for (M, N, K) in [(512, 768, 640), (64, 4000, 4096)]:
        p = inputs.make_problem("det", M, N, K, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1), seed=M)
        a, _ = run(p, h)
        b, _ = run(p, h)
        assert np.array_equal(a, b)


def test_torch_binding_matches_oracle(h):
    """The tensor-level binding infers sizes and leading dimensions correctly."""
    p = inputs.make_problem("bind", 200, 300, 100, 1, 0, "bf16", "bf16", ("normal", 0, 1), ("normal", 0, 1), seed=12)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.empty(200, 300, dtype=torch.bfloat16, device="cuda")
    G.gemm(A, B, C, transA=True, transB=False, handle=h)
    torch.cuda.synchronize()
    R, Mag = oracle_full(p)
    assert_close(C.double().cpu().numpy(), R, Mag, False, "binding")


def test_launch_count_and_plan_agree(h):
    p = inputs.make_problem("cnt", 333, 517, 301, 0, 0, "bf16", "f32", lda=301, ldb=519, ldc=517, seed=1)
    plan = G.plan(p.M, p.N, p.K, 0, 0, lda=p.lda, ldb=p.ldb, ldc=p.ldc)
    Ad, Bd, Cd, ldc = device_problem(p)
    before = h.launch_count()
    launch(p, h, Ad, Bd, Cd, ldc)
    assert h.status()[0] == G.OK
    assert h.launch_count() - before == plan.launches == 3


@pytest.mark.parametrize("shape,code", [((300, 264, 200), G.BF16_F32), ((40, 1000, 512), G.BF16_BF16),
                                        ((260, 200, 96), G.F32_F32)])
def test_plan_cache_hits_use_the_calls_own_pointers(h, shape, code):
    """Repeated calls of one shape on different buffers reuse the cached plan
    (a swapped problem and the split fp32 operands included) and each writes
    its own product; a differently aligned pointer plans anew."""
    import oracle
    M, N, K = shape
    dt = torch.float32 if code == G.F32_F32 else torch.bfloat16
    ct = torch.bfloat16 if code == G.BF16_BF16 else torch.float32
    g = torch.Generator().manual_seed(sum(shape))
    pairs = [(torch.randn(M, K, generator=g).to(dt), torch.randn(N, K, generator=g).to(dt)) for _ in range(3)]
    hits0, misses0 = h.plan_cache_stats()
    outs = []
    for A, B in pairs:
        Ad, Bd = A.cuda(), B.cuda()
        C = torch.full((M, N), float("nan"), dtype=ct, device="cuda")
        assert h.run_raw(0, 1, M, N, K, 1.0, Ad.data_ptr(), K, Bd.data_ptr(), K, 0.0, C.data_ptr(), N, code,
                         None) == G.OK
        torch.cuda.synchronize()
        outs.append(C.cpu().double().numpy())
    hits, misses = h.plan_cache_stats()
    assert hits - hits0 >= 2 and misses - misses0 <= 1
    # a C 4 bytes off a 16-byte boundary is a different plan (direct stores)
    Cbig = torch.full((M * N + 4,), float("nan"), dtype=torch.float32, device="cuda")
    Ad, Bd = pairs[0][0].cuda(), pairs[0][1].cuda()
    if ct == torch.float32:
        assert h.run_raw(0, 1, M, N, K, 1.0, Ad.data_ptr(), K, Bd.data_ptr(), K, 0.0, Cbig.data_ptr() + 4, N, code,
                         None) == G.OK
        torch.cuda.synchronize()
        assert h.plan_cache_stats()[1] == misses + 1
        outs_shift = Cbig[1:1 + M * N].view(M, N).cpu().double().numpy()
        assert np.array_equal(outs_shift, outs[0])
    for (A, B), out in zip(pairs, outs):
        if dt == torch.float32:
            R, Mag = oracle.gemm(0, 1, M, N, K, 1.0, A.numpy(), K, B.numpy(), K, 0.0, None, N, oracle.IN_F32)
            assert oracle.within_tolerance(out, R, Mag, True, tf32x3_k=K).all()
        else:
            bits = lambda t: t.contiguous().view(torch.uint16).numpy()
            R, Mag = oracle.gemm(0, 1, M, N, K, 1.0, bits(A), K, bits(B), K, 0.0, None, N, oracle.IN_BF16)
            assert_close(out, R, Mag, ct == torch.float32, "plan cache")


def test_tensor_map_cache_reuses_maps_of_the_same_buffers(h):
    """A repeated call on the same buffers copies its tensor maps from the
    handle's cache instead of encoding them; a call on another buffer encodes
    that buffer's map anew, and every result is the oracle's."""
    # (a shape no other test uses, so no earlier call left maps of these extents)
    p = inputs.make_problem("tmap", 296, 328, 200, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1), seed=61)
    R, Mag = oracle_full(p)
    Ad, Bd = p.A.cuda(), p.B.cuda()
    C1 = torch.full((p.M, p.N), float("nan"), device="cuda")
    C2 = torch.full((p.M, p.N), float("nan"), device="cuda")
    hits0, misses0 = h.tensor_map_cache_stats()
    for _ in range(4):
        launch(p, h, Ad, Bd, C1, p.N)
    hits1, misses1 = h.tensor_map_cache_stats()
    assert misses1 - misses0 <= 3 and hits1 - hits0 >= 9      # 3 maps a call (A, B, C), encoded once
    launch(p, h, Ad, Bd, C2, p.N)                             # only C's map is new
    hits2, misses2 = h.tensor_map_cache_stats()
    assert misses2 - misses1 == 1 and hits2 - hits1 == 2
    assert h.status()[0] == G.OK
    for C in (C1, C2):
        assert_close(C.double().cpu().numpy(), R, Mag, True, "tensor-map cache")
