"""GPU parity of the 8-bit float path (tcgen05.mma kind::f8f6f4) against the
CPU oracle, element by element: both FP8 formats and their mixed pairs, every
output type, ragged sizes (K not a multiple of the 128-element k-slice),
every 8-bit tile configuration with one and two k-slices per stage, stream-K
and split-K fix-ups, the swapped skinny path, repacked operands and exact
small-integer products.  Every call goes through the C ABI."""
import contextlib

import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, assert_close, dtype_code, oracle_at, oracle_full, run

pytestmark = pytest.mark.gpu

CONFIGS8 = [(1, 64), (1, 128), (2, 128), (2, 256)]
PATHS = {1: G.PATH_TC_1CTA, 2: G.PATH_TC_2CTA}
PAIRS = [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")]


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


@contextlib.contextmanager
def options(h, **kw):
    codes = {"path": G.OPT_FORCE_PATH, "bn": G.OPT_FORCE_BN, "split": G.OPT_SPLIT_K, "grid": G.OPT_MAX_GRID,
             "stream_k": G.OPT_STREAM_K, "kdepth": G.OPT_KDEPTH}
    try:
        for k, v in kw.items():
            h.set_option(codes[k], v)
        yield
    finally:
        for k in kw:
            h.set_option(codes[k], 0)


def problem(name, M, N, K, fa="e4m3", fb="e4m3", out="f32", seed=0, dist=("normal", 0, 1), **kw):
    return inputs.make_problem(name, M, N, K, 0, 1, fa, out, dist, dist, seed=seed, b_dtype=fb, **kw)


def check(p, h, guard_cols=5):
    out, full = run(p, h, guard_rows=3, guard_cols=guard_cols)
    R, Mag = oracle_full(p)
    assert_close(out, R, Mag, p.out_dtype == "f32", p.name)
    pad = full.clone().to(torch.float64)
    pad[:p.M, :p.N] = SENTINEL
    assert torch.all(pad == SENTINEL), "C written outside the M x N block"


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("fa,fb", PAIRS)
def test_formats_and_outputs(h, fa, fb, out):
    """Ragged in every dimension (K = 300: two full 128-element slices and a partial one)."""
    p = problem("f8", 300, 520, 300, fa, fb, out, seed=len(fa + fb + out), alpha=0.5, beta=-0.75)
    check(p, h)


@pytest.mark.parametrize("kdepth", [1, 2])
@pytest.mark.parametrize("cg,bn", CONFIGS8)
def test_every_configuration(h, cg, bn, kdepth):
    """K = 700: five full k-slices and a partial sixth; bulk-store epilogue (guard keeps rows aligned)."""
    p = problem("f8cfg", 600, 904, 700, "e4m3", "e5m2", "bf16", seed=bn + cg + kdepth)
    with options(h, path=PATHS[cg], bn=bn, kdepth=kdepth):
        plan = G.plan(p.M, p.N, p.K, 0, 1, dtype_code(p), handle=h, ldc=p.ldc + 8)
        assert plan.bn == bn and plan.path == PATHS[cg] and plan.kdepth == kdepth and plan.bk == 128 * kdepth
        assert plan.bulk_store == G.BULK_ROWS
        check(p, h, guard_cols=8)


@pytest.mark.parametrize("cg,bn", CONFIGS8)
def test_stream_k(h, cg, bn):
    """Stream-K tail forced on a small grid, and a deep K shared by every tile."""
    grid = {1: 13, 2: 14}[cg]
    p = problem("f8sk", 700, 900, 1500, "e4m3", "e4m3", "f32", seed=grid + bn, alpha=1.25, beta=0.5)
    with options(h, path=PATHS[cg], bn=bn, grid=grid, stream_k=2):
        plan = G.plan(p.M, p.N, p.K, 0, 1, dtype_code(p), handle=h, beta=p.beta)
        assert plan.schedule == G.SCHED_STREAM_K
        check(p, h)
    q = problem("f8deep", 250, 250, 6000, "e5m2", "e4m3", "f16", seed=bn * cg)
    with options(h, path=PATHS[cg], bn=bn, stream_k=2):
        assert G.plan(q.M, q.N, q.K, 0, 1, dtype_code(q), handle=h).dp_tiles == 0
        check(q, h)


@pytest.mark.parametrize("split", [2, 5])
def test_split_k(h, split):
    p = problem("f8split", 300, 520, 1100, "e4m3", "e4m3", "f32", seed=split, beta=1.5)
    with options(h, split=split):
        assert G.plan(p.M, p.N, p.K, 0, 1, dtype_code(p), handle=h, beta=p.beta).split_k == split
        check(p, h)


@pytest.mark.parametrize("M,N,K", [(64, 3000, 4096), (1, 1032, 256), (40, 1000, 700)])
def test_skinny_swapped(h, M, N, K):
    """Short M: C^T = B A^T with the operands' formats swapped too (A E4M3, B E5M2)."""
    p = problem("f8skinny", M, N, K, "e4m3", "e5m2", "f32", seed=N)
    assert G.plan(M, N, K, 0, 1, dtype_code(p)).swap_ab == 1
    check(p, h, guard_cols=8)


def test_misaligned_rows_are_repacked(h):
    """Row pitches that are not multiples of 16 bytes: the 8-bit repack kernel."""
    p = problem("f8mis", 333, 517, 301, "e5m2", "e4m3", "f32", seed=9, lda=309, ldb=307)
    plan = G.plan(p.M, p.N, p.K, 0, 1, dtype_code(p), lda=p.lda, ldb=p.ldb, ldc=p.ldc + 5)
    assert plan.repack_a == 1 and plan.repack_b == 1
    check(p, h)


@pytest.mark.parametrize("fa,fb", PAIRS)
def test_small_integers_bit_exact(h, fa, fb):
    """Integers in {-8..8} are exact in both formats and their products and sums
    are exact in fp32: the GPU must equal the oracle bit for bit."""
    p = problem("f8ints", 384, 640, 2048, fa, fb, "f32", seed=5, dist=("ints", -8, 8), alpha=2.0)
    out, _ = run(p, h)
    R, _ = oracle_full(p)
    assert np.array_equal(out, R)


def test_full_size_square_sampled(h):
    """4096^3 E4M3 NT in the launch configuration the benchmark times, checked on
    sampled outputs (every tile row and column band, edges included)."""
    p = inputs.square_4096_fp8_nt("e4m3", "f32")
    out, _ = run(p, h)
    g = np.random.default_rng(0)
    rows = np.concatenate([[0, 4095, 255, 256], g.integers(0, 4096, 400)])
    cols = np.concatenate([[4095, 0, 256, 255], g.integers(0, 4096, 400)])
    r, m = oracle_at(p, rows, cols)
    assert_close(out[rows, cols], r, m, True, p.name)
