"""GPU parity of the fused epilogue (gemm_run_ex): per-column bias, ReLU / GELU
and the output scale, against the oracle's epilogue applied to the fp64 GEMM,
on every store path: bulk stores of rows, bulk stores of transposed blocks
(swapped problems), direct stores (beta != 0, misaligned C), stream-K and
split-K fix-ups, 8-bit inputs, the quantised E4M3 output and K == 0."""
import contextlib

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, dtype_code, oracle_full

pytestmark = pytest.mark.gpu

ACTS = [G.ACT_NONE, G.ACT_RELU, G.ACT_GELU]
_T = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn}


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


@contextlib.contextmanager
def options(h, **kw):
    codes = {"path": G.OPT_FORCE_PATH, "bn": G.OPT_FORCE_BN, "split": G.OPT_SPLIT_K, "grid": G.OPT_MAX_GRID,
             "stream_k": G.OPT_STREAM_K}
    try:
        for k, v in kw.items():
            h.set_option(codes[k], v)
        yield
    finally:
        for k in kw:
            h.set_option(codes[k], 0)


def bias_for(N, seed):
    return torch.from_numpy(np.random.default_rng(seed).normal(0, 2, N).astype(np.float32))


def run_ex(p, h, bias, act, scale, guard_cols=8, expect_bulk=None):
    """Run p through gemm_run_ex; returns (C as fp64 numpy M x N, whole C buffer)."""
    ldc = p.ldc + guard_cols
    out_t = _T[p.out_dtype]
    if p.out_dtype == "e4m3":
        Cd = torch.full((p.M + 2, ldc), 0x3C, dtype=torch.uint8, device="cuda").view(out_t)  # 1.5 as sentinel
    else:
        Cd = torch.full((p.M + 2, ldc), SENTINEL, dtype=out_t, device="cuda")
        if p.beta != 0.0:
            Cd[:p.M, :p.N] = p.C0[:, :p.N].cuda()
        else:
            Cd[:p.M, :p.N] = float("nan")
    if expect_bulk is not None:
        plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, dtype_code(p), handle=h, ldc=ldc, beta=p.beta)
        assert plan.bulk_store == expect_bulk, plan.as_dict()
    Ad, Bd = p.A.cuda(), p.B.cuda()
    bd = bias.cuda() if bias is not None else None
    st = h.run_ex_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, Ad.data_ptr(), p.lda, Bd.data_ptr(), p.ldb,
                      p.beta, Cd.data_ptr(), ldc, dtype_code(p), None,
                      bias=bd.data_ptr() if bd is not None else 0, act=act, out_scale=scale)
    assert st == G.OK, G.STATUS.get(st)
    assert h.status()[0] == G.OK
    full = Cd.cpu()
    return full[:p.M, :p.N].to(torch.float64).numpy(), full


def check(p, h, bias, act, scale, **kw):
    out, full = run_ex(p, h, bias, act, scale, **kw)
    R, Mag = oracle_full(p)
    R, Mag = oracle.epilogue(R, Mag, bias=None if bias is None else bias.numpy(), act=act, scale=scale)
    e4 = p.out_dtype == "e4m3"
    ok = oracle.within_tolerance(out, R, Mag, p.out_dtype == "f32", e4m3=e4)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError("%s: %d outside tolerance; first %s gpu %r oracle %r mag %r"
                             % (p.name, (~ok).sum(), i, out[i], R[i], Mag[i]))
    # nothing outside the M x N block was written
    if e4:
        raw = full.view(torch.uint8).clone()
        raw[:p.M, :p.N] = 0x3C
        assert bool((raw == 0x3C).all())
    else:
        pad = full.clone().to(torch.float64)
        pad[:p.M, :p.N] = SENTINEL
        assert bool((pad == SENTINEL).all())


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_rows_bulk_store(h, act, out):
    """beta == 0 and aligned C: bulk stores of rows carry the fused operations."""
    p = inputs.make_problem("epi_rows", 600, 904, 300, 0, 1, "bf16", out, ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.5, seed=act)
    check(p, h, bias_for(p.N, 1), act, 0.75, expect_bulk=G.BULK_ROWS)


@pytest.mark.parametrize("act", ACTS)
def test_transposed_bulk_store(h, act):
    """Swapped problem (M = 40): the bias runs along the kernel's rows."""
    p = inputs.make_problem("epi_swap", 40, 2000, 700, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            seed=10 + act)
    check(p, h, bias_for(p.N, 2), act, -1.25, expect_bulk=G.BULK_TRANSPOSED)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1)])
def test_direct_store_with_blend(h, act, transA, transB):
    """beta != 0: the blend with the old C comes before the bias and activation."""
    p = inputs.make_problem("epi_blend", 300, 520, 200, transA, transB, "f16", "f16", ("uniform", -1, 1),
                            ("uniform", -1, 1), alpha=1.5, beta=-0.5, seed=20 + act)
    check(p, h, bias_for(p.N, 3), act, 2.0, guard_cols=5, expect_bulk=G.BULK_NONE)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("out,guard", [("f32", 5), ("bf16", 3), ("f32", 7)])
@pytest.mark.parametrize("mode", [0, 3, 4])
def test_misaligned_c(h, act, out, guard, mode):
    """C whose rows bulk tensor stores cannot write (misaligned, or ending
    inside a 16-byte piece): the operations ride on the row-class stores (fp32
    C, auto), on the per-row bulk copies (GEMM_OPT_EPILOGUE = 4) or on the bulk
    stores into the aligned workspace copy that the copy kernel then writes
    into C (3), M x N elements only."""
    if mode == 0 and out != "f32":
        pytest.skip("row classes are planned for fp32 C")
    p = inputs.make_problem("epi_misaligned", 1100, 1001, 300, 0, 1, "bf16", out, ("normal", 0, 1),
                            ("normal", 0, 1), alpha=0.5, seed=40 + act + guard)
    h.set_option(G.OPT_EPILOGUE, mode)
    try:
        expect = {0: G.BULK_ROW_CLASSES, 3: G.BULK_STAGED, 4: G.BULK_ROW_COPIES}[mode]
        check(p, h, bias_for(p.N, 5), act, 0.75, guard_cols=guard, expect_bulk=expect)
    finally:
        h.set_option(G.OPT_EPILOGUE, 0)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 1)])
def test_bulk_store_with_blend(h, act, transA, transB):
    """beta != 0 with rows bulk stores can write: the old C arrives by tensor
    loads into the staging buffer; the blend comes before the bias and activation."""
    p = inputs.make_problem("epi_blend_bulk", 300, 520, 200, transA, transB, "f16", "f16", ("uniform", -1, 1),
                            ("uniform", -1, 1), alpha=1.5, beta=-0.5, seed=30 + act)
    check(p, h, bias_for(p.N, 4), act, 2.0, guard_cols=8, expect_bulk=G.BULK_ROWS)


@pytest.mark.parametrize("sched", ["split", "stream_k"])
def test_fix_up_paths(h, sched):
    """Split tiles: the operations apply once, to the summed tile, never to partials."""
    p = inputs.make_problem("epi_sk", 700, 904, 1500, 0, 1, "bf16", "bf16", ("normal", 0, 1), ("normal", 0, 1),
                            seed=31)
    kw = dict(split=3) if sched == "split" else dict(grid=14, stream_k=2, path=G.PATH_TC_2CTA)
    with options(h, **kw):
        check(p, h, bias_for(p.N, 4), G.ACT_GELU, 0.5)


def test_no_bias_scale_only(h):
    p = inputs.make_problem("epi_scale", 256, 384, 512, 0, 1, "bf16", "f32", seed=4)
    check(p, h, None, G.ACT_NONE, 3.0)


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e4m3", "e5m2")])
def test_fp8_inputs(h, fa, fb):
    p = inputs.make_problem("epi_f8", 300, 520, 700, 0, 1, fa, "bf16", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.125, seed=5, b_dtype=fb)
    check(p, h, bias_for(p.N, 5), G.ACT_RELU, 1.0)


@pytest.mark.parametrize("act", [G.ACT_NONE, G.ACT_GELU])
@pytest.mark.parametrize("fin", ["bf16", "e4m3"])
@pytest.mark.parametrize("N", [1024, 1000])
def test_e4m3_quantised_output(h, act, fin, N):
    """E4M3 C: out_scale is the quantisation scale, values saturate at +-448.
    N = 1000 with a 1008-wide C keeps 16-byte rows (vector stores); the scale
    drives part of the outputs past 448."""
    p = inputs.make_problem("epi_q8", 300, N, 512, 0, 1, fin, "e4m3", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=1.0 / 16, seed=6)
    check(p, h, bias_for(p.N, 6), act, 100.0, guard_cols=8, expect_bulk=G.BULK_NONE)


@pytest.mark.parametrize("out", ["f32", "bf16", "e4m3"])
def test_k_zero_applies_the_operations(h, out):
    """K == 0: z = beta * C + bias, then the activation and scale."""
    M, N = 70, 90
    beta = 0.5 if out != "e4m3" else 0.0
    p = inputs.make_problem("epi_k0", M, N, 0, 0, 0, "bf16", out, beta=beta, seed=7)
    check(p, h, bias_for(N, 7), G.ACT_GELU, 1.5, guard_cols=3)


def test_bad_epilogue_arguments(h):
    A = torch.zeros(8, 8, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(8, 8, device="cuda")
    st = h.run_ex_raw(0, 1, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0, C.data_ptr(), 8, G.BF16_F32,
                      None, act=7)
    assert st == G.ERR_INVALID_ARG
    st = h.run_ex_raw(0, 1, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0, C.data_ptr(), 8, G.BF16_F32,
                      None, out_scale=float("inf"))
    assert st == G.ERR_INVALID_ARG
    b = torch.zeros(16, device="cuda")
    st = h.run_ex_raw(0, 1, 8, 8, 8, 1.0, A.data_ptr(), 8, A.data_ptr(), 8, 0.0, C.data_ptr(), 8, G.BF16_F32,
                      None, bias=b.data_ptr() + 2)
    assert st == G.ERR_INVALID_ARG


def test_tensor_binding_bias_gelu(h):
    p = inputs.make_problem("epi_bind", 200, 300, 100, 0, 1, "bf16", "bf16", seed=8)
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.empty(200, 300, dtype=torch.bfloat16, device="cuda")
    b = bias_for(300, 8)
    G.gemm(A, B, C, transB=True, bias=b.cuda(), act=G.ACT_GELU, out_scale=0.5, handle=h)
    torch.cuda.synchronize()
    R, Mag = oracle_full(p)
    R, Mag = oracle.epilogue(R, Mag, bias=b.numpy(), act=G.ACT_GELU, scale=0.5)
    assert oracle.within_tolerance(C.double().cpu().numpy(), R, Mag, False).all()


EW_CASES = [  # name, M, N, K, transA, transB, inputs, C, beta, guard columns, GEMM_OPT_EPILOGUE, store path
    ("rows", 600, 904, 300, 0, 1, "bf16", "f32", 0.0, 8, 0, G.BULK_ROWS),
    ("rows_bf16", 600, 904, 300, 0, 1, "bf16", "bf16", 0.0, 8, 0, G.BULK_ROWS),
    ("blend", 300, 520, 200, 1, 1, "f16", "f16", -0.5, 8, 0, G.BULK_ROWS),
    ("direct_blend", 300, 520, 200, 0, 0, "f16", "f16", -0.5, 5, 0, G.BULK_NONE),
    ("classes", 1100, 1001, 300, 0, 1, "bf16", "f32", 0.0, 5, 0, G.BULK_ROW_CLASSES),
    ("row_copies", 1100, 1001, 300, 0, 1, "bf16", "bf16", 0.0, 3, 4, G.BULK_ROW_COPIES),
    ("staged", 1100, 1001, 300, 0, 1, "bf16", "f32", 0.0, 7, 3, G.BULK_STAGED),
]


@pytest.mark.parametrize("ew", [4, 8])
@pytest.mark.parametrize("case", EW_CASES, ids=lambda c: c[0])
def test_epilogue_warps(h, case, ew):
    """The 256-wide CTA-pair tile with four or with eight epilogue warps (two
    per tensor-memory lane quarter, each storing half of a tile's columns) on
    every store path, with the fused operations."""
    name, M, N, K, ta, tb, fin, fout, beta, guard, mode, bulk = case
    p = inputs.make_problem("epi_ew_" + name, M, N, K, ta, tb, fin, fout, ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.5, beta=beta, seed=50 + ew + len(name))
    h.set_option(G.OPT_EPILOGUE, mode)
    h.set_option(G.OPT_EPILOGUE_WARPS, ew)
    try:
        with options(h, path=G.PATH_TC_2CTA, bn=256):
            plan = G.plan(p.M, p.N, p.K, ta, tb, dtype_code(p), handle=h, ldc=p.ldc + guard, beta=p.beta)
            assert plan.epilogue_warps == ew and plan.bn == 256 and plan.bm == 256
            check(p, h, bias_for(p.N, 6), G.ACT_GELU, 0.75, guard_cols=guard, expect_bulk=bulk)
    finally:
        h.set_option(G.OPT_EPILOGUE, 0)
        h.set_option(G.OPT_EPILOGUE_WARPS, 0)


@pytest.mark.parametrize("sched", ["split", "stream_k"])
def test_epilogue_warps_fix_up(h, sched):
    """Eight epilogue warps on split tiles: each warp writes and sums its half
    of the columns of every partial."""
    p = inputs.make_problem("epi_ew_sk", 700, 904, 1500, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            seed=57)
    kw = dict(split=3) if sched == "split" else dict(grid=14, stream_k=2)
    h.set_option(G.OPT_EPILOGUE_WARPS, 8)
    try:
        with options(h, path=G.PATH_TC_2CTA, bn=256, **kw):
            assert G.plan(p.M, p.N, p.K, 0, 1, handle=h, ldc=p.ldc + 8).epilogue_warps == 8
            check(p, h, bias_for(p.N, 7), G.ACT_RELU, 1.5)
    finally:
        h.set_option(G.OPT_EPILOGUE_WARPS, 0)
