"""GPU parity of fp32 inputs against the oracle's fp64 product of the fp32
values: the fp32 GEMM from three TF32 products (GEMM_F32_F32) within the
bound of that emulation, one TF32 product per product (GEMM_TF32_F32) within
the TF32 bound.  Every layout (MN-major operands are written K-major first),
ragged sizes and leading dimensions, misaligned rows, the blend with C,
swapped skinny problems, split-K and stream-K, the fused epilogue, strided
batches, groups, K == 0 and the full 4096^3 size on sampled outputs.  The cut
to TF32 must not depend on the layout: an operand read as it is and the same
operand written K-major first give the same bits."""
import contextlib

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, oracle_at, oracle_full, run, sample_indices

pytestmark = pytest.mark.gpu

NORMAL = ("normal", 0.0, 1.0)


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


def check_close(out, R, Mag, K, code, what):
    if code == G.F32_F32:
        ok = oracle.within_tolerance(out, R, Mag, True, tf32x3_k=K)
    else:
        ok = oracle.within_tolerance(out, R, Mag, True, tf32=True)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError("%s: %d of %d outside tolerance; first %s gpu %r oracle %r mag %r"
                             % (what, (~ok).sum(), ok.size, i, out[i], R[i], Mag[i]))


def check(p, h, code, guard_cols=4):
    out, full = run(p, h, guard_rows=2, guard_cols=guard_cols, code=code)
    R, Mag = oracle_full(p)
    check_close(out, R, Mag, p.K, code, p.name)
    pad = full.clone().double()
    pad[:p.M, :p.N] = SENTINEL
    assert bool((pad == SENTINEL).all()), "C written outside M x N"
    return out, R, Mag


CODES = [G.F32_F32, G.TF32_F32]


@pytest.mark.parametrize("code", CODES)
@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_layouts(h, code, transA, transB):
    """Ragged M, N, K (K = 301: rows of 1204 bytes, so the one-pass path writes
    its K-major operands too) and a blend with C."""
    p = inputs.make_problem("f32_%d%d" % (transA, transB), 300, 328, 301, transA, transB, "f32", "f32", NORMAL,
                            NORMAL, alpha=0.75, beta=-0.5, seed=transA + 2 * transB)
    check(p, h, code)


@pytest.mark.parametrize("code", CODES)
def test_aligned_k_major_read_directly(h, code):
    p = inputs.make_problem("f32_nt", 520, 904, 512, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=5)
    plan = G.plan(p.M, p.N, p.K, 0, 1, code, handle=h)
    assert (plan.repack_a, plan.repack_b) == ((1, 1) if code == G.F32_F32 else (0, 0))
    check(p, h, code)


def test_tf32_cut_does_not_depend_on_layout(h):
    """NT operands read as they are vs the same values stored NN / TN (written
    K-major and cut on the way): bit-identical C."""
    p = inputs.make_problem("cut_nt", 384, 512, 640, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=6)
    out_nt, _ = run(p, h, code=G.TF32_F32)
    q = inputs.make_problem("cut_tn", 384, 512, 640, 1, 0, "f32", "f32", NORMAL, NORMAL, seed=6)
    q.A = p.A.t().contiguous()
    q.B = p.B.t().contiguous()
    q.lda, q.ldb = 384, 512
    assert G.plan(q.M, q.N, q.K, 1, 0, G.TF32_F32, handle=h).launches == 3
    out_tn, _ = run(q, h, code=G.TF32_F32)
    assert np.array_equal(out_nt, out_tn)


def test_three_products_beat_one(h):
    """The same inputs: the error of three TF32 products is far below one's
    (one: ~2^-11 relative per input; three: ~2^-22 plus the fp32 sum)."""
    p = inputs.make_problem("f32_acc", 512, 512, 1024, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=7)
    R, Mag = oracle_full(p)
    out3, _ = run(p, h, code=G.F32_F32)
    out1, _ = run(p, h, code=G.TF32_F32)
    e3 = np.abs(out3 - R) / Mag
    e1 = np.abs(out1 - R) / Mag
    check_close(out3, R, Mag, p.K, G.F32_F32, "3xTF32")
    check_close(out1, R, Mag, p.K, G.TF32_F32, "TF32")
    print("max err / mag: 3xTF32 %.3g (2^%.1f), TF32 %.3g (2^%.1f); median %.3g vs %.3g"
          % (e3.max(), np.log2(e3.max()), e1.max(), np.log2(e1.max()), np.median(e3), np.median(e1)))
    assert np.median(e1) > 256 * np.median(e3)


def test_three_products_statistical_bound_at_k4096(h):
    """A statistical check beside the worst-case rule: at K = 4096, on N(0, 1)
    inputs, the three-product result stays within 2^-16 of the magnitude m at
    every element (observed about 2^-21), a bound one TF32 product (about
    2^-12 of m) fails.  The worst-case rule alone, (3K 2^-23 + 2^-20) m = 2^-9.4
    m at this K, cannot tell the two apart."""
    p = inputs.make_problem("f32_k4096", 1024, 1024, 4096, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=12)
    R, Mag = oracle_full(p)
    out3, _ = run(p, h, code=G.F32_F32)
    out1, _ = run(p, h, code=G.TF32_F32)
    e3 = float((np.abs(out3 - R) / Mag).max())
    e1 = float((np.abs(out1 - R) / Mag).max())
    print("K = 4096, max err / mag: 3xTF32 2^%.1f, TF32 2^%.1f" % (np.log2(e3), np.log2(e1)))
    check_close(out3, R, Mag, p.K, G.F32_F32, "3xTF32 K=4096")
    assert e3 <= 2.0 ** -16, "three TF32 products: max err / mag 2^%.1f" % np.log2(e3)
    assert e1 > 2.0 ** -16, "one TF32 product should not meet the three-product bound"


@pytest.mark.parametrize("sched", ["split", "stream_k"])
def test_split_tiles(h, sched):
    p = inputs.make_problem("f32_sk", 700, 904, 1500, 0, 1, "f32", "f32", NORMAL, NORMAL, beta=0.25, seed=8)
    kw = dict(split=3) if sched == "split" else dict(grid=14, stream_k=2, path=G.PATH_TC_2CTA)
    with options(h, **kw):
        plan = G.plan(p.M, p.N, p.K, 0, 1, G.F32_F32, handle=h, beta=p.beta)
        assert (plan.split_k == 3) if sched == "split" else (plan.schedule == G.SCHED_STREAM_K)
        check(p, h, G.F32_F32)


@pytest.mark.parametrize("code", CODES)
def test_swapped_skinny(h, code):
    p = inputs.make_problem("f32_skinny", 16, 1000, 512, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=9)
    assert G.plan(p.M, p.N, p.K, 0, 1, code, handle=h).swap_ab == 1
    check(p, h, code)


def test_fused_epilogue(h):
    p = inputs.make_problem("f32_epi", 300, 520, 700, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=10)
    bias = torch.from_numpy(np.random.default_rng(10).normal(0, 2, p.N).astype(np.float32))
    C = torch.full((p.M, p.N), float("nan"), device="cuda")
    Ad, Bd, bd = p.A.cuda(), p.B.cuda(), bias.cuda()   # held until the kernel has run
    st = h.run_ex_raw(0, 1, p.M, p.N, p.K, 1.0, Ad.data_ptr(), p.lda, Bd.data_ptr(), p.ldb, 0.0,
                      C.data_ptr(), p.N, G.F32_F32, None, bias=bd.data_ptr(), act=G.ACT_GELU, out_scale=0.5)
    assert st == G.OK and h.status()[0] == G.OK
    R0, Mag0 = oracle_full(p)
    R, _ = oracle.epilogue(R0, Mag0, bias=bias.numpy(), act=G.ACT_GELU, scale=0.5)
    # GELU's slope is at most ~1.13, so the GEMM's error passes on scaled by at
    # most that; z = acc + bias and 0.5 z (1 + erf(z / sqrt 2)) in fp32 add a
    # few ulp of |z| (erf near -1 cancels in 1 + erf: the error is absolute).
    z = np.abs(R0 + bias.numpy().astype(np.float64))
    out = C.double().cpu().numpy()
    bound = 0.5 * (1.2 * (3 * p.K * 2.0 ** -23 + 2.0 ** -20) * Mag0 + 2.0 ** -20 * z) + 1e-30
    ok = np.abs(out - R) <= bound
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError("%d outside; first %s gpu %r oracle %r z %r bound %r"
                             % ((~ok).sum(), i, out[i], R[i], R0[i] + bias[i[1]].item(), bound[i]))


def test_strided_batches(h):
    M, N, K, batch = 200, 264, 150, 3
    p = inputs.make_batched_problem("f32_b", batch, M, N, K, 0, 0, "f32", "f32", NORMAL, NORMAL, beta=-0.25,
                                    seed=11, lda=K + 2, ldb=N + 4, ldc=N + 4, strideA=M * (K + 2) + 6,
                                    strideB=K * (N + 4) + 4, strideC=M * (N + 4) + 4)
    total = p.strideC * (batch - 1) + M * p.ldc + 16
    Cd = torch.full((total,), SENTINEL, device="cuda")
    for b in range(batch):
        Cd[b * p.strideC:b * p.strideC + M * p.ldc].view(M, p.ldc)[:, :N] = \
            p.C0[b * p.strideC:b * p.strideC + M * p.ldc].view(M, p.ldc)[:, :N].cuda()
    Ad, Bd = p.A.cuda(), p.B.cuda()
    st = h.run_batched_raw(0, 0, M, N, K, p.alpha, Ad.data_ptr(), p.lda, p.strideA, Bd.data_ptr(), p.ldb,
                           p.strideB, p.beta, Cd.data_ptr(), p.ldc, p.strideC, batch, G.F32_F32, None)
    assert st == G.OK and h.status()[0] == G.OK
    R, Mag = oracle.gemm_batched(0, 0, M, N, K, p.alpha, inputs.bits(p.A), p.lda, p.strideA, inputs.bits(p.B),
                                 p.ldb, p.strideB, p.beta, p.C0.numpy(), p.ldc, p.strideC, oracle.IN_F32, batch)
    full = Cd.cpu()
    for b in range(batch):
        out = full[b * p.strideC:b * p.strideC + M * p.ldc].view(M, p.ldc)[:, :N].double().numpy()
        check_close(out, R[b], Mag[b], K, G.F32_F32, "batch %d" % b)


def test_groups(h):
    sizes = [5, 0, 130, 1, 257]
    p = inputs.make_grouped_problem("f32_g", sizes, 264, 200, 1, "f32", "f32", NORMAL, NORMAL, seed=12)
    M = sum(sizes)
    Cd = torch.full((M + 2, p.ldc), SENTINEL, device="cuda")
    Ad, Bd = p.A.cuda(), p.B.cuda()
    st = h.run_grouped_raw(1, sizes, p.N, p.K, p.alpha, Ad.data_ptr(), p.lda, Bd.data_ptr(), p.ldb, p.strideB,
                           0.0, Cd.data_ptr(), p.ldc, G.F32_F32, None)
    assert st == G.OK and h.status()[0] == G.OK
    R, Mag = oracle.gemm_grouped(1, sizes, p.N, p.K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B), p.ldb,
                                 p.strideB, 0.0, None, p.ldc, oracle.IN_F32)
    full = Cd.cpu().double()
    check_close(full[:M, :p.N].numpy(), R, Mag, p.K, G.F32_F32, "groups")
    full[:M, :p.N] = SENTINEL
    assert bool((full == SENTINEL).all())


def test_k_zero(h):
    p = inputs.make_problem("f32_k0", 40, 50, 0, 0, 0, "f32", "f32", beta=-2.0, seed=13)
    check(p, h, G.F32_F32)


@pytest.mark.parametrize("code", CODES)
def test_square_4096_sampled(h, code):
    """4096^3 NT at the full size, in the launch configuration the benchmark times;
    2000 sampled outputs plus the edges against the oracle one by one."""
    p = inputs.make_problem("f32_4096", 4096, 4096, 4096, 0, 1, "f32", "f32", NORMAL, NORMAL, seed=14)
    out, _ = run(p, h, code=code)
    rows, cols = sample_indices(p.M, p.N, 2000, seed=14)
    R, Mag = oracle_at(p, rows, cols)
    check_close(out[rows, cols], R, Mag, p.K, code, p.name)


def test_tensor_binding(h):
    g = torch.Generator().manual_seed(15)
    A = torch.randn(300, 200, generator=g)
    B = torch.randn(200, 260, generator=g)
    ref = (A.double() @ B.double()).numpy()
    mag = (A.double().abs() @ B.double().abs()).numpy()
    for tf32 in (False, True):
        C = torch.empty(300, 260, device="cuda")
        G.gemm(A.cuda(), B.cuda(), C, tf32=tf32, handle=h)
        torch.cuda.synchronize()
        out = C.double().cpu().numpy()
        ok = oracle.within_tolerance(out, ref, mag, True, tf32=True) if tf32 else \
            oracle.within_tolerance(out, ref, mag, True, tf32x3_k=200)
        assert ok.all()
