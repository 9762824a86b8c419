"""GPU parity of strided batched GEMM (gemm_run_strided_batched) against the
batched oracle, batch by batch: every layout, gaps between batches (aligned
and misaligned, the latter repacked), shared A or B (stride 0), many small
GEMMs filling the GPU together, attention-shaped products, swapped skinny
batches, split-K and stream-K across batches, 8-bit inputs, K == 0 and the
fused bias.  The memory between and after the batches' C must stay untouched."""
import contextlib

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, assert_close, dtype_code

pytestmark = pytest.mark.gpu

_T = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
_OIN = {"bf16": oracle.IN_BF16, "f16": oracle.IN_F16, "e4m3": oracle.IN_E4M3, "e5m2": oracle.IN_E5M2}


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


def oracle_batched(p, bias=None):
    if p.beta == 0.0 or p.C0 is None:
        c0, ct = None, oracle.C_F32
    elif p.out_dtype == "f32":
        c0, ct = p.C0.numpy(), oracle.C_F32
    else:
        c0, ct = inputs.bits(p.C0), oracle.C_BF16 if p.out_dtype == "bf16" else oracle.C_F16
    R, Mag = oracle.gemm_batched(p.transA, p.transB, p.M, p.N, p.K, p.alpha, inputs.bits(p.A), p.lda, p.strideA,
                                 inputs.bits(p.B), p.ldb, p.strideB, p.beta, c0, p.ldc, p.strideC,
                                 _OIN[p.in_dtype], p.batch, c_type=ct, b_type=_OIN[p.b_dtype])
    if bias is not None:
        for b in range(p.batch):
            R[b], Mag[b] = oracle.epilogue(R[b], Mag[b], bias=bias.numpy())
    return R, Mag


def run_batched(p, h, bias=None):
    """Run p; returns (outputs as fp64 batch x M x N, the whole C buffer)."""
    total = p.strideC * (p.batch - 1) + p.M * p.ldc + 64   # 64 guard elements after the last batch
    Cd = torch.full((total,), SENTINEL, dtype=_T[p.out_dtype], device="cuda")
    for b in range(p.batch):
        view = Cd[b * p.strideC:b * p.strideC + p.M * p.ldc].view(p.M, p.ldc)
        if p.beta != 0.0:
            view[:, :p.N] = p.C0[b * p.strideC:b * p.strideC + p.M * p.ldc].view(p.M, p.ldc)[:, :p.N].cuda()
        else:
            view[:, :p.N] = float("nan")
    Ad, Bd = p.A.cuda(), p.B.cuda()
    bd = bias.cuda() if bias is not None else None
    st = h.run_batched_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, Ad.data_ptr(), p.lda, p.strideA,
                           Bd.data_ptr(), p.ldb, p.strideB, p.beta, Cd.data_ptr(), p.ldc, p.strideC, p.batch,
                           dtype_code(p), None, bias=bd.data_ptr() if bd is not None else 0)
    assert st == G.OK, G.STATUS.get(st)
    assert h.status()[0] == G.OK
    full = Cd.cpu()
    outs = np.stack([full[b * p.strideC:b * p.strideC + p.M * p.ldc].view(p.M, p.ldc)[:, :p.N].double().numpy()
                     for b in range(p.batch)])
    return outs, full


def check(p, h, bias=None):
    out, full = run_batched(p, h, bias)
    R, Mag = oracle_batched(p, bias)
    for b in range(p.batch):
        assert_close(out[b], R[b], Mag[b], p.out_dtype == "f32", "%s batch %d" % (p.name, b))
    pad = full.clone().double()
    for b in range(p.batch):
        pad[b * p.strideC:b * p.strideC + p.M * p.ldc].view(p.M, p.ldc)[:, :p.N] = SENTINEL
    assert bool((pad == SENTINEL).all()), "C written outside the batches' M x N blocks"


def plan_of(p, h=None):
    return G.plan_batched(p.M, p.N, p.K, p.batch, p.transA, p.transB, dtype_code(p), lda=p.lda, ldb=p.ldb,
                          ldc=p.ldc, strideA=p.strideA, strideB=p.strideB, strideC=p.strideC, beta=p.beta,
                          handle=h)


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_layouts_with_gaps(h, transA, transB, out):
    """Ragged sizes, leading dimensions and 16-byte-aligned gaps between batches."""
    M, N, K, batch = 200, 328, 150, 3
    a_rows, b_rows = (K if transA else M), (N if transB else K)
    up8 = lambda x: (x + 7) // 8 * 8 + 8            # 16-byte rows with padding
    lda, ldb = up8(M if transA else K), up8(K if transB else N)
    p = inputs.make_batched_problem("bl", batch, M, N, K, transA, transB, "bf16", out, ("normal", 0, 1),
                                    ("normal", 0, 1), alpha=0.5, beta=-0.25, seed=transA + 2 * transB,
                                    lda=lda, ldb=ldb, ldc=N + 8, strideA=a_rows * lda + 16,
                                    strideB=b_rows * ldb + 32, strideC=M * (N + 8) + 8)
    plan = plan_of(p)
    assert plan.batch == batch and plan.repack_a == 0 and plan.repack_b == 0
    check(p, h)


@pytest.mark.parametrize("shared", ["A", "B"])
def test_shared_operand(h, shared):
    p = inputs.make_batched_problem("bs", 5, 300, 264, 200, 0, 1, "f16", "f32", ("uniform", -1, 1),
                                    ("uniform", -1, 1), seed=11, strideA=0 if shared == "A" else None,
                                    strideB=0 if shared == "B" else None)
    check(p, h)


def test_misaligned_batch_strides_repack(h):
    p = inputs.make_batched_problem("bm", 4, 130, 200, 70, 0, 0, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                                    seed=12, strideA=130 * 70 + 3, strideB=70 * 200 + 5, strideC=130 * 200 + 3)
    plan = plan_of(p)
    # (C's batches start off 16-byte boundaries: each row leaves through its own bulk copy)
    assert plan.repack_a == 1 and plan.repack_b == 1 and plan.bulk_store == G.BULK_ROW_COPIES
    check(p, h)


def test_many_small_gemms_fill_the_gpu(h):
    """64 GEMMs of 64 x 96 x 64: one tile each, all in one launch."""
    p = inputs.make_batched_problem("bsmall", 64, 64, 96, 64, 0, 1, "bf16", "bf16", ("normal", 0, 1),
                                    ("normal", 0, 1), seed=13)
    plan = plan_of(p)
    assert plan.tiles >= 64 and plan.launches == 1
    check(p, h)


@pytest.mark.parametrize("which", ["scores", "values"])
def test_attention_shapes(h, which):
    """Q K^T (NT, alpha 1/sqrt(d)) and P V (NN) for 8 heads of 512 tokens, d = 64."""
    if which == "scores":
        p = inputs.make_batched_problem("qk", 8, 512, 512, 64, 0, 1, "bf16", "bf16", ("normal", 0, 1),
                                        ("normal", 0, 1), alpha=0.125, seed=14)
    else:
        p = inputs.make_batched_problem("pv", 8, 512, 64, 512, 0, 0, "bf16", "bf16", ("uniform", 0, 1.0 / 256),
                                        ("normal", 0, 1), seed=15)
    check(p, h)


def test_swapped_skinny_batches(h):
    """M = 16 per batch: the swap to C^T holds per batch; B shared."""
    p = inputs.make_batched_problem("bsk", 4, 16, 1000, 256, 0, 1, "bf16", "f32", ("normal", 0, 1),
                                    ("normal", 0, 1), seed=16, strideB=0)
    assert plan_of(p).swap_ab == 1
    check(p, h)


@pytest.mark.parametrize("sched", ["split", "stream_k"])
def test_split_tiles_across_batches(h, sched):
    p = inputs.make_batched_problem("bsplit", 3, 300, 520, 960, 0, 1, "bf16", "f32", ("normal", 0, 1),
                                    ("normal", 0, 1), beta=0.5, seed=17)
    kw = dict(split=3) if sched == "split" else dict(grid=14, stream_k=2, path=G.PATH_TC_2CTA)
    with options(h, **kw):
        plan = plan_of(p, h)
        assert (plan.split_k == 3) if sched == "split" else (plan.schedule == G.SCHED_STREAM_K)
        check(p, h)


def test_fp8_batches(h):
    p = inputs.make_batched_problem("b8", 3, 256, 384, 300, 0, 1, "e4m3", "f32", ("normal", 0, 1),
                                    ("normal", 0, 1), seed=18, b_dtype="e5m2")
    check(p, h)


def test_k_zero_batches(h):
    p = inputs.make_batched_problem("bk0", 3, 40, 50, 0, 0, 0, "bf16", "f32", beta=-2.0, seed=19,
                                    strideC=40 * 50 + 10)
    check(p, h)


def test_bias_shared_by_batches(h):
    p = inputs.make_batched_problem("bbias", 3, 200, 264, 128, 0, 1, "bf16", "bf16", ("normal", 0, 1),
                                    ("normal", 0, 1), seed=20)
    bias = torch.from_numpy(np.random.default_rng(20).normal(0, 2, 264).astype(np.float32))
    check(p, h, bias=bias)
