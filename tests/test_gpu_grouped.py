"""GPU parity of grouped GEMM (gemm_run_grouped: stacked rows, one weight
matrix per group, as a mixture-of-experts layer routes tokens) against the
grouped oracle: empty, single-row and multi-tile groups, both weight
layouts, the blend with C, 8-bit inputs, the fused epilogue, split-K and
stream-K fix-ups, shared weights and K == 0.  Rows past the last group and
columns past N must stay untouched."""
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


def oracle_grouped(p, bias=None, act=G.ACT_NONE, scale=1.0):
    if p.beta == 0.0:
        c0, ct = None, oracle.C_F32
    elif p.out_dtype == "f32":
        c0, ct = p.C0.numpy(), oracle.C_F32
    else:
        c0, ct = inputs.bits(p.C0), oracle.C_BF16 if p.out_dtype == "bf16" else oracle.C_F16
    R, Mag = oracle.gemm_grouped(p.transB, p.m_sizes, p.N, p.K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B),
                                 p.ldb, p.strideB, p.beta, c0, p.ldc, _OIN[p.in_dtype], c_type=ct,
                                 b_type=_OIN[p.b_dtype])
    if bias is not None or act != G.ACT_NONE or scale != 1.0:
        R, Mag = oracle.epilogue(R, Mag, bias=None if bias is None else bias.numpy(), act=act, scale=scale)
    return R, Mag


def check(p, h, bias=None, act=G.ACT_NONE, scale=1.0, guard_rows=3):
    M = p.M
    Cd = torch.full((M + guard_rows, p.ldc), SENTINEL, dtype=_T[p.out_dtype], device="cuda")
    if p.beta != 0.0:
        Cd[:M, :p.N] = p.C0[:, :p.N].cuda()
    else:
        Cd[:M, :p.N] = float("nan")
    Ad, Bd = p.A.cuda(), p.B.cuda()
    bd = bias.cuda() if bias is not None else None
    st = h.run_grouped_raw(p.transB, p.m_sizes, p.N, p.K, p.alpha, Ad.data_ptr(), p.lda, Bd.data_ptr(), p.ldb,
                           p.strideB, p.beta, Cd.data_ptr(), p.ldc, dtype_code(p), None,
                           bias=bd.data_ptr() if bd is not None else 0, act=act, out_scale=scale)
    assert st == G.OK, G.STATUS.get(st)
    assert h.status()[0] == G.OK
    full = Cd.cpu()
    R, Mag = oracle_grouped(p, bias, act, scale)
    if M:
        assert_close(full[:M, :p.N].double().numpy(), R, Mag, p.out_dtype == "f32", p.name)
    pad = full.clone().double()
    pad[:M, :p.N] = SENTINEL
    assert bool((pad == SENTINEL).all()), "C written outside the groups' rows and columns"


SIZES = [5, 0, 130, 1, 257, 64]


@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_groups_both_weight_layouts(h, transB, out):
    """Empty, single-row and multi-tile groups; tiles that straddle two groups' rows."""
    p = inputs.make_grouped_problem("grp", SIZES, 300, 200, transB, "bf16", out, seed=transB, alpha=2.0,
                                    ldc=305)
    check(p, h)


def test_blend_with_c(h):
    p = inputs.make_grouped_problem("grpb", SIZES, 264, 320, 1, "f16", "f16", ("uniform", -1, 1), ("uniform", -1, 1),
                                    alpha=1.5, beta=-0.5, seed=3)
    check(p, h)


def test_fp8_groups(h):
    p = inputs.make_grouped_problem("grp8", SIZES, 256, 384, 1, "e4m3", "f32", ("normal", 0, 1), ("normal", 0, 1),
                                    seed=4, b_dtype="e5m2")
    check(p, h)


@pytest.mark.parametrize("act", [G.ACT_RELU, G.ACT_GELU])
def test_fused_epilogue(h, act):
    p = inputs.make_grouped_problem("grpe", SIZES, 272, 256, 1, "bf16", "bf16", seed=5)
    bias = torch.from_numpy(np.random.default_rng(5).normal(0, 1, 272).astype(np.float32))
    check(p, h, bias=bias, act=act, scale=0.5)


@pytest.mark.parametrize("sched", ["split", "stream_k"])
def test_split_groups(h, sched):
    p = inputs.make_grouped_problem("grps", [200, 0, 70, 300], 520, 960, 1, "bf16", "f32", seed=6, beta=0.25)
    kw = dict(split=3) if sched == "split" else dict(grid=10, stream_k=2, path=G.PATH_TC_1CTA)
    with options(h, **kw):
        check(p, h)


@pytest.mark.parametrize("path", [G.PATH_TC_1CTA, G.PATH_TC_2CTA])
def test_every_path(h, path):
    p = inputs.make_grouped_problem("grpp", [300, 40, 0, 500, 9], 400, 192, 1, "bf16", "f32", seed=7)
    with options(h, path=path):
        assert G.plan_grouped(p.m_sizes, p.N, p.K, 1, handle=h).path == path
        check(p, h)


def test_shared_weights_and_k_zero(h):
    p = inputs.make_grouped_problem("grpw", [40, 33, 0, 90], 200, 96, 1, "bf16", "f32", seed=8, strideB=0)
    check(p, h)
    q = inputs.make_grouped_problem("grpk0", [4, 0, 7], 50, 0, 1, "bf16", "f32", seed=9, beta=2.0)
    check(q, h)


def test_moe_layer_shape(h):
    """16 experts, 2048 routed tokens (uneven), d_model 1024 -> d_ff 512."""
    sizes = inputs.moe_routing(2048, 16, seed=1)
    p = inputs.make_grouped_problem("moe", sizes, 512, 1024, 1, "bf16", "bf16", seed=10)
    check(p, h)


def test_no_groups_is_a_noop(h):
    C = torch.full((4, 4), 7.0, device="cuda")
    st = h.run_grouped_raw(1, [], 4, 4, 1.0, 0, 4, 0, 4, 16, 0.0, C.data_ptr(), 4, G.BF16_F32, None)
    assert st == G.OK and bool((C == 7.0).all())
