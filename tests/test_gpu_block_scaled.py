"""GPU parity of block-scaled GEMMs (gemm_run_block_scaled: MXFP8 codes with
E8M0 scales per 32 values of k, NVFP4 E2M1 codes with unsigned E4M3 scales per
16) against the block-scaled oracle: every code pair, ragged M, N and K
(partial last blocks, odd K for FP4), padded leading dimensions, the blend
with C, every output type, swapped skinny problems, the fused epilogue, K == 0
and sampled outputs at 4096^3.  Scale rows are padded with NaN codes and
matrix rows with 0xFF bytes, which must never be read; nothing outside C's
M x N block may be written."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, assert_close, sample_indices

pytestmark = pytest.mark.gpu

_T = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
_ET = {"e4m3": oracle.IN_E4M3, "e5m2": oracle.IN_E5M2, "e2m1": oracle.IN_E2M1}


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


def code_of(p):
    if p.fmt == "nvfp4":
        return {"f32": G.NVFP4_F32, "bf16": G.NVFP4_BF16, "f16": G.NVFP4_F16}[p.out_dtype]
    return G.mxfp8_dtype(p.a_elem, p.b_elem, p.out_dtype)


def reference(p, rows=None, cols=None):
    c0, ct = None, oracle.C_F32
    if p.beta != 0.0:
        c0 = p.C0.numpy() if p.out_dtype == "f32" else inputs.bits(p.C0)
        ct = {"f32": oracle.C_F32, "bf16": oracle.C_BF16, "f16": oracle.C_F16}[p.out_dtype]
    return oracle.gemm_block_scaled(p.M, p.N, p.K, p.alpha, p.A.numpy(), p.lda, p.SFA.numpy(), p.ld_sfa, p.B.numpy(),
                                    p.ldb, p.SFB.numpy(), p.ld_sfb, p.beta, c0, p.ldc, _ET[p.a_elem], _ET[p.b_elem],
                                    oracle.SF_E8M0 if p.fmt == "mxfp8" else oracle.SF_UE4M3, p.block, rows=rows,
                                    cols=cols, c_type=ct)


def run(p, h, bias=None, act=G.ACT_NONE, scale=1.0, guard=2):
    Cd = torch.full((p.M + guard, p.ldc + guard), SENTINEL, dtype=_T[p.out_dtype], device="cuda")
    if p.beta != 0.0:
        Cd[:p.M, :p.N] = p.C0[:, :p.N].cuda()
    else:
        Cd[:p.M, :p.N] = float("nan")
    A, B, SA, SB = p.A.cuda(), p.B.cuda(), p.SFA.cuda(), p.SFB.cuda()
    bd = bias.cuda() if bias is not None else None
    st = h.run_block_scaled_raw(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, SA.data_ptr(), p.ld_sfa, B.data_ptr(),
                                p.ldb, SB.data_ptr(), p.ld_sfb, p.beta, Cd.data_ptr(), p.ldc + guard, code_of(p), None,
                                bias=bd.data_ptr() if bd is not None else 0, act=act, out_scale=scale)
    assert st == G.OK, G.STATUS.get(st)
    assert h.status()[0] == G.OK
    full = Cd.cpu().double()
    out = full[:p.M, :p.N].numpy().copy()
    full[:p.M, :p.N] = SENTINEL
    assert bool((full == SENTINEL).all()), "C written outside M x N"
    return out


PAIRS = [("mxfp8", "e4m3", "e4m3"), ("mxfp8", "e4m3", "e5m2"), ("mxfp8", "e5m2", "e4m3"), ("mxfp8", "e5m2", "e5m2"),
         ("nvfp4", "e2m1", "e2m1")]


@pytest.mark.parametrize("fmt,a,b", PAIRS)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_formats_ragged(h, fmt, a, b, out):
    """M, N not multiples of the tile, K with a partial last block, a blend with C."""
    p = inputs.make_block_scaled_problem("bs_%s_%s_%s" % (fmt, a, b), 300, 264, 200, fmt, out, a, b, alpha=0.5,
                                         beta=-0.25, seed=len(a) + 3 * len(b))
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, out == "f32", p.name)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_padded_pitches_and_fp16_out(h, fmt):
    K = 192
    per16 = 32 if fmt == "nvfp4" else 16
    # (alpha keeps C inside fp16's range: the blocks' values reach 2^6 x 448)
    p = inputs.make_block_scaled_problem("bs_pad", 130, 136, K, fmt, "f16", lda=K + 2 * per16, ldb=K + per16,
                                         ld_sf=48, ldc=150, seed=7, alpha=2.0 ** -6)
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, False, p.name)


def test_fp4_odd_k_ignores_the_last_high_nibble(h):
    """K = 37: the last byte of each row holds one value; its high four bits are
    set to -6 here and must not count."""
    p = inputs.make_block_scaled_problem("bs_odd", 70, 90, 37, "nvfp4", seed=8, lda=64, ldb=64)
    for X in (p.A, p.B):
        X[:, 18] |= 0xF0
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, True, p.name)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_swapped_skinny(h, fmt):
    """M = 40: the GEMM runs as C^T with the weights on the MMA's rows."""
    p = inputs.make_block_scaled_problem("bs_skinny", 40, 1000, 512, fmt, "bf16", seed=9)
    assert G.plan_block_scaled(p.M, p.N, p.K, code_of(p), handle=h).swap_ab == 1
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, False, p.name)


def test_fused_epilogue(h):
    p = inputs.make_block_scaled_problem("bs_epi", 256, 384, 256, "mxfp8", "bf16", seed=10)
    bias = torch.from_numpy(np.random.default_rng(10).normal(0, 2, p.N).astype(np.float32))
    R, Mag = reference(p)
    R, Mag = oracle.epilogue(R, Mag, bias=bias.numpy(), act=G.ACT_GELU, scale=0.5)
    assert_close(run(p, h, bias=bias, act=G.ACT_GELU, scale=0.5), R, Mag, False, p.name)


def test_k_zero(h):
    p = inputs.make_block_scaled_problem("bs_k0", 30, 40, 0, "nvfp4", seed=11, beta=2.0)
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, True, p.name)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4"])
def test_square_4096_sampled(h, fmt):
    p = inputs.make_block_scaled_problem("bs_4096", 4096, 4096, 4096, fmt, "f32", seed=12, alpha=1.0 / 64)
    out = run(p, h)
    rows, cols = sample_indices(p.M, p.N, 1500, seed=12)
    R, Mag = reference(p, rows, cols)
    assert_close(out[rows, cols], R, Mag, True, p.name)


def test_bad_arguments(h):
    A = torch.zeros(64, 64, dtype=torch.uint8, device="cuda")
    C = torch.zeros(64, 64, device="cuda")
    # a block-scaled type through the plain entry point, and a plain type here
    assert h.run_raw(0, 1, 64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 64, 0.0, C.data_ptr(), 64, G.NVFP4_F32,
                     None) == G.ERR_INVALID_ARG
    assert h.run_block_scaled_raw(64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 16, A.data_ptr(), 64,
                                  A.data_ptr(), 16, 0.0, C.data_ptr(), 64, G.E4M3_F32, None) == G.ERR_INVALID_ARG
    # missing scales, scale rows too short, odd FP4 pitch
    assert h.run_block_scaled_raw(64, 64, 64, 1.0, A.data_ptr(), 64, 0, 16, A.data_ptr(), 64, A.data_ptr(), 16, 0.0,
                                  C.data_ptr(), 64, G.mxfp8_dtype(), None) == G.ERR_INVALID_ARG
    assert h.run_block_scaled_raw(64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 1, A.data_ptr(), 64, A.data_ptr(),
                                  16, 0.0, C.data_ptr(), 64, G.mxfp8_dtype(), None) == G.ERR_INVALID_ARG
    assert h.run_block_scaled_raw(64, 64, 64, 1.0, A.data_ptr(), 65, A.data_ptr(), 16, A.data_ptr(), 64,
                                  A.data_ptr(), 16, 0.0, C.data_ptr(), 64, G.NVFP4_F32, None) == G.ERR_INVALID_ARG


# ---------------------------------------------------- codes converted in the GEMM --

def _dq_plan(p, h):
    return G.plan_block_scaled(p.M, p.N, p.K, code_of(p), lda=p.lda, ldb=p.ldb, ld_sfa=p.ld_sfa, ld_sfb=p.ld_sfb,
                               ldc=p.ldc + 2, handle=h)


@pytest.mark.parametrize("fmt,a,b", PAIRS)
@pytest.mark.parametrize("M,N,K", [(40, 1000, 200), (1, 257, 64), (64, 520, 1000)])
def test_dq_kernel_formats(h, fmt, a, b, M, N, K):
    """M <= 64: the weights B stay in their codes and the GEMM's converter warps
    write their 16-bit values into the ring (A alone goes through the pass).
    Ragged N, K with partial k-slices and blocks; the same result as the pass
    for both operands (GEMM_OPT_DEQUANT_IN_KERNEL = 1), within the tolerance."""
    p = inputs.make_block_scaled_problem("bs_dq_%s_%s_%s" % (fmt, a, b), M, N, K, fmt, "f32", a, b, alpha=0.5,
                                         seed=M + N + K + len(a) + 3 * len(b))
    plan = _dq_plan(p, h)
    assert plan.swap_ab == 1 and plan.launches == 2 and plan.repack_b == 0, plan.as_dict()
    R, Mag = reference(p)
    out = run(p, h)
    assert_close(out, R, Mag, True, p.name)
    h.set_option(G.OPT_DEQUANT_IN_KERNEL, 1)
    try:
        assert _dq_plan(p, h).launches == 3
        assert_close(run(p, h), R, Mag, True, p.name + " (pass)")
    finally:
        h.set_option(G.OPT_DEQUANT_IN_KERNEL, 0)


def test_dq_kernel_fp4_odd_k(h):
    """K = 37 on the converting path: the last code byte of each weight row holds
    one value, its high four bits set to -6 here; the product past K is zero
    because A's 16-bit copy is zero there."""
    p = inputs.make_block_scaled_problem("bs_dq_odd", 40, 300, 37, "nvfp4", seed=18, lda=64, ldb=64)
    for X in (p.A, p.B):
        X[:, 18] |= 0xF0
    assert _dq_plan(p, h).launches == 2
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, True, p.name)


@pytest.mark.parametrize("fmt,out", [("nvfp4", "bf16"), ("mxfp8", "f32")])
def test_dq_kernel_lm_head_full(h, fmt, out):
    """The LM head, 64 x 32000 x 4096, every element against the oracle
    (stream-K over all SMs, transposed bulk stores of C)."""
    p = inputs.make_block_scaled_problem("bs_dq_lmhead", 64, 32000, 4096, fmt, out, seed=19, alpha=1.0 / 64)
    plan = _dq_plan(p, h)
    assert plan.launches == 2 and plan.schedule == G.SCHED_STREAM_K
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, out == "f32", p.name)


def test_dq_kernel_timeout_then_clean(h):
    """A dropped load on the converting path: the converter warps' and the MMA's
    bounded waits run out, the status reports a timeout, and the next call on
    the same handle is correct."""
    p = inputs.make_block_scaled_problem("bs_dq_drop", 40, 1000, 512, "nvfp4", "f32", seed=20)
    assert _dq_plan(p, h).launches == 2
    Cd = torch.zeros(p.M, p.ldc, device="cuda")
    A, B, SA, SB = p.A.cuda(), p.B.cuda(), p.SFA.cuda(), p.SFB.cuda()
    h.set_option(G.OPT_WAIT_LIMIT_NS, 50_000_000)
    h.set_option(G.OPT_TEST_DROP_LOAD, 3)
    try:
        st = h.run_block_scaled_raw(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, SA.data_ptr(), p.ld_sfa, B.data_ptr(),
                                    p.ldb, SB.data_ptr(), p.ld_sfb, 0.0, Cd.data_ptr(), p.ldc, code_of(p), None)
        assert st == G.OK
        st, word = h.status()
        assert st == G.ERR_TIMEOUT and word & 0xFF == 6
    finally:
        h.set_option(G.OPT_TEST_DROP_LOAD, 0)
        h.set_option(G.OPT_WAIT_LIMIT_NS, 2_000_000_000)
    R, Mag = reference(p)
    assert_close(run(p, h), R, Mag, True, p.name)


@pytest.mark.parametrize("elem", ["e4m3", "e5m2", "e2m1"])
def test_dq_kernel_every_code_exact(h, elem):
    """Every code of the weights' format through the converting path, one
    product per output: token i is 1.0 at k = i and 0 elsewhere, so C[i, j] is
    weight (j, i) times its row's scale, exactly (the E8M0 scales keep every
    product inside bf16's normal range; E2M1 x E4M3 products are exact in
    fp16).  Rows 0 .. 255 hold every finite code at every position of a
    k-slice; rows 256 .. 511 hold the special codes too (E4M3 NaN, E5M2
    infinities and NaNs), whose columns come out NaN as in the oracle."""
    fmt = "nvfp4" if elem == "e2m1" else "mxfp8"
    M, N, K = 64, 512, 64
    p = inputs.make_block_scaled_problem("bs_dq_codes_" + elem, M, N, K, fmt, "f32", elem, elem, seed=21)
    A, B, SA, SB = p.A.numpy(), p.B.numpy(), p.SFA.numpy(), p.SFB.numpy()
    nblk = K // p.block
    A[:, :] = 0
    j = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    if fmt == "nvfp4":
        A[np.arange(M), np.arange(M) // 2] = np.where(np.arange(M) % 2 == 0, 0x02, 0x20)  # E2M1 1.0
        SA[:, :nblk] = 0x38                                                                # UE4M3 1.0
        nib = (j + k) % 16
        B[:, :K // 2] = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
        SB[:, :nblk] = np.array([0x38, 0x01, 0x7E, 0x08, 0x40, 0x20, 0x30, 0x50], np.uint8)[np.arange(N) % 8, None]
    else:
        A[np.arange(M), np.arange(M)] = 0x38 if elem == "e4m3" else 0x3C                # 1.0
        SA[:, :nblk] = 127
        codes = (j * 64 + k) % 256
        special = (codes & 0x7F) == 0x7F if elem == "e4m3" else (codes & 0x7C) == 0x7C
        codes = np.where(special & (j < N // 2), 0, codes)
        B[:, :K] = codes.astype(np.uint8)
        top = 240 if elem == "e4m3" else 225   # largest code x 2^(top - 127) finite in bf16
        SB[:, :nblk] = np.array([17, 60, 100, 127, 150, 200, top, 127], np.uint8)[np.arange(N) % 8, None]
    assert _dq_plan(p, h).launches == 2
    R, _ = reference(p)
    out = run(p, h)
    np.testing.assert_array_equal(out.astype(np.float32), R.astype(np.float32))
    assert np.isfinite(out[:, :N // 2]).all()
    if fmt == "mxfp8":
        assert np.isnan(out[:, N // 2:]).any()
