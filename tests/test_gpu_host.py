"""GPU parity of gemm_run_host (host buffers in and out, copies overlapped with
the GEMM in blocks of C) against the oracle: every layout, row chunks
(M >= 1024), row and column chunks (M, N >= 1024) and single-block calls,
ragged last chunks, the blend with
C, 16-bit and fp32 C, page-locked and pageable host memory, K == 0, a growing
sequence of calls that reuses and grows the handle's device copies, and the
order with other work on the same stream.  Host C's padding columns must stay
untouched."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import SENTINEL, assert_close, dtype_code, oracle_full

pytestmark = pytest.mark.gpu

_T = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


def run_host(p, h, pinned=True, pad=3):
    """Run p through gemm_run_host; returns (C as fp64 M x N, the whole host C)."""
    ldc = p.ldc + pad
    C = torch.full((p.M, ldc), SENTINEL, dtype=_T[p.out_dtype])
    if p.beta != 0.0:
        C[:, :p.N] = p.C0[:, :p.N]
    else:
        C[:, :p.N] = float("nan")
    A, B = p.A.contiguous(), p.B.contiguous()
    if pinned:
        A, B, C = A.pin_memory(), B.pin_memory(), C.pin_memory()
    s = torch.cuda.current_stream()
    st = G.lib().gemm_run_host(h.ptr, p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(),
                               p.ldb, p.beta, C.data_ptr(), ldc, dtype_code(p), s.cuda_stream)
    assert st == G.OK, G.STATUS.get(st)
    s.synchronize()
    assert h.status()[0] == G.OK
    full = C.double()
    out = full[:, :p.N].numpy().copy()
    full[:, :p.N] = SENTINEL
    assert bool((full == SENTINEL).all()), "host C written outside M x N"
    return out


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_layouts_chunked_and_blend(h, transA, transB, out):
    """M = 1100: three row chunks of 512 rows (the last 76)."""
    p = inputs.make_problem("host_%d%d" % (transA, transB), 1100, 300, 200, transA, transB, "bf16", out,
                            ("normal", 0, 1), ("normal", 0, 1), alpha=0.5, beta=-0.25, seed=transA + 2 * transB)
    R, Mag = oracle_full(p)
    assert_close(run_host(p, h), R, Mag, out == "f32", p.name)


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_blocks_of_c(h, transA, transB, beta):
    """M, N >= 1024: C in 3 x 3 blocks of 512 (the last 76) computed as A's row
    chunks and B's column chunks arrive, every layout, with and without the blend."""
    p = inputs.make_problem("host_2d_%d%d" % (transA, transB), 1100, 1100, 200, transA, transB, "bf16", "f32",
                            ("normal", 0, 1), ("normal", 0, 1), alpha=0.75, beta=beta, seed=30 + transA + 2 * transB)
    R, Mag = oracle_full(p)
    assert_close(run_host(p, h), R, Mag, True, p.name)


@pytest.mark.parametrize("pinned", [True, False])
def test_pageable_and_pinned(h, pinned):
    p = inputs.make_problem("host_mem", 2048, 520, 384, 0, 1, "f16", "f16", ("uniform", -1, 1), ("uniform", -1, 1),
                            seed=5)
    R, Mag = oracle_full(p)
    assert_close(run_host(p, h, pinned=pinned), R, Mag, False, p.name)


def test_small_single_chunk_and_k_zero(h):
    p = inputs.make_problem("host_small", 70, 90, 40, 0, 0, "bf16", "f32", seed=6)
    R, Mag = oracle_full(p)
    assert_close(run_host(p, h), R, Mag, True, p.name)
    q = inputs.make_problem("host_k0", 1500, 64, 0, 0, 0, "bf16", "f32", beta=2.0, seed=7)
    R, Mag = oracle_full(q)
    assert_close(run_host(q, h), R, Mag, True, q.name)


def test_growing_calls_reuse_the_device_copies(h):
    for i, (M, N, K) in enumerate([(256, 256, 128), (3000, 700, 512), (1024, 1024, 1024), (4096, 256, 64)]):
        p = inputs.make_problem("host_grow%d" % i, M, N, K, 0, 1, "bf16", "f32", ("normal", 0, 1),
                                ("normal", 0, 1), seed=10 + i)
        R, Mag = oracle_full(p, nthreads=0)
        assert_close(run_host(p, h), R, Mag, True, p.name)


def test_stream_order_with_other_work(h):
    """A device GEMM queued before the host call writes a buffer that a device
    GEMM queued after it reads; the host call in between must neither wait on
    the host nor break that order, and host C is complete after one stream sync."""
    p = inputs.make_problem("host_order", 1536, 256, 256, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            seed=20)
    A, B = p.A.pin_memory(), p.B.pin_memory()
    C = torch.empty(p.M, p.N).pin_memory()
    X = torch.randn(512, 512, device="cuda").to(torch.bfloat16)
    Y = torch.empty(512, 512, dtype=torch.bfloat16, device="cuda")
    Z = torch.empty(512, 512, device="cuda")
    s = torch.cuda.current_stream()
    assert h.run_raw(0, 0, 512, 512, 512, 1.0, X.data_ptr(), 512, X.data_ptr(), 512, 0.0, Y.data_ptr(), 512,
                     G.BF16_BF16, s.cuda_stream) == G.OK
    assert G.lib().gemm_run_host(h.ptr, 0, 1, p.M, p.N, p.K, 1.0, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, 0.0,
                                 C.data_ptr(), p.N, G.BF16_F32, s.cuda_stream) == G.OK
    assert h.run_raw(0, 0, 512, 512, 512, 1.0, Y.data_ptr(), 512, X.data_ptr(), 512, 0.0, Z.data_ptr(), 512,
                     G.BF16_F32, s.cuda_stream) == G.OK
    s.synchronize()
    R, Mag = oracle_full(p)
    assert_close(C.double().numpy(), R, Mag, True, p.name)
    y = Y.cpu()
    bits = lambda t: t.contiguous().view(torch.uint16).numpy()
    Ry, My = oracle.gemm(0, 0, 512, 512, 512, 1.0, bits(X.cpu()), 512, bits(X.cpu()), 512, 0.0, None, 512,
                         oracle.IN_BF16)
    assert_close(y.double().numpy(), Ry, My, False, "Y")
    Rz, Mz = oracle.gemm(0, 0, 512, 512, 512, 1.0, bits(y), 512, bits(X.cpu()), 512, 0.0, None, 512, oracle.IN_BF16)
    assert_close(Z.double().cpu().numpy(), Rz, Mz, True, "Z")


def test_tensor_binding(h):
    g = torch.Generator().manual_seed(30)
    A = torch.randn(1200, 256, generator=g).to(torch.bfloat16).pin_memory()
    B = torch.randn(256, 384, generator=g).to(torch.bfloat16).pin_memory()
    C = torch.empty(1200, 384).pin_memory()
    G.gemm_host(A, B, C, handle=h)
    torch.cuda.current_stream().synchronize()
    ref = (A.double() @ B.double()).numpy()
    mag = (A.double().abs() @ B.double().abs()).numpy()
    assert oracle.within_tolerance(C.double().numpy(), ref, mag, True).all()
    with pytest.raises(ValueError):
        G.gemm_host(A.cuda(), B, C, handle=h)


def test_block_scaled_types_are_refused(h):
    A = torch.zeros(64, 64, dtype=torch.uint8)
    C = torch.zeros(64, 64)
    assert G.lib().gemm_run_host(h.ptr, 0, 1, 64, 64, 64, 1.0, A.data_ptr(), 64, A.data_ptr(), 64, 0.0, C.data_ptr(),
                                 64, G.NVFP4_F32, None) == G.ERR_UNSUPPORTED
