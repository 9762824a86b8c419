"""gemm_run_noalloc, the entry point for callers that must not allocate device
memory (their memory is reserved up front by their own allocator, or they
cannot afford the device synchronisation cudaMalloc can imply).  It keeps its
scratch in fixed device arrays of the library instead of a handle's workspace.

Every result is checked element by element against the CPU oracle, and against
the handle-based gemm_run within the same tolerance, on two calls in a row, so
that whatever the first call leaves in the shared arrays (partial sums,
counters) cannot leak into the second.  The path's own status word is read
back through gemm_noalloc_get_status.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import assert_close, oracle_full

pytestmark = pytest.mark.gpu


def _status():
    word = ctypes.c_int32(0)
    st = G.lib().gemm_noalloc_get_status(None, ctypes.byref(word))
    return st, word.value


def _run_noalloc(p, A, B, C):
    return G.lib().gemm_run_noalloc(p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda,
                                    B.data_ptr(), p.ldb, p.beta, C.data_ptr(), p.ldc, G.BF16_F32, None)


def _problem(seed):
    # M = 64 against N = 3000 tiles: the plan shares every tile's k-blocks out
    # (stream-K), so the run stores partial sums in the scratch array; ldb = 4104
    # keeps B's rows 16-byte aligned, ldc = 3003 forces the scalar-store epilogue.
    return inputs.make_problem("noalloc", 64, 3000, 4096, 0, 1, "bf16", "f32", ("normal", 0, 1),
                               ("normal", 0, 0.02), alpha=1.25, beta=0.5, seed=seed, ldb=4104, ldc=3003)


def test_noalloc_matches_oracle_and_gemm_run_twice():
    h = G.Handle(0)
    try:
        for seed in (7, 8):  # two calls in a row on the shared scratch
            p = _problem(seed)
            plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, lda=p.lda, ldb=p.ldb, ldc=p.ldc, beta=p.beta)
            assert plan.schedule == G.SCHED_STREAM_K and plan.workspace_bytes <= 16 << 20
            A, B = p.A.cuda(), p.B.cuda()
            C_ref = p.C0.cuda()
            C_new = p.C0.cuda()
            assert h.run_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(),
                             p.ldb, p.beta, C_ref.data_ptr(), p.ldc, G.BF16_F32, None) == G.OK
            assert _run_noalloc(p, A, B, C_new) == G.OK
            assert _status() == (G.OK, 0)
            assert h.status()[0] == G.OK
            R, Mag = oracle_full(p)
            new = C_new[:, :p.N].double().cpu().numpy()
            ref = C_ref[:, :p.N].double().cpu().numpy()
            assert_close(new, R, Mag, True, "gemm_run_noalloc call with seed %d" % seed)
            assert_close(new, ref, Mag, True, "gemm_run_noalloc against gemm_run, seed %d" % seed)
            # the padding columns of C (NaN in the generated C0) are untouched
            assert bool(torch.isnan(C_new[:, p.N:]).all())
    finally:
        h.close()


def test_noalloc_replans_without_stream_k():
    """A plan whose stream-K partial sums overflow the 16 MiB array (256 x 2048 x
    8192: 16 tiles shared by every SM pair, 19 MB of partials) is planned again
    on whole tiles, which need no partial sums, and runs."""
    p = inputs.make_problem("noalloc_replan", 256, 2048, 8192, 0, 1, "bf16", "f32", ("normal", 0, 1),
                            ("normal", 0, 0.02), seed=11)
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB)
    assert plan.schedule == G.SCHED_STREAM_K and plan.workspace_bytes > 16 << 20
    A, B = p.A.cuda(), p.B.cuda()
    C = torch.full((p.M, p.N), float("nan"), device="cuda")
    assert _run_noalloc(p, A, B, C) == G.OK
    assert _status() == (G.OK, 0)
    R, Mag = oracle_full(p)
    assert_close(C.double().cpu().numpy(), R, Mag, True, "re-planned gemm_run_noalloc")


def test_noalloc_timeout_is_reported_then_clean():
    """The test hook drops one load, so one barrier never completes: the kernel's
    bounded wait runs out, the path's status word records it, the status read
    reports GEMM_ERR_TIMEOUT and clears it, and the next call is correct."""
    L = G.lib()
    p = _problem(9)
    A, B = p.A.cuda(), p.B.cuda()
    try:
        assert L.gemm_noalloc_set_option(G.OPT_WAIT_LIMIT_NS, 50_000_000) == G.OK
        assert L.gemm_noalloc_set_option(G.OPT_TEST_DROP_LOAD, 3) == G.OK
        C = p.C0.cuda()
        assert _run_noalloc(p, A, B, C) == G.OK
        st, word = _status()
        assert st == G.ERR_TIMEOUT
        assert word & 0xFF == 6 and (word >> 8) & 0xF in (1, 2, 3)
        assert _status() == (G.OK, 0)   # the read cleared it
    finally:
        L.gemm_noalloc_set_option(G.OPT_TEST_DROP_LOAD, 0)
        L.gemm_noalloc_set_option(G.OPT_WAIT_LIMIT_NS, 2_000_000_000)
    C = p.C0.cuda()
    assert _run_noalloc(p, A, B, C) == G.OK
    assert _status() == (G.OK, 0)
    R, Mag = oracle_full(p)
    assert_close(C[:, :p.N].double().cpu().numpy(), R, Mag, True, "gemm_run_noalloc after a timeout")


def test_noalloc_rejects_what_does_not_fit():
    """A repack larger than the 16 MiB scratch array is refused, not allocated."""
    lib = G.lib()
    M = N = K = 4097          # odd leading dimensions: both operands need repacking (2 x 33.6 MB)
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    st = lib.gemm_run_noalloc(0, 0, M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(), N,
                              G.BF16_F32, None)
    assert st == G.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert _status() == (G.OK, 0)
