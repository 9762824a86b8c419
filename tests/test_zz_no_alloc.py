"""gemm_run_noalloc, the entry point for callers that must not allocate device
memory (their memory is reserved up front by their own allocator, or they
cannot afford the device synchronisation cudaMalloc can imply).  It keeps its
scratch in fixed device arrays of the library instead of a handle's workspace.

Checked through the C ABI against the handle-based gemm_run on two calls in a
row, so that whatever the first call leaves in the shared arrays (partial sums,
counters) cannot leak into the second.  This file is collected last."""
import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import oracle_full

pytestmark = pytest.mark.gpu


def _problem(seed):
    # M = 64 against N = 3000 tiles: the plan shares every tile's k-blocks out
    # (stream-K), so the run stores partial sums in the scratch array; ldb = 4100
    # keeps B's rows 16-byte aligned, ldc = 3003 forces the scalar-store epilogue.
    return inputs.make_problem("noalloc", 64, 3000, 4096, 0, 1, "bf16", "f32", ("normal", 0, 1),
                               ("normal", 0, 0.02), alpha=1.25, beta=0.5, seed=seed, ldb=4104, ldc=3003)


def test_noalloc_matches_gemm_run_twice():
    lib = G.lib()
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
            assert lib.gemm_run_noalloc(p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda,
                                        B.data_ptr(), p.ldb, p.beta, C_new.data_ptr(), p.ldc, G.BF16_F32,
                                        None) == G.OK
            torch.cuda.synchronize()
            assert h.status()[0] == G.OK
            ref = C_ref[:, :p.N].double().cpu().numpy()
            new = C_new[:, :p.N].double().cpu().numpy()
            _, Mag = oracle_full(p)
            assert np.all(np.abs(new - ref) <= 1e-3 * Mag + 1e-5)
            # the padding columns of C (NaN in the generated C0) are untouched
            assert bool(torch.isnan(C_new[:, p.N:]).all())
    finally:
        h.close()


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
