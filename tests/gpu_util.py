"""Helpers for the GPU parity tests: move a seeded problem to the device, run it
through the C ABI, and compare against the CPU oracle element by element."""
import numpy as np
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

_TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
_ORACLE_IN = {"bf16": oracle.IN_BF16, "f16": oracle.IN_F16, "e4m3": oracle.IN_E4M3, "e5m2": oracle.IN_E5M2,
              "f32": oracle.IN_F32}
SENTINEL = 1536.0   # exact in fp32, bf16 and fp16


def dtype_code(p):
    if p.in_dtype in inputs.FP8:
        return G.fp8_dtype(p.in_dtype, p.b_dtype, p.out_dtype)
    return {("bf16", "f32"): G.BF16_F32, ("bf16", "bf16"): G.BF16_BF16, ("f16", "f32"): G.F16_F32,
            ("f16", "f16"): G.F16_F16, ("bf16", "e4m3"): G.BF16_E4M3,
            ("f16", "e4m3"): G.F16_E4M3, ("f32", "f32"): G.F32_F32}[(p.in_dtype, p.out_dtype)]


def device_problem(p, guard_rows=0, guard_cols=0):
    """Device copies of A, B and a C buffer.  C has `guard_cols` extra columns
    (beyond ldc's own padding) and `guard_rows` extra rows holding a sentinel;
    when beta == 0 the C region starts as NaN, so reading it would show."""
    Ad = p.A.cuda()
    Bd = p.B.cuda()
    ldc = p.ldc + guard_cols
    Cd = torch.full((p.M + guard_rows, ldc), SENTINEL, dtype=_TORCH[p.out_dtype], device="cuda")
    if p.beta != 0.0:
        Cd[:p.M, :p.N] = p.C0[:, :p.N].cuda()
    else:
        Cd[:p.M, :p.N] = float("nan")
    return Ad, Bd, Cd, ldc


def launch(p, h, Ad, Bd, Cd, ldc, stream=None, code=None):
    st = h.run_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, Ad.data_ptr(), p.lda, Bd.data_ptr(), p.ldb,
                   p.beta, Cd.data_ptr(), ldc, dtype_code(p) if code is None else code, stream)
    if st != G.OK:
        raise G.GemmError(st, "gemm_run")


def run(p, h, guard_rows=0, guard_cols=0, code=None):
    """Run p on the GPU (dtype code `code`, default the problem's own); returns
    (C as fp64 numpy M x N, whole C buffer on the CPU)."""
    Ad, Bd, Cd, ldc = device_problem(p, guard_rows, guard_cols)
    launch(p, h, Ad, Bd, Cd, ldc, code=code)
    st, detail = h.status()
    assert st == G.OK, "kernel status %s (word 0x%x)" % (G.STATUS.get(st), detail)
    full = Cd.cpu()
    return full[:p.M, :p.N].to(torch.float64).numpy(), full


def _c0_for_oracle(p):
    if p.C0 is None:
        return None, oracle.C_F32
    if p.out_dtype == "f32":
        return p.C0.numpy(), oracle.C_F32
    return inputs.bits(p.C0), (oracle.C_BF16 if p.out_dtype == "bf16" else oracle.C_F16)


def oracle_full(p, nthreads=0):
    c0, ct = _c0_for_oracle(p)
    return oracle.gemm(p.transA, p.transB, p.M, p.N, p.K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B),
                       p.ldb, p.beta, c0, p.ldc, _ORACLE_IN[p.in_dtype], c_type=ct, nthreads=nthreads,
                       b_type=_ORACLE_IN[p.b_dtype])


def oracle_at(p, rows, cols, nthreads=0):
    c0, ct = _c0_for_oracle(p)
    return oracle.gemm_at(p.transA, p.transB, p.M, p.N, p.K, p.alpha, inputs.bits(p.A), p.lda,
                          inputs.bits(p.B), p.ldb, p.beta, c0, p.ldc, _ORACLE_IN[p.in_dtype], rows, cols,
                          c_type=ct, nthreads=nthreads, b_type=_ORACLE_IN[p.b_dtype])


def assert_close(out, r, m, out_is_f32, what=""):
    ok = oracle.within_tolerance(out, r, m, out_is_f32)
    if not ok.all():
        bad = np.argwhere(~ok.reshape(np.shape(out))) if np.ndim(out) > 1 else np.argwhere(~ok)
        first = tuple(bad[0])
        raise AssertionError("%s: %d of %d outside tolerance; first at %s: gpu %r oracle %r mag %r"
                             % (what, (~ok).sum(), ok.size, first, np.asarray(out)[first], r[first],
                                m[first]))


def sample_indices(M, N, count, seed, edge=64):
    """Random entries plus the corners and stretches of the first / last rows and columns."""
    g = np.random.Generator(np.random.PCG64(seed))
    rows = [g.integers(0, M, count)]
    cols = [g.integers(0, N, count)]
    for r in {0, M - 1}:
        rows.append(np.full(edge, r))
        cols.append(g.integers(0, N, edge))
    for c in {0, N - 1}:
        rows.append(g.integers(0, M, edge))
        cols.append(np.full(edge, c))
    rows.append(np.array([0, 0, M - 1, M - 1]))
    cols.append(np.array([0, N - 1, 0, N - 1]))
    # the last tile row / column (ragged tails live there)
    rows.append(g.integers(max(0, M - 128), M, edge))
    cols.append(g.integers(0, N, edge))
    rows.append(g.integers(0, M, edge))
    cols.append(g.integers(max(0, N - 256), N, edge))
    return np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64)
