"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: the value
definitions of the 16-bit and 8-bit formats and a library decoder over every
bit pattern, closed forms (identity, permutation, rank-1 products), exact integer
arithmetic, a brute-force loop written independently in pure Python, the
degenerate sizes, and invariants of the tolerance magnitude.  Together they
catch a dropped term, a wrong sign, a wrong index or stride, and a transposed
operand anywhere in the oracle.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _stored(transX, rows, cols):
    """Stored shape of op(X) = rows x cols."""
    return (cols, rows) if transX else (rows, cols)


def _op(stored, trans):
    return np.ascontiguousarray(stored.T) if trans else stored


# ---------------------------------------------------------------------------
# Decoding the 16-bit formats
# ---------------------------------------------------------------------------

def test_bf16_decode_known_values():
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC040) == -3.0
    assert oracle.bf16_value(0x4049) == 3.140625
    assert oracle.bf16_value(0x0001) == 2.0 ** -133           # smallest subnormal
    assert oracle.bf16_value(0x0080) == 2.0 ** -126           # smallest normal
    assert oracle.bf16_value(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert oracle.bf16_value(0x8000) == 0.0 and math.copysign(1, oracle.bf16_value(0x8000)) < 0
    assert oracle.bf16_value(0x7F80) == math.inf
    assert math.isnan(oracle.bf16_value(0x7FC0))


def test_f16_decode_known_values():
    assert oracle.f16_value(0x3C00) == 1.0
    assert oracle.f16_value(0xC200) == -3.0
    assert oracle.f16_value(0x3555) == 0.333251953125
    assert oracle.f16_value(0x0001) == 2.0 ** -24             # smallest subnormal
    assert oracle.f16_value(0x0400) == 2.0 ** -14             # smallest normal
    assert oracle.f16_value(0x7BFF) == 65504.0
    assert oracle.f16_value(0xFC00) == -math.inf
    assert math.isnan(oracle.f16_value(0x7E00))


def test_bf16_decode_every_pattern_matches_library():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    mine = np.array([oracle.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_f16_decode_every_pattern_matches_library():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    mine = np.array([oracle.f16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


# ---------------------------------------------------------------------------
# Decoding the 8-bit formats (E4M3 / E5M2: OCP 8-bit float layouts)
# ---------------------------------------------------------------------------

def test_fp8_decode_known_values():
    """Values fixed by the format definitions."""
    e4, e5 = oracle.e4m3_value, oracle.e5m2_value
    assert e4(0x38) == 1.0 and e4(0xB8) == -1.0
    assert e4(0x7E) == 448.0                      # largest finite E4M3
    assert e4(0x08) == 2.0 ** -6                  # smallest normal
    assert e4(0x01) == 2.0 ** -9                  # smallest subnormal
    assert e4(0x07) == 7.0 / 8.0 * 2.0 ** -6      # largest subnormal
    assert e4(0x78) == 256.0 and e4(0x3C) == 1.5
    assert math.isnan(e4(0x7F)) and math.isnan(e4(0xFF))   # the only NaNs; no infinities
    assert math.copysign(1.0, e4(0x80)) == -1.0 and e4(0x80) == 0.0
    assert e5(0x3C) == 1.0 and e5(0xBC) == -1.0
    assert e5(0x7B) == 57344.0                    # largest finite E5M2
    assert e5(0x04) == 2.0 ** -14 and e5(0x01) == 2.0 ** -16
    assert e5(0x7C) == math.inf and e5(0xFC) == -math.inf
    assert all(math.isnan(e5(b)) for b in (0x7D, 0x7E, 0x7F, 0xFD))
    assert e5(0x3E) == 1.5


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_decode_every_pattern_matches_library(fmt):
    codes = np.arange(256, dtype=np.uint8)
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    ref = torch.from_numpy(codes.copy()).view(dt).to(torch.float64).numpy()
    dec = oracle.e4m3_value if fmt == "e4m3" else oracle.e5m2_value
    mine = np.array([dec(int(b)) for b in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def _decoded(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_fp8_product_matches_library_matmul(transA, transB, fa, fb):
    """8-bit inputs, each operand with its own format, against numpy's matmul
    of the library-decoded values (fp64, exact products, order-only rounding)."""
    M, N, K = 13, 11, 150
    p = inputs.make_problem("f8", M, N, K, transA, transB, fa, "f32", ("normal", 0, 2), ("normal", 0, 2),
                            alpha=0.75, beta=-0.5, seed=41, b_dtype=fb)
    codes = {"e4m3": oracle.IN_E4M3, "e5m2": oracle.IN_E5M2}
    R, Mag = oracle.gemm(transA, transB, M, N, K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B), p.ldb,
                         p.beta, p.C0.numpy(), p.ldc, codes[fa], b_type=codes[fb])
    a = _op(_decoded(p.A[:, :(M if transA else K)]), transA)
    b = _op(_decoded(p.B[:, :(K if transB else N)]), transB)
    ref = p.alpha * (a @ b) + p.beta * p.C0[:, :N].double().numpy()
    assert np.allclose(R, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(Mag, abs(p.alpha) * (np.abs(a) @ np.abs(b)) + abs(p.beta) * np.abs(p.C0[:, :N].double().numpy()),
                       rtol=1e-12, atol=1e-12)


def test_fp8_small_integers_exact():
    """Integers in {-8..8} are exact in both formats; the integer product is exact."""
    M, N, K = 20, 24, 300
    p = inputs.make_problem("f8i", M, N, K, 0, 1, "e4m3", "f32", ("ints", -8, 8), ("ints", -8, 8), seed=3,
                            b_dtype="e5m2")
    R, _ = oracle.gemm(0, 1, M, N, K, 1.0, inputs.bits(p.A), K, inputs.bits(p.B), K, 0.0, None, N,
                       oracle.IN_E4M3, b_type=oracle.IN_E5M2)
    a = p.A.to(torch.float32).numpy().astype(np.int64)
    b = p.B.to(torch.float32).numpy().astype(np.int64)
    assert np.array_equal(R, (a @ b.T).astype(np.float64))


def test_fp8_code_width_is_checked():
    with pytest.raises(TypeError):
        oracle.gemm(0, 0, 2, 2, 2, 1.0, np.zeros((2, 2), np.uint16), 2, np.zeros((2, 2), np.uint8), 2, 0.0,
                    None, 2, oracle.IN_E4M3)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def _as_dtype_bits(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16 if dtype == "bf16" else torch.float16)
    return inputs.bits(t), t.to(torch.float64).numpy()


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_identity_left(transA, transB, dtype):
    """A = I (M = K): r = alpha * B + beta * C0, exactly."""
    M = K = 23
    N = 17
    in_type = oracle.IN_BF16 if dtype == "bf16" else oracle.IN_F16
    a_bits, _ = _as_dtype_bits(np.eye(M), dtype)
    b = inputs.draw(_stored(transB, K, N), ("uniform", -2, 2), 5, dtype)
    b_bits, b_val = inputs.bits(b), b.to(torch.float64).numpy()
    c0 = inputs.draw((M, N), ("normal", 0, 1), 6, "f32").numpy()
    alpha, beta = 1.25, -0.75
    R, Mag = oracle.gemm(transA, transB, M, N, K, alpha, a_bits, M, b_bits, b_bits.shape[1], beta,
                         c0, N, in_type)
    opb = _op(b_val, transB)
    assert np.array_equal(R, alpha * opb + beta * c0.astype(np.float64))
    assert np.array_equal(Mag, abs(alpha) * np.abs(opb) + abs(beta) * np.abs(c0.astype(np.float64)))


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
def test_identity_right(transA, transB):
    """B = I (K = N): r = alpha * op(A), exactly."""
    M, K = 19, 32
    a = inputs.draw(_stored(transA, M, K), ("uniform", -1, 1), 7, "bf16")
    a_bits, a_val = inputs.bits(a), a.to(torch.float64).numpy()
    b_bits, _ = _as_dtype_bits(np.eye(K), "bf16")
    R, _ = oracle.gemm(transA, transB, M, K, K, -2.0, a_bits, a_bits.shape[1], b_bits, K, 0.0, None,
                       K, oracle.IN_BF16)
    assert np.array_equal(R, -2.0 * _op(a_val, transA))


@pytest.mark.parametrize("transA", [0, 1])
def test_permutation(transA):
    """A = P: the rows of r are the rows of B taken in the order of P."""
    M = K = 31
    N = 9
    perm = np.random.Generator(np.random.PCG64(11)).permutation(M)
    P = np.zeros((M, K))
    P[np.arange(M), perm] = 1.0
    a_bits, _ = _as_dtype_bits(P.T if transA else P, "bf16")
    b = inputs.draw((K, N), ("uniform", -1, 1), 12, "bf16")
    b_bits, b_val = inputs.bits(b), b.to(torch.float64).numpy()
    R, _ = oracle.gemm(transA, 0, M, N, K, 1.0, a_bits, M, b_bits, N, 0.0, None, N, oracle.IN_BF16)
    assert np.array_equal(R, b_val[perm, :])


@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
def test_rank_one_closed_form(transA, transB):
    """a(i, k) = u_i and b(k, j) = v_j: r_ij = alpha * K * u_i * v_j + beta * c0_ij, exactly."""
    M, N, K = 12, 10, 40
    g = np.random.Generator(np.random.PCG64(3))
    u = 2.0 ** g.integers(-3, 4, size=M) * g.choice([-1, 1], size=M)
    v = 2.0 ** g.integers(-3, 4, size=N) * g.choice([-1, 1], size=N)
    opa = np.repeat(u[:, None], K, axis=1)
    opb = np.repeat(v[None, :], K, axis=0)
    a_bits, _ = _as_dtype_bits(opa.T if transA else opa, "f16")
    b_bits, _ = _as_dtype_bits(opb.T if transB else opb, "f16")
    c0 = g.integers(-8, 9, size=(M, N)).astype(np.float32)
    alpha, beta = 0.5, 2.0
    R, Mag = oracle.gemm(transA, transB, M, N, K, alpha, a_bits, a_bits.shape[1], b_bits,
                         b_bits.shape[1], beta, c0, N, oracle.IN_F16)
    want = alpha * K * np.outer(u, v) + beta * c0
    assert np.array_equal(R, want)
    assert np.array_equal(Mag, abs(alpha) * K * np.abs(np.outer(u, v)) + abs(beta) * np.abs(c0))


# ---------------------------------------------------------------------------
# Exact integer arithmetic
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("transA", [0, 1])
@pytest.mark.parametrize("transB", [0, 1])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_small_integers_exact(transA, transB, dtype):
    """Entries in {-4..4}: every partial sum is an integer far below 2^53, so the
    oracle must equal the exact integer product, whatever the order of the sum.
    Non-square shapes and padded leading dimensions catch a transposed operand
    or a wrong stride."""
    M, N, K = 13, 7, 29
    pa, pb = 3, 5   # padding columns (filled with NaN bits, which must never be read)
    in_type = oracle.IN_BF16 if dtype == "bf16" else oracle.IN_F16
    sa, sb = _stored(transA, M, K), _stored(transB, K, N)
    p = inputs.make_problem("ints", M, N, K, transA, transB, dtype, "f32", ("ints", -4, 4),
                            ("ints", -4, 4), alpha=1.5, beta=0.5, dist_c=("ints", -9, 9), seed=21,
                            lda=sa[1] + pa, ldb=sb[1] + pb, ldc=N + 2)
    A_int = p.A[:, :sa[1]].to(torch.float64).numpy().astype(np.int64)
    B_int = p.B[:, :sb[1]].to(torch.float64).numpy().astype(np.int64)
    C_int = p.C0[:, :N].numpy().astype(np.int64)
    exact = _op(A_int, transA) @ _op(B_int, transB)
    R, Mag = oracle.gemm(transA, transB, M, N, K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B),
                         p.ldb, p.beta, p.C0.numpy(), p.ldc, in_type)
    assert np.array_equal(R, 1.5 * exact + 0.5 * C_int)
    absprod = np.abs(_op(A_int, transA)) @ np.abs(_op(B_int, transB))
    assert np.array_equal(Mag, 1.5 * absprod + 0.5 * np.abs(C_int))


def test_small_integers_exact_at_full_depth():
    """K = 4096 with entries in {-4..4}: |partial sums| <= 65536, still exact."""
    M, N, K = 5, 6, 4096
    p = inputs.make_problem("ints_deep", M, N, K, 0, 1, "bf16", "f32", ("ints", -4, 4), ("ints", -4, 4),
                            seed=40)
    A_int = p.A.to(torch.float64).numpy().astype(np.int64)
    B_int = p.B.to(torch.float64).numpy().astype(np.int64)
    R, _ = oracle.gemm(0, 1, M, N, K, 1.0, inputs.bits(p.A), K, inputs.bits(p.B), K, 0.0, None, N,
                       oracle.IN_BF16)
    assert np.array_equal(R, (A_int @ B_int.T).astype(np.float64))


# ---------------------------------------------------------------------------
# Brute force: an independent loop in pure Python, other loop order, other decoder
# ---------------------------------------------------------------------------

def _py_value(h, dtype):
    h = int(h)
    if dtype == "f16":
        return struct.unpack("<e", struct.pack("<H", h))[0]
    return struct.unpack("<f", struct.pack("<I", h << 16))[0]


def _brute(transA, transB, M, N, K, alpha, Abits, lda, Bbits, ldb, beta, C0, ldc, dtype):
    Af, Bf = Abits.reshape(-1), Bbits.reshape(-1)
    out = [[0.0] * N for _ in range(M)]
    for j in range(N):
        for i in range(M):
            acc = 0.0
            for k in range(K):
                ha = Af[k * lda + i] if transA else Af[i * lda + k]
                hb = Bf[j * ldb + k] if transB else Bf[k * ldb + j]
                acc += _py_value(ha, dtype) * _py_value(hb, dtype)
            v = alpha * acc
            if beta != 0.0:
                v += beta * float(C0.reshape(-1)[i * ldc + j])
            out[i][j] = v
    return np.array(out)


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (7, 2, 13), (11, 13, 1), (24, 24, 24), (1, 17, 23)])
@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_brute_force_agreement(shape, transA, transB, dtype):
    M, N, K = shape
    seed = 100 + M * 7 + N * 3 + K + 2 * transA + transB
    g = np.random.Generator(np.random.PCG64(seed))
    alpha = float(g.uniform(-2, 2))
    beta = float(g.choice([0.0, float(g.uniform(-2, 2))]))
    p = inputs.make_problem("brute", M, N, K, transA, transB, dtype, "f32", ("normal", 0, 1),
                            ("uniform", -3, 3), alpha=alpha, beta=beta, seed=seed,
                            lda=_stored(transA, M, K)[1] + 1, ldb=_stored(transB, K, N)[1] + 2,
                            ldc=N + 1)
    in_type = oracle.IN_BF16 if dtype == "bf16" else oracle.IN_F16
    c0 = p.C0.numpy() if p.C0 is not None else None
    R, Mag = oracle.gemm(transA, transB, M, N, K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B),
                         p.ldb, p.beta, c0, p.ldc, in_type)
    want = _brute(transA, transB, M, N, K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B), p.ldb,
                  p.beta, c0, p.ldc, dtype)
    assert np.all(np.abs(R - want) <= 1e-12 * Mag + 1e-300)


def test_bf16_output_c0_is_decoded():
    """beta != 0 with a bf16 C0: the oracle must read C0 as bf16 bits."""
    M, N, K = 4, 6, 8
    p = inputs.make_problem("c16", M, N, K, 0, 0, "bf16", "bf16", ("ints", -2, 2), ("ints", -2, 2),
                            alpha=1.0, beta=-2.0, dist_c=("ints", -5, 5), seed=9)
    R, _ = oracle.gemm(0, 0, M, N, K, 1.0, inputs.bits(p.A), K, inputs.bits(p.B), N, -2.0,
                       inputs.bits(p.C0), N, oracle.IN_BF16, c_type=oracle.C_BF16)
    exact = p.A.double().numpy() @ p.B.double().numpy() - 2.0 * p.C0.double().numpy()
    assert np.array_equal(R, exact)


# ---------------------------------------------------------------------------
# Degenerate sizes, invariants, the sampled mode
# ---------------------------------------------------------------------------

def test_k_zero_gives_beta_c0():
    M, N = 6, 5
    c0 = inputs.draw((M, N), ("normal", 0, 1), 1, "f32").numpy()
    a = np.zeros((M, 1), dtype=np.uint16)
    b = np.zeros((1, N), dtype=np.uint16)
    R, Mag = oracle.gemm(0, 0, M, N, 0, 3.0, a, 1, b, N, -0.5, c0, N, oracle.IN_BF16)
    assert np.array_equal(R, -0.5 * c0.astype(np.float64))
    assert np.array_equal(Mag, 0.5 * np.abs(c0.astype(np.float64)))


def test_beta_zero_ignores_nan_c0():
    M, N, K = 3, 4, 5
    p = inputs.make_problem("nanc", M, N, K, 0, 0, "bf16", "f32", ("ints", -2, 2), ("ints", -2, 2), seed=2)
    c0 = np.full((M, N), np.nan, dtype=np.float32)
    R, _ = oracle.gemm(0, 0, M, N, K, 1.0, inputs.bits(p.A), K, inputs.bits(p.B), N, 0.0, c0, N,
                       oracle.IN_BF16)
    assert np.all(np.isfinite(R))


def test_empty_sizes():
    R, Mag = oracle.gemm(0, 0, 0, 5, 3, 1.0, np.zeros((1, 3), np.uint16), 3, np.zeros((3, 5), np.uint16),
                         5, 0.0, None, 5, oracle.IN_BF16)
    assert R.shape == (0, 5)
    R, Mag = oracle.gemm(0, 0, 4, 0, 3, 1.0, np.zeros((4, 3), np.uint16), 3, np.zeros((3, 1), np.uint16),
                         1, 0.0, None, 1, oracle.IN_BF16)
    assert R.shape == (4, 0)


def test_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.gemm(0, 0, 4, 4, 8, 1.0, np.zeros((4, 8), np.uint16), 7, np.zeros((8, 4), np.uint16), 4,
                    0.0, None, 4, oracle.IN_BF16)   # lda < K


def test_magnitude_bounds_result():
    """|r| <= m always (triangle inequality), with equality when every term is >= 0."""
    p = inputs.make_problem("mag", 20, 30, 50, 1, 0, "f16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=-1.5, beta=0.25, seed=4)
    R, Mag = oracle.gemm(1, 0, 20, 30, 50, -1.5, inputs.bits(p.A), 20, inputs.bits(p.B), 30, 0.25,
                         p.C0.numpy(), 30, oracle.IN_F16)
    assert np.all(np.abs(R) <= Mag * (1 + 1e-15))
    q = inputs.make_problem("pos", 9, 8, 70, 0, 0, "bf16", "f32", ("uniform", 0, 1), ("uniform", 0, 1), seed=8)
    R, Mag = oracle.gemm(0, 0, 9, 8, 70, 2.0, inputs.bits(q.A), 70, inputs.bits(q.B), 8, 0.0, None, 8,
                         oracle.IN_BF16)
    assert np.array_equal(R, Mag)


def test_sampled_mode_equals_full_mode():
    p = inputs.make_problem("samp", 37, 41, 64, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.7, beta=1.1, seed=13)
    R, Mag = oracle.gemm(0, 1, 37, 41, 64, 0.7, inputs.bits(p.A), 64, inputs.bits(p.B), 64, 1.1,
                         p.C0.numpy(), 41, oracle.IN_BF16, nthreads=3)
    g = np.random.Generator(np.random.PCG64(0))
    rows = g.integers(0, 37, 200)
    cols = g.integers(0, 41, 200)
    r, m = oracle.gemm_at(0, 1, 37, 41, 64, 0.7, inputs.bits(p.A), 64, inputs.bits(p.B), 64, 1.1,
                          p.C0.numpy(), 41, oracle.IN_BF16, rows, cols, nthreads=5)
    assert np.array_equal(r, R[rows, cols]) and np.array_equal(m, Mag[rows, cols])


def test_thread_count_does_not_change_results():
    p = inputs.make_problem("thr", 50, 20, 33, 0, 0, "f16", "f32", ("normal", 0, 1), ("normal", 0, 1), seed=17)
    args = (0, 0, 50, 20, 33, 1.0, inputs.bits(p.A), 33, inputs.bits(p.B), 20, 0.0, None, 20, oracle.IN_F16)
    R1, _ = oracle.gemm(*args, nthreads=1)
    R7, _ = oracle.gemm(*args, nthreads=7)
    assert np.array_equal(R1, R7)


# ---------------------------------------------------------------------------
# fp32 inputs (the FP32 GEMM emulated with three TF32 products)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_fp32_inputs_match_library_matmul(transA, transB):
    M, N, K = 17, 23, 90
    p = inputs.make_problem("of32", M, N, K, transA, transB, "f32", "f32", ("normal", 0, 1), ("normal", 0, 1),
                            alpha=0.5, beta=2.0, seed=6)
    R, Mag = oracle.gemm(transA, transB, M, N, K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B), p.ldb, p.beta,
                         p.C0.numpy(), p.ldc, oracle.IN_F32)
    a = _op(p.A.double().numpy(), transA)
    b = _op(p.B.double().numpy(), transB)
    ref = p.alpha * (a @ b) + p.beta * p.C0.double().numpy()
    assert np.allclose(R, ref, rtol=1e-13, atol=1e-13)


def test_fp32_inputs_exact_integers_and_types():
    p = inputs.make_problem("of32i", 30, 40, 500, 0, 0, "f32", "f32", ("ints", -50, 50), ("ints", -50, 50), seed=7)
    R, _ = oracle.gemm(0, 0, 30, 40, 500, 1.0, inputs.bits(p.A), 500, inputs.bits(p.B), 40, 0.0, None, 40,
                       oracle.IN_F32)
    assert np.array_equal(R, (p.A.numpy().astype(np.int64) @ p.B.numpy().astype(np.int64)).astype(np.float64))
    with pytest.raises(TypeError):   # fp32 inputs are float32 arrays, not codes
        oracle.gemm(0, 0, 2, 2, 2, 1.0, np.zeros((2, 2), np.uint16), 2, np.zeros((2, 2), np.uint16), 2, 0.0, None,
                    2, oracle.IN_F32)


def test_fp32_batched_and_grouped_offsets():
    """fp32 operands advance by 4 bytes per element in batches and groups."""
    p = inputs.make_batched_problem("ob32", 3, 6, 5, 40, 0, 1, "f32", "f32", ("normal", 0, 1), ("normal", 0, 1), seed=8)
    R, _ = oracle.gemm_batched(0, 1, 6, 5, 40, 1.0, inputs.bits(p.A), 40, p.strideA, inputs.bits(p.B), 40, p.strideB,
                               0.0, None, 5, p.strideC, oracle.IN_F32, 3)
    a = p.A.double().numpy().reshape(3, 6, 40)
    b = p.B.double().numpy().reshape(3, 5, 40)
    assert np.allclose(R, np.einsum("bik,bjk->bij", a, b), rtol=1e-13, atol=1e-13)
    q = inputs.make_grouped_problem("og32", [2, 0, 4], 5, 40, 1, "f32", "f32", seed=9)
    Rg, _ = oracle.gemm_grouped(1, [2, 0, 4], 5, 40, 1.0, inputs.bits(q.A), 40, inputs.bits(q.B), 40, q.strideB,
                                0.0, None, 5, oracle.IN_F32)
    w = q.B.double().numpy().reshape(3, 5, 40)
    aa = q.A.double().numpy()
    assert np.allclose(Rg[:2], aa[:2] @ w[0].T, rtol=1e-13) and np.allclose(Rg[2:], aa[2:] @ w[2].T, rtol=1e-13)


def test_tf32_tolerance_rule():
    r = np.array([1.0, 1.0, 0.0])
    m = np.array([1.0, 1.0, 1.0])
    assert list(oracle.within_tolerance(np.array([1.0 + 3.8e-3, 1.0 + 4.1e-3, np.inf]), r, m, True, tf32=True)) \
        == [True, False, False]


def test_tf32x3_tolerance_rule():
    """K = 64: (192 * 2^-23 + 2^-20) = 2^-15.32...; a 1-ulp fp32 error passes, 2^-14 does not."""
    r = np.array([1.0, 1.0, 1.0, 0.0, 5.0])
    m = np.array([1.0, 1.0, 1.0, 0.0, 5.0])
    bound = 192 * 2.0 ** -23 + 2.0 ** -20
    out = np.array([1.0 + 2.0 ** -23, 1.0 + 0.99 * bound, 1.0 + 2.0 ** -14, 0.0, np.nan])
    assert list(oracle.within_tolerance(out, r, m, True, tf32x3_k=64)) == [True, True, False, True, False]
    # the error bound of the split itself: x - hi - lo for hi, lo rounded to TF32
    g = np.random.default_rng(1)
    x = g.standard_normal(10000).astype(np.float32).astype(np.float64)
    def tf32(v):   # round to nearest on 10 fraction bits (ties away from zero)
        e = np.floor(np.log2(np.abs(v)))
        q = 2.0 ** (e - 10)
        return np.sign(v) * np.floor(np.abs(v) / q + 0.5) * q
    hi = tf32(x)
    lo = np.where(x != hi, tf32(np.where(x != hi, x - hi, 1.0)), 0.0)
    assert np.all(np.abs(x - hi) <= 2.0 ** -11 * np.abs(x))
    assert np.all(np.abs(x - hi - lo) <= 2.0 ** -22 * np.abs(x))


# ---------------------------------------------------------------------------
# Strided batched GEMM
# ---------------------------------------------------------------------------

def _batch_mats(flat, count, stride, rows, ld, cols):
    """Decoded fp64 matrices of a flat batch (stride 0: the same one each time)."""
    x = flat.to(torch.float64).numpy()
    return [x[b * stride:b * stride + rows * ld].reshape(rows, ld)[:, :cols] for b in range(count)]


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("bcast", ["none", "A", "B"])
def test_batched_matches_per_batch_library_matmul(transA, transB, bcast):
    """Each batch against numpy's matmul of the library-decoded matrices, with
    padded leading dimensions, gaps between batches and broadcast operands."""
    batch, M, N, K = 4, 9, 11, 37
    a_rows = K if transA else M
    b_rows = N if transB else K
    lda = (M if transA else K) + 3
    ldb = (K if transB else N) + 2
    p = inputs.make_batched_problem("ob", batch, M, N, K, transA, transB, "bf16", "f32", ("normal", 0, 1),
                                    ("normal", 0, 1), alpha=-0.5, beta=1.25, seed=3, lda=lda, ldb=ldb,
                                    ldc=N + 1, strideA=0 if bcast == "A" else a_rows * lda + 5,
                                    strideB=0 if bcast == "B" else b_rows * ldb + 7, strideC=M * (N + 1) + 4)
    R, Mag = oracle.gemm_batched(transA, transB, M, N, K, p.alpha, inputs.bits(p.A), p.lda, p.strideA,
                                 inputs.bits(p.B), p.ldb, p.strideB, p.beta, p.C0.numpy(), p.ldc, p.strideC,
                                 oracle.IN_BF16, batch)
    As = _batch_mats(p.A, batch, p.strideA, a_rows, lda, M if transA else K)
    Bs = _batch_mats(p.B, batch, p.strideB, b_rows, ldb, K if transB else N)
    Cs = _batch_mats(p.C0, batch, p.strideC, M, N + 1, N)
    for b in range(batch):
        a = As[b].T if transA else As[b]
        bb = Bs[b].T if transB else Bs[b]
        ref = p.alpha * (a @ bb) + p.beta * Cs[b]
        assert np.allclose(R[b], ref, rtol=1e-12, atol=1e-12), b
        assert np.allclose(Mag[b], abs(p.alpha) * (np.abs(a) @ np.abs(bb)) + abs(p.beta) * np.abs(Cs[b]),
                           rtol=1e-12, atol=1e-12)


def test_batched_fp8_and_empty_batch():
    p = inputs.make_batched_problem("ob8", 3, 5, 6, 70, 0, 1, "e4m3", "f32", ("normal", 0, 1), ("normal", 0, 1),
                                    seed=9, b_dtype="e5m2")
    R, _ = oracle.gemm_batched(0, 1, 5, 6, 70, 1.0, inputs.bits(p.A), 70, p.strideA, inputs.bits(p.B), 70,
                               p.strideB, 0.0, None, 6, p.strideC, oracle.IN_E4M3, 3, b_type=oracle.IN_E5M2)
    for b in range(3):
        a = p.A[b * 350:(b + 1) * 350].to(torch.float64).numpy().reshape(5, 70)
        bb = p.B[b * 420:(b + 1) * 420].to(torch.float64).numpy().reshape(6, 70)
        assert np.allclose(R[b], a @ bb.T, rtol=1e-12, atol=1e-12)
    R0, M0 = oracle.gemm_batched(0, 0, 4, 4, 4, 1.0, np.zeros(16, np.uint16), 4, 16, np.zeros(16, np.uint16), 4,
                                 16, 0.0, None, 4, 16, oracle.IN_BF16, 0)
    assert R0.shape == (0, 4, 4)


# ---------------------------------------------------------------------------
# Grouped GEMM (stacked rows, one weight matrix per group)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("transB", [0, 1])
def test_grouped_matches_per_group_library_matmul(transB):
    sizes = [5, 0, 17, 1, 9]
    N, K = 13, 40
    p = inputs.make_grouped_problem("og", sizes, N, K, transB, "bf16", "f32", alpha=1.5, beta=-0.5, seed=4,
                                    lda=K + 3, ldb=(K if transB else N) + 2, ldc=N + 1)
    b_rows = N if transB else K
    ldb = (K if transB else N) + 2
    R, Mag = oracle.gemm_grouped(transB, sizes, N, K, p.alpha, inputs.bits(p.A), p.lda, inputs.bits(p.B), p.ldb,
                                 p.strideB, p.beta, p.C0.numpy(), p.ldc, oracle.IN_BF16)
    a = p.A.to(torch.float64).numpy()[:, :K]
    c0 = p.C0.to(torch.float64).numpy()[:, :N]
    Bs = _batch_mats(p.B, len(sizes), p.strideB, b_rows, ldb, K if transB else N)
    off = 0
    for g, m in enumerate(sizes):
        bg = Bs[g].T if transB else Bs[g]
        ref = p.alpha * (a[off:off + m] @ bg) + p.beta * c0[off:off + m]
        assert np.allclose(R[off:off + m], ref, rtol=1e-12, atol=1e-12), g
        off += m
    assert R.shape == (sum(sizes), N)


def test_grouped_single_group_is_the_plain_gemm():
    p = inputs.make_grouped_problem("og1", [37], 21, 50, 1, "f16", "f32", seed=5)
    R, Mag = oracle.gemm_grouped(1, [37], 21, 50, 1.0, inputs.bits(p.A), 50, inputs.bits(p.B), 50, p.strideB, 0.0,
                                 None, 21, oracle.IN_F16)
    R1, M1 = oracle.gemm(0, 1, 37, 21, 50, 1.0, inputs.bits(p.A), 50, inputs.bits(p.B), 50, 0.0, None, 21,
                         oracle.IN_F16)
    assert np.array_equal(R, R1) and np.array_equal(Mag, M1)


def test_moe_routing_sizes():
    s = inputs.moe_routing(8192, 64, seed=0)
    assert len(s) == 64 and sum(s) == 8192 and min(s) >= 0 and max(s) > 2 * 8192 // 64   # uneven


# ---------------------------------------------------------------------------
# Fused epilogue: bias, activation, output scale
# ---------------------------------------------------------------------------

def _grid(M=7, N=9, seed=1):
    g = np.random.default_rng(seed)
    return g.normal(0, 3, (M, N)), g.uniform(0.5, 2.0, (M, N)), g.normal(0, 1, N).astype(np.float32)


def test_epilogue_identity_and_bias():
    R, Mag, b = _grid()
    R0, M0 = oracle.epilogue(R, Mag)
    assert np.array_equal(R0, R) and np.array_equal(M0, Mag)
    R1, M1 = oracle.epilogue(R, Mag, bias=b)
    assert np.array_equal(R1, R + b.astype(np.float64)[None, :])       # one value per column
    assert np.array_equal(M1, Mag + np.abs(b.astype(np.float64))[None, :])


def test_epilogue_relu_and_scale():
    R, Mag, b = _grid(seed=2)
    out, m = oracle.epilogue(R, Mag, bias=b, act=oracle.ACT_RELU, scale=-0.5)
    z = R + b.astype(np.float64)[None, :]
    assert np.array_equal(out, -0.5 * np.where(z > 0, z, 0.0))
    assert np.allclose(m, 0.5 * (Mag + np.abs(b)[None, :]), rtol=0, atol=1e-15)


def test_epilogue_gelu_matches_library_and_closed_forms():
    x = np.linspace(-8, 8, 1601)
    R = x[None, :]
    out, m = oracle.epilogue(R, np.ones_like(R), act=oracle.ACT_GELU)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="none").numpy()
    assert np.allclose(out[0], ref, rtol=1e-14, atol=1e-15)
    neg, _ = oracle.epilogue(-R, np.ones_like(R), act=oracle.ACT_GELU)
    assert np.allclose(out[0] - neg[0], x, rtol=0, atol=1e-13)         # GELU(x) - GELU(-x) = x
    one, _ = oracle.epilogue(np.array([[1.0, 0.0]]), np.ones((1, 2)), act=oracle.ACT_GELU)
    assert abs(one[0, 0] - 0.8413447460685429) < 1e-15 and one[0, 1] == 0.0   # Phi(1); GELU(0) = 0
    assert np.all(m == 1.13)                                           # the largest slope bounds the error


def test_e4m3_output_tolerance():
    r = np.array([1.0, 1.0, 500.0, 0.0, 0.0, 3.0])
    m = np.zeros(6)
    out = np.array([1.0625, 1.07, 448.0, 2 ** -10, 2 ** -9, np.nan])
    assert list(oracle.within_tolerance(out, r, m, True, e4m3=True)) == [True, False, True, True, False, False]


def test_tolerance_rule():
    r = np.array([1.0, 1.0, 0.0, 1.0])
    m = np.array([1.0, 1.0, 10.0, 1.0])
    out = np.array([1.0 + 0.9e-3, 1.0 + 1.2e-3, 9e-3, np.nan])
    assert list(oracle.within_tolerance(out, r, m, True)) == [True, False, True, False]
    out16 = np.array([1.0 + 8.5e-3, 1.0 + 1e-2, 0.0, 1.0])
    assert list(oracle.within_tolerance(out16, r, m, False)) == [True, False, True, True]


# ---------------------------------------------------------------------------
# Block-scaled inputs (MXFP8, NVFP4)
# ---------------------------------------------------------------------------

def test_e2m1_codes():
    """FP4 E2M1: sign bit 3, exponent bits 2..1 (bias 1), fraction bit 0."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert v == (-1.0 if c & 8 else 1.0) * mags[c & 7]
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_scale_factor_codes():
    for c in range(255):
        assert oracle.e8m0_value(c) == math.ldexp(1.0, c - 127)
    assert math.isnan(oracle.e8m0_value(255))
    e4 = torch.arange(128, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        v = oracle.ue4m3_value(c)
        if (c & 0x7F) == 0x7F:
            assert math.isnan(v)
        else:
            assert v == e4[c & 0x7F]


def _decode_block_scaled(p, which):
    """Independent decode with torch / numpy: the fp64 matrix (rows x K) of values x scales."""
    X, SF, ld, elem, rows = (p.A, p.SFA, p.lda, p.a_elem, p.M) if which == "A" else \
        (p.B, p.SFB, p.ldb, p.b_elem, p.N)
    raw = X.numpy()
    if elem == "e2m1":
        codes = np.empty((rows, raw.shape[1] * 2), dtype=np.uint8)
        codes[:, 0::2] = raw & 0xF
        codes[:, 1::2] = raw >> 4
        table = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
        vals = np.where(codes & 8, -1.0, 1.0) * table[codes & 7]
    else:
        dt = torch.float8_e4m3fn if elem == "e4m3" else torch.float8_e5m2
        vals = torch.from_numpy(raw.copy()).view(dt).double().numpy()
    vals = vals[:, :p.K]
    sf = SF.numpy()[:, :-(-p.K // p.block)].astype(np.int64)
    if p.fmt == "mxfp8":
        scale = np.ldexp(1.0, sf - 127)
    else:
        scale = torch.from_numpy((sf & 0x7F).astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    return vals * np.repeat(scale, p.block, axis=1)[:, :p.K]


def _oracle_block_scaled(p, rows=None, cols=None):
    et = {"e4m3": oracle.IN_E4M3, "e5m2": oracle.IN_E5M2, "e2m1": oracle.IN_E2M1}
    sft = oracle.SF_E8M0 if p.fmt == "mxfp8" else oracle.SF_UE4M3
    c0 = None if p.beta == 0.0 else p.C0.numpy()
    return oracle.gemm_block_scaled(p.M, p.N, p.K, p.alpha, p.A.numpy(), p.lda, p.SFA.numpy(), p.ld_sfa,
                                    p.B.numpy(), p.ldb, p.SFB.numpy(), p.ld_sfb, p.beta, c0, p.ldc,
                                    et[p.a_elem], et[p.b_elem], sft, p.block, rows=rows, cols=cols)


@pytest.mark.parametrize("fmt,a,b,K", [("mxfp8", "e4m3", "e4m3", 96), ("mxfp8", "e4m3", "e5m2", 70),
                                       ("mxfp8", "e5m2", "e5m2", 33), ("nvfp4", "e2m1", "e2m1", 64),
                                       ("nvfp4", "e2m1", "e2m1", 37)])
def test_block_scaled_against_numpy(fmt, a, b, K):
    """Decoded with torch's FP8 and a table for FP4, scaled and multiplied by numpy."""
    p = inputs.make_block_scaled_problem("bs", 9, 11, K, fmt, a_elem=a, b_elem=b, alpha=0.75, beta=-0.5, seed=K)
    R, Mag = _oracle_block_scaled(p)
    Ad, Bd = _decode_block_scaled(p, "A"), _decode_block_scaled(p, "B")
    c0 = p.C0.numpy()[:, :p.N].astype(np.float64)
    assert np.allclose(R, 0.75 * Ad @ Bd.T - 0.5 * c0, rtol=1e-12, atol=1e-12)
    assert np.allclose(Mag, 0.75 * np.abs(Ad) @ np.abs(Bd).T + 0.5 * np.abs(c0), rtol=1e-12)
    rows, cols = np.array([0, 8, 3]), np.array([10, 0, 5])
    r, m = _oracle_block_scaled(p, rows, cols)
    assert np.array_equal(r, R[rows, cols]) and np.array_equal(m, Mag[rows, cols])


def test_block_scale_placement_closed_form():
    """K = 64, two MXFP8 blocks: A all 1.0 with block scales 2^1 and 2^-2 in row 0,
    B all 1.0 with scale 1: C = 32 * 2 + 32 * 0.25 = 72 exactly."""
    A = np.full((1, 64), 0x38, dtype=np.uint8)     # E4M3 1.0
    B = np.full((2, 64), 0x38, dtype=np.uint8)
    SFA = np.zeros((1, 16), dtype=np.uint8)
    SFA[0, :2] = [128, 125]
    SFB = np.full((2, 16), 127, dtype=np.uint8)
    SFB[1, 1] = 130                                 # column 1: second block times 8
    R, _ = oracle.gemm_block_scaled(1, 2, 64, 1.0, A, 64, SFA, 16, B, 64, SFB, 16, 0.0, None, 2,
                                    oracle.IN_E4M3, oracle.IN_E4M3, oracle.SF_E8M0, 32)
    assert R.tolist() == [[72.0, 32 * 2 + 32 * 0.25 * 8]]


def test_fp4_nibble_order():
    """The even element of a pair is the low four bits: byte 0x21 is (0.5, 1.0)."""
    A = np.array([[0x21]], dtype=np.uint8)
    B = np.array([[0x42], [0x24]], dtype=np.uint8)  # (1.0, 2.0) and (2.0, 1.0)
    SF = np.full((2, 16), 0x38, dtype=np.uint8)     # UE4M3 1.0
    R, _ = oracle.gemm_block_scaled(1, 2, 2, 1.0, A, 2, SF[:1], 16, B, 2, SF, 16, 0.0, None, 2,
                                    oracle.IN_E2M1, oracle.IN_E2M1, oracle.SF_UE4M3, 16)
    assert R.tolist() == [[0.5 * 1.0 + 1.0 * 2.0, 0.5 * 2.0 + 1.0 * 1.0]]


def test_block_scaled_generator_reconstructs():
    """The quantised blocks stay close to the drawn values: MXFP8 E4M3 within
    2^-3 of the block maximum, NVFP4 within half its coarsest step, 1/3 of the
    maximum (plus the E4M3 rounding of the scale)."""
    for fmt, tol in (("mxfp8", 2.0 ** -3), ("nvfp4", 0.36)):
        p = inputs.make_block_scaled_problem("rq", 4, 4, 96, fmt, seed=3)
        x = inputs._block_values(4, 96, p.block, 3, 6).reshape(4, -1)[:, :96]
        d = _decode_block_scaled(p, "A")
        amax = np.repeat(np.abs(x.reshape(4, -1, p.block)).max(axis=2), p.block, axis=1)
        assert np.all(np.abs(d - x) <= tol * amax + 1e-30)
        assert np.all(p.SFA.numpy()[:, -(-96 // p.block):] == 0xFF)     # scale padding never read
