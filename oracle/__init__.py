"""CPU oracle for C = alpha * op(A) * op(B) + beta * C0 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library never calls it and the
two share no code: the oracle is a plain fp64 triple loop in ``gemm_oracle.c``
(the definition of "CUDA GEMM 矩阵乘法优化指南", section 2.1, checked in double
precision as the page at m.lqnn.cn/news/285670 does in its section 1.2).

Inputs are the raw bit patterns of the matrices, in the row-major storage
convention described in ``gemm_oracle.c``: numpy ``uint16`` for bf16 / fp16,
``uint8`` for the 8-bit E4M3 / E5M2 formats and for packed FP4 E2M1 (two
elements a byte, the even one in the low four bits), ``float32`` for fp32.
Every function here is pinned by ``tests/test_oracle.py``.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_gemm.so")

IN_BF16, IN_F16, IN_E4M3, IN_E5M2, IN_F32, IN_E2M1 = 0, 1, 2, 3, 4, 5
SF_E8M0, SF_UE4M3 = 0, 1
C_F32, C_BF16, C_F16 = 0, 1, 2

_lib = None


def build(force=False):
    """Compile the oracle with gcc (plain C, fp-contraction off so that the
    same source gives the same roundings on x86-64 and aarch64)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp,
           "-lpthread", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # ORACLE_LIB points the pins at another build of the oracle source; the
    # mutation test uses it to show that a planted mistake fails the pins.
    path = os.environ.get("ORACLE_LIB") or build()
    lib = ctypes.CDLL(path)
    i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
    lib.oracle_gemm_ab.restype = i32
    lib.oracle_gemm_ab.argtypes = [i32, i32, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i32, i64,
                                   i32, i32, vp, vp, i64, i32]
    lib.oracle_gemm_at_ab.restype = i32
    lib.oracle_gemm_at_ab.argtypes = [i32, i32, i64, i64, i64, dbl, vp, i64, vp, i64, dbl, vp, i32,
                                      i64, i32, i32, i64, vp, vp, vp, vp, i32]
    lib.oracle_bf16_value.restype = dbl
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_value.restype = dbl
    lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_gemm_batched.restype = i32
    lib.oracle_gemm_batched.argtypes = [i32, i32, i64, i64, i64, dbl, vp, i64, i64, vp, i64, i64, dbl, vp, i32,
                                        i64, i64, i32, i32, i64, vp, vp, i64, i32]
    lib.oracle_gemm_grouped.restype = i32
    lib.oracle_gemm_grouped.argtypes = [i32, i64, vp, i64, i64, dbl, vp, i64, vp, i64, i64, dbl, vp, i32, i64, i32,
                                        i32, vp, vp, i64, i32]
    lib.oracle_epilogue.restype = i32
    lib.oracle_epilogue.argtypes = [i64, i64, vp, vp, i64, vp, i32, dbl]
    lib.oracle_e4m3_value.restype = dbl
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e5m2_value.restype = dbl
    lib.oracle_e5m2_value.argtypes = [ctypes.c_uint8]
    for name in ("oracle_e2m1_value", "oracle_e8m0_value", "oracle_ue4m3_value"):
        getattr(lib, name).restype = dbl
        getattr(lib, name).argtypes = [ctypes.c_uint8]
    lib.oracle_gemm_block_scaled.restype = i32
    lib.oracle_gemm_block_scaled.argtypes = [i64, i64, i64, dbl, vp, i64, vp, i64, vp, i64, vp, i64, dbl, vp, i32,
                                             i64, i32, i32, i32, i64, i64, vp, vp, vp, vp, i64, i32]
    _lib = lib
    return lib


def bf16_value(bits):
    """Value of one bfloat16 bit pattern, decoded from the format definition."""
    return _load().oracle_bf16_value(int(bits) & 0xFFFF)


def f16_value(bits):
    """Value of one IEEE binary16 bit pattern, decoded from the format definition."""
    return _load().oracle_f16_value(int(bits) & 0xFFFF)


def e4m3_value(bits):
    """Value of one FP8 E4M3 bit pattern, decoded from the format definition."""
    return _load().oracle_e4m3_value(int(bits) & 0xFF)


def e5m2_value(bits):
    """Value of one FP8 E5M2 bit pattern, decoded from the format definition."""
    return _load().oracle_e5m2_value(int(bits) & 0xFF)


def e2m1_value(bits):
    """Value of one FP4 E2M1 code (low four bits), decoded from the format definition."""
    return _load().oracle_e2m1_value(int(bits) & 0xF)


def e8m0_value(bits):
    """Value of one E8M0 scale-factor code: 2^(bits - 127), NaN for 255."""
    return _load().oracle_e8m0_value(int(bits) & 0xFF)


def ue4m3_value(bits):
    """Value of one unsigned E4M3 scale-factor code (sign bit ignored)."""
    return _load().oracle_ue4m3_value(int(bits) & 0xFF)


def _codes(X, in_type):
    """The stored matrix as an array of codes of the type's width."""
    want = np.uint8 if in_type in (IN_E4M3, IN_E5M2, IN_E2M1) else np.float32 if in_type == IN_F32 else np.uint16
    X = np.ascontiguousarray(X)
    if X.dtype != want:
        raise TypeError("input of type %d must be %s codes" % (in_type, want.__name__))
    return X


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c0_array(C0, c_type):
    if C0 is None:
        return None
    want = np.float32 if c_type == C_F32 else np.uint16
    C0 = np.ascontiguousarray(C0)
    if C0.dtype != want:
        raise TypeError("C0 must be %s for c_type %d" % (want.__name__, c_type))
    return C0


def gemm(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, in_type, c_type=C_F32,
         nthreads=0, b_type=None):
    """Full oracle.  Returns (R, Mag): fp64 M x N arrays of r_ij and m_ij.

    A, B: code arrays holding the stored matrices (row-major, leading
    dimensions lda / ldb); A has type in_type, B has b_type (default: the
    same).  C0: float32 (c_type C_F32) or uint16 bits, M x N with leading
    dimension ldc; ignored when beta == 0.
    """
    lib = _load()
    b_type = in_type if b_type is None else b_type
    A = _codes(A, in_type)
    B = _codes(B, b_type)
    C0 = _c0_array(C0, c_type) if beta != 0.0 else None
    R = np.zeros((M, N), dtype=np.float64)
    Mag = np.zeros((M, N), dtype=np.float64)
    rc = lib.oracle_gemm_ab(int(transA), int(transB), M, N, K, float(alpha), _ptr(A), lda, _ptr(B),
                            ldb, float(beta), _ptr(C0), int(c_type), ldc, int(in_type), int(b_type),
                            _ptr(R), _ptr(Mag), N, int(nthreads))
    if rc < 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return R, Mag


def gemm_batched(transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C0, ldc, strideC,
                 in_type, batch, c_type=C_F32, nthreads=0, b_type=None):
    """Strided batched oracle.  Returns (R, Mag): fp64 arrays of shape (batch, M, N).
    A, B, C0: flat code / value arrays holding every batch at the given element
    strides (0 = the same matrix for every batch)."""
    lib = _load()
    b_type = in_type if b_type is None else b_type
    A = _codes(A, in_type).reshape(-1)
    B = _codes(B, b_type).reshape(-1)
    C0 = _c0_array(C0, c_type).reshape(-1) if beta != 0.0 else None
    R = np.zeros((batch, M, N), dtype=np.float64)
    Mag = np.zeros((batch, M, N), dtype=np.float64)
    rc = lib.oracle_gemm_batched(int(transA), int(transB), M, N, K, float(alpha), _ptr(A), lda, strideA,
                                 _ptr(B), ldb, strideB, float(beta), _ptr(C0), int(c_type), ldc, strideC,
                                 int(in_type), int(b_type), batch, _ptr(R), _ptr(Mag), N, int(nthreads))
    if rc < 0:
        raise ValueError("oracle_gemm_batched rejected its arguments")
    return R, Mag


def gemm_grouped(transB, m_sizes, N, K, alpha, A, lda, B, ldb, strideB, beta, C0, ldc, in_type, c_type=C_F32,
                 nthreads=0, b_type=None):
    """Grouped oracle.  Returns (R, Mag): fp64 arrays of shape (sum(m_sizes), N)."""
    lib = _load()
    b_type = in_type if b_type is None else b_type
    sizes = np.ascontiguousarray(m_sizes, dtype=np.int64)
    A = _codes(A, in_type).reshape(-1)
    B = _codes(B, b_type).reshape(-1)
    C0 = _c0_array(C0, c_type).reshape(-1) if beta != 0.0 else None
    rows = int(sizes.sum())
    R = np.zeros((rows, N), dtype=np.float64)
    Mag = np.zeros((rows, N), dtype=np.float64)
    rc = lib.oracle_gemm_grouped(int(transB), sizes.size, _ptr(sizes), N, K, float(alpha), _ptr(A), lda, _ptr(B),
                                 ldb, strideB, float(beta), _ptr(C0), int(c_type), ldc, int(in_type), int(b_type),
                                 _ptr(R), _ptr(Mag), N, int(nthreads))
    if rc < 0:
        raise ValueError("oracle_gemm_grouped rejected its arguments")
    return R, Mag


def gemm_at(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, in_type, rows, cols,
            c_type=C_F32, nthreads=0, b_type=None):
    """Sampled oracle: r and m at the listed (rows[e], cols[e]) entries."""
    lib = _load()
    b_type = in_type if b_type is None else b_type
    A = _codes(A, in_type)
    B = _codes(B, b_type)
    C0 = _c0_array(C0, c_type) if beta != 0.0 else None
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in length")
    r = np.zeros(rows.shape, dtype=np.float64)
    m = np.zeros(rows.shape, dtype=np.float64)
    rc = lib.oracle_gemm_at_ab(int(transA), int(transB), M, N, K, float(alpha), _ptr(A), lda, _ptr(B),
                               ldb, float(beta), _ptr(C0), int(c_type), ldc, int(in_type), int(b_type),
                               rows.size, _ptr(rows), _ptr(cols), _ptr(r), _ptr(m), int(nthreads))
    if rc < 0:
        raise ValueError("oracle_gemm_at rejected its arguments")
    return r, m


def gemm_block_scaled(M, N, K, alpha, A, lda, SFA, ld_sfa, B, ldb, SFB, ld_sfb, beta, C0, ldc, a_type, b_type,
                      sf_type, block, rows=None, cols=None, c_type=C_F32, nthreads=0):
    """Block-scaled oracle (MXFP8: E4M3 / E5M2 with an E8M0 scale per 32 values
    of k; NVFP4: packed E2M1 with an unsigned E4M3 scale per 16).  A is stored
    M x K, B N x K (K contiguous, lda / ldb in elements); SFA / SFB are uint8
    scale codes, one per block of k, rows of ld_sfa / ld_sfb codes.  Returns
    (R, Mag): M x N arrays, or arrays of the sampled entries when rows / cols
    are given."""
    lib = _load()
    A = _codes(A, a_type)
    B = _codes(B, b_type)
    SFA = np.ascontiguousarray(SFA, dtype=np.uint8)
    SFB = np.ascontiguousarray(SFB, dtype=np.uint8)
    C0 = _c0_array(C0, c_type) if beta != 0.0 else None
    if rows is None:
        R = np.zeros((M, N), dtype=np.float64)
        Mag = np.zeros((M, N), dtype=np.float64)
        count, rp, cp = 0, None, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        if rows.shape != cols.shape:
            raise ValueError("rows and cols differ in length")
        R = np.zeros(rows.shape, dtype=np.float64)
        Mag = np.zeros(rows.shape, dtype=np.float64)
        count, rp, cp = rows.size, _ptr(rows), _ptr(cols)
    rc = lib.oracle_gemm_block_scaled(M, N, K, float(alpha), _ptr(A), lda, _ptr(SFA), ld_sfa, _ptr(B), ldb,
                                      _ptr(SFB), ld_sfb, float(beta), _ptr(C0), int(c_type), ldc, int(a_type),
                                      int(b_type), int(sf_type), int(block), count, rp, cp, _ptr(R), _ptr(Mag), N,
                                      int(nthreads))
    if rc < 0:
        raise ValueError("oracle_gemm_block_scaled rejected its arguments")
    return R, Mag


ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2
E4M3_MAX = 448.0


def epilogue(R, Mag, bias=None, act=ACT_NONE, scale=1.0):
    """The fused epilogue applied to a full oracle result (see oracle_epilogue in
    gemm_oracle.c): out = scale * act(r + bias_j), with the magnitude carried
    through the same steps.  Returns new arrays."""
    R = np.array(R, dtype=np.float64, order="C", copy=True)
    Mag = np.array(Mag, dtype=np.float64, order="C", copy=True)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if b is not None and b.shape != (R.shape[1],):
        raise ValueError("bias must hold one value per column")
    rc = _load().oracle_epilogue(R.shape[0], R.shape[1], _ptr(R), _ptr(Mag), R.shape[1], _ptr(b), int(act),
                                 float(scale))
    if rc != 0:
        raise ValueError("oracle_epilogue rejected its arguments")
    return R, Mag


def within_tolerance(out, r, m, out_is_f32, e4m3=False, tf32=False, tf32x3_k=None):
    """Elementwise comparison rule for a GPU result ``out`` against (r, m).

    fp32 output:       |out - r| <= 1e-3 * m + 1e-5
    bf16 / fp16 output: |out - r| <= 8e-3 * |r| + 1e-3 * m + 1e-5
    E4M3 output (e4m3=True): r saturates at +-448 first (the format's largest
    value), then |out - r| <= 2^-4 * |r| + 1e-3 * m + 2^-10 (half a unit in the
    last of E4M3's 3 fraction bits, and half its smallest subnormal).
    Products of TF32-rounded inputs (tf32=True, one pass; each input keeps
    10 fraction bits, so a product is off by up to ~2^-10 relative):
    |out - r| <= 2^-8 * m + 1e-5.
    fp32 products from three TF32 products (tf32x3_k = K): each x = hi + lo +
    e with hi, lo TF32 values and |e| <= 2^-22 |x|; dropping lo_a lo_b and
    the two e terms costs at most 2^-20 |a b| per product; the fp32 sum of 3K
    terms (each partial sum at most m, each addition off by at most 2^-23 of
    it, truncation included) adds at most 3K * 2^-23 * m:
    |out - r| <= (3K * 2^-23 + 2^-20) * m + 2^-126.
    A NaN or Inf in ``out`` where r is finite fails.
    Returns a boolean array (True = within tolerance).
    """
    out = np.asarray(out, dtype=np.float64)
    if tf32x3_k is not None:
        ok = np.abs(out - r) <= (3 * int(tf32x3_k) * 2.0 ** -23 + 2.0 ** -20) * m + 2.0 ** -126
        ok &= np.isfinite(out) | ~np.isfinite(r)
        return ok
    if tf32:
        ok = np.abs(out - r) <= 2.0 ** -8 * m + 1e-5
        ok &= np.isfinite(out) | ~np.isfinite(r)
        return ok
    if e4m3:
        r = np.clip(r, -E4M3_MAX, E4M3_MAX)
        bound = 2.0 ** -4 * np.abs(r) + 1e-3 * m + 2.0 ** -10
        ok = np.abs(out - r) <= bound
        ok &= np.isfinite(out) | ~np.isfinite(r)
        return ok
    err = np.abs(out - r)
    bound = 1e-3 * m + 1e-5
    if not out_is_f32:
        bound = bound + 8e-3 * np.abs(r)
    ok = err <= bound
    ok &= np.isfinite(out) | ~np.isfinite(r)
    return ok
