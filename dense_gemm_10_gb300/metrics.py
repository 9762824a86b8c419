"""Work and traffic accounting for C = alpha * op(A) * op(B) + beta * C.

FLOPs follow "CUDA GEMM 矩阵乘法优化指南", section 2.1: each of the M x N outputs
takes K multiply-adds, 2 * M * N * K floating-point operations in all.
Algorithmic bytes follow section 2.2 of the same page (the ideal traffic, each
matrix moved once): A and B read once, C written once, and C read once more
when beta != 0 (the blend needs its old value).  The arithmetic intensity is
their ratio.
"""

ELEM_BYTES = {"bf16": 2, "f16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}


def flops(M, N, K):
    return 2 * int(M) * int(N) * int(K)


def algorithmic_bytes(M, N, K, in_dtype="bf16", out_dtype="f32", beta=0.0):
    e_in = ELEM_BYTES[in_dtype]
    e_out = ELEM_BYTES[out_dtype]
    n = (int(M) * int(K) + int(K) * int(N)) * e_in + int(M) * int(N) * e_out
    if beta != 0.0:
        n += int(M) * int(N) * e_out
    return n


def arithmetic_intensity(M, N, K, in_dtype="bf16", out_dtype="f32", beta=0.0):
    return flops(M, N, K) / algorithmic_bytes(M, N, K, in_dtype, out_dtype, beta)
