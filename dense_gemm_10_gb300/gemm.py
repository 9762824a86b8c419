"""Thin ctypes binding of include/gemm_gb300.h (argument marshalling only).

Every step of the GEMM runs in the CUDA library; this module only turns
tensors into pointers, sizes and leading dimensions.  There is no fallback: if
the library has not been built, every call raises.
"""
import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgemm_gb300.so")

OP_N, OP_T = 0, 1
BF16_F32, BF16_BF16, F16_F32, F16_F16, BF16_E4M3, F16_E4M3 = 0, 1, 2, 3, 4, 5
F32_F32, TF32_F32 = 6, 7   # fp32 inputs: three TF32 products per product, or one
NVFP4_F32, NVFP4_BF16, NVFP4_F16 = 48, 49, 50   # block-scaled E2M1 (gemm_run_block_scaled)


def mxfp8_dtype(a="e4m3", b=None, c="f32"):
    """gemm_dtype_t of a block-scaled MXFP8 pair (E8M0 scales per 32 values of k)."""
    b = a if b is None else b
    return 32 + (a == "e5m2") + 2 * (b == "e5m2") + 4 * {"f32": 0, "bf16": 1, "f16": 2}[c]
_FP8_FORMATS = ("e4m3", "e5m2")
_C_TYPES = ("f32", "bf16", "f16", "e4m3")
ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2


def fp8_dtype(a="e4m3", b="e4m3", c="f32"):
    """gemm_dtype_t code for 8-bit inputs: 16 + (A E5M2) + 2 (B E5M2) + 4 (C type)."""
    return 16 + _FP8_FORMATS.index(a) + 2 * _FP8_FORMATS.index(b) + 4 * _C_TYPES.index(c)


E4M3_F32, E5M2_F32, E4M3_BF16, E5M2_BF16 = fp8_dtype(), fp8_dtype("e5m2", "e5m2"), fp8_dtype(c="bf16"), \
    fp8_dtype("e5m2", "e5m2", "bf16")
STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED", 3: "GEMM_ERR_NO_DEVICE",
          4: "GEMM_ERR_CUDA", 5: "GEMM_ERR_TENSORMAP", 6: "GEMM_ERR_TIMEOUT", 7: "GEMM_ERR_WORKSPACE"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NO_DEVICE, ERR_CUDA, ERR_TENSORMAP, ERR_TIMEOUT, ERR_WORKSPACE = range(8)
PATH_NOOP, PATH_SCALE_C, PATH_TC_1CTA, PATH_TC_2CTA = 0, 1, 2, 3
(OPT_WAIT_LIMIT_NS, OPT_FORCE_PATH, OPT_SPLIT_K, OPT_RASTER_GROUP, OPT_FORCE_BN, OPT_TEST_DROP_LOAD, OPT_MAX_GRID,
 OPT_STREAM_K, OPT_STAGES) = range(9)
OPT_EPILOGUE = 10
OPT_KDEPTH = 11
OPT_PDL = 12
OPT_PLAN_CACHE = 13
OPT_DEQUANT_IN_KERNEL = 15
OPT_EPILOGUE_WARPS = 16
BULK_NONE, BULK_ROWS, BULK_TRANSPOSED, BULK_STAGED, BULK_ROW_COPIES, BULK_ROW_CLASSES = 0, 1, 2, 3, 4, 5  # bulk_store
SCHED_TILES, SCHED_STREAM_K = 0, 1

# Exported functions and their (restype, argtypes).
_i32, _i64, _u64, _f32, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p


class Epilogue(ctypes.Structure):
    """gemm_epilogue_t: C = convert(out_scale * act(alpha A B + beta C + bias[j]))."""
    _fields_ = [("bias", _vp), ("activation", _i32), ("out_scale", _f32)]


class Plan(ctypes.Structure):
    _fields_ = [(n, _i32) for n in ("path", "swap_ab", "a_kmajor", "b_kmajor", "bm", "bn", "bk", "stages",
                                    "split_k", "raster_group", "repack_a", "repack_b", "vector_store",
                                    "grid", "launches", "schedule")] + \
               [(n, _i64) for n in ("tiles", "units", "workspace_bytes")] + \
               [(n, _i32) for n in ("tiles_i", "tiles_j", "num_kb", "dp_tiles", "sk_slots", "cluster", "kdepth",
                                    "bulk_store", "batch", "epilogue_warps")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


SIGNATURES = {
    "gemm_create": (_i32, [ctypes.POINTER(_vp), ctypes.c_int]),
    "gemm_run": (_i32, [_vp, _i32, _i32, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                        _i32, _vp]),
    "gemm_get_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "gemm_status_string": (ctypes.c_char_p, [_i32]),
    "gemm_last_cuda_error": (ctypes.c_int, [_vp]),
    "gemm_destroy": (_i32, [_vp]),
    "gemm_plan": (_i32, [_vp, ctypes.c_int, _i32, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _f32, _vp,
                         _i64, _i32, ctypes.POINTER(Plan)]),
    "gemm_set_option": (_i32, [_vp, _i32, _i64]),
    "gemm_launch_count": (_i32, [_vp, ctypes.POINTER(_u64)]),
    "gemm_run_noalloc": (_i32, [_i32, _i32, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _i32,
                                _vp]),
    "gemm_noalloc_get_status": (_i32, [_vp, ctypes.POINTER(_i32)]),
    "gemm_noalloc_set_option": (_i32, [_i32, _i64]),
    "gemm_run_ex": (_i32, [_vp, _i32, _i32, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                           _i32, ctypes.POINTER(Epilogue), _vp]),
    "gemm_run_strided_batched": (_i32, [_vp, _i32, _i32, _i64, _i64, _i64, _f32, _vp, _i64, _i64, _vp, _i64,
                                        _i64, _f32, _vp, _i64, _i64, _i64, _i32, ctypes.POINTER(Epilogue), _vp]),
    "gemm_plan_strided_batched": (_i32, [_vp, ctypes.c_int, _i32, _i32, _i64, _i64, _i64, _vp, _i64, _i64, _vp,
                                         _i64, _i64, _f32, _vp, _i64, _i64, _i64, _i32, ctypes.POINTER(Plan)]),
    "gemm_run_grouped": (_i32, [_vp, _i32, _i64, _vp, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _i64, _f32, _vp, _i64,
                                _i32, ctypes.POINTER(Epilogue), _vp]),
    "gemm_plan_grouped": (_i32, [_vp, ctypes.c_int, _i32, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _f32, _vp,
                                 _i64, _i32, ctypes.POINTER(Plan)]),
    "gemm_plan_cache_stats": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "gemm_tensor_map_cache_stats": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "gemm_probe_tma_tile": (_i32, [_vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "gemm_run_host": (_i32, [_vp, _i32, _i32, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _i32,
                             _vp]),
    "gemm_run_block_scaled": (_i32, [_vp, _i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32,
                                     _vp, _i64, _i32, ctypes.POINTER(Epilogue), _vp]),
    "gemm_plan_block_scaled": (_i32, [_vp, ctypes.c_int, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i64,
                                      _f32, _vp, _i64, _i32, ctypes.POINTER(Plan)]),
}

_lib = None
_lock = threading.Lock()


class GemmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s" % (what or "gemm", STATUS.get(status, str(status))))


def lib():
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("the GEMM CUDA library is not built (%s missing); run "
                                   "dense_gemm_10_gb300.build.build()" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
        return _lib


def _check(status, what):
    if status != OK:
        raise GemmError(status, what)


def plan(M, N, K, transA=0, transB=0, dtype=BF16_F32, lda=None, ldb=None, ldc=None, sm_count=152,
         A=0x1000, B=0x1000, C=0x1000, beta=0.0, handle=None):
    """Host-only planner query (no GPU needed); pointers matter only for alignment."""
    lda = lda if lda is not None else (M if transA else K)
    ldb = ldb if ldb is not None else (K if transB else N)
    ldc = ldc if ldc is not None else N
    p = Plan()
    h = handle.ptr if handle is not None else None
    st = lib().gemm_plan(h, sm_count, transA, transB, M, N, K, A, lda, B, ldb, beta, C, ldc, dtype,
                         ctypes.byref(p))
    _check(st, "gemm_plan")
    return p


class Handle:
    """A library handle bound to one CUDA device."""

    def __init__(self, device=0):
        h = _vp()
        _check(lib().gemm_create(ctypes.byref(h), int(device)), "gemm_create")
        self.ptr = h.value
        self.device = int(device)

    def close(self):
        if self.ptr:
            lib().gemm_destroy(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, opt, value):
        _check(lib().gemm_set_option(self.ptr, opt, int(value)), "gemm_set_option")

    def launch_count(self):
        n = _u64()
        _check(lib().gemm_launch_count(self.ptr, ctypes.byref(n)), "gemm_launch_count")
        return n.value

    def status(self, stream=None):
        """Synchronise `stream` and return (status code, raw status word)."""
        d = _i32()
        st = lib().gemm_get_status(self.ptr, stream, ctypes.byref(d))
        return st, d.value

    def run_raw(self, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, stream):
        """gemm_run on raw device pointers; returns the status code (no raise)."""
        return lib().gemm_run(self.ptr, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                              dtype, stream)

    def run_batched_raw(self, transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                        strideC, batch, dtype, stream, bias=0, act=ACT_NONE, out_scale=1.0):
        """gemm_run_strided_batched on raw device pointers; returns the status code."""
        epi = Epilogue(bias or None, int(act), float(out_scale))
        return lib().gemm_run_strided_batched(self.ptr, transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb,
                                              strideB, beta, C, ldc, strideC, batch, dtype, ctypes.byref(epi),
                                              stream)

    def run_grouped_raw(self, transB, m_sizes, N, K, alpha, A, lda, B, ldb, strideB, beta, C, ldc, dtype, stream,
                        bias=0, act=ACT_NONE, out_scale=1.0):
        """gemm_run_grouped on raw device pointers, group sizes from a Python list; returns the status."""
        sizes = (ctypes.c_int64 * max(1, len(m_sizes)))(*m_sizes)
        epi = Epilogue(bias or None, int(act), float(out_scale))
        return lib().gemm_run_grouped(self.ptr, transB, len(m_sizes), ctypes.cast(sizes, _vp), N, K, alpha, A, lda, B,
                                      ldb, strideB, beta, C, ldc, dtype, ctypes.byref(epi), stream)

    def plan_cache_stats(self):
        """(hits, misses) of the handle's plan cache."""
        hits, misses = ctypes.c_uint64(), ctypes.c_uint64()
        _check(lib().gemm_plan_cache_stats(self.ptr, ctypes.byref(hits), ctypes.byref(misses)),
               "gemm_plan_cache_stats")
        return hits.value, misses.value

    def tensor_map_cache_stats(self):
        """(hits, misses) of the handle's tensor-map cache."""
        hits, misses = ctypes.c_uint64(), ctypes.c_uint64()
        _check(lib().gemm_tensor_map_cache_stats(self.ptr, ctypes.byref(hits), ctypes.byref(misses)),
               "gemm_tensor_map_cache_stats")
        return hits.value, misses.value

    def run_block_scaled_raw(self, M, N, K, alpha, A, lda, SFA, ld_sfa, B, ldb, SFB, ld_sfb, beta, C, ldc, dtype,
                             stream, bias=0, act=ACT_NONE, out_scale=1.0):
        """gemm_run_block_scaled on raw device pointers; returns the status."""
        epi = Epilogue(bias or None, int(act), float(out_scale))
        return lib().gemm_run_block_scaled(self.ptr, M, N, K, alpha, A, lda, SFA, ld_sfa, B, ldb, SFB, ld_sfb, beta, C,
                                           ldc, dtype, ctypes.byref(epi), stream)

    def run_ex_raw(self, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dtype, stream,
                   bias=0, act=ACT_NONE, out_scale=1.0):
        """gemm_run_ex on raw device pointers (bias: device pointer or 0); returns the status code."""
        epi = Epilogue(bias or None, int(act), float(out_scale))
        return lib().gemm_run_ex(self.ptr, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                 dtype, ctypes.byref(epi), stream)


_default = {}


def default_handle(device=None):
    import torch
    dev = torch.cuda.current_device() if device is None else int(device)
    h = _default.get(dev)
    if h is None:
        h = _default[dev] = Handle(dev)
    return h


def plan_batched(M, N, K, batch, transA=0, transB=0, dtype=BF16_F32, lda=None, ldb=None, ldc=None,
                 strideA=None, strideB=None, strideC=None, sm_count=152, A=0x1000, B=0x1000, C=0x1000, beta=0.0,
                 handle=None):
    """Host-only planner query for a strided batched call (strides default to packed)."""
    lda = lda if lda is not None else (M if transA else K)
    ldb = ldb if ldb is not None else (K if transB else N)
    ldc = ldc if ldc is not None else N
    strideA = strideA if strideA is not None else (K if transA else M) * lda
    strideB = strideB if strideB is not None else (N if transB else K) * ldb
    strideC = strideC if strideC is not None else M * ldc
    p = Plan()
    h = handle.ptr if handle is not None else None
    st = lib().gemm_plan_strided_batched(h, sm_count, transA, transB, M, N, K, A, lda, strideA, B, ldb, strideB,
                                         beta, C, ldc, strideC, batch, dtype, ctypes.byref(p))
    _check(st, "gemm_plan_strided_batched")
    return p


def plan_block_scaled(M, N, K, dtype, lda=None, ldb=None, ld_sfa=None, ld_sfb=None, ldc=None, sm_count=152,
                      A=0x1000, B=0x1000, SFA=0x1000, SFB=0x1000, C=0x1000, beta=0.0, handle=None):
    """Host-only planner query for a block-scaled call (default pitches: K values,
    scale rows padded to 16 bytes)."""
    block = 16 if dtype >= NVFP4_F32 else 32
    nblk = -(-K // block)
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ld_sfa = -(-max(nblk, 1) // 16) * 16 if ld_sfa is None else ld_sfa
    ld_sfb = ld_sfa if ld_sfb is None else ld_sfb
    ldc = N if ldc is None else ldc
    p = Plan()
    h = handle.ptr if handle is not None else None
    st = lib().gemm_plan_block_scaled(h, sm_count, M, N, K, A, lda, SFA, ld_sfa, B, ldb, SFB, ld_sfb, beta, C, ldc,
                                      dtype, ctypes.byref(p))
    _check(st, "gemm_plan_block_scaled")
    return p


def plan_grouped(m_sizes, N, K, transB=1, dtype=BF16_F32, lda=None, ldb=None, strideB=None, ldc=None, sm_count=152,
                 A=0x1000, B=0x1000, C=0x1000, beta=0.0, handle=None):
    """Host-only planner query for a grouped call."""
    lda = K if lda is None else lda
    ldb = ldb if ldb is not None else (K if transB else N)
    ldc = N if ldc is None else ldc
    strideB = strideB if strideB is not None else (N if transB else K) * ldb
    sizes = (ctypes.c_int64 * max(1, len(m_sizes)))(*m_sizes)
    p = Plan()
    h = handle.ptr if handle is not None else None
    st = lib().gemm_plan_grouped(h, sm_count, transB, len(m_sizes), ctypes.cast(sizes, _vp), N, K, A, lda, B, ldb,
                                 strideB, beta, C, ldc, dtype, ctypes.byref(p))
    _check(st, "gemm_plan_grouped")
    return p


def dtype_code(in_dtype, out_dtype, b_dtype=None, tf32=False):
    """gemm_dtype_t code for torch dtypes of A (and B, default the same) and C.
    fp32 inputs: the fp32 GEMM from three TF32 products, or one TF32 product
    per product with tf32=True."""
    import torch
    b_dtype = in_dtype if b_dtype is None else b_dtype
    if in_dtype == torch.float32 and b_dtype == torch.float32 and out_dtype == torch.float32:
        return TF32_F32 if tf32 else F32_F32
    table = {(torch.bfloat16, torch.float32): BF16_F32, (torch.bfloat16, torch.bfloat16): BF16_BF16,
             (torch.float16, torch.float32): F16_F32, (torch.float16, torch.float16): F16_F16}
    if b_dtype == in_dtype and (in_dtype, out_dtype) in table:
        return table[(in_dtype, out_dtype)]
    if b_dtype == in_dtype and out_dtype == torch.float8_e4m3fn and in_dtype in (torch.bfloat16, torch.float16):
        return BF16_E4M3 if in_dtype == torch.bfloat16 else F16_E4M3
    f8 = {torch.float8_e4m3fn: "e4m3", torch.float8_e5m2: "e5m2"}
    cty = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16", torch.float8_e4m3fn: "e4m3"}
    if in_dtype in f8 and b_dtype in f8 and out_dtype in cty:
        return fp8_dtype(f8[in_dtype], f8[b_dtype], cty[out_dtype])
    raise TypeError("unsupported dtypes %s x %s -> %s" % (in_dtype, b_dtype, out_dtype))


def _ld(t, name):
    if t.dim() != 2 or (t.stride(1) != 1 and t.shape[1] > 1):
        raise ValueError("%s must be a 2-D row-major tensor (unit column stride)" % name)
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1], 1)


def gemm(A, B, C, transA=False, transB=False, alpha=1.0, beta=0.0, handle=None, stream=None, M=None,
         N=None, K=None, bias=None, act=ACT_NONE, out_scale=1.0, tf32=False):
    """C = convert(out_scale * act(alpha * op(A) * op(B) + beta * C + bias)) on
    CUDA tensors, enqueued on `stream` (default: torch's current stream).  A and
    B are stored row-major as (M, K) / (K, M) and (K, N) / (N, K) per transA /
    transB; C is (M, N); bias (optional) is a CUDA fp32 tensor of N values.
    fp32 A, B and C: the fp32 GEMM from three TF32 products, or one TF32
    product per product with tf32=True.  Sizes default to the logical extents
    of the tensors."""
    import torch
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % n)
    ta, tb = int(bool(transA)), int(bool(transB))
    M = M if M is not None else (A.shape[1] if ta else A.shape[0])
    K = K if K is not None else (A.shape[0] if ta else A.shape[1])
    N = N if N is not None else (B.shape[0] if tb else B.shape[1])
    code = dtype_code(A.dtype, C.dtype, B.dtype, tf32)
    h = handle if handle is not None else default_handle(C.device.index)
    if stream is None:
        stream = torch.cuda.current_stream(C.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if bias is not None and (not bias.is_cuda or bias.dtype != torch.float32 or bias.numel() < N
                             or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous CUDA float32 tensor of N values")
    st = h.run_ex_raw(ta, tb, M, N, K, float(alpha), A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"),
                      float(beta), C.data_ptr(), _ld(C, "C"), code, stream,
                      bias=bias.data_ptr() if bias is not None else 0, act=act, out_scale=out_scale)
    _check(st, "gemm_run")
    return C


def gemm_host(A, B, C, transA=False, transB=False, alpha=1.0, beta=0.0, handle=None, stream=None):
    """End-to-end call on CPU tensors (gemm_run_host): A, B (and C when beta
    != 0) go to the device, the GEMM runs, C comes back, overlapped in row
    chunks; use page-locked tensors (``pin_memory()``) for the overlap.  The
    call is asynchronous on `stream` (default: torch's current stream):
    synchronise it before reading C."""
    import torch
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if t.is_cuda:
            raise ValueError("%s must be a host tensor" % n)
    ta, tb = int(bool(transA)), int(bool(transB))
    M = A.shape[1] if ta else A.shape[0]
    K = A.shape[0] if ta else A.shape[1]
    N = B.shape[0] if tb else B.shape[1]
    code = dtype_code(A.dtype, C.dtype, B.dtype)
    h = handle if handle is not None else default_handle(0)
    if stream is None:
        stream = torch.cuda.current_stream(h.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    st = lib().gemm_run_host(h.ptr, ta, tb, M, N, K, alpha, A.data_ptr(), _ld(A, "A"), B.data_ptr(), _ld(B, "B"),
                             beta, C.data_ptr(), _ld(C, "C"), code, sptr)
    _check(st, "gemm_run_host")
    return C
