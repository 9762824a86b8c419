"""Seeded synthetic GEMM inputs, shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays them out; it holds none of the
GEMM's arithmetic.  Both the oracle side and the GPU side receive exactly the
tensors built here.

Recipe (one rule for every workload):
  * a workload has one integer seed s; A is drawn from seed s, B from s + 1,
    the initial C from s + 2 (numpy PCG64 streams);
  * samples are drawn in float32 (uniform or normal), then rounded once to the
    input type with round-to-nearest-even (torch ``.to(...)``: bfloat16,
    float16, or the 8-bit float8_e4m3fn / float8_e5m2; the distributions used
    stay inside the 8-bit formats' ranges);
  * a matrix is drawn directly in its stored shape (row-major storage, see
    ``Problem``), so the "op" flags change the layout, not the distribution;
    the one exception is a problem made with ``logical=True`` (the fp16
    blend workload): there op(A) (M x K) and op(B) (K x N) are drawn in their
    logical shapes and stored transposed where the layout says, so that every
    layout of the workload multiplies the same two matrices;
  * padding columns beyond a leading dimension hold a NaN bit pattern, so a
    kernel that reads past the logical width shows up as NaN in its output.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

_TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32,
             "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
_NAN_BITS = {"bf16": 0x7FC1, "f16": 0x7E01}
_NAN_BITS8 = {"e4m3": 0x7F, "e5m2": 0x7F}
FP8 = ("e4m3", "e5m2")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(int(seed)))


def draw(shape, dist, seed, dtype):
    """Draw a CPU tensor of ``dtype`` ("bf16", "f16", "f32", "e4m3", "e5m2") in ``shape``.

    dist: ("uniform", lo, hi) | ("normal", mean, std) | ("ints", lo, hi)
    (integers uniform in [lo, hi], inclusive) | ("zeros",).
    """
    g = _rng(seed)
    kind = dist[0]
    if kind == "uniform":
        x = g.random(size=shape, dtype=np.float32) * np.float32(dist[2] - dist[1]) + np.float32(dist[1])
    elif kind == "normal":
        x = g.standard_normal(size=shape, dtype=np.float32) * np.float32(dist[2]) + np.float32(dist[1])
    elif kind == "ints":
        x = g.integers(dist[1], dist[2] + 1, size=shape).astype(np.float32)
    elif kind == "zeros":
        x = np.zeros(shape, dtype=np.float32)
    else:
        raise ValueError("unknown distribution %r" % (dist,))
    return torch.from_numpy(np.ascontiguousarray(x)).to(_TORCH_DT[dtype])


def _pad_columns(t, ld, dtype):
    """Return a (rows, ld) tensor holding ``t`` in its first columns and NaN bits after."""
    rows, cols = t.shape
    if ld == cols:
        return t.contiguous()
    out = torch.empty((rows, ld), dtype=t.dtype)
    if dtype in _NAN_BITS:
        out.view(torch.int16).fill_(_NAN_BITS[dtype])
    elif dtype in _NAN_BITS8:
        out.view(torch.uint8).fill_(_NAN_BITS8[dtype])
    else:
        out.fill_(float("nan"))
    out[:, :cols] = t
    return out


@dataclass
class Problem:
    """One GEMM instance: C = alpha * op(A) * op(B) + beta * C0 (row-major storage).

    transA 0: A stored M x K (lda >= K); 1: A stored K x M (lda >= M).
    transB 0: B stored K x N (ldb >= N); 1: B stored N x K (ldb >= K).
    C0 is M x N with ldc >= N, in the output type; None when beta == 0.
    A has type in_dtype, B has b_dtype (the same unless a mixed 8-bit pair).
    """
    name: str
    M: int
    N: int
    K: int
    transA: int
    transB: int
    in_dtype: str
    out_dtype: str
    alpha: float
    beta: float
    A: torch.Tensor
    lda: int
    B: torch.Tensor
    ldb: int
    C0: object
    ldc: int
    seed: int
    recipe: dict = field(default_factory=dict)
    b_dtype: str = None

    def __post_init__(self):
        if self.b_dtype is None:
            self.b_dtype = self.in_dtype

    @property
    def layout(self):
        return ("T" if self.transA else "N") + ("T" if self.transB else "N")


def make_problem(name, M, N, K, transA=0, transB=0, in_dtype="bf16", out_dtype="f32",
                 dist_a=("uniform", -1.0, 1.0), dist_b=("uniform", -1.0, 1.0), alpha=1.0,
                 beta=0.0, dist_c=("normal", 0.0, 1.0), seed=0, lda=None, ldb=None, ldc=None, b_dtype=None,
                 logical=False):
    b_dtype = in_dtype if b_dtype is None else b_dtype
    a_shape = (K, M) if transA else (M, K)
    b_shape = (N, K) if transB else (K, N)
    lda = a_shape[1] if lda is None else lda
    ldb = b_shape[1] if ldb is None else ldb
    ldc = N if ldc is None else ldc
    if lda < a_shape[1] or ldb < b_shape[1] or ldc < N:
        raise ValueError("leading dimension smaller than the stored width")
    if logical:   # op(A) and op(B) drawn as M x K and K x N, stored per the layout
        a = draw((M, K), dist_a, seed, in_dtype)
        b = draw((K, N), dist_b, seed + 1, b_dtype)
        a = a.t().contiguous() if transA else a
        b = b.t().contiguous() if transB else b
    else:
        a = draw(a_shape, dist_a, seed, in_dtype)
        b = draw(b_shape, dist_b, seed + 1, b_dtype)
    A = _pad_columns(a, lda, in_dtype)
    B = _pad_columns(b, ldb, b_dtype)
    C0 = None
    if beta != 0.0:
        C0 = _pad_columns(draw((M, N), dist_c, seed + 2, out_dtype), ldc, out_dtype)
    recipe = {"dist_a": list(dist_a), "dist_b": list(dist_b), "dist_c": list(dist_c) if beta else None,
              "seeds": [seed, seed + 1, seed + 2], "drawn": "logical" if logical else "stored"}
    return Problem(name, M, N, K, transA, transB, in_dtype, out_dtype, float(alpha), float(beta),
                   A, lda, B, ldb, C0, ldc, seed, recipe, b_dtype)


@dataclass
class BatchedProblem:
    """A strided batch of GEMMs C_b = alpha * op(A_b) * op(B_b) + beta * C0_b,
    b < batch, with A_b = A[b * strideA :] etc. (row-major storage as in
    Problem; a stride of 0 reuses one matrix for every batch).  A, B, C0 are
    flat tensors of the input / output types."""
    name: str
    batch: int
    M: int
    N: int
    K: int
    transA: int
    transB: int
    in_dtype: str
    out_dtype: str
    alpha: float
    beta: float
    A: torch.Tensor
    lda: int
    strideA: int
    B: torch.Tensor
    ldb: int
    strideB: int
    C0: object
    ldc: int
    strideC: int
    seed: int
    b_dtype: str = None

    def __post_init__(self):
        if self.b_dtype is None:
            self.b_dtype = self.in_dtype


def _stack(mats, stride, dtype):
    """Lay the matrices out flat at `stride` elements apart (NaN bits between)."""
    rows, ld = mats[0].shape
    if stride == 0:
        return mats[0].reshape(-1).clone()
    if stride < rows * ld:
        raise ValueError("batch stride smaller than one matrix")
    flat = torch.empty(stride * (len(mats) - 1) + rows * ld, dtype=mats[0].dtype)
    if dtype in _NAN_BITS:
        flat.view(torch.int16).fill_(_NAN_BITS[dtype])
    elif dtype in _NAN_BITS8:
        flat.view(torch.uint8).fill_(_NAN_BITS8[dtype])
    else:
        flat.fill_(float("nan"))
    for b, m in enumerate(mats):
        flat[b * stride:b * stride + rows * ld] = m.reshape(-1)
    return flat


def make_batched_problem(name, batch, M, N, K, transA=0, transB=0, in_dtype="bf16", out_dtype="f32",
                         dist_a=("uniform", -1.0, 1.0), dist_b=("uniform", -1.0, 1.0), alpha=1.0, beta=0.0,
                         dist_c=("normal", 0.0, 1.0), seed=0, lda=None, ldb=None, ldc=None, strideA=None,
                         strideB=None, strideC=None, b_dtype=None):
    """Batch b draws A from seed + 3b, B from seed + 3b + 1, C0 from seed + 3b + 2
    (one draw when that operand's stride is 0); strides default to packed."""
    b_dtype = in_dtype if b_dtype is None else b_dtype
    a_shape = (K, M) if transA else (M, K)
    b_shape = (N, K) if transB else (K, N)
    lda = a_shape[1] if lda is None else lda
    ldb = b_shape[1] if ldb is None else ldb
    ldc = N if ldc is None else ldc
    strideA = a_shape[0] * lda if strideA is None else strideA
    strideB = b_shape[0] * ldb if strideB is None else strideB
    strideC = M * ldc if strideC is None else strideC
    nA = 1 if strideA == 0 else batch
    nB = 1 if strideB == 0 else batch
    A = _stack([_pad_columns(draw(a_shape, dist_a, seed + 3 * b, in_dtype), lda, in_dtype) for b in range(nA)],
               strideA, in_dtype)
    B = _stack([_pad_columns(draw(b_shape, dist_b, seed + 3 * b + 1, b_dtype), ldb, b_dtype) for b in range(nB)],
               strideB, b_dtype)
    C0 = None
    if beta != 0.0:
        C0 = _stack([_pad_columns(draw((M, N), dist_c, seed + 3 * b + 2, out_dtype), ldc, out_dtype)
                     for b in range(batch)], strideC, out_dtype)
    return BatchedProblem(name, batch, M, N, K, transA, transB, in_dtype, out_dtype, float(alpha), float(beta),
                          A, lda, strideA, B, ldb, strideB, C0, ldc, strideC, seed, b_dtype)


@dataclass
class GroupedProblem:
    """Grouped GEMMs with stacked rows (mixture-of-experts routing): group g owns
    rows [off_g, off_g + m_sizes[g]) of A (sum(m) x K) and C (sum(m) x N) and
    multiplies them by B_g = B[g * strideB:] (N x K when transB, else K x N)."""
    name: str
    m_sizes: list
    N: int
    K: int
    transB: int
    in_dtype: str
    out_dtype: str
    alpha: float
    beta: float
    A: torch.Tensor
    lda: int
    B: torch.Tensor
    ldb: int
    strideB: int
    C0: object
    ldc: int
    seed: int
    b_dtype: str = None

    def __post_init__(self):
        if self.b_dtype is None:
            self.b_dtype = self.in_dtype

    @property
    def M(self):
        return int(sum(self.m_sizes))


def make_grouped_problem(name, m_sizes, N, K, transB=1, in_dtype="bf16", out_dtype="f32",
                         dist_a=("normal", 0.0, 1.0), dist_b=("normal", 0.0, 0.02), alpha=1.0, beta=0.0,
                         dist_c=("normal", 0.0, 1.0), seed=0, lda=None, ldb=None, strideB=None, ldc=None,
                         b_dtype=None):
    """A from seed, C0 from seed + 2, expert g's weights from seed + 3 + g."""
    b_dtype = in_dtype if b_dtype is None else b_dtype
    M = int(sum(m_sizes))
    b_shape = (N, K) if transB else (K, N)
    lda = K if lda is None else lda
    ldb = b_shape[1] if ldb is None else ldb
    ldc = N if ldc is None else ldc
    strideB = b_shape[0] * ldb if strideB is None else strideB
    A = _pad_columns(draw((M, K), dist_a, seed, in_dtype), lda, in_dtype)
    B = _stack([_pad_columns(draw(b_shape, dist_b, seed + 3 + g, b_dtype), ldb, b_dtype)
                for g in range(len(m_sizes))], strideB, b_dtype)
    C0 = None
    if beta != 0.0:
        C0 = _pad_columns(draw((M, N), dist_c, seed + 2, out_dtype), ldc, out_dtype)
    return GroupedProblem(name, [int(m) for m in m_sizes], N, K, transB, in_dtype, out_dtype, float(alpha),
                          float(beta), A, lda, B, ldb, strideB, C0, ldc, seed, b_dtype)


def moe_routing(tokens=8192, experts=64, seed=0):
    """Uneven tokens per expert for a mixture-of-experts layer: a seeded
    multinomial draw of `tokens` routed tokens over `experts` experts."""
    g = _rng(seed)
    w = g.gamma(2.0, 1.0, experts)
    return [int(x) for x in g.multinomial(tokens, w / w.sum())]


# ---------------------------------------------------------------------------
# The workloads, named by what they are.
# ---------------------------------------------------------------------------

def tiny_256():
    """M = N = K = 256, A and B row-major, bf16 U[-1, 1], alpha 1, beta 0, fp32 C."""
    return make_problem("tiny_256_bf16_nn", 256, 256, 256, 0, 0, "bf16", "f32")


def square_4096_bf16_nt(out_dtype="f32", size=4096):
    """M = N = K = 4096, A row-major, B column-major (NT), bf16 N(0, 1)/sqrt(K)."""
    std = 1.0 / math.sqrt(size)
    return make_problem("square_%d_bf16_nt_%s" % (size, out_dtype), size, size, size, 0, 1, "bf16",
                        out_dtype, ("normal", 0.0, std), ("normal", 0.0, std))


def square_4096_f16_blend(transA, transB, size=4096):
    """M = N = K = 4096, fp16 U[-1, 1], alpha 1.5, beta 0.5, fp32 C0 ~ N(0, 1).
    The four layouts store the same logical A and B (drawn as M x K and K x N)."""
    lay = ("T" if transA else "N") + ("T" if transB else "N")
    return make_problem("square_%d_f16_blend_%s" % (size, lay.lower()), size, size, size, transA,
                        transB, "f16", "f32", alpha=1.5, beta=0.5, dist_c=("normal", 0.0, 1.0), logical=True)


LLM_SHAPES = {
    # name: (M, K, N) -- M is batch x sequence
    "qkv_proj": (8192, 4096, 12288),
    "ffn_up": (8192, 4096, 16384),
    "ffn_down": (8192, 16384, 4096),
}


def llm_projection(name, transB=0):
    """LLM projection: activations N(0, 1), weights N(0, 0.02), bf16, beta 0, fp32 C."""
    M, K, N = LLM_SHAPES[name]
    return make_problem("%s_%s" % (name, "nt" if transB else "nn"), M, N, K, 0, transB, "bf16", "f32",
                        ("normal", 0.0, 1.0), ("normal", 0.0, 0.02))


def ragged_4095_4097_1000():
    """Ragged tile edges: M = 4095, N = 4097, K = 1000, NN, bf16 as the LLM shapes."""
    return make_problem("ragged_4095x4097x1000_nn", 4095, 4097, 1000, 0, 0, "bf16", "f32",
                        ("normal", 0.0, 1.0), ("normal", 0.0, 0.02))


def attention_scores(batch_heads=32, seq=2048, head_dim=128):
    """Attention scores Q K^T for batch x heads pairs: Q (S x d) and K (S x d)
    row-major, so the product is NT; bf16 N(0, 1), alpha 1/sqrt(d), bf16 out."""
    return make_batched_problem("attn_qk_%dx%dx%d" % (batch_heads, seq, head_dim), batch_heads, seq, seq,
                                head_dim, 0, 1, "bf16", "bf16", ("normal", 0.0, 1.0), ("normal", 0.0, 1.0),
                                alpha=1.0 / math.sqrt(head_dim))


def lm_head_64():
    """Skinny LM head: M = 64 (decode batch), K = 4096, N = 32000 (vocabulary).

    Weights are stored vocabulary-major (N x K), i.e. the NT layout.
    """
    return make_problem("lm_head_64x32000x4096_nt", 64, 32000, 4096, 0, 1, "bf16", "f32",
                        ("normal", 0.0, 1.0), ("normal", 0.0, 0.02))


def square_4096_fp8_nt(fmt="e4m3", out_dtype="f32", size=4096):
    """M = N = K = 4096, A row-major, B column-major (NT), 8-bit float inputs
    N(0, 1) (inside both formats' ranges), alpha 1 / K so that C is O(1)."""
    return make_problem("square_%d_%s_nt_%s" % (size, fmt, out_dtype), size, size, size, 0, 1, fmt,
                        out_dtype, ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), alpha=1.0 / size)


def square_4096_f32_nt(size=4096):
    """M = N = K = 4096 fp32, A row-major, B column-major (NT), entries N(0, 1),
    alpha 1 / K so that C is O(1): the fp32 GEMM emulated with TF32 products."""
    return make_problem("square_%d_f32_nt_f32" % size, size, size, size, 0, 1, "f32", "f32",
                        ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), alpha=1.0 / size)


# ----------------------------------------------------------------------------
# Block-scaled inputs: MXFP8 (E4M3 / E5M2 codes, one E8M0 scale per 32 values
# of k) and NVFP4 (E2M1 codes packed two to a byte, one unsigned E4M3 scale per
# 16).  Values are drawn in float32 as N(0, 1) times a per-block power of two
# 2^t, t uniform in [-6, 6], so that the scales differ from block to block;
# each block is then quantised the usual way for its format:
#   MXFP8: shared exponent e = floor(log2(max |x|)) - emax (emax 8 for E4M3,
#          15 for E5M2), scale code e + 127, codes = RNE(x / 2^e) saturated;
#   NVFP4: scale = RNE_E4M3(max |x| / 6), codes = the nearest E2M1 value of
#          x / scale (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).
# This prepares data; the GEMM arithmetic on it lives in the oracle and the
# kernels.  Scale rows are padded to 16 bytes with the code 0xFF (NaN as
# E8M0), matrix rows past K with 0xFF bytes: neither may be read.

BLOCK_FORMATS = {"mxfp8": ("e8m0", 32), "nvfp4": ("ue4m3", 16)}
_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def _block_values(rows, K, block, seed, seed_t):
    g, gt = _rng(seed), _rng(seed_t)
    nblk = -(-K // block)
    t = gt.integers(-6, 7, size=(rows, nblk)).astype(np.float32)
    x = g.standard_normal(size=(rows, nblk * block), dtype=np.float32)
    x = x.reshape(rows, nblk, block) * np.exp2(t)[..., None]
    if nblk * block > K:   # the last block's tail lies past K: no values there
        flat = x.reshape(rows, nblk * block)
        flat[:, K:] = 0.0
    return x


def _quantise(x, fmt, elem):
    """x: rows x nblk x block float32 -> (codes rows x nblk*block uint8, scale codes rows x nblk uint8)."""
    rows, nblk, block = x.shape
    amax = np.abs(x).max(axis=2)
    if fmt == "mxfp8":
        emax, vmax = (8, 448.0) if elem == "e4m3" else (15, 57344.0)
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - emax
        e = np.clip(e, -127, 127)
        sf = (e + 127).astype(np.uint8)
        q = np.clip(x / np.exp2(e)[..., None], -vmax, vmax).astype(np.float32)
        codes = torch.from_numpy(np.ascontiguousarray(q.reshape(rows, -1))).to(_TORCH_DT[elem])
        return codes.view(torch.uint8).numpy(), sf
    sf_t = torch.from_numpy(np.ascontiguousarray((amax / 6.0).astype(np.float32))).to(torch.float8_e4m3fn)
    sf = sf_t.view(torch.uint8).numpy().copy()
    scale = sf_t.to(torch.float32).numpy()
    q = x / np.where(scale > 0, scale, 1.0)[..., None]
    idx = np.abs(np.abs(q)[..., None] - _E2M1_MAGS).argmin(axis=-1).astype(np.uint8)
    codes = idx | ((q < 0).astype(np.uint8) << 3)
    return codes.reshape(rows, -1), sf


def _store_codes(codes, K, ld, elem):
    """rows x >= K codes -> rows x bytes-per-row uint8 tensor (E2M1: two per byte, even one low)."""
    rows = codes.shape[0]
    if elem == "e2m1":
        c = np.zeros((rows, ld), dtype=np.uint8)
        c[:, :K] = codes[:, :K]
        packed = c[:, 0::2] | (c[:, 1::2] << 4)
        packed[:, -(-K // 2):] = 0xFF
        return torch.from_numpy(np.ascontiguousarray(packed))
    out = np.full((rows, ld), 0xFF, dtype=np.uint8)
    out[:, :K] = codes[:, :K]
    return torch.from_numpy(out)


@dataclass
class BlockScaledProblem:
    """C = alpha * A' * B'^T + beta * C0 with A' (M x K) and B' (N x K) given as
    block-scaled codes: A, B uint8 tensors of the stored rows (lda / ldb in
    elements; E2M1 packs two elements a byte), SFA (M x ld_sfa) and SFB (N x
    ld_sfb) the scale codes, one per `block` values of k."""
    name: str
    M: int
    N: int
    K: int
    fmt: str          # "mxfp8" | "nvfp4"
    a_elem: str       # "e4m3" | "e5m2" | "e2m1"
    b_elem: str
    out_dtype: str
    alpha: float
    beta: float
    A: torch.Tensor
    lda: int
    SFA: torch.Tensor
    ld_sfa: int
    B: torch.Tensor
    ldb: int
    SFB: torch.Tensor
    ld_sfb: int
    C0: object
    ldc: int
    block: int
    seed: int


def make_block_scaled_problem(name, M, N, K, fmt="mxfp8", out_dtype="f32", a_elem=None, b_elem=None, alpha=1.0,
                              beta=0.0, seed=0, lda=None, ldb=None, ldc=None, ld_sf=None):
    """A from seeds (s, s + 3), B from (s + 1, s + 4), C0 from s + 2.  Default
    leading dimensions: K rounded up to 16 bytes of codes; scale rows padded
    to 16 bytes."""
    _, block = BLOCK_FORMATS[fmt]
    a_elem = a_elem or ("e4m3" if fmt == "mxfp8" else "e2m1")
    b_elem = b_elem or a_elem
    per16 = 32 if fmt == "nvfp4" else 16          # elements in 16 bytes
    up = lambda v, m: -(-v // m) * m
    lda = up(K, per16) if lda is None else lda
    ldb = up(K, per16) if ldb is None else ldb
    ldc = N if ldc is None else ldc
    nblk = -(-K // block)
    ld_sf = up(max(nblk, 1), 16) if ld_sf is None else ld_sf
    mats = []
    for rows, elem, sv, st, ld in ((M, a_elem, seed, seed + 3, lda), (N, b_elem, seed + 1, seed + 4, ldb)):
        codes, sf = _quantise(_block_values(rows, K, block, sv, st), fmt, elem)
        sfs = np.full((rows, ld_sf), 0xFF, dtype=np.uint8)
        sfs[:, :nblk] = sf
        mats.append((_store_codes(codes, K, ld, elem), torch.from_numpy(sfs)))
    C0 = None
    if beta != 0.0:
        C0 = _pad_columns(draw((M, N), ("normal", 0.0, 1.0), seed + 2, out_dtype), ldc, out_dtype)
    return BlockScaledProblem(name, M, N, K, fmt, a_elem, b_elem, out_dtype, float(alpha), float(beta),
                              mats[0][0], lda, mats[0][1], ld_sf, mats[1][0], ldb, mats[1][1], ld_sf, C0, ldc,
                              block, seed)


def bits(t):
    """Raw bit patterns of an input tensor, without copying values: numpy
    uint16 for bf16 / fp16, uint8 for the 8-bit formats, float32 as it is."""
    if t.element_size() == 1:
        return t.contiguous().view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.contiguous().numpy()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
