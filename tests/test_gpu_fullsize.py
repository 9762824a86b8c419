"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times.

Full matrix: every element of C is compared with the oracle for the square
4096^3 bf16 NT workload (fp32 and bf16 C), the fp16 blend workload in its four
layouts, the QKV projection (NN), the ragged 4095 x 4097 x 1000 workload, the
LM head and the extreme shapes.  The oracle runs once per distinct logical
product: the fp32- and bf16-output runs of the square workload share one, and
so do the four blend layouts, which store the same logical A and B four ways.
The oracle's share of the suite's time is about 5 minutes on 16 host cores
(3.6 GFLOP/s: 137 GFLOP for each square product, 825 GFLOP for QKV).

Sampled (random entries, corners, first / last rows and columns, the ragged
last tiles): the FFN-up and FFN-down projections and the NT layouts of the
projections, 1.1 TFLOP each, which would add about 5 minutes apiece."""
import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import assert_close, device_problem, launch, oracle_at, oracle_full, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


_ORACLE = {}


def _oracle_once(key, p):
    """The oracle's full result for logical product `key`, computed once and kept
    while consecutive tests use it (one at a time: QKV's alone is 1.6 GB)."""
    if key not in _ORACLE:
        _ORACLE.clear()
        _ORACLE[key] = oracle_full(p)
    return _ORACLE[key]


def _run(p, h):
    Ad, Bd, Cd, ldc = device_problem(p)
    launch(p, h, Ad, Bd, Cd, ldc)
    st, word = h.status()
    assert st == G.OK, "status %s word 0x%x" % (G.STATUS.get(st), word)
    return Cd


def _full(p, h, key):
    Cd = _run(p, h)
    out = Cd[:p.M, :p.N].double().cpu().numpy()
    del Cd
    R, Mag = _oracle_once(key, p)
    assert_close(out, R, Mag, p.out_dtype == "f32", p.name)


def _sampled(p, h, count=3000):
    Cd = _run(p, h)
    rows, cols = sample_indices(p.M, p.N, count, seed=p.M * 7 + p.N)
    ri = torch.from_numpy(rows).cuda()
    ci = torch.from_numpy(cols).cuda()
    out = Cd[ri, ci].double().cpu().numpy()
    r, m = oracle_at(p, rows, cols)
    assert_close(out, r, m, p.out_dtype == "f32", p.name)
    # every output is finite (beta == 0 runs start from a NaN-filled C)
    assert bool(torch.isfinite(Cd[:p.M, :p.N]).all())


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_square_4096_bf16_nt(h, out_dtype):
    _full(inputs.square_4096_bf16_nt(out_dtype), h, "square_4096_bf16_nt")


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_square_4096_f16_blend(h, transA, transB):
    _full(inputs.square_4096_f16_blend(transA, transB), h, "square_4096_f16_blend")


def test_qkv_projection_nn_full(h):
    _full(inputs.llm_projection("qkv_proj", 0), h, "qkv_proj_nn")


@pytest.mark.parametrize("name,transB", [("qkv_proj", 1), ("ffn_up", 0), ("ffn_up", 1), ("ffn_down", 0),
                                         ("ffn_down", 1)])
def test_llm_projections_sampled(h, name, transB):
    _sampled(inputs.llm_projection(name, transB), h, count=1500)


def test_ragged_4095_4097_1000(h):
    _full(inputs.ragged_4095_4097_1000(), h, "ragged")


def test_lm_head_64(h):
    p = inputs.lm_head_64()
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB)
    assert plan.swap_ab == 1
    _full(p, h, "lm_head")


@pytest.mark.parametrize("M,N,K,transA,transB", [
    (1, 4096, 4096, 0, 1),        # one row of C (swapped: the 4096 columns on the MMA's rows)
    (4096, 1, 4096, 0, 0),        # one column of C
    (128, 136, 131072, 0, 1),     # very long K: every k-block of one tile row, split across the grid
    (262144, 64, 128, 0, 0),      # 2048 tile rows, one tile column
    (3, 5, 7, 1, 1),              # smaller than every tile in all three dimensions
])
def test_extreme_shapes(h, M, N, K, transA, transB):
    p = inputs.make_problem("extreme_%dx%dx%d" % (M, N, K), M, N, K, transA, transB, "bf16", "f32",
                            ("normal", 0.0, 1.0), ("normal", 0.0, 1.0), seed=M % 97 + K % 89)
    _full(p, h, p.name)


def test_largest_extent_is_refused_not_run(h):
    """Extents past the kernels' 32-bit index range are refused at planning time."""
    with pytest.raises(G.GemmError) as e:
        G.plan(1 << 31, 64, 64, 0, 1, handle=h)
    assert e.value.status == G.ERR_UNSUPPORTED
