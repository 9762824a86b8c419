"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times, on sampled outputs the oracle computes one by one (random
entries, corners, first / last rows and columns, the ragged last tiles)."""
import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import assert_close, device_problem, launch, oracle_at, sample_indices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


def _sampled(p, h, count=3000):
    Ad, Bd, Cd, ldc = device_problem(p)
    launch(p, h, Ad, Bd, Cd, ldc)
    st, word = h.status()
    assert st == G.OK, "status %s word 0x%x" % (G.STATUS.get(st), word)
    rows, cols = sample_indices(p.M, p.N, count, seed=p.M * 7 + p.N)
    ri = torch.from_numpy(rows).cuda()
    ci = torch.from_numpy(cols).cuda()
    out = Cd[ri, ci].double().cpu().numpy()
    r, m = oracle_at(p, rows, cols)
    assert_close(out, r, m, p.out_dtype == "f32", p.name)
    # every output is finite (beta == 0 runs start from a NaN-filled C)
    assert bool(torch.isfinite(Cd[:p.M, :p.N]).all())
    return Cd


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_square_4096_bf16_nt(h, out_dtype):
    _sampled(inputs.square_4096_bf16_nt(out_dtype), h)


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_square_4096_f16_blend(h, transA, transB):
    _sampled(inputs.square_4096_f16_blend(transA, transB), h, count=2000)


@pytest.mark.parametrize("name", ["qkv_proj", "ffn_up", "ffn_down"])
@pytest.mark.parametrize("transB", [0, 1])
def test_llm_projections(h, name, transB):
    _sampled(inputs.llm_projection(name, transB), h, count=1500)


def test_ragged_4095_4097_1000(h):
    _sampled(inputs.ragged_4095_4097_1000(), h, count=4000)


def test_lm_head_64(h):
    p = inputs.lm_head_64()
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB)
    assert plan.swap_ab == 1
    Cd = _sampled(p, h, count=6000)
    # M = 64 is small enough to check one full row of the vocabulary as well
    from gpu_util import oracle_at as _at
    cols = np.arange(p.N, dtype=np.int64)
    rows = np.full(p.N, 17, dtype=np.int64)
    r, m = _at(p, rows, cols)
    assert_close(Cd[17, :p.N].double().cpu().numpy(), r, m, True, "lm_head row 17")


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
    _sampled(p, h, count=2000)


def test_largest_extent_is_refused_not_run(h):
    """Extents past the kernels' 32-bit index range are refused at planning time."""
    with pytest.raises(G.GemmError) as e:
        G.plan(1 << 31, 64, 64, 0, 1, handle=h)
    assert e.value.status == G.ERR_UNSUPPORTED
