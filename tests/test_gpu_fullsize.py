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
