"""The seeded input generators (no GPU): the fp16 blend workload's four layouts
hold the same logical matrices, so one oracle product serves all four."""
import torch

from dense_gemm_10_gb300 import inputs


def _logical(t, trans):
    return t.t() if trans else t


def test_blend_layouts_share_logical_operands():
    ref = inputs.square_4096_f16_blend(0, 0, size=96)
    for ta, tb in ((0, 1), (1, 0), (1, 1)):
        p = inputs.square_4096_f16_blend(ta, tb, size=96)
        assert p.layout == ("T" if ta else "N") + ("T" if tb else "N")
        assert tuple(p.A.shape) == ((96, 96)) and p.transA == ta and p.transB == tb
        assert torch.equal(_logical(p.A, ta).view(torch.int16), ref.A.view(torch.int16))
        assert torch.equal(_logical(p.B, tb).view(torch.int16), ref.B.view(torch.int16))
        assert torch.equal(p.C0, ref.C0)


def test_blend_layouts_differ_in_storage():
    """The transposed layouts really store the transpose (not the same bytes)."""
    nn = inputs.square_4096_f16_blend(0, 0, size=64)
    tt = inputs.square_4096_f16_blend(1, 1, size=64)
    assert not torch.equal(tt.A.view(torch.int16), nn.A.view(torch.int16))
    assert not torch.equal(tt.B.view(torch.int16), nn.B.view(torch.int16))


def test_stored_draws_are_unchanged_for_other_workloads():
    """Problems without logical=True still draw each matrix in its stored shape."""
    a = inputs.make_problem("x", 8, 12, 16, 1, 0, "bf16", "f32", seed=5)
    b = inputs.draw((16, 8), ("uniform", -1.0, 1.0), 5, "bf16")
    assert torch.equal(a.A.view(torch.int16), b.view(torch.int16))
