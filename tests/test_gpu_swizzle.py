"""The 128-byte swizzle, pinned on the hardware: one tile load issued the way
the GEMM loads a K-major 16-bit operand tile puts element (r, c) at 16-bit
position r * 64 + (c ^ ((r & 7) << 3)) of shared memory, the layout the MMA's
shared-memory descriptors assume ("[CUDA 优化实战] hgemm sm120 - 100KB SMEM
中的“微雕”战争", section 4).  The source holds each element's own index, so the
test reads the permutation directly."""
import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    gh = G.Handle(0)
    yield gh
    gh.close()


_TIMED_OUT = []   # a timed-out probe ends the module's probe launches


def probe(h, rows, cols, ld):
    if _TIMED_OUT:
        pytest.fail("an earlier probe timed out (%s): no further probe is launched" % _TIMED_OUT[0])
    r = np.arange(rows)[:, None]
    c = np.arange(ld)[None, :]
    src_np = (r * 64 + c).astype(np.uint16)          # element (r, c) holds r * 64 + c (c < 64)
    src_np[:, cols:] = 0xFFFF                         # past cols: must not arrive
    src = torch.from_numpy(src_np.view(np.int16)).cuda()
    dst = torch.full((rows * 64,), -1, dtype=torch.int16, device="cuda")
    st = G.lib().gemm_probe_tma_tile(h.ptr, src.data_ptr(), ld, cols, rows, dst.data_ptr(), None)
    assert st == G.OK, G.STATUS.get(st)
    status = h.status()[0]
    if status == G.ERR_TIMEOUT:
        _TIMED_OUT.append("rows %d, cols %d, ld %d" % (rows, cols, ld))
    assert status == G.OK
    return dst.cpu().numpy().view(np.uint16).reshape(rows, 64)


@pytest.mark.parametrize("rows,cols,ld", [(8, 64, 64), (64, 64, 72), (256, 64, 64), (40, 64, 200)])
def test_swizzle_128b_layout(h, rows, cols, ld):
    got = probe(h, rows, cols, ld)
    for r in range(rows):
        for c in range(64):
            assert got[r, c ^ ((r & 7) << 3)] == r * 64 + c, (r, c)


def test_columns_past_the_matrix_arrive_as_zeros(h):
    got = probe(h, 16, 40, 48)
    for r in range(16):
        for c in range(64):
            want = r * 64 + c if c < 40 else 0
            assert got[r, c ^ ((r & 7) << 3)] == want, (r, c)
