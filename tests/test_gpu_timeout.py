"""Failure detection without a GPU fault: the test hook makes CTA 0 skip one
k-block load, so one mbarrier phase never completes.  The kernel's bounded
wait must run out (short limit), record a timeout in the status word, leave
every role's loop and free Tensor Memory; gemm_get_status reports
GEMM_ERR_TIMEOUT, and the next GEMM on the same handle and context is correct.
No trap, no fault, no unbounded loop is involved."""
import numpy as np
import pytest
import torch

from dense_gemm_10_gb300 import gemm as G
from dense_gemm_10_gb300 import inputs

from gpu_util import assert_close, device_problem, launch, oracle_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path,stream_k", [(G.PATH_TC_1CTA, 1), (G.PATH_TC_2CTA, 1), (G.PATH_TC_2CTA, 2),
                                           (G.PATH_TC_1CTA, 2)])
def test_dropped_load_times_out_then_recovers(path, stream_k):
    h = G.Handle(0)
    try:
        p = inputs.make_problem("drop", 640, 768, 1024, 0, 1, "bf16", "f32", ("normal", 0, 1), ("normal", 0, 1),
                                seed=path + 10 * stream_k)
        h.set_option(G.OPT_FORCE_PATH, path)
        h.set_option(G.OPT_STREAM_K, stream_k)
        h.set_option(G.OPT_MAX_GRID, 14)          # several units per CTA, an incomplete last wave
        h.set_option(G.OPT_WAIT_LIMIT_NS, 50_000_000)
        h.set_option(G.OPT_TEST_DROP_LOAD, 3)
        Ad, Bd, Cd, ldc = device_problem(p)
        launch(p, h, Ad, Bd, Cd, ldc)
        st, word = h.status()
        assert st == G.ERR_TIMEOUT
        assert word & 0xFF == 6 and (word >> 8) & 0xF in (1, 2, 3)
        # the status word was cleared: a second read is clean
        assert h.status()[0] == G.OK
        # the same handle, same configuration, without the hook: correct again
        h.set_option(G.OPT_TEST_DROP_LOAD, 0)
        Ad, Bd, Cd, ldc = device_problem(p)
        launch(p, h, Ad, Bd, Cd, ldc)
        st, word = h.status()
        assert st == G.OK, hex(word)
        R, Mag = oracle_full(p)
        assert_close(Cd[:p.M, :p.N].double().cpu().numpy(), R, Mag, True, "after timeout")
    finally:
        h.close()
