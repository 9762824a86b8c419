"""The multi-GPU path is replicas only (the GEMM exchanges no data between
GPUs): every rank runs its own GEMM and rank 0 reports all ranks' work over the
slowest rank's time.  Checked here on CPU with world-size-2 gloo groups: the
max-over-ranks timing, the whole-job value, a rank that fails before the
barrier (the other gets an error, not a hang), and the reference arm under
torchrun (rank 0 prints, rank 1 exits 0 without work)."""
import datetime
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, mode, results):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", timeout=datetime.timedelta(seconds=5))
    try:
        if mode == "fail" and rank == 1:
            raise SystemExit(3)      # leaves before the barrier, with nothing in flight
        if mode == "fail":
            try:
                dist.barrier()
                results[rank] = "no error"
            except Exception as e:   # the peer never arrives: a timeout or a closed connection
                results[rank] = "error: " + type(e).__name__
            return
        ms = bench.slowest_over_ranks(10.0 * (rank + 1))
        ws, r, _ = bench.dist_env()
        results[rank] = (ms, ws, r, bench.job_value(137438953472, ws, 20, ms))
    finally:
        if mode != "fail" or rank == 0:
            try:
                dist.destroy_process_group()
            except Exception:
                pass


def _run(mode):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, PORT[0], mode, results))
                 for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(60)
            assert p.exitcode is not None, "a rank hung"
        return dict(results), [p.exitcode for p in procs]


PORT = [0]


@pytest.fixture(autouse=True)
def _port():
    PORT[0] = _free_port()


def test_slowest_rank_sets_the_time():
    res, codes = _run("time")
    assert codes == [0, 0]
    for rank in (0, 1):
        ms, ws, r, value = res[rank]
        assert ms == 20.0 and ws == 2 and r == rank
        # two ranks' FLOPs over the slower one's 20 ms for 20 steps
        assert value == pytest.approx(2 * 137438953472 * 20 / 0.020 / 1e12)


def test_a_rank_that_leaves_is_seen_as_an_error():
    res, codes = _run("fail")
    assert codes[1] == 3
    assert res[0].startswith("error")


def test_reference_arm_under_torchrun():
    """Rank 0 alone times the oracle and prints one JSON line; rank 1 exits 0."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
