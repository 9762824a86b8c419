"""The C ABI from a plain C program (tests/c_abi_example.c, built here with
gcc against include/gemm_gb300.h and the library), and gemm_run captured in a
CUDA graph and replayed."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_10_gb300 import gemm as G

from gpu_util import assert_close

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_program(repo_tmp):
    G.lib()   # the library is built
    cuda = "/usr/local/cuda"
    exe = repo_tmp / "c_abi_example"
    libdir = os.path.dirname(G.LIB_PATH)
    subprocess.run(["gcc", "-O1", "-std=c11", os.path.join(ROOT, "tests", "c_abi_example.c"), "-o", str(exe),
                    "-I" + os.path.join(ROOT, "include"), "-I" + cuda + "/include", "-L" + libdir,
                    "-L" + cuda + "/lib64", "-lgemm_gb300", "-lcudart", "-lm", "-Wl,-rpath," + libdir,
                    "-Wl,-rpath," + cuda + "/lib64"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr


def test_cuda_graph_replay():
    """Three dependent GEMMs captured once and replayed: each replay recomputes
    from the current contents of the input buffers."""
    h = G.Handle(0)
    try:
        g = torch.Generator().manual_seed(5)
        X = torch.randn(512, 384, generator=g).to(torch.bfloat16).cuda()
        W1 = (torch.randn(384, 640, generator=g) / 16).to(torch.bfloat16).cuda()
        W2 = (torch.randn(640, 256, generator=g) / 16).to(torch.bfloat16).cuda()
        H = torch.empty(512, 640, dtype=torch.bfloat16, device="cuda")
        Y = torch.empty(512, 256, device="cuda")
        s = torch.cuda.Stream()

        def step():
            assert h.run_raw(0, 0, 512, 640, 384, 1.0, X.data_ptr(), 384, W1.data_ptr(), 640, 0.0, H.data_ptr(),
                             640, G.BF16_BF16, s.cuda_stream) == G.OK
            assert h.run_raw(0, 0, 512, 256, 640, 1.0, H.data_ptr(), 640, W2.data_ptr(), 256, 0.0, Y.data_ptr(),
                             256, G.BF16_F32, s.cuda_stream) == G.OK

        with torch.cuda.stream(s):
            step()                 # plans, workspace and launches set up outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
        bits = lambda t: t.contiguous().view(torch.uint16).numpy()
        for rep in range(2):
            X.copy_(torch.randn(512, 384, generator=g).to(torch.bfloat16))
            Y.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert h.status()[0] == G.OK
            Hc = H.cpu()
            R1, M1 = oracle.gemm(0, 0, 512, 640, 384, 1.0, bits(X.cpu()), 384, bits(W1.cpu()), 640, 0.0, None, 640,
                                 oracle.IN_BF16)
            assert_close(Hc.double().numpy(), R1, M1, False, "H, replay %d" % rep)
            R2, M2 = oracle.gemm(0, 0, 512, 256, 640, 1.0, bits(Hc), 640, bits(W2.cpu()), 256, 0.0, None, 256,
                                 oracle.IN_BF16)
            assert_close(Y.cpu().double().numpy(), R2, M2, True, "Y, replay %d" % rep)
    finally:
        h.close()
