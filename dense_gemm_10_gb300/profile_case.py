"""Run one benchmark workload a few times through the library, for a profiler.

    python -m dense_gemm_10_gb300.profile_case CASE [--launches N] [--raster-group G] [--option OPT_X=V ...]

Every case is one of the benchmark's workloads (seeded synthetic inputs of the
benchmark's shapes), called N times back to back on one stream through the
public entry points; the handle's status is checked at the end and the
process exits non-zero on any error.  --raster-group sets the number of tile
rows per raster group of the persistent schedule (0: the library's choice);
--option sets any other handle option by its binding name (OPT_STREAM_K=1:
no stream-K).
Under a profiler, skip the first calls (their set-up and cold caches) and
capture one or two of the later ones:

    ncu --set full --clock-control none -k regex:tc_gemm_kernel -s 2 -c 1 \\
        -o prof python -m dense_gemm_10_gb300.profile_case square_4096_nt_f32
"""
import argparse
import sys

import torch

from . import gemm as G
from . import inputs


def _plain(p, code):
    return p, code


CASES = {
    "square_4096_nt_f32": lambda: _plain(inputs.square_4096_bf16_nt("f32"), G.BF16_F32),
    "square_4096_nt_bf16": lambda: _plain(inputs.square_4096_bf16_nt("bf16"), G.BF16_BF16),
    "blend_4096_tn_f16": lambda: _plain(inputs.square_4096_f16_blend(1, 0), G.F16_F32),
    "qkv_8192x12288x4096_nn": lambda: _plain(inputs.llm_projection("qkv_proj", 0), G.BF16_F32),
    "ragged_4095x4097x1000_nn": lambda: _plain(inputs.ragged_4095_4097_1000(), G.BF16_F32),
    "lm_head_64x32000x4096_nt": lambda: _plain(inputs.lm_head_64(), G.BF16_F32),
    "square_4096_e4m3_nt": lambda: _plain(inputs.square_4096_fp8_nt("e4m3", "f32"), G.fp8_dtype("e4m3", "e4m3", "f32")),
}
BLOCK_CASES = ("lm_head_64x32000x4096_nvfp4",)


def run(case, launches, raster_group=0, options=()):
    h = G.Handle(0)
    try:
        if raster_group:
            h.set_option(G.OPT_RASTER_GROUP, raster_group)
        for opt, value in options:
            h.set_option(opt, value)
        if case in BLOCK_CASES:
            p = inputs.make_block_scaled_problem(case, 64, 32000, 4096, "nvfp4", "bf16", seed=0, alpha=1.0 / 64)
            A, SA, B, SB = p.A.cuda(), p.SFA.cuda(), p.B.cuda(), p.SFB.cuda()
            C = torch.empty(p.M, p.ldc, dtype=torch.bfloat16, device="cuda")
            for _ in range(launches):
                st = h.run_block_scaled_raw(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, SA.data_ptr(), p.ld_sfa,
                                            B.data_ptr(), p.ldb, SB.data_ptr(), p.ld_sfb, 0.0, C.data_ptr(), p.ldc,
                                            G.NVFP4_BF16, None)
                if st != G.OK:
                    raise G.GemmError(st, "gemm_run_block_scaled")
        else:
            p, code = CASES[case]()
            out = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.out_dtype]
            A, B = p.A.cuda(), p.B.cuda()
            C = p.C0.cuda() if p.C0 is not None else torch.empty(p.M, p.ldc, dtype=out, device="cuda")
            for _ in range(launches):
                st = h.run_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                               p.beta, C.data_ptr(), p.ldc, code, None)
                if st != G.OK:
                    raise G.GemmError(st, "gemm_run")
        st, word = h.status()
        if st != G.OK:
            raise RuntimeError("%s: status %s (0x%x)" % (case, G.STATUS.get(st), word))
    finally:
        h.close()
    print("%s: %d calls, status ok" % (case, launches))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("case", choices=sorted(CASES) + list(BLOCK_CASES))
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--raster-group", type=int, default=0)
    ap.add_argument("--option", action="append", default=[], metavar="OPT_NAME=V")
    a = ap.parse_args(argv)
    if a.raster_group < 0:
        ap.error("--raster-group must be >= 0")
    options = []
    for item in a.option:
        name, _, value = item.partition("=")
        if not name.startswith("OPT_") or not hasattr(G, name) or not value.lstrip("-").isdigit():
            ap.error("--option wants OPT_NAME=INTEGER, got %r" % item)
        options.append((getattr(G, name), int(value)))
    run(a.case, a.launches, a.raster_group, options)
    return 0


if __name__ == "__main__":
    sys.exit(main())
