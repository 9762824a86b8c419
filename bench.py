"""Benchmark of the GB300 dense GEMM: one JSON line on stdout (rank 0).

A step is one GEMM over one batch of synthetic input already resident in HBM:
the square M = N = K = 4096 bf16 problem, A row-major and B column-major (NT),
entries N(0, 1)/sqrt(K), fp32 output, alpha 1, beta 0.  The metric is TFLOP/s
(2*M*N*K per step).  Steps rotate over several input sets whose total exceeds
the L2 cache, so no step starts with its operands in L2.

Also reported, in the same line:
  roofline      the GEMM kernel's achieved TFLOP/s against the measured bf16 peak
  e2e           the same metric through the public API with host buffers, the
                host<->device copies inside the timed region
  cpu_baseline  the CPU oracle (plain fp64 triple loop) on a bounded sample
  skinny        the LM-head GEMM (M = 64, K = 4096, N = 32000) in GB/s
  bf16_out      the same 4096^3 GEMM writing bf16 C (the other output type
                of the square workload) in TFLOP/s
  fp8           the 4096^3 GEMM with 8-bit E4M3 inputs in TFLOP/s
  fp32          the 4096^3 fp32 GEMM from three TF32 products (and with one
                TF32 product) in TFLOP/s of fp32 work
  clocks        SM clocks and throttle reasons sampled during the timed region

`--impl reference` times the CPU oracle instead (the reference arm).
Under torchrun every rank runs its own replica (the GEMM does not exchange
data); value = all ranks' FLOPs / the slowest rank's time.
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BF16 GEMM TFLOPS & % of dense tensor peak at 4096³; GB/s on skinny M=64"
WORKLOAD = "square_4096_bf16_nt_f32"
SIZE = 4096
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--skinny-steps", type=int, default=4000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-skinny", action="store_true")
    ap.add_argument("--bf16-out-steps", type=int, default=20000)
    ap.add_argument("--no-bf16-out", action="store_true")
    ap.add_argument("--fp8-steps", type=int, default=4000)
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--fp32-steps", type=int, default=300)
    ap.add_argument("--no-fp32", action="store_true")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def slowest_over_ranks(ms, device="cpu"):
    """The largest of every rank's timed-region milliseconds (the job takes as
    long as its slowest replica); ms itself when running alone."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank_step, ws, steps, ms_slowest):
    """Whole-job throughput: every rank's units over the slowest rank's time,
    in units per second / 1e12 (TFLOP/s for FLOPs)."""
    return ws * units_per_rank_step * steps / (ms_slowest / 1e3) / 1e12


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# --------------------------------------------------------------- CPU oracle --

def oracle_sample(seconds, problem=None):
    """Time the CPU oracle on whole rows of the 4096^3 workload's C, 16 rows at a
    time, until about `seconds` have passed.  Returns (TFLOP/s, description)."""
    import numpy as np
    import oracle
    from dense_gemm_10_gb300 import inputs
    p = problem or inputs.square_4096_bf16_nt("f32", SIZE)
    a_bits, b_bits = inputs.bits(p.A), inputs.bits(p.B)
    rows_done = 0
    t0 = time.perf_counter()
    block = 16
    while True:
        rows = np.repeat(np.arange(rows_done, rows_done + block) % p.M, p.N)
        cols = np.tile(np.arange(p.N), block)
        oracle.gemm_at(p.transA, p.transB, p.M, p.N, p.K, p.alpha, a_bits, p.lda, b_bits, p.ldb, p.beta, None,
                       p.ldc, oracle.IN_BF16, rows, cols, nthreads=0)
        rows_done += block
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    flops = 2.0 * rows_done * p.N * p.K
    desc = "%d full rows of C (%d of %d outputs, K=%d) of the %s workload, fp64, all cores" % (
        rows_done, rows_done * p.N, p.M * p.N, p.K, WORKLOAD)
    return flops / el / 1e12, desc, el


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from dense_gemm_10_gb300 import inputs
    p = inputs.square_4096_bf16_nt("f32", SIZE)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_sample(0.5, p)
    total_flops_time = []
    for _ in range(args.steps):
        v, desc, el = oracle_sample(per_step, p)
        total_flops_time.append((v, el))
    value = sum(v * el for v, el in total_flops_time) / sum(el for _, el in total_flops_time)
    cores = cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * sum(el for _, el in total_flops_time) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "M": SIZE, "N": SIZE, "K": SIZE, "layout": "NT",
                                        "out": "f32"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            scratch = os.path.join(ROOT, ".scratch")   # inside the repository, git-ignored
            os.makedirs(scratch, exist_ok=True)
            fd, self.path = tempfile.mkstemp(suffix=".csv", dir=scratch)
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- our arm --

def kernel_source_hash():
    """Hash of the sources that decide what the tensor-core kernel does: its
    code, its instantiations and the planner (the copy and conversion kernels
    of aux_kernels.cu and the swizzle probe of probe.cu are left out)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_gemm_10_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in ("aux_kernels.cu", "probe.cu"):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(kernel_key)
    except Exception:
        return None
    if not d or d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from dense_gemm_10_gb300 import build as gbuild
    from dense_gemm_10_gb300 import gemm as G
    from dense_gemm_10_gb300 import inputs, metrics
    gbuild.build()

    h = G.Handle(local)
    p = inputs.square_4096_bf16_nt("f32", SIZE)
    flops = metrics.flops(p.M, p.N, p.K)
    set_bytes = p.A.numel() * 2 + p.B.numel() * 2 + p.M * p.N * 4
    n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)
    A0, B0 = p.A.to(dev), p.B.to(dev)
    sets = [(A0.clone(), B0.clone(), torch.empty(p.M, p.N, dtype=torch.float32, device=dev)) for _ in range(n_sets)]
    del A0, B0
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, G.BF16_F32, sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)

    def step(i):
        A, B, C = sets[i % n_sets]
        st = h.run_raw(p.transA, p.transB, p.M, p.N, p.K, 1.0, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, 0.0,
                       C.data_ptr(), p.N, G.BF16_F32, sptr)
        if st != G.OK:
            raise G.GemmError(st, "gemm_run")

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            step(i)
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("warm-up kernel status %s (0x%x)" % (G.STATUS.get(st), word))

    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    clocks = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.25)
    launches0 = h.launch_count()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(K):
            step(i)
        ev[1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    launches = h.launch_count() - launches0
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("timed kernel status %s (0x%x)" % (G.STATUS.get(st), word))
    ms = slowest_over_ranks(ev[0].elapsed_time(ev[1]), dev)
    value = job_value(flops, ws, K, ms)
    kernel_ms = ms / K   # one kernel launch per step, back to back on one stream

    # End to end through the public API on host buffers (gemm_run_host): every
    # step copies A and B from page-locked host memory, runs the GEMM and copies
    # C back, the copies overlapping the GEMM in row chunks.
    A_h = p.A.pin_memory()
    B_h = p.B.pin_memory()
    C_h = torch.empty(p.M, p.N, dtype=torch.float32).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(3):
            G.gemm_host(A_h, B_h, C_h, False, True, handle=h, stream=stream)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            G.gemm_host(A_h, B_h, C_h, False, True, handle=h, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    e2e = {"value": flops / (e2e_ms / 1e3) / 1e12 * ws, "unit": "TFLOP/s",
           "h2d_bytes_per_step": A_h.numel() * 2 + B_h.numel() * 2, "d2h_bytes_per_step": C_h.numel() * 4,
           "ms_per_step": e2e_ms, "steps": args.e2e_steps}

    pk, pk_src = peaks()
    peak_b = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_s = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = flops / (kernel_ms / 1e3) / 1e12
    cg = 2 if plan.path == G.PATH_TC_2CTA else 1
    kernel_key = "tc_gemm_kernel<%d,%d>:%s" % (plan.bn, cg, WORKLOAD)
    # The timed region runs the kernel back to back for seconds under the power
    # cap, as the sustained cuBLAS figure was measured; a short region compares
    # against the burst figure.
    sustained = wall >= 1.0
    peak = peak_s if sustained else peak_b
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": recorded_traffic(kernel_key),
                "peak_source": "%s %s (cuBLAS bf16; %s)" % (
                    pk_src, "bf16_tflops_sustained" if sustained else "bf16_tflops",
                    "this run is back to back for %.3f s" % wall),
                "frac_of_burst": achieved / peak_b, "frac_of_sustained": achieved / peak_s,
                "frac_of_nominal_2250": achieved / 2250.0,
                "kernel": "tc_gemm_kernel<BN=%d, CTA group %d>" % (plan.bn, cg), "kernel_ms": kernel_ms,
                "algorithmic_flops_per_launch": flops,
                "traffic_note": "DRAM bytes per launch from the committed ncu summary, if taken on these sources"}

    bf16_out = None
    if not args.no_bf16_out:
        bf16_out = run_bf16_out(args, G, h, inputs, metrics, dev, stream, pk, pk_src)
    skinny = None
    if not args.no_skinny:
        skinny = run_skinny(args, G, h, inputs, metrics, dev, stream, pk, pk_src)
    fp8 = None
    if not args.no_fp8:
        fp8 = run_fp8(args, G, h, inputs, metrics, dev, stream, pk, pk_src)
    fp32 = None
    if not args.no_fp32:
        fp32 = run_fp32(args, G, h, inputs, metrics, dev, stream, pk, pk_src)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, el = oracle_sample(args.cpu_seconds, p)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc,
               "seconds": el, "cpu": cpu_model()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": p.M, "N": p.N, "K": p.K, "layout": "NT", "in": "bf16",
                       "out": "f32", "alpha": 1.0, "beta": 0.0, "dist": "N(0,1)/sqrt(K), seeds 0/1",
                       "l2": "%d rotating input sets of %.0f MB (%.0f MB total > %d MB L2)" % (
                           n_sets, set_bytes / 2 ** 20, n_sets * set_bytes / 2 ** 20, L2_BYTES // 2 ** 20),
                       "plan": plan.as_dict(), "parallelism": "replicas" if ws > 1 else "single GPU",
                       "wall_s_timed_region": wall},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "bf16_out": bf16_out, "skinny": skinny, "fp8": fp8, "fp32": fp32,
        }
        print(json.dumps(line), flush=True)
    h.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


def run_bf16_out(args, G, h, inputs, metrics, dev, stream, pk, pk_src):
    """The square 4096^3 bf16 NT GEMM writing bf16 C (RNE), against the measured
    bf16 peak: the sustained figure when the timed region lasts a second or
    more (back to back under the power cap), else the burst figure."""
    import torch
    p = inputs.square_4096_bf16_nt("bf16", SIZE)
    set_bytes = p.A.numel() * 2 + p.B.numel() * 2 + p.M * p.N * 2
    n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)
    sets = [(p.A.to(dev), p.B.to(dev), torch.empty(p.M, p.N, dtype=torch.bfloat16, device=dev))
            for _ in range(n_sets)]
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, G.BF16_BF16)
    sptr = stream.cuda_stream

    def step(i):
        A, B, C = sets[i % n_sets]
        st = h.run_raw(p.transA, p.transB, p.M, p.N, p.K, 1.0, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, 0.0,
                       C.data_ptr(), p.N, G.BF16_BF16, sptr)
        if st != G.OK:
            raise G.GemmError(st, "gemm_run")

    with torch.cuda.stream(stream):
        for i in range(20):
            step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.perf_counter()
        e0.record(stream)
        for i in range(args.bf16_out_steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("bf16-output kernel status %s (0x%x)" % (G.STATUS.get(st), word))
    ms = e0.elapsed_time(e1) / args.bf16_out_steps
    tflops = metrics.flops(p.M, p.N, p.K) / (ms / 1e3) / 1e12
    sustained = wall >= 1.0
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = float(pk.get(key, FALLBACK_PEAKS[key]))
    return {"workload": "square_4096_bf16_nt_bf16", "value": tflops, "unit": "TFLOP/s", "us_per_call": ms * 1e3,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "frac_of_nominal_2250": tflops / 2250.0,
                         "peak_source": "%s %s (this leg is back to back for %.3f s)" % (pk_src, key, wall),
                         "traffic": None},
            "plan": plan.as_dict(), "l2": "%d rotating input sets (%.0f MB total)" % (
                n_sets, n_sets * set_bytes / 2 ** 20)}


def run_fp8(args, G, h, inputs, metrics, dev, stream, pk, pk_src):
    """4096^3 with 8-bit E4M3 inputs (A M x K, B N x K), fp32 C: TFLOP/s against
    the measured bf16 burst peak scaled by the nominal FP8 / bf16 ratio (2)."""
    import torch
    p = inputs.square_4096_fp8_nt("e4m3", "f32", SIZE)
    code = G.fp8_dtype("e4m3", "e4m3", "f32")
    set_bytes = p.A.numel() + p.B.numel() + p.M * p.N * 4
    n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)
    sets = [(p.A.to(dev), p.B.to(dev), torch.empty(p.M, p.N, dtype=torch.float32, device=dev))
            for _ in range(n_sets)]
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, code)
    sptr = stream.cuda_stream

    def step(i):
        A, B, C = sets[i % n_sets]
        st = h.run_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                       0.0, C.data_ptr(), p.N, code, sptr)
        if st != G.OK:
            raise G.GemmError(st, "gemm_run")

    with torch.cuda.stream(stream):
        for i in range(20):
            step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.fp8_steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("fp8 kernel status %s (0x%x)" % (G.STATUS.get(st), word))
    ms = e0.elapsed_time(e1) / args.fp8_steps
    tflops = metrics.flops(p.M, p.N, p.K) / (ms / 1e3) / 1e12
    peak = 2.0 * float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    cg = plan.bm // 128
    return {"workload": "square_4096_e4m3_nt_f32", "value": tflops, "unit": "TFLOP/s", "us_per_call": ms * 1e3,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "frac_of_nominal_4500": tflops / 4500.0,
                         "peak_source": "%s bf16_tflops x 2 (nominal FP8 / bf16 dense ratio 4.5 / 2.25)" % pk_src,
                         "traffic": recorded_traffic("tc_gemm_kernel<%d,%d,e4m3>:square_4096_e4m3_nt_f32"
                                                     % (plan.bn, cg))},
            "plan": plan.as_dict(), "l2": "%d rotating input sets (%.0f MB total)" % (
                n_sets, n_sets * set_bytes / 2 ** 20)}


def run_fp32(args, G, h, inputs, metrics, dev, stream, pk, pk_src):
    """4096^3 with fp32 inputs and C (A M x K, B N x K): the fp32 GEMM from
    three TF32 products per product (two split launches and one GEMM over 3K)
    and, for comparison, one TF32 product per product (one launch).  Values are
    TFLOP/s of fp32 work (2 M N K per call); the roofline counts the TF32
    products the tensor cores execute against the measured bf16 burst peak
    scaled by the nominal TF32 / bf16 dense ratio (1.1 / 2.25)."""
    import torch
    p = inputs.square_4096_f32_nt(SIZE)
    set_bytes = (p.A.numel() + p.B.numel() + p.M * p.N) * 4
    n_sets = max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)
    sets = [(p.A.to(dev), p.B.to(dev), torch.empty(p.M, p.N, dtype=torch.float32, device=dev))
            for _ in range(n_sets)]
    sptr = stream.cuda_stream
    peak = 1.1 / 2.25 * float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    out = {"workload": "square_4096_f32_nt_f32", "unit": "TFLOP/s",
           "l2": "%d rotating input sets (%.0f MB total)" % (n_sets, n_sets * set_bytes / 2 ** 20)}
    for name, code, parts in (("f32_3xtf32", G.F32_F32, 3), ("tf32", G.TF32_F32, 1)):
        def step(i):
            A, B, C = sets[i % n_sets]
            st = h.run_raw(0, 1, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, 0.0,
                           C.data_ptr(), p.N, code, sptr)
            if st != G.OK:
                raise G.GemmError(st, "gemm_run")

        steps = args.fp32_steps * (3 if parts == 1 else 1)
        with torch.cuda.stream(stream):
            for i in range(5):
                step(i)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                step(i)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        st, word = h.status(sptr)
        if st != G.OK:
            raise RuntimeError("fp32 kernel status %s (0x%x)" % (G.STATUS.get(st), word))
        ms = e0.elapsed_time(e1) / steps
        tflops = metrics.flops(p.M, p.N, p.K) / (ms / 1e3) / 1e12
        plan = G.plan(p.M, p.N, p.K, 0, 1, code)
        out[name] = {"value": tflops, "us_per_call": ms * 1e3, "launches_per_call": plan.launches,
                     "roofline": {"bound": "tensor", "achieved": parts * tflops, "peak": peak, "unit": "TFLOP/s",
                                  "frac": parts * tflops / peak,
                                  "peak_source": "%s bf16_tflops x 1.1 / 2.25 (nominal TF32 / bf16 dense ratio)"
                                                 % pk_src,
                                  "achieved_counts": "%d TF32 products per product, whole call" % parts},
                     "plan": plan.as_dict()}
    out["value"] = out["f32_3xtf32"]["value"]
    return out


def run_skinny(args, G, h, inputs, metrics, dev, stream, pk, pk_src):
    """LM-head GEMM, M = 64 x K = 4096 x N = 32000, weights N x K (NT), fp32 out:
    HBM GB/s of algorithmic bytes against the measured copy bandwidth."""
    import torch
    p = inputs.lm_head_64()
    A = p.A.to(dev)
    Bs = [p.B.to(dev) for _ in range(2)]   # 2 x 262 MB of weights > L2
    C = torch.empty(p.M, p.N, dtype=torch.float32, device=dev)
    plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, G.BF16_F32)
    sptr = stream.cuda_stream

    def step(i):
        st = h.run_raw(p.transA, p.transB, p.M, p.N, p.K, 1.0, A.data_ptr(), p.lda, Bs[i % 2].data_ptr(), p.ldb,
                       0.0, C.data_ptr(), p.N, G.BF16_F32, sptr)
        if st != G.OK:
            raise G.GemmError(st, "gemm_run")

    with torch.cuda.stream(stream):
        for i in range(20):
            step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.skinny_steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("skinny kernel status %s (0x%x)" % (G.STATUS.get(st), word))
    ms = e0.elapsed_time(e1) / args.skinny_steps
    nbytes = metrics.algorithmic_bytes(p.M, p.N, p.K, "bf16", "f32")
    gbs = nbytes / (ms / 1e3) / 1e9
    hbm = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"workload": "lm_head_64x32000x4096_nt_f32", "value": gbs, "unit": "GB/s", "us_per_call": ms * 1e3,
            "tflops": metrics.flops(p.M, p.N, p.K) / (ms / 1e3) / 1e12,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "frac_of_8000": gbs / 8000.0, "peak_source": "%s hbm_gbs (copy)" % pk_src,
                         "algorithmic_bytes_per_launch": nbytes,
                         "traffic": recorded_traffic("tc_gemm_kernel<%d,%d>:lm_head_64x32000x4096_nt_f32"
                                                     % (plan.bn, plan.bm // 128))},
            "plan": plan.as_dict(), "l2": "2 weight copies of 262 MB alternate"}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
