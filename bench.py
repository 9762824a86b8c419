"""Benchmark of the GB300 dense GEMM: one JSON line on stdout (rank 0).

A step is one GEMM over one batch of synthetic input already resident in HBM:
the square M = N = K = 4096 bf16 problem, A row-major and B column-major (NT),
entries N(0, 1)/sqrt(K), fp32 output, alpha 1, beta 0.  The metric is TFLOP/s
(2*M*N*K per step).  Steps rotate over several input sets whose total exceeds
the L2 cache, so no step starts with its operands in L2.

Also reported, in the same line (kept under 2 KB; --detail FILE writes every
leg's plan, timings and notes to a file):
  roofline      the GEMM kernel's achieved TFLOP/s against the measured bf16 peak
  e2e           the same metric through the public API with host buffers, the
                host<->device copies inside the timed region
  cpu_baseline  the CPU oracle (plain fp64 triple loop) on a bounded sample
  clocks        SM clocks and throttle reasons sampled during the timed region
  legs          the other workloads, each [value, fraction of its roofline]:
                c1 256^3 (device and host microseconds per call), c2 the
                4096^3 workload with bf16 C, c3 4096^3 fp16 alpha 1.5 beta 0.5
                in four layouts, c4 the LLM projections (QKV, FFN-up,
                FFN-down, NN) and the ragged 4095 x 4097 x 1000, c5 the LM head
                64 x 32000 x 4096 in GB/s, and the FP8 and fp32 GEMMs at 4096^3

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
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tiny-steps", type=int, default=2000)
    ap.add_argument("--bf16-out-steps", type=int, default=20000)
    ap.add_argument("--llm-steps", type=int, default=200)
    ap.add_argument("--skinny-steps", type=int, default=4000)
    ap.add_argument("--fp8-steps", type=int, default=4000)
    ap.add_argument("--fp32-steps", type=int, default=300)
    ap.add_argument("--skip", default="", help="comma-separated legs to leave out: " + ",".join(
        n for n, _ in LEGS))
    ap.add_argument("--detail", default="", help="write per-leg plans and timings to this JSON file")
    a = ap.parse_args()
    a.skip = set(x for x in a.skip.split(",") if x)
    return a


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
    desc = "%d of %d rows of C, fp64, all cores" % (rows_done, p.M)
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


def _sig(x, digits=4):
    """x rounded to `digits` significant figures (keeps the JSON line short)."""
    if x is None or x == 0 or not math.isfinite(x):
        return x
    return round(x, digits - 1 - int(math.floor(math.log10(abs(x)))))


def n_rotating_sets(set_bytes):
    """Input sets to rotate over so that every step's operands and C miss L2:
    together at least twice the L2 size, and at least two sets unless one set
    alone is four times the L2 size."""
    if set_bytes > 4 * L2_BYTES:
        return 1
    return max(2, math.ceil(2 * L2_BYTES / set_bytes) + 1)


def time_steps(step, n, stream, dev, warm=10):
    """Average device milliseconds of `step(i)` over n back-to-back calls on
    `stream` (CUDA events on that stream, synchronised on both sides), and the
    wall seconds of the timed region."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warm):
            step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        wall0 = time.perf_counter()
        e0.record(stream)
        for i in range(n):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / n, time.perf_counter() - wall0


def device_operands(p, dev):
    """Device copies of a problem's A and B, and its C: the initial C0 when
    beta != 0 (read and updated in place by every step), else an empty buffer
    of C's type and leading dimension."""
    import torch
    out = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[p.out_dtype]
    C = p.C0.to(dev) if p.C0 is not None else torch.empty(p.M, p.ldc, dtype=out, device=dev)
    return p.A.to(dev), p.B.to(dev), C


class GemmLeg:
    """One workload timed through gemm_run on device buffers: rotating input
    sets larger than L2, back-to-back calls, status checked afterwards."""

    def __init__(self, G, h, p, code, dev, stream):
        self.G, self.h, self.p, self.code, self.stream = G, h, p, code, stream
        A, B, C = device_operands(p, dev)
        set_bytes = A.numel() * A.element_size() + B.numel() * B.element_size() + C.numel() * C.element_size()
        self.n_sets = n_rotating_sets(set_bytes)
        self.sets = [(A, B, C)] + [(A.clone(), B.clone(), C.clone()) for _ in range(self.n_sets - 1)]
        self.set_mb = set_bytes / 2 ** 20
        self.sptr = stream.cuda_stream
        self.plan = G.plan(p.M, p.N, p.K, p.transA, p.transB, code, lda=p.lda, ldb=p.ldb, ldc=p.ldc,
                           beta=p.beta, handle=h)

    def step(self, i):
        p = self.p
        A, B, C = self.sets[i % self.n_sets]
        st = self.h.run_raw(p.transA, p.transB, p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(),
                            p.ldb, p.beta, C.data_ptr(), p.ldc, self.code, self.sptr)
        if st != self.G.OK:
            raise self.G.GemmError(st, "gemm_run " + p.name)

    def time(self, n, dev, warm=10):
        ms, wall = time_steps(self.step, n, self.stream, dev, warm)
        st, word = self.h.status(self.sptr)
        if st != self.G.OK:
            raise RuntimeError("%s: kernel status %s (0x%x)" % (self.p.name, self.G.STATUS.get(st), word))
        return ms, wall

    def free(self):
        self.sets = None


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
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    p = inputs.square_4096_bf16_nt("f32", SIZE)
    flops = metrics.flops(p.M, p.N, p.K)
    main = GemmLeg(G, h, p, G.BF16_F32, dev, stream)
    plan = main.plan

    # The clock sampler starts first and has its first samples taken before the
    # warm-up, so that the warm-up steps run right before the timed ones (an
    # idle gap there would let the timed region start on an idle GPU).
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            main.step(i)
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("warm-up kernel status %s (0x%x)" % (G.STATUS.get(st), word))

    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = h.launch_count()
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(K):
            main.step(i)
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
    main_l2 = "%d rotating sets of %.0f MB" % (main.n_sets, main.set_mb)
    main.free()

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
    e2e = {"value": _sig(flops / (e2e_ms / 1e3) / 1e12 * ws), "unit": "TFLOP/s",
           "h2d_bytes_per_step": A_h.numel() * 2 + B_h.numel() * 2, "d2h_bytes_per_step": C_h.numel() * 4}
    del A_h, B_h, C_h

    pk, pk_src = peaks()
    peak_b = float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_s = float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = flops / (kernel_ms / 1e3) / 1e12
    cg = 2 if plan.path == G.PATH_TC_2CTA else 1
    # The timed region runs the kernel back to back for seconds under the power
    # cap, as the sustained cuBLAS figure was measured; a short region compares
    # against the burst figure.
    sustained = wall >= 1.0
    peak = peak_s if sustained else peak_b
    roofline = {"bound": "tensor", "achieved": _sig(achieved), "peak": peak, "unit": "TFLOP/s",
                "frac": _sig(achieved / peak),
                "traffic": recorded_traffic("tc_gemm_kernel<%d,%d>:%s" % (plan.bn, cg, WORKLOAD)),
                "peak_key": "%s %s" % (pk_src, "bf16_tflops_sustained" if sustained else "bf16_tflops"),
                "frac_nominal_2250": _sig(achieved / 2250.0)}
    detail = {"main": {"plan": plan.as_dict(), "kernel_ms": kernel_ms, "wall_s": wall, "l2": main_l2,
                       "peak_source": "%s (cuBLAS bf16); timed region back to back for %.3f s" % (
                           roofline["peak_key"], wall)},
              "e2e": {"ms_per_step": e2e_ms, "steps": args.e2e_steps}}

    legs = {}
    ctx = dict(args=args, G=G, h=h, inputs=inputs, metrics=metrics, dev=dev, stream=stream, pk=pk,
               peak_b=peak_b, peak_s=peak_s, legs=legs, detail=detail)
    for name, fn in LEGS:
        if name not in args.skip:
            fn(ctx)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, el = oracle_sample(args.cpu_seconds, p)
        cpu = {"value": _sig(v), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc}
        detail["cpu_baseline"] = {"seconds": el, "cpu": cpu_model()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": _sig(value, 5), "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
            "warmup": args.warmup, "ms_per_step": _sig(ms / K, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": p.M, "N": p.N, "K": p.K, "layout": "NT", "out": "f32",
                       "l2": main_l2 + " > L2", "parallelism": "replicas" if ws > 1 else "1 GPU"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "legs": legs,
            "legs_key": LEGS_KEY,
        }
        if args.detail:
            detail["clocks"] = clk
            with open(args.detail, "w") as f:
                json.dump(detail, f, indent=1)
        print(json.dumps(line, separators=(",", ":"), ensure_ascii=False), flush=True)
    h.close()
    if ws > 1:
        dist.destroy_process_group()
    return 0


LEGS_KEY = ("[v, frac]: _tf TFLOP/s vs bf16 peak (fp8 x2; fp32: 3 TF32 products vs x1.1/2.25), "
            "_gbs GB/s vs copy; c1: [device, host] us per call")


def _tensor_leg(ctx, key, p, code, steps, peak_scale=1.0, work_scale=1.0):
    """Time one GEMM workload; record [TFLOP/s, frac of the bf16 peak x peak_scale]."""
    leg = GemmLeg(ctx["G"], ctx["h"], p, code, ctx["dev"], ctx["stream"])
    ms, wall = leg.time(steps, ctx["dev"])
    tflops = ctx["metrics"].flops(p.M, p.N, p.K) / (ms / 1e3) / 1e12
    sustained = wall >= 1.0
    peak = (ctx["peak_s"] if sustained else ctx["peak_b"]) * peak_scale
    ctx["legs"][key] = [_sig(tflops), _sig(work_scale * tflops / peak, 3)]
    ctx["detail"][key] = {"workload": p.name, "us_per_call": ms * 1e3, "tflops": tflops, "peak": peak,
                          "sustained": sustained, "wall_s": wall, "plan": leg.plan.as_dict(),
                          "l2": "%d rotating sets of %.0f MB" % (leg.n_sets, leg.set_mb)}
    leg.free()
    return ms


def leg_tiny(ctx):
    """256^3 NN bf16 -> fp32 (latency-bound): device microseconds per call over
    back-to-back calls, and host microseconds per gemm_run call."""
    G, h, stream, dev = ctx["G"], ctx["h"], ctx["stream"], ctx["dev"]
    p = ctx["inputs"].tiny_256()
    leg = GemmLeg(G, h, p, G.BF16_F32, dev, stream)
    ms, _ = leg.time(ctx["args"].tiny_steps, dev)
    # host time of the call alone (the launch is asynchronous), repeated on
    # one set of buffers as a decode loop calls it: plan and tensor maps come
    # from the handle's caches
    import torch
    n = ctx["args"].tiny_steps
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for _ in range(n):
            leg.step(0)
        host_us = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize(dev)
    ctx["legs"]["c1_256_us"] = [_sig(ms * 1e3, 3), _sig(host_us, 3)]
    ctx["detail"]["c1_256_us"] = {"workload": p.name, "device_us_per_call": ms * 1e3, "host_us_per_call": host_us,
                                  "plan": leg.plan.as_dict(),
                                  "l2": "%d rotating sets of %.2f MB" % (leg.n_sets, leg.set_mb)}
    leg.free()


def leg_bf16_out(ctx):
    """The 4096^3 bf16 NT workload with bf16 C (its other output type)."""
    _tensor_leg(ctx, "c2_bf16c_tf", ctx["inputs"].square_4096_bf16_nt("bf16", SIZE), ctx["G"].BF16_BF16,
                ctx["args"].bf16_out_steps)


def leg_blend(ctx):
    """4096^3 fp16, alpha 1.5, beta 0.5 (C read and written), four layouts."""
    for ta, tb in ((0, 0), (0, 1), (1, 0), (1, 1)):
        lay = ("t" if ta else "n") + ("t" if tb else "n")
        _tensor_leg(ctx, "c3_%s_tf" % lay, ctx["inputs"].square_4096_f16_blend(ta, tb, SIZE), ctx["G"].F16_F32,
                    ctx["args"].llm_steps)


def leg_llm(ctx):
    """LLM projections NN (weights K x N) and the ragged 4095 x 4097 x 1000 NN."""
    inp = ctx["inputs"]
    for name, key in (("qkv_proj", "c4_qkv_tf"), ("ffn_up", "c4_up_tf"), ("ffn_down", "c4_down_tf")):
        _tensor_leg(ctx, key, inp.llm_projection(name, 0), ctx["G"].BF16_F32, ctx["args"].llm_steps)
    _tensor_leg(ctx, "c4_ragged_tf", inp.ragged_4095_4097_1000(), ctx["G"].BF16_F32, ctx["args"].llm_steps)


def leg_skinny(ctx):
    """LM head M = 64 x K = 4096 x N = 32000, weights N x K (NT), fp32 C: GB/s of
    algorithmic bytes against the measured copy bandwidth."""
    G, metrics = ctx["G"], ctx["metrics"]
    p = ctx["inputs"].lm_head_64()
    leg = GemmLeg(G, ctx["h"], p, G.BF16_F32, ctx["dev"], ctx["stream"])
    ms, wall = leg.time(ctx["args"].skinny_steps, ctx["dev"], warm=20)
    nbytes = metrics.algorithmic_bytes(p.M, p.N, p.K, "bf16", "f32")
    gbs = nbytes / (ms / 1e3) / 1e9
    hbm = float(ctx["pk"].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ctx["legs"]["c5_lmhead_gbs"] = [_sig(gbs), _sig(gbs / hbm, 3)]
    ctx["detail"]["c5_lmhead_gbs"] = {
        "workload": p.name, "us_per_call": ms * 1e3, "gbs": gbs, "frac_of_8000": gbs / 8000.0,
        "algorithmic_bytes_per_launch": nbytes, "plan": leg.plan.as_dict(),
        "traffic": recorded_traffic("tc_gemm_kernel<%d,%d>:lm_head_64x32000x4096_nt_f32"
                                    % (leg.plan.bn, leg.plan.bm // 128)),
        "l2": "%d rotating sets of %.0f MB" % (leg.n_sets, leg.set_mb)}
    leg.free()


def leg_fp8(ctx):
    """4096^3 E4M3 NT -> fp32 against 2 x the measured bf16 burst peak."""
    G = ctx["G"]
    p = ctx["inputs"].square_4096_fp8_nt("e4m3", "f32", SIZE)
    _tensor_leg(ctx, "fp8_tf", p, G.fp8_dtype("e4m3", "e4m3", "f32"), ctx["args"].fp8_steps, peak_scale=2.0)


def leg_fp32(ctx):
    """4096^3 fp32 NT -> fp32 from three TF32 products: TFLOP/s of fp32 work; the
    frac counts the three TF32 products against bf16 x 1.1 / 2.25."""
    G = ctx["G"]
    p = ctx["inputs"].square_4096_f32_nt(SIZE)
    _tensor_leg(ctx, "fp32_tf", p, G.F32_F32, ctx["args"].fp32_steps, peak_scale=1.1 / 2.25, work_scale=3.0)


def leg_nvfp4_lm_head(ctx):
    """The LM head with NVFP4 operands (E2M1 codes, an unsigned E4M3 scale per 16
    values), bf16 C: GB/s of algorithmic bytes (codes, scale codes, C) against
    the measured copy bandwidth.  The weights stay in their codes; the GEMM
    converts them as they arrive."""
    import torch
    G, dev = ctx["G"], ctx["dev"]
    inp = ctx["inputs"]
    p = inp.make_block_scaled_problem("lm_head_64x32000x4096_nvfp4", 64, 32000, 4096, "nvfp4", "bf16", seed=0,
                                      alpha=1.0 / 64)
    ops = [p.A.to(dev), p.SFA.to(dev), p.B.to(dev), p.SFB.to(dev)]
    set_bytes = sum(t.numel() for t in ops) + p.M * p.ldc * 2
    n = n_rotating_sets(set_bytes)
    sets = [ops] + [[t.clone() for t in ops] for _ in range(n - 1)]
    C = torch.empty(p.M, p.ldc, dtype=torch.bfloat16, device=dev)
    h, sptr = ctx["h"], ctx["stream"].cuda_stream

    def step(i):
        A, SA, B, SB = sets[i % n]
        st = h.run_block_scaled_raw(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, SA.data_ptr(), p.ld_sfa,
                                    B.data_ptr(), p.ldb, SB.data_ptr(), p.ld_sfb, 0.0, C.data_ptr(), p.ldc,
                                    G.NVFP4_BF16, sptr)
        if st != G.OK:
            raise G.GemmError(st, "gemm_run_block_scaled")

    ms, wall = time_steps(step, ctx["args"].skinny_steps, ctx["stream"], dev, warm=20)
    st, word = h.status(sptr)
    if st != G.OK:
        raise RuntimeError("nvfp4 kernel status %s (0x%x)" % (G.STATUS.get(st), word))
    nbytes = sum(t.numel() for t in ops) + p.M * p.N * 2
    gbs = nbytes / (ms / 1e3) / 1e9
    hbm = float(ctx["pk"].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    plan = G.plan_block_scaled(p.M, p.N, p.K, G.NVFP4_BF16, lda=p.lda, ldb=p.ldb, ld_sfa=p.ld_sfa,
                               ld_sfb=p.ld_sfb, ldc=p.ldc, handle=h)
    ctx["legs"]["f1_nvfp4_lm_gbs"] = [_sig(gbs), _sig(gbs / hbm, 3)]
    ctx["detail"]["f1_nvfp4_lm_gbs"] = {"workload": p.name, "us_per_call": ms * 1e3, "gbs": gbs,
                                        "algorithmic_bytes_per_call": nbytes, "plan": plan.as_dict(),
                                        "l2": "%d rotating sets of %.0f MB" % (n, set_bytes / 2 ** 20)}


LEGS = [("tiny", leg_tiny), ("bf16_out", leg_bf16_out), ("blend", leg_blend), ("llm", leg_llm),
        ("skinny", leg_skinny), ("nvfp4", leg_nvfp4_lm_head), ("fp8", leg_fp8), ("fp32", leg_fp32)]


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
