"""Benchmark: GEMM TFLOP/s (2MNK/t) of bf16 NN 4096^3 on GB300, through the C ABI.

One step = one GEMM C = A @ B, M = N = K = 4096, bf16 in / bf16 out, fp32
accumulation, alpha = 1, beta = 0, inputs normal(0,1) rounded to bf16 from
seed 1 (the tensorcore gemm.md "Measured perf" 4096^3 shape; the tessl
architecture.md "Column-Panel Grid Swizzling" bf16 4096^3 figure).

Timing: inputs resident in HBM; every step starts from a cold L2 -- by
default each step reads its own copy of the operands (R >= 2 copies in
turn, R x step bytes >= 2.5 x L2); ``--l2 flush`` writes a buffer twice the
L2 size before every step instead; each step's GEMM is bracketed by CUDA
events on the stream it is launched on (nothing else inside the events);
W warm-up steps, then exactly K timed steps, with a barrier and a device
synchronize on both sides.  Under torchrun every rank runs an independent
replica on its own GPU (the path does not shard), the time is the max over
ranks and the value is the total over ranks.

Also reported: the roofline of the dominant kernel against the measured
peak, the end-to-end figure through the host-buffer ABI call (copies
included), SM clocks sampled during the timed region, the CPU oracle timed
on a bounded row band as a baseline, and (last in the line) every other
named workload's time and fraction of its roofline, measured before the
headline's warm-up.  ``--impl reference`` times the CPU oracle (the
reference arm of this benchmark) instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M = N = K = 4096
HEADLINE = "bf16_nn_4096"
SETTLE_MS = 30.0           # default of --settle-ms (see run_ours)
HOST_AHEAD_CYCLES = 400000  # device spin (~0.2 ms) before the timed region's first event
WORKLOAD = "bf16 NN GEMM M=N=K=4096, bf16 out, fp32 accumulate, alpha=1 beta=0, normal(0,1) from seed 1"
METRIC = "GEMM TFLOP/s (2MNK/t) bf16 4096^3 NN"
PAGES_BASELINE = 29.0     # TFLOP/s, bf16 4096^3 NN, Apple M5 Pro (tessl architecture.md, column-panel swizzle)
PAGES_REF = "29.0 TFLOP/s bf16 4096^3 NN on Apple M5 Pro (tessl architecture.md, Column-Panel Grid Swizzling)"
FLOPS = 2.0 * M * N * K


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["bf16_tflops"], d.get("bf16_tflops_sustained"), d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def profile_traffic(workload: str, src_hash: str):
    """DRAM bytes (read + write) per launch of the workload's dominant kernel,
    from the committed ncu figures in profiles/dram_traffic.txt (one line per
    workload: name, kernel-source hash, bytes), if they were taken on the
    current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload:
                    return int(parts[2]) if parts[1] == src_hash else None
    except (OSError, ValueError):
        return None
    return None


def kernel_source_hash() -> str:
    """Hash of the sources of the tensor-core kernel and its launch code."""
    h = hashlib.sha256()
    for name in ("tc_mma.cu", "ptx.cuh", "internal.h", "elem.cuh"):
        with open(os.path.join(ROOT, "matrix_multiply_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The maximum of a per-rank figure over all ranks (each rank is one
    replica on its own GPU; the slowest rank sets the job's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_step: float, steps: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs the same steps (replicas, weak
    scaling), so the job did world * steps * flops in the slowest rank's time."""
    return world * flops_per_step * steps / (max_ms / 1e3) / 1e12


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cpu_baseline(target_s: float = 12.0):
    """The CPU oracle, as it stands, on a band of output rows of the same
    workload, grown until one run takes about target_s seconds."""
    import oracle
    import synthetic
    p = synthetic.bf16_nn_4096()
    lib = oracle.load_library()
    rows = 16
    while True:
        t0 = time.perf_counter()
        oracle.gemm(p, 0, rows, lib=lib)
        dt = time.perf_counter() - t0
        if dt >= 0.8 * target_s or rows >= M:
            break
        rows = int(min(M, max(2 * rows, rows * target_s / max(dt, 1e-3))))
    flops = 2.0 * rows * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(lib),
            "kind": "oracle", "sample": f"rows 0..{rows - 1} of the {M}x{N}x{K} problem ({dt:.1f} s)",
            "seconds": round(dt, 2)}


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores.
    Each step is one oracle call on a bounded sample of the headline problem,
    sized so that all warm-up and timed steps take about 90 s: a band of
    output rows (the oracle's main path, which decodes B once per call),
    or, when even one row per step would not fit, a sample of single output
    elements (its one-dot-product-per-element path)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    import synthetic
    p = synthetic.bf16_nn_4096()
    lib = oracle.load_library()
    rng = np.random.default_rng(0)
    budget = 90.0 / max(args.steps + args.warmup, 1)        # seconds per step

    # calibrate: cost of a call with 8 rows and with 32 rows
    t0 = time.perf_counter(); oracle.gemm(p, 0, 8, lib=lib); c8 = time.perf_counter() - t0
    t0 = time.perf_counter(); oracle.gemm(p, 0, 32, lib=lib); c32 = time.perf_counter() - t0
    per_row = max((c32 - c8) / 24, 1e-6)
    fixed = max(c8 - 8 * per_row, 0.0)
    if fixed + per_row <= budget:
        rows = int(min(M, max(1, (budget - fixed) / per_row)))
        units, flops_per_step = f"rows 0..{rows - 1} of the {M}x{N}x{K} problem per step", 2.0 * rows * N * K
        step = lambda: oracle.gemm(p, 0, rows, lib=lib)         # noqa: E731
    else:
        r, c = rng.integers(0, M, 256), rng.integers(0, N, 256)
        t0 = time.perf_counter(); oracle.gemm_points(p, r, c, lib=lib)
        per_point = (time.perf_counter() - t0) / 256
        points = int(max(16, min(1 << 16, budget / max(per_point, 1e-9))))
        r, c = rng.integers(0, M, points), rng.integers(0, N, points)
        units, flops_per_step = f"{points} sampled output elements of the {M}x{N}x{K} problem per step", 2.0 * K * points
        step = lambda: oracle.gemm_points(p, r, c, lib=lib)     # noqa: E731
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        step()
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    tot = sum(times)
    value = flops_per_step * len(times) / tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(times) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": units},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(lib),
                         "kind": "oracle", "sample": units},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- workloads
# Every named GEMM configuration: (name, problem factory, single GEMM or a
# grouped batch).  The headline is bf16_nn_4096; the others are timed for
# the per-workload roofline summary and can be run alone with --workload.

def workload_registry():
    import synthetic
    reg = {
        "bf16_nn_4096": lambda: [synthetic.bf16_nn_4096()],
        "fp32_nn_256": lambda: [synthetic.fp32_nn_256()],
        "bf16_tn_4096x4096x8192": lambda: [synthetic.bf16_tn_nt_4096x8192("TN")],
        "bf16_nt_4096x4096x8192": lambda: [synthetic.bf16_tn_nt_4096x8192("NT")],
        "bf16_tn_splitk_256x256x16384": lambda: [synthetic.bf16_tn_splitk_256x16384()],
        "fp16_nn_8192x384x4096": lambda: [synthetic.fp16_nn_narrow_8192x384x4096()],
        "fp16_ragged_64": lambda: synthetic.fp16_ragged(),
    }
    for n in synthetic.SQUARE_SIZES:
        reg[f"fp16_nn_square_{n}"] = (lambda n=n: [synthetic.fp16_nn_square(n)])

    # the fused bias + GELU epilogue (tessl architecture.md, "Fused Epilogue")
    def epilogue(shape):
        p, bias = synthetic.bf16_epilogue(*shape)
        p.bias, p.activation = bias, "gelu_tanh"
        return [p]
    for (m, n, k) in synthetic.EPILOGUE_SHAPES:
        tag = f"{m}" if m == n == k else f"{m}x{n}x{k}"
        reg[f"bf16_bias_gelu_{tag}"] = (lambda s=(m, n, k): epilogue(s))
    # the same operands without the epilogue: what the fused bias + GELU
    # costs over the plain GEMM
    for (m, n, k) in synthetic.EPILOGUE_SHAPES:
        tag = f"{m}" if m == n == k else f"{m}x{n}x{k}"
        reg[f"bf16_plain_{tag}"] = (lambda s=(m, n, k): [synthetic.bf16_epilogue(*s)[0]])
    # the small-M decode shape (the skinny-product kernel)
    for (m, n, k) in synthetic.DECODE_SHAPES:
        reg[f"f16_decode_m{m}_{n}x{k}"] = (lambda s=(m, n, k): [synthetic.f16_decode(*s)])

    # the same decode shapes over int8 weights with per-row scales (Foundry
    # metal.md, "Custom Compute Kernels": fm_sgemm_q8 / fm_matvec_q8)
    def q8(shape):
        p, scale = synthetic.q8_decode(*shape)
        p.q8_scale = scale
        return [p]
    for (m, n, k) in synthetic.DECODE_SHAPES:
        reg[f"q8w_decode_m{m}_{n}x{k}"] = (lambda s=(m, n, k): q8(s))

    # fp32 at 4096^3: the exact path and the relaxed (bf16-split) path
    def relaxed():
        p = synthetic.fp32_nn_4096()
        p.precision = "relaxed"
        return [p]
    reg["fp32_nn_4096"] = lambda: [synthetic.fp32_nn_4096()]
    reg["fp32_relaxed_nn_4096"] = relaxed

    # int8 x int8 -> per-column dequantised fp32 (exact accumulation)
    def i8():
        p, scale = synthetic.i8_dequant_4096()
        p.col_scale = scale
        return [p]
    reg["i8_dequant_nn_4096"] = i8
    return reg


def ffma_peak_tflops(sms: int, mhz: float) -> float:
    """fp32 FFMA peak: SMs x 128 fp32 lanes x 2 flop x SM clock."""
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def roofline(probs, seconds, sms):
    """Algorithmic flops/bytes of a step against the measured peaks: the
    bound is whichever of compute and HBM traffic takes longer."""
    burst, _sustained, hbm, src = peaks()
    es = {"f16": 2, "bf16": 2, "f32": 4, "i8": 1}
    flops = sum(2.0 * p.M * p.N * p.K for p in probs)
    # each operand at its own element size (the int8-weight product mixes
    # half-precision activations with one-byte weights), plus the per-column
    # bias or scale vectors
    nbytes = sum(p.M * p.K * p.A.element_size() + p.K * p.N * p.B.element_size() +
                 p.M * p.N * es[p.c_dtype] * (2 if p.beta != 0 else 1) +
                 (p.N * es[p.c_dtype] if getattr(p, "bias", None) is not None else 0) +
                 (p.N * 4 if getattr(p, "q8_scale", None) is not None else 0) for p in probs)
    # fp32 operands: the exact path runs on the FFMA lanes; the relaxed path
    # on the bf16 tensor cores at three bf16 products per fp32 product
    relaxed = getattr(probs[0], "precision", None) == "relaxed"
    fp32 = probs[0].ab_dtype == "f32" and not relaxed
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = json.load(f).get("sm_max_mhz", 2070.0)
    except Exception:
        mhz = 2070.0
    peak_c = ffma_peak_tflops(sms, mhz) if fp32 else burst / 3.0 if relaxed else burst
    t_c = flops / (peak_c * 1e12)
    t_m = nbytes / (hbm * 1e9)
    if t_c >= t_m:
        bound, achieved, peak, unit = ("alu" if fp32 else "tensor"), flops / seconds / 1e12, peak_c, "TFLOP/s"
    else:
        bound, achieved, peak, unit = "hbm", nbytes / seconds / 1e9, hbm, "GB/s"
    what = ("FFMA lanes x clock (derived)" if fp32 else "HBM copy" if bound == "hbm" else
            "bf16 dense burst / 3 (three bf16 products per fp32 product)" if relaxed else "bf16 dense burst")
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "flops_per_step": flops, "bytes_per_step": nbytes, "peak_source": f"{src}: {what}"}


def torch_int8():
    import torch
    return torch.int8


def step_bytes(probs) -> int:
    """Bytes of the operands one step reads or writes (A, B, C, vectors)."""
    n = 0
    for p in probs:
        n += p.A.numel() * p.A.element_size() + p.B.numel() * p.B.element_size() + p.C.numel() * p.C.element_size()
    return n


class Cold:
    """Cold L2 before every timed step, one of two ways:
    rotate -- every step reads its own copy of the operands: R >= 2 copies
              with R x (bytes of a step) >= 2.5 x L2, used in turn, so a
              step's operands were evicted by the R - 1 steps before it (the
              rules' "inputs larger than L2"; nothing extra runs between
              steps);
    flush  -- one copy, and a write of >= 2 x L2 before every step (outside
              the timed events); the flush leaves the L2 full of dirty lines,
              which a read-bound step then pays to write back."""

    def __init__(self, torch, mode: str, l2_bytes: int):
        self.torch, self.mode, self.l2 = torch, mode, l2_bytes
        self.buf = (torch.empty(max(2 * l2_bytes, 256 << 20) // 4, dtype=torch.float32, device="cuda")
                    if mode == "flush" else None)

    def copies(self, probs) -> int:
        if self.mode != "rotate":
            return 1
        nbytes = max(step_bytes(probs), 1)
        return int(min(4096, max(2, -(-int(2.5 * self.l2) // nbytes))))

    def before_step(self):
        if self.buf is not None:
            self.buf.zero_()

    def describe(self) -> str:
        if self.mode == "flush":
            return "flushed before every step (write of >= 2x L2); flush outside the timed events"
        return ("cold L2: each step reads its own copy of the operands, R >= 2 copies in turn with "
                "R x step bytes >= 2.5x L2 (no flush kernel)")


class Runner:
    """Device-resident operands of one workload (``copies`` copies, used in
    turn) and its launch."""

    def __init__(self, tg, ctx, stream, probs, copies: int = 1):
        self.tg, self.ctx, self.stream, self.probs = tg, ctx, stream, probs
        self.copies, self.k = copies, 0
        self.As = [[p.A.cuda() for p in probs] for _ in range(copies)]
        self.Bs = [[p.B.cuda() for p in probs] for _ in range(copies)]
        self.Cs = [[p.C.cuda() for p in probs] for _ in range(copies)]
        self.d = [tg.make_desc(p.M, p.N, p.K, p.ab_dtype, p.c_dtype, transpose_a=p.transpose_a,
                               transpose_b=p.transpose_b, alpha=p.alpha, beta=p.beta,
                               b_dtype="i8" if p.B.dtype == torch_int8() else None) for p in probs]
        # a group's arguments are marshalled once per copy; each step is one C call
        self.groups = ([tg.GroupedGemm(self.d, a, b, c) for a, b, c in zip(self.As, self.Bs, self.Cs)]
                       if len(probs) > 1 else None)
        # the fused-epilogue workloads carry a bias and an activation
        p0 = probs[0]
        self.activation = getattr(p0, "activation", None)
        self.bias = p0.bias.cuda() if getattr(p0, "bias", None) is not None else None
        self.relaxed = getattr(p0, "precision", None) == "relaxed"
        self.col_scale = p0.col_scale.cuda() if getattr(p0, "col_scale", None) is not None else None
        self.q8_scale = p0.q8_scale.cuda() if getattr(p0, "q8_scale", None) is not None else None
        # a single product's arguments are marshalled once per copy as well
        self.calls = ([tg.PreparedGemm(ctx, self.d[0], a[0], b[0], c[0], stream, bias=self.bias,
                                       activation=self.activation, relaxed=self.relaxed, col_scale=self.col_scale,
                                       q8_scale=self.q8_scale) for a, b, c in zip(self.As, self.Bs, self.Cs)]
                      if len(probs) == 1 else None)

    def step(self):
        """One step: the next copy's product (or group), one C call."""
        self.k = (self.k + 1) % self.copies
        if self.calls:
            self.calls[self.k].enqueue()
        else:
            self.groups[self.k].enqueue(self.ctx, self.stream)


def timed_loop(torch, runner, tstream, cold, steps, per_step):
    """Device time (ms) of `steps` steps issued back to back on the launching
    stream, as a list with one entry per step.  per_step: an event pair
    around every step (each step then also pays the gap between kernels
    that an event in the stream imposes); else one pair around all of them
    (the throughput of back-to-back steps), each entry the mean."""
    torch.cuda._sleep(HOST_AHEAD_CYCLES)      # the host queues ahead of the first event (see run_ours)
    if per_step:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            cold.before_step()
            starts[i].record(tstream)
            runner.step()
            ends[i].record(tstream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(starts, ends)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(tstream)
    for i in range(steps):
        cold.before_step()
        runner.step()
    end.record(tstream)
    torch.cuda.synchronize()
    return [start.elapsed_time(end) / steps] * steps


def time_steps(torch, runner, tstream, cold, steps, warmup, per_step=False):
    for _ in range(warmup):
        cold.before_step()
        runner.step()
    torch.cuda.synchronize()
    return timed_loop(torch, runner, tstream, cold, steps, per_step)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import matrix_multiply_gb300 as tg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    ctx = tg.Context(local)
    tstream = torch.cuda.current_stream()
    stream = tg.Stream(ctx, torch_stream=tstream)
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count
    cold = Cold(torch, args.l2, props.L2_cache_size)
    reg = workload_registry()
    name = args.workload
    probs = reg[name]()
    runner = Runner(tg, ctx, stream, probs, cold.copies(probs))
    n_copies = runner.copies
    flops = sum(2.0 * p.M * p.N * p.K for p in probs)

    # Untimed: the step repeated for --settle-ms of wall time, so that the
    # SM clock has left its idle state, then the W warm-up steps.  The
    # headline is timed before the summary of the other workloads, so that
    # seconds of other work do not leave the GPU at its power cap: this is
    # the kernel timed alone, against the burst peak.
    t_settle = time.perf_counter()
    while time.perf_counter() - t_settle < args.settle_ms / 1e3:
        for _ in range(8):
            cold.before_step()
            runner.step()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        cold.before_step()
        runner.step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()

    launches0 = ctx.launch_count
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        # (timed_loop first queues a short device-side spin ahead of the
        # first event, so that the host has queued the first steps by the
        # time the GPU reaches it: without it the first step, launched onto
        # an idle GPU, also times the host's launch latency, ~20 us)
        ms = timed_loop(torch, runner, tstream, cold, args.steps, args.timing == "step")
        t_wall = time.perf_counter() - t_wall
    barrier()
    torch.cuda.synchronize()
    stream.sync()
    launches = ctx.launch_count - launches0
    kernel = ctx.last_kernel
    total_ms = max_over_ranks(sum(ms), world)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, flops, args.steps, total_ms)

    # end to end through the host-buffer ABI call (copies inside the timed region)
    e2e = None
    if (len(probs) == 1 and runner.activation is None and not runner.relaxed and runner.col_scale is None
            and runner.q8_scale is None):
        # (no host-buffer call carries the epilogue or the relaxed mode)
        p = probs[0]
        Ah, Bh, Ch = p.A.pin_memory(), p.B.pin_memory(), p.C.clone().pin_memory()
        d = runner.d[0]
        for _ in range(2):
            tg.tc_gemm_host(ctx, d, Ah, Bh, Ch)
        e2e_steps = max(5, min(args.steps, 30))
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            tg.tc_gemm_host(ctx, d, Ah, Bh, Ch)
        e2e_ms = max_over_ranks((time.perf_counter() - t0) / e2e_steps * 1e3, world)
        es = {"f16": 2, "bf16": 2, "f32": 4}
        e2e = {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": (p.M * p.K + p.K * p.N) * es[p.ab_dtype] +
               (p.M * p.N * es[p.c_dtype] if p.beta != 0 else 0),
               "d2h_bytes_per_step": p.M * p.N * es[p.c_dtype], "ms_per_step": e2e_ms,
               "call": "tc_gemm_host (pinned host A, B, C)"}

    if world > 1:
        dist.barrier()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    # every other named workload (cold L2 per step, about a third of a
    # second each), after the headline's timed region
    work = None
    if args.summary and name == HEADLINE and world == 1:
        del runner
        torch.cuda.empty_cache()
        work = summary(torch, tg, ctx, stream, tstream, cold, reg, sms, args.timing == "step")

    rl = roofline(probs, statistics.mean(ms) / 1e3, sms)
    rl["traffic"] = profile_traffic(name, kernel_source_hash())
    p0 = probs[0]
    line = {
        "metric": METRIC if name == HEADLINE else f"GEMM TFLOP/s (2MNK/t) {name}",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": value / (world * PAGES_BASELINE) if name == HEADLINE else None,
        "dtype": p0.ab_dtype, "data": "synthetic",
        "config": {"workload": WORKLOAD if name == HEADLINE else name, "problems": len(probs),
                   "M": p0.M, "N": p0.N, "K": p0.K, "layout": p0.layout, "global_batch": len(probs),
                   "parallelism": f"replicas{world}" if world > 1 else "single", "variant": kernel,
                   "l2": cold.describe(), "copies": n_copies, "settle_ms": args.settle_ms,
                   "timing": ("one CUDA event pair around each step" if args.timing == "step" else
                              "one CUDA event pair around the back-to-back timed steps")},
        "roofline": rl,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(t_wall, 3),
    }
    if name == HEADLINE:
        line["config"]["vs_baseline_ref"] = PAGES_REF
    if not args.no_cpu_baseline and name == HEADLINE:
        line["cpu_baseline"] = cpu_baseline()
    if work is not None:
        # the full per-workload record (variant names, achieved rates) on
        # stderr; the line itself ends with the compact map
        # {workload: [us per step, fraction of roofline, bound]}, last so
        # that a reader keeping only the end of the line still has it
        print(json.dumps({"workloads_detail": work}), file=sys.stderr, flush=True)
        line["workloads_key"] = "[us_per_step, roofline_frac, bound]"
        line["workloads"] = {k: [round(v["ms"] * 1e3, 1), round(v["frac"], 3), v["bound"]]
                             for k, v in work.items()}
    print(json.dumps(line, separators=(",", ":")), flush=True)
    stream.close()
    ctx.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def summary(torch, tg, ctx, stream, tstream, cold, reg, sms, per_step=False):
    """Every other named workload: TFLOP/s and roofline fraction, each timed
    for about a third of a second of device time (cold L2 per step)."""
    out = {}
    for name, factory in reg.items():
        if name == HEADLINE:
            continue
        probs = factory()
        runner = Runner(tg, ctx, stream, probs, cold.copies(probs))
        probe = time_steps(torch, runner, tstream, cold, 3, 2)
        steps = int(max(10, min(2000, 0.3e3 / max(statistics.mean(probe), 1e-3))))
        ms = time_steps(torch, runner, tstream, cold, steps, 3, per_step)
        t = statistics.mean(ms) / 1e3
        flops = sum(2.0 * p.M * p.N * p.K for p in probs)
        rl = roofline(probs, t, sms)
        out[name] = {"tflops": flops / t / 1e12, "ms": t * 1e3, "steps": steps,
                     "bound": rl["bound"], "achieved": rl["achieved"], "unit": rl["unit"],
                     "frac": rl["frac"], "variant": ctx.last_kernel}
        del runner
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=HEADLINE,
                    help="which named workload to time (default: the headline bf16 NN 4096^3)")
    ap.add_argument("--no-summary", dest="summary", action="store_false",
                    help="skip the per-workload roofline summary of the other workloads")
    ap.add_argument("--settle-ms", type=float, default=SETTLE_MS,
                    help="untimed repetitions of the step (wall ms) before the warm-up steps; 0 for "
                         "profiler runs that list every launch")
    ap.add_argument("--timing", choices=["stream", "step"], default="stream",
                    help="one event pair around the back-to-back timed steps (stream), or one per step")
    ap.add_argument("--l2", choices=["rotate", "flush"], default="rotate",
                    help="how every timed step starts from a cold L2 (see Cold)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
