"""Benchmark of the block-scaled FP4 GEMM on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--results PATH]

A step is one pass of the whole hot path over one problem: one call of
fp4_gemm_nvfp4 / fp4_gemm_mxfp4 (the C ABI) on plain scales. The call reorders
sfA and sfB into the 128x4 atom layout (one launch), then launches the
persistent tcgen05 GEMM on the reordered scales as a programmatic dependent of
the reorder; where the plan is a single launch (the narrow-M CUDA-core kernel,
which reads the plain scales in place), that launch alone. Nothing is recorded
between the reorder and the GEMM (an event there would break their overlap),
so the GEMM's own duration, for the roofline, is timed separately: the GEMM
alone on scales reordered once before the loop, launched between the timed
steps after its own L2 flush, with CUDA events around it.
Inputs are seeded synthetic data resident in HBM; L2 is
flushed (a 256 MiB write) between timed steps, outside each step's events, and
a spin kernel queued before each step keeps host launch overhead out of them.

`value` is whole-job TFLOP/s (2*M*N*K per step, summed over ranks, divided by
the slowest rank's time). `roofline` is for the GEMM kernel: its FLOPs per
launch over its CUDA-event duration, against the dense FP4 tensor peak (the
measured bf16 burst peak times the nominal FP4:bf16 ratio 13.5:2.25 = 6).
`e2e` is the same metric through fp4_gemm_host with pinned host buffers, the
host<->device copies inside the timed region; consecutive steps alternate
between two streams, so one step's result download overlaps the next step's
upload (two requests in flight). `cpu_baseline` is the fp64 CPU
oracle on a bounded row sample of the same problem, on all host cores.

Multi-GPU (torchrun): replicas only -- every rank runs the same problem on its
own GPU with no collective in the data path (weak scaling).

--impl reference times the CPU oracle (the only reference this project has)
on the same workload, one bounded row sample per step.

--op fused times the GEMM with a fused epilogue (fp4_gemm_fused: bias,
ReLU, squared ReLU or SwiGLU applied to the accumulator before the cast) on
the FFN workloads ffn_*; same metric, roofline and legs, with the oracle's
GEMM plus its epilogue as the cpu_baseline and e2e through pinned host
buffers copied on the stream around the same call.

--op grouped times the grouped (mixture-of-experts) GEMM, fp4_gemm_grouped,
on the moe_* workloads: a step is one grouped call on plain scales (one
reorder launch for the routed activations' and the experts' weight scales,
then the one grouped GEMM launch over all experts); the GEMM alone on
prepacked scales is timed between the steps for the roofline, as above. Same
metric (2 * M_total * N * K per step).

--op quantize measures the quantisation step that feeds the GEMM instead
(fp4_quantize: bf16 or fp32 activations -> E2M1 codes + atom-layout scales),
against the HBM roofline: its bytes (values read, codes and scale atoms
written) over its CUDA-event duration, with the CPU oracle's quantiser on a
row sample as the cpu_baseline. Its workloads are the quant_* names.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "block-scaled FP4 GEMM TFLOP/s on 1 GB300 and % of dense FP4 tensor peak"
DEFAULT_WORKLOAD = "nvfp4_8192_f32"
DEFAULT_FUSED_WORKLOAD = "ffn_swiglu_nvfp4_m8192_n28672_k4096"
DEFAULT_GROUPED_WORKLOAD = "moe_nvfp4_e64_t4096_top8_n2048_k4096"
FP4_PER_BF16 = 13.5 / 2.25       # nominal dense FP4 : dense bf16 tensor throughput on GB300
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
SPACER_CYCLES = 400_000          # ~0.2 ms at 2 GHz


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, FALLBACK_HBM_GBS, "fallback"


GEMM_SOURCES = ("block_scaled_fp4_sfa_gb300/csrc/fp4_gemm.cu", "block_scaled_fp4_sfa_gb300/csrc/ptx.cuh",
                "block_scaled_fp4_sfa_gb300/csrc/epilogue.cuh")
GEMV_SOURCES = ("block_scaled_fp4_sfa_gb300/csrc/fp4_gemv.cu", "block_scaled_fp4_sfa_gb300/csrc/epilogue.cuh")
QUANT_SOURCES = ("block_scaled_fp4_sfa_gb300/csrc/fp4_quant.cu", "block_scaled_fp4_sfa_gb300/csrc/ptx.cuh")


def kernel_source_hash(sources=GEMM_SOURCES):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, sources=GEMM_SOURCES):
    """DRAM bytes per launch of the workload's kernel from the committed ncu
    summary (profiles/traffic.json), if it was taken on the current kernel
    source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash(sources):
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle sampling (every 20 ms) while the timed region
    runs; only samples stamped inside the region (mark_start / mark_end) count."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None
        self.lines = []

    def __enter__(self):
        if self.index < 0:
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    @staticmethod
    def _stamp(text):
        try:
            whole, _, frac = text.strip().partition(".")
            return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
        except ValueError:
            return None

    def summary(self):
        sm, mx, reasons = [], [], set()
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            ts = self._stamp(f[0])
            if ts is None or self.t0 is None or not (self.t0 <= ts <= (self.t1 or ts)):
                continue
            try:
                sm.append(float(f[2]))
                mx.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_rows_tflops(inp, rows, nthreads=0, act=None, bias=None):
    import oracle
    t0 = time.perf_counter()
    y, _ = oracle.gemm_rows(inp, rows, nthreads=nthreads)
    if act is not None:
        oracle.epilogue(y, bias, act)
    dt = time.perf_counter() - t0
    return 2.0 * len(rows) * inp.N * inp.K / dt / 1e12, dt


def cpu_sample_rows(inp, target_s):
    """Row sample whose oracle time is about target_s seconds (at least 1 row)."""
    probe = np.arange(min(8, inp.M))
    oracle_rows_tflops(inp, probe[:1])                 # first call: library load, thread start
    _, dt = oracle_rows_tflops(inp, probe)
    per_row = dt / len(probe)
    n = int(max(1, min(inp.M, target_s / max(per_row, 1e-9))))
    return np.linspace(0, inp.M - 1, n).astype(np.int64)


def run_reference(args, inp):
    """The CPU oracle timed as the reference arm: each step one bounded row sample."""
    # each step a bounded sample; the whole run stays within about two minutes
    rows = cpu_sample_rows(inp, min(args.ref_step_s, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_rows_tflops(inp, rows[: max(1, len(rows) // 8)])
    times = []
    for _ in range(args.steps):
        _, dt = oracle_rows_tflops(inp, rows)
        times.append(dt)
    flops = 2.0 * len(rows) * inp.N * inp.K
    value = flops * len(times) / sum(times) / 1e12
    cores = os.cpu_count()
    sample = "%d of %d rows of %s (all %d columns), fp64 C oracle, OpenMP on %d cores" % (
        len(rows), inp.M, inp.name, inp.N, cores)
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(workload_config(inp), parallelism="replicas" if args.gpus > 1 else "single"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def slowest_rank_ms(local_ms, world_size, device=None):
    """Max over ranks of the timed-region milliseconds (replicas run concurrently)."""
    if world_size <= 1:
        return float(local_ms)
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step, steps, world_size, total_ms):
    """Units all ranks processed (every rank runs `steps` steps) over the slowest rank's time."""
    return flops_per_step * steps * world_size / (total_ms * 1e-3) / 1e12


def workload_config(inp, act=None, bias=None):
    c = {"workload": inp.name, "format": inp.fmt, "M": inp.M, "N": inp.N, "K": inp.K, "out": inp.out,
         "alpha": inp.alpha, "l2": "flushed between steps (256 MiB write, outside the step events)"}
    if act is not None:
        c["epilogue"] = act
        c["bias"] = bias is not None
    return c


def run_ours(args, inp, rank, ws, local, act=None, bias=None):
    import torch
    import block_scaled_fp4_sfa_gb300 as fp4

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp4.load()
    stream = torch.cuda.current_stream()
    vec = inp.vec
    hA, hsA, hB, hsB = (torch.from_numpy(np.ascontiguousarray(getattr(inp, k))) for k in ("A", "sfA", "B", "sfB"))
    A, sfA, B, sfB = (t.to(dev) for t in (hA, hsA, hB, hsB))
    atomA = torch.empty(fp4.scale_atom_bytes(inp.M, inp.K, vec), dtype=torch.uint8, device=dev)
    atomB = torch.empty(fp4.scale_atom_bytes(inp.N, inp.K, vec), dtype=torch.uint8, device=dev)
    odt = torch.float32 if inp.out == "f32" else torch.bfloat16
    fused = act is not None
    d_cols = inp.N // 2 if act == "swiglu" else inp.N
    D = torch.empty(inp.M, d_cols, dtype=odt, device=dev)
    hbias = torch.from_numpy(bias) if bias is not None else None
    dbias = hbias.to(dev) if bias is not None else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    s = stream.cuda_stream
    # The step is the call a user makes on plain scales: it reorders them and
    # launches the GEMM as a programmatic dependent of the reorder. The GEMM's
    # own duration (for the roofline) is timed alone, on scales reordered once
    # before the loop, between the timed steps and after its own L2 flush: an
    # event recorded between the reorder and the GEMM would break their overlap.
    # A plan of one launch (the narrow-M kernel reads plain scales in place)
    # needs no second leg: the step is the kernel.
    plan = fp4.gemm_plan(inp.fmt, inp.M, inp.N, inp.K, inp.out, act=act or "none")
    narrow = plan["kernel"] == "narrow"
    single = plan["launches"] == 1
    kplan = fp4.gemm_plan(inp.fmt, inp.M, inp.N, inp.K, inp.out, act=act or "none", prepacked=True)
    leg_launches = 0 if single else kplan["launches"]
    plain_call = fp4.gemm_nvfp4 if inp.fmt == "nvfp4" else fp4.gemm_mxfp4
    pre_call = fp4.gemm_nvfp4_prepacked if inp.fmt == "nvfp4" else fp4.gemm_mxfp4_prepacked

    def gemm_call(a, sa, b, sb, d, bb, pre):
        if fused:
            fp4.gemm_fused(inp.fmt, a, sa, b, sb, inp.alpha, d, inp.M, inp.N, inp.K, inp.out, act=act, bias=bb,
                           prepacked=pre, stream=s)
        else:
            (pre_call if pre else plain_call)(a, sa, b, sb, inp.alpha, d, inp.M, inp.N, inp.K, inp.out, stream=s)

    def spacer():
        # a spin kernel keeps the GPU busy while the host enqueues the step, so no
        # host launch overhead falls between the events that bracket the kernels
        torch.cuda._sleep(SPACER_CYCLES)

    def step():
        gemm_call(A, sfA, B, sfB, D, dbias, False)

    def kernel_alone():
        gemm_call(A, atomA, B, atomB, D, dbias, True)

    if not single:
        fp4.scale_reorder2(sfA, atomA, inp.M, sfB, atomB, inp.N, inp.K, vec, stream=s)
    for _ in range(args.warmup):
        flush.zero_()
        spacer()
        step()
        if not single:
            flush.zero_()
            spacer()
            kernel_alone()
    torch.cuda.synchronize()
    st = fp4.get_device_status(s)
    if st != 0:
        raise RuntimeError("device status after warm-up: %s" % fp4.status_string(st))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if not single else starts
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] if not single else ends
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sp0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local if not args.quick else -1) as clk:
        time.sleep(0.5)
        clk.mark_start()
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            sp0[i].record(stream)
            spacer()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            if not single:
                flush.zero_()
                spacer()
                g0[i].record(stream)
                kernel_alone()
                g1[i].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        clk.mark_end()
        if ws > 1:
            torch.distributed.barrier()
    st = fp4.get_device_status(s)
    if st != 0:
        raise RuntimeError("device status after timing: %s" % fp4.status_string(st))
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    gemm_ms = [a.elapsed_time(b) for a, b in zip(g0, g1)]
    # SM clock between the steps: the spin kernel runs SPACER_CYCLES clock cycles
    spin_mhz = statistics.median(SPACER_CYCLES / (a.elapsed_time(b) * 1e3) for a, b in zip(sp0, starts))
    total_ms = slowest_rank_ms(sum(step_ms), ws, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(inp.flops, args.steps, ws, total_ms)

    result_quick = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "ms_per_step": ms_per_step,
                    "gemm_us": 1e3 * sum(gemm_ms) / len(gemm_ms), "config": workload_config(inp, act, bias)}
    if args.quick:
        return result_quick

    # e2e: host buffers, pinned memory, copies inside the timed region -- through
    # fp4_gemm_host, or for a fused epilogue the same copies on the stream around
    # fp4_gemm_fused (plain scales: it reorders them itself). Consecutive steps
    # go to two streams in turn (each with its own result buffer, and for the
    # fused call its own device buffers), as two requests in flight would: one
    # step's result download overlaps the next step's upload on the full-duplex
    # host link. The events bracket all steps on both streams.
    pA, psA, pB, psB = (t.pin_memory() for t in (hA, hsA, hB, hsB))
    pbias = hbias.pin_memory() if hbias is not None else None
    lanes = []
    for i in range(2):
        st = stream if i == 0 else torch.cuda.Stream()
        lane = {"stream": st, "pD": torch.empty(inp.M, d_cols, dtype=odt).pin_memory()}
        if fused:
            lane.update({"A": A if i == 0 else torch.empty_like(A), "sfA": sfA if i == 0 else torch.empty_like(sfA),
                         "B": B if i == 0 else torch.empty_like(B), "sfB": sfB if i == 0 else torch.empty_like(sfB),
                         "D": D if i == 0 else torch.empty_like(D),
                         "bias": dbias if (i == 0 or dbias is None) else torch.empty_like(dbias)})
        lanes.append(lane)

    def e2e_step(i):
        lane = lanes[i % 2]
        st = lane["stream"]
        if not fused:
            fp4.gemm_host(inp.fmt, pA, psA, pB, psB, inp.alpha, lane["pD"], inp.M, inp.N, inp.K, inp.out,
                          stream=st.cuda_stream)
            return
        with torch.cuda.stream(st):
            for key, src in (("A", pA), ("sfA", psA), ("B", pB), ("sfB", psB), ("bias", pbias)):
                if lane[key] is not None:
                    lane[key].copy_(src, non_blocking=True)
            fp4.gemm_fused(inp.fmt, lane["A"], lane["sfA"], lane["B"], lane["sfB"], inp.alpha, lane["D"], inp.M,
                           inp.N, inp.K, inp.out, act=act, bias=lane["bias"], stream=st.cuda_stream)
            lane["pD"].copy_(lane["D"], non_blocking=True)

    e_steps = max(4, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    lanes[1]["stream"].wait_event(e0)
    for i in range(e_steps):
        e2e_step(i)
    done1 = torch.cuda.Event()
    done1.record(lanes[1]["stream"])
    stream.wait_event(done1)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    h2d = sum(t.numel() * t.element_size() for t in (hA, hsA, hB, hsB) + ((hbias,) if hbias is not None else ()))
    d2h = lanes[0]["pD"].numel() * lanes[0]["pD"].element_size()

    bf16_peak, hbm_peak, peak_src = peaks()
    gemm_avg_ms = sum(gemm_ms) / len(gemm_ms)
    achieved = inp.flops / (gemm_avg_ms * 1e-3) / 1e12
    fp4_peak = bf16_peak * FP4_PER_BF16
    kname = "gemv_kernel" if narrow else "fp4_gemm_kernel"
    traffic = ncu_traffic(inp.name, GEMV_SOURCES if narrow else GEMM_SOURCES)
    alg_bytes = ((inp.M + inp.N) * (inp.K // 2 + inp.K // vec) + inp.M * d_cols * (4 if inp.out == "f32" else 2)
                 + (4 * inp.N if bias is not None else 0))
    # the binding roof: HBM when the arithmetic intensity is below the ridge
    # (skinny shapes), else the FP4 tensor rate
    hbm_bound = inp.flops / alg_bytes < fp4_peak * 1e12 / (hbm_peak * 1e9)
    achieved_gbs = alg_bytes / (gemm_avg_ms * 1e-3) / 1e9
    if hbm_bound:
        roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                    "peak_source": "%s HBM copy bandwidth" % peak_src,
                    "tensor_tflops": achieved, "tensor_frac": achieved / fp4_peak}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp4_peak, "traffic": traffic,
                    "peak_source": "%s bf16 burst %.1f TFLOP/s x %.0f (nominal FP4:bf16)" % (
                        peak_src, bf16_peak, FP4_PER_BF16)}
    clocks = clk.summary()
    clocks["sm_mhz_spin"] = spin_mhz
    mhz = clocks["sm_mhz"] or spin_mhz
    roofline.update({"kernel": kname, "gemm_us": 1e3 * gemm_avg_ms, "algorithmic_bytes": alg_bytes,
                     # kernel time x median SM clock = its cycles, so runs at other clocks compare
                     "gemm_us_x_sm_mhz": 1e3 * gemm_avg_ms * mhz, "sm_mhz_used": mhz,
                     "hbm_frac_at_algorithmic_bytes": achieved_gbs / hbm_peak,
                     "timed": "the step itself" if single else
                     "alone on prepacked scales, between the timed steps, L2 flushed before each launch"})
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1", "data": "synthetic",
        "config": dict(workload_config(inp, act, bias), parallelism="replicas" if ws > 1 else "single"),
        "roofline": roofline,
        "e2e": {"value": inp.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": (plan["launches"] + leg_launches) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    return result


QUANT_METRIC = "FP4 activation quantisation GB/s on 1 GB300 and % of HBM bandwidth"
DEFAULT_QUANT_WORKLOAD = "quant_nvfp4_8192x4096_bf16"


def quant_bytes(rows, K, vec, in_bytes, atom_bytes):
    return rows * K * in_bytes + rows * K // 2 + atom_bytes


def run_quant(args, rank, ws, local):
    """Times fp4_quantize (atom-layout scales) on a named activation workload."""
    import torch
    import block_scaled_fp4_sfa_gb300 as fp4
    name = args.workload if args.workload in W.QUANT_WORKLOADS else DEFAULT_QUANT_WORKLOAD
    fmt, X = W.make_quant_workload(name, seed=rank)
    rows, K = X.shape
    vec = 16 if fmt == "nvfp4" else 32
    in_dtype = "bf16" if X.dtype == np.uint16 else "f32"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp4.load()
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    hX = torch.from_numpy(X.view(np.int16) if X.dtype == np.uint16 else X)
    Xd = hX.to(dev)
    atom_bytes = fp4.scale_atom_bytes(rows, K, vec)
    codes = torch.empty(rows * K // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(atom_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    nbytes = quant_bytes(rows, K, vec, X.itemsize, atom_bytes)

    def step():
        fp4.quantize(fmt, Xd, rows, K, codes, sf, in_dtype=in_dtype, layout="atom", stream=s)

    for _ in range(args.warmup):
        flush.zero_()
        torch.cuda._sleep(SPACER_CYCLES)
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local if not args.quick else -1) as clk:
        time.sleep(0.5)
        clk.mark_start()
        for e0, e1 in ev:
            flush.zero_()
            torch.cuda._sleep(SPACER_CYCLES)
            e0.record(stream)
            step()
            e1.record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        if ws > 1:
            torch.distributed.barrier()
    st = fp4.get_device_status(s)
    if st != 0:
        raise RuntimeError("device status after timing: %s" % fp4.status_string(st))
    ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = slowest_rank_ms(sum(ms), ws, dev)
    ms_per_step = total_ms / args.steps
    value = nbytes * args.steps * ws / (total_ms * 1e-3) / 1e9
    cfg = {"workload": name, "format": fmt, "rows": rows, "K": K, "in": in_dtype, "scales": "atom",
           "l2": "flushed between steps (256 MiB write, outside the step events)",
           "parallelism": "replicas" if ws > 1 else "single"}
    res = {"metric": QUANT_METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": in_dtype + "->e2m1", "data": "synthetic", "config": cfg}
    if args.quick:
        return res
    # e2e: pinned host values in, codes and scales back to pinned host memory;
    # consecutive steps on two streams in turn, each with its own buffers (as
    # for the GEMM line: one step's download overlaps the next one's upload)
    pX = hX.pin_memory()
    lanes = []
    for i in range(2):
        lanes.append({"stream": stream if i == 0 else torch.cuda.Stream(),
                      "X": Xd if i == 0 else torch.empty_like(Xd),
                      "codes": codes if i == 0 else torch.empty_like(codes),
                      "sf": sf if i == 0 else torch.empty_like(sf),
                      "pc": torch.empty(rows * K // 2, dtype=torch.uint8).pin_memory(),
                      "ps": torch.empty(atom_bytes, dtype=torch.uint8).pin_memory()})

    def e2e_step(i):
        lane = lanes[i % 2]
        with torch.cuda.stream(lane["stream"]):
            lane["X"].copy_(pX, non_blocking=True)
            fp4.quantize(fmt, lane["X"], rows, K, lane["codes"], lane["sf"], in_dtype=in_dtype, layout="atom",
                         stream=lane["stream"].cuda_stream)
            lane["pc"].copy_(lane["codes"], non_blocking=True)
            lane["ps"].copy_(lane["sf"], non_blocking=True)

    e_steps = max(4, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    lanes[1]["stream"].wait_event(e0)
    for i in range(e_steps):
        e2e_step(i)
    done1 = torch.cuda.Event()
    done1.record(lanes[1]["stream"])
    stream.wait_event(done1)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    pc, ps = lanes[0]["pc"], lanes[0]["ps"]
    _, hbm_peak, peak_src = peaks()
    avg_ms = sum(ms) / len(ms)
    achieved = nbytes / (avg_ms * 1e-3) / 1e9
    res.update({
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": ncu_traffic(name, QUANT_SOURCES),
                     "peak_source": "%s HBM copy bandwidth" % peak_src, "kernel": "quantize_kernel",
                     "kernel_us": 1e3 * avg_ms, "algorithmic_bytes": nbytes},
        "e2e": {"value": nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": hX.numel() * hX.element_size(), "d2h_bytes_per_step": pc.numel() + ps.numel()},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    })
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        n = 64
        t0 = time.perf_counter()
        oracle.quantize(X[:n], fmt)
        dt = time.perf_counter() - t0
        n = int(max(1, min(rows, n * args.cpu_sample_s / 4 / max(dt, 1e-6))))
        # whole passes over the sample until about cpu_sample_s / 2 seconds have run
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.quantize(X[:n], fmt)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= args.cpu_sample_s / 2 or reps >= 1000:
                break
        res["cpu_baseline"] = {"value": reps * quant_bytes(n, K, vec, X.itemsize, 0) / dt / 1e9, "unit": "GB/s",
                               "cores": os.cpu_count(), "kind": "oracle",
                               "sample": "first %d of %d rows of %s, %d passes, %.1f s, C oracle (fp32 decisions), "
                                         "plain scales" % (n, rows, name, reps, dt)}
    return res


def run_grouped(args, rank, ws, local):
    """Times fp4_gemm_grouped on a named MoE workload."""
    import torch
    import block_scaled_fp4_sfa_gb300 as fp4
    gin, act = W.make_grouped_workload(args.workload, seed=rank)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp4.load()
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    vec, M, N, K, G = gin.vec, gin.M, gin.N, gin.K, gin.G
    hA, hsA, hB, hsB = (torch.from_numpy(np.ascontiguousarray(getattr(gin, k))) for k in ("A", "sfA", "B", "sfB"))
    A, sfA, B, sfB = (t.to(dev) for t in (hA, hsA, hB, hsB))
    atomA = torch.empty(max(16, fp4.scale_atom_bytes_grouped(gin.offsets, K, vec)), dtype=torch.uint8, device=dev)
    assert N % 128 == 0            # then one reorder of all G*N weight rows is the per-expert atom layout
    atomB = torch.empty(fp4.scale_atom_bytes(G * N, K, vec), dtype=torch.uint8, device=dev)
    odt = torch.float32 if gin.out == "f32" else torch.bfloat16
    d_cols = N // 2 if act == "swiglu" else N
    D = torch.empty(M, d_cols, dtype=odt, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    # The step is the grouped call on plain scales (one reorder launch for the
    # routed activations' and the experts' scales, then the GEMM as its
    # programmatic dependent). The GEMM alone, on scales reordered once before
    # the loop, is timed between the steps for the roofline.
    def step():
        fp4.gemm_grouped(gin.fmt, gin.offsets, A, sfA, B, sfB, gin.alpha, D, N, K, gin.out, act=act, stream=s)

    def kernel_alone():
        fp4.gemm_grouped(gin.fmt, gin.offsets, A, atomA, B, atomB, gin.alpha, D, N, K, gin.out, act=act,
                         weights_prepacked=True, acts_prepacked=True, stream=s)

    fp4.scale_reorder_grouped(sfA, atomA, gin.offsets, K, vec, stream=s)
    fp4.scale_reorder(sfB, atomB, G * N, K, vec, stream=s)
    for _ in range(args.warmup):
        for f in (step, kernel_alone):
            flush.zero_()
            torch.cuda._sleep(SPACER_CYCLES)
            f()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local if not args.quick else -1) as clk:
        time.sleep(0.5)
        clk.mark_start()
        for i in range(args.steps):
            flush.zero_()
            torch.cuda._sleep(SPACER_CYCLES)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            flush.zero_()
            torch.cuda._sleep(SPACER_CYCLES)
            g0[i].record(stream)
            kernel_alone()
            g1[i].record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        if ws > 1:
            torch.distributed.barrier()
    st = fp4.get_device_status(s)
    if st != 0:
        raise RuntimeError("device status after timing: %s" % fp4.status_string(st))
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    gemm_ms = [a.elapsed_time(b) for a, b in zip(g0, g1)]
    total_ms = slowest_rank_ms(sum(step_ms), ws, dev)
    value = whole_job_tflops(gin.flops, args.steps, ws, total_ms)
    sizes = np.diff(gin.offsets)
    cfg = {"workload": gin.name, "format": gin.fmt, "experts": G, "M_total": M, "N": N, "K": K, "out": gin.out,
           "epilogue": act, "rows_per_expert": {"min": int(sizes.min()), "max": int(sizes.max()),
                                                "empty": int((sizes == 0).sum())},
           "l2": "flushed between steps (256 MiB write, outside the step events)",
           "parallelism": "replicas" if ws > 1 else "single"}
    res = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "e2m1", "data": "synthetic", "config": cfg,
           "gemm_us": 1e3 * sum(gemm_ms) / len(gemm_ms)}
    if args.quick:
        return res
    # e2e: pinned host buffers copied in, the plain-scale grouped call, D copied
    # back; consecutive steps on two streams in turn, each with its own buffers
    # (as for the GEMM line)
    pA, psA, pB, psB = (t.pin_memory() for t in (hA, hsA, hB, hsB))
    lanes = []
    for i in range(2):
        lane = {"stream": stream if i == 0 else torch.cuda.Stream(),
                "pD": torch.empty(M, d_cols, dtype=odt).pin_memory()}
        for key, t in (("A", A), ("sfA", sfA), ("B", B), ("sfB", sfB), ("D", D)):
            lane[key] = t if i == 0 else torch.empty_like(t)
        lanes.append(lane)

    def e2e_step(i):
        lane = lanes[i % 2]
        with torch.cuda.stream(lane["stream"]):
            for key, src in (("A", pA), ("sfA", psA), ("B", pB), ("sfB", psB)):
                lane[key].copy_(src, non_blocking=True)
            fp4.gemm_grouped(gin.fmt, gin.offsets, lane["A"], lane["sfA"], lane["B"], lane["sfB"], gin.alpha,
                             lane["D"], N, K, gin.out, act=act, stream=lane["stream"].cuda_stream)
            lane["pD"].copy_(lane["D"], non_blocking=True)

    e_steps = max(4, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    lanes[1]["stream"].wait_event(e0)
    for i in range(e_steps):
        e2e_step(i)
    done1 = torch.cuda.Event()
    done1.record(lanes[1]["stream"])
    stream.wait_event(done1)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e_steps
    pD = lanes[0]["pD"]
    bf16_peak, hbm_peak, peak_src = peaks()
    gemm_avg_ms = sum(gemm_ms) / len(gemm_ms)
    achieved = gin.flops / (gemm_avg_ms * 1e-3) / 1e12
    fp4_peak = bf16_peak * FP4_PER_BF16
    used = int((sizes > 0).sum())
    alg_bytes = (M * (K // 2 + K // vec) + used * N * (K // 2 + K // vec)
                 + M * d_cols * (4 if gin.out == "f32" else 2))
    achieved_gbs = alg_bytes / (gemm_avg_ms * 1e-3) / 1e9
    if gin.flops / alg_bytes < fp4_peak * 1e12 / (hbm_peak * 1e9):
        roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved_gbs / hbm_peak, "peak_source": "%s HBM copy bandwidth" % peak_src,
                    "tensor_tflops": achieved, "tensor_frac": achieved / fp4_peak}
    else:
        roofline = {"bound": "tensor", "achieved": achieved, "peak": fp4_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp4_peak, "peak_source": "%s bf16 burst %.1f TFLOP/s x %.0f (nominal FP4:bf16)"
                    % (peak_src, bf16_peak, FP4_PER_BF16)}
    roofline.update({"traffic": ncu_traffic(gin.name), "kernel": "fp4_gemm_kernel (grouped)",
                     "gemm_us": 1e3 * gemm_avg_ms, "algorithmic_bytes": alg_bytes,
                     "hbm_frac_at_algorithmic_bytes": achieved_gbs / hbm_peak})
    res.update({
        "roofline": roofline,
        "e2e": {"value": gin.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hA, hsA, hB, hsB)),
                "d2h_bytes_per_step": pD.numel() * pD.element_size()},
        "gpu_launches": 3 * args.steps,      # step: reorder + GEMM; then the GEMM alone
        "clocks": clk.summary(),
    })
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        probe = np.arange(min(8, M))
        oracle.grouped_gemm_rows(gin, probe[:1])
        t0 = time.perf_counter()
        oracle.grouped_gemm_rows(gin, probe)
        per_row = (time.perf_counter() - t0) / len(probe)
        n = int(max(1, min(M, args.cpu_sample_s / max(per_row, 1e-9))))
        rows = np.linspace(0, M - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        y, _ = oracle.grouped_gemm_rows(gin, rows)
        oracle.epilogue(y, None, act)
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": 2.0 * n * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                               "kind": "oracle",
                               "sample": "%d of %d routed rows of %s (all %d columns), %.1f s, fp64 C oracle per "
                                         "expert + its %s epilogue" % (n, M, gin.name, N, dt, act)}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["gemm", "fused", "grouped", "quantize"], default="gemm")
    ap.add_argument("--workload", default=None,
                    choices=W.config_names() + sorted(W.FUSED_WORKLOADS) + sorted(W.GROUPED_WORKLOADS)
                    + sorted(W.QUANT_WORKLOADS))
    ap.add_argument("--cpu-sample-s", type=float, default=12.0, help="oracle seconds for cpu_baseline")
    ap.add_argument("--ref-step-s", type=float, default=3.0, help="oracle seconds per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--results", default=None, help="also append the JSON line to this file")
    ap.add_argument("--quick", action="store_true",
                    help="GEMM steps only: no e2e, clock or CPU legs (for profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if args.workload is None:
        args.workload = {"quantize": DEFAULT_QUANT_WORKLOAD, "fused": DEFAULT_FUSED_WORKLOAD,
                         "grouped": DEFAULT_GROUPED_WORKLOAD}.get(args.op, DEFAULT_WORKLOAD)
    table = {"quantize": W.QUANT_WORKLOADS, "fused": W.FUSED_WORKLOADS, "grouped": W.GROUPED_WORKLOADS}.get(args.op)
    valid = table if table is not None else W.config_names()
    if args.workload not in valid:
        ap.error("--op %s does not take workload %s" % (args.op, args.workload))
    if args.op != "gemm" and args.impl == "reference":
        ap.error("--impl reference times the GEMM's oracle; use --op gemm")

    if args.op in ("quantize", "grouped"):
        if ws > 1:
            import torch
            torch.cuda.set_device(local)
            torch.distributed.init_process_group("nccl")
        res = (run_quant if args.op == "quantize" else run_grouped)(args, rank, ws, local)
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
    elif args.impl == "reference":
        if rank != 0:
            return
        inp = W.make_config(args.workload)
        res = run_reference(args, inp)
    else:
        if ws > 1:
            import torch
            torch.cuda.set_device(local)
            torch.distributed.init_process_group("nccl")
        act = bias = None
        if args.op == "fused":
            inp, act, bias = W.make_fused(args.workload)
        else:
            inp = W.make_config(args.workload)
        res = run_ours(args, inp, rank, ws, local, act, bias)
        if rank == 0 and not args.no_cpu_baseline and not args.quick:
            rows = cpu_sample_rows(inp, args.cpu_sample_s)
            v, dt = oracle_rows_tflops(inp, rows, act=act, bias=bias)
            what = "fp64 C oracle" + (" + its %s epilogue" % act if act else "")
            res["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                   "sample": "%d of %d rows of %s (all %d columns), %.1f s, %s"
                                             % (len(rows), inp.M, inp.name, inp.N, dt, what)}
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
    if rank == 0:
        line = json.dumps(res)
        print(line, flush=True)
        if args.results:
            with open(args.results, "a") as f:
                f.write(line + "\n")


if __name__ == "__main__":
    main()
