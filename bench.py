#!/usr/bin/env python
"""RankMixer block forward + backward throughput on GB300.

One step = rmx_forward + rmx_backward of the whole block over one batch
(B=1024, T=64, D=1280, H=2560, bf16 storage by default), inputs resident in
HBM.  Prints one JSON line (rank 0).  Timing follows the page's protocol
("Subgraph-fusion-based Mega-kernel Generation", section "Exact timing
behavior"): warm-up, an L2 flush and a barrier before every measured step
(outside the timed region), CUDA events around the complete forward+backward.

Multi-GPU (--gpus N under torchrun): N independent replicas, one per GPU, each
on its own batch (the block needs no exchange at EP=1); value = all rows
processed / the slowest rank's time.

--impl reference times the float64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "RankMixer fwd+bwd rows/s (B*T) at B1024/T64/D1280/H2560; % of roofline"
WORKLOAD_NAMES = {
    "c3": "RankMixer production block B=1024 T=64 D=1280 H=2560 bf16",
    "c4": "RankMixer ragged block B=1000 T=40 D=1200 H=3600 fp16",
    "c2": "RankMixer mid block B=256 T=32 D=512 H=1536 bf16",
    "c1": "RankMixer small block B=64 T=16 D=256 H=512 fp32",
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# FP32 FMA peak of the CUDA cores (the strict fp32 contract's contractions):
# 152 SMs x 128 fp32 lanes x 2 FLOP per FMA x 2.07 GHz (maximum SM clock).
GB300_SMS, FP32_LANES_PER_SM, SM_MAX_GHZ = 152, 128, 2.07
FFMA_TFLOPS = GB300_SMS * FP32_LANES_PER_SM * 2 * SM_MAX_GHZ / 1e3


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference", "unfused"], default="ours",
                    help="ours; reference = the float64 oracle on the host cores; unfused = a plain PyTorch "
                         "eager composition of the block on the GPU (the per-op sequence the fused path is "
                         "compared with for time, memory and DRAM bytes)")
    ap.add_argument("--config", default="c3")
    ap.add_argument("--batch", type=int, default=None, help="override B (profiling a smaller case)")
    ap.add_argument("--tokens", type=int, default=None, help="override T (profiling a smaller case)")
    ap.add_argument("--dim", type=int, default=None, help="override D (profiling a smaller case)")
    ap.add_argument("--hidden", type=int, default=None, help="override H (profiling a smaller case)")
    ap.add_argument("--graph", action="store_true",
                    help="time the step as a replay of a captured CUDA graph (rmx_graph_launch) instead of the "
                         "two calls")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-reps", type=int, default=6, help="timed oracle calls of the CPU baseline")
    ap.add_argument("--oracle-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--samples", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--reps", type=int, default=1, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ---------------------------------------------------------------- accounting

def flops_per_step(s) -> float:
    """18 * B*T*D*H: the four forward contractions (2 x 2*B*T*D*2H ... ) and
    the eight backward ones (dgrad + wgrad of each)."""
    return 18.0 * s.B * s.T * s.D * s.H


def min_bytes_per_step(s) -> float:
    """Bytes the API forces: x, dy read; y, dx written; parameters read in the
    forward and the backward; parameter gradients written once."""
    e = 4 if s.dtype == "f32" else 2
    act = 4 * s.B * s.T * s.D * e
    params = (3 * s.T * s.D * s.H + s.T * 2 * s.H + s.T * s.D + 6 * s.D + 4 * s.H) * e
    return act + 3 * params


def gemm_flops_per_launch(s) -> dict:
    BTDH = s.B * s.T * s.D * s.H
    return {
        "gemm1_fwd": 4.0 * BTDH, "gemm2_fwd": 2.0 * BTDH,
        "gemm2_dgrad": 2.0 * BTDH, "gemm2_wgrad": 2.0 * BTDH,
        "gemm1_dgrad": 4.0 * BTDH, "gemm1_wgrad": 4.0 * BTDH,
    }


def row_bytes_per_launch(s) -> dict:
    """Algorithmic HBM bytes of each row pass (reads + writes of full tensors)."""
    e = 4 if s.dtype == "f32" else 2
    N = s.B * s.T
    BTD, BTH = N * s.D * e, N * s.H * e
    return {
        "ln01_fwd": 3 * BTD,                        # x in; s1 and out1 out (one CTA per sample)
        "ln0_fwd_mixed": 2 * BTD,                   # x in, token_mix(norm0(x)) out (large samples)
        "ln1_fwd": 4 * BTD,                         # mix, x in; s1 and out1 out (large samples)
        "gate_fwd": 2 * BTH + BTH,                  # Z in, hidden out (row statistics merged in-pass)
        "ln2_fwd": 2 * BTD,                         # s2 in, y out
        "ln2_bwd": 3 * BTD,                         # dy, s2 in, ds2 out
        "gate_bwd": BTH + 2 * BTH + 2 * BTH,        # dh, Z in, dZ out (single pass)
        "ln1_bwd": 3 * BTD,                         # dout1, s1 in; ds1 out
        "ln0_bwd_gather": 3 * BTD,                  # ds1, x in, dx out (the mix read from a stripe of ds1)
        "ln1_bwd_mixed": 4 * BTD,                   # dout1, s1 in; ds1 and token_mix(ds1) out
        "ln0_bwd": 4 * BTD,                         # token_mix(ds1), x, ds1 in, dx out
    }


def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


PEAK_RULE = "burst peak when the median SM clock of the timed region is within 5% of the maximum, else sustained"


def tensor_peak(peaks: dict, clocks: dict) -> tuple[float, float, str]:
    """(burst, sustained, which) bf16 tensor peaks in TFLOP/s.  The burst
    figure was measured at full clock and the sustained one under the power
    cap: the denominator is the burst figure when the timed region ran at
    (nearly) the maximum SM clock, so a kernel is not flattered by a peak
    taken at a lower clock than its own."""
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = sm is None or smax is None or sm >= 0.95 * smax
    return burst, sustained, "burst" if at_max else "sustained"


# Source file of each kernel (besides the headers every kernel includes).
KERNEL_SOURCES = {
    "gemm": "gemm_tc.cu", "gate_bwd": "gate_bwd.cu", "ln01_fwd": "ln01_fwd.cu", "ln0_bwd_gather": "ln0_bwd.cu",
    "ln1_bwd": "ln_bwd.cu", "ln2_bwd": "ln_bwd.cu", "gate_fwd": "rows.cu", "ln2_fwd": "rows.cu", "colsums": "rows.cu",
}
SHARED_SOURCES = ("common.cuh", "launch.cuh", "kernels.h")


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the sources a kernel is built from (its file and the shared
    headers; every kernel file when `kernel` is None or unknown): a profile
    taken on other sources is stale."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ffn_block_gb300", "csrc")
    key = "gemm" if kernel and kernel.startswith("gemm") else kernel
    if key in KERNEL_SOURCES:
        names = sorted({KERNEL_SOURCES[key], *SHARED_SOURCES})
    else:
        names = sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks

def gpu_selector(dev: int) -> str:
    """nvidia-smi -i argument for torch device `dev` (by UUID when known)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        pass
    return str(dev)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- oracle (CPU)

def oracle_worker(args) -> None:
    """Times the float64 oracle on `--samples` samples of the workload (one
    forward + backward per repetition) and prints a JSON line."""
    import numpy as np
    from ffn_block_gb300 import inputs as I
    from oracle import rmx_oracle as O

    shape = I.shape_of(args.config)
    sub = I.Shape(B=args.samples, T=shape.T, D=shape.D, H=shape.H, dtype=shape.dtype)
    arrays = I.to_float64(I.make_inputs(sub))
    p = {k: arrays[k] for k in I.PARAM_NAMES}
    times = []
    for _ in range(args.reps):
        t0 = time.perf_counter()
        O.forward_backward(arrays["x"], arrays["dy"], p)
        times.append(time.perf_counter() - t0)
    print(json.dumps({"samples": args.samples, "rows": args.samples * shape.T, "times": times,
                      "numpy": np.__version__}))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_oracle(config: str, samples: int, reps: int) -> dict:
    cores = host_cores()
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-worker", "--config", config,
           "--samples", str(samples), "--reps", str(reps)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {r.stderr[-2000:]}")
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = cores
    return out


# One sample rule for both CPU legs (the cpu_baseline of the GPU line and the
# reference arm): every oracle call takes the first ORACLE_SAMPLES samples of
# the workload (all of them when the batch is smaller).  numpy's per-token
# matmuls run faster on more rows, so a rate measured on another sample size
# would not be comparable.
ORACLE_SAMPLES = 32


def oracle_samples(config: str) -> int:
    from ffn_block_gb300 import inputs as I
    return max(1, min(I.shape_of(config).B, ORACLE_SAMPLES))


def cpu_baseline(config: str, reps: int) -> dict:
    """Oracle rows/s: `reps` float64 forward+backward calls on the fixed
    sample (the first warms up and is not counted)."""
    samples = oracle_samples(config)
    res = run_oracle(config, samples, reps + 1)
    times = res["times"][1:]
    t = sum(times) / len(times)
    rows = res["rows"]
    return {"value": rows / t, "unit": "rows/s", "cores": res["cores"], "kind": "oracle",
            "sample": f"first {samples} of the workload's samples ({rows} rows) per call, float64 "
                      f"forward+backward in numpy, mean of {len(times)} calls after one warm-up call "
                      f"({t:.2f} s each); BLAS threads = cores"}


# ---------------------------------------------------------------- GPU arm

def dist_setup(n_gpus: int):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, local, ws


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, ws: int) -> float:
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(rows_per_rank: int, ms_max: float, ws: int) -> float:
    """Whole-job throughput: rows of every rank over the slowest rank's time."""
    return rows_per_rank * ws / (ms_max / 1e3)


def workload_name(args, shape) -> str:
    base = WORKLOAD_NAMES.get(args.config, args.config)
    if all(v is None for v in (args.batch, args.tokens, args.dim, args.hidden)):
        return base
    return f"RankMixer block B={shape.B} T={shape.T} D={shape.D} H={shape.H} {shape.dtype} (reduced case)"


def workload_shape(args):
    from ffn_block_gb300 import inputs as I
    d = dict(I.CONFIGS[args.config])
    if args.batch is not None:
        d["B"] = args.batch
    if args.tokens is not None:
        d["T"] = args.tokens
    if args.dim is not None:
        d["D"] = args.dim
    if args.hidden is not None:
        d["H"] = args.hidden
    return I.Shape(**d)


def run_ours(args) -> dict | None:
    import numpy as np
    import torch

    from ffn_block_gb300 import binding as B
    from ffn_block_gb300 import inputs as I
    from ffn_block_gb300.device import RankMixerDevice

    rank, local, ws = dist_setup(args.gpus)
    shape = workload_shape(args)
    arrays = I.make_inputs(shape, seed=I.DEFAULT_SEED + rank)
    torch.cuda.reset_peak_memory_stats()
    blk = RankMixerDevice(shape, arrays, device=f"cuda:{torch.cuda.current_device()}")
    del arrays
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 0)):
        blk.step(stream)
    torch.cuda.synchronize()
    B.check(B.rmx_check(stream), "warm-up")
    memory = {"peak_allocated_bytes": torch.cuda.max_memory_allocated(),
              "saved_bytes": blk.saved_bytes, "workspace_bytes": blk.ws_bytes,
              "note": "every device buffer of the step: inputs, outputs, parameters, gradients, saved, scratch"}
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")

    # Per-kernel breakdown from a separate pass (every launch bracketed by
    # events): it names the dominant kernel.  The timed region below brackets
    # only that kernel's launches, so the step runs as it does unprofiled.
    B.rmx_profile_read()
    B.rmx_profile_select(None)
    B.rmx_profile_enable(True)
    for _ in range(max(1, min(args.steps, 3))):
        flush.zero_()
        blk.step(stream)
    torch.cuda.synchronize()
    B.rmx_profile_enable(False)
    breakdown = B.rmx_profile_read()
    dom = max(breakdown, key=lambda k: breakdown[k][1]) if breakdown else None

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(gpu_selector(torch.cuda.current_device()))
    sampler.start()
    # Keep the GPU under load while the sampler starts (about half a second of
    # untimed steps), so that the clock samples around the short timed region
    # are taken at work, not idle.
    soak_end = time.perf_counter() + 0.5
    while time.perf_counter() < soak_end:
        blk.step(stream)
        torch.cuda.synchronize()
    # Timed region: K steps with no event inside a step (the library's
    # per-kernel timing is off), so the kernels run back to back as in use.
    graph = None
    timed_step = lambda: blk.step(stream)
    if args.graph:
        graph = B.rmx_graph_create(blk.cfg, blk.x, blk.dy, blk.c_params, blk.saved, blk.saved_bytes, blk.y, blk.dx,
                                   blk.c_grads, blk.ws, blk.ws_bytes)
        timed_step = lambda: B.check(B.rmx_graph_launch(graph, stream), "rmx_graph_launch")
        for _ in range(max(args.warmup, 1)):
            timed_step()
        torch.cuda.synchronize()
    launches0 = B.rmx_launch_count()
    # No garbage-collection pause of the Python host loop inside the timed
    # steps (with the launch queue full, the host paces the device).
    gc.collect()
    gc.disable()
    barrier(ws)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                                    # L2 flush, outside the events
        torch.cuda.nvtx.range_push("rmx_step")
        starts[i].record(stream)
        timed_step()
        ends[i].record(stream)
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    gc.enable()
    barrier(ws)
    wall = time.perf_counter() - wall0
    launches = B.rmx_launch_count() - launches0
    if graph is not None:
        B.rmx_graph_destroy(graph)
    # The dominant kernel's own time from a second pass of K steps in which
    # only its launches are bracketed by events (on the stream they are
    # launched on), the others running back to back.
    B.rmx_profile_read()
    B.rmx_profile_select(dom)
    B.rmx_profile_enable(True)
    for i in range(args.steps):
        flush.zero_()
        blk.step(stream)
    torch.cuda.synchronize()
    B.rmx_profile_enable(False)
    B.rmx_profile_select(None)
    clocks = sampler.stop()
    B.check(B.rmx_check(stream), "timed region")
    live = B.rmx_profile_read()  # the dominant kernel, timed inside whole steps
    samples = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = float(np.mean(samples))
    ms_max = reduce_max(ms, ws)
    rows = shape.B * shape.T
    value = aggregate(rows, ms_max, ws)

    # ---- end to end through the host-memory entry point
    e2e = None
    if not args.no_e2e:
        hx = blk.x.cpu().pin_memory()
        hdy = blk.dy.cpu().pin_memory()
        hy = torch.empty_like(hx).pin_memory()
        hdx = torch.empty_like(hx).pin_memory()
        staging = [torch.empty_like(blk.x) for _ in range(4)]
        dev = B.rmx_device_io(*[t.data_ptr() for t in staging])
        host = B.rmx_host_io(hx.data_ptr(), hdy.data_ptr(), hy.data_ptr(), hdx.data_ptr())

        def host_step():
            B.check(B.rmx_step_host(blk.cfg, host, dev, blk.c_params, blk.c_grads, blk.saved,
                                    blk.saved_bytes, blk.ws, blk.ws_bytes, stream), "rmx_step_host")

        for _ in range(max(args.warmup, 1)):
            host_step()
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        gc.collect()
        gc.disable()
        barrier(ws)
        for i in range(args.steps):
            flush.zero_()
            es[i].record(stream)
            host_step()
            ee[i].record(stream)
        torch.cuda.synchronize()
        gc.enable()
        B.check(B.rmx_check(stream), "e2e")
        e_samples = [a.elapsed_time(b) for a, b in zip(es, ee)]
        e_ms = reduce_max(float(np.mean(e_samples)), ws)
        nbytes = hx.numel() * hx.element_size()
        e2e = {"value": aggregate(rows, e_ms, ws), "unit": "rows/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": 2 * nbytes, "d2h_bytes_per_step": 2 * nbytes,
               "samples_ms": [round(v, 4) for v in e_samples],
               # value is the mean (whole-job throughput); the median shows
               # a step's time without the host's occasional stalls
               "median_ms": round(float(np.median(e_samples)), 4)}

    if rank != 0:
        return None

    # ---- roofline of the dominant kernel and of the whole step
    peaks, peak_src = load_peaks()
    kernels = {k: {"launches": n, "ms_total": t, "ms_per_launch": t / max(n, 1)} for k, (n, t) in breakdown.items()}
    total_ms = sum(v["ms_total"] for v in kernels.values()) or 1.0
    for v in kernels.values():
        v["share"] = v["ms_total"] / total_ms
    if dom is not None and dom in live:
        n_live, t_live = live[dom]
        kernels[dom]["ms_per_launch_timed_region"] = t_live / max(n_live, 1)
    gflops, rbytes = gemm_flops_per_launch(shape), row_bytes_per_launch(shape)
    burst, sustained, peak_name = tensor_peak(peaks, clocks)
    roofline = None
    if dom is not None:
        per = kernels[dom].get("ms_per_launch_timed_region", kernels[dom]["ms_per_launch"]) / 1e3
        if dom.endswith(".ffma") and dom.split(".")[0] in gflops:
            ach = gflops[dom.split(".")[0]] / per / 1e12
            roofline = {"kernel": dom, "bound": "alu", "achieved": ach, "peak": FFMA_TFLOPS, "unit": "TFLOP/s",
                        "frac": ach / FFMA_TFLOPS,
                        "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 FLOP per FMA x 2.07 GHz",
                        "traffic": profiled_traffic(dom, args.config)}
        elif dom in gflops:
            ach = gflops[dom] / per / 1e12
            tensor = shape.dtype != "f32"
            peak = (burst if peak_name == "burst" else sustained) if tensor else None
            roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                        "frac": (ach / peak) if peak else None,
                        "frac_of_sustained": (ach / sustained) if tensor else None,
                        "peak_source": f"{peak_src} bf16_tflops{'' if peak_name == 'burst' else '_sustained'} "
                                       f"({peak_name}: {PEAK_RULE}; fp16 at the bf16 rate, nominal ratio 1)",
                        "traffic": profiled_traffic(dom, args.config)}
        else:
            ach = rbytes.get(dom, 0.0) / per / 1e9
            roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": ach / peaks["hbm_gbs"], "peak_source": f"{peak_src} hbm_gbs",
                        "traffic": profiled_traffic(dom, args.config)}
    tpeak = burst if peak_name == "burst" else sustained
    for k, v in kernels.items():
        per = v["ms_per_launch"] / 1e3
        if k.split(".")[0] in gflops and shape.dtype == "f32":
            v["gflops"] = gflops[k.split(".")[0]] / per / 1e9   # CUDA-core (FFMA) contraction
        elif k in gflops and shape.dtype != "f32":
            v["tflops"] = gflops[k] / per / 1e12
            v["frac_of_peak"] = v["tflops"] / tpeak
        elif k in rbytes:
            v["gbs"] = rbytes[k] / per / 1e9
            v["frac_of_peak"] = v["gbs"] / peaks["hbm_gbs"]
    t_mem = min_bytes_per_step(shape) / (peaks["hbm_gbs"] * 1e9)

    def step_frac(tflops):
        # strict fp32: the contractions run on the CUDA cores (FFMA peak)
        t_compute = flops_per_step(shape) / ((tflops if shape.dtype != "f32" else FFMA_TFLOPS) * 1e12)
        return max(t_compute, t_mem), t_compute

    t_roof, t_compute = step_frac(tpeak)
    step_roofline = {"bound": ("tensor" if shape.dtype != "f32" else "alu") if t_compute >= t_mem else "hbm",
                     "t_ms": t_roof * 1e3,
                     "flops": flops_per_step(shape), "min_bytes": min_bytes_per_step(shape),
                     "frac": (t_roof * 1e3) / ms,
                     "frac_of_sustained": step_frac(sustained)[0] * 1e3 / ms,
                     "peaks": (f"{peak_src}: {peak_name} bf16 {tpeak} TFLOP/s ({PEAK_RULE}), "
                               if shape.dtype != "f32" else f"derived FFMA {FFMA_TFLOPS:.1f} TFLOP/s, ")
                              + f"hbm_gbs={peaks['hbm_gbs']}"}

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"f32": "f32", "bf16": "bf16", "f16": "f16"}[shape.dtype],
        "data": "synthetic (seeded he-uniform weights, standard-normal x and dy)",
        "config": {"workload": workload_name(args, shape), "B": shape.B, "T": shape.T,
                   "D": shape.D, "H": shape.H, "storage": shape.dtype, "parallelism": f"replicas x{ws}",
                   "l2": "flushed before every step (outside the timed region)",
                   "launch": "CUDA graph replay" if args.graph else "rmx_forward + rmx_backward"},
        "step_roofline": step_roofline,
        "roofline": roofline,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches,
        "wall_s": wall,
        "samples_ms": samples,
        "memory": memory,
        "kernels": kernels,
        "kernels_note": "per-kernel times from a separate pass with every launch bracketed by events; the "
                        "timed region has no event inside a step; the dominant kernel's "
                        "ms_per_launch_timed_region comes from a further pass of K steps in which only its "
                        "launches are bracketed",
    }
    return line


def run_reference(args) -> dict | None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from ffn_block_gb300 import inputs as I
    shape = I.shape_of(args.config)
    samples = oracle_samples(args.config)
    res = run_oracle(args.config, samples, args.steps + args.warmup)
    times = res["times"][args.warmup:] or res["times"]
    t = sum(times) / len(times)
    rows = samples * shape.T
    value = rows / t
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": 1,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAMES.get(args.config, args.config), "B": shape.B, "T": shape.T,
                   "D": shape.D, "H": shape.H, "storage": shape.dtype},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": res["cores"], "kind": "oracle",
                         "sample": f"first {samples} of the workload's samples ({rows} rows) per step, "
                                   f"float64 forward+backward in numpy; BLAS threads = cores"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def unfused_forward_backward(x, dy, p):
    """The block as a plain PyTorch eager composition (one op per step of the
    page's "Exact computation" section, autograd for the backward): the
    unfused per-op sequence the fused path is compared with.  x, dy [B,T,D]
    and the parameters in their page layouts, all on one device and dtype.
    Returns y, dx and the parameter gradients."""
    import torch
    import torch.nn.functional as F
    B_, T, D = x.shape
    H = p["lnx_w"].shape[0]
    C = D // T
    x = x.detach().requires_grad_(True)
    q = {k: v.detach().requires_grad_(True) for k, v in p.items()}
    a0 = F.layer_norm(x, (D,), q["gamma0"], q["beta0"], 1e-3)
    mixed = a0.reshape(B_, T, T, C).transpose(1, 2).reshape(B_, T, D)      # swap the two T axes
    out1 = F.layer_norm(mixed + x, (D,), q["gamma1"], q["beta1"], 1e-3)
    Z = torch.baddbmm(q["b1"].unsqueeze(1), out1.transpose(0, 1), q["w1"])  # [T, B, 2H]
    U, G = Z.split(H, dim=-1)
    hidden = F.layer_norm(U, (H,), q["lnx_w"], q["lnx_b"], 1e-5) * F.silu(
        F.layer_norm(G, (H,), q["lng_w"], q["lng_b"], 1e-5))
    out2 = torch.baddbmm(q["bout"].unsqueeze(1), hidden, q["wout"])        # [T, B, D]
    y = F.layer_norm(out1 + out2.transpose(0, 1), (D,), q["gamma2"], q["beta2"], 1e-3)
    y.backward(dy)
    return y.detach(), x.grad, {k: v.grad for k, v in q.items()}


def run_unfused(args) -> dict | None:
    import numpy as np
    import torch

    from ffn_block_gb300 import inputs as I
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    shape = workload_shape(args)
    arrays = I.make_inputs(shape, seed=I.DEFAULT_SEED)
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[shape.dtype]
    dev = torch.device("cuda")
    torch.cuda.reset_peak_memory_stats()
    x = torch.from_numpy(np.ascontiguousarray(arrays["x"], dtype=np.float32)).to(dev, dt)
    dy = torch.from_numpy(np.ascontiguousarray(arrays["dy"], dtype=np.float32)).to(dev, dt)
    p = {k: torch.from_numpy(np.ascontiguousarray(arrays[k], dtype=np.float32)).to(dev, dt) for k in I.PARAM_NAMES}
    del arrays
    for _ in range(max(args.warmup, 0)):
        unfused_forward_backward(x, dy, p)
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stream = torch.cuda.current_stream()
    for i in range(args.steps):
        flush.zero_()
        torch.cuda.nvtx.range_push("rmx_step")
        starts[i].record(stream)
        unfused_forward_backward(x, dy, p)
        ends[i].record(stream)
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)]))
    rows = shape.B * shape.T
    return {"impl": "unfused", "metric": METRIC, "value": rows / (ms / 1e3), "unit": "rows/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": shape.dtype, "data": "synthetic (the same seeded inputs as the fused path)",
            "config": {"workload": workload_name(args, shape), "B": shape.B, "T": shape.T, "D": shape.D,
                       "H": shape.H, "storage": shape.dtype},
            "memory": {"peak_allocated_bytes": peak}}


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_worker:
        oracle_worker(args)
        return
    if args.impl in ("reference", "unfused"):
        line = run_reference(args) if args.impl == "reference" else run_unfused(args)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line = run_ours(args)
    if line is None:
        return
    if not args.no_cpu_baseline and int(os.environ.get("WORLD_SIZE", "1")) == 1:
        try:
            line["cpu_baseline"] = cpu_baseline(args.config, args.cpu_reps)
        except Exception as e:  # report, do not hide the GPU number
            line["cpu_baseline"] = {"value": None, "error": str(e)[:300]}
    elif int(os.environ.get("WORLD_SIZE", "1")) > 1:
        line["cpu_baseline"] = None
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
