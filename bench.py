"""Throughput of the fused linear cross-entropy forward + backward on GB300.

One step = one flce_forward_backward call over the whole batch (every chunk:
logits GEMM with its log-sum-exp epilogue, combine, dlogits, dx GEMM, dW
GEMM, loss reduction). Default workload: the Llama-3-shaped batch,
N = 16384 tokens (4 x 4096), H = 4096, V = 128256, bf16, Zipf(1.1) targets,
5% ignored. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on the host cores.
Under torchrun each rank runs an independent replica of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FLCE fwd+bwd tokens/s & % of bf16 tensor peak (6·N·H·V FLOPs); peak HBM GB"
UNIT = "tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HBM_BOUND = {"dlogits_inplace", "lse_combine", "combine_dlogits", "dx_split_reduce", "count_valid",
             "loss_finalize", "device_result"}
ALU_BOUND = {"simt_gemm_f32"}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="llama3_bf16")
    p.add_argument("--chunk", type=int, default=0)
    p.add_argument("--budget-gib", type=float, default=0.0)
    p.add_argument("--dlogits", choices=["auto", "inplace", "recompute", "slabs"], default="auto")
    p.add_argument("--cta", choices=["auto", "single", "pair", "wide"], default="auto",
                   help="GEMM tile shape: one CTA per 128x256 tile, CTA pairs per 256x256, "
                        "or CTA pairs per 256x512 sharing A (wide)")
    p.add_argument("--backward", choices=["auto", "separate", "one_launch"], default="auto",
                   help="dx and dW GEMMs of a chunk in two launches or one (CTA pairs)")
    p.add_argument("--token-parallel", action="store_true",
                   help="shard the batch's tokens over the ranks (NEXT-3): each step all-reduces "
                        "the non-ignored token count, then dW and the loss; strong scaling. "
                        "Default: independent replicas")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle sample")
    return p.parse_args()


# ------------------------------------------------------------ distributed

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    # under torchrun the token-parallel mode joins its rendezvous even with one
    # rank (an explicit tcp:// group there would wait on the launcher's store)
    launched = "MASTER_PORT" in os.environ and "RANK" in os.environ
    if ws > 1 or (args.impl == "ours" and args.token_parallel and launched):
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend, rank=rank, world_size=ws)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, value: float, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ws, tokens_per_rank: int, ms_local: float, device=None):
    """Whole-job throughput of independent replicas: every rank processed
    tokens_per_rank tokens; the job took as long as the slowest rank."""
    ms_max = max_over_ranks(ws, ms_local, device)
    return ms_max, ws * tokens_per_rank / (ms_max / 1e3)


L2_BYTES = 129 * 10**6   # GB300 L2


def l2_note(w_bytes: int, buf_bytes: int) -> str:
    """How the timed steps stand to L2: every step streams W and the chunk
    buffer, so the inputs are larger than L2 when either is."""
    size = f"W {w_bytes / 1e9:.3g} GB, chunk buffer {buf_bytes / 1e9:.3g} GB"
    if max(w_bytes, buf_bytes) > L2_BYTES:
        return f"inputs larger than L2 ({size}; L2 129 MB)"
    return f"inputs smaller than L2 ({size}; L2 129 MB): steps may hit in L2, no flush"


# The pages' own figures for this shape, other hardware: context, not targets.
PAGE_CONTEXT = {
    "full_logits_bf16_gb": 4.20,
    "standard_pytorch_loss_peak_gb": 36.02,
    "fused_triton_loss_peak_gb": 5.04,
    "hardware": "A100 (FLCE page, section on memory measured at 16,384 tokens)",
    "strategies_16b_model_128k_context": {
        "full logits": "110+ GB, 1.0x throughput", "chunked loss, 8K chunks": "14 GB, 0.85x",
        "LM-head gradient checkpointing": "4 GB, 0.70x", "fused Triton loss": "6 GB, 1.05x",
        "hardware": "A100/H100 class, unspecified"},
}

# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        after = False
        if not rows:
            # a timed region shorter than nvidia-smi's start-up and sampling
            # interval: one sample taken right after it, marked as such
            try:
                out = subprocess.run(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=10).stdout
                rows = [[p.strip() for p in line.split(",")] for line in out.splitlines()
                        if len(line.split(",")) >= 9]
                after = bool(rows)
            except (OSError, subprocess.SubprocessError):
                rows = []
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        res = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
               "samples": 0 if after else len(rows),
               "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                                  default=None)}
        if after:
            res["note"] = "timed region shorter than the sampling interval: one sample right after it"
        return res


# ------------------------------------------------------------------- peaks

def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_hash() -> str:
    from linear_cross_entropy_token_gb300.build import source_hash
    return source_hash()


def traffic_for(kernel: str, workload: str, chunk: int, dlogits: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or
    None if there is none for this workload, chunk and dlogits mode, or the
    kernels changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash():
        return None
    k = d.get("kernels", {}).get(kernel)
    if (not k or d.get("workload") != workload or d.get("chunk") != chunk
            or d.get("dlogits", "inplace") != dlogits):
        return None
    return k.get("dram_bytes_per_launch")


# ------------------------------------------------------------- cpu oracle

def blas_threads() -> int:
    """Threads numpy's BLAS runs the oracle's products on."""
    try:
        from threadpoolctl import threadpool_info
        n = [p["num_threads"] for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def oracle_sample_rate(w, target_s: float, max_tokens: int = 4096):
    """The fp64 oracle on the first n tokens of the workload (all of W), n
    grown until one run takes about target_s seconds; a workload too small
    for that is run whole, repeatedly, for about target_s seconds. Returns
    tokens/s, tokens per run, seconds, cores, runs."""
    import numpy as np
    import oracle
    Wd = w.W_f64()
    cores = blas_threads()
    max_tokens = min(max_tokens, w.N)
    n = min(8, max_tokens)
    while True:
        xs = w.x_f64(np.arange(n))
        t0 = time.perf_counter()
        oracle.flce_reference(xs, Wd, w.t[:n], w.ignore_index)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5:
            return n / dt, n, dt, cores, 1
        if n >= max_tokens:
            runs = max(1, int(target_s / max(dt, 1e-4)))
            t0 = time.perf_counter()
            for _ in range(runs):
                oracle.flce_reference(xs, Wd, w.t[:n], w.ignore_index)
            dt = time.perf_counter() - t0
            return n * runs / dt, n, dt, cores, runs
        n = min(max_tokens, max(n * 2, int(n * target_s / max(dt, 1e-3))))


# -------------------------------------------------------------------- main

def run_reference(args, ws, rank):
    """--impl reference: the fp64 CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    import workloads
    w = workloads.make(args.config)
    Wd = w.W_f64()
    # each step a sample sized so that warm-up plus timed steps take ~90 s
    per_step = max(0.2, min(args.cpu_seconds, 6.0, 90.0 / max(1, args.steps + args.warmup)))
    _, n, dt, cores, _ = oracle_sample_rate(w, target_s=per_step)
    xs = w.x_f64(np.arange(n))
    ts = w.t[:n]
    for _ in range(args.warmup):
        oracle.flce_reference(xs, Wd, ts, w.ignore_index)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.flce_reference(xs, Wd, ts, w.ignore_index)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = (f"first {n} tokens of {args.config} (N={w.N}, H={w.H}, V={w.V}) per step, "
              f"float64 numpy oracle, all of W")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.config, "N": w.N, "H": w.H, "V": w.V,
                                            "sample_tokens": n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, ws, rank, local):
    import numpy as np
    import torch

    import workloads
    from linear_cross_entropy_token_gb300 import FLCE

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workloads.make(args.config)
    N, H, V = w.N, w.H, w.V
    if args.chunk == 0 and w.spec.chunk:
        args.chunk = w.spec.chunk   # a configuration that names its chunk (tiny fp32: 64) runs it
    bf16 = w.x.dtype == np.uint16   # bf16 configs hold RNE-rounded bit patterns
    if bf16:
        x_h = torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16)
        W_h = torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16)
    else:
        x_h = torch.from_numpy(w.x)
        W_h = torch.from_numpy(w.W)
    esize = x_h.element_size()
    t_h = torch.from_numpy(w.t)
    x, W, t = x_h.to(dev), W_h.to(dev), t_h.to(dev)
    dx = torch.empty_like(x)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    budget = int(args.budget_gib * (1 << 30))
    h = FLCE("bf16" if bf16 else "fp32", local, hbm_budget_bytes=budget, dlogits_mode=args.dlogits, cta=args.cta,
             backward=args.backward)
    stream = torch.cuda.current_stream(dev)

    free0, _ = torch.cuda.mem_get_info(dev)
    h.forward_backward(x, W, t, chunk=args.chunk, dx=dx, dW=dW)
    free1, _ = torch.cuda.mem_get_info(dev)
    plan = h.last_plan()
    # the timed steps are enqueued with the sync-free entry: each step's loss
    # lands in device memory and is read after the timed region, so a stall
    # of the host thread cannot leave the GPU idle between steps
    loss_buf = torch.empty(max(1, args.steps), dtype=torch.float32, device=dev)
    nv_buf = torch.empty((), dtype=torch.int32, device=dev)
    for _ in range(max(0, args.warmup - 1)):
        h.forward_backward_async(x, W, t, chunk=args.chunk, loss=loss_buf[0], n_valid=nv_buf,
                                 dx=dx, dW=dW)
    torch.cuda.synchronize(dev)
    h.async_status()

    def run_steps(n):
        for i in range(n):
            h.forward_backward_async(x, W, t, chunk=args.chunk, loss=loss_buf[i], n_valid=nv_buf,
                                     dx=dx, dW=dW)

    def timed(fn):
        """Device time per step of fn() over args.steps steps, CUDA events on the
        call stream, a barrier and a synchronize on both sides."""
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        return e0.elapsed_time(e1) / args.steps

    # ---------------------------------------------------- timed region
    # the steps as a caller runs them: no per-launch events
    launches0 = h.launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    ms = timed(lambda: run_steps(args.steps))
    clk = clocks.stop()
    h.async_status()   # raises if any timed step recorded a device-side error
    losses = loss_buf[:args.steps].tolist()
    launches = h.launch_count() - launches0

    # the same steps with CUDA events around every launch (on the stream each
    # kernel runs on): the per-kernel times of the roofline; the events cost a
    # few microseconds per launch, visible only on the smallest workloads
    h.set_profiling(True)
    h.profile_reset()
    ms_events = timed(lambda: run_steps(args.steps))
    prof = h.profile()
    h.set_profiling(False)
    h.async_status()

    # one call captured in a CUDA graph and replayed: the host's launch work
    # leaves the step (the call allocates nothing once its workspace exists)
    ms_graph = None
    if ws == 1:
        try:
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    h.forward_backward_async(x, W, t, chunk=args.chunk, loss=loss_buf[0],
                                             n_valid=nv_buf, dx=dx, dW=dW)
            stream.wait_stream(cap)
            g.replay()
            torch.cuda.synchronize(dev)

            def replays():
                for _ in range(args.steps):
                    g.replay()
            ms_graph = timed(replays)
            h.async_status()
            del g
        except RuntimeError as err:   # reported, not fatal: the eager steps stand
            ms_graph = f"not measured: {err}"[:200]
    tokens = N
    ms_max, value = aggregate(ws, tokens, ms, dev if ws > 1 else None)
    flops = 6.0 * N * H * V
    tflops = flops / (ms_max / 1e3) / 1e12
    peaks, peaks_kind = load_peaks()
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    peak_clk = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")

    # dominant kernel and its roofline; the slab backward runs its dx and dW
    # GEMMs side by side on two streams, so their event times overlap and the
    # dominant kernel is the main-stream one with the most time
    side_stream = {"gemm_dw"} if (plan["dlogits"] == "slabs" or plan["dw_beside_dx"]) else set()
    dom = max(((k, v) for k, v in prof.items() if k not in side_stream), key=lambda kv: kv[1]["total_ms"])
    name, pk = dom
    per_launch_ms = pk["total_ms"] / pk["launches"]
    if name in HBM_BOUND:
        achieved = pk["bytes"] / pk["launches"] / (per_launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    elif name in ALU_BOUND:
        # fp32 CUDA-core FMAs: SMs x 128 FP32 lanes x 2 FLOP x the maximum SM clock
        achieved = pk["flops"] / pk["launches"] / (per_launch_ms / 1e3) / 1e12
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = sms * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        achieved = pk["flops"] / pk["launches"] / (per_launch_ms / 1e3) / 1e12
        # the kernel is timed alone (per-launch events within a step of tens
        # of ms), so the burst peak applies; the sustained one, measured over
        # seconds under the power cap, is reported beside it
        roof = {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                "peak_sustained": sustained, "frac_sustained": achieved / sustained}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_for(name, args.config, plan["chunk"], plan["dlogits"])
    roof["kernel"] = name
    roof["timing"] = ("per-launch CUDA events on each kernel's stream over a second run of the "
                      "timed steps (the headline run records none)")
    if side_stream:
        roof["note"] = ("the dx and dW GEMMs overlap on two streams: their per-launch times "
                        "include the time they share the GPU")
    roof["peak_source"] = {"tensor": f"{peaks_kind} (burst bf16; sustained beside it)",
                           "hbm": f"{peaks_kind} (hbm copy)",
                           "alu": "derived: SMs x 128 fp32 lanes x 2 x max SM clock"}[roof["bound"]]
    kernels = {k: {"launches": v["launches"], "ms_per_launch": v["total_ms"] / v["launches"],
                   "share": v["total_ms"] / sum(q["total_ms"] for q in prof.values()),
                   ("tflops" if k not in HBM_BOUND else "gbs"):
                       (v["flops"] / v["total_ms"] / 1e9 if k not in HBM_BOUND
                        else v["bytes"] / v["total_ms"] / 1e6)}
               for k, v in prof.items()}

    # ---------------------------------------------- end to end, host buffers
    e2e = None
    if not args.no_e2e:
        xp, Wp, tp = x_h.pin_memory(), W_h.pin_memory(), t_h.pin_memory()

        def sync_steps():
            for _ in range(args.steps):
                h.forward_backward_host(xp, Wp, tp, chunk=args.chunk, dx=dx, dW=dW)

        def pipelined_steps():
            # every step copies its inputs in and reads its loss back; the
            # copies of step k+1 overlap the compute of step k
            prev, _, _ = h.submit_host(xp, Wp, tp, chunk=args.chunk, dx=dx, dW=dW)
            for _ in range(args.steps - 1):
                cur, _, _ = h.submit_host(xp, Wp, tp, chunk=args.chunk, dx=dx, dW=dW)
                h.wait(prev)
                prev = cur
            h.wait(prev)

        sync_steps()
        pipelined_steps()
        sync_ms = timed(sync_steps)
        pipe_ms = timed(pipelined_steps)
        ems, evalue = aggregate(ws, tokens, pipe_ms, dev if ws > 1 else None)
        sync_max, _ = aggregate(ws, tokens, sync_ms, dev if ws > 1 else None)

        # the copies alone, from CUDA events on the stream that runs them, in
        # a further run of each form with the library's profiling on
        def copy_time(fn):
            h.set_profiling(True)
            h.profile_reset()
            fn()
            torch.cuda.synchronize(dev)
            c = h.profile().get("h2d_copy")
            h.set_profiling(False)
            h.profile_reset()
            if not c or not c["launches"]:
                return None, None
            return c["total_ms"] / c["launches"], c["bytes"] / c["total_ms"] / 1e6
        copy_pipe_ms, copy_pipe_gbs = copy_time(pipelined_steps)
        copy_sync_ms, copy_sync_gbs = copy_time(sync_steps)
        e2e = {"value": evalue, "unit": UNIT,
               "h2d_bytes_per_step": int((x_h.numel() + W_h.numel()) * esize + t_h.numel() * 8),
               "d2h_bytes_per_step": 4 * 16, "ms_per_step": ems,
               "path": "flce_submit_host / flce_wait: pinned host x, W, t copied in every step on "
                       "the library's copy stream (overlapping the previous step's compute); "
                       "the step's control words, with its loss, read back",
               "sync_ms_per_step": sync_max,
               "sync_path": "flce_forward_backward_host: copy in, compute, read back, one after another",
               "copy_ms_per_step": {"beside_compute": copy_pipe_ms, "alone": copy_sync_ms},
               "copy_gbs": {"beside_compute": copy_pipe_gbs, "alone": copy_sync_gbs},
               "copy_timing": "CUDA events around each step's host-to-device copies on the stream "
                              "that runs them (the copy stream when pipelined), in a further run of "
                              "each form with per-launch profiling on"}

    # --------------------------------------------------- cpu oracle sample
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, n, dt, cores, runs = oracle_sample_rate(w, args.cpu_seconds)
        what = (f"the first {n} tokens of the workload" if n < N else f"the whole workload ({n} tokens)")
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{what} with all of W, float64 numpy oracle, "
                         + (f"{runs} runs, " if runs > 1 else "") + f"{dt:.1f} s"}

    h.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if bf16 else "f32", "data": "synthetic",
        "ms_per_step_with_kernel_events": ms_events,
        "ms_per_step_graph_replay": ms_graph,
        "config": {"workload": args.config, "N": N, "H": H, "V": V, "chunk": plan["chunk"],
                   "num_chunks": plan["num_chunks"], "dx_splits": plan["dx_splits"],
                   "dlogits": plan["dlogits"],
                   "gemm_tiles": ({(128, 256): "128x256, one CTA", (256, 256): "256x256, CTA pairs",
                                   (256, 512): "256x512, CTA pairs sharing A through the collector"}[
                                      (plan["tile_m"], plan["tile_n"])]
                                  if bf16 else "fp32 CUDA-core GEMMs"),
                   "backward_gemms": ("one launch, work units handed out dynamically (dx first)"
                                      if plan["backward_one_launch"] else "two launches"),
                   "targets": w.spec.targets, "ignore_frac": float(w.spec.ignore_frac),
                   "l2": l2_note(V * H * esize, plan["logits_bytes"]),
                   "parallelism": "replicas" if ws > 1 else "single"},
        "tflops": tflops, "frac_of_bf16_peak": tflops / burst,
        "frac_of_bf16_peak_sustained": tflops / sustained,
        "peak_source": peaks_kind,
        "peak_clocks": {"burst": "cuBLAS 8192^3 bf16, best of 10 launches",
                        "sustained": (f"cuBLAS back to back for seconds, SM clock median {peak_clk} MHz"
                                      if peak_clk else "cuBLAS back to back for seconds"),
                        "this_run_sm_mhz": clk.get("sm_mhz")},
        "peak_extra_hbm_gb": plan["workspace_bytes"] / 1e9,
        "peak_extra_hbm_measured_gb": max(0, free0 - free1) / 1e9,
        "full_logits_gb": N * V * 2 / 1e9,
        "page_context": PAGE_CONTEXT if (N, H, V) == (16384, 4096, 128256) else None,
        "loss": losses[-1] if losses else None,
        "gpu_launches": launches,
        "kernels": kernels,
        "roofline": roof,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def aggregate_sharded(ws, batch_tokens: int, ms_local: float, device=None):
    """Whole-job throughput of one token-sharded batch: the batch's tokens
    once, over the slowest rank's time."""
    ms_max = max_over_ranks(ws, ms_local, device)
    return ms_max, batch_tokens / (ms_max / 1e3)


def run_token_parallel(args, ws, rank, local):
    """--token-parallel: one batch split by tokens over the ranks; every step
    is the token_parallel wrapper's count all-reduce, the rank's fused call
    with the batch's divisor, and the all-reduces of dW and the loss."""
    import socket

    import numpy as np
    import torch
    import torch.distributed as dist

    import workloads
    from linear_cross_entropy_token_gb300 import FLCE
    from linear_cross_entropy_token_gb300.token_parallel import (shard_bounds,
                                                                 token_parallel_forward_backward)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    own_group = not dist.is_initialized()
    if own_group:   # one plain process: the collectives run over a one-rank NCCL group
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                                device_id=dev)
    w = workloads.make(args.config)
    if args.chunk == 0 and w.spec.chunk:
        args.chunk = w.spec.chunk
    a, b = shard_bounds(w.N, ws, rank)
    bf16 = w.x.dtype == np.uint16
    xs = w.x[a:b]
    if bf16:
        x = torch.from_numpy(np.ascontiguousarray(xs).view(np.int16)).view(torch.bfloat16).to(dev)
        W = torch.from_numpy(w.W.view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        x = torch.from_numpy(np.ascontiguousarray(xs)).to(dev)
        W = torch.from_numpy(w.W).to(dev)
    t = torch.from_numpy(np.ascontiguousarray(w.t[a:b])).to(dev)
    dx = torch.empty_like(x)
    dW = torch.empty((w.V, w.H), dtype=torch.float32, device=dev)
    h = FLCE("bf16" if bf16 else "fp32", local, hbm_budget_bytes=int(args.budget_gib * (1 << 30)),
             dlogits_mode=args.dlogits, cta=args.cta, backward=args.backward)
    stream = torch.cuda.current_stream(dev)

    def step():
        return token_parallel_forward_backward(h, x, W, t, chunk=args.chunk, dx=dx, dW=dW)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    h.async_status()
    plan = h.last_plan()

    def timed():
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            loss = step()[0]
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        return e0.elapsed_time(e1) / args.steps, loss

    launches0 = h.launch_count()
    clocks = ClockSampler(local)
    clocks.start()
    ms, loss = timed()
    clk = clocks.stop()
    h.async_status()
    launches = h.launch_count() - launches0
    h.set_profiling(True)
    h.profile_reset()
    ms_events, _ = timed()
    prof = h.profile()
    h.set_profiling(False)
    ms_max, value = aggregate_sharded(ws, w.N, ms, dev)
    flops = 6.0 * w.N * w.H * w.V
    tflops = flops / (ms_max / 1e3) / 1e12
    peaks, peaks_kind = load_peaks()
    name, pk = max(((k, v) for k, v in prof.items() if k != "gemm_dw" or not plan["dw_beside_dx"]),
                   key=lambda kv: kv[1]["total_ms"])
    achieved = pk["flops"] / pk["total_ms"] / 1e9 if name not in HBM_BOUND else pk["bytes"] / pk["total_ms"] / 1e6
    roof_peak = peaks["hbm_gbs"] if name in HBM_BOUND else peaks["bf16_tflops"]
    loss_v = float(loss.item())
    h.close()
    if own_group:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "bf16" if bf16 else "f32", "data": "synthetic",
        "ms_per_step_with_kernel_events": ms_events,
        "config": {"workload": args.config, "N": w.N, "H": w.H, "V": w.V, "tokens_per_rank": b - a,
                   "chunk": plan["chunk"], "num_chunks": plan["num_chunks"], "dlogits": plan["dlogits"],
                   "l2": l2_note(w.V * w.H * x.element_size(), plan["logits_bytes"]),
                   "parallelism": f"token-parallel over {ws} rank(s): all-reduce of n_valid, then of "
                                  "dW and the loss shares (NCCL)"},
        "tflops": tflops, "frac_of_bf16_peak": tflops / peaks["bf16_tflops"], "peak_source": peaks_kind,
        "loss": loss_v, "gpu_launches": launches,
        "roofline": {"bound": "hbm" if name in HBM_BOUND else "tensor", "achieved": achieved,
                     "peak": roof_peak, "unit": "GB/s" if name in HBM_BOUND else "TFLOP/s",
                     "frac": achieved / roof_peak, "traffic": None, "kernel": name,
                     "timing": "per-launch CUDA events over a second run of the timed steps"},
        "clocks": clk,
        "e2e": None,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.token_parallel:
        run_token_parallel(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
