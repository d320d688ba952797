#!/usr/bin/env python
"""Benchmark of the Stable LatentMoE layer forward (QB routing) on GB300.

One step = one moe_latent_forward over one batch of the workload (router,
Quantile Balancing, top-k, dispatch, latent down-projection, grouped SiTU-GLU
experts, combine + RMSNorm, up-projection + merged shared expert).  Prints one
JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload prefill|decode|prefill_mxfp4|decode_mxfp4|route_qb|route_qb_gs]

The default workload is the largest single-GPU configuration: the K3-shape
layer at prefill size (16384 tokens, bf16).

Multi-GPU (torchrun): every rank runs an independent replica on its own batch
(the path has no data exchange on one replica); value = all ranks' tokens /
max-over-ranks time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import qb_inputs as QI  # noqa: E402

WORKLOADS = {"decode": QI.DECODE, "prefill": QI.PREFILL, "prefill_mxfp4": QI.PREFILL_MXFP4,
             "decode_mxfp4": QI.DECODE_MXFP4, "route_qb": QI.ROUTE_QB, "route_qb_gs": QI.ROUTE_QB}
ROUTE_WORKLOADS = ("route_qb", "route_qb_gs")
METRIC = "MoE-layer fwd routed tokens/s on 1 GB300; % of HBM / tensor-core roofline"
ROUTE_METRIC = "QB routing tokens/s on 1 GB300; % of HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha256():
    """Hash of the tensor-core kernel's code (comments and whitespace removed,
    so that a recorded traffic figure survives edits of comments only)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "tc_ptx.cuh"):
        with open(os.path.join(ROOT, "quantile_balanced_routing_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    """Per-launch DRAM bytes of `kernel` on `workload` from an ncu summary under
    profiles/ (a `traffic: <kernel> <workload> <bytes>` line), if the summary
    was taken with the current kernel source; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = kernel_source_sha256()
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        file_sha, found = None, None
        with open(os.path.join(pdir, name)) as f:
            for line in f:
                if line.startswith("kernel_source_sha256:"):
                    file_sha = line.split(":", 1)[1].strip()
                elif line.startswith("traffic:"):
                    parts = line.split(":", 1)[1].split()
                    if len(parts) == 3 and parts[0] == kernel and parts[1] == workload:
                        found = int(parts[2])
        if found is not None and file_sha == sha:
            return found
    return None


def weight_bytes_per_elt(shape):
    return (0.5 + 1.0 / 32.0) if shape.wfmt == "mxfp4" else (4 if shape.wfmt == "f32" else 2)


def stage_work(shape, T):
    """Algorithmic (bytes, flops) per launch of each stage: what the method
    must move and compute once, ignoring re-reads."""
    a = 4 if shape.dtype == "f32" else 2
    wb = weight_bytes_per_elt(shape)
    n, k, d, L, m, ms = shape.n, shape.k, shape.d, shape.latent, shape.m, shape.m_s
    R = T * k
    # grouped expert work touches every expert that receives a token; with QB
    # every expert does when T*k >= n
    used = min(n, R)
    w = {
        "router": (n * d * a + T * d * a + T * n * 4, 2 * T * n * d),
        "expert_gate_up": (used * 2 * m * L * wb + T * L * a + R * m * a, 2 * R * L * 2 * m),
        "expert_down": (used * L * m * wb + R * m * a + R * L * a, 2 * R * m * L),
        "xside_gemm": ((L + 2 * ms) * d * a + T * d * a + T * (L + ms) * a, 2 * T * d * (L + 2 * ms)),
        "down_proj": (L * d * a + T * d * a + T * L * a, 2 * T * d * L),
        "shared_gate_up": (2 * ms * d * a + T * d * a + T * ms * a, 2 * T * d * 2 * ms),
        "combine_rmsnorm": (R * L * a + T * L * a + R * 8, 4 * R * L),
        "up_proj_shared": (d * (L + ms) * a + T * (L + ms) * a + T * d * a, 2 * T * d * (L + ms)),
    }
    return w


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Max of x over the ranks (NCCL on GPUs, gloo on CPU)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank, ms_local, world):
    """Whole-job routed tokens/s of `world` independent replicas: all ranks'
    tokens over the slowest rank's time (weak scaling)."""
    ms = max_over_ranks(ms_local, world)
    return tokens_per_rank * world / (ms * 1e-3), ms


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------

class OracleSample:
    """The CPU oracle on a bounded sample of a workload: the routing of the
    whole batch (router GEMM, QB sweep and biased top-k over all T tokens:
    QB's quantiles are over the batch) and then the dense layer of n_tok
    seeded sampled tokens.  The n_tok tokens are the units counted: each has
    gone through the complete layer when the clock stops.  Weight draws (and
    fp32 copies of the sampled tokens' experts) are made once, before any
    clock starts, as the GPU's weights are resident before its clock."""

    def __init__(self, shape, n_tok, seed=0):
        from oracle import qb_oracle as O
        self.O = O
        self.shape = shape
        self.inp = QI.LayerInputs(shape)
        rng = np.random.default_rng(seed)
        self.tokens = np.sort(rng.choice(shape.T, n_tok, replace=False))

        class Cached(O.LayerWeights):
            def __init__(self, inputs):
                super().__init__(inputs)
                self.cache = {}

            def expert(self, name, e):
                return self.cache[(name, int(e))].astype(np.float64)

        W = Cached(self.inp)
        for nm in ("x", "w_router", "router_offset", "w_down", "gamma", "w_proj_up", "w_shared_gate",
                   "w_shared_up", "w_shared_out"):
            if nm in self.inp.specs:
                W.dense(nm)
        logits = O.router_logits(W.dense("x"), W.dense("w_router"), W.dense("router_offset"))
        idx = O.moe_route_qb(logits, None, shape.k, shape.qb_sweeps)[2]
        for e in np.unique(idx[self.tokens]):
            for nm in ("w_gate", "w_up", "w_out"):
                W.cache[(nm, int(e))] = O.LayerWeights.expert(W, nm, e).astype(np.float32)
        self.W = W

    def run(self):
        """Seconds of one pass: the routing of all T tokens (inside
        layer_forward, from the router GEMM on) and the dense layer of the
        sampled tokens."""
        O, W = self.O, self.W
        t0 = time.perf_counter()
        O.layer_forward(self.inp, tokens=self.tokens, weights=W)
        return time.perf_counter() - t0

    def describe(self, sec, runs):
        s = self.shape
        return (f"numpy oracle, {runs} pass(es), mean {sec:.2f} s: router GEMM (fp64), QB sweep and top-k of "
                f"all {s.T} tokens, then the dense layer of {len(self.tokens)} seeded sampled tokens; "
                f"value counts those {len(self.tokens)} tokens (no extrapolation); BLAS threads = cores")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(shape, n_tok, min_seconds=10.0):
    """The oracle as it stands on a bounded sample (about 10-30 s of work)."""
    sample = OracleSample(shape, n_tok)
    times = []
    t_end = time.perf_counter() + min_seconds
    while not times or time.perf_counter() < t_end:
        times.append(sample.run())
    sec = statistics.mean(times)
    return {"value": n_tok / sec, "unit": "routed tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": sample.describe(sec, len(times))}


# ---------------------------------------------------------------------------

def run_reference(args, shape, world, rank):
    if rank != 0:
        return
    n_tok = max(1, int(os.environ.get("QB_ORACLE_TOKENS", "4")))
    times = []
    if args.workload in ROUTE_WORKLOADS:
        # the oracle's routing of the whole batch from the same fp32 logits
        from oracle import qb_oracle as O
        inp = QI.LayerInputs(shape)
        logits = O.router_logits(inp.values("x"), inp.values("w_router"), inp.values("router_offset"))
        mode = "gauss_seidel" if args.workload == "route_qb_gs" else "jacobi"
        steps = min(args.warmup + args.steps, 4) if mode == "gauss_seidel" else args.warmup + args.steps
        for i in range(steps):
            t0 = time.perf_counter()
            O.moe_route_qb(logits, None, shape.k, 1, mode)
            if i >= min(args.warmup, steps - 1):
                times.append(time.perf_counter() - t0)
        n_tok = shape.T
    else:
        sample = OracleSample(shape, n_tok)
        for i in range(args.warmup + args.steps):
            t = sample.run()
            if i >= args.warmup:
                times.append(t)
    sec = statistics.mean(times)
    val = n_tok / sec
    route = args.workload in ROUTE_WORKLOADS
    line = {"impl": "reference", "metric": ROUTE_METRIC if route else METRIC, "value": val,
            "unit": "routed tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32" if route else "f64",
            "data": "synthetic (seeded)",
            "config": route_config(shape, args) if route else config_of(shape, args),
            "cpu_baseline": {"value": val, "unit": "routed tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": (f"each step: the oracle's routing of all {shape.T} tokens" +
                                        ("" if args.workload in ROUTE_WORKLOADS else
                                         f" (router GEMM, QB sweep, top-k) and its dense layer of {n_tok} seeded "
                                         f"sampled tokens; value = those {n_tok} tokens / step time"))},
            "e2e": {"value": val, "unit": "routed tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def route_config(shape, args):
    gs = args.workload == "route_qb_gs"
    return {"workload": shape.name + ("_gauss_seidel" if gs else "_jacobi"), "T": shape.T, "n_experts": shape.n,
            "top_k": shape.k, "qb_sweeps": 1, "l2": "flushed between steps (512 MB write)",
            "parallelism": f"replicas x{args.gpus}"}


def route_balance(logits, k, qb_loads, T, n):
    """Max/mean expert load after one QB sweep (the timed routing's loads)
    and after DeepSeek-V3's fixed-step sign rule (moe_route_signsgd) for a few
    step sizes and step counts, on the same logits, from the GPU kernels."""
    import quantile_balanced_routing_gb300 as Q
    mean = T * k / n
    out = {"qb_one_sweep": float(qb_loads.max().item()) / mean}
    for gamma in (0.01, 0.03, 0.1):
        for steps in (0, 1, 8, 32):
            loads = Q.route_signsgd(logits, k, steps, gamma)[4]
            out[f"sign_gamma{gamma}_steps{steps}"] = float(loads.max().item()) / mean
    return {"max_over_mean_load": out}


def cpu_route_baseline(logits, k, gs):
    """The oracle's routing of the same fp32 logits on the host cores: one
    cyclic sweep (about 20 s at 4096 x 896), or Jacobi sweeps repeated for at
    least 3 s."""
    from oracle import qb_oracle as O
    mode = "gauss_seidel" if gs else "jacobi"
    times = []
    t_end = time.perf_counter() + 3.0
    while True:
        t0 = time.perf_counter()
        O.moe_route_qb(logits, None, k, 1, mode)
        times.append(time.perf_counter() - t0)
        if gs or time.perf_counter() >= t_end:
            break
    sec = statistics.mean(times)
    T, n = logits.shape
    return {"value": T / sec, "unit": "routed tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": (f"numpy oracle: {mode} routing of the same {T} x {n} fp32 logits, "
                       f"{len(times)} run(s), mean {sec:.3f} s")}


def config_of(shape, args):
    return {"workload": shape.name, "T": shape.T, "d": shape.d, "latent": shape.latent, "n_experts": shape.n,
            "top_k": shape.k, "expert_inter": shape.m, "shared_inter": shape.m_s, "expert_weights": shape.wfmt,
            "qb_sweeps": shape.qb_sweeps, "seed": shape.seed,
            "l2": "inputs larger than L2 (all weights are streamed every step)",
            "parallelism": f"replicas x{args.gpus}"}


def expert_gemm_roofline(shape, stages, pk, src, mx_peak=None):
    """Roofline of the dominant kernel: the grouped expert GEMM (the tcgen05
    kernel in grouped mode), launched twice per step, for the expert gate/up
    (with the SiTU-GLU epilogue) and the expert down-projection.  Achieved =
    the two launches' algorithmic work / their summed CUDA-event durations
    (the average launch's work over its average duration).  Tensor-bound
    workloads (prefill) are taken against the burst bf16 peak (the kernel is
    timed alone, between events), or the measured block-scaled peak for
    MXFP4 experts; weight-streaming ones (decode) against the HBM copy."""
    st = dict(stages)
    work = stage_work(shape, shape.T)
    names = ("expert_gate_up", "expert_down")
    if not all(nm in st for nm in names):
        return None
    b = sum(work[nm][0] for nm in names)
    f = sum(work[nm][1] for nm in names)
    ms = sum(st[nm] for nm in names)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if f / b >= ridge:
        if shape.wfmt == "mxfp4":
            # E2M1 weights x E4M3 token pairs on kind::mxf8f6f4: the MMA issues
            # twice the layer's flops (hi and lo token planes).  Peak: the
            # measured bf16 burst times the block-scaled : bf16 MMA rate ratio
            # the library's probe measures on this GPU.
            achieved = 2.0 * f / (ms * 1e-3) / 1e12
            if mx_peak:
                ratio, probe = mx_peak
                peak = pk["bf16_tflops"] * ratio
                note = (f"measured bf16 burst x measured mxf8f6f4:bf16 MMA rate ratio {ratio:.3f} (probe: "
                        f"{probe['mxf8f6f4']:.0f} / {probe['bf16']:.0f} TFLOP/s raw back-to-back MMAs)")
            else:
                peak = 2.0 * pk["bf16_tflops"]
                note = "2 x measured bf16 burst (nominal fp8:bf16 ratio; the probe was unavailable)"
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "peak_note": note + "; issued MMA flops = 2 x layer flops (hi and lo token planes)"}
        else:
            achieved = f / (ms * 1e-3) / 1e12
            peak = pk["bf16_tflops"]
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "peak_note": "measured cuBLAS bf16 burst"}
    else:
        achieved = b / (ms * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "peak_note": "measured copy bandwidth"}
    roof["frac"] = achieved / peak
    # both roofs, whichever binds: the bf16 (or block-scaled) tensor peak and
    # the HBM copy bandwidth, each against the same two launches
    if shape.wfmt == "mxfp4":
        t_peak = pk["bf16_tflops"] * mx_peak[0] if mx_peak else 2.0 * pk["bf16_tflops"]
        t_frac = 2.0 * f / (ms * 1e-3) / 1e12 / t_peak
    else:
        t_frac = f / (ms * 1e-3) / 1e12 / pk["bf16_tflops"]
    roof["tensor_frac"] = t_frac
    roof["hbm_frac"] = b / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]
    tr = [recorded_traffic(nm, shape.name) for nm in names]
    roof.update({"traffic": sum(tr) / 2 if all(t is not None for t in tr) else None,
                 "kernel": "k_tc_gemm grouped (expert gate/up + expert down launches)",
                 "launches_per_step": 2, "ms_per_launch": ms / 2, "algorithmic_bytes_per_launch": b / 2,
                 "algorithmic_flops_per_launch": f / 2, "peak_source": src,
                 "per_launch_ms": {nm: round(st[nm], 4) for nm in names}})
    return roof


def pipelined_e2e(steps, stream, h2d, compute, d2h):
    """End-to-end steps as a user's pipeline would run them: each step copies
    its input from pinned host memory (h2d, on one copy stream), computes (on
    `stream`) and copies its result back (d2h, on another copy stream), with
    two buffer slots so that step i's copies overlap the neighbouring steps'
    compute.  Every step's copies are inside the timed region; returns ms per
    step from the first input copy to the last result copy."""
    import torch
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    Ev = torch.cuda.Event
    in_ready = [Ev() for _ in range(steps)]
    done = [Ev() for _ in range(steps)]
    out_done = [Ev() for _ in range(steps)]
    e0, e1 = Ev(enable_timing=True), Ev(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        slot = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(done[i - 2])      # step i-2 has read this input slot
            h2d(slot)
            in_ready[i].record(s_in)
        stream.wait_event(in_ready[i])
        if i >= 2:
            stream.wait_event(out_done[i - 2])    # step i-2's result has left this output slot
        compute(slot)
        done[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[i])
            d2h(slot)
            out_done[i].record(s_out)
    e1.record(s_out)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / max(steps, 1)


def run_ours(args, shape, world, rank, local):
    import torch
    from qb_inputs.device import layer_for, upload
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = QI.LayerInputs(shape.with_(seed=shape.seed + rank))
    d = upload(inp, dev)
    lay = layer_for(shape)
    lay.set_weights(**{k: v for k, v in d.items() if k != "x"})
    x = d["x"]
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        lay.forward(x, out=out)
    rc = lay.status()
    if rc:
        raise RuntimeError(f"device status {rc} after warm-up")
    launches_per_step = lay.last_launch_count()
    # the headline loop: no per-stage events inside it
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            lay.forward(x, out=out)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = start.elapsed_time(end) / max(args.steps, 1)
    rc = lay.status()
    if rc:
        raise RuntimeError(f"device status {rc} in the timed region")
    value_job, ms_max = replica_throughput(shape.T, ms, world)

    # per-stage times from a separate pass with CUDA events between the stages
    lay.set_timing(max(args.steps, 1))
    for _ in range(args.steps):
        lay.forward(x, out=out)
    stages = lay.stage_times()
    lay.set_timing(0)

    # end to end: pinned host input -> device, forward, device -> host output,
    # double-buffered so that copies overlap the neighbouring steps' forwards
    x_host = x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]

    def h2d(slot):
        x_dev[slot].copy_(x_host, non_blocking=True)

    def fwd(slot):
        lay.forward(x_dev[slot], out=out_dev[slot])

    def d2h(slot):
        out_host.copy_(out_dev[slot], non_blocking=True)

    pipelined_e2e(2, stream, h2d, fwd, d2h)
    barrier(world)
    ms_e2e = max_over_ranks(pipelined_e2e(args.steps, stream, h2d, fwd, d2h), world)
    lay.close()
    mx_peak = None
    if shape.wfmt == "mxfp4" and rank == 0:
        mx_peak = mma_peak_ratio()

    if rank != 0:
        return
    pk, src = peaks()
    roof = expert_gemm_roofline(shape, stages, pk, src, mx_peak)
    n_cpu_tok = int(os.environ.get("QB_ORACLE_TOKENS", "8"))
    cpu = cpu_baseline(shape, n_cpu_tok) if world == 1 and not args.no_cpu else None
    tok = shape.T * world
    line = {
        "metric": METRIC, "value": value_job, "unit": "routed tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if shape.wfmt == "bf16" else ("bf16+mxfp4" if shape.wfmt == "mxfp4" else "f32"),
        "data": "synthetic (seeded, random-init weights)", "config": config_of(shape, args),
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": tok / (ms_e2e * 1e-3), "unit": "routed tokens/s",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size()},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "stages_ms": {nm: round(t, 4) for nm, t in stages},
    }
    print(json.dumps(line), flush=True)


def mma_peak_ratio():
    """(block-scaled mxf8f6f4 : bf16 MMA rate ratio, the probe's raw rates in
    TFLOP/s), measured by the library's own probe kernel on this GPU; None if
    the probe is unavailable."""
    try:
        import quantile_balanced_routing_gb300 as Q
        probe = {k: Q.mma_peak_tflops(k) for k in ("bf16", "mxf8f6f4")}
        return probe["mxf8f6f4"] / probe["bf16"], probe
    except Exception:
        return None


def run_route(args, shape, world, rank, local):
    """The QB-routing workload alone: moe_route_qb (one Jacobi sweep) or
    moe_route_qb_gs (one cyclic sweep) on fp32 logits x W_r^T + o resident
    in HBM.  Its working set fits in L2, so L2 is flushed (a 512 MB write)
    between timed steps, outside each step's event pair."""
    import torch
    import quantile_balanced_routing_gb300 as Q
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = QI.LayerInputs(shape.with_(seed=shape.seed + rank))
    x = torch.from_numpy(inp.values("x")).to(dev)
    wr = torch.from_numpy(inp.values("w_router")).to(dev)
    o = torch.from_numpy(inp.values("router_offset")).to(dev)
    logits = (x @ wr.T + o).contiguous()          # input preparation (not timed)
    del x, wr
    gs = args.workload == "route_qb_gs"
    T, n, k = shape.T, shape.n, shape.k
    scores = torch.empty((T, n), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    loads = torch.empty((n,), dtype=torch.int32, device=dev)
    bias = torch.empty((n,), dtype=torch.float32, device=dev)
    lib = Q.load_library()
    need = lib.qbmoe_route_gs_workspace_bytes(T, n, k) if gs else Q.qbmoe_route_workspace_bytes(T, n, k)
    ws = torch.empty((need,), dtype=torch.uint8, device=dev)
    flush = torch.empty((512 << 20,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    p = lambda t: t.data_ptr()

    def step():
        if gs:
            rc = lib.moe_route_qb_gs(T, n, k, 1, 0, p(logits), None, p(bias), p(scores), p(idx), p(w), p(loads),
                                     None, p(ws), ws.numel(), stream.cuda_stream or None)
            launches = 2 * n + 6
        else:
            rc = Q.moe_route_qb(T, n, k, 1, p(logits), None, p(bias), p(scores), p(idx), p(w), p(loads), p(ws),
                                ws.numel(), stream.cuda_stream or None)
            launches = lib.qbmoe_route_last_launch_count()
        if rc:
            raise Q.QbmoeError(rc, "routing")
        return launches

    for _ in range(args.warmup):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    launches = 0
    with ClockSampler(local) as clocks:
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            launches += step()
            b.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = sum(a.elapsed_time(b) for a, b in ev) / max(args.steps, 1)
    value_job, ms_max = replica_throughput(T, ms, world)

    # end to end: pinned host logits -> device, routing, device -> host indices
    # and weights, double-buffered (two sets of routing buffers) so that the
    # copies overlap the neighbouring steps' routing
    lg_host = logits.cpu().pin_memory()
    idx_host = torch.empty((T, k), dtype=torch.int32).pin_memory()
    w_host = torch.empty((T, k), dtype=torch.float32).pin_memory()
    bufs = [dict(logits=torch.empty_like(logits), scores=torch.empty_like(scores), idx=torch.empty_like(idx),
                 w=torch.empty_like(w), loads=torch.empty_like(loads), bias=torch.empty_like(bias),
                 ws=torch.empty_like(ws)) for _ in range(2)]

    def h2d(slot):
        bufs[slot]["logits"].copy_(lg_host, non_blocking=True)

    def route(slot):
        nonlocal logits, scores, idx, w, loads, bias, ws
        keep = (logits, scores, idx, w, loads, bias, ws)
        b = bufs[slot]
        logits, scores, idx, w, loads, bias, ws = (b["logits"], b["scores"], b["idx"], b["w"], b["loads"],
                                                   b["bias"], b["ws"])
        step()
        logits, scores, idx, w, loads, bias, ws = keep

    def d2h(slot):
        idx_host.copy_(bufs[slot]["idx"], non_blocking=True)
        w_host.copy_(bufs[slot]["w"], non_blocking=True)

    pipelined_e2e(2, stream, h2d, route, d2h)
    barrier(world)
    ms_e2e = max_over_ranks(pipelined_e2e(args.steps, stream, h2d, route, d2h), world)
    if rank != 0:
        return
    balance = route_balance(logits, k, loads, T, n) if not gs else None
    cpu = cpu_route_baseline(lg_host.numpy(), k, gs) if world == 1 and not args.no_cpu else None
    pk, src = peaks()
    b_alg = T * n * 4 * 2 + T * k * 8 + n * 8       # logits in, scores out, idx/w out, bias/loads
    achieved = b_alg / (ms_max * 1e-3) / 1e9
    line = {"metric": ROUTE_METRIC, "value": value_job,
            "unit": "routed tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded)",
            "config": route_config(shape, args),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "traffic": None, "kernel": "routing (all kernels)",
                         "algorithmic_bytes": b_alg, "peak_source": src},
            "cpu_baseline": cpu,
            "e2e": {"value": T * world / (ms_e2e * 1e-3), "unit": "routed tokens/s",
                    "h2d_bytes_per_step": logits.numel() * logits.element_size(),
                    "d2h_bytes_per_step": idx.numel() * idx.element_size() + w.numel() * w.element_size()},
            "gpu_launches": launches, "clocks": clocks.summary()}
    if balance:
        line["balance"] = balance
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling only: scale the workload down to this many experts, keeping tokens per expert")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    shape = WORKLOADS[args.workload]
    if args.experts:
        shape = shape.with_(name=f"{shape.name}_scaled_n{args.experts}", n=args.experts,
                            T=max(1, shape.T * args.experts // shape.n))
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, shape, int(os.environ.get("WORLD_SIZE", "1")), rank)
        return
    world, rank, local = dist_setup()
    if args.workload in ROUTE_WORKLOADS:
        run_route(args, shape, world, rank, local)
    else:
        run_ours(args, shape, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
