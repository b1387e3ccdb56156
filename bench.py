"""Benchmark of the K3-shaped sparse MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one forward pass of the whole layer (every stage of moe_forward)
over one batch of synthetic tokens of the workload (default: the K3-shaped
decode batch, 64 tokens).  The forward is captured once in a CUDA graph and
each step replays it (--eager: plain launches; the eager time is reported
either way).  Inputs and weights are resident in HBM before the timed region;
L2 is flushed (a 512 MB write) between timed steps, outside the per-step CUDA
events.  Prints one JSON line (rank 0), with a sub-record of the same layer at
8192 tokens (prefill) timed the same way in the same run.

--impl reference times the CPU oracle instead (the reference arm): each step
is the oracle's forward over a bounded sample of the same workload's tokens on
this machine's host cores.

Multi-GPU: the layer is replicated (each rank runs its own full batch, no
collective on the data path); value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; % HBM roofline (decode) / % FP4 tensor peak (prefill)"
MX4_BYTES_PER_ELT = 17 / 32          # 4-bit element + 8-bit scale per 32
MX8_BYTES_PER_ELT = 33 / 32


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


CPU_BASELINE_SECONDS = 10.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the layer's
# kernels from an ncu capture, stored with a hash of the kernel sources it
# was taken on; a figure stands only while the sources are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
SOURCE_FILES = ("api.cu", "gemm.cu", "kernels.cu", "peak.cu", "router.cu", "ep.cu", "balance.cu", "internal.h", "mx.cuh", "ptx.cuh")


def kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) of the library's CUDA sources and header."""
    import hashlib
    h = hashlib.sha256()
    src = os.path.join(ROOT, "moe_expert_layer_top16_gb300", "csrc")
    for f in SOURCE_FILES + ("../../include/moe.h",):
        with open(os.path.join(src, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """(DRAM bytes of one forward, per-kernel dict) from the stored capture of
    `workload`, or (None, None) when there is none or the sources changed."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None, None
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None, None
    return rec.get("layer_dram_bytes"), rec.get("kernels")


def workload_config(wl, T):
    """The `config` keys both arms report for a workload of T tokens."""
    return {"workload": wl.name, "tokens": T, "d_model": wl.d_model, "d_latent": wl.d_latent,
            "experts": wl.n_experts, "top_k": wl.top_k, "expert_inter": wl.expert_inter,
            "shared": wl.n_shared, "shared_inter": wl.shared_inter, "bias": wl.bias,
            "precision": getattr(wl, "precision", "mx")}


def launches_per_forward(T, wl=None):
    """Kernels of this library one forward of T tokens launches: quantiser
    (not in the mixed scheme with latent routing), A2, router (or its
    tensor-core estimate), top-k, per-expert scan (batches over 128 tokens;
    folded into the work-list kernel below that), work lists, dispatch, A7,
    A8, combine, A10."""
    n = 10 + (1 if (T + 31) // 32 > 4 else 0)
    if wl is not None and getattr(wl, "precision", "mx") == "mixed" and wl.route == "latent":
        n -= 1
    return n


def algorithmic_work(wl, T, counts):
    """Per-stage algorithmic bytes and MX FLOPs of one forward of T tokens.
    `counts` = realised tokens per expert (touched experts are those > 0)."""
    D, L, E, k, I, S, Is = (wl.d_model, wl.d_latent, wl.n_experts, wl.top_k, wl.expert_inter, wl.n_shared,
                            wl.shared_inter)
    touched = int((np.asarray(counts) > 0).sum())
    TK = T * k
    rows_a2 = L + 2 * S * Is
    kcat = L + S * Is
    # the mixed scheme keeps the projections and shared experts in bf16, and
    # their inputs (x, h_s, c) too
    mixed = getattr(wl, "precision", "mx") == "mixed"
    wb = 2.0 if mixed else MX4_BYTES_PER_ELT          # bytes per weight element of A2 / A10
    ab = 2.0 if mixed else MX8_BYTES_PER_ELT          # bytes per input element of A2 / A10
    w = {
        "gemm_down_shared": (rows_a2 * D * wb + T * D * ab
                             + T * L * (4 + MX8_BYTES_PER_ELT) + T * S * Is * ab,
                             2.0 * T * rows_a2 * D),
        "router": (E * L * 4 + T * L * 4 + T * E * 4, 2.0 * T * E * L),
        "gemm_gate_up": (touched * 2 * I * L * MX4_BYTES_PER_ELT + TK * L * MX8_BYTES_PER_ELT
                         + TK * I * MX8_BYTES_PER_ELT, 2.0 * TK * 2 * I * L),
        "gemm_down": (touched * L * I * MX4_BYTES_PER_ELT + TK * I * MX8_BYTES_PER_ELT + TK * L * 4,
                      2.0 * TK * L * I),
        "combine": (TK * L * 4 + T * L * ab, 2.0 * TK * L),
        "gemm_up_shared": (D * kcat * wb + T * kcat * ab + T * D * 4,
                           2.0 * T * D * kcat),
        "quant_x": (0.0 if mixed and wl.route == "latent" else T * D * (2 + MX8_BYTES_PER_ELT), 0.0),
        "dispatch": (TK * L * MX8_BYTES_PER_ELT * 2, 0.0),
    }
    expert_weight_bytes = touched * 3 * I * L * MX4_BYTES_PER_ELT + 3 * S * Is * D * wb
    return w, touched, expert_weight_bytes


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    """Ranks from the launcher's environment; one process per GPU over NCCL
    (gloo where no GPU is visible, for the host-side logic)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(world, tokens_per_step, steps, slowest_ms):
    """Whole-job tokens/s: each of `world` ranks runs `steps` steps of
    `tokens_per_step` tokens (weak scaling); the job takes the slowest rank's
    time."""
    return world * tokens_per_step * steps / (slowest_ms / 1e3)


def max_over_ranks(world, v: float) -> float:
    """The largest of the ranks' values (every rank gets it)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle (CPU) timing
def oracle_sample(wl, n_tokens, device):
    """Encode (oracle encoder) the weights a sample of tokens needs and return
    a closure that runs the oracle forward over those tokens."""
    import torch
    import oracle
    import synth

    dev = device

    def fetch(name, i):
        if name == "bias":
            b = synth.router_bias(wl, device="cpu")
            return None if b is None else b.numpy()
        return synth.weight(wl, name, i, device=dev).cpu().numpy()

    x = synth.hidden_states(wl, n_tokens, device="cpu")
    xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    base = oracle.encode_layer(wl, fetch, experts=[])
    r = oracle.moe_forward(wl, base, xb, route_only=True, want=("idx",))
    experts = sorted(set(int(e) for e in r["idx"].ravel()))
    lw = oracle.encode_layer(wl, fetch, experts=experts)

    def run():
        return oracle.moe_forward(wl, lw, xb, want=("y",))

    return run, len(experts)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def run_reference(args, wl, world, rank):
    import torch
    if rank != 0:
        return 0
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    n_tok = args.reference_tokens
    run, n_exp = oracle_sample(wl, n_tok, dev)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = n_tok * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(wl, wl.tokens), tokens_per_step=n_tok, parallelism="rank 0 only"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{n_tok} tokens of {wl.name} ({n_exp} experts) per step; fp64 C oracle, OpenMP, "
                                   f"{cpu_model()}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- CUDA path
def measure_tensor_peaks(dev, reps=5):
    """Issue rate of the tensor cores on this GPU (moe_mma_probe): the
    layer's block-scaled kind::mxf8f6f4 MMA (E2M1 x E4M3, N = 240) and
    kind::f16 (bf16, N = 256), best of `reps` timed launches, TFLOP/s."""
    import torch
    import moe_expert_layer_top16_gb300 as moe
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = {}
    for name, kind, n, iters in (("mxf8f6f4_e2m1_e4m3", moe.PROBE_MX_E2M1_E4M3, 240, 20000),
                                 ("f16_bf16", moe.PROBE_BF16, 256, 20000)):
        rates = []
        for i in range(reps + 2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            flops = moe.mma_probe(kind, n, iters, status)
            b.record()
            torch.cuda.synchronize()
            if i >= 2:
                rates.append(flops / (a.elapsed_time(b) / 1e3) / 1e12)
        if int(status.item()) != 0:
            raise RuntimeError("device-side time-out in the tensor-core probe")
        out[name] = max(rates)
    return out


def time_layer(plan, wl, T, x, y, flush, steps, warmup, world, with_stages=True, graph=True):
    """Warm-up, an untimed per-stage pass (events between the stages), then
    exactly `steps` forwards each between two events on the forward's stream,
    with the L2 flush outside the events.  With `graph` the forward (all its
    kernels, unchanged) is captured once in a CUDA graph and each timed step
    replays it, as a serving loop runs a batch bucket; the eager time of the
    same forward is measured too.  Returns (step_ms list, mean stage ms,
    realised counts, clocks, wall seconds of the timed region, eager ms per
    step or None)."""
    import torch
    import moe_expert_layer_top16_gb300 as moe
    dev = x.device
    counts = torch.zeros(wl.n_experts, dtype=torch.int32, device=dev)
    for i in range(max(warmup, 1)):
        plan.forward(x, out=y, debug={"counts": counts} if i == 0 else None)
    torch.cuda.synchronize()
    if plan.device_status() != moe.MOE_OK:
        raise RuntimeError("device-side error during warm-up")
    counts_h = counts.cpu().numpy()
    nst = moe.NUM_STAGES
    stage_ms = None
    if with_stages:
        n_stage = min(steps, 20)
        stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(n_stage)]
        for evs in stage_ev:                 # torch creates the CUDA events at their first record
            for e in evs:
                e.record()
        torch.cuda.synchronize()
        for i in range(n_stage):
            flush.fill_(float(i))
            plan.forward(x, out=y, stage_events=stage_ev[i])
        torch.cuda.synchronize()
        stage_ms = np.array([[stage_ev[i][s].elapsed_time(stage_ev[i][s + 1]) for s in range(nst)]
                             for i in range(n_stage)]).mean(axis=0)
    eager_ms = None
    g = None
    if graph:
        # eager reference of the same forward, then the capture
        ea = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(min(steps, 20))]
        for i, (a, b) in enumerate(ea):
            flush.fill_(float(i))
            a.record()
            plan.forward(x, out=y)
            b.record()
        torch.cuda.synchronize()
        eager_ms = float(np.median([a.elapsed_time(b) for a, b in ea]))
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            plan.forward(x, out=y)
            cs.synchronize()
            with torch.cuda.graph(g, stream=cs):
                plan.forward(x, out=y)
        torch.cuda.current_stream().wait_stream(cs)
        for _ in range(max(warmup, 1)):
            g.replay()
        torch.cuda.synchronize()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(dev.index)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(float(i))                       # L2 flush, outside the step events
        ev0[i].record()
        if g is not None:
            g.replay()
        else:
            plan.forward(x, out=y)
        ev1[i].record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if plan.device_status() != moe.MOE_OK:
        raise RuntimeError("device-side error in the timed region")
    step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(steps)]
    del g
    return step_ms, stage_ms, counts_h, clocks, wall, eager_ms


def layer_roofline(wl, T, ms_per_step, stage_ms, counts_h, hbm, tensor_peak, peak_source):
    """Roofline of the whole layer step and of its dominant kernel.  The
    layer figure is the headline: decode-sized batches (below 4096 tokens)
    on expert-weight bytes over the measured HBM copy bandwidth,
    prefill-sized ones on MX FLOPs over the measured block-scaled MMA rate.
    The dominant stage's own figure rides along under "kernel"."""
    import moe_expert_layer_top16_gb300 as moe
    work, touched, expert_bytes = algorithmic_work(wl, T, counts_h)
    step_s = ms_per_step / 1e3
    layer_flops = sum(f for _, f in work.values())
    names = moe.STAGE_NAMES
    dom = int(np.argmax(stage_ms))
    dom_name = names[dom]
    k_bytes, k_flops = work.get(dom_name, (0.0, 0.0))
    k_s = stage_ms[dom] / 1e3
    tensor_bound = T >= 4096
    traffic, per_kernel = ncu_traffic(wl.name)
    kernel = {"name": dom_name, "ms": float(stage_ms[dom]),
              "hbm": {"achieved": k_bytes / k_s / 1e9, "frac": k_bytes / k_s / 1e9 / hbm, "algorithmic_bytes": k_bytes},
              "tensor": {"achieved": k_flops / k_s / 1e12, "frac": k_flops / k_s / 1e12 / tensor_peak,
                         "flops": k_flops},
              "traffic": (per_kernel or {}).get(dom_name)}
    if tensor_bound:
        roof = {"bound": "tensor", "scope": "layer: MX FLOPs per step", "achieved": layer_flops / step_s / 1e12,
                "peak": tensor_peak, "unit": "TFLOP/s", "frac": layer_flops / step_s / 1e12 / tensor_peak,
                "peak_source": peak_source}
    else:
        roof = {"bound": "hbm", "scope": "layer: expert-weight bytes per step",
                "achieved": expert_bytes / step_s / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": expert_bytes / step_s / 1e9 / hbm, "peak_source": "measured copy bandwidth"}
    roof["traffic"] = traffic
    roof["traffic_note"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum over one forward's kernels, "
                            "taken on the current kernel sources" if traffic is not None
                            else "no ncu capture of the current kernel sources")
    roof["kernel"] = kernel
    roof["kernel_frac"] = kernel["tensor" if tensor_bound else "hbm"]["frac"]
    layer = {"touched_experts": touched, "expert_weight_bytes": expert_bytes,
             "expert_weight_GBps": expert_bytes / step_s / 1e9,
             "expert_weight_frac_hbm": expert_bytes / step_s / 1e9 / hbm,
             "mx_tflops": layer_flops / step_s / 1e12, "mx_frac_tensor_peak": layer_flops / step_s / 1e12 / tensor_peak,
             "max_over_mean_load": float(counts_h.max() / max(counts_h.mean(), 1e-9)),
             "stage_ms": {n: float(v) for n, v in zip(names, stage_ms)}}
    return roof, layer


def routing_check(plan, wl, x, n_tok, dev):
    """The GPU's selection for the first n_tok tokens against the oracle's
    (on its own latent): tokens whose lists differ, and how many of those are
    certified near-ties (key gap within twice the selected logits' error)."""
    import torch
    import oracle
    import synth
    import moe_expert_layer_top16_gb300 as moe

    def fetch(name, i):
        if name == "bias":
            b = synth.router_bias(wl, device="cpu")
            return None if b is None else b.numpy()
        return synth.weight(wl, name, i, device=dev).cpu().numpy()

    T = x.shape[0]
    dbg = moe.debug_buffers(wl, T, dev, ("topk_idx", "logits"))
    plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    idx = dbg["topk_idx"][:n_tok].cpu().numpy()
    lg = dbg["logits"][:n_tok].cpu().numpy().astype(np.float64)
    xb = x[:n_tok].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    r = oracle.moe_forward(wl, oracle.encode_layer(wl, fetch, experts=[]), xb, route_only=True,
                           want=("idx", "logits"))
    bias = synth.router_bias(wl, device="cpu")
    b = 0.0 if bias is None else bias.numpy().astype(np.float64)
    keys = r["logits"] if bias is None else 1.0 / (1.0 + np.exp(-r["logits"])) + b
    differ, near = 0, 0
    for t in range(n_tok):
        if list(idx[t]) == list(r["idx"][t]):
            continue
        differ += 1
        sel = idx[t].astype(np.int64)
        delta = float(np.max(np.abs(lg[t, sel] - r["logits"][t, sel])))
        if all(abs(keys[t, a] - keys[t, c]) <= 2 * delta + 1e-12 for a, c in zip(idx[t], r["idx"][t]) if a != c):
            near += 1
    return {"tokens": n_tok, "differing": differ, "certified_near_ties": near}


def run_cuda(args, wl, world, rank, local):
    import torch
    import synth
    import moe_expert_layer_top16_gb300 as moe
    from moe_expert_layer_top16_gb300 import build as mbuild
    from moe_expert_layer_top16_gb300.weights import encode_layer

    mbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    T = wl.tokens
    pre = None if args.no_prefill or T >= args.prefill_tokens else wl.with_tokens(args.prefill_tokens)

    def fetch(name, i):
        if name == "bias":
            return synth.router_bias(wl, device=dev)
        return synth.weight(wl, name, i, device=dev)

    W = encode_layer(wl, fetch, dev)
    plan = moe.Plan(wl, W, max_tokens=max(T, pre.tokens if pre else 0))
    del W
    torch.cuda.empty_cache()
    hbm, bf16, bf16_sus, peak_kind = peaks()
    tpk = measure_tensor_peaks(dev)
    tensor_peak = tpk["mxf8f6f4_e2m1_e4m3"]
    peak_source = "measured: tcgen05.mma kind::mxf8f6f4 E2M1 x E4M3 issue rate (moe_mma_probe), this GPU"
    x = synth.hidden_states(wl, T, device=dev, offset=rank * T)
    y = torch.empty(T, wl.d_model, dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    K = args.steps
    step_ms, stage_ms, counts_h, clocks, wall, eager_ms = time_layer(plan, wl, T, x, y, flush, K, args.warmup, world,
                                                                     graph=not args.eager)
    total_ms = max_over_ranks(world, float(np.sum(step_ms)))
    ms_per_step = total_ms / K
    value = job_throughput(world, T, K, total_ms)

    # end to end through the C ABI with host buffers (copies inside the timed region)
    xh = x.cpu().pin_memory()
    yh = torch.empty(T, wl.d_model, dtype=torch.float32).pin_memory()
    for _ in range(2):
        plan.forward_host(xh, yh)
    barrier(world)
    t0 = time.perf_counter()
    n_e2e = max(3, min(K, 50))
    for _ in range(n_e2e):
        plan.forward_host(xh, yh)
    e2e_s = max_over_ranks(world, time.perf_counter() - t0)
    e2e_value = world * T * n_e2e / e2e_s

    roof, layer = layer_roofline(wl, T, ms_per_step, stage_ms, counts_h, hbm, tensor_peak, peak_source)
    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "step_ms": {"median": float(np.median(step_ms)), "p10": float(np.percentile(step_ms, 10)),
                    "p90": float(np.percentile(step_ms, 90))},
        "launch": ("each step replays one CUDA graph of the whole forward (its kernels unchanged)"
                   if eager_ms is not None else "eager launches"),
        "eager_ms_per_step": eager_ms,
        "dtype": ("mxfp4 x mxfp8 routed experts, bf16 projections and shared experts, fp32 accumulate"
                  if getattr(wl, "precision", "mx") == "mixed" else "mxfp4 weights x mxfp8 activations, fp32 accumulate"),
        "data": "synthetic",
        "config": dict(workload_config(wl, T),
                       l2="flushed by a 512 MB write between timed steps (outside the step events)",
                       parallelism=f"replicas x{world}"),
        "roofline": roof,
        "layer": layer,
        "tensor_peaks_tflops": dict(tpk, note="issue rate of back-to-back MMAs on shared-memory operands, "
                                              "one CTA per SM, best of 5 launches; kind::mxf4 is not probed: "
                                              "a W4A8 product cannot use it"),
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": int(T * wl.d_model * 2),
                "d2h_bytes_per_step": int(T * wl.d_model * 4)},
        "gpu_launches": launches_per_forward(T, wl) * K,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if args.ep_ranks > 0:
        # expert-parallel dispatch and combine of this batch over virtual ranks
        R = min(args.ep_ranks, wl.n_experts)
        plan.forward(x, out=y)
        wire, offs = plan.ep_dispatch(T, R)
        o = torch.zeros(T * wl.top_k, wl.d_latent, dtype=torch.float32, device=dev)
        plan.ep_combine(T, wire, o)
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(10)]
        for e3 in evs:
            e3[0].record()
            plan.ep_dispatch(T, R)
            e3[1].record()
            plan.ep_combine(T, wire, o)
            e3[2].record()
        torch.cuda.synchronize()
        rows = np.diff(offs.cpu().numpy())
        rb = plan.ep_row_bytes()
        result["ep"] = {"ranks": R, "tokens": T,
                        "payload_bytes_per_token": wl.top_k * (wl.d_latent + wl.d_latent // 32),
                        "wire_bytes_per_token": wl.top_k * rb,
                        "combine_bytes_per_token_fp32": wl.top_k * wl.d_latent * 4,
                        "pages_2kd_fp8_bytes_per_token": 2 * wl.top_k * wl.d_model,
                        "rows_per_rank_min_max": [int(rows.min()), int(rows.max())],
                        "dispatch_ms": float(np.median([a.elapsed_time(b) for a, b, _ in evs])),
                        "combine_ms": float(np.median([b.elapsed_time(c) for _, b, c in evs]))}
        del wire, offs, o
    if pre is not None:
        # the same layer at the prefill batch, timed the same way in the same run
        Tp = pre.tokens
        xp = synth.hidden_states(pre, Tp, device=dev, offset=rank * Tp)
        yp = torch.empty(Tp, wl.d_model, dtype=torch.float32, device=dev)
        Kp = max(5, min(K, 40))
        p_ms, p_stage, p_counts, p_clocks, p_wall, p_eager = time_layer(plan, pre, Tp, xp, yp, flush, Kp, args.warmup,
                                                                        world, graph=not args.eager)
        p_total = max_over_ranks(world, float(np.sum(p_ms)))
        p_roof, p_layer = layer_roofline(pre, Tp, p_total / Kp, p_stage, p_counts, hbm, tensor_peak, peak_source)
        result["prefill"] = {"workload": pre.name, "tokens": Tp, "steps": Kp, "ms_per_step": p_total / Kp,
                             "eager_ms_per_step": p_eager,
                             "value": job_throughput(world, Tp, Kp, p_total), "unit": "tokens/s",
                             "step_ms": {"median": float(np.median(p_ms)), "p10": float(np.percentile(p_ms, 10)),
                                         "p90": float(np.percentile(p_ms, 90))},
                             "roofline": p_roof, "layer": p_layer, "gpu_launches": launches_per_forward(Tp, pre) * Kp,
                             "clocks": p_clocks, "wall_s_timed_region": p_wall}
        result["gpu_launches"] += launches_per_forward(Tp, pre) * Kp
        del xp, yp
    if rank == 0 and not args.no_cpu_baseline:
        n_tok = min(args.cpu_tokens, T)
        result["layer"]["routing_check"] = routing_check(plan, wl, x, n_tok, dev)
    plan.close()
    del flush
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle as it stands, repeated over the same token sample until
        # about CPU_BASELINE_SECONDS of work have been timed
        n_tok = min(args.cpu_tokens, T)
        run, n_exp = oracle_sample(wl, n_tok, dev)
        reps, t0 = 0, time.perf_counter()
        while True:
            run()
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= CPU_BASELINE_SECONDS or reps >= 100:
                break
        result["cpu_baseline"] = {"value": n_tok * reps / dt, "unit": "tokens/s", "cores": cpu_cores(),
                                  "kind": "oracle",
                                  "sample": f"{n_tok} tokens of {wl.name} ({n_exp} experts) x {reps} passes "
                                            f"({dt:.1f} s); fp64 C oracle with OpenMP on {cpu_model()}; "
                                            f"weight encoding excluded"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


def run_sweep(args, wl, rank, local):
    """The layer at every batch size of the sweep (one plan), against both
    rooflines: expert-weight bytes over HBM bandwidth, MX FLOPs over the
    tensor peak.  The crossover is where the second overtakes the first."""
    import torch
    import synth
    import moe_expert_layer_top16_gb300 as moe
    from moe_expert_layer_top16_gb300 import build as mbuild
    from moe_expert_layer_top16_gb300.weights import encode_layer

    mbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    Tmax = max(synth.SWEEP_TOKENS)

    def fetch(name, i):
        if name == "bias":
            return synth.router_bias(wl, device=dev)
        return synth.weight(wl, name, i, device=dev)

    W = encode_layer(wl, fetch, dev)
    plan = moe.Plan(wl, W, max_tokens=Tmax)
    del W
    torch.cuda.empty_cache()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    hbm, bf16, _, _ = peaks()
    tensor_peak = measure_tensor_peaks(dev)["mxf8f6f4_e2m1_e4m3"]
    for T in synth.SWEEP_TOKENS:
        x = synth.hidden_states(wl, T, device=dev)
        y = torch.empty(T, wl.d_model, dtype=plan.out_dtype, device=dev)
        steps = max(5, min(args.steps, (200 * 64) // T))
        # the same timing as the headline: graph replay, L2 flushed between steps
        step_ms, _, counts_h, _, _, eager_ms = time_layer(plan, wl, T, x, y, flush, steps, max(args.warmup, 3), 1,
                                                          with_stages=False, graph=not args.eager)
        ms = float(np.median(step_ms))
        work, touched, expert_bytes = algorithmic_work(wl, T, counts_h)
        flops = sum(f for _, f in work.values())
        line = {"impl": "sweep", "workload": wl.name, "tokens": T, "ms_median": ms, "eager_ms_median": eager_ms,
                "tokens_per_s": T / (ms / 1e3),
                "touched_experts": touched, "expert_weight_GBps": expert_bytes / (ms / 1e3) / 1e9,
                "expert_weight_frac_hbm": expert_bytes / (ms / 1e3) / 1e9 / hbm,
                "mx_tflops": flops / (ms / 1e3) / 1e12, "mx_frac_tensor_peak": flops / (ms / 1e3) / 1e12 / tensor_peak,
                "tensor_peak_tflops": tensor_peak,
                "steps": steps, "l2": "flushed between steps"}
        if rank == 0:
            print(json.dumps(line), flush=True)
    plan.close()
    return 0


PAGES_BATCHES = (1, 8, 64, 256, 1024, 4096)


def pages_uniform_gb_per_token():
    """The pages' uniform-routing column (GB per token by batch), from the
    stored copy of their printed table."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", "expert_amortisation.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                parts = ln.split()
                out[int(parts[0])] = float(parts[1])
    return out


def run_multilayer(args, wl, rank, local):
    """A decode step through N layers of the K3-shaped MoE: layer l has its
    own weights (seed 1000 + l) and its own seeded hidden states.  Between two
    MoE layers a model runs attention, a residual add and a norm, which this
    library does not implement; feeding one layer's raw output into the next
    would correlate the tokens and skew the routing, while the pages'
    amortisation table assumes uniform routing.  For every batch size the N
    forwards are captured once in a CUDA graph and the graph is replayed; one
    JSON line per batch size reports the step time, the experts each layer
    touched, the expert-weight bytes streamed per token, and the achieved
    bandwidth.  The pages' uniform column (GB per token at an assumed 1.5 GB
    per expert for the whole model) rides along, rescaled to this stack's
    bytes per expert, so that the two curves can be compared by shape."""
    import dataclasses
    import torch
    import synth
    import moe_expert_layer_top16_gb300 as moe
    from moe_expert_layer_top16_gb300 import build as mbuild
    from moe_expert_layer_top16_gb300.weights import encode_layer

    mbuild.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    batches = [int(b) for b in args.batches.split(",")]
    N = args.layers
    layers = [dataclasses.replace(wl, seed=1000 + l) for l in range(N)]
    plans = []
    for lw in layers:
        def fetch(name, i, lw=lw):
            if name == "bias":
                return synth.router_bias(lw, device=dev)
            return synth.weight(lw, name, i, device=dev)
        W = encode_layer(lw, fetch, dev)
        plans.append(moe.Plan(lw, W, max_tokens=max(batches)))
        del W
        torch.cuda.empty_cache()
    hbm, _, _, _ = peaks()
    pages = pages_uniform_gb_per_token()
    D, L, I, S, Is = wl.d_model, wl.d_latent, wl.expert_inter, wl.n_shared, wl.shared_inter
    per_expert = 3 * I * L * MX4_BYTES_PER_ELT                  # bytes of one routed expert in one layer
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    for B in batches:
        xs = [synth.hidden_states(lw, B, device=dev) for lw in layers]
        bufs = [torch.empty(B, D, dtype=torch.float32, device=dev) for _ in range(2)]
        # one eager pass: the experts each layer touches (the graph exports nothing)
        touched = []
        for l, plan in enumerate(plans):
            counts = torch.zeros(wl.n_experts, dtype=torch.int32, device=dev)
            plan.forward(xs[l], out=bufs[l % 2], debug={"counts": counts})
            touched.append(int((counts > 0).sum().item()))
        torch.cuda.synchronize()
        for plan in plans:
            if plan.device_status() != moe.MOE_OK:
                raise RuntimeError(f"device-side error at batch {B}")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            plans[0].forward(xs[0], out=bufs[0])               # warm-up on the capture stream
            stream.synchronize()
            with torch.cuda.graph(graph, stream=stream):
                for l, plan in enumerate(plans):
                    plan.forward(xs[l], out=bufs[l % 2])
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        steps = max(3, min(args.steps, 20))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush.fill_(float(i))
                evs[i][0].record()
                graph.replay()
                evs[i][1].record()
        torch.cuda.synchronize()
        for plan in plans:
            if plan.device_status() != moe.MOE_OK:
                raise RuntimeError(f"device-side error at batch {B}")
        ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
        routed = sum(touched) * per_expert
        dense = N * ((L + 2 * S * Is) * D + D * (L + S * Is)) * MX4_BYTES_PER_ELT
        line = {"impl": "multilayer", "workload": wl.name, "layers": N, "tokens": B, "ms_per_step": ms,
                "ms_per_layer": ms / N, "tokens_per_s": B / (ms / 1e3),
                "touched_per_layer": float(np.mean(touched)),
                "routed_weight_GB_per_token": routed / B / 1e9,
                "all_weight_GB_per_token": (routed + dense) / B / 1e9,
                "weight_GBps": (routed + dense) / (ms / 1e3) / 1e9,
                "weight_frac_hbm": (routed + dense) / (ms / 1e3) / 1e9 / hbm,
                "pages_uniform_GB_per_token": pages.get(B),
                "pages_uniform_rescaled_GB_per_token": (pages[B] / 1.5e9 * per_expert * N) if B in pages else None,
                "steps": steps, "graph": "one CUDA graph of the N forwards, replayed",
                "l2": "flushed between steps"}
        if rank == 0:
            print(json.dumps(line), flush=True)
        del graph
    for plan in plans:
        plan.close()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode64")
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=64)
    ap.add_argument("--reference-tokens", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill sub-record (the same layer at --prefill-tokens tokens)")
    ap.add_argument("--prefill-tokens", type=int, default=8192)
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches of the forward instead of replays of its CUDA graph")
    ap.add_argument("--ep-ranks", type=int, default=64,
                    help="virtual ranks of the expert-parallel dispatch/combine record (0: skip)")
    ap.add_argument("--sweep", action="store_true",
                    help="token-count sweep of the workload's layer: one JSON line per batch size")
    ap.add_argument("--layers", type=int, default=0,
                    help="multi-layer decode step: N layers with their own weights, one CUDA graph per batch size")
    ap.add_argument("--batches", default=",".join(str(b) for b in PAGES_BATCHES))
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    import synth
    wl = synth.workload(args.workload)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, wl, world, rank)
    if args.sweep:
        return run_sweep(args, wl, rank, local)
    if args.layers > 0:
        return run_multilayer(args, wl, rank, local)
    return run_cuda(args, wl, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
