"""Benchmark of the K3-shaped sparse MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one forward pass of the whole layer (every stage of moe_forward)
over one batch of synthetic tokens of the workload (default: the K3-shaped
decode batch, 64 tokens).  Inputs and weights are resident in HBM before the
timed region; L2 is flushed (a 512 MB write) between timed steps, outside the
per-step CUDA events.  Prints one JSON line (rank 0).

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

# DRAM bytes (read + write) per launch of a stage's kernel from one ncu
# capture, and the commit the capture was taken at; a capture stands only
# until its kernel changes (summaries under profiles/).
NCU_TRAFFIC = {
    ("decode64", "gemm_gate_up"): (1.331121e9 + 3.783424e6, "60ceff4", "profiles/gate_up_decode64.md"),
    ("prefill8192", "gemm_gate_up"): (2.266878e9 + 69.639424e6, "60ceff4", "profiles/gate_up_prefill8192.md"),
}


def workload_config(wl, T):
    """The `config` keys both arms report for a workload of T tokens."""
    return {"workload": wl.name, "tokens": T, "d_model": wl.d_model, "d_latent": wl.d_latent,
            "experts": wl.n_experts, "top_k": wl.top_k, "expert_inter": wl.expert_inter,
            "shared": wl.n_shared, "shared_inter": wl.shared_inter, "bias": wl.bias}


def launches_per_forward(T):
    """Kernels of this library one forward of T tokens launches: quantiser, A2,
    router (or its tensor-core estimate), top-k, per-expert scan (batches over
    128 tokens; folded into the work-list kernel below that), work lists,
    dispatch, A7, A8, combine, A10."""
    return 10 + (1 if (T + 31) // 32 > 4 else 0)


def algorithmic_work(wl, T, counts):
    """Per-stage algorithmic bytes and MX FLOPs of one forward of T tokens.
    `counts` = realised tokens per expert (touched experts are those > 0)."""
    D, L, E, k, I, S, Is = (wl.d_model, wl.d_latent, wl.n_experts, wl.top_k, wl.expert_inter, wl.n_shared,
                            wl.shared_inter)
    touched = int((np.asarray(counts) > 0).sum())
    TK = T * k
    rows_a2 = L + 2 * S * Is
    kcat = L + S * Is
    w = {
        "gemm_down_shared": (rows_a2 * D * MX4_BYTES_PER_ELT + T * D * MX8_BYTES_PER_ELT
                             + T * L * (4 + MX8_BYTES_PER_ELT) + T * S * Is * MX8_BYTES_PER_ELT,
                             2.0 * T * rows_a2 * D),
        "router": (E * L * 4 + T * L * 4 + T * E * 4, 2.0 * T * E * L),
        "gemm_gate_up": (touched * 2 * I * L * MX4_BYTES_PER_ELT + TK * L * MX8_BYTES_PER_ELT
                         + TK * I * MX8_BYTES_PER_ELT, 2.0 * TK * 2 * I * L),
        "gemm_down": (touched * L * I * MX4_BYTES_PER_ELT + TK * I * MX8_BYTES_PER_ELT + TK * L * 4,
                      2.0 * TK * L * I),
        "combine": (TK * L * 4 + T * L * MX8_BYTES_PER_ELT, 2.0 * TK * L),
        "gemm_up_shared": (D * kcat * MX4_BYTES_PER_ELT + T * kcat * MX8_BYTES_PER_ELT + T * D * 4,
                           2.0 * T * D * kcat),
        "quant_x": (T * D * (2 + MX8_BYTES_PER_ELT), 0.0),
        "dispatch": (TK * L * MX8_BYTES_PER_ELT * 2, 0.0),
    }
    expert_weight_bytes = touched * 3 * I * L * MX4_BYTES_PER_ELT + 3 * S * Is * D * MX4_BYTES_PER_ELT
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

    def fetch(name, i):
        if name == "bias":
            return synth.router_bias(wl, device=dev)
        return synth.weight(wl, name, i, device=dev)

    W = encode_layer(wl, fetch, dev)
    plan = moe.Plan(wl, W, max_tokens=T)
    del W
    torch.cuda.empty_cache()
    x = synth.hidden_states(wl, T, device=dev, offset=rank * T)
    y = torch.empty(T, wl.d_model, dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    counts = torch.zeros(wl.n_experts, dtype=torch.int32, device=dev)

    nst = moe.NUM_STAGES
    # warm-up (also captures the realised expert histogram)
    for i in range(max(args.warmup, 1)):
        plan.forward(x, out=y, debug={"counts": counts} if i == 0 else None)
    torch.cuda.synchronize()
    if plan.device_status() != moe.MOE_OK:
        raise RuntimeError("device-side error during warm-up")
    counts_h = counts.cpu().numpy()

    K = args.steps
    # per-stage breakdown: a separate, untimed pass with events between the stages
    n_stage = min(K, 20)
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
                         for i in range(n_stage)])

    # timed region: exactly K forwards, each between two events on the forward's
    # stream; the L2 flush sits between steps, outside the events
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(float(i))                       # L2 flush, outside the step events
        ev0[i].record()
        plan.forward(x, out=y)
        ev1[i].record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if plan.device_status() != moe.MOE_OK:
        raise RuntimeError("device-side error in the timed region")

    step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(K)]
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

    hbm, bf16, bf16_sus, peak_kind = peaks()
    work, touched, expert_bytes = algorithmic_work(wl, T, counts_h)
    mean_stage = stage_ms.mean(axis=0)
    names = moe.STAGE_NAMES
    dom = int(np.argmax(mean_stage))
    dom_name = names[dom]
    bytes_, flops = work.get(dom_name, (0.0, 0.0))
    stage_s = mean_stage[dom] / 1e3
    key = (wl.name, dom_name)
    traffic = NCU_TRAFFIC[key][0] if key in NCU_TRAFFIC else None
    # decode-sized batches are judged on HBM bytes, prefill-sized ones (4096
    # tokens and up) on the tensor pipe; the other roof's fraction rides along,
    # since a grouped GEMM near 150 tokens per expert sits at the ridge of both
    peak_t = bf16 * 2.0          # W4A8 block-scaled MMA: measured bf16 peak x nominal mxf8f6f4 / bf16 (4.5 / 2.25)
    t_roof = {"bound": "tensor", "kernel": dom_name, "achieved": flops / stage_s / 1e12, "peak": peak_t,
              "unit": "TFLOP/s", "frac": flops / stage_s / 1e12 / peak_t, "traffic": traffic,
              "peak_source": f"{peak_kind} bf16 burst {bf16} TFLOP/s x 2 (nominal fp8/bf16 ratio)"}
    h_roof = {"bound": "hbm", "kernel": dom_name, "achieved": bytes_ / stage_s / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": bytes_ / stage_s / 1e9 / hbm, "traffic": traffic, "peak_source": f"{peak_kind} copy bandwidth"}
    tensor_bound = T >= 4096 and flops > 0
    roof, other = (t_roof, h_roof) if tensor_bound else (h_roof, t_roof)
    roof["other_roof"] = {"bound": other["bound"], "achieved": other["achieved"], "unit": other["unit"],
                          "frac": other["frac"]}
    if traffic is not None:
        roof["traffic_source"] = f"ncu dram__bytes_read.sum + dram__bytes_write.sum, {NCU_TRAFFIC[key][2]}, " \
                                 f"commit {NCU_TRAFFIC[key][1]}"
    layer_bytes = sum(b for b, _ in work.values())
    layer_flops = sum(f for _, f in work.values())
    step_s = ms_per_step / 1e3
    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "step_ms": {"median": float(np.median(step_ms)), "p10": float(np.percentile(step_ms, 10)),
                    "p90": float(np.percentile(step_ms, 90))},
        "dtype": "mxfp4 weights x mxfp8 activations, fp32 accumulate", "data": "synthetic",
        "config": dict(workload_config(wl, T),
                       l2="flushed by a 512 MB write between timed steps (outside the step events)",
                       parallelism=f"replicas x{world}"),
        "roofline": roof,
        "layer": {"touched_experts": touched, "expert_weight_bytes": expert_bytes,
                  "expert_weight_GBps": expert_bytes / step_s / 1e9,
                  "expert_weight_frac_hbm": expert_bytes / step_s / 1e9 / hbm,
                  "algorithmic_bytes": layer_bytes, "mx_tflops": layer_flops / step_s / 1e12,
                  "mx_frac_fp8_peak": layer_flops / step_s / 1e12 / (bf16 * 2.0),
                  # the same against the FP4-only rate (kind::mxf4, nominally 6x bf16), which a
                  # W4A8 product cannot reach: at most 1/3 of it
                  "mx_frac_fp4_peak": layer_flops / step_s / 1e12 / (bf16 * 6.0),
                  "max_over_mean_load": float(counts_h.max() / max(counts_h.mean(), 1e-9)),
                  "stage_ms": {n: float(v) for n, v in zip(names, mean_stage)}},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": int(T * wl.d_model * 2),
                "d2h_bytes_per_step": int(T * wl.d_model * 4)},
        "gpu_launches": launches_per_forward(T) * K,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
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
    for T in synth.SWEEP_TOKENS:
        x = synth.hidden_states(wl, T, device=dev)
        y = torch.empty(T, wl.d_model, dtype=plan.out_dtype, device=dev)
        counts = torch.zeros(wl.n_experts, dtype=torch.int32, device=dev)
        for i in range(args.warmup):
            plan.forward(x, out=y, debug={"counts": counts} if i == 0 else None)
        torch.cuda.synchronize()
        steps = max(5, min(args.steps, (200 * 64) // T))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for i in range(steps):
            flush.fill_(float(i))
            ev[i][0].record()
            plan.forward(x, out=y)
            ev[i][1].record()
        torch.cuda.synchronize()
        if plan.device_status() != moe.MOE_OK:
            raise RuntimeError(f"device-side error at T={T}")
        ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
        work, touched, expert_bytes = algorithmic_work(wl, T, counts.cpu().numpy())
        flops = sum(f for _, f in work.values())
        line = {"impl": "sweep", "workload": wl.name, "tokens": T, "ms_median": ms, "tokens_per_s": T / (ms / 1e3),
                "touched_experts": touched, "expert_weight_GBps": expert_bytes / (ms / 1e3) / 1e9,
                "expert_weight_frac_hbm": expert_bytes / (ms / 1e3) / 1e9 / hbm,
                "mx_tflops": flops / (ms / 1e3) / 1e12, "mx_frac_fp8_peak": flops / (ms / 1e3) / 1e12 / (bf16 * 2.0),
                "steps": steps, "l2": "flushed between steps"}
        if rank == 0:
            print(json.dumps(line), flush=True)
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
    ap.add_argument("--sweep", action="store_true",
                    help="token-count sweep of the workload's layer: one JSON line per batch size")
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
    return run_cuda(args, wl, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
