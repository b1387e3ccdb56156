"""Seeded synthetic inputs for the K3-shaped sparse MoE layer.

This module draws random tensors and nothing else: it holds none of the
layer's arithmetic (no quantisation, no routing, no GEMM).  Both sides of
every parity check -- the CPU oracle under ``oracle/`` and the CUDA path in
``moe_expert_layer_top16_gb300`` -- take their inputs from here.

Workload shapes follow the Kimi K3 layer described on the pages
("Kimi K3 and the New Open-Weights Moat", section "Sparse computation:
latent experts and routing"): 896 routed experts, top-16, two shared
experts at width 7168, routed path in a 3584-wide latent.  The routed and
shared inner widths (512 and 2048) are not on the pages; they are the
assumed values of the workload definitions below.

Distributions:
  * hidden states x ~ N(0, 1), rounded to bf16 (round-to-nearest-even);
  * every weight ~ N(0, 0.02) in fp32 (the MX weights are encoded from these
    by each side's own encoder);
  * router weights ~ N(0, 0.02) in fp32;
  * selection bias: zero, except for the skewed workload, where expert ranks
    come from a seeded permutation and b_e = -1.1 * ZIPF_GAMMA * ln(rank_e),
    so that the bias follows Zipf(s=1.1) log-popularity.

Every tensor has its own seed, derived from (master seed, tensor name,
index), so any single expert can be regenerated without the others.
Generation uses torch's generator on the requested device; the CPU and CUDA
generators give different streams, so a check that needs the same tensor on
both sides draws it once and copies it.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, replace
from typing import Optional

import torch

# Strength of the Zipf-shaped selection bias (see module docstring).  With
# logits of std ~2 this makes the hottest experts receive well over 10x the
# mean load; the realised histogram is measured, not assumed.
ZIPF_GAMMA = 0.05
ZIPF_S = 1.1
WEIGHT_STD = 0.02


@dataclass(frozen=True)
class Workload:
    name: str
    d_model: int
    d_latent: int
    n_experts: int
    top_k: int
    expert_inter: int
    n_shared: int
    shared_inter: int
    tokens: int
    score: str          # "sigmoid" (sigmoid + selection bias) or "softmax" (toy gates)
    bias: str           # "zero" or "zipf"
    seed: int = 0
    route: str = "latent"   # router input: "latent" (z, [E][L] router) or "hidden" (x, [E][D] router)
    out: str = "f32"        # output dtype of y: "f32" or "bf16"
    precision: str = "mx"   # "mx": every weight MXFP4; "mixed": bf16 latent projections and shared experts

    def with_tokens(self, t: int) -> "Workload":
        return replace(self, tokens=int(t), name=f"{self.name.split('@')[0]}@T{t}")


K3 = dict(d_model=7168, d_latent=3584, n_experts=896, top_k=16, expert_inter=512,
          n_shared=2, shared_inter=2048, score="sigmoid")

WORKLOADS = {
    # Small layer the oracle finishes in well under a second.
    "tiny": Workload("tiny", d_model=256, d_latent=128, n_experts=32, top_k=4,
                     expert_inter=64, n_shared=1, shared_inter=128, tokens=64,
                     score="softmax", bias="zero", seed=0),
    # K3-shaped layer, decode-sized batch.
    "decode64": Workload("decode64", tokens=64, bias="zero", seed=0, **K3),
    # K3-shaped layer, prefill-sized batch.
    "prefill8192": Workload("prefill8192", tokens=8192, bias="zero", seed=0, **K3),
    # K3-shaped layer, skewed routing through a Zipf-shaped selection bias.
    "zipf16384": Workload("zipf16384", tokens=16384, bias="zipf", seed=0, **K3),
}
SWEEP_TOKENS = (1, 8, 64, 512, 4096, 32768)


def workload(name: str) -> Workload:
    """A named workload; "name@T<n>" overrides the token count, "name+hidden"
    routes on the hidden state, "name+bf16" writes a bf16 output, "name+mixed"
    keeps the latent projections and shared experts in bf16 (only the routed
    experts MXFP4)."""
    base, *opts = name.split("+")
    if "@T" in base:
        b, t = base.split("@T")
        w = WORKLOADS[b].with_tokens(int(t))
    else:
        w = WORKLOADS[base]
    for o in opts:
        if o == "hidden":
            w = replace(w, route="hidden")
        elif o == "bf16":
            w = replace(w, out="bf16")
        elif o == "mixed":
            w = replace(w, precision="mixed")
        else:
            raise KeyError(name)
    if opts:
        w = replace(w, name=name)
    return w


def tensor_seed(master: int, name: str, index: int = 0) -> int:
    h = hashlib.blake2b(f"{master}/{name}/{index}".encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _normal(shape, std: float, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


# Weight tensors: name -> (shape function, count function).  Shapes are
# [out_features][in_features], i.e. the reduction dim is innermost.
def weight_shape(w: Workload, name: str):
    D, L, I, Is = w.d_model, w.d_latent, w.expert_inter, w.shared_inter
    return {
        "p_down": (L, D), "p_up": (D, L),
        "w_gate": (I, L), "w_up": (I, L), "w_down": (L, I),
        "s_gate": (Is, D), "s_up": (Is, D), "s_down": (D, Is),
        "router": (w.n_experts, L if w.route == "latent" else D),
    }[name]


def weight_count(w: Workload, name: str) -> int:
    if name in ("w_gate", "w_up", "w_down"):
        return w.n_experts
    if name in ("s_gate", "s_up", "s_down"):
        return w.n_shared
    return 1


def weight(w: Workload, name: str, index: int = 0, device="cpu") -> torch.Tensor:
    """fp32 weight tensor `name` (expert / shared-expert `index`), ~N(0, 0.02)."""
    if not 0 <= index < weight_count(w, name):
        raise IndexError(f"{name}[{index}]")
    return _normal(weight_shape(w, name), WEIGHT_STD, tensor_seed(w.seed, name, index), device)


def hidden_states(w: Workload, tokens: Optional[int] = None, device="cpu", offset: int = 0) -> torch.Tensor:
    """bf16 hidden states [T][d_model] ~ N(0, 1).

    Rows are drawn in 1024-row chunks with their own seeds, so row r is the
    same whatever T is; `offset` selects the first row.
    """
    T = w.tokens if tokens is None else int(tokens)
    out = torch.empty(T, w.d_model, dtype=torch.bfloat16, device=device)
    CH = 1024
    r = 0
    while r < T:
        row = offset + r
        chunk, within = divmod(row, CH)
        blk = _normal((CH, w.d_model), 1.0, tensor_seed(w.seed, "x", chunk), device)
        n = min(CH - within, T - r)
        out[r:r + n] = blk[within:within + n].to(torch.bfloat16)
        r += n
    return out


def router_bias(w: Workload, device="cpu") -> Optional[torch.Tensor]:
    """Selection bias [E] (fp32) or None when the workload has none."""
    if w.bias == "zero":
        return None
    if w.bias != "zipf":
        raise ValueError(w.bias)
    g = torch.Generator(device="cpu")
    g.manual_seed(tensor_seed(w.seed, "zipf_rank"))
    perm = torch.randperm(w.n_experts, generator=g)
    rank = torch.empty(w.n_experts, dtype=torch.float64)
    rank[perm] = torch.arange(1, w.n_experts + 1, dtype=torch.float64)
    b = (-ZIPF_S * ZIPF_GAMMA) * torch.log(rank)
    return b.to(torch.float32).to(device)
