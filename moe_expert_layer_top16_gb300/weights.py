"""Assemble a layer's MXFP4 weight dict from fp32 tensors, with libmoe's
own encoder (``moe_mxfp4_encode``) on the device.

`fetch(name, index)` returns one fp32 CUDA tensor: name in p_down, p_up,
w_gate, w_up, w_down (index = expert), s_gate, s_up, s_down (index = shared
expert), router; shapes [out_features][in_features].  Experts are encoded
one at a time, so the fp32 copy of the routed weights never has to exist in
full.
"""
from __future__ import annotations

import torch

from . import mxfp4_encode


def encode_layer(cfg, fetch, device) -> dict:
    E, S = cfg.n_experts, cfg.n_shared
    mixed = getattr(cfg, "precision", "mx") == "mixed"
    out = {}
    if mixed:
        # the mixed scheme keeps the projections and shared experts in bf16
        # (fp32 rounded to nearest even)
        for name in ("p_down", "p_up"):
            out[name + "_bf16"] = fetch(name, 0).to(torch.bfloat16).contiguous()
        if S > 0:
            for name in ("s_gate", "s_up", "s_down"):
                out[name + "_bf16"] = torch.stack([fetch(name, i).to(torch.bfloat16) for i in range(S)]).contiguous()
    else:
        for name in ("p_down", "p_up"):
            out[name] = mxfp4_encode(fetch(name, 0))
    shared = () if mixed else (("s_gate", S), ("s_up", S), ("s_down", S))
    for name, count in (("w_gate", E), ("w_up", E), ("w_down", E)) + shared:
        if count == 0:
            continue
        first = fetch(name, 0)
        rows, K = first.shape
        codes = torch.empty(count, rows, K // 2, dtype=torch.uint8, device=device)
        scales = torch.empty(count, rows, K // 32, dtype=torch.uint8, device=device)
        for i in range(count):
            w = first if i == 0 else fetch(name, i)
            c, s = mxfp4_encode(w)
            codes[i].copy_(c)
            scales[i].copy_(s)
            del w
        out[name] = (codes, scales)
    out["router"] = fetch("router", 0).contiguous()
    b = fetch("bias", 0)
    if b is not None:
        out["bias"] = b.contiguous()
    return out
