"""Expert-parallel dispatch and combine emulated on one GPU ("Kimi K3: 2.8
Trillion Parameters, Four Bits at a Time", section "What it takes to serve
it"; "What Kimi K3 asks of the hardware", section "Width: 896 experts and the
interconnect").

The 896 experts of the K3-shaped layer are split into R contiguous slices
(virtual ranks).  After a forward, the dispatch packs one wire row per
(token, slot) -- header {token, expert, slot, gate}, the token's MXFP8 latent
codes and scales -- in the layer's dispatch order.  Checked against the
oracle's permutation of the GPU's selection: every rank's segment bounds,
every header field and every payload byte; the byte count per token is
k (L + L/32) of payload, against the pages' k d_model at FP8 for a hidden
state.  The combine of the experts' outputs (in wire order) must reproduce
the layer's own combine bit for bit (its MXFP8 codes and scales) and the
oracle's fp64 combine within rounding."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from gpu_util import DEV, gpu_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k3():
    wl = synth.workload("decode64")
    plan, _ = gpu_plan(wl, max_tokens=512)
    yield wl, plan
    plan.close()


@pytest.mark.parametrize("T,R", [(64, 8), (64, 64), (512, 64), (512, 896), (300, 7)])
def test_ep_dispatch_and_combine(k3, T, R):
    wl, plan = k3
    E, k, L = wl.n_experts, wl.top_k, wl.d_latent
    x = synth.hidden_states(wl, T, device=DEV)
    dbg = moe.debug_buffers(wl, T, DEV, ("topk_idx", "topk_w", "zq", "zs", "o", "cq", "cs"))
    plan.forward(x, debug=dbg)
    wire, offs = plan.ep_dispatch(T, R)
    c = plan.ep_combine(T, wire, dbg["o"])
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    g = {f: v.cpu().numpy() for f, v in dbg.items()}
    wire_h, offs_h, c_h = wire.cpu().numpy(), offs.cpu().numpy(), c.cpu().numpy()
    rb = plan.ep_row_bytes()
    assert rb == -(-(16 + L + L // 32) // 16) * 16 and wire_h.shape == (T * k, rb)
    # rank segments: the oracle's per-expert offsets at the slice boundaries
    counts, offsets, order = oracle.permute(g["topk_idx"], E)
    bounds = np.array([offsets[E * r // R] for r in range(R + 1)])
    assert np.array_equal(offs_h, bounds)
    assert offs_h[0] == 0 and offs_h[-1] == T * k and (np.diff(offs_h) >= 0).all()
    # every row: the (token, slot) of the oracle's permutation and its payload
    hdr = wire_h[:, :16].copy().view(np.int32)
    tok, slot = order // k, order % k
    assert np.array_equal(hdr[:, 0], tok) and np.array_equal(hdr[:, 2], slot)
    assert np.array_equal(hdr[:, 1], g["topk_idx"][tok, slot])
    assert np.array_equal(hdr[:, 3].view(np.float32), g["topk_w"][tok, slot])
    assert np.array_equal(wire_h[:, 16:16 + L], g["zq"][tok])
    assert np.array_equal(wire_h[:, 16 + L:16 + L + L // 32], g["zs"][tok])
    assert not wire_h[:, 16 + L + L // 32:].any()
    # every row of rank r holds an expert of rank r's slice
    for r in range(R):
        seg = hdr[offs_h[r]:offs_h[r + 1], 1]
        assert ((seg >= E * r // R) & (seg < E * (r + 1) // R)).all()
    payload = k * (L + L // 32)
    print(f"T={T} R={R}: {payload} payload bytes per token dispatched (pages: k d_model = {k * wl.d_model} at FP8 "
          f"for a hidden state), rows per rank {np.diff(offs_h).min()}..{np.diff(offs_h).max()}")
    # the combine of the experts' outputs in wire order is the layer's combine
    cq, cs = oracle.mxfp8_quantize(c_h)
    assert np.array_equal(cq, g["cq"]) and np.array_equal(cs, g["cs"])
    o_tok = np.zeros((T, k, L))
    o_tok[tok, slot] = g["o"].astype(np.float64)
    ref = np.einsum("tj,tjl->tl", g["topk_w"].astype(np.float64), o_tok)
    assert np.abs(c_h - ref).max() <= 1e-6 * np.abs(ref).max()
