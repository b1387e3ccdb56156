"""Top-k on exact ties, at every selection path of the CUDA layer.

The K3-shaped layer with a router whose rows come in identical pairs
(row 2i + 1 = row 2i): the logits of experts 2i and 2i + 1 are then equal
bit for bit, estimates and exact values alike, so every selection meets
ties and must break them toward the lower expert id.  64 tokens take the
one-CTA-per-token path on exact logits, 300 tokens the warp-per-token path
refining tensor-core estimates, 1024 tokens the same above the small-batch
limit.  On the logits the GPU exports, its selection, slot order and gates
must equal the oracle's selection rule exactly; the dispatch built from the
selection must be exact too.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from moe_expert_layer_top16_gb300.weights import encode_layer
from gpu_util import DEV, fetch_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def paired():
    wl = synth.workload("decode64")
    base = fetch_device(wl)

    def fetch(name, i):
        w = base(name, i)
        if name == "router":
            w = w.clone()
            w[1::2] = w[0::2]
        return w

    plan = moe.Plan(wl, encode_layer(wl, fetch, DEV), max_tokens=1024)
    yield wl, plan
    plan.close()


@pytest.mark.parametrize("T", [64, 300, 1024])
def test_paired_router_ties(paired, T):
    wl, plan = paired
    x = synth.hidden_states(wl, T, device=DEV)
    dbg = moe.debug_buffers(wl, T, DEV, ("logits", "topk_idx", "topk_w", "counts", "offsets", "sorted_token"))
    plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    g = {k: v.cpu().numpy() for k, v in dbg.items()}
    lg = g["logits"]
    E, k = wl.n_experts, wl.top_k
    # the pairs tie on the exported logits (exact values and estimates alike)
    assert np.array_equal(lg[:, 0::2], lg[:, 1::2])
    idx_ref, gates_ref = oracle.route(lg, k, softmax=(wl.score == "softmax"), bias=None)
    assert np.array_equal(g["topk_idx"], idx_ref)
    np.testing.assert_allclose(g["topk_w"], gates_ref, rtol=3e-6, atol=1e-7)
    # an odd expert is only ever taken right after its even twin
    for t in range(T):
        sel = list(g["topk_idx"][t])
        for j, e in enumerate(sel):
            if e % 2:
                assert j > 0 and sel[j - 1] == e - 1, f"token {t}: {sel}"
    counts, offsets, order = oracle.permute(g["topk_idx"], E)
    assert np.array_equal(g["counts"], counts) and np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["sorted_token"], order // k)
