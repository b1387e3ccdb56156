"""Parity of the CUDA layer with the oracle under the mixed precision scheme
of "Kimi K3 and the New Open-Weights Moat", section "Precision and
deployment", Fig. 6: MXFP4 weights and MXFP8 inputs on the routed experts
only; the latent projections and the shared experts run on the bf16 tensor
cores (kind::f16) with bf16 weights and bf16 inputs (x as given, the shared
activation and the combine output rounded to bf16).

Same contract as the all-MX layer: exact top-k on the exported logits and
exact dispatch over the whole batch; sampled tokens against the oracle
(selected logits exact, tensor-core estimates within the proven bound,
selections equal) and y within max |err| <= 2e-2 rms(y_ref),
sum|err| / sum|y_ref| <= 2e-3.  On the small layer the latent z is also
compared element by element (the projection's fp32 accumulation against the
oracle's fp64 sum)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from gpu_util import DEV, OracleLayer, bf16_bits, gpu_plan, run_sampled_parity

pytestmark = pytest.mark.gpu


def test_tiny_mixed():
    wl = synth.workload("tiny+mixed")
    plan, _ = gpu_plan(wl)
    try:
        ol = OracleLayer(wl)
        accepted, errs, counts = run_sampled_parity(wl, plan, ol, wl.tokens, range(wl.tokens))
        assert len(accepted) == 0
        x = synth.hidden_states(wl, device=DEV)
        dbg = moe.debug_buffers(wl, wl.tokens, DEV, ("z", "zq", "zs"))
        plan.forward(x, debug=dbg)
        torch.cuda.synchronize()
        ref = oracle.moe_forward(wl, ol.ensure([]), bf16_bits(x), route_only=True, want=("z",))
        z = dbg["z"].cpu().numpy().astype(np.float64)
        assert np.sqrt(np.mean((z - ref["z"]) ** 2)) <= 1e-5 * np.sqrt(np.mean(ref["z"].astype(np.float64) ** 2))
    finally:
        plan.close()


@pytest.fixture(scope="module")
def k3_mixed():
    wl = synth.workload("decode64+mixed")
    plan, _ = gpu_plan(wl, max_tokens=4096)
    ol = OracleLayer(wl)
    yield wl, plan, ol
    plan.close()


@pytest.mark.parametrize("T", [1, 64, 512, 4096])
def test_k3_mixed(k3_mixed, T):
    wl, plan, ol = k3_mixed
    accepted, errs, counts = run_sampled_parity(wl, plan, ol, T, np.linspace(0, T - 1, num=min(T, 16)).astype(int))
    assert len(accepted) == 0
    assert counts.sum() == T * wl.top_k
