"""Quantile Balancing on the GPU ("Kimi K3 and the New Open-Weights Moat",
section "How the router picks 16 of 896", Fig. 2) against the oracle's
update, on the K3-shaped layer with the Zipf-shaped selection bias: from the
logits of one forward and the current bias, the new bias must equal the
oracle's (fp64 margins, exact quantile search; equal up to the final fp32
rounding).  Installed with a damped step and repeated, the updates must pull
the skewed per-expert load toward the mean."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from gpu_util import DEV, gpu_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zipf():
    wl = synth.workload("zipf16384")
    plan, _ = gpu_plan(wl, max_tokens=2048)
    yield wl, plan
    plan.close()


@pytest.mark.parametrize("T", [64, 2048])
def test_update_matches_oracle_and_balances(zipf, T):
    wl, plan = zipf
    E, k = wl.n_experts, wl.top_k
    x = synth.hidden_states(wl, T, device=DEV)
    bias = synth.router_bias(wl, device=DEV).clone()
    plan.set_bias(bias)
    target = int((T * k + E // 2) // E)
    ratios = []
    for it in range(6):
        dbg = moe.debug_buffers(wl, T, DEV, ("logits", "counts"))
        plan.forward(x, debug=dbg)
        alpha = 1.0 if it == 0 else 0.5
        new = plan.quantile_balance(T, alpha=alpha)
        torch.cuda.synchronize()
        assert plan.device_status() == moe.MOE_OK
        c = dbg["counts"].cpu().numpy()
        ratios.append(c.max() / c.mean())
        ref = oracle.quantile_balance(dbg["logits"].cpu().numpy(), bias.cpu().numpy(), k, target, alpha)
        got = new.cpu().numpy().astype(np.float64)
        assert np.abs(got - ref).max() <= 2.0 ** -22 * np.maximum(1.0, np.abs(ref)).max(), np.abs(got - ref).max()
        bias = new
        plan.set_bias(bias)
    print(f"T={T}: max/mean load per update {np.round(ratios, 2).tolist()}")
    if T >= 1024:                       # enough tokens per expert for the load to converge
        assert ratios[0] > 3.0
        assert ratios[-1] < ratios[0] / 2
    # put the workload's own bias back for the other tests of the module
    plan.set_bias(synth.router_bias(wl, device=DEV))
