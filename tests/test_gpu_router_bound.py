"""The tensor-core router estimate and its proven error bound under inputs
built to break a fixed error band.

Above 128 tokens the layer estimates the logits with one TF32 product on the
tensor cores and recomputes in exact fp32 only the candidates whose key
interval (estimate +- the per-(token, expert) bound) reaches the k-th largest
lower end.  The bound scales with |z_t| |R_e|, so it holds for any input
scale.  Two adversarial variants of the K3-shaped layer push the estimate
error far beyond a fixed band of 2e-2:
  * hidden states scaled by 64 (every logit and every estimate error 64x);
  * eight router rows scaled by 64 (their experts' logits and errors 64x).
The selection must still be exact: on the exported logits for the whole
batch, and against the oracle (no near-ties) on sampled tokens, with every
estimate inside the proven bound."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from moe_expert_layer_top16_gb300.weights import encode_layer
from gpu_util import DEV, OracleLayer, fetch_device, route_exact_on_exports, sampled_y

pytestmark = pytest.mark.gpu

BIG_ROWS = [3, 100, 257, 400, 511, 640, 777, 895]


class ScaledRouterLayer(OracleLayer):
    """The oracle's weights of the layer with eight router rows scaled."""

    def __init__(self, wl):
        super().__init__(wl)
        r = self.enc["router"].copy()
        r[BIG_ROWS] *= 64.0
        self.enc["router"] = r
        self._lw = None


def plan_for(wl, scaled_rows):
    base = fetch_device(wl)

    def fetch(name, i):
        w = base(name, i)
        if name == "router" and scaled_rows:
            w = w.clone()
            w[BIG_ROWS] *= 64.0
        return w

    return moe.Plan(wl, encode_layer(wl, fetch, DEV), max_tokens=1024)


@pytest.fixture(scope="module")
def layers():
    wl = synth.workload("decode64")
    plain, scaled = plan_for(wl, False), plan_for(wl, True)
    yield wl, (plain, OracleLayer(wl)), (scaled, ScaledRouterLayer(wl))
    plain.close()
    scaled.close()


def run(wl, plan, ol, x, T):
    fields = ("xq", "xs", "z", "logits", "topk_idx", "topk_w", "counts", "offsets", "sorted_token")
    dbg = moe.debug_buffers(wl, T, DEV, fields)
    y = plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    g = {k: v.cpu().numpy() for k, v in dbg.items()}
    y = y.float().cpu().numpy()
    assert np.isfinite(y).all()
    route_exact_on_exports(wl, ol, g)
    sample = np.linspace(0, T - 1, num=24).astype(int)
    accepted, errs, est_err = sampled_y(wl, ol, T, x, g, y, sample)
    return accepted, est_err


@pytest.mark.parametrize("T", [300, 1024])
def test_scaled_hidden_states(layers, T):
    wl, (plan, ol), _ = layers
    x = synth.hidden_states(wl, T, device=DEV) * 64          # exact in bf16: a power of two
    accepted, est_err = run(wl, plan, ol, x, T)
    assert len(accepted) == 0
    assert est_err > 2e-2, f"the inputs did not push the estimate error past 2e-2 ({est_err:.3e})"


@pytest.mark.parametrize("T", [300, 1024])
def test_scaled_router_rows(layers, T):
    wl, _, (plan, ol) = layers
    x = synth.hidden_states(wl, T, device=DEV)
    accepted, est_err = run(wl, plan, ol, x, T)
    assert len(accepted) == 0
    assert est_err > 2e-2, f"the inputs did not push the estimate error past 2e-2 ({est_err:.3e})"
