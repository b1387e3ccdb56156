"""Parity of the CUDA layer with the oracle under the configuration options:
routing on the hidden state instead of the latent, and a bf16 output.

The hidden-state router reads x itself (bf16, exact in fp32) with an [E][D]
router: on the K3-shaped layer at 64 tokens (fp32 SIMT router) and at 512
tokens (tensor-core router with exact refinement of the candidates).  Same
checks as the latent layer: exact top-k on the GPU's own logits and exact
dispatch over the whole batch; sampled tokens against the oracle.  A bf16
output is the fp32 result rounded once, so it must stay within the same
output tolerance.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_top16_gb300 as moe
import synth
from gpu_util import DEV, OracleLayer, gpu_plan, run_sampled_parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny+hidden", "tiny+bf16", "tiny+hidden+bf16"])
def test_tiny_options(name):
    wl = synth.workload(name)
    plan, _ = gpu_plan(wl)
    try:
        accepted, errs, counts = run_sampled_parity(wl, plan, OracleLayer(wl), wl.tokens, range(wl.tokens))
        assert len(accepted) <= 1
        assert counts.sum() == wl.tokens * wl.top_k
    finally:
        plan.close()


@pytest.fixture(scope="module")
def k3_hidden():
    wl = synth.workload("decode64+hidden")
    plan, _ = gpu_plan(wl, max_tokens=512)
    ol = OracleLayer(wl)
    yield wl, plan, ol
    plan.close()


@pytest.mark.parametrize("T", [64, 512])
def test_k3_hidden_routing(k3_hidden, T):
    wl, plan, ol = k3_hidden
    accepted, errs, counts = run_sampled_parity(wl, plan, ol, T, [0, T // 3, T - 1])
    assert len(accepted) <= 1
    assert counts.sum() == T * wl.top_k


def test_bf16_output_is_the_rounded_fp32_output():
    """Same layer, same input: the bf16 plan's y equals the fp32 plan's y
    rounded to bf16, element for element."""
    wl32 = synth.workload("tiny")
    wl16 = synth.workload("tiny+bf16")
    p32, _ = gpu_plan(wl32)
    p16, _ = gpu_plan(wl16)
    try:
        x = synth.hidden_states(wl32, device=DEV)
        y32 = p32.forward(x)
        y16 = p16.forward(x)
        torch.cuda.synchronize()
        assert y16.dtype == torch.bfloat16
        assert torch.equal(y16, y32.to(torch.bfloat16))
    finally:
        p32.close()
        p16.close()
