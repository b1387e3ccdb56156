"""The forward's launch paths give bit-identical outputs.

A plain forward launches its kernels with programmatic dependent launch and,
from 1024 tokens on, runs the shared experts' gate/up on the plan's side
stream (beside the routing steps, or, in a captured forward, beside the
combine).  With per-stage events recorded it launches
every kernel plainly, one after another, on the caller's stream.  The same
kernels run on the same data in the same order of accumulation, so y (and
every intermediate a later step reads) must be equal bit for bit, and
repeated forwards must reproduce it: the layer's output does not depend on
scheduling.  Checked on the K3-shaped layer at 64 and 2048 tokens, and for
a forward captured in a CUDA graph and replayed.
"""
import pytest
import torch

import moe_expert_layer_top16_gb300 as moe
import synth
from gpu_util import DEV, gpu_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def k3():
    wl = synth.workload("decode64")
    plan, _ = gpu_plan(wl, max_tokens=2048)
    yield wl, plan
    plan.close()


@pytest.mark.parametrize("T", [64, 2048])
def test_launch_paths_bit_identical(k3, T):
    wl, plan = k3
    x = synth.hidden_states(wl, T, device=DEV)
    y_fast = plan.forward(x).clone()
    y_again = plan.forward(x).clone()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(moe.NUM_STAGES + 1)]
    for e in events:                      # torch creates CUDA events at their first record
        e.record()
    y_plain = plan.forward(x, stage_events=events).clone()
    # the same forward captured once in a CUDA graph and replayed
    y_graph = torch.empty_like(y_fast)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device=DEV)
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        plan.forward(x, out=y_graph)
        cs.synchronize()
        with torch.cuda.graph(g, stream=cs):
            plan.forward(x, out=y_graph)
    torch.cuda.current_stream().wait_stream(cs)
    y_graph.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    assert torch.isfinite(y_fast).all()
    assert torch.equal(y_fast, y_again)
    assert torch.equal(y_fast, y_plain)
    assert torch.equal(y_fast, y_graph)
    del g
