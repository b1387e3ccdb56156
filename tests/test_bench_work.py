"""The measurement arithmetic of bench.py, checked against figures derived by
hand from the layer's shapes: MXFP4 costs 17/32 bytes per element (4-bit
codes plus one 8-bit scale per 32), one K3 routed expert (gate, up, down of
inner 512 on the 3584 latent) is 5,505,024 elements, and the MX work of one
token is the four block-scaled GEMMs' multiply-adds."""
import importlib.util
import os

import numpy as np

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_expert_weight_bytes():
    b = _bench()
    wl = synth.workload("decode64")
    counts = np.zeros(wl.n_experts, np.int32)
    counts[:1] = 1
    _, touched, one = b.algorithmic_work(wl, 1, counts)
    shared = 3 * 2 * 2048 * 7168 * 17 // 32              # 46,792,704 B
    assert touched == 1
    assert one == 2_924_544 + shared                      # 5,505,024 elements x 17/32
    counts[:] = 3
    _, touched, allb = b.algorithmic_work(wl, 168, counts)
    assert touched == 896
    assert allb == 896 * 2_924_544 + shared               # all routed experts: 2.620 GB


def test_mx_flops_per_token():
    b = _bench()
    wl = synth.workload("decode64")
    counts = np.ones(wl.n_experts, np.int32)
    work, _, _ = b.algorithmic_work(wl, 64, counts)
    mx = sum(work[s][1] for s in ("gemm_down_shared", "gemm_gate_up", "gemm_down", "gemm_up_shared"))
    # projections + shared (2 x 11776 x 7168 + 2 x 7168 x 7680) and routed (16 x 2 x (1024 + 512) x 3584)
    assert mx / 64 == 455_081_984


def test_launches_per_forward():
    b = _bench()
    # the per-expert scan is its own kernel above 128 tokens (four bitmap words)
    assert b.launches_per_forward(1) == 10
    assert b.launches_per_forward(128) == 10
    assert b.launches_per_forward(129) == 11
    assert b.launches_per_forward(8192) == 11


def test_mixed_scheme_bytes():
    """In the mixed scheme the projections and shared experts move 2 bytes per
    weight element: the shared experts' 3 x 2 x 2048 x 7168 = 88,080,384
    elements are 176,160,768 bytes instead of 46,792,704, and one quantiser
    launch fewer."""
    b = _bench()
    wl = synth.workload("decode64+mixed")
    counts = np.zeros(wl.n_experts, np.int32)
    counts[0] = 1
    _, touched, b1 = b.algorithmic_work(wl, 1, counts)
    assert touched == 1
    assert b1 == 2_924_544 + 176_160_768
    work, _, _ = b.algorithmic_work(wl, 64, counts)
    assert work["gemm_down_shared"][0] >= (3584 + 2 * 2 * 2048) * 7168 * 2
    assert b.launches_per_forward(64, wl) == 9 and b.launches_per_forward(64, synth.workload("decode64")) == 10


def test_traffic_record_used_only_for_its_sources(tmp_path):
    # The stored ncu traffic of a workload is reported only while the kernel
    # sources hash to the value recorded with it; a stale record, a missing
    # workload or a missing file reads as no capture.
    import json
    b = _bench()
    h = b.kernel_source_hash()
    assert len(h) == 16 and all(c in "0123456789abcdef" for c in h)
    rec = {"source_hash": h, "layer_dram_bytes": 123.0, "kernels": {"gemm_gate_up": 100.0}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps({"w": rec, "old": dict(rec, source_hash="0" * 16)}))
    b.TRAFFIC_FILE = str(path)
    assert b.ncu_traffic("w") == (123.0, {"gemm_gate_up": 100.0})
    assert b.ncu_traffic("old") == (None, None)
    assert b.ncu_traffic("absent") == (None, None)
    b.TRAFFIC_FILE = str(tmp_path / "missing.json")
    assert b.ncu_traffic("w") == (None, None)
