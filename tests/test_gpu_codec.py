"""GPU MX codecs against the oracle, bit-exact on identical inputs.

MXFP8 activation quantisation ("Kimi K3 and the New Open-Weights Moat",
section "Precision and deployment", Fig. 6) is checked over every finite
bf16 value through the layer's first step; the MXFP4 weight encoder ("Kimi
K3: 2.8 Trillion Parameters, Four Bits at a Time", section "Four bits from
the start") over random blocks, planted ties, zeros and extreme exponents.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from gpu_util import DEV, gpu_plan

pytestmark = pytest.mark.gpu


def finite_bf16_patterns():
    allb = np.arange(65536, dtype=np.uint32)
    return allb[((allb >> 7) & 0xFF) != 0xFF]


def test_quant_x_every_finite_bf16_bit_exact():
    wl = synth.workload("tiny")
    pats = finite_bf16_patterns()
    rng = np.random.default_rng(3)
    D = wl.d_model
    rows_sorted = pats[: (len(pats) // D) * D].reshape(-1, D)
    rows_mixed = rng.permutation(pats)[: 64 * D].reshape(-1, D)
    bits = np.concatenate([rows_sorted, rows_mixed]).astype(np.uint16)
    T = bits.shape[0]
    plan, _ = gpu_plan(wl, max_tokens=T)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    dbg = moe.debug_buffers(wl, T, DEV, fields=("xq", "xs"))
    plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    q_ref, s_ref = oracle.mxfp8_quantize(xf)
    s_gpu = dbg["xs"].cpu().numpy()
    q_gpu = dbg["xq"].cpu().numpy()
    assert (s_gpu == s_ref).all(), f"scale mismatches: {int((s_gpu != s_ref).sum())}"
    mism = np.argwhere(q_gpu != q_ref)
    assert mism.size == 0, f"{len(mism)} code mismatches, first {[(int(bits[r, c]), int(q_gpu[r, c]), int(q_ref[r, c])) for r, c in mism[:8]]}"


@pytest.mark.parametrize("route", ["latent", "hidden"])
def test_quant_x_odd_tile_count_bit_exact(route):
    # d_model = 384: three 128-wide tiles, so the quantiser's last 256-wide
    # span has one tile and the upper half of its warp stores nothing; 203
    # tokens leave a ragged last token tile.  Hidden routing also has the
    # kernel write x as fp32.
    wl = dataclasses.replace(synth.workload("tiny"), name="tiny384", d_model=384, route=route)
    pats = finite_bf16_patterns()
    rng = np.random.default_rng(11)
    T = 203
    bits = rng.choice(pats, size=(T, wl.d_model)).astype(np.uint16)
    plan, _ = gpu_plan(wl, max_tokens=T)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    dbg = moe.debug_buffers(wl, T, DEV, fields=("xq", "xs"))
    plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    xf = (bits.astype(np.uint32) << 16).view(np.float32)
    q_ref, s_ref = oracle.mxfp8_quantize(xf)
    assert (dbg["xs"].cpu().numpy() == s_ref).all()
    assert (dbg["xq"].cpu().numpy() == q_ref).all()


def _encoder_inputs():
    rng = np.random.default_rng(17)
    blocks = [rng.normal(0, 0.02, size=(512, 256)).astype(np.float32)]
    w = rng.normal(size=(64, 256)).astype(np.float32)
    w *= np.float32(2.0) ** rng.integers(-140, 120, size=(64, 8)).repeat(32, axis=1).astype(np.float32)
    blocks.append(w)
    # exact midpoints of the E2M1 grid at scale 1 (amax 4 in the block)
    mids = np.array([4.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, 0.0,
                     -0.0, 6.0, 7.0, 1e-30, -1e-38, 3.0, 2.0, 0.5] + [1.0] * 8, np.float32)
    blocks.append(np.tile(mids, (4, 8)))
    z = np.zeros((4, 256), np.float32)
    z[1, 40] = -0.0
    z[2, :32] = 1e-45          # smallest subnormals
    blocks.append(z)
    return np.concatenate(blocks)


def test_mxfp4_encoder_matches_oracle():
    w = _encoder_inputs()
    c_ref, s_ref = oracle.mxfp4_encode(w)
    c, s = moe.mxfp4_encode(torch.from_numpy(w).to(DEV))
    torch.cuda.synchronize()
    c = c.cpu().numpy()
    s = s.cpu().numpy()
    assert (s == s_ref).all(), f"scale mismatches {int((s != s_ref).sum())}"
    assert (c == c_ref).all(), f"code mismatches {int((c != c_ref).sum())}"


def test_mxfp4_encoder_on_k3_expert_matches_oracle():
    wl = synth.workload("decode64")
    for name in ("w_gate", "w_down"):
        w = synth.weight(wl, name, 5, device=DEV)
        c, s = moe.mxfp4_encode(w)
        c_ref, s_ref = oracle.mxfp4_encode(w.cpu().numpy())
        assert (s.cpu().numpy() == s_ref).all() and (c.cpu().numpy() == c_ref).all(), name
