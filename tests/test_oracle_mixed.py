"""Pins for the oracle's mixed-precision scheme ("Kimi K3 and the New
Open-Weights Moat", section "Precision and deployment", Fig. 6: only the
routed experts' weights are MXFP4 and their inputs MXFP8; the latent-MoE
projections, the shared experts and the router stay at higher precision,
read here as BF16 weights and BF16 inputs, fp32 router).

Pinned against: round-to-nearest-even on the bf16 grid (hand cases, and the
conversion of a library, torch, on random fp32 values); a dense
recomputation of the small layer from numpy matmuls of the decoded bf16
weights; and one-hot projection rows, which make the latent an exact copy of
components of x and the output an exact copy of components of bf16(c).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import synth


def test_bf16_round_hand_cases():
    def r(v):
        return int(oracle.bf16_round(np.array([v], np.float32))[0])
    assert r(1.0) == 0x3F80
    assert r(-2.0) == 0xC000
    assert r(-0.0) == 0x8000
    assert r(1.0 + 2.0 ** -8) == 0x3F80             # halfway to 0x3F81: ties to the even 0x3F80
    assert r(1.0 + 3 * 2.0 ** -8) == 0x3F82         # halfway between 0x3F81 and 0x3F82: to 0x3F82
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -20) == 0x3F81    # just above halfway: up
    assert r(np.float32(3.4028235e38)) == 0x7F80    # rounds past the largest bf16: infinity
    assert r(np.inf) == 0x7F80 and r(-np.inf) == 0xFF80
    n = r(np.nan)
    assert (n & 0x7F80) == 0x7F80 and (n & 0x7F) != 0
    assert r(2.0 ** -133) == 0x0001                 # smallest bf16 subnormal is exact
    assert r(1.5 * 2.0 ** -133) == 0x0002           # halfway between 1 and 2 units: to even 2


def test_bf16_round_matches_the_library_conversion():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(0, 1, 100000), rng.normal(0, 0.02, 100000),
                        np.ldexp(rng.uniform(1, 2, 100000), rng.integers(-140, 120, 100000))]).astype(np.float32)
    ours = oracle.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    np.testing.assert_array_equal(oracle.bf16_decode(ours), torch.from_numpy(v).to(torch.bfloat16).double().numpy())


def mixed_tiny(fetch_override=None):
    wl = synth.workload("tiny+mixed")

    def fetch(name, i):
        if fetch_override is not None:
            w = fetch_override(name, i)
            if w is not None:
                return w
        if name == "bias":
            return None
        return synth.weight(wl, name, i).numpy()

    return wl, oracle.encode_layer(wl, fetch)


def bits(x):
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def silu(g):
    return g / (1.0 + np.exp(-g))


def test_mixed_layer_dense_recomputation():
    wl, W = mixed_tiny()
    enc = W.enc
    x = bits(synth.hidden_states(wl))
    out = oracle.moe_forward(wl, W, x, want=("y", "z", "zq", "zs", "hs", "logits", "idx", "gates", "o", "c"))
    T, L, E, k = wl.tokens, wl.d_latent, wl.n_experts, wl.top_k
    xf = oracle.bf16_decode(x)                       # x enters the projections as it is (bf16)
    z = (xf @ oracle.bf16_decode(enc["p_down_bf16"]).T).astype(np.float32)
    np.testing.assert_array_max_ulp(z, out["z"], maxulp=1)
    zq, zs = oracle.mxfp8_quantize(out["z"])
    assert (zq == out["zq"]).all() and (zs == out["zs"]).all()
    g = (xf @ oracle.bf16_decode(enc["s_gate_bf16"][0]).T).astype(np.float32)
    u = (xf @ oracle.bf16_decode(enc["s_up_bf16"][0]).T).astype(np.float32)
    hs = (silu(g.astype(np.float64)) * u).astype(np.float32)
    np.testing.assert_allclose(hs, out["hs"], rtol=1e-6, atol=1e-12)
    # routing on the fp32 latent, as in the all-MX layer
    logits = out["z"].astype(np.float64) @ enc["router"].astype(np.float64).T
    np.testing.assert_allclose(logits, out["logits"], rtol=0, atol=1e-12)
    idx, gates = oracle.route(out["logits"], k, softmax=(wl.score == "softmax"))
    assert (idx == out["idx"]).all()
    # routed experts: MXFP4 x MXFP8, as in the all-MX layer
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            gt = oracle.mx_matmul(*enc[("w_gate", e)], zq[t:t + 1], zs[t:t + 1]).astype(np.float32)
            ut = oracle.mx_matmul(*enc[("w_up", e)], zq[t:t + 1], zs[t:t + 1]).astype(np.float32)
            h = (silu(gt.astype(np.float64)) * ut).astype(np.float32)
            hq, hqs = oracle.mxfp8_quantize(h)
            o = oracle.mx_matmul(*enc[("w_down", e)], hq, hqs).astype(np.float32)
            np.testing.assert_array_equal(o[0], out["o"][t, j])
    c = np.einsum("tj,tjl->tl", gates, out["o"].astype(np.float64)).astype(np.float32)
    np.testing.assert_allclose(c, out["c"], rtol=1e-6, atol=1e-12)
    # the up-projection reads bf16(c) and bf16(h_s)
    cb = oracle.bf16_decode(oracle.bf16_round(out["c"]))
    hb = oracle.bf16_decode(oracle.bf16_round(out["hs"]))
    y = cb @ oracle.bf16_decode(enc["p_up_bf16"]).T + hb @ oracle.bf16_decode(enc["s_down_bf16"][0]).T
    np.testing.assert_allclose(y.astype(np.float32), out["y"], rtol=1e-6, atol=1e-7)


def test_mixed_layer_one_hot_projections_copy_exactly():
    """P_down rows one-hot at columns dz, P_up rows one-hot at columns dy and
    a zero shared gate: z is exactly x[:, dz] (a bf16 value times 1), the
    shared activation SiLU(0) * u is exactly 0, and y is exactly
    bf16(c)[:, dy]."""
    wl0 = synth.workload("tiny+mixed")
    D, L = wl0.d_model, wl0.d_latent
    dz = (5 * np.arange(L) + 3) % D
    dy = (7 * np.arange(D) + 1) % L
    p_down = np.zeros((L, D), np.float32)
    p_down[np.arange(L), dz] = 1.0
    p_up = np.zeros((D, L), np.float32)
    p_up[np.arange(D), dy] = 1.0

    def override(name, i):
        if name == "p_down":
            return p_down
        if name == "p_up":
            return p_up
        if name == "s_gate":
            return np.zeros(synth.weight_shape(wl0, "s_gate"), np.float32)
        return None

    wl, W = mixed_tiny(override)
    x = bits(synth.hidden_states(wl))
    out = oracle.moe_forward(wl, W, x, want=("y", "z", "hs", "c"))
    xf = oracle.bf16_decode(x)
    assert np.array_equal(out["z"].astype(np.float64), xf[:, dz])
    assert not out["hs"].any()
    cb = oracle.bf16_decode(oracle.bf16_round(out["c"]))
    assert np.array_equal(out["y"].astype(np.float64), cb[:, dy])
    assert np.abs(out["y"]).sum() > 0
