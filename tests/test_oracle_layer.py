"""Layer-level pins for the oracle on the small (Tiny) layer.

The oracle's per-token forward is checked against a dense recomputation that
evaluates every expert for every token and then masks by the selection,
assembled from the oracle's separately pinned primitives (block-scaled
product, MXFP8 quantiser, router).  Layer structure: "Kimi K3 and the New
Open-Weights Moat", sections "Sparse computation: latent experts and
routing" and "How the router picks 16 of 896" (Fig. 2); the dense loop over
tokens and their experts mirrors the reference check of the one-page data
path in "Kimi K3: 2.8 Trillion Parameters, Four Bits at a Time".
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def tiny_layer():
    wl = synth.workload("tiny")

    def fetch(name, i):
        if name == "bias":
            b = synth.router_bias(wl)
            return None if b is None else b.numpy()
        return synth.weight(wl, name, i).numpy()

    return wl, oracle.encode_layer(wl, fetch)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


ALL = ("y", "xq", "xs", "z", "zq", "zs", "hs", "hsq", "hss", "logits", "idx", "gates",
       "h", "hq", "hqs", "o", "c", "cq", "cs")


@pytest.fixture(scope="module")
def tiny():
    wl, W = tiny_layer()
    x = bf16_bits(synth.hidden_states(wl))
    out = oracle.moe_forward(wl, W, x, want=ALL)
    return wl, W, x, out


def silu(g):
    return g / (1.0 + np.exp(-g))


def test_dense_all_experts_masked_recomputation(tiny):
    wl, W, x, out = tiny
    enc = W.enc
    T, E, k, I, L = wl.tokens, wl.n_experts, wl.top_k, wl.expert_inter, wl.d_latent
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    xq, xs = oracle.mxfp8_quantize(xf)
    assert (xq == out["xq"]).all() and (xs == out["xs"]).all()
    z = oracle.mx_matmul(*enc["p_down"], xq, xs).astype(np.float32)
    np.testing.assert_array_equal(z, out["z"])
    zq, zs = oracle.mxfp8_quantize(z)
    assert (zq == out["zq"]).all() and (zs == out["zs"]).all()
    hs = []
    for s in range(wl.n_shared):
        g = oracle.mx_matmul(*enc[("s_gate", s)], xq, xs).astype(np.float32)
        u = oracle.mx_matmul(*enc[("s_up", s)], xq, xs).astype(np.float32)
        hs.append((silu(g.astype(np.float64)) * u).astype(np.float32))
    hs = np.concatenate(hs, axis=1)
    np.testing.assert_array_equal(hs, out["hs"])
    hsq, hss = oracle.mxfp8_quantize(hs)
    logits = z.astype(np.float64) @ enc["router"].astype(np.float64).T
    np.testing.assert_allclose(logits, out["logits"], rtol=0, atol=1e-12)
    idx, gates = oracle.route(out["logits"], k, softmax=(wl.score == "softmax"))
    assert (idx == out["idx"]).all()
    np.testing.assert_array_equal(gates, out["gates"])
    # every expert for every token
    o_all = np.zeros((E, T, L), np.float32)
    for e in range(E):
        g = oracle.mx_matmul(*enc[("w_gate", e)], zq, zs).astype(np.float32)
        u = oracle.mx_matmul(*enc[("w_up", e)], zq, zs).astype(np.float32)
        h = (silu(g.astype(np.float64)) * u).astype(np.float32)
        hq, hqs = oracle.mxfp8_quantize(h)
        o_all[e] = oracle.mx_matmul(*enc[("w_down", e)], hq, hqs).astype(np.float32)
    sel = np.zeros((T, E), bool)
    sel[np.arange(T)[:, None], idx] = True
    assert sel.sum() == T * k
    c = np.zeros((T, L))
    for t in range(T):
        for j in range(k):            # slot order
            c[t] += gates[t, j] * o_all[idx[t, j], t].astype(np.float64)
        # masked experts contribute nothing
        assert np.count_nonzero(sel[t]) == k
    c = c.astype(np.float32)
    np.testing.assert_array_equal(c, out["c"])
    cq, cs = oracle.mxfp8_quantize(c)
    y = (oracle.mx_matmul(*enc["p_up"], cq, cs)
         + sum(oracle.mx_matmul(*enc[("s_down", s)],
                                np.ascontiguousarray(hsq[:, s * wl.shared_inter:(s + 1) * wl.shared_inter]),
                                np.ascontiguousarray(hss[:, s * wl.shared_inter // 32:(s + 1) * wl.shared_inter // 32]))
               for s in range(wl.n_shared)))
    np.testing.assert_allclose(y.astype(np.float32), out["y"], rtol=1e-6, atol=1e-7)


def test_forced_routing(tiny):
    wl, W, x, out = tiny
    same = oracle.moe_forward(wl, W, x, force_idx=out["idx"], want=("y", "gates"))
    np.testing.assert_array_equal(same["y"], out["y"])
    np.testing.assert_array_equal(same["gates"], out["gates"])
    # a different selection: gates are the softmax of the forced winners
    forced = np.roll(out["idx"], 1, axis=0)
    res = oracle.moe_forward(wl, W, x, force_idx=forced, want=("y", "gates", "idx"))
    assert (res["idx"] == forced).all()
    lg = np.take_along_axis(out["logits"], forced.astype(np.int64), 1)
    ex = np.exp(lg - lg.max(1, keepdims=True))
    np.testing.assert_allclose(res["gates"], ex / ex.sum(1, keepdims=True), rtol=1e-13)
    assert not np.array_equal(res["y"], out["y"])


def test_rows_are_independent(tiny):
    wl, W, x, out = tiny
    part = oracle.moe_forward(wl, W, x[17:23], want=("y",))
    np.testing.assert_array_equal(part["y"], out["y"][17:23])


def test_output_scale(tiny):
    wl, W, x, out = tiny
    y = out["y"]
    assert np.isfinite(y).all() and y.std() > 0


def test_forced_routing_sigmoid_gates_on_negated_router_rows():
    """Forced selection in sigmoid mode ("How the router picks 16 of 896",
    Fig. 2: the winners' raw sigmoid scores over their sum, the bias left
    out).  The router's rows come in negated pairs, R[2i+1] = -R[2i], so the
    logits of a pair are exactly l and -l, and sigmoid(l) + sigmoid(-l) = 1.
    Forcing two whole pairs makes the normaliser exactly 2: every gate is
    sigmoid(l_j) / 2 and each pair's gates add to 1/2 -- values a softmax
    over the winners, a missing normalisation or a bias inside the gates
    would all miss."""
    from dataclasses import replace
    wl = replace(synth.workload("tiny"), score="sigmoid")
    base = synth.weight(wl, "router", 0).numpy()
    router = base.copy()
    router[1::2] = -base[0::2]
    rng = np.random.default_rng(5)
    bias = rng.normal(0, 0.5, size=wl.n_experts).astype(np.float32)
    x = bf16_bits(synth.hidden_states(wl))
    T = x.shape[0]
    forced = np.tile(np.array([4, 5, 10, 11], np.int32), (T, 1))
    outs = []
    for b in (None, bias):
        def fetch(name, i, b=b):
            if name == "router":
                return router
            if name == "bias":
                return b
            return synth.weight(wl, name, i).numpy()
        lw = oracle.encode_layer(wl, fetch)
        outs.append(oracle.moe_forward(wl, lw, x, force_idx=forced, want=("gates", "logits", "idx")))
    for r in outs:
        lg = r["logits"]
        assert np.array_equal(lg[:, 1::2], -lg[:, 0::2])
        assert (r["idx"] == forced).all()
        g = r["gates"]
        np.testing.assert_allclose(g[:, 0] + g[:, 1], 0.5, rtol=0, atol=1e-15)
        np.testing.assert_allclose(g[:, 2] + g[:, 3], 0.5, rtol=0, atol=1e-15)
        sel = np.take_along_axis(lg, forced.astype(np.int64), 1)
        np.testing.assert_allclose(g, 0.5 / (1.0 + np.exp(-sel)), rtol=1e-14, atol=0)
    # the selection bias changes nothing in the forced gates
    np.testing.assert_array_equal(outs[0]["gates"], outs[1]["gates"])
