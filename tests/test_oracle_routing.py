"""Pins for the oracle's routing, dispatch and combine.

Sources: "Kimi K3: 2.8 Trillion Parameters, Four Bits at a Time", section
"What it takes to serve it" (the one-page MoE data path and its printed
output), and "Kimi K3 and the New Open-Weights Moat", section "How the
router picks 16 of 896" / Fig. 2 (sigmoid score, selection-only bias,
winners' scores normalised by their sum).
"""
import numpy as np

import oracle
from conftest import read_golden


def _toy_inputs():
    rng = np.random.default_rng(0)
    T, D, E, K = 8, 16, 32, 4
    x = rng.normal(size=(T, D)).astype(np.float32)
    W = rng.normal(size=(E, D, D)).astype(np.float32) * 0.1
    router = rng.normal(size=(D, E)).astype(np.float32)
    return T, D, E, K, x, W, router


def test_toy_data_path_reproduces_printed_output():
    g = {r[0]: r[1:] for r in read_golden("toy_moe_data_path.txt")}
    T, D, E, K, x, W, router = _toy_inputs()
    logits = x @ router
    idx, gates = oracle.route(logits, K, softmax=True)
    # the page's selection, argsort(-logits)[:, :K], on the same logits
    assert (idx == np.argsort(-logits, axis=1)[:, :K]).all()
    counts, offsets, order = oracle.permute(idx, E)
    assert counts.tolist() == [int(v) for v in g["tokens_per_expert"]]
    assert order.size == int(g["permuted_buffer_rows"][0])
    assert 2 * K * D * x.itemsize == int(g["wire_bytes_per_token"][0])
    xp = x[order // K]
    yp = np.empty_like(xp, dtype=np.float64)
    for e in range(E):                   # one matrix per expert segment
        s, t = offsets[e], offsets[e + 1]
        if t > s:
            yp[s:t] = xp[s:t].astype(np.float64) @ W[e].astype(np.float64)
    y = oracle.combine(yp, order, gates, T, K)
    y_ref = np.zeros((T, D))
    for t in range(T):
        for j in range(K):
            y_ref[t] += gates[t, j] * (x[t].astype(np.float64) @ W[idx[t, j]].astype(np.float64))
    assert np.allclose(y, y_ref, atol=1e-5) == (g["matches_dense_loop"][0] == "True")


def _brute_topk(key, k):
    E = key.shape[0]
    order = sorted(range(E), key=lambda e: (-key[e], e))
    return order[:k]


def test_sigmoid_route_brute_force_and_invariants():
    rng = np.random.default_rng(4)
    T, E, k = 48, 896, 16
    logits = rng.normal(0, 2.0, size=(T, E))
    bias = (rng.normal(size=E) * 0.01).astype(np.float32)
    # plant exact ties in the key to exercise the lower-id rule
    logits[0, 10] = logits[0, 20] = 9.0
    logits[1, 5] = logits[1, 700] = logits[1, 3] = 8.0
    bias[[3, 5, 10, 20, 700]] = 0.2    # dominate the random biases
    idx, gates = oracle.route(logits, k, softmax=False, bias=bias)
    for t in range(T):
        key = 1.0 / (1.0 + np.exp(-logits[t])) + bias.astype(np.float64)
        assert idx[t].tolist() == _brute_topk(key, k)
    assert idx[0, 0] == 10 and idx[0, 1] == 20
    assert idx[1, :3].tolist() == [3, 5, 700]
    assert (gates >= 0).all()
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=0, atol=1e-12)
    assert all(len(set(r)) == k for r in idx.tolist())
    assert ((idx >= 0) & (idx < E)).all()
    # gates are the winners' sigmoid scores over their sum -- no bias in them
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx.astype(np.int64), 1)))
    np.testing.assert_allclose(gates, s / s.sum(1, keepdims=True), rtol=1e-14)


def test_bias_moves_selection_not_weights():
    rng = np.random.default_rng(8)
    T, E, k = 16, 64, 4
    logits = rng.normal(size=(T, E))
    bias = np.zeros(E, np.float32)
    bias[7] = 5.0                      # a bias this large always selects expert 7
    idx_b, g_b = oracle.route(logits, k, softmax=False, bias=bias)
    assert (idx_b[:, 0] == 7).all()
    # the gate of expert 7 is its raw score share, independent of the bias
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx_b.astype(np.int64), 1)))
    np.testing.assert_allclose(g_b, s / s.sum(1, keepdims=True), rtol=1e-14)
    idx_0, _ = oracle.route(logits, k, softmax=False)
    assert not (idx_0 == idx_b).all()


def test_softmax_route_gates():
    rng = np.random.default_rng(9)
    logits = rng.normal(size=(10, 32)).astype(np.float32)
    idx, gates = oracle.route(logits, 4, softmax=True)
    sel = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), 1)
    np.testing.assert_allclose(gates, np.exp(sel) / np.exp(sel).sum(1, keepdims=True), rtol=1e-13)
    assert (np.diff(sel, axis=1) <= 0).all()          # slot order = descending logit


def test_permute_invariants():
    rng = np.random.default_rng(12)
    T, E, k = 300, 96, 8
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, order = oracle.permute(idx, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[-1] == T * k and (np.diff(offsets) == counts).all()
    assert sorted(order.tolist()) == list(range(T * k))
    flat_e = idx.ravel()
    assert (order == np.argsort(flat_e, kind="stable")).all()
    for e in range(E):
        toks = order[offsets[e]:offsets[e + 1]] // k
        assert (np.diff(toks) > 0).all()
        assert (flat_e[order[offsets[e]:offsets[e + 1]]] == e).all()


def test_permute_degenerate_all_to_one_expert():
    T, E, k = 40, 16, 1
    idx = np.full((T, k), 5, np.int32)
    counts, offsets, order = oracle.permute(idx, E)
    assert counts[5] == T and counts.sum() == T
    assert order.tolist() == list(range(T))


def test_touched_expert_closed_form_matches_printed_simulation():
    # Expected distinct experts under uniform routing: E (1 - (1 - k/E)^B).
    # The page's GB/token column is touched * 1.5 GB / B.
    E, k = 896, 16
    rows = {int(r[0]): float(r[1]) for r in read_golden("expert_amortisation.txt")}
    for B, gb in rows.items():
        touched = E * (1 - (1 - k / E) ** B)
        assert abs(touched * 1.5 / B - gb) <= 0.02 * gb + 0.01
    # and the oracle's router on iid logits gives the same expectation
    rng = np.random.default_rng(21)
    for B in (8, 64):
        t = []
        for _ in range(16):
            idx, _ = oracle.route(rng.normal(size=(B, E)), k, softmax=False)
            counts, _, _ = oracle.permute(idx, E)
            t.append((counts > 0).sum())
        assert abs(np.mean(t) * 1.5 / B - rows[B]) <= 0.03 * rows[B]


def _one_hot_router(E, K, stride=7, offset=3):
    """Router rows that pick one input dimension each: row e = unit vector at
    (stride * e + offset) % K."""
    r = np.zeros((E, K), np.float32)
    dims = (stride * np.arange(E) + offset) % K
    r[np.arange(E), dims] = 1.0
    return r, dims


def _layer_with_router(wl, router):
    import synth

    def fetch(name, i):
        if name == "router":
            return router
        if name == "bias":
            return None
        return synth.weight(wl, name, i).numpy()
    return oracle.encode_layer(wl, fetch)


def test_router_input_hidden_reads_x_and_latent_reads_z():
    """With one-hot router rows each logit is one component of the router's
    input: of x itself (its exact bf16 value) when routing on the hidden
    state, of the oracle's own latent z otherwise."""
    import synth
    import torch
    for route in ("hidden", "latent"):
        wl = synth.workload("tiny" + ("+hidden" if route == "hidden" else "")).with_tokens(6)
        K = wl.d_model if route == "hidden" else wl.d_latent
        router, dims = _one_hot_router(wl.n_experts, K)
        lw = _layer_with_router(wl, router)
        x = synth.hidden_states(wl, 6)
        xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
        r = oracle.moe_forward(wl, lw, xb, route_only=True, want=("logits", "z"))
        src = x.float().numpy() if route == "hidden" else r["z"]
        assert np.array_equal(r["logits"], src[:, dims].astype(np.float64))


def test_sigmoid_keys_without_bias_keep_their_order_past_saturation():
    """sigmoid is strictly increasing, so without a bias the selection key
    sigmoid(l) orders the experts exactly as their logits do -- also where
    sigmoid(l) rounds to 1.0 in fp64 (l above about 37), where a comparison
    of the rounded keys would see ties and fall back to the expert id."""
    E, k = 12, 4
    logits = np.zeros((1, E))
    logits[0, [2, 5, 7, 9, 11]] = [39.0, 41.0, 40.0, 38.5, 45.0]
    assert 1.0 / (1.0 + np.exp(-39.0)) == 1.0 / (1.0 + np.exp(-41.0)) == 1.0   # the rounded keys tie
    idx, gates = oracle.route(logits, k, softmax=False)
    assert idx[0].tolist() == [11, 5, 7, 2]
    np.testing.assert_allclose(gates, 0.25, rtol=0, atol=1e-15)
    # with a bias the key is sigmoid(l) + b as written, evaluated in fp64
    bias = np.zeros(E, np.float32)
    bias[3] = 2.0
    idx_b, _ = oracle.route(logits, k, softmax=False, bias=bias)
    assert idx_b[0, 0] == 3
