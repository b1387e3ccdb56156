"""Pins for the oracle's Quantile Balancing update ("Kimi K3 and the New
Open-Weights Moat", section "How the router picks 16 of 896", Fig. 2: each
expert's selection bias is updated from the distribution of its score
margins so that its routed token count approaches the target load).

The pages give no formula; the reading (moe_oracle.c) moves the midpoint of
an expert's target-th and (target+1)-th largest margins to zero.  Pinned
here by what that reading must achieve, checked by brute force: an expert
updated alone with a full step lands exactly on the target count; the update
does not depend on a constant added to every bias; repeated damped updates
of all experts at once drive a Zipf-skewed load toward the mean."""
import numpy as np

import oracle


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def counts_fp64(logits, bias, k):
    """Brute force: each token's k largest keys sigmoid(l) + b (fp64, lower id
    on ties), counted per expert."""
    keys = sigmoid(logits) + bias[None, :]
    T, E = keys.shape
    order = np.lexsort((np.tile(np.arange(E), (T, 1)), -keys), axis=1)[:, :k]
    return np.bincount(order.ravel(), minlength=E)


def test_full_step_puts_one_expert_exactly_on_target():
    rng = np.random.default_rng(11)
    T, E, k = 300, 64, 4
    logits = rng.normal(0, 2, size=(T, E))
    bias = (rng.normal(0, 0.05, size=E)).astype(np.float32)
    target = 19
    new = oracle.quantile_balance(logits, bias, k, target, 1.0)
    before = counts_fp64(logits, bias.astype(np.float64), k)
    moved = 0
    for e in range(E):
        b = bias.astype(np.float64)
        b[e] = new[e]
        assert counts_fp64(logits, b, k)[e] == target, e
        moved += before[e] != target
    assert moved > E // 2                     # the batch was not balanced to begin with


def test_update_ignores_a_common_shift_of_the_bias():
    rng = np.random.default_rng(12)
    logits = rng.normal(0, 2, size=(200, 32))
    bias = (rng.normal(0, 0.05, size=32)).astype(np.float32)
    a = oracle.quantile_balance(logits, bias, 2, 12, 0.7)
    b = oracle.quantile_balance(logits, bias + np.float32(0.25), 2, 12, 0.7)
    np.testing.assert_allclose(b - 0.25, a, rtol=0, atol=1e-6)   # 0.25 is exact in fp32


def test_damped_updates_balance_a_zipf_skewed_load():
    rng = np.random.default_rng(13)
    T, E, k = 4096, 128, 8
    logits = rng.normal(0, 1, size=(T, E))
    rank = rng.permutation(E) + 1
    bias = (-0.3 * np.log(rank)).astype(np.float32)
    target = T * k // E
    loads = []
    for it in range(30):
        c = counts_fp64(logits, bias.astype(np.float64), k)
        loads.append(c.max() / c.mean())
        bias = oracle.quantile_balance(logits, bias, k, target, 0.5).astype(np.float32)
    c = counts_fp64(logits, bias.astype(np.float64), k)
    loads.append(c.max() / c.mean())
    assert loads[0] > 3.0
    assert loads[-1] < 1.25, loads[-5:]
    assert loads[-1] < loads[0] / 2
