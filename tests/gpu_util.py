"""Shared helpers of the GPU parity tests: build the same synthetic layer for
the CUDA path (encoded by libmoe's encoder on the device) and for the oracle
(encoded by the oracle's own encoder from the same fp32 tensors, copied to
the host), and compare outputs with the tolerances of the parity contract."""
import numpy as np
import torch

import oracle
import synth
import moe_expert_layer_top16_gb300 as moe
from moe_expert_layer_top16_gb300.weights import encode_layer

DEV = torch.device("cuda:0")

# Output tolerance (fp32 y): max |err| <= 2e-2 * rms(y_ref) and
# sum|err| / sum|y_ref| <= 2e-3.
Y_MAX_REL_RMS = 2e-2
Y_REL_L1 = 2e-3


def fetch_device(wl, device=DEV):
    def fetch(name, i):
        if name == "bias":
            return synth.router_bias(wl, device=device)
        return synth.weight(wl, name, i, device=device)
    return fetch


def gpu_plan(wl, max_tokens=None):
    W = encode_layer(wl, fetch_device(wl), DEV)
    plan = moe.Plan(wl, W, max_tokens=max_tokens)
    return plan, W


def oracle_weights(wl, experts=None):
    """Oracle-encoded weights drawn from the same device tensors."""
    def fetch(name, i):
        if name == "bias":
            b = synth.router_bias(wl, device="cpu")
            return None if b is None else b.numpy()
        return synth.weight(wl, name, i, device=DEV).cpu().numpy()
    return oracle.encode_layer(wl, fetch, experts=experts)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def y_errors(y, y_ref):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    err = np.abs(y - y_ref)
    rms = np.sqrt(np.mean(y_ref ** 2))
    return err.max() / rms, err.sum() / np.abs(y_ref).sum()


def assert_y_close(y, y_ref, what="", out_bf16=False):
    """The output tolerance (stated for fp32).  A bf16 output carries one more
    rounding, to nearest bf16 (at most 2^-9 of the value): it is compared
    with the fp32 bound plus that rounding, element by element."""
    if not out_bf16:
        mx, l1 = y_errors(y, y_ref)
        assert mx <= Y_MAX_REL_RMS and l1 <= Y_REL_L1, f"{what}: max|err|/rms={mx:.3e} relL1={l1:.3e}"
        return mx, l1
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    err = np.abs(y - y_ref)
    rms = np.sqrt(np.mean(y_ref ** 2))
    rnd = np.ldexp(np.abs(y), -9)                     # half an ulp of bf16 at the output's value
    mx = float(np.max((err - rnd) / rms))
    l1 = float(np.maximum(err - rnd, 0.0).sum() / np.abs(y_ref).sum())
    assert mx <= Y_MAX_REL_RMS and l1 <= Y_REL_L1, f"{what}: max(|err|-rnd)/rms={mx:.3e} relL1={l1:.3e}"
    return mx, l1


def code_step_diff(a, b):
    """|difference| in E4M3 magnitude-code steps, for codes of equal sign
    (sign flips count as a large difference unless both are zeros)."""
    a = np.asarray(a, np.int32)
    b = np.asarray(b, np.int32)
    sa, sb = a >> 7, b >> 7
    ma, mb = a & 0x7F, b & 0x7F
    d = np.abs(ma - mb)
    flip = (sa != sb) & ~((ma == 0) & (mb == 0))
    d[flip] = ma[flip] + mb[flip]
    return d


def assert_codes_close(q, q_ref, s, s_ref, what="", min_equal=0.999):
    """Intermediate MXFP8 codes from fp32 inputs that differ at the rounding
    level: values equal in >= min_equal of elements, all within one code step
    (a scale change by one power of two shifts codes by 8 steps: compare the
    decoded values instead when scales differ)."""
    vq = oracle.mxfp8_decode(np.asarray(q), np.asarray(s))
    vr = oracle.mxfp8_decode(np.asarray(q_ref), np.asarray(s_ref))
    eq = (vq == vr).mean()
    same_scale = np.repeat(np.asarray(s) == np.asarray(s_ref), 32, axis=-1)
    steps = code_step_diff(q, q_ref)
    bad = same_scale & (steps > 1)
    # where the block scale moved by one, the value may differ by one step of the coarser grid
    smax = np.repeat(np.maximum(np.asarray(s, np.int32), np.asarray(s_ref, np.int32)), 32, axis=-1)
    tol = 0.13 * np.abs(vr) + np.ldexp(1.0, smax - 127 - 8)     # a grid step, or two subnormal steps
    bad |= ~same_scale & (np.abs(vq - vr) > tol)
    assert eq >= min_equal and not bad.any(), f"{what}: equal={eq:.5f} bad={int(bad.sum())}"
    return eq


class OracleLayer:
    """Oracle-encoded weights of one workload; routed experts are encoded on
    demand (the oracle never needs all 896 for a sampled check)."""

    def __init__(self, wl):
        self.wl = wl
        self.enc = {}

        def fetch(name, i):
            return synth.weight(wl, name, i, device=DEV).cpu().numpy()

        self._fetch = fetch
        if getattr(wl, "precision", "mx") == "mixed":
            # bf16 projections and shared experts, rounded by the oracle's own conversion
            for name in ("p_down", "p_up"):
                self.enc[name + "_bf16"] = oracle.bf16_round(fetch(name, 0))
            if wl.n_shared > 0:
                for name in ("s_gate", "s_up", "s_down"):
                    self.enc[name + "_bf16"] = np.stack([oracle.bf16_round(fetch(name, s))
                                                         for s in range(wl.n_shared)])
        else:
            for name in ("p_down", "p_up"):
                self.enc[name] = oracle.mxfp4_encode(fetch(name, 0))
            for s in range(wl.n_shared):
                for name in ("s_gate", "s_up", "s_down"):
                    self.enc[(name, s)] = oracle.mxfp4_encode(fetch(name, s))
        self.enc["router"] = fetch("router", 0)
        b = synth.router_bias(wl, device="cpu")
        self.enc["bias"] = None if b is None else b.numpy()
        self._lw = None

    def ensure(self, experts):
        new = [int(e) for e in set(int(v) for v in np.ravel(experts)) if ("w_gate", int(e)) not in self.enc]
        for e in new:
            for name in ("w_gate", "w_up", "w_down"):
                self.enc[(name, e)] = oracle.mxfp4_encode(self._fetch(name, e))
        if new or self._lw is None:
            self._lw = oracle.LayerWeights(self.wl, self.enc)
        return self._lw

    def keys(self, logits):
        """Selection keys of the oracle (fp64) for logits [n][E]."""
        lg = np.asarray(logits, np.float64)
        if self.wl.score == "softmax":
            return lg
        b = 0.0 if self.enc["bias"] is None else self.enc["bias"].astype(np.float64)
        return 1.0 / (1.0 + np.exp(-lg)) + b


def certify_routing(ol, idx_gpu, idx_ref, logits_gpu, logits_ref):
    """Compare per-token selections.  Tokens whose lists differ are accepted
    only at a near-tie: every expert picked by one side and not the other (or
    placed in a different slot) has an oracle key within 2*delta + 1e-12 of
    the key it displaced, where delta = max |logit_gpu - logit_ref| over the
    experts the GPU selected -- logits it recomputed exactly in fp32, so delta
    measures only the fp32 rounding and the GPU's own latent z, never a
    tensor-core estimate.  Returns the list of accepted tokens; raises on any
    other difference."""
    accepted = []
    keys = ol.keys(logits_ref)
    for t in range(idx_gpu.shape[0]):
        a, b = list(idx_gpu[t]), list(idx_ref[t])
        if a == b:
            continue
        sel = np.asarray(a, np.int64)
        delta = float(np.max(np.abs(np.asarray(logits_gpu[t], np.float64)[sel] - np.asarray(logits_ref[t])[sel])))
        tol = 2 * delta + 1e-12
        for ga, rb in zip(a, b):
            if ga != rb:
                assert abs(keys[t, ga] - keys[t, rb]) <= tol, (
                    f"token {t}: gpu {a} vs oracle {b}, key gap {abs(keys[t, ga] - keys[t, rb]):.3e} > {tol:.3e}")
        accepted.append(t)
    return accepted


def tf32_rna(v):
    """fp32 -> nearest TF32 value (10 explicit mantissa bits, ties away from
    zero), as fp32: the rounding the layer applies to the tensor-core router's
    operands."""
    b = np.ascontiguousarray(v, np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x1000) & 0xFFFFE000).astype(np.uint32)
    return b.view(np.float32)


def tc_router_bound(z_rows, R):
    """The layer's proven error bound of its tensor-core router estimates
    (delta_te = |z_hi||R_lo_e| + (|z_lo| + g_tc (1 + 2^-11)|z_hi| + g_32 (|z_hi|
    + |z_lo|)) |R_e|, 2-norms, g_tc = (K + 8) 2^-22, g_32 = (K/32 + 8) 2^-24),
    evaluated in fp64 for the GPU's latent rows z_rows [n][K] and router R
    [E][K]: [n][E]."""
    K = R.shape[1]
    z = np.asarray(z_rows, np.float32)
    zh = tf32_rna(z).astype(np.float64)
    zl = z.astype(np.float64) - zh
    Rh = tf32_rna(R).astype(np.float64)
    Rl = np.asarray(R, np.float64) - Rh
    nzh, nzl = np.linalg.norm(zh, axis=1), np.linalg.norm(zl, axis=1)
    nR, nRl = np.linalg.norm(np.asarray(R, np.float64), axis=1), np.linalg.norm(Rl, axis=1)
    g_tc, g_32 = (K + 8) * 2.0 ** -22, (K // 32 + 8) * 2.0 ** -24
    B = nzl + g_tc * (1 + 2.0 ** -11) * nzh + g_32 * (nzh + nzl)
    return nzh[:, None] * nRl[None, :] + B[:, None] * nR[None, :]


def route_exact_on_exports(wl, ol, g):
    """Top-k on the logits the GPU exports, whole batch: the oracle's
    selection rule on those values must reproduce the GPU's selection, gates
    and dispatch exactly (the exports are exact for every candidate and
    provably below the k-th exact logit elsewhere)."""
    E, k = wl.n_experts, wl.top_k
    idx_ref, gates_ref = oracle.route(g["logits"], k, softmax=(wl.score == "softmax"), bias=ol.enc["bias"])
    assert np.array_equal(idx_ref, g["topk_idx"]), \
        f"{int((idx_ref != g['topk_idx']).any(axis=1).sum())} tokens differ on the exported logits"
    np.testing.assert_allclose(g["topk_w"], gates_ref, rtol=3e-6, atol=1e-7)
    counts, offsets, order = oracle.permute(g["topk_idx"], E)
    assert (g["counts"] == counts).all() and (g["offsets"] == offsets).all()
    assert (g["sorted_token"] == order // k).all()


def check_router_logits(wl, ol, T, g_logits, g_idx, z_gpu, z_ref):
    """Router logits of sampled tokens against fp64 dot products of the GPU's
    own router input z_gpu with R, each within a rounding bound of its path
    (2-norms): the SIMT router (batches of up to 128 tokens, fp32 chains of at
    most K + 8 roundings) and the exact recomputation of the selected experts
    (K/32 + 8) bound their error by gamma |z| |R_e|; every other logit above
    128 tokens is a tensor-core estimate, within the layer's proven bound.
    The selected logits also stay within |z_gpu - z_ref| |R_e| (plus the
    rounding bound) of the oracle's own logits.  Returns the largest error
    of any logit (estimates included)."""
    R = ol.enc["router"].astype(np.float64)
    K = R.shape[1]
    zg = np.asarray(z_gpu, np.float32).astype(np.float64)
    exact = zg @ R.T
    nR = np.linalg.norm(R, axis=1)
    nz = np.linalg.norm(zg, axis=1)
    sel = g_idx.astype(np.int64)
    err = np.abs(g_logits.astype(np.float64) - exact)
    gamma = ((K + 8) if T <= 128 else (K // 32 + 8)) * 2.0 ** -24
    rnd = 1.001 * gamma * nz[:, None] * nR[None, :]
    sel_err = np.take_along_axis(err, sel, 1)
    assert (sel_err <= np.take_along_axis(rnd, sel, 1)).all(), f"selected logits off by {sel_err.max():.3e}"
    if T > 128:
        bound = tc_router_bound(z_gpu, ol.enc["router"])
        assert (err <= bound).all(), f"estimate error {err.max():.3e} beyond the proven bound"
    else:
        assert (err <= rnd).all(), f"logits off by {err.max():.3e}"
    zr = np.asarray(z_ref, np.float32).astype(np.float64)
    ref = zr @ R.T
    dz = np.linalg.norm(zg - zr, axis=1)
    d_ref = np.abs(np.take_along_axis(g_logits.astype(np.float64), sel, 1) - np.take_along_axis(ref, sel, 1))
    lim = np.take_along_axis(rnd + dz[:, None] * nR[None, :] * 1.001, sel, 1) + 1e-12
    assert (d_ref <= lim).all(), f"selected logits {d_ref.max():.3e} from the oracle's"
    return float(err.max())


def run_sampled_parity(wl, plan, ol, T, sample, x=None):
    """One forward of T tokens; whole-batch exact checks (top-k on the GPU's
    logits, dispatch), then oracle parity on the sampled tokens.  Returns
    (accepted near-tie tokens, y errors, realised counts)."""
    if x is None:
        x = synth.hidden_states(wl, T, device=DEV)
    fields = ("xq", "xs", "z", "logits", "topk_idx", "topk_w", "counts", "offsets", "sorted_token")
    dbg = moe.debug_buffers(wl, T, DEV, fields)
    y = plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    g = {k: v.cpu().numpy() for k, v in dbg.items()}
    y = y.float().cpu().numpy()
    assert np.isfinite(y).all()
    route_exact_on_exports(wl, ol, g)
    accepted, errs, _ = sampled_y(wl, ol, T, x, g, y, sample)
    return accepted, errs, g["counts"]


def sampled_y(wl, ol, T, x, g, y, sample):
    """Sampled tokens against the oracle layer: x codes exact, router logits
    (check_router_logits), selections equal except at certified near-ties,
    y within the output tolerance with the GPU's selection forced."""
    sample = np.asarray(sorted(set(int(s) for s in sample if 0 <= s < T)))
    xb = bf16_bits(x[torch.as_tensor(sample, device=DEV)])
    r0 = oracle.moe_forward(wl, ol.ensure([]), xb, route_only=True, want=("idx", "logits", "xq", "xs", "z"))
    if getattr(wl, "precision", "mx") != "mixed":        # the mixed scheme reads x as it is
        assert (r0["xq"] == g["xq"][sample]).all() and (r0["xs"] == g["xs"][sample]).all()
    if wl.route == "latent":
        z_gpu, z_ref = g["z"][sample], r0["z"]
    else:
        z_gpu = z_ref = (xb.astype(np.uint32) << 16).view(np.float32)
    est_err = check_router_logits(wl, ol, T, g["logits"][sample], g["topk_idx"][sample], z_gpu, z_ref)
    accepted = certify_routing(ol, g["topk_idx"][sample], r0["idx"], g["logits"][sample], r0["logits"])
    print(f"{wl.name} T={T}: {len(sample)} sampled tokens, {len(accepted)} certified near-ties")
    lw = ol.ensure(np.concatenate([g["topk_idx"][sample].ravel(), r0["idx"].ravel()]))
    ref = oracle.moe_forward(wl, lw, xb, force_idx=g["topk_idx"][sample], want=("y",))
    errs = assert_y_close(y[sample], ref["y"], f"{wl.name} T={T}", out_bf16=getattr(wl, "out", "f32") == "bf16")
    return accepted, errs, est_err


def grouped_item_tokens(T, k, E):
    """Rows of the most loaded expert that the item parity compares at batch
    size T: about three times the mean tokens per expert, a multiple of 16
    between 16 and 240, at most T rounded up to 16.  The engine's work items
    hold no more (at most 224 tokens on CTA pairs, 240 unpaired), so the rows
    cover that expert's first work item whole."""
    per_expert = -(-T * k // E)
    return int(min(max(-(-3 * per_expert // 16) * 16, 16), 240, -(-T // 16) * 16))


def silu(g):
    return g / (1.0 + np.exp(-g))


def run_item_parity(wl, plan, ol, T, n_sample=256, x=None):
    """One forward of T tokens with the full exports, then:
      * the whole-batch exact checks (top-k on the exported logits, dispatch);
      * the grouped GEMMs element by element on the most loaded expert's first
        grouped_item_tokens rows (its first work item whole, and more where
        its items are smaller): the GPU's MXFP8 activation codes and scales (A7) against
        MXFP8(SiLU(g) u) of the oracle's exact block-scaled products on the
        GPU's own latent codes, and the GPU's expert outputs (A8) against the
        oracle's exact product of the GPU's activation codes, within the
        tensor core's accumulation bound;
      * y of at least n_sample tokens -- that item's tokens plus evenly spaced
        others -- against the oracle layer.
    Returns (accepted near-ties, y errors, counts, rows compared)."""
    if x is None:
        x = synth.hidden_states(wl, T, device=DEV)
    E, k, I, L = wl.n_experts, wl.top_k, wl.expert_inter, wl.d_latent
    fields = ("xq", "xs", "z", "zq", "zs", "logits", "topk_idx", "topk_w", "counts", "offsets", "sorted_token",
              "hq", "hqs", "o")
    dbg = moe.debug_buffers(wl, T, DEV, fields)
    y = plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    small = ("xq", "xs", "z", "logits", "topk_idx", "topk_w", "counts", "offsets", "sorted_token")
    g = {f: dbg[f].cpu().numpy() for f in small}
    y = y.float().cpu().numpy()
    assert np.isfinite(y).all()
    route_exact_on_exports(wl, ol, g)
    # the hottest expert's first work item
    e = int(np.argmax(g["counts"]))
    n_item = min(int(g["counts"][e]), grouped_item_tokens(T, k, E))
    p0 = int(g["offsets"][e])
    rows = torch.arange(p0, p0 + n_item, device=DEV)
    toks = g["sorted_token"][p0:p0 + n_item].astype(np.int64)
    tt = torch.as_tensor(toks, device=DEV)
    zq, zs = dbg["zq"][tt].cpu().numpy(), dbg["zs"][tt].cpu().numpy()
    hq, hqs, o = dbg["hq"][rows].cpu().numpy(), dbg["hqs"][rows].cpu().numpy(), dbg["o"][rows].cpu().numpy()
    del dbg
    ol.ensure([e])
    gate, up, down = ol.enc[("w_gate", e)], ol.enc[("w_up", e)], ol.enc[("w_down", e)]
    gv = oracle.mx_matmul(*gate, zq, zs).astype(np.float32).astype(np.float64)
    uv = oracle.mx_matmul(*up, zq, zs).astype(np.float32).astype(np.float64)
    h = (silu(gv) * uv).astype(np.float32)
    hq_ref, hqs_ref = oracle.mxfp8_quantize(h)
    assert_codes_close(hq, hq_ref, hqs, hqs_ref, f"A7 expert {e} rows 0..{n_item - 1}")
    o_ref = oracle.mx_matmul(*down, hq, hqs)
    mag = oracle.mx_matmul(down[0] & 0x77, down[1], hq & 0x7F, hqs)       # sum of |terms|
    o_err = np.abs(o.astype(np.float64) - o_ref)
    assert (o_err <= mag * ((I + 8) * 2.0 ** -22) + np.abs(o_ref) * 2.0 ** -24).all(), \
        f"A8 expert {e}: max err {o_err.max():.3e}"
    # y of the item's tokens and evenly spaced others
    extra = np.linspace(0, T - 1, num=max(0, n_sample - len(toks)) + 2).astype(np.int64)
    sample = np.unique(np.concatenate([toks, extra]))
    accepted, errs, _ = sampled_y(wl, ol, T, x, g, y, sample)
    assert len(sample) >= min(n_sample, T)
    return accepted, errs, g["counts"], n_item
