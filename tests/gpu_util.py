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
    the key it displaced, delta = max |logit_gpu - logit_ref| of that token.
    Returns the list of accepted tokens; raises on any other difference."""
    accepted = []
    keys = ol.keys(logits_ref)
    for t in range(idx_gpu.shape[0]):
        a, b = list(idx_gpu[t]), list(idx_ref[t])
        if a == b:
            continue
        delta = float(np.max(np.abs(np.asarray(logits_gpu[t], np.float64) - logits_ref[t])))
        tol = 2 * delta + 1e-12
        for ga, rb in zip(a, b):
            if ga != rb:
                assert abs(keys[t, ga] - keys[t, rb]) <= tol, (
                    f"token {t}: gpu {a} vs oracle {b}, key gap {abs(keys[t, ga] - keys[t, rb]):.3e} > {tol:.3e}")
        accepted.append(t)
    return accepted


def run_sampled_parity(wl, plan, ol, T, sample, x=None):
    """One forward of T tokens; whole-batch exact checks (top-k on the GPU's
    logits, dispatch), then oracle parity on the sampled tokens.  Returns
    (accepted near-tie tokens, y errors, realised counts)."""
    if x is None:
        x = synth.hidden_states(wl, T, device=DEV)
    fields = ("xq", "xs", "logits", "topk_idx", "topk_w", "counts", "offsets", "sorted_token")
    dbg = moe.debug_buffers(wl, T, DEV, fields)
    y = plan.forward(x, debug=dbg)
    torch.cuda.synchronize()
    assert plan.device_status() == moe.MOE_OK
    g = {k: v.cpu().numpy() for k, v in dbg.items()}
    y = y.float().cpu().numpy()
    assert np.isfinite(y).all()
    E, k = wl.n_experts, wl.top_k
    # exact on identical logits: selection, gates, dispatch
    idx_ref, gates_ref = oracle.route(g["logits"], k, softmax=(wl.score == "softmax"), bias=ol.enc["bias"])
    same = (idx_ref == g["topk_idx"]).all(axis=1)
    if not same.all():
        certify_routing(ol, g["topk_idx"], idx_ref, g["logits"], g["logits"].astype(np.float64))
    np.testing.assert_allclose(g["topk_w"][same], gates_ref[same], rtol=3e-6, atol=1e-7)
    counts, offsets, order = oracle.permute(g["topk_idx"], E)
    assert (g["counts"] == counts).all() and (g["offsets"] == offsets).all()
    assert (g["sorted_token"] == order // k).all()
    # sampled tokens against the oracle layer
    sample = np.asarray(sorted(set(int(s) for s in sample if 0 <= s < T)))
    xb = bf16_bits(x[torch.as_tensor(sample, device=DEV)])
    r0 = oracle.moe_forward(wl, ol.ensure([]), xb, route_only=True, want=("idx", "logits", "xq", "xs"))
    assert (r0["xq"] == g["xq"][sample]).all() and (r0["xs"] == g["xs"][sample]).all()
    # the selected experts' logits are fp32-accurate; above 128 tokens the
    # others are tensor-core estimates (one TF32 product), within the bound
    # the top-k refinement assumes (2e-2)
    sel = g["topk_idx"][sample].astype(np.int64)
    assert np.max(np.abs(np.take_along_axis(g["logits"][sample], sel, 1)
                         - np.take_along_axis(r0["logits"], sel, 1))) <= 1e-4
    assert np.max(np.abs(g["logits"][sample] - r0["logits"])) <= (2e-2 if T > 128 else 1e-4)
    accepted = certify_routing(ol, g["topk_idx"][sample], r0["idx"], g["logits"][sample], r0["logits"])
    lw = ol.ensure(np.concatenate([g["topk_idx"][sample].ravel(), r0["idx"].ravel()]))
    ref = oracle.moe_forward(wl, lw, xb, force_idx=g["topk_idx"][sample], want=("y",))
    errs = assert_y_close(y[sample], ref["y"], f"{wl.name} T={T}", out_bf16=getattr(wl, "out", "f32") == "bf16")
    return accepted, errs, g["counts"]
