"""Python binding of libmoe: the K3-style sparse MoE layer on one GB300.

Argument marshalling only: every step of the layer runs in the CUDA kernels
of libmoe (``csrc/``), reached through the C ABI declared in
``include/moe.h``.  PyTorch supplies device memory and the current stream.
There is no CPU fallback: if the library is missing or no sm_103a device is
present, the calls raise.

    from moe_expert_layer_top16_gb300 import Plan, mxfp4_encode
    plan = Plan(cfg, weights)            # weights: dict of CUDA tensors (see Plan)
    y = plan.forward(x)                  # x: bf16 [T][D] CUDA tensor -> y fp32 [T][D]
"""
from __future__ import annotations

import ctypes as C
import os
import threading
from typing import Optional

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_OOM, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = range(7)
SCORE_SIGMOID_BIAS, SCORE_SOFTMAX = 0, 1
ROUTE_ON_LATENT, ROUTE_ON_HIDDEN = 0, 1
OUT_F32, OUT_BF16 = 0, 1
PRECISION_MX, PRECISION_MIXED = 0, 1

# Entry points declared in include/moe.h.
ENTRY_POINTS = ("moe_plan", "moe_forward", "moe_forward_host", "moe_get_device_status", "moe_workspace_bytes",
                "moe_free", "moe_status_str", "moe_mxfp4_encode", "moe_mx_gemm", "moe_mma_probe",
                "moe_ep_row_bytes", "moe_ep_dispatch", "moe_ep_combine", "moe_quantile_balance", "moe_set_bias",
                "moe_mx_gemm_noalloc")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_str(code)} ({code})")
        self.code = code


class _Config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("d_model", "d_latent", "n_experts", "top_k", "expert_inter",
                                          "n_shared", "shared_inter", "max_tokens", "score_fn", "route_input",
                                          "out_dtype", "precision")]


class _MX4(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p)]


class _Weights(C.Structure):
    _fields_ = [(n, _MX4) for n in ("p_down", "p_up", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")] + \
               [("router_w", C.c_void_p), ("router_bias", C.c_void_p)] + \
               [(n + "_bf16", C.c_void_p) for n in ("p_down", "p_up", "s_gate", "s_up", "s_down")]


DEBUG_FIELDS = ("xq", "xs", "z", "zq", "zs", "hsq", "hss", "logits", "topk_idx", "topk_w", "counts", "offsets",
                "sorted_token", "hq", "hqs", "o", "cq", "cs")


NUM_STAGES = 11
STAGE_NAMES = ("quant_x", "gemm_down_shared", "router", "topk", "expert_counts", "worklists", "dispatch",
               "gemm_gate_up", "gemm_down", "combine", "gemm_up_shared")


class _Debug(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in DEBUG_FIELDS] + [("stage_events", C.c_void_p)]


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = False):
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"libmoe is not built ({path}); run moe_expert_layer_top16_gb300.build.build()")
                _build.build()
            L = C.CDLL(path)
            P, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
            L.moe_plan.restype = C.c_int
            L.moe_plan.argtypes = [C.POINTER(_Config), C.POINTER(_Weights), C.c_int, C.POINTER(C.c_void_p)]
            L.moe_forward.restype = C.c_int
            L.moe_forward.argtypes = [P, P, i32, P, P, C.POINTER(_Debug)]
            L.moe_forward_host.restype = C.c_int
            L.moe_forward_host.argtypes = [P, P, i32, P, P]
            L.moe_get_device_status.restype = C.c_int
            L.moe_get_device_status.argtypes = [P]
            L.moe_workspace_bytes.restype = C.c_size_t
            L.moe_workspace_bytes.argtypes = [P]
            L.moe_free.restype = None
            L.moe_free.argtypes = [P]
            L.moe_status_str.restype = C.c_char_p
            L.moe_status_str.argtypes = [C.c_int]
            L.moe_mxfp4_encode.restype = C.c_int
            L.moe_mxfp4_encode.argtypes = [P, i64, i64, P, P, P]
            L.moe_mx_gemm.restype = C.c_int
            L.moe_mx_gemm.argtypes = [P, P, i32, P, P, i32, i32, P, P, P]
            L.moe_ep_row_bytes.restype = C.c_int64
            L.moe_ep_row_bytes.argtypes = [P]
            L.moe_ep_dispatch.restype = C.c_int
            L.moe_ep_dispatch.argtypes = [P, i32, i32, P, P, P]
            L.moe_ep_combine.restype = C.c_int
            L.moe_ep_combine.argtypes = [P, i32, P, P, P, P]
            L.moe_quantile_balance.restype = C.c_int
            L.moe_quantile_balance.argtypes = [P, i32, i32, C.c_double, P, P]
            L.moe_set_bias.restype = C.c_int
            L.moe_set_bias.argtypes = [P, P]
            L.moe_mma_probe.restype = C.c_int
            L.moe_mma_probe.argtypes = [i32, i32, i32, P, C.POINTER(C.c_double), P]
            L.moe_mx_gemm_noalloc.restype = C.c_int
            L.moe_mx_gemm_noalloc.argtypes = [P, P, i32, P, P, i32, i32, P, P, P]
            _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().moe_status_str(int(code)).decode()


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoeError(code, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "tensors passed to libmoe must be contiguous CUDA tensors"
    return C.c_void_p(t.data_ptr())


def _stream_ptr(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def config_struct(cfg) -> _Config:
    """`cfg` is any object with the synth.Workload fields (or a dict of them)."""
    g = (lambda k: cfg[k]) if isinstance(cfg, dict) else (lambda k: getattr(cfg, k))
    score = g("score")
    route = g("route") if _has(cfg, "route") else "latent"
    out = g("out") if _has(cfg, "out") else "f32"
    precision = g("precision") if _has(cfg, "precision") else "mx"
    return _Config(g("d_model"), g("d_latent"), g("n_experts"), g("top_k"), g("expert_inter"), g("n_shared"),
                   g("shared_inter"), int(g("max_tokens")) if _has(cfg, "max_tokens") else g("tokens"),
                   SCORE_SOFTMAX if score == "softmax" else SCORE_SIGMOID_BIAS,
                   ROUTE_ON_HIDDEN if route == "hidden" else ROUTE_ON_LATENT,
                   OUT_BF16 if out == "bf16" else OUT_F32,
                   PRECISION_MIXED if precision == "mixed" else PRECISION_MX)


def _has(cfg, k):
    return (k in cfg) if isinstance(cfg, dict) else hasattr(cfg, k)


def mxfp4_encode(w: torch.Tensor, stream=None):
    """MXFP4-encode a float32 CUDA tensor [..., K] -> (codes [..., K/2], scales [..., K/32])."""
    assert w.dtype == torch.float32 and w.is_cuda
    w = w.contiguous()
    K = w.shape[-1]
    rows = w.numel() // K
    codes = torch.empty(*w.shape[:-1], K // 2, dtype=torch.uint8, device=w.device)
    scales = torch.empty(*w.shape[:-1], K // 32, dtype=torch.uint8, device=w.device)
    _check(lib().moe_mxfp4_encode(_ptr(w), rows, K, _ptr(codes), _ptr(scales), _stream_ptr(stream)),
           "moe_mxfp4_encode")
    return codes, scales


def mx_gemm(a_codes, a_scales, b_codes, b_scales, out=None, status=None, stream=None) -> torch.Tensor:
    """out[n][m] = sum_k dq(B[n][k]) dq(A[m][k]); A MXFP4 [M][K], B MXFP8 [N][K]."""
    M = a_codes.shape[0]
    N, K = b_codes.shape
    if out is None:
        out = torch.empty(N, M, dtype=torch.float32, device=a_codes.device)
    _check(lib().moe_mx_gemm(_ptr(a_codes), _ptr(a_scales), M, _ptr(b_codes), _ptr(b_scales), N, K, _ptr(out),
                             _ptr(status), _stream_ptr(stream)), "moe_mx_gemm")
    return out


PROBE_MX_E2M1_E4M3, PROBE_MX_E4M3_E4M3, PROBE_BF16 = 0, 1, 2


def mma_probe(kind: int, n: int, iters: int, status: torch.Tensor, stream=None) -> float:
    """Enqueue the tensor-core rate probe (see moe_mma_probe in include/moe.h);
    returns the FLOPs of the launch."""
    flops = C.c_double(0.0)
    _check(lib().moe_mma_probe(int(kind), int(n), int(iters), _ptr(status), C.byref(flops), _stream_ptr(stream)),
           "moe_mma_probe")
    return flops.value


class Plan:
    """A planned layer on one device.

    weights: dict with MXFP4 pairs ``(codes, scales)`` for 'p_down' [L][D],
    'p_up' [D][L], 'w_gate'/'w_up' [E][I][L], 'w_down' [E][L][I],
    's_gate'/'s_up' [S][Is][D], 's_down' [S][D][Is]; 'router' fp32 [E][L];
    optional 'bias' fp32 [E].  With the mixed precision scheme, bf16 tensors
    'p_down_bf16', 'p_up_bf16', 's_gate_bf16', 's_up_bf16', 's_down_bf16'
    replace the MXFP4 projections and shared experts.  All CUDA tensors on
    one device; the plan copies them, so they may be freed afterwards.
    """

    def __init__(self, cfg, weights: dict, max_tokens: Optional[int] = None):
        c = config_struct(cfg)
        if max_tokens is not None:
            c.max_tokens = int(max_tokens)
        self.cfg = c
        dev = weights["router"].device
        self.device = dev

        def mx(name):
            pair = weights.get(name)
            if pair is None:
                return _MX4(None, None)
            return _MX4(_ptr(pair[0]), _ptr(pair[1]))

        bias = weights.get("bias")
        bf = [_ptr(weights.get(n + "_bf16")) for n in ("p_down", "p_up", "s_gate", "s_up", "s_down")]
        w = _Weights(mx("p_down"), mx("p_up"), mx("w_gate"), mx("w_up"), mx("w_down"), mx("s_gate"), mx("s_up"),
                     mx("s_down"), _ptr(weights["router"]), _ptr(bias), *bf)
        h = C.c_void_p()
        with torch.cuda.device(dev):
            torch.cuda.synchronize()
            _check(lib().moe_plan(C.byref(c), C.byref(w), dev.index, C.byref(h)), "moe_plan")
        self._h = h
        self.max_tokens = c.max_tokens

    @property
    def handle(self):
        return self._h

    @property
    def out_dtype(self):
        return torch.bfloat16 if self.cfg.out_dtype == OUT_BF16 else torch.float32

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, debug: Optional[dict] = None,
                stream=None, stage_events=None) -> torch.Tensor:
        """y = layer(x); x bf16 [T][D] on the plan's device.  `debug` maps
        moe_debug field names to preallocated CUDA tensors to fill;
        `stage_events` is a list of NUM_STAGES + 1 torch.cuda.Event recorded
        between the stages."""
        assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.shape[1] == self.cfg.d_model
        x = x.contiguous()
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.cfg.d_model, dtype=self.out_dtype, device=x.device)
        assert out.dtype == self.out_dtype and out.shape == (T, self.cfg.d_model)
        dbg = None
        if debug or stage_events:
            dbg = _Debug()
            for k, t in (debug or {}).items():
                setattr(dbg, k, _ptr(t).value)
            if stage_events:
                assert len(stage_events) == NUM_STAGES + 1
                self._ev_arr = (C.c_void_p * (NUM_STAGES + 1))(*[e.cuda_event for e in stage_events])
                dbg.stage_events = C.cast(self._ev_arr, C.c_void_p)
        _check(lib().moe_forward(self._h, _ptr(x), T, _ptr(out), _stream_ptr(stream),
                                 C.byref(dbg) if dbg is not None else None), "moe_forward")
        return out

    def forward_host(self, x_host: torch.Tensor, y_host: torch.Tensor, stream=None):
        """End-to-end call with host buffers (bf16 [T][D] in, [T][D] out in the plan's output dtype)."""
        assert x_host.dtype == torch.bfloat16 and not x_host.is_cuda and y_host.dtype == self.out_dtype
        T = x_host.shape[0]
        _check(lib().moe_forward_host(self._h, C.c_void_p(x_host.data_ptr()), T, C.c_void_p(y_host.data_ptr()),
                                      _stream_ptr(stream)), "moe_forward_host")
        return y_host

    def quantile_balance(self, T: int, alpha: float = 1.0, target: int = 0, stream=None) -> torch.Tensor:
        """Quantile Balancing update of the selection bias from the last
        forward's T tokens (see moe_quantile_balance): the new bias, fp32 [E]."""
        out = torch.empty(self.cfg.n_experts, dtype=torch.float32, device=self.device)
        _check(lib().moe_quantile_balance(self._h, int(T), int(target), float(alpha), _ptr(out), _stream_ptr(stream)),
               "moe_quantile_balance")
        return out

    def set_bias(self, bias: torch.Tensor):
        """Install a new selection bias (fp32 [E] on the plan's device)."""
        assert bias.dtype == torch.float32 and bias.numel() == self.cfg.n_experts
        _check(lib().moe_set_bias(self._h, _ptr(bias.contiguous())), "moe_set_bias")

    def ep_row_bytes(self) -> int:
        """Bytes of one expert-parallel wire row (header, latent codes, scales, padding)."""
        return int(lib().moe_ep_row_bytes(self._h))

    def ep_dispatch(self, T: int, ranks: int, stream=None):
        """Expert-parallel dispatch of the last forward's T tokens over `ranks`
        virtual ranks: (wire uint8 [T*k][row_bytes], rank_offsets int64 [ranks+1])."""
        k = self.cfg.top_k
        wire = torch.empty(T * k, self.ep_row_bytes(), dtype=torch.uint8, device=self.device)
        offs = torch.empty(ranks + 1, dtype=torch.int64, device=self.device)
        _check(lib().moe_ep_dispatch(self._h, int(T), int(ranks), _ptr(wire), _ptr(offs), _stream_ptr(stream)),
               "moe_ep_dispatch")
        return wire, offs

    def ep_combine(self, T: int, wire: torch.Tensor, expert_out: torch.Tensor, stream=None) -> torch.Tensor:
        """c [T][L] fp32 from expert outputs in wire-row order (the matching combine)."""
        c = torch.empty(T, self.cfg.d_latent, dtype=torch.float32, device=self.device)
        _check(lib().moe_ep_combine(self._h, int(T), _ptr(wire), _ptr(expert_out.contiguous()), _ptr(c),
                                    _stream_ptr(stream)), "moe_ep_combine")
        return c

    def device_status(self) -> int:
        return lib().moe_get_device_status(self._h)

    def workspace_bytes(self) -> int:
        return lib().moe_workspace_bytes(self._h)

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().moe_free(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def debug_buffers(cfg, T: int, device, fields=DEBUG_FIELDS) -> dict:
    """Allocate CUDA tensors for the requested moe_debug fields of a T-token call."""
    D, L, E, k, I = cfg.d_model, cfg.d_latent, cfg.n_experts, cfg.top_k, cfg.expert_inter
    SIs = cfg.n_shared * cfg.shared_inter
    u8, f32, i32 = torch.uint8, torch.float32, torch.int32
    spec = {
        "xq": ((T, D), u8), "xs": ((T, D // 32), u8), "z": ((T, L), f32), "zq": ((T, L), u8),
        "zs": ((T, L // 32), u8), "hsq": ((T, SIs), u8), "hss": ((T, SIs // 32), u8),
        "logits": ((T, E), f32), "topk_idx": ((T, k), i32), "topk_w": ((T, k), f32), "counts": ((E,), i32),
        "offsets": ((E + 1,), i32), "sorted_token": ((T * k,), i32), "hq": ((T * k, I), u8),
        "hqs": ((T * k, I // 32), u8), "o": ((T * k, L), f32), "cq": ((T, L), u8), "cs": ((T, L // 32), u8),
    }
    return {f: torch.zeros(*spec[f][0], dtype=spec[f][1], device=device) for f in fields}
