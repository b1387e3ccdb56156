"""CPU oracle for the K3-style sparse MoE layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links or calls
it, and the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64), whose header lists
the passages of the pages each step follows and every reading taken where the
pages are silent.  This module only compiles that file (gcc, OpenMP) and
marshals numpy arrays through ctypes.

Parity status per function (what pins it is in ``tests/test_oracle_*.py``):
  mxfp4_encode   pinned: the printed table of "Four bits from the start",
                 hand cases of the tie rule, the E2M1 grid.
  mxfp8_quantize pinned: hand cases from the OCP E4M3 definition, an
                 independent exact-rational rounding over every bf16 value,
                 scale equivariance.
  decode tables  pinned: OCP element definitions (hand cases).
  mx_matmul      pinned: exact rational sum on small shapes; reduces to a
                 numpy matmul when every scale is 2^0.
  route/permute/combine  pinned: the printed output of the one-page data
                 path ("What it takes to serve it"), brute force, invariants.
  moe_forward    pinned by its parts, by a dense all-experts recomputation on
                 the small layer, and by linearity of the combine; the pages
                 print no K3-shaped output, so end-to-end K3 values beyond
                 that are parity unpinned.
  bf16_round     pinned: hand cases of round-to-nearest-even on the bf16 grid,
                 and the library conversion (torch) on random fp32 values.
  quantile_balance  pinned: with a step of 1, an expert updated alone gets
                 exactly the target load (brute force over the batch); the
                 update is unchanged when every bias shifts by a constant;
                 repeated damped updates drive a Zipf-skewed load toward the
                 mean.
  moe_forward, mixed scheme (BF16 projections and shared experts): pinned by
                 a dense recomputation from numpy matmuls of the decoded bf16
                 weights, and by one-hot projection rows that copy x into z.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _MX(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p)]


class _Cfg(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("D", "L", "E", "k", "I", "S", "Is", "softmax", "route_hidden", "mixed")]


class _Weights(C.Structure):
    _fields_ = [("p_down", _MX), ("p_up", _MX),
                ("w_gate", C.POINTER(_MX)), ("w_up", C.POINTER(_MX)), ("w_down", C.POINTER(_MX)),
                ("s_gate", C.POINTER(_MX)), ("s_up", C.POINTER(_MX)), ("s_down", C.POINTER(_MX)),
                ("router", C.c_void_p), ("bias", C.c_void_p),
                ("p_down_bf", C.c_void_p), ("p_up_bf", C.c_void_p), ("s_gate_bf", C.c_void_p),
                ("s_up_bf", C.c_void_p), ("s_down_bf", C.c_void_p)]


_OUT_FIELDS = ["y", "xq", "xs", "z", "zq", "zs", "hs", "hsq", "hss", "logits", "idx", "gates",
               "h", "hq", "hqs", "o", "c", "cq", "cs"]


class _Out(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in _OUT_FIELDS]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            i64 = C.c_int64
            L.orc_e2m1_decode.restype = C.c_double
            L.orc_e2m1_decode.argtypes = [C.c_int]
            L.orc_e4m3_decode.restype = C.c_double
            L.orc_e4m3_decode.argtypes = [C.c_int]
            L.orc_e8m0_decode.restype = C.c_double
            L.orc_e8m0_decode.argtypes = [C.c_int]
            L.orc_e4m3_encode.restype = C.c_uint8
            L.orc_e4m3_encode.argtypes = [C.c_double]
            for fn in ("orc_mxfp4_encode_f64", "orc_mxfp4_encode_f32", "orc_mxfp8_quantize"):
                getattr(L, fn).restype = None
                getattr(L, fn).argtypes = [P, i64, i64, P, P]
            L.orc_mx_matmul.restype = None
            L.orc_mx_matmul.argtypes = [P, P, i64, P, P, i64, i64, P]
            L.orc_route.restype = None
            L.orc_route.argtypes = [P, P, i64, C.c_int, C.c_int, C.c_int, P, P]
            L.orc_permute.restype = None
            L.orc_permute.argtypes = [P, i64, C.c_int, C.c_int, P, P, P]
            L.orc_combine.restype = None
            L.orc_combine.argtypes = [P, P, P, i64, C.c_int, i64, P]
            L.orc_quantile_balance.restype = None
            L.orc_quantile_balance.argtypes = [P, P, i64, C.c_int, C.c_int, i64, C.c_double, P]
            L.orc_bf16_round_array.restype = None
            L.orc_bf16_round_array.argtypes = [P, i64, P]
            L.orc_moe_forward.restype = C.c_int
            L.orc_moe_forward.argtypes = [C.POINTER(_Cfg), C.POINTER(_Weights), P, i64, P, C.c_int,
                                          C.POINTER(_Out)]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- element codecs
def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e8m0_decode(code: int) -> float:
    return lib().orc_e8m0_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def mxfp4_encode(w: np.ndarray):
    """MXFP4 encode of [rows][K] (fp32 or fp64) -> (codes [rows][K/2], scales [rows][K/32])."""
    w = np.ascontiguousarray(w)
    rows, K = w.shape
    assert K % 32 == 0
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    if w.dtype == np.float64:
        lib().orc_mxfp4_encode_f64(_p(w), rows, K, _p(codes), _p(scales))
    else:
        w = np.ascontiguousarray(w, dtype=np.float32)
        lib().orc_mxfp4_encode_f32(_p(w), rows, K, _p(codes), _p(scales))
    return codes, scales


def mxfp4_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Values of an MXFP4 matrix (fp64), via the oracle's element decoders."""
    rows, kh = codes.shape
    K = kh * 2
    tab = np.array([e2m1_decode(c) for c in range(16)])
    sc = np.array([e8m0_decode(c) for c in range(256)])
    lo = tab[codes & 15]
    hi = tab[codes >> 4]
    v = np.empty((rows, K))
    v[:, 0::2] = lo
    v[:, 1::2] = hi
    return v * np.repeat(sc[scales], 32, axis=1)


def mxfp8_quantize(v: np.ndarray):
    """MXFP8 quantise of fp32 [rows][K] -> (codes [rows][K], scales [rows][K/32])."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    if v.ndim == 1:
        v = v[None]
    rows, K = v.shape
    assert K % 32 == 0
    codes = np.zeros((rows, K), np.uint8)
    scales = np.zeros((rows, K // 32), np.uint8)
    lib().orc_mxfp8_quantize(_p(v), rows, K, _p(codes), _p(scales))
    return codes, scales


def bf16_round(v: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), nearest with ties to even."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, np.uint16)
    lib().orc_bf16_round_array(_p(v), v.size, _p(out))
    return out


def bf16_decode(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> their exact values (fp64): the upper half of an fp32."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def mxfp8_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    tab = np.array([e4m3_decode(c) for c in range(256)])
    sc = np.array([e8m0_decode(c) for c in range(256)])
    return tab[codes] * np.repeat(sc[scales], 32, axis=-1)


def mx_matmul(a_codes, a_scales, b_codes, b_scales) -> np.ndarray:
    """out[n][m] = sum_k dq(B[n][k]) dq(A[m][k]); A MXFP4 [M][K], B MXFP8 [N][K]."""
    M = a_codes.shape[0]
    N, K = b_codes.shape
    out = np.zeros((N, M), np.float64)
    lib().orc_mx_matmul(_p(np.ascontiguousarray(a_codes)), _p(np.ascontiguousarray(a_scales)), M,
                        _p(np.ascontiguousarray(b_codes)), _p(np.ascontiguousarray(b_scales)), N, K,
                        _p(out))
    return out


# ---------------------------------------------------------------- routing / dispatch
def route(logits: np.ndarray, k: int, softmax: bool, bias=None):
    """Top-k selection and gates for logits [T][E] (fp32 or fp64 values)."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    gates = np.zeros((T, k), np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    lib().orc_route(_p(lg), None if b is None else _p(b), T, E, k, int(bool(softmax)), _p(idx), _p(gates))
    return idx, gates


def quantile_balance(logits: np.ndarray, bias, k: int, target: int, alpha: float) -> np.ndarray:
    """Quantile Balancing update of the selection bias from logits [T][E]
    (the reading in moe_oracle.c); returns the new bias (fp64 [E])."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = lg.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.zeros(E, np.float64)
    lib().orc_quantile_balance(_p(lg), None if b is None else _p(b), T, E, k, int(target), float(alpha), _p(out))
    return out


def permute(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    order = np.zeros(T * k, np.int32)
    lib().orc_permute(_p(idx), T, k, E, _p(counts), _p(offsets), _p(order))
    return counts, offsets, order


def combine(rows: np.ndarray, order: np.ndarray, gates: np.ndarray, T: int, k: int):
    rows = np.ascontiguousarray(rows, dtype=np.float64)
    D = rows.shape[1]
    y = np.zeros((T, D), np.float64)
    lib().orc_combine(_p(rows), _p(np.ascontiguousarray(order, dtype=np.int32)),
                      _p(np.ascontiguousarray(gates, dtype=np.float64).ravel()), T, k, D, _p(y))
    return y


# ---------------------------------------------------------------- the layer
class LayerWeights:
    """MXFP4 weights of one layer in the oracle's byte layout.

    `enc` maps a tensor name ('p_down', 'p_up', 'router', 'bias') to arrays,
    and ('w_gate', e) / ('s_gate', s) style keys to (codes, scales) per expert.
    Experts that are absent may not be selected.
    """

    def __init__(self, wl, enc: dict):
        self.wl = wl
        self.enc = enc
        E, S = wl.n_experts, wl.n_shared
        self._keep = []

        def mx(pair):
            if pair is None:
                return _MX(None, None)
            c, s = (np.ascontiguousarray(a) for a in pair)
            self._keep += [c, s]
            return _MX(c.ctypes.data, s.ctypes.data)

        def arr(name, n):
            a = (_MX * n)()
            for i in range(n):
                a[i] = mx(enc.get((name, i)))
            self._keep.append(a)
            return a

        router = np.ascontiguousarray(enc["router"], dtype=np.float32)
        bias = enc.get("bias")
        bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self._keep += [router, bias]

        def bf(name):
            a = enc.get(name + "_bf16")
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=np.uint16)
            self._keep.append(a)
            return a.ctypes.data

        self.cw = _Weights(mx(enc.get("p_down")), mx(enc.get("p_up")),
                           arr("w_gate", E), arr("w_up", E), arr("w_down", E),
                           arr("s_gate", S), arr("s_up", S), arr("s_down", S),
                           router.ctypes.data, None if bias is None else bias.ctypes.data,
                           bf("p_down"), bf("p_up"), bf("s_gate"), bf("s_up"), bf("s_down"))


def moe_forward(wl, weights: LayerWeights, x_bf16_bits: np.ndarray, force_idx=None,
                route_only: bool = False, want=("y",)):
    """Run the oracle layer on tokens x (uint16 bf16 bit patterns [n][D]).

    Returns a dict with the requested outputs (names of the C struct orc_out).
    """
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    n, D = x.shape
    L, E, k, I, S, Is = wl.d_latent, wl.n_experts, wl.top_k, wl.expert_inter, wl.n_shared, wl.shared_inter
    shapes = {
        "y": ((n, D), np.float32), "xq": ((n, D), np.uint8), "xs": ((n, D // 32), np.uint8),
        "z": ((n, L), np.float32), "zq": ((n, L), np.uint8), "zs": ((n, L // 32), np.uint8),
        "hs": ((n, S * Is), np.float32), "hsq": ((n, S * Is), np.uint8),
        "hss": ((n, S * Is // 32), np.uint8), "logits": ((n, E), np.float64),
        "idx": ((n, k), np.int32), "gates": ((n, k), np.float64),
        "h": ((n, k, I), np.float32), "hq": ((n, k, I), np.uint8), "hqs": ((n, k, I // 32), np.uint8),
        "o": ((n, k, L), np.float32), "c": ((n, L), np.float32), "cq": ((n, L), np.uint8),
        "cs": ((n, L // 32), np.uint8),
    }
    res = {}
    out = _Out()
    for name in want:
        shp, dt = shapes[name]
        res[name] = np.zeros(shp, dt)
        setattr(out, name, res[name].ctypes.data)
    mixed = getattr(wl, "precision", "mx") == "mixed"
    if mixed:
        for name in ("p_down", "p_up") + (("s_gate", "s_up", "s_down") if S > 0 else ()):
            assert weights.enc.get(name + "_bf16") is not None, f"mixed scheme needs bf16 {name}"
    cfg = _Cfg(D, L, E, k, I, S, Is, 1 if wl.score == "softmax" else 0, 1 if wl.route == "hidden" else 0,
               1 if mixed else 0)
    fi = None
    if force_idx is not None:
        fi = np.ascontiguousarray(force_idx, dtype=np.int32)
        assert fi.shape == (n, k)
    rc = lib().orc_moe_forward(C.byref(cfg), C.byref(weights.cw), _p(x), n,
                               None if fi is None else _p(fi), int(route_only), C.byref(out))
    if rc != 0:
        raise RuntimeError(f"oracle forward failed with code {rc}")
    return res


def encode_layer(wl, fetch, experts=None, device_hint=None) -> LayerWeights:
    """Encode a layer's fp32 weights with the oracle's MXFP4 encoder.

    `fetch(name, index)` returns the fp32 weight as a numpy array (the
    synthetic generator, possibly copied from another device).  `experts`
    limits which routed experts are encoded (None = all).
    """
    enc = {}
    if getattr(wl, "precision", "mx") == "mixed":
        # the mixed scheme: bf16 latent projections and shared experts
        for name in ("p_down", "p_up"):
            enc[name + "_bf16"] = bf16_round(fetch(name, 0))
        if wl.n_shared > 0:
            for name in ("s_gate", "s_up", "s_down"):
                enc[name + "_bf16"] = np.stack([bf16_round(fetch(name, s)) for s in range(wl.n_shared)])
    else:
        for name in ("p_down", "p_up"):
            enc[name] = mxfp4_encode(fetch(name, 0))
        for s in range(wl.n_shared):
            for name in ("s_gate", "s_up", "s_down"):
                enc[(name, s)] = mxfp4_encode(fetch(name, s))
    for e in (range(wl.n_experts) if experts is None else experts):
        for name in ("w_gate", "w_up", "w_down"):
            enc[(name, e)] = mxfp4_encode(fetch(name, e))
    enc["router"] = np.ascontiguousarray(fetch("router", 0), dtype=np.float32)
    enc["bias"] = fetch("bias", 0)
    return LayerWeights(wl, enc)
