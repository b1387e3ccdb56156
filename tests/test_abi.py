"""The C-ABI library builds, loads without a GPU, exports every entry point
that include/moe.h declares, and rejects bad arguments on the host before it
touches a device."""
import ctypes as C
import os
import re
import subprocess

import pytest

import moe_expert_layer_top16_gb300 as moe
from moe_expert_layer_top16_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mbuild.build()
    return moe.lib()


def declared_entry_points():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"MOE_API\s+[^;(]*?\b(moe_\w+)\s*\(", text)))


def test_header_lists_the_binding_entry_points():
    assert declared_entry_points() == sorted(moe.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", mbuild.LIB], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in declared_entry_points():
        assert name in exported, name
        assert getattr(L, name) is not None
    # nothing else leaks out of the library
    assert {n for n in exported if not n.startswith("_")} <= set(declared_entry_points())


def test_status_strings(L):
    for code in range(7):
        assert moe.status_str(code)
    assert moe.status_str(0) == "ok"


def _cfg(**kw):
    base = dict(d_model=256, d_latent=128, n_experts=32, top_k=4, expert_inter=64, n_shared=1, shared_inter=128,
                max_tokens=64, score_fn=1, route_input=0, out_dtype=0, precision=0)
    base.update(kw)
    return moe._Config(*[base[f] for f, _ in moe._Config._fields_])


@pytest.mark.parametrize("bad", [dict(d_model=200), dict(d_latent=96), dict(expert_inter=48), dict(top_k=0),
                                 dict(top_k=33), dict(top_k=40, n_experts=32), dict(n_experts=0), dict(n_experts=2048),
                                 dict(route_input=2), dict(out_dtype=2), dict(route_input=-1),
                                 dict(max_tokens=0), dict(max_tokens=70000), dict(score_fn=7),
                                 dict(n_shared=1, shared_inter=0), dict(precision=2), dict(precision=-1)])
def test_plan_rejects_bad_config_without_a_device(L, bad):
    w = moe._Weights()
    h = C.c_void_p(123)
    rc = L.moe_plan(C.byref(_cfg(**bad)), C.byref(w), 0, C.byref(h))
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert not h.value


def test_plan_rejects_missing_weights(L):
    h = C.c_void_p()
    assert L.moe_plan(C.byref(_cfg()), C.byref(moe._Weights()), 0, C.byref(h)) == moe.MOE_ERR_INVALID_ARG
    # the mixed scheme needs the bf16 projections and shared experts, the MXFP4 ones do not stand in
    p = C.c_void_p(256)
    w = moe._Weights()
    for n in ("p_down", "p_up", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down"):
        setattr(w, n, moe._MX4(p, p))
    w.router_w = p
    assert L.moe_plan(C.byref(_cfg(precision=1)), C.byref(w), 0, C.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_plan(C.byref(_cfg()), None, 0, C.byref(h)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_plan(None, None, 0, C.byref(h)) == moe.MOE_ERR_INVALID_ARG


def test_expert_parallel_calls_reject_bad_arguments(L):
    p = C.c_void_p(256)
    assert L.moe_quantile_balance(None, 64, 0, 1.0, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_set_bias(None, p) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_ep_row_bytes(None) == 0
    assert L.moe_ep_dispatch(None, 1, 8, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_ep_combine(None, 1, p, p, p, None) == moe.MOE_ERR_INVALID_ARG


def test_null_plan_calls(L):
    assert L.moe_forward(None, None, 1, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_host(None, None, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_get_device_status(None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_bytes(None) == 0
    L.moe_free(None)


def test_utility_argument_checks(L):
    p = C.c_void_p(256)
    assert L.moe_mxfp4_encode(p, 4, 48, p, p, None) == moe.MOE_ERR_INVALID_ARG    # K % 32
    assert L.moe_mxfp4_encode(None, 4, 64, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_mxfp4_encode(C.c_void_p(258), 4, 64, p, p, None) == moe.MOE_ERR_INVALID_ARG  # misaligned
    assert L.moe_mx_gemm(p, p, 100, p, p, 4, 128, p, None, None) == moe.MOE_ERR_INVALID_ARG   # M % 128
    assert L.moe_mx_gemm(p, p, 128, p, p, 4, 96, p, None, None) == moe.MOE_ERR_INVALID_ARG    # K % 128
    assert L.moe_mx_gemm(p, p, 128, p, p, 0, 128, p, None, None) == moe.MOE_ERR_INVALID_ARG   # N
    assert L.moe_mx_gemm(C.c_void_p(272), p, 128, p, p, 4, 128, p, None, None) == moe.MOE_ERR_INVALID_ARG
