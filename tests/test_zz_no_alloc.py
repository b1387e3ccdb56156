"""moe_mx_gemm_noalloc: the block-scaled GEMM for callers that cannot
allocate device memory (their memory belongs to another allocator with a
fixed budget, or they cannot afford cudaFree's device-wide synchronisation).
It keeps its scratch in a fixed device array inside the library instead of
allocating; its results must match those of moe_mx_gemm, call after call,
although the shared array keeps whatever the previous call left in it, and
both must match the oracle's exact block-scaled product within the tensor
core's fp32 accumulation bound."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import moe_expert_layer_top16_gb300 as moe

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SCRATCH_BYTES = 4 << 20     # MOE_NOALLOC_SCRATCH_BYTES in include/moe.h


def operands(seed, M, N, K):
    rng = np.random.default_rng(seed)
    ac = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    as_ = rng.integers(118, 128, size=(M, K // 32), dtype=np.uint8)
    bc = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    bc[(bc & 0x7F) == 0x7F] = 0x3E
    bs = rng.integers(112, 124, size=(N, K // 32), dtype=np.uint8)
    return ac, as_, bc, bs


def call(fn, ops, status):
    M = ops[0].shape[0]
    N, K = ops[2].shape
    t = [torch.from_numpy(a).to(DEV) for a in ops]
    out = torch.full((N, M), float("nan"), dtype=torch.float32, device=DEV)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(C.c_void_p(t[0].data_ptr()), C.c_void_p(t[1].data_ptr()), M, C.c_void_p(t[2].data_ptr()),
            C.c_void_p(t[3].data_ptr()), N, K, C.c_void_p(out.data_ptr()), C.c_void_p(status.data_ptr()), stream)
    assert rc == moe.MOE_OK, moe.status_str(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.cpu().numpy()


def test_noalloc_matches_allocating_gemm_on_consecutive_calls():
    L = moe.lib(build_if_missing=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # two calls in a row with different shapes: the second runs on scratch
    # that still holds the first call's scale factors
    for seed, (M, N, K) in ((1, (256, 300, 1024)), (2, (128, 37, 512))):
        ops = operands(seed, M, N, K)
        got = call(L.moe_mx_gemm_noalloc, ops, status)
        ref = call(L.moe_mx_gemm, ops, status)
        exact = oracle.mx_matmul(*ops)
        mag = oracle.mx_matmul(ops[0] & 0x77, ops[1], ops[2] & 0x7F, ops[3])   # sum of |terms|
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= mag * (K * 2.0 ** -23) + 1e-30).all()
        # each product is added with at most two units in the last place of
        # the running sum; the result is one more fp32 rounding
        bound = mag * ((K + 8) * 2.0 ** -22) + np.abs(exact) * 2.0 ** -24 + 1e-30
        assert (np.abs(got - exact) <= bound).all()
        assert (np.abs(ref - exact) <= bound).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = moe.lib(build_if_missing=True)
    buf = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    p = C.c_void_p(buf.data_ptr())
    M, K = 8192, 16384                     # M*K/32 alone is the whole scratch
    assert M * K // 32 + 256 > SCRATCH_BYTES
    rc = L.moe_mx_gemm_noalloc(p, p, M, p, p, 16, K, p, None, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
