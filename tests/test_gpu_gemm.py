"""The tcgen05 block-scaled GEMM engine (moe_mx_gemm) against the oracle's
exact block-scaled product.

out[n][m] = sum_k dq(B[n][k]) dq(A[m][k]) with MXFP4 A (weights) and MXFP8 B
(tokens), scales applied per 32 along K inside the MMA ("Kimi K3: 2.8
Trillion Parameters, Four Bits at a Time", section "What has to change in the
serving stacks": block-scaled FP4 weights against FP8 activations).  The GPU
accumulates in fp32; the bound below is the fp32 accumulation error relative
to sum_k |a_k b_k|.
"""
import numpy as np
import pytest
import torch

import oracle
import moe_expert_layer_top16_gb300 as moe
from gpu_util import DEV

pytestmark = pytest.mark.gpu


def random_operands(rng, M, N, K, a_scale=(118, 128), b_scale=(112, 124)):
    ac = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    as_ = rng.integers(*a_scale, size=(M, K // 32), dtype=np.uint8)
    bc = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    bc[(bc & 0x7F) == 0x7F] = 0x3E            # no NaN codes
    bs = rng.integers(*b_scale, size=(N, K // 32), dtype=np.uint8)
    return ac, as_, bc, bs


def run_gpu(ac, as_, bc, bs):
    t = [torch.from_numpy(a).to(DEV) for a in (ac, as_, bc, bs)]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = moe.mx_gemm(*t, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return out.cpu().numpy()


def check(ac, as_, bc, bs, what):
    got = run_gpu(ac, as_, bc, bs)
    ref = oracle.mx_matmul(ac, as_, bc, bs)
    mag = oracle.mx_matmul(ac & 0x77, as_, bc & 0x7F, bs)       # sum of |terms|
    K = bc.shape[1]
    err = np.abs(got - ref)
    bound = mag * (K * 2.0 ** -23) + 1e-30
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), (f"{what}: {int((err > bound).sum())} of {err.size} outside; worst n,m={worst} "
                                  f"got={got[worst]:.6g} ref={ref[worst]:.6g}")


def test_gemm_all_ones():
    M, N, K = 128, 16, 256
    ac = np.full((M, K // 2), 0x22, np.uint8)        # E2M1 1.0 in both nibbles
    as_ = np.full((M, K // 32), 127, np.uint8)
    bc = np.full((N, K), 0x38, np.uint8)             # E4M3 1.0
    bs = np.full((N, K // 32), 127, np.uint8)
    got = run_gpu(ac, as_, bc, bs)
    assert np.all(got == K), f"values seen: {np.unique(got)[:8]}"


def test_gemm_structured_rows_and_scales():
    # A row m = level (m % 8) everywhere, scale 2^(m % 5); B row n: 1.0 with
    # scale 2^(n % 3) on K-block (n % (K/32)), zero elsewhere.  Each output
    # isolates one (row scale, column scale, K-block) combination.
    M, N, K = 256, 48, 512
    lv = np.arange(M) % 8
    ac = np.repeat(((lv | (lv << 4)).astype(np.uint8))[:, None], K // 2, axis=1)
    as_ = np.repeat((127 + np.arange(M) % 5).astype(np.uint8)[:, None], K // 32, axis=1)
    bc = np.zeros((N, K), np.uint8)
    bs = np.full((N, K // 32), 127, np.uint8)
    for n in range(N):
        kb = n % (K // 32)
        bc[n, kb * 32:(kb + 1) * 32] = 0x38
        bs[n, kb] = 127 + n % 3
    got = run_gpu(ac, as_, bc, bs)
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    exp = np.array([[32 * e2m1[m % 8] * 2.0 ** (m % 5) * 2.0 ** (n % 3) for m in range(M)] for n in range(N)])
    bad = np.argwhere(got != exp)
    assert bad.size == 0, f"{len(bad)} wrong, first (n, m, got, exp): " + str(
        [(int(n), int(m), float(got[n, m]), float(exp[n, m])) for n, m in bad[:6]])


@pytest.mark.parametrize("M,N,K", [(128, 1, 128), (128, 16, 256), (256, 37, 512), (384, 240, 1024),
                                   (128, 241, 128), (256, 500, 384), (128, 3, 7168)])
def test_gemm_random_against_oracle(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 13 + K)
    check(*random_operands(rng, M, N, K), f"M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(256, 257, 256), (512, 3585, 384), (1024, 4063, 256), (768, 1000, 1024),
                                   (384, 700, 256)])
def test_gemm_wide_items_on_cta_pairs(M, N, K):
    # Batches above 256 tokens form wide items; with an even number of
    # 128-row weight tiles two CTAs share each MMA (M = 256, each CTA loading
    # half of the item's token rows) and items hold up to 224 tokens.  Last
    # items of 113, 1 and 31 tokens (N = 257, 3585, 4063) give pair halves of
    # 56, 8 and 16 rows; M = 384 has an odd tile count and stays unpaired.
    rng = np.random.default_rng(M * 11 + N * 3 + K)
    check(*random_operands(rng, M, N, K), f"M={M} N={N} K={K}")


def test_gemm_rejects_bad_shapes():
    t = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError):
        moe.mx_gemm(t.view(128, 2), t[:128].view(128, 1), t.view(1, 256)[:, :96], t[:3].view(1, 3))
