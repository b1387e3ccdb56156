// Tensor-core issue-rate probe: the peak that the layer's GEMMs are measured
// against, measured on the GPU at hand instead of taken from a data sheet.
//
// One CTA per SM issues back-to-back tcgen05.mma instructions of one kind on
// operand tiles that stay in shared memory (no global loads), accumulating
// into one TMEM accumulator of 128 lanes x N columns.  Kinds:
//   PROBE_MX_E2M1_E4M3  kind::mxf8f6f4, A E2M1 (unpacked), B E4M3, E8M0
//                       block scales -- the layer's block-scaled MMA
//   PROBE_MX_E4M3_E4M3  kind::mxf8f6f4, both E4M3
//   PROBE_BF16          kind::f16 with bf16 operands, fp32 accumulate
// Each instruction is M = 128 x N x (32 bytes of K per row: 32 fp8 / 16 bf16
// elements); four of them cover one 128-byte K row of the swizzled tiles.
// The final commit is waited on with a bounded wait.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeSmem = 160 * 1024;    // keeps one CTA per SM (one TMEM allocation each)

template <int KIND>
__global__ void __launch_bounds__(kProbeThreads, 1) mma_probe_kernel(int iters, int n, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* a_tile = base;                     // 128 rows x 128 B
    uint8_t* b_tile = base + 16384;             // n rows x 128 B (n <= 256)
    uint8_t* sf = base + 16384 + 32768;         // 512 B of A scales, 2 x 512 B of B scales
    uint64_t* bar = reinterpret_cast<uint64_t*>(sf + 2048);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int warp = threadIdx.x >> 5;
    // operands: small finite values (codes 0x38: 1.0 in E4M3, 1.5 in E2M1;
    // bf16 1.0), scales 2^0
    for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += blockDim.x) {
        uint32_t v = 0x38383838u;
        if (KIND == PROBE_BF16) v = 0x3F803F80u;
        reinterpret_cast<uint32_t*>(base)[i] = v;
    }
    for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sf)[i] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp == 1) {
        const uint64_t adesc = sdesc_sw128(smem_u32(a_tile));
        const uint64_t bdesc = sdesc_sw128(smem_u32(b_tile));
        const uint32_t sfa_col = tmem + 256, sfb_col = tmem + 260;
        if constexpr (KIND != PROBE_BF16) {
            if (elect_one()) {
                tc_cp_32x128b_x4(sfa_col, sdesc_rows16(smem_u32(sf)));
                tc_cp_32x128b_x4(sfb_col, sdesc_rows16(smem_u32(sf + 512)));
                tc_cp_32x128b_x4(sfb_col + 4, sdesc_rows16(smem_u32(sf + 1024)));
            }
            __syncwarp();
        }
        const uint32_t idesc0 = (KIND == PROBE_BF16) ? idesc_bf16(128, n)
                                : idesc_mxf8f6f4(128, n, KIND == PROBE_MX_E2M1_E4M3 ? 5 : 0, 0, 0, 0);
        for (int it = 0; it < iters; ++it) {
            if (elect_one()) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t acc = (it | j) != 0 ? 1u : 0u;
                    if constexpr (KIND == PROBE_BF16) {
                        mma_bf16(tmem, adesc + 2 * j, bdesc + 2 * j, idesc0, acc);
                    } else {
                        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(j) << 4) |
                                               (static_cast<uint32_t>(j) << 29);
                        mma_mxf8f6f4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col, sfb_col, acc);
                    }
                }
            }
            __syncwarp();
        }
        if (elect_one()) {
            tc_commit(bar);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicCAS(status, 0, DEV_TIMEOUT_MMA);
                    break;
                }
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_mma_probe(int kind, int n, int iters, int grid, int* status, double* flops, cudaStream_t s) {
    if (n < 16 || n > 256 || (n & 15) || iters < 1 || grid < 1 || !status) return cudaErrorInvalidValue;
    if (kind != PROBE_BF16 && n > kNMax) return cudaErrorInvalidValue;       // scale columns share the 512
    const double k_per_instr = (kind == PROBE_BF16) ? 16.0 : 32.0;
    *flops = 2.0 * 128.0 * n * k_per_instr * 4.0 * iters * grid;
    cudaError_t err = cudaSuccess;
    switch (kind) {
        case PROBE_MX_E2M1_E4M3:
            err = cudaFuncSetAttribute(mma_probe_kernel<PROBE_MX_E2M1_E4M3>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
            if (err == cudaSuccess)
                mma_probe_kernel<PROBE_MX_E2M1_E4M3><<<grid, kProbeThreads, kProbeSmem, s>>>(iters, n, status);
            break;
        case PROBE_MX_E4M3_E4M3:
            err = cudaFuncSetAttribute(mma_probe_kernel<PROBE_MX_E4M3_E4M3>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
            if (err == cudaSuccess)
                mma_probe_kernel<PROBE_MX_E4M3_E4M3><<<grid, kProbeThreads, kProbeSmem, s>>>(iters, n, status);
            break;
        case PROBE_BF16:
            err = cudaFuncSetAttribute(mma_probe_kernel<PROBE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kProbeSmem);
            if (err == cudaSuccess) mma_probe_kernel<PROBE_BF16><<<grid, kProbeThreads, kProbeSmem, s>>>(iters, n, status);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe
