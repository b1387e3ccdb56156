// Block-scaled MXFP4 x MXFP8 GEMM engine on tcgen05 (sm_103a).
//
// out[token][feature] = sum_k dq(B[token][k]) * dq(A[feature][k])
//
// A = weights (MXFP4, the MMA's M=128 operand), B = tokens (MXFP8, the MMA's
// N operand, N = 16..240 per work item).  Putting the weights on M lets a
// ragged expert segment of n tokens run as one MMA of N = round16(n) instead
// of padding tokens to 128 -- the tile waste of grouped GEMMs over runtime-
// sized groups that "Kimi K3: 2.8 Trillion Parameters, Four Bits at a Time",
// section "What has to change in the serving stacks", describes.  The
// block scales are applied inside the MMA (kind::mxf8f6f4.block_scale),
// with E8M0 scales per 32 elements along K for both operands.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0     TMA producer: per 128-wide K tile, one 128x128 MXFP4 box of A
//              (unpacked into 16-byte groups in shared memory by the
//              16U4_ALIGN16B tensor type), ceil(N/16) 16-row boxes of B, and
//              two bulk copies for the scale factors.
//   warp 1     owns TMEM (512 columns) and issues the MMAs: per K tile it
//              re-arranges B's scales, copies both scale tiles shared->TMEM
//              (tcgen05.cp), issues 4 MMAs (K = 32 each) and commits the
//              stage back to the producer.
//   warps 2-5  epilogue: TMEM -> registers (tcgen05.ld), then fp32 stores or
//              MXFP8 quantisation (one warp = 32 consecutive output features =
//              one MX block) or SiLU-gating + MXFP8.
// Two TMEM accumulators let the epilogue of one item overlap the MMAs of the
// next.  Work items come from a device-side list (grouped GEMMs) or from a
// dense m-tile x n-tile grid; CTAs take items blockIdx.x, +gridDim.x, ...
//
// Every wait is bounded; on a time-out the kernel records a status code,
// drains what it issued and frees TMEM before returning.
#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kABytes = kBlockM * kBlockK;  // 128 rows x 128 B in shared memory (4-bit elements padded)
constexpr int kTmemCols = 512;

struct Item {
    int a_row0, b_row0, n, mt;
};

__device__ __forceinline__ Item get_item(const GemmParams& p, int it) {
    Item w;
    if (p.dense) {
        const int mt = it % p.m_tiles;
        const int nt = it / p.m_tiles;
        w.a_row0 = mt * kBlockM;
        w.b_row0 = nt * p.n_max;
        w.n = min(p.n_max, p.n_tokens - w.b_row0);
        w.mt = mt;
    } else {
        const int4 v = p.items[it];
        w.a_row0 = v.x;
        w.b_row0 = v.y;
        w.n = v.z;
        w.mt = v.w;
        // reject items that would read or write outside the buffers
        if (w.n <= 0 || w.n > p.n_max || w.a_row0 < 0 || (w.a_row0 & (kBlockM - 1)) ||
            w.a_row0 + kBlockM > p.a_rows || w.b_row0 < 0 || (w.b_row0 & 3) ||
            w.b_row0 + ((w.n + 15) & ~15) > p.b_rows || w.mt < 0) {
            w.n = -1;
        }
    }
    return w;
}

struct SmemLayout {
    int offB, offSFA, offSFBatom, offSFBraw;
};

__host__ __device__ __forceinline__ SmemLayout stage_layout(int n_max) {
    SmemLayout l;
    l.offB = kABytes;
    l.offSFA = l.offB + n_max * kBlockK;
    l.offSFBatom = l.offSFA + 512;
    l.offSFBraw = l.offSFBatom + ((n_max + 127) / 128) * 512;
    return l;
}

// Shared memory after the stages: epilogue exchange buffer (2 x 2 warps x
// 32 lanes x 16 floats), then the barriers.
constexpr int kXbufBytes = 2 * 2 * 32 * 16 * 4;
constexpr int kMaxStages = 16;
constexpr int kBarBytes = (2 * kMaxStages + 5) * 8 + 16;

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// All 128 epilogue threads agree on `ok` (named barrier 1 with an AND reduction).
__device__ __forceinline__ bool epi_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u)
        : "memory");
    return r != 0;
}

// Wait used while tearing down: bounded, ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_teardown(uint64_t* bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicCAS(status, 0, DEV_TIMEOUT_TEARDOWN);
            return false;
        }
    }
    return true;
}

template <int KIND>
__global__ void __launch_bounds__(kGemmThreads, 1) mx_gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr bool kMX = (KIND == KIND_MX);
    constexpr int kTileElems = kMX ? kBlockK : 32;      // K elements per 128-byte row of a stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    const SmemLayout L = stage_layout(p.n_max);
    uint8_t* tail = base + S * p.stage_bytes;
    float* xbuf = reinterpret_cast<float*>(tail);
    uint64_t* full = reinterpret_cast<uint64_t*>(tail + kXbufBytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;   // [2]
    uint64_t* tempty = tfull + 2;           // [2]
    uint64_t* tdown = tempty + 2;           // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tdown + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(tdown, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tmA);
        prefetch_tmap(&p.tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_items = p.dense ? p.m_tiles * ((p.n_tokens + p.n_max - 1) / p.n_max) : *p.n_items;
    const uint32_t sf_base_col = 2u * static_cast<uint32_t>(p.n_max);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, issued_parity = 0;   // per-stage bits for the teardown drain
            for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
                const Item w = get_item(p, it);
                if (w.n <= 0) {
                    if (w.n < 0) atomicCAS(p.status, 0, DEV_BAD_WORK);
                    continue;
                }
                const int nm = (w.n + 15) & ~15;
                const uint32_t tx = kMX ? static_cast<uint32_t>(p.a_tx_bytes + (nm / 16) * 2048 + 512 + nm * 4)
                                        : static_cast<uint32_t>(kBlockM * 128 + (nm / 16) * 2048);
                const uint8_t* sfa_tile = kMX ? p.sfa + static_cast<size_t>(w.a_row0 / kBlockM) * p.KT * 512 : nullptr;
                bool ok = true;
                for (int kt = 0; kt < p.KT; ++kt) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const int seg = kt / p.kseg_tiles;
                    const int kin = (kt - seg * p.kseg_tiles) * kTileElems;
                    uint8_t* sb = base + stage * p.stage_bytes;
                    mbar_arrive_expect_tx(&full[stage], tx);
                    tma_load_2d(sb, &p.tmA, &full[stage], p.a_seg_x[seg] + kin, w.a_row0);
                    for (int c = 0; c < nm / 16; ++c)
                        tma_load_2d(sb + L.offB + c * 2048, &p.tmB, &full[stage], p.b_seg_x[seg] + kin,
                                    w.b_row0 + c * 16);
                    if constexpr (kMX) {
                        bulk_load(sb + L.offSFA, sfa_tile + static_cast<size_t>(kt) * 512, 512, &full[stage]);
                        bulk_load(sb + L.offSFBraw,
                                  p.sfb + (static_cast<size_t>(kt) * p.sfb_pitch + w.b_row0) * 4,
                                  static_cast<uint32_t>(nm * 4), &full[stage]);
                    }
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == static_cast<uint32_t>(S)) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                // drain: every issued stage's copies must land before exit
                for (int s = 0; s < S; ++s)
                    if (issued & (1u << s)) mbar_wait_teardown(&full[s], (issued_parity >> s) & 1u, p.status);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool any = false;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item w = get_item(p, it);
            if (w.n <= 0) continue;
            const int nm = (w.n + 15) & ~15;
            const int natoms = (nm + 127) / 128;
            bool ok = mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_MMA);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * static_cast<uint32_t>(p.n_max);
            const uint32_t idesc_n = static_cast<uint32_t>(nm);
            for (int kt = 0; kt < p.KT; ++kt) {
                ok = mbar_wait(&full[stage], phase, abort_flag, p.status, DEV_TIMEOUT_MMA);
                if (!__all_sync(0xffffffffu, ok)) goto mma_done;
                tc_fence_after();
                if constexpr (!kMX) {
                    uint8_t* sb = base + stage * p.stage_bytes;
                    if (lane == 0) {
                        const uint64_t adesc = sdesc_sw128(smem_u32(sb));
                        const uint64_t bdesc = sdesc_sw128(smem_u32(sb + L.offB));
                        const uint32_t idesc = idesc_tf32(kBlockM, static_cast<int>(idesc_n));
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_tf32(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (kt | j) != 0 ? 1u : 0u);
                        tc_commit(&empty[stage]);
                    }
                    any = true;
                    __syncwarp();
                } else {
                    uint8_t* sb = base + stage * p.stage_bytes;
                    // B scales arrive as one uint32 per token row (4 bytes = the 4
                    // K-blocks of this tile).  The 32x128b copy wants 32 rows of
                    // 16 bytes where row i holds tokens i, i+32, i+64, i+96.
                    const uint32_t* raw = reinterpret_cast<const uint32_t*>(sb + L.offSFBraw);
                    for (int a = 0; a < natoms; ++a) {
                        const int r0 = a * 128 + lane;
                        uint4 v;
                        v.x = (r0 < nm) ? raw[r0] : 0u;
                        v.y = (r0 + 32 < nm) ? raw[r0 + 32] : 0u;
                        v.z = (r0 + 64 < nm) ? raw[r0 + 64] : 0u;
                        v.w = (r0 + 96 < nm) ? raw[r0 + 96] : 0u;
                        *reinterpret_cast<uint4*>(sb + L.offSFBatom + a * 512 + lane * 16) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t sfa_col = tmem + sf_base_col + static_cast<uint32_t>(kt & 1) * 12u;
                        const uint32_t sfb_col = sfa_col + 4u;
                        tc_cp_32x128b_x4(sfa_col, sdesc_rows16(smem_u32(sb + L.offSFA)));
                        for (int a = 0; a < natoms; ++a)
                            tc_cp_32x128b_x4(sfb_col + 4u * a, sdesc_rows16(smem_u32(sb + L.offSFBatom + a * 512)));
                        const uint64_t adesc = sdesc_sw128(smem_u32(sb));
                        const uint64_t bdesc = sdesc_sw128(smem_u32(sb + L.offB));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t idesc = idesc_mxf8f6f4(kBlockM, static_cast<int>(idesc_n), 5, 0, j, j);
                            mma_mxf8f6f4(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col, sfb_col,
                                         (kt | j) != 0 ? 1u : 0u);
                        }
                        tc_commit(&empty[stage]);
                    }
                    any = true;
                    __syncwarp();
                }
                if (++stage == static_cast<uint32_t>(p.stages)) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (lane == 0) tc_commit(&tfull[acc]);
            __syncwarp();
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    mma_done:
        // every tcgen05 operation issued above must finish before TMEM is freed
        if (lane == 0 && any) {
            tc_commit(tdown);
            mbar_wait_teardown(tdown, 0, p.status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        uint32_t acc = 0, acc_phase = 0;
        int chunk_parity = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item w = get_item(p, it);
            if (w.n <= 0) continue;
            const int nm = (w.n + 15) & ~15;
            bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status, DEV_TIMEOUT_EPILOGUE);
            if (!epi_all(ok && !*abort_flag)) break;
            tc_fence_after();
            const int region = (p.dense && w.mt >= p.epi_split) ? 1 : 0;
            const EpiParams& E = p.epi[region];
            const uint32_t t_base = tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * static_cast<uint32_t>(p.n_max);
            const int rel_mt = w.mt - E.m_tile0;
            for (int n0 = 0; n0 < nm; n0 += 16) {
                float v[16];
                tmem_ld16(t_base + static_cast<uint32_t>(n0), v);
                if (E.mode == EPI_SILU_QUANT) {
                    float* xb = xbuf + chunk_parity * (2 * 32 * 16);
                    chunk_parity ^= 1;
                    if (q >= 2) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) xb[(q - 2) * 512 + i * 32 + lane] = v[i];
                    }
                    named_bar_sync(2, 128);
                    if (q < 2) {
                        const int64_t col = E.col0 + static_cast<int64_t>(rel_mt) * 64 + 32 * q + lane;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int n = n0 + i;
                            if (n < w.n) {
                                const float h = silu_f(v[i]) * xb[q * 512 + i * 32 + lane];
                                uint8_t sc;
                                const uint8_t code = warp_mx8_quant(h, &sc);
                                const int64_t row = w.b_row0 + n;
                                E.out_q[row * E.ld_q + col] = code;
                                if (lane == 0) E.out_sf[sf_byte_offset(row, col, E.sf_pitch)] = sc;
                            }
                        }
                    }
                } else {
                    const int64_t col = E.col0 + static_cast<int64_t>(rel_mt) * 128 + 32 * q + lane;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = n0 + i;
                        if (n < w.n) {
                            const int64_t row = w.b_row0 + n;
                            if (E.out_f32) {
                                if (E.f32_split) {
                                    const float hi = tf32_round(v[i]);
                                    E.out_f32[row * E.ld_f32 + col] = hi;
                                    E.out_f32[row * E.ld_f32 + col + E.f32_split] = v[i] - hi;
                                } else {
                                    E.out_f32[row * E.ld_f32 + col] = v[i];
                                }
                            }
                            if (E.mode == EPI_QUANT) {
                                uint8_t sc;
                                const uint8_t code = warp_mx8_quant(v[i], &sc);
                                E.out_q[row * E.ld_q + col] = code;
                                if (lane == 0) E.out_sf[sf_byte_offset(row, col, E.sf_pitch)] = sc;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int gemm_stage_bytes(int n_max) {
    const SmemLayout l = stage_layout(n_max);
    const int bytes = l.offSFBraw + ((n_max * 4 + 15) & ~15);
    return (bytes + 1023) & ~1023;
}

size_t gemm_smem_bytes(int n_max, int stages) {
    return 1024 + static_cast<size_t>(stages) * gemm_stage_bytes(n_max) + kXbufBytes + kBarBytes;
}

int gemm_stages(int n_max) {
    int s = kMaxStages;
    while (s > 2 && gemm_smem_bytes(n_max, s) > static_cast<size_t>(kSmemLimit)) --s;
    return s;
}

cudaError_t gemm_setup() {
    cudaError_t err =
        cudaFuncSetAttribute(mx_gemm_kernel<KIND_MX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(mx_gemm_kernel<KIND_TF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t s) {
    const size_t smem = gemm_smem_bytes(p.n_max, p.stages);
    if (p.kseg_tiles <= 0 || p.KT > 3 * p.kseg_tiles) return cudaErrorInvalidValue;
    if (p.kind == KIND_TF32)
        mx_gemm_kernel<KIND_TF32><<<grid, kGemmThreads, smem, s>>>(p);
    else
        mx_gemm_kernel<KIND_MX><<<grid, kGemmThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
