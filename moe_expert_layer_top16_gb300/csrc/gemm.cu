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
// Persistent kernel, one CTA per SM.  A thread that issues tcgen05.mma gets
// one MMA through per ~250 cycles whatever its N, while MMAs from different
// threads proceed concurrently; a thread issuing TMA copies is similarly
// limited.  So a CTA runs G "groups" side by side, each with its own
// producer warp, MMA warp, shared-memory stage ring and TMEM accumulator(s),
// and splits every work item's K tiles into G contiguous ranges:
//   warps 0..G-1     TMA producers: per 128-wide K tile, one 128x128 MXFP4
//                    box of A (unpacked into 16-byte groups in shared memory
//                    by the 16U4_ALIGN16B tensor type), ceil(N/16) 16-row
//                    boxes of B, and bulk copies of both scale tiles.
//   warps G..2G-1    MMA issuers: per K tile, re-arrange B's scales,
//                    tcgen05.cp both scale tiles into TMEM, 4 MMAs (K = 32
//                    each), commit the stage back to the producer.
//   warps 2G..2G+3   epilogue: wait for all G partial accumulators of the
//                    item, add them (group order, fp32), then fp32 stores,
//                    MXFP8 quantisation (one warp = 32 consecutive output
//                    features = one MX block) or SiLU-gating + MXFP8.
// With two accumulator buffers per group the epilogue of one item overlaps
// the MMAs of the next.  Work items come from per-expert tables (grouped
// GEMMs) or a dense m-tile x n-tile grid; CTAs take items blockIdx.x,
// +gridDim.x, ...
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

// Item `it`.  Grouped items come from the per-expert tables staged in shared
// memory (ioff, seg, counts): binary search for the expert, then token tile j
// and weight tile m of that expert.
__device__ __forceinline__ Item get_item(const GemmParams& p, int it, const int* ioff, const int* seg,
                                         const int* cnt) {
    Item w;
    if (p.dense) {
        const int mt = it % p.m_tiles;
        const int nt = it / p.m_tiles;
        w.a_row0 = mt * kBlockM;
        w.b_row0 = nt * p.n_max;
        w.n = min(p.n_max, p.n_tokens - w.b_row0);
        w.mt = mt;
    } else {
        int lo = 0, hi = p.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ioff[mid] <= it) lo = mid;
            else hi = mid - 1;
        }
        const int local = it - ioff[lo];
        const int j = local / p.mt_per_e, m = local - j * p.mt_per_e;
        w.a_row0 = lo * p.rows_per_e + m * kBlockM;
        w.b_row0 = seg[lo] + j * p.n_max;
        w.n = min(p.n_max, cnt[lo] - j * p.n_max);
        w.mt = m;
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

// K tiles [kb, ke) of an item handled by group g of G.
__device__ __forceinline__ void group_range(int KT, int g, int G, int& kb, int& ke) {
    kb = (KT * g) / G;
    ke = (KT * (g + 1)) / G;
}

// Shared memory after the stages: epilogue exchange buffer (2 x 2 warps x
// 32 lanes x 16 floats), then the barriers, then the grouped-item tables.
constexpr int kXbufBytes = 2 * 2 * 32 * 16 * 4;
constexpr int kMaxStagesPerGroup = 16;
constexpr int kBarBytes = (kMaxGroups * (2 * kMaxStagesPerGroup + 2 * 2 + 1)) * 8 + 16;
__host__ __device__ __forceinline__ int table_bytes(int E) { return E > 0 ? ((3 * (E + 1) * 4 + 15) & ~15) : 0; }

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
__global__ void __launch_bounds__(kGemmMaxThreads, 1) mx_gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr bool kMX = (KIND == KIND_MX);
    constexpr int kTileElems = kMX ? kBlockK : 32;      // K elements per 128-byte row of a stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int G = p.groups;
    const int S = p.stages;                 // per group
    const int NB = p.acc_bufs;              // accumulator buffers per group
    const SmemLayout L = stage_layout(p.n_max);
    uint8_t* tail = base + G * S * p.stage_bytes;
    float* xbuf = reinterpret_cast<float*>(tail);
    uint64_t* full = reinterpret_cast<uint64_t*>(tail + kXbufBytes);      // [G][kMaxStagesPerGroup]
    uint64_t* empty = full + kMaxGroups * kMaxStagesPerGroup;              // [G][kMaxStagesPerGroup]
    uint64_t* tfull = empty + kMaxGroups * kMaxStagesPerGroup;             // [G][2]
    uint64_t* tempty = tfull + kMaxGroups * 2;                             // [G][2]
    uint64_t* tdown = tempty + kMaxGroups * 2;                             // [G]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tdown + kMaxGroups);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* ioff_s = reinterpret_cast<int*>(tail + kXbufBytes + kBarBytes);
    int* seg_s = ioff_s + (p.dense ? 0 : p.E + 1);
    int* cnt_s = seg_s + (p.dense ? 0 : p.E + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int g = 0; g < G; ++g) {
            for (int s = 0; s < S; ++s) {
                mbar_init(&full[g * kMaxStagesPerGroup + s], 1);
                mbar_init(&empty[g * kMaxStagesPerGroup + s], 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&tfull[g * 2 + b], 1);
                mbar_init(&tempty[g * 2 + b], 4);
            }
            mbar_init(&tdown[g], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tmA);
        prefetch_tmap(&p.tmB);
    }
    if (warp == G) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (!p.dense) {
        for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
            ioff_s[i] = p.ioff[i];
            seg_s[i] = p.seg[i];
            cnt_s[i] = (i < p.E) ? p.counts[i] : 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_items = p.dense ? p.m_tiles * ((p.n_tokens + p.n_max - 1) / p.n_max) : ioff_s[p.E];
    const uint32_t cols_per_group = static_cast<uint32_t>(NB * p.n_max + 24);

    if (warp < G) {
        // ------------------------------------------------------------ producer of group g
        const int g = warp;
        if (lane == 0) {
            uint64_t* fullg = full + g * kMaxStagesPerGroup;
            uint64_t* emptyg = empty + g * kMaxStagesPerGroup;
            uint8_t* ring = base + g * S * p.stage_bytes;
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, issued_parity = 0;   // per-stage bits for the teardown drain
            for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
                const Item w = get_item(p, it, ioff_s, seg_s, cnt_s);
                if (w.n <= 0) {
                    if (w.n < 0 && g == 0) atomicCAS(p.status, 0, DEV_BAD_WORK);
                    continue;
                }
                int kb, ke;
                group_range(p.KT, g, G, kb, ke);
                const int nm = (w.n + 15) & ~15;
                const uint32_t tx = kMX ? static_cast<uint32_t>(p.a_tx_bytes + (nm / 16) * 2048 + 512 + nm * 4)
                                        : static_cast<uint32_t>(kBlockM * 128 + (nm / 16) * 2048);
                const uint8_t* sfa_tile = kMX ? p.sfa + static_cast<size_t>(w.a_row0 / kBlockM) * p.KT * 512 : nullptr;
                bool ok = true;
                for (int kt = kb; kt < ke; ++kt) {
                    if (!mbar_wait(&emptyg[stage], phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const int seg = kt / p.kseg_tiles;
                    const int kin = (kt - seg * p.kseg_tiles) * kTileElems;
                    uint8_t* sb = ring + stage * p.stage_bytes;
                    mbar_arrive_expect_tx(&fullg[stage], tx);
                    tma_load_2d(sb, &p.tmA, &fullg[stage], p.a_seg_x[seg] + kin, w.a_row0);
                    for (int c = 0; c < nm / 16; ++c)
                        tma_load_2d(sb + L.offB + c * 2048, &p.tmB, &fullg[stage], p.b_seg_x[seg] + kin,
                                    w.b_row0 + c * 16);
                    if constexpr (kMX) {
                        bulk_load(sb + L.offSFA, sfa_tile + static_cast<size_t>(kt) * 512, 512, &fullg[stage]);
                        bulk_load(sb + L.offSFBraw,
                                  p.sfb + (static_cast<size_t>(kt) * p.sfb_pitch + w.b_row0) * 4,
                                  static_cast<uint32_t>(nm * 4), &fullg[stage]);
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
                    if (issued & (1u << s)) mbar_wait_teardown(&fullg[s], (issued_parity >> s) & 1u, p.status);
            }
        }
    } else if (warp < 2 * G) {
        // ------------------------------------------------------------ MMA issuer of group g
        const int g = warp - G;
        uint64_t* fullg = full + g * kMaxStagesPerGroup;
        uint64_t* emptyg = empty + g * kMaxStagesPerGroup;
        uint8_t* ring = base + g * S * p.stage_bytes;
        const uint32_t gcol = tmem + static_cast<uint32_t>(g) * cols_per_group;
        const uint32_t sf_base = gcol + static_cast<uint32_t>(NB * p.n_max);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool any = false;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item w = get_item(p, it, ioff_s, seg_s, cnt_s);
            if (w.n <= 0) continue;
            int kb, ke;
            group_range(p.KT, g, G, kb, ke);
            if (ke <= kb) continue;
            const int nm = (w.n + 15) & ~15;
            const int natoms = (nm + 127) / 128;
            bool ok = mbar_wait(&tempty[g * 2 + acc], acc_phase ^ 1, abort_flag, p.status, DEV_TIMEOUT_MMA);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t d_tmem = gcol + acc * static_cast<uint32_t>(p.n_max);
            for (int kt = kb; kt < ke; ++kt) {
                ok = mbar_wait(&fullg[stage], phase, abort_flag, p.status, DEV_TIMEOUT_MMA);
                if (!__all_sync(0xffffffffu, ok)) goto mma_done;
                tc_fence_after();
                {
                    uint8_t* sb = ring + stage * p.stage_bytes;
                    const uint32_t accum_first = (kt == kb) ? 0u : 1u;
                    if constexpr (!kMX) {
                        if (lane == 0) {
                            const uint64_t adesc = sdesc_sw128(smem_u32(sb));
                            const uint64_t bdesc = sdesc_sw128(smem_u32(sb + L.offB));
                            const uint32_t idesc = idesc_tf32(kBlockM, nm);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                mma_tf32(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (accum_first | j) != 0 ? 1u : 0u);
                            tc_commit(&emptyg[stage]);
                        }
                    } else {
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
                            const uint32_t sfa_col = sf_base + static_cast<uint32_t>(kt & 1) * 12u;
                            const uint32_t sfb_col = sfa_col + 4u;
                            tc_cp_32x128b_x4(sfa_col, sdesc_rows16(smem_u32(sb + L.offSFA)));
                            for (int a = 0; a < natoms; ++a)
                                tc_cp_32x128b_x4(sfb_col + 4u * a, sdesc_rows16(smem_u32(sb + L.offSFBatom + a * 512)));
                            const uint64_t adesc = sdesc_sw128(smem_u32(sb));
                            const uint64_t bdesc = sdesc_sw128(smem_u32(sb + L.offB));
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t idesc = idesc_mxf8f6f4(kBlockM, nm, 5, 0, j, j);
                                mma_mxf8f6f4(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col, sfb_col,
                                             (accum_first | j) != 0 ? 1u : 0u);
                            }
                            tc_commit(&emptyg[stage]);
                        }
                    }
                    any = true;
                    __syncwarp();
                }
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (lane == 0) tc_commit(&tfull[g * 2 + acc]);
            __syncwarp();
            if (++acc == static_cast<uint32_t>(NB)) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    mma_done:
        // every tcgen05 operation issued above must finish before TMEM is freed
        if (lane == 0 && any) {
            tc_commit(&tdown[g]);
            mbar_wait_teardown(&tdown[g], 0, p.status);
        }
        __syncwarp();
    } else if (warp < 2 * G + 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        uint32_t acc = 0, acc_phase = 0;
        int chunk_parity = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item w = get_item(p, it, ioff_s, seg_s, cnt_s);
            if (w.n <= 0) continue;
            const int nm = (w.n + 15) & ~15;
            bool ok = true;
            for (int g = 0; g < G; ++g) {
                int kb, ke;
                group_range(p.KT, g, G, kb, ke);
                if (ke > kb && ok)
                    ok = mbar_wait(&tfull[g * 2 + acc], acc_phase, abort_flag, p.status, DEV_TIMEOUT_EPILOGUE);
            }
            if (!epi_all(ok && !*abort_flag)) break;
            tc_fence_after();
            const int region = (p.dense && w.mt >= p.epi_split) ? 1 : 0;
            const EpiParams& E = p.epi[region];
            const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
            const int rel_mt = w.mt - E.m_tile0;
            for (int n0 = 0; n0 < nm; n0 += 16) {
                // sum of the groups' partial accumulators, in group order
                float v[16];
                bool first = true;
                for (int g = 0; g < G; ++g) {
                    int kb, ke;
                    group_range(p.KT, g, G, kb, ke);
                    if (ke <= kb) continue;
                    float u[16];
                    tmem_ld16(tmem + t_lane + static_cast<uint32_t>(g) * cols_per_group +
                                  acc * static_cast<uint32_t>(p.n_max) + static_cast<uint32_t>(n0),
                              u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = first ? u[i] : v[i] + u[i];
                    first = false;
                }
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
            if (lane == 0) {
                for (int g = 0; g < G; ++g) {
                    int kb, ke;
                    group_range(p.KT, g, G, kb, ke);
                    if (ke > kb) mbar_arrive(&tempty[g * 2 + acc]);
                }
            }
            if (++acc == static_cast<uint32_t>(NB)) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == G) {
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

size_t gemm_smem_bytes(int n_max, int groups, int stages, int E) {
    return 1024 + static_cast<size_t>(groups) * stages * gemm_stage_bytes(n_max) + kXbufBytes + kBarBytes +
           table_bytes(E);
}

int gemm_stages(int n_max, int groups, int E) {
    int s = kMaxStagesPerGroup;
    while (s > 2 && gemm_smem_bytes(n_max, groups, s, E) > static_cast<size_t>(kSmemLimit)) --s;
    return s;
}

bool gemm_config_ok(int n_max, int groups, int acc_bufs) {
    if (groups < 1 || groups > kMaxGroups || acc_bufs < 1 || acc_bufs > 2) return false;
    if (n_max < 16 || n_max > kNMax || (n_max & 15)) return false;
    return groups * (acc_bufs * n_max + 24) <= kTmemCols;
}

cudaError_t gemm_setup() {
    cudaError_t err =
        cudaFuncSetAttribute(mx_gemm_kernel<KIND_MX>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(mx_gemm_kernel<KIND_TF32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t s) {
    if (!gemm_config_ok(p.n_max, p.groups, p.acc_bufs)) return cudaErrorInvalidValue;
    if (p.stages < 2 || p.stages > kMaxStagesPerGroup) return cudaErrorInvalidValue;
    const size_t smem = gemm_smem_bytes(p.n_max, p.groups, p.stages, p.dense ? 0 : p.E);
    if (smem > static_cast<size_t>(kSmemLimit)) return cudaErrorInvalidValue;
    if (p.kseg_tiles <= 0 || p.KT > 3 * p.kseg_tiles) return cudaErrorInvalidValue;
    if (!p.dense && (p.E <= 0 || p.E > 1024)) return cudaErrorInvalidValue;
    const int threads = (2 * p.groups + 4) * 32;
    if (p.kind == KIND_TF32)
        mx_gemm_kernel<KIND_TF32><<<grid, threads, smem, s>>>(p);
    else
        mx_gemm_kernel<KIND_MX><<<grid, threads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
