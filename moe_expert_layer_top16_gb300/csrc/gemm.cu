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
// Persistent kernel, one CTA per SM, organised as G "groups", each with its
// own TMA producer warp, MMA warp, shared-memory stage ring and TMEM
// accumulator(s).  Groups form IP item lanes x KS K-splits: the CTA's items
// (blockIdx.x, +gridDim.x, ...) are dealt round-robin to the item lanes, and
// the KS groups of a lane split each item's K tiles into contiguous ranges.
// Independent issuers matter because one thread's tcgen05 / TMA issue rate,
// not the tensor pipe, bounds small-N items: several item lanes keep the
// pipe and HBM busy on short-K GEMMs, K-splits on long-K ones.
//   warps 0..G-1     TMA producers: per 128-wide K tile, one 128x128 MXFP4
//                    box of A (unpacked into 16-byte groups in shared memory
//                    by the 16U4_ALIGN16B tensor type), ceil(N/16) 16-row
//                    boxes of B, and bulk copies of both scale tiles.
//   warps G..2G-1    MMA issuers: per K tile, re-arrange B's scales,
//                    tcgen05.cp both scale tiles into TMEM, 4 MMAs (K = 32
//                    each), commit the stage back to the producer.
//   warps 2G..2G+7   epilogue, two warpgroups taking the CTA's items in
//                    turn: wait for the KS partial accumulators of the item,
//                    add them (group order, fp32), then fp32 stores, MXFP8
//                    quantisation (one warp = 32 consecutive output features
//                    = one MX block) or SiLU-gating + MXFP8.
// Both roles that issue asynchronous work run warp-converged and issue from
// one elected lane.  With two accumulator buffers per group the epilogue of
// one item overlaps the MMAs of the next.  Work items come from per-expert
// tables (grouped GEMMs) or a dense m-tile x n-tile grid.
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

// Scalar launch parameters held in registers for the whole kernel (reading
// them from the parameter space would repeat after every asm statement that
// clobbers memory).
struct Hot {
    int KT, n_max, stage_bytes, a_tx_bytes, kseg_tiles, b_box, b_row1, b_producer;
    int dense, m_tiles, mt_base, n_tokens, a_rows, b_rows, E, mt_per_e, rows_per_e, epi_split;
    int ax0, ax1, ax2, bx0, bx1, bx2;
    int64_t sfb_pitch;
    const uint8_t* sfa;
    const uint8_t* sfb;
    int* status;
};

__device__ __forceinline__ Hot load_hot(const GemmParams& p) {
    Hot h;
    h.KT = pin(p.KT);
    h.n_max = pin(p.n_max);
    h.stage_bytes = pin(p.stage_bytes);
    h.a_tx_bytes = pin(p.a_tx_bytes);
    h.kseg_tiles = pin(p.kseg_tiles);
    h.b_box = pin(p.b_box);
    h.b_row1 = pin(p.b_row1);
    h.b_producer = pin(p.b_producer);
    h.dense = pin(p.dense);
    h.m_tiles = pin(p.m_tiles);
    h.mt_base = pin(p.mt_base);
    h.n_tokens = pin(p.n_tokens);
    h.a_rows = pin(p.a_rows);
    h.b_rows = pin(p.b_rows);
    h.E = pin(p.E);
    h.mt_per_e = pin(p.mt_per_e);
    h.rows_per_e = pin(p.rows_per_e);
    h.epi_split = pin(p.epi_split);
    h.ax0 = pin(p.a_seg_x[0]);
    h.ax1 = pin(p.a_seg_x[1]);
    h.ax2 = pin(p.a_seg_x[2]);
    h.bx0 = pin(p.b_seg_x[0]);
    h.bx1 = pin(p.b_seg_x[1]);
    h.bx2 = pin(p.b_seg_x[2]);
    h.sfb_pitch = pin(p.sfb_pitch);
    h.sfa = pin(p.sfa);
    h.sfb = pin(p.sfb);
    h.status = pin(p.status);
    return h;
}

__device__ __forceinline__ void pin_epi(EpiParams& e) {
    e.mode = pin(e.mode);
    e.m_tile0 = pin(e.m_tile0);
    e.col0 = pin(e.col0);
    e.f32_split = pin(e.f32_split);
    e.out_f32 = pin(e.out_f32);
    e.ld_f32 = pin(e.ld_f32);
    e.out_q = pin(e.out_q);
    e.ld_q = pin(e.ld_q);
    e.out_sf = pin(e.out_sf);
    e.sf_pitch = pin(e.sf_pitch);
    e.sf_item = pin(e.sf_item);
    e.out_bf16 = pin(e.out_bf16);
}

// Item `it`.  Grouped items come from the per-expert tables staged in shared
// memory (ioff, seg, counts): the expert is found from `e`, the expert of the
// caller's previous item (callers visit their items in increasing order), by
// a short walk forward, else a binary search; then token tile j and weight
// tile m of that expert.
__device__ __forceinline__ Item get_item(const Hot& h, int it, const int* ioff, const int* seg, const int* cnt,
                                         int& e) {
    Item w;
    if (h.dense) {
        const int mt = h.mt_base + it % h.m_tiles;
        const int nt = it / h.m_tiles;
        w.a_row0 = mt * kBlockM;
        w.b_row0 = nt * h.n_max;
        w.n = min(h.n_max, h.n_tokens - w.b_row0);
        w.mt = mt;
    } else {
        int lo = (e < 0 || ioff[e] > it) ? 0 : e;
        for (int step = 0; step < 4 && lo + 1 < h.E && ioff[lo + 1] <= it; ++step) ++lo;
        if (lo + 1 < h.E && ioff[lo + 1] <= it) {
            int hi = h.E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (ioff[mid] <= it) lo = mid;
                else hi = mid - 1;
            }
        }
        e = lo;
        const int local = it - ioff[lo];
        const int j = local / h.mt_per_e, m = local - j * h.mt_per_e;
        w.a_row0 = lo * h.rows_per_e + m * kBlockM;
        w.b_row0 = seg[lo] + j * h.n_max;
        w.n = min(h.n_max, cnt[lo] - j * h.n_max);
        w.mt = m;
        // reject items that would read or write outside the buffers
        if (w.n <= 0 || w.n > h.n_max || w.a_row0 < 0 || (w.a_row0 & (kBlockM - 1)) ||
            w.a_row0 + kBlockM > h.a_rows || w.b_row0 < 0 || (w.b_row0 & 15) ||
            w.b_row0 + ((w.n + 15) & ~15) > h.b_rows || w.mt < 0) {
            w.n = -1;
        }
    }
    return w;
}

struct SmemLayout {
    int offB, offSFA, offSFB;
};

// One stage: A tile, B rows, then the scale atoms of A (512 B) and of B
// (512 B per started 128 tokens), both copied as they sit in global memory.
// A CTA of a pair holds half of the token rows (pair_b_rows).
__host__ __device__ __forceinline__ SmemLayout stage_layout(int n_max, bool pair = false) {
    SmemLayout l;
    l.offB = kABytes;
    l.offSFA = l.offB + (pair ? pair_b_rows(n_max) : n_max) * kBlockK;
    l.offSFB = l.offSFA + 512;
    return l;
}

// K tiles [kb, ke) of an item handled by K-split g of G.
__device__ __forceinline__ void group_range(int KT, int g, int G, int& kb, int& ke) {
    kb = (KT * g) / G;
    ke = (KT * (g + 1)) / G;
}

// Shared memory after the stages: epilogue exchange buffer (2 x 2 warps x
// 32 lanes x 16 floats), then the barriers, then the grouped-item tables.
constexpr int kSplitChunksMin = 32;   // items of this many tokens or more share their chunks among warpgroups
constexpr int kXchgBytes = kEpiGroups * 2 * 2 * 32 * 16 * 4;    // SiLU exchange, per warpgroup: 2 chunks x 2 warps
constexpr int kQStageBytes = 4 * kEpiGroups * 512;              // per epilogue warp: 16 tokens x 32 codes
constexpr int kXbufBytes = kXchgBytes + kQStageBytes;
constexpr int kMaxStagesPerGroup = 16;
// barriers, TMEM slot + abort flag (16 bytes), then the [G][2] item slots
constexpr int kBarBytes = (kMaxGroups * (2 * kMaxStagesPerGroup + 2 * 2 + 1)) * 8 + 16 + kMaxGroups * 2 * 16;
__host__ __device__ __forceinline__ int table_bytes(int E) { return E > 0 ? ((3 * (E + 1) * 4 + 15) & ~15) : 0; }

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// The 128 threads of an epilogue warpgroup agree on `ok` (named barrier
// `bar` with an AND reduction).
__device__ __forceinline__ bool epi_all(bool ok, int bar) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "r"(bar)
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

// Epilogue code compiled into a kernel instance: each launch carries only the
// output paths it can take.
enum EpiSet : int {
    SET_F32 = 0,        // EPI_F32 only
    SET_QUANT = 1,      // EPI_F32 / EPI_QUANT
    SET_SILU = 2,       // EPI_SILU_QUANT only
    SET_DUAL = 3        // EPI_F32 / EPI_QUANT (epi[0]) and EPI_SILU_QUANT (epi[1])
};

template <int KIND, int SET, bool PAIR = false>
__global__ void __launch_bounds__(kGemmMaxThreads, 1) mx_gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr bool kMX = (KIND == KIND_MX);
    constexpr bool kBF16 = (KIND == KIND_BF16);
    constexpr bool kSilu = (SET == SET_SILU || SET == SET_DUAL);
    constexpr bool kQuant = (SET == SET_QUANT || SET == SET_DUAL);
    constexpr bool kOnlySilu = (SET == SET_SILU);
    constexpr int kTileElems = kMX ? kBlockK : (kBF16 ? 64 : 32);   // K elements per 128-byte row of a stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Hot h = load_hot(p);
    const int G = pin(p.groups);
    const int KS = pin(p.ksplit);           // groups per item
    const int IP = G / KS;                  // item lanes
    const int S_all = pin(p.stages);        // stages of all groups; group g has S_all / G (+1 for g < S_all % G)
    const int NB = pin(p.acc_bufs);         // accumulator buffers per group
    const SmemLayout L = stage_layout(h.n_max, PAIR);
    // CTA pairs: this CTA's rank in the pair; the even CTA issues the MMAs
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    constexpr int kXbuf = (kSilu || kQuant) ? kXbufBytes : 0;
    uint8_t* tail = base + S_all * h.stage_bytes;
    float* xbuf = reinterpret_cast<float*>(tail);
    // MXFP8 codes of a chunk are staged per warp, then stored as 16-byte rows
    uint8_t* qstage = tail + kXchgBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(tail + kXbuf);           // [G][kMaxStagesPerGroup]
    uint64_t* empty = full + kMaxGroups * kMaxStagesPerGroup;              // [G][kMaxStagesPerGroup]
    uint64_t* tfull = empty + kMaxGroups * kMaxStagesPerGroup;             // [G][2]
    uint64_t* tempty = tfull + kMaxGroups * 2;                             // [G][2]
    uint64_t* tdown = tempty + kMaxGroups * 2;                             // [G]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tdown + kMaxGroups);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // item handed from each group's MMA warp to the epilogue with its accumulator
    Item* item_slot = reinterpret_cast<Item*>(reinterpret_cast<uint8_t*>(tmem_slot) + 16);    // [G][2]
    int* ioff_s = reinterpret_cast<int*>(tail + kXbuf + kBarBytes);
    int* seg_s = ioff_s + (h.dense ? 0 : h.E + 1);
    int* cnt_s = seg_s + (h.dense ? 0 : h.E + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_trigger();

    if (threadIdx.x == 0) {
        for (int g = 0; g < G; ++g) {
            const int S = S_all / G + (g < S_all % G ? 1 : 0);
            for (int s = 0; s < S; ++s) {
                mbar_init(&full[g * kMaxStagesPerGroup + s], 1);
                mbar_init(&empty[g * kMaxStagesPerGroup + s], 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&tfull[g * 2 + b], 2);      // the MMAs' commit + the item slot
                // released by every epilogue warp that works on the item (in
                // a pair: the even CTA's by the epilogue warps of both CTAs)
                mbar_init(&tempty[g * 2 + b],
                          (PAIR && rank == 0 ? 2 : 1) * (h.n_max >= kSplitChunksMin ? 4 * kEpiGroups : 4));
            }
            mbar_init(&tdown[g], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tmA);
        prefetch_tmap(&p.tmB);
        if (h.b_row1) prefetch_tmap(&p.tmB1);
        if (PAIR) {
            prefetch_tmap(&p.tmSFA);
            prefetch_tmap(&p.tmSFB);
        }
    }
    if (warp == G) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_slot, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    // everything above touches only this CTA's resources; from here on the
    // kernel reads and writes buffers of earlier kernels
    pdl_wait();
    if (!h.dense) {
        for (int i = threadIdx.x; i <= h.E; i += blockDim.x) {
            ioff_s[i] = p.ioff[i];
            seg_s[i] = p.seg[i];
            cnt_s[i] = (i < h.E) ? p.counts[i] : 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    // a pair's barriers are initialised before either CTA signals the other's
    if constexpr (PAIR) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // pairs: item i of the launch is engine item 2i + rank of this CTA
    const int n_items_all = h.dense ? h.m_tiles * ((h.n_tokens + h.n_max - 1) / h.n_max) : ioff_s[h.E];
    const int n_items = PAIR ? (n_items_all >> 1) : n_items_all;
    const int cta = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int n_cta = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    // this CTA's items: it_begin + c * it_step for c = 0, 1, ... while below
    // it_end -- a contiguous range (narrow items: consecutive items mostly
    // share an expert), or every n_cta-th item
    const bool contiguous = p.contiguous != 0;
    const int it_begin = contiguous ? static_cast<int>(static_cast<int64_t>(n_items) * cta / n_cta) : cta;
    const int it_end = contiguous ? static_cast<int>(static_cast<int64_t>(n_items) * (cta + 1) / n_cta) : n_items;
    const int it_step = contiguous ? 1 : n_cta;
    const uint32_t cols_per_group = static_cast<uint32_t>(NB * h.n_max + 24);

    if (warp < G) {
        // ------------------------------------------------------------ producer of group g
        // The whole warp runs the loop; one elected lane issues the copies.
        const int g = warp;
        const int ip = g / KS;
        int kb, ke;
        group_range(h.KT, g % KS, KS, kb, ke);
        // a single-lane pair streams its K tiles as two rings: this producer
        // the first half of the stages and K tiles, the second producer warp
        // the rest (one CTA streams a ring at about one stage per 340 ns,
        // two rings about twice that)
        const bool dual = PAIR && h.b_producer;
        if (dual) ke = (h.KT + 1) / 2;
        uint64_t* fullg = full + g * kMaxStagesPerGroup;
        uint64_t* emptyg = empty + g * kMaxStagesPerGroup;
        const int S = dual ? (S_all + 1) / 2 : S_all / G + (g < S_all % G ? 1 : 0);
        uint8_t* ring = base + (g * (S_all / G) + min(g, S_all % G)) * h.stage_bytes;
        uint32_t stage = 0, phase = 0;
        uint32_t issued = 0, issued_parity = 0;   // per-stage bits for the teardown drain
        bool ok = true;
        int ecur = -1;
        for (int it = it_begin + ip * it_step; ok && it < it_end && ke > kb; it += IP * it_step) {
            const Item w = get_item(h, PAIR ? 2 * it + rank : it, ioff_s, seg_s, cnt_s, ecur);
            if (w.n <= 0) {
                if (w.n < 0 && g == 0 && lane == 0) atomicCAS(h.status, 0, DEV_BAD_WORK);
                continue;
            }
            const int nm = (w.n + 15) & ~15;
            const int natoms = (nm + 127) / 128;
            const int nbox = (nm + h.b_box - 1) / h.b_box;           // B boxes of b_box rows
            // an item of fewer than 16 tokens loads only its own token rows
            // (one-row boxes) and, up to 32 tokens, only its own scale slots:
            // the MMA still reads 16 rows, and the accumulator columns of the
            // rows left as they were are never stored
            const bool row_loads = kMX && h.b_row1 && w.n < 16;
            const uint32_t b_bytes = row_loads ? static_cast<uint32_t>(w.n * kBlockK)
                                               : static_cast<uint32_t>(nbox * h.b_box * kBlockK);
            const uint32_t sfb_bytes = (w.n <= 32) ? static_cast<uint32_t>(w.n * 16) : static_cast<uint32_t>(natoms * 512);
            // a pair's stage: both CTAs' weight tiles and scale atoms, and
            // one box of token rows and one of token scales per CTA (the even
            // CTA counts them all on its barrier)
            const uint32_t tx = PAIR ? 2u * (static_cast<uint32_t>(h.a_tx_bytes) + 512u +
                                             static_cast<uint32_t>(((h.n_max + 127) / 128) * 512 + h.b_box * kBlockK))
                              : kMX ? static_cast<uint32_t>(h.a_tx_bytes) + b_bytes + 512u + sfb_bytes
                                    : static_cast<uint32_t>(kBlockM * 128) + b_bytes;
            const uint8_t* sfa_tile = kMX ? h.sfa + static_cast<size_t>(w.a_row0 / kBlockM) * h.KT * 512 : nullptr;
            for (int kt = kb; kt < ke; ++kt) {
                ok = mbar_wait(&emptyg[stage], phase ^ 1, abort_flag, h.status, DEV_TIMEOUT_PRODUCER);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const int sg = kt / h.kseg_tiles;
                const int kin = (kt - sg * h.kseg_tiles) * kTileElems;
                const int ax = (sg == 0 ? h.ax0 : (sg == 1 ? h.ax1 : h.ax2)) + kin;
                const int bx = (sg == 0 ? h.bx0 : (sg == 1 ? h.bx1 : h.bx2)) + kin;
                uint8_t* sb = ring + stage * h.stage_bytes;
                if constexpr (PAIR) {
                    if (elect_one()) {
                        const uint32_t fb = mapa_shared(smem_u32(&fullg[stage]), 0);
                        // the even CTA counts the pair's bytes on its own barrier
                        // (a CTA-local arrive: the cluster-scope form costs about a
                        // microsecond per stage)
                        if (rank == 0) mbar_arrive_expect_tx(&fullg[stage], tx);
                        tma_load_2d_pair(sb, &p.tmA, fb, ax, w.a_row0);
                        tma_load_2d_pair(sb + L.offSFA, &p.tmSFA, fb, 0, ((w.a_row0 / kBlockM) * h.KT + kt) * 2);
                        // this CTA's half of the token rows, and all of their scales
                        tma_load_2d_pair(sb + L.offB, &p.tmB, fb, bx, w.b_row0 + rank * (nm >> 1));
                        tma_load_2d_pair(sb + L.offSFB, &p.tmSFB, fb, 0,
                                         (static_cast<int>(kt * h.sfb_pitch) + w.b_row0) >> 4);
                    }
                } else if (elect_one()) {
                    mbar_arrive_expect_tx(&fullg[stage], tx);
                    tma_load_2d(sb, &p.tmA, &fullg[stage], ax, w.a_row0);
                    if (!h.b_producer) {
                        if (row_loads) {
                            for (int r = 0; r < w.n; ++r)
                                tma_load_2d(sb + L.offB + r * kBlockK, &p.tmB1, &fullg[stage], bx, w.b_row0 + r);
                        } else {
                            for (int c = 0; c < nbox; ++c)
                                tma_load_2d(sb + L.offB + c * h.b_box * kBlockK, &p.tmB, &fullg[stage], bx,
                                            w.b_row0 + c * h.b_box);
                        }
                    }
                    if constexpr (kMX) {
                        bulk_load(sb + L.offSFA, sfa_tile + static_cast<size_t>(kt) * 512, 512, &fullg[stage]);
                        if (!h.b_producer)
                            bulk_load(sb + L.offSFB, h.sfb + (static_cast<size_t>(kt) * h.sfb_pitch + w.b_row0) * 16,
                                      sfb_bytes, &fullg[stage]);
                    }
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if constexpr (PAIR) {
            // the even CTA's MMAs read this CTA's stages and their commits
            // arrive on its barriers: before this CTA may exit, every stage
            // must have been released
            for (int i = 0; ok && i < S; ++i) {
                ok = mbar_wait(&emptyg[stage], phase ^ 1, abort_flag, h.status, DEV_TIMEOUT_PRODUCER);
                ok = __all_sync(0xffffffffu, ok);
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (*abort_flag && lane == 0 && rank == 0) {
            // drain: every issued stage's copies must land before exit (a
            // pair's copies all count on the even CTA's barriers)
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) mbar_wait_teardown(&fullg[s], (issued_parity >> s) & 1u, h.status);
        }
        __syncwarp();
    } else if (warp < 2 * G) {
        // ------------------------------------------------------------ MMA issuer of group g
        const int g = warp - G;
        const int ip = g / KS;
        int kb, ke;
        group_range(h.KT, g % KS, KS, kb, ke);
        uint64_t* fullg = full + g * kMaxStagesPerGroup;
        uint64_t* emptyg = empty + g * kMaxStagesPerGroup;
        const int S = S_all / G + (g < S_all % G ? 1 : 0);
        uint8_t* ring = base + (g * (S_all / G) + min(g, S_all % G)) * h.stage_bytes;
        const uint32_t gcol = tmem + static_cast<uint32_t>(g) * cols_per_group;
        const uint32_t sf_base = gcol + static_cast<uint32_t>(NB * h.n_max);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        // paired launches: stage and phase of each ring (ring 1: single lane only)
        const int pS0 = (PAIR && h.b_producer) ? (S + 1) / 2 : S, pS1 = S - pS0;
        uint32_t pst0 = 0, pph0 = 0, pst1 = 0, pph1 = 0;
        uint32_t pused = 0;                   // stages consumed so far: the scale columns rotate
        // scale-column sets of a paired launch (minus one): 4 where the
        // group's columns leave room, else 2
        const uint32_t psets = (PAIR && h.b_producer && NB * h.n_max + 4 * 12 <= kTmemCols) ? 3u : 1u;
        // shared-memory descriptors of stage 0 of this group's ring
        const uint64_t pdA = PAIR ? sdesc_sw128(smem_u32(ring)) : 0, pdB = PAIR ? sdesc_sw128(smem_u32(ring + L.offB)) : 0;
        const uint64_t pdSA = PAIR ? sdesc_rows16(smem_u32(ring + L.offSFA)) : 0,
                       pdSB = PAIR ? sdesc_rows16(smem_u32(ring + L.offSFB)) : 0;
        bool any = false;
        int ecur = -1;
        for (int it = it_begin + ip * it_step; it < it_end && ke > kb; it += IP * it_step) {
            // every item takes an accumulator turn, so that the epilogue can
            // follow the item lanes round-robin; a rejected item (n <= 0)
            // issues no MMAs.  In a pair the even CTA issues the MMAs of both
            // (its accumulator buffer is free once both epilogues released
            // it); the odd CTA only hands its item to its epilogue.
            const Item w = get_item(h, PAIR ? 2 * it + rank : it, ioff_s, seg_s, cnt_s, ecur);
            const int nm = (w.n + 15) & ~15;
            const int natoms = (nm + 127) / 128;
            bool ok = mbar_wait(&tempty[g * 2 + acc], acc_phase ^ 1, abort_flag, h.status, DEV_TIMEOUT_MMA);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t d_tmem = gcol + acc * static_cast<uint32_t>(h.n_max);
            if constexpr (PAIR) {
                // one ring per lane, or (single lane) two rings taken in turn:
                // K tiles 0, KT0, 1, KT0 + 1, ... -- a fixed order
                const bool dual = h.b_producer != 0;
                const int KT0 = dual ? (h.KT + 1) / 2 : h.KT, KT1 = h.KT - KT0;
                const uint32_t idesc0 = idesc_mxf8f6f4(2 * kBlockM, nm, 5, 0, 0, 0);
                for (int v = 0; v < ((w.n > 0 && rank == 0) ? h.KT : 0); ++v) {
                    const bool r1 = (v < 2 * KT1) && (v & 1);      // the v-th stage is ring 1's
                    const uint32_t si = r1 ? pS0 + pst1 : pst0;      // its stage index
                    // a stage that is already full is seen so by every lane at
                    // once: the warp-wide vote only on the waiting path
                    if (!mbar_try_wait(&fullg[si], r1 ? pph1 : pph0)) {
                        ok = mbar_wait(&fullg[si], r1 ? pph1 : pph0, abort_flag, h.status, DEV_TIMEOUT_MMA);
                        if (!__all_sync(0xffffffffu, ok)) goto mma_done;
                    }
                    // the stage barrier orders the copies' writes before the
                    // MMAs' reads (both async proxy): no tcgen05 fence per stage.
                    // Descriptors of stage si: stage 0's plus its offset (the
                    // start-address field counts 16-byte units)
                    const uint64_t soff = static_cast<uint64_t>(si) * (static_cast<uint32_t>(h.stage_bytes) >> 4);
                    const uint64_t adesc = pdA + soff, bdesc = pdB + soff;
                    // consecutive stages (across items too) use different scale columns
                    const uint32_t sfa_col = sf_base + (pused++ & psets) * 12u;
                    const uint32_t sfb_col = sfa_col + 4u;
                    if (elect_one()) {
                        tc_cp_32x128b_x4_pair(sfa_col, pdSA + soff);
                        for (int a = 0; a < natoms; ++a)
                            tc_cp_32x128b_x4_pair(sfb_col + 4u * a, pdSB + soff + static_cast<uint64_t>(a * (512 >> 4)));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t idesc = idesc0 | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
                            mma_mxf8f6f4_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col, sfb_col,
                                              (v | j) != 0 ? 1u : 0u);
                        }
                        tc_commit_pair(&emptyg[si], 3);
                    }
                    any = true;
                    if (r1) {
                        if (++pst1 == static_cast<uint32_t>(pS1)) {
                            pst1 = 0;
                            pph1 ^= 1;
                        }
                    } else if (++pst0 == static_cast<uint32_t>(pS0)) {
                        pst0 = 0;
                        pph0 ^= 1;
                    }
                }
            } else
            for (int kt = kb; kt < ((w.n > 0 && rank == 0) ? ke : kb); ++kt) {
                ok = mbar_wait(&fullg[stage], phase, abort_flag, h.status, DEV_TIMEOUT_MMA);
                if (!__all_sync(0xffffffffu, ok)) goto mma_done;
                tc_fence_after();
                {
                    uint8_t* sb = ring + stage * h.stage_bytes;
                    const uint32_t accum_first = (kt == kb) ? 0u : 1u;
                    const uint64_t adesc = sdesc_sw128(smem_u32(sb));
                    const uint64_t bdesc = sdesc_sw128(smem_u32(sb + L.offB));
                    if constexpr (kBF16) {
                        const uint32_t idesc = idesc_bf16(kBlockM, nm);
                        if (elect_one()) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                mma_bf16(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (accum_first | j) != 0 ? 1u : 0u);
                            tc_commit(&emptyg[stage]);
                        }
                    } else if constexpr (!kMX) {
                        const uint32_t idesc = idesc_tf32(kBlockM, nm);
                        if (elect_one()) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                mma_tf32(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (accum_first | j) != 0 ? 1u : 0u);
                            tc_commit(&emptyg[stage]);
                        }
                    } else {
                        // both scale operands arrive as 32x128b copy images
                        const uint32_t sfa_col = sf_base + static_cast<uint32_t>(kt & 1) * 12u;
                        const uint32_t sfb_col = sfa_col + 4u;
                        {
                        const uint32_t idesc0 = idesc_mxf8f6f4(kBlockM, nm, 5, 0, 0, 0);
                        if (elect_one()) {
                            tc_cp_32x128b_x4(sfa_col, sdesc_rows16(smem_u32(sb + L.offSFA)));
                            for (int a = 0; a < natoms; ++a)
                                tc_cp_32x128b_x4(sfb_col + 4u * a, sdesc_rows16(smem_u32(sb + L.offSFB + a * 512)));
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                // scale-factor ids (byte j of each 32-bit scale column) sit
                                // at bits 4..5 (B) and 29..30 (A) of the instruction descriptor
                                const uint32_t idesc = idesc0 | (static_cast<uint32_t>(j) << 4) |
                                                       (static_cast<uint32_t>(j) << 29);
                                mma_mxf8f6f4(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col, sfb_col,
                                             (accum_first | j) != 0 ? 1u : 0u);
                            }
                            tc_commit(&emptyg[stage]);
                        }
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
            if (elect_one()) {
                item_slot[g * 2 + acc] = w;
                mbar_arrive(&tfull[g * 2 + acc]);      // release: the slot is visible with the phase
                if constexpr (PAIR) {
                    if (rank == 0) tc_commit_pair(&tfull[g * 2 + acc], 3);
                } else {
                    tc_commit(&tfull[g * 2 + acc]);
                }
            }
            __syncwarp();
            if (++acc == static_cast<uint32_t>(NB)) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    mma_done:
        // every tcgen05 operation issued above must finish before TMEM is freed
        if (any) {
            if (elect_one()) {
                if constexpr (PAIR)
                    tc_commit_pair(&tdown[g], 1);
                else
                    tc_commit(&tdown[g]);
                mbar_wait_teardown(&tdown[g], 0, h.status);
            }
            __syncwarp();
        }
    } else if (warp < 2 * G + 4 * kEpiGroups) {
        // ------------------------------------------------------------ epilogue
        // kEpiGroups warpgroups take the CTA's items in turn; the four warps of
        // a warpgroup cover the four TMEM lane quarters of an accumulator
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int wg = (warp - 2 * G) >> 2;
        const int bar_agree = 1 + 2 * wg, bar_xchg = 2 + 2 * wg;     // named barriers of this warpgroup
        const uint32_t t_lane = static_cast<uint32_t>(32 * q) << 16;
        // both output descriptions in registers; an item selects scalars
        EpiParams E0 = p.epi[0];
        EpiParams E1 = p.epi[1];
        pin_epi(E0);
        pin_epi(E1);
        int chunk_parity = 0;
        const int n_mine = (it_end > it_begin) ? (it_end - it_begin + it_step - 1) / it_step : 0;
        const int ip_shift = (IP == 4) ? 2 : (IP == 2 ? 1 : 0);       // IP is 1, 2 or 4
        // items of several chunks: every warpgroup takes every item, and its
        // 16-token chunks in turn; single-chunk items: warpgroups take the
        // items in turn
        const bool split_chunks = h.n_max >= kSplitChunksMin;
        const int c_first = split_chunks ? 0 : wg, c_step = split_chunks ? 1 : kEpiGroups;
        const int n_first = split_chunks ? 16 * wg : 0, n_step = split_chunks ? 16 * kEpiGroups : 16;
        for (int c = c_first; c < n_mine; c += c_step) {
            // item c: item lane c % IP, that lane's (c / IP)-th accumulator turn
            const int ip = c & (IP - 1);
            const uint32_t turn = static_cast<uint32_t>(c >> ip_shift);
            const uint32_t acc = (NB == 2) ? (turn & 1u) : 0u;
            const uint32_t acc_phase = (NB == 2) ? ((turn >> 1) & 1u) : (turn & 1u);
            const int g0 = ip * KS;
            bool ok = true;
            for (int ks = 0; ks < KS; ++ks) {
                int kb, ke;
                group_range(h.KT, ks, KS, kb, ke);
                if (ke > kb && ok)
                    ok = mbar_wait(&tfull[(g0 + ks) * 2 + acc], acc_phase, abort_flag, h.status, DEV_TIMEOUT_EPILOGUE);
            }
            // the SiLU exchange synchronises the four warps, so there all of
            // them must leave together; elsewhere each warp decides alone
            // (every wait is bounded, and a failure raises the abort flag)
            if (kSilu ? !epi_all(ok && !*abort_flag, bar_agree) : !__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            tc_fence_after();
            const Item w = item_slot[g0 * 2 + acc];
            const int nm = (w.n > 0) ? ((w.n + 15) & ~15) : 0;
            const bool second = h.dense && w.mt >= h.epi_split;
            EpiParams E;
            E.mode = second ? E1.mode : E0.mode;
            E.m_tile0 = second ? E1.m_tile0 : E0.m_tile0;
            E.col0 = second ? E1.col0 : E0.col0;
            E.f32_split = second ? E1.f32_split : E0.f32_split;
            E.out_f32 = second ? E1.out_f32 : E0.out_f32;
            E.ld_f32 = second ? E1.ld_f32 : E0.ld_f32;
            E.out_q = second ? E1.out_q : E0.out_q;
            E.ld_q = second ? E1.ld_q : E0.ld_q;
            E.out_sf = second ? E1.out_sf : E0.out_sf;
            E.sf_pitch = second ? E1.sf_pitch : E0.sf_pitch;
            E.sf_item = second ? E1.sf_item : E0.sf_item;
            E.out_bf16 = second ? E1.out_bf16 : E0.out_bf16;
            const int rel_mt = w.mt - E.m_tile0;
            bool stored = false;
            if constexpr (SET == SET_F32) {
              if (KS == 1 && !E.out_bf16 && E.f32_split == 0) {
                stored = true;
                // fp32 output of one accumulator: the next chunk's TMEM load is
                // in flight while this chunk is stored
                const uint32_t a0 = tmem + t_lane + static_cast<uint32_t>(g0) * cols_per_group +
                                    acc * static_cast<uint32_t>(h.n_max);
                const int64_t col = E.col0 + static_cast<int64_t>(rel_mt) * 128 + 32 * q + lane;
                uint32_t cur[16], nxt[16];
                if (n_first < nm) {
                    tmem_ld16_async(a0 + static_cast<uint32_t>(n_first), cur);
                    tmem_wait16(cur);
                }
                for (int n0 = n_first; n0 < nm; n0 += n_step) {
                    const bool more = n0 + n_step < nm;
                    if (more) tmem_ld16_async(a0 + static_cast<uint32_t>(n0 + n_step), nxt);
                    const int nv = min(16, w.n - n0);
                    float* o = E.out_f32 + (w.b_row0 + n0) * E.ld_f32 + col;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (i >= nv) break;
                        o[0] = __uint_as_float(cur[i]);
                        o += E.ld_f32;
                    }
                    if (more) {
                        tmem_wait16(nxt);
#pragma unroll
                        for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
                    }
                }
              }
            }
            for (int n0 = n_first; n0 < (stored ? n_first : nm); n0 += n_step) {
                // sum of the K-split partial accumulators, in group order
                float v[16];
                bool first = true;
                for (int ks = 0; ks < KS; ++ks) {
                    int kb, ke;
                    group_range(h.KT, ks, KS, kb, ke);
                    if (ke <= kb) continue;
                    float u[16];
                    tmem_ld16(tmem + t_lane + static_cast<uint32_t>(g0 + ks) * cols_per_group +
                                  acc * static_cast<uint32_t>(h.n_max) + static_cast<uint32_t>(n0),
                              u);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = first ? u[i] : v[i] + u[i];
                    first = false;
                }
                if (kOnlySilu || (kSilu && (E.mode == EPI_SILU_QUANT || E.mode == EPI_SILU_BF16))) {
                    // rows 0..63 of the tile are gate, 64..127 up: warp q < 2 holds
                    // the gate of feature block q, warp q + 2 its up.  The pair
                    // swaps halves of the chunk through shared memory, then warp
                    // q < 2 finishes tokens 0..7 of block q and warp q + 2 tokens
                    // 8..15: all four warps gate and quantise.
                    float* xb = xbuf + (wg * 2 + chunk_parity) * (2 * 32 * 16);     // [block][token][lane]
                    chunk_parity ^= 1;
                    const int blk = q & 1;
                    const bool gate_warp = q < 2;
                    const int t0 = gate_warp ? 0 : 8;            // tokens this warp finishes
#pragma unroll
                    for (int i = 0; i < 8; ++i)                  // hand over the other half
                        xb[blk * 512 + ((gate_warp ? 8 : 0) + i) * 32 + lane] = gate_warp ? v[8 + i] : v[i];
                    named_bar_sync(bar_xchg, 128);
                    const int64_t col_blk = E.col0 + static_cast<int64_t>(rel_mt) * 64 + 32 * blk;
                    const int nv = min(8, w.n - n0 - t0);
                    if (E.mode == EPI_SILU_BF16) {
                        // bf16 activation (mixed precision): one value per lane and token
                        __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(E.out_q) +
                                            (w.b_row0 + n0 + t0) * E.ld_q + col_blk + lane;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            if (i >= nv) break;
                            const float mine = gate_warp ? v[i] : v[8 + i];
                            const float other = xb[blk * 512 + (t0 + i) * 32 + lane];
                            const float hv = gate_warp ? silu_f(mine) * other : silu_f(other) * mine;
                            ob[0] = __float2bfloat16_rn(hv);
                            ob += E.ld_q;
                        }
                        __syncwarp();
                        continue;
                    }
                    uint8_t* stg = qstage + (warp - 2 * G) * 512;            // [token][32 codes]
                    uint8_t my_sc = 0;                                       // lane i: scale of token i
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (i >= nv) break;
                        const float mine = gate_warp ? v[i] : v[8 + i];
                        const float other = xb[blk * 512 + (t0 + i) * 32 + lane];
                        const float hv = gate_warp ? silu_f(mine) * other : silu_f(other) * mine;
                        uint8_t sc;
                        stg[i * 32 + lane] = warp_mx8_quant(hv, &sc);
                        if (lane == i) my_sc = sc;
                    }
                    __syncwarp();
                    const int64_t row0 = w.b_row0 + n0 + t0;
                    if (lane < 2 * nv) {
                        const int i = lane >> 1, hf = lane & 1;
                        *reinterpret_cast<uint4*>(E.out_q + (row0 + i) * E.ld_q + col_blk + 16 * hf) =
                            *reinterpret_cast<const uint4*>(stg + i * 32 + 16 * hf);
                    }
                    if (lane < nv)
                        E.out_sf[E.sf_item ? sf_atom_offset(w.b_row0, n0 + t0 + lane, col_blk, E.sf_pitch)
                                           : sf_byte_offset(row0 + lane, col_blk, E.sf_pitch)] = my_sc;
                    __syncwarp();
                } else {
                    const int64_t col = E.col0 + static_cast<int64_t>(rel_mt) * 128 + 32 * q + lane;
                    const int nv = min(16, w.n - n0);                 // valid tokens of this chunk
                    const int64_t row0 = w.b_row0 + n0;
                    if (!kQuant || E.mode != EPI_QUANT) {
                        // fp32 (or bf16) only: one store per valid token through a running pointer
                        float* o = E.out_f32 + row0 * E.ld_f32 + col;
                        if (E.out_bf16) {
                            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(E.out_f32) + row0 * E.ld_f32 + col;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (i >= nv) break;
                                ob[0] = __float2bfloat16_rn(v[i]);
                                ob += E.ld_f32;
                            }
                        } else if (E.f32_split) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (i >= nv) break;
                                o[0] = tf32_round(v[i]);
                                o[E.f32_split] = v[i];
                                o += E.ld_f32;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (i >= nv) break;
                                o[0] = v[i];
                                o += E.ld_f32;
                            }
                        }
                    } else {
                        uint8_t* stg = qstage + (warp - 2 * G) * 512;        // [token][32 codes]
                        uint8_t my_sc = 0;                                   // lane i: scale of token i
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (i >= nv) break;
                            const int64_t row = row0 + i;
                            if (E.out_f32) {
                                if (E.f32_split) {
                                    E.out_f32[row * E.ld_f32 + col] = tf32_round(v[i]);
                                    E.out_f32[row * E.ld_f32 + col + E.f32_split] = v[i];
                                } else {
                                    E.out_f32[row * E.ld_f32 + col] = v[i];
                                }
                            }
                            uint8_t sc;
                            stg[i * 32 + lane] = warp_mx8_quant(v[i], &sc);
                            if (lane == i) my_sc = sc;
                        }
                        __syncwarp();
                        const int64_t col_blk = col - lane;
                        if (lane < 2 * nv) {
                            const int i = lane >> 1, hf = lane & 1;
                            *reinterpret_cast<uint4*>(E.out_q + (row0 + i) * E.ld_q + col_blk + 16 * hf) =
                                *reinterpret_cast<const uint4*>(stg + i * 32 + 16 * hf);
                        }
                        if (lane < nv)
                            E.out_sf[E.sf_item ? sf_atom_offset(w.b_row0, n0 + lane, col_blk, E.sf_pitch)
                                               : sf_byte_offset(row0 + lane, col_blk, E.sf_pitch)] = my_sc;
                        __syncwarp();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                for (int ks = 0; ks < KS; ++ks) {
                    int kb, ke;
                    group_range(h.KT, ks, KS, kb, ke);
                    if (ke > kb) mbar_arrive(&tempty[(g0 + ks) * 2 + acc]);
                }
                // the even CTA of a pair refills both CTAs' accumulators (this
                // warp's TMEM loads are complete: tcgen05.wait::ld)
                if (PAIR && rank == 1) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tempty[g0 * 2 + acc]), 0));
            }
        }
    } else if (PAIR && h.b_producer && warp == 2 * G + 4 * kEpiGroups) {
        // ------------------------------------------------------------ second ring of a single-lane pair
        // The second half of every item's K tiles through the second half of
        // the stages: weight tile, token half and all scales, counted on the
        // even CTA's stage barrier like producer 0's.
        const int S0 = (S_all + 1) / 2, S = S_all - S0;
        const int KT0 = (h.KT + 1) / 2;
        uint64_t* fullr = full + S0;
        uint64_t* emptyr = empty + S0;
        uint8_t* ringr = base + S0 * h.stage_bytes;
        uint32_t stage = 0, phase = 0;
        uint32_t issued = 0, issued_parity = 0;
        bool ok = true;
        int ecur = -1;
        const uint32_t tx = 2u * (static_cast<uint32_t>(h.a_tx_bytes) + 512u +
                                  static_cast<uint32_t>(((h.n_max + 127) / 128) * 512 + h.b_box * kBlockK));
        for (int it = it_begin; ok && S > 0 && it < it_end; it += it_step) {
            const Item w = get_item(h, 2 * it + rank, ioff_s, seg_s, cnt_s, ecur);
            if (w.n <= 0) continue;
            const int nm = (w.n + 15) & ~15;
            for (int kt = KT0; kt < h.KT; ++kt) {
                ok = mbar_wait(&emptyr[stage], phase ^ 1, abort_flag, h.status, DEV_TIMEOUT_PRODUCER);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const int sg = kt / h.kseg_tiles;
                const int kin = (kt - sg * h.kseg_tiles) * kTileElems;
                const int ax = (sg == 0 ? h.ax0 : (sg == 1 ? h.ax1 : h.ax2)) + kin;
                const int bx = (sg == 0 ? h.bx0 : (sg == 1 ? h.bx1 : h.bx2)) + kin;
                uint8_t* sb = ringr + stage * h.stage_bytes;
                if (elect_one()) {
                    const uint32_t fb = mapa_shared(smem_u32(&fullr[stage]), 0);
                    if (rank == 0) mbar_arrive_expect_tx(&fullr[stage], tx);
                    tma_load_2d_pair(sb, &p.tmA, fb, ax, w.a_row0);
                    tma_load_2d_pair(sb + L.offSFA, &p.tmSFA, fb, 0, ((w.a_row0 / kBlockM) * h.KT + kt) * 2);
                    tma_load_2d_pair(sb + L.offB, &p.tmB, fb, bx, w.b_row0 + rank * (nm >> 1));
                    tma_load_2d_pair(sb + L.offSFB, &p.tmSFB, fb, 0,
                                     (static_cast<int>(kt * h.sfb_pitch) + w.b_row0) >> 4);
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // the even CTA's MMAs read this CTA's stages and their commits arrive
        // on its barriers: before this CTA may exit, every stage must have
        // been released
        for (int i = 0; ok && i < S; ++i) {
            ok = mbar_wait(&emptyr[stage], phase ^ 1, abort_flag, h.status, DEV_TIMEOUT_PRODUCER);
            ok = __all_sync(0xffffffffu, ok);
            if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (*abort_flag && lane == 0 && rank == 0) {
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) mbar_wait_teardown(&fullr[s], (issued_parity >> s) & 1u, h.status);
        }
        __syncwarp();
    } else if (!PAIR && h.b_producer && warp == 2 * G + 4 * kEpiGroups) {
        // ------------------------------------------------------------ token-side producer (groups == 1)
        // Follows producer 0 stage by stage: the same items and K tiles, the
        // same free stages; it issues the token rows and their scales, whose
        // bytes producer 0 has counted on the stage barrier (or is about to:
        // a barrier's byte count may dip below zero meanwhile, and the phase
        // cannot complete before producer 0 has arrived).
        const int S = S_all;
        uint32_t stage = 0, phase = 0;
        uint32_t issued = 0, issued_parity = 0;
        bool ok = true;
        int ecur = -1;
        for (int it = it_begin; ok && it < it_end; it += it_step) {
            const Item w = get_item(h, it, ioff_s, seg_s, cnt_s, ecur);
            if (w.n <= 0) continue;
            const int nm = (w.n + 15) & ~15;
            const int natoms = (nm + 127) / 128;
            const int nbox = (nm + h.b_box - 1) / h.b_box;
            const bool row_loads = kMX && h.b_row1 && w.n < 16;
            const uint32_t sfb_bytes = (w.n <= 32) ? static_cast<uint32_t>(w.n * 16) : static_cast<uint32_t>(natoms * 512);
            for (int kt = 0; kt < h.KT; ++kt) {
                ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, h.status, DEV_TIMEOUT_PRODUCER);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                const int sg = kt / h.kseg_tiles;
                const int kin = (kt - sg * h.kseg_tiles) * kTileElems;
                const int bx = (sg == 0 ? h.bx0 : (sg == 1 ? h.bx1 : h.bx2)) + kin;
                uint8_t* sb = base + stage * h.stage_bytes;
                if (elect_one()) {
                    if (row_loads) {
                        for (int r = 0; r < w.n; ++r)
                            tma_load_2d(sb + L.offB + r * kBlockK, &p.tmB1, &full[stage], bx, w.b_row0 + r);
                    } else {
                        for (int c = 0; c < nbox; ++c)
                            tma_load_2d(sb + L.offB + c * h.b_box * kBlockK, &p.tmB, &full[stage], bx,
                                        w.b_row0 + c * h.b_box);
                    }
                    if constexpr (kMX)
                        bulk_load(sb + L.offSFB, h.sfb + (static_cast<size_t>(kt) * h.sfb_pitch + w.b_row0) * 16,
                                  sfb_bytes, &full[stage]);
                }
                __syncwarp();
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == static_cast<uint32_t>(S)) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (*abort_flag && lane == 0) {
            for (int s = 0; s < S; ++s)
                if (issued & (1u << s)) mbar_wait_teardown(&full[s], (issued_parity >> s) & 1u, h.status);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA of a pair frees the pair's TMEM or leaves while the other
    // may still signal its barriers
    if constexpr (PAIR) cluster_sync_all();
    if (warp == G) {
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem, kTmemCols);
        else
            tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int gemm_stage_bytes(int n_max, bool pair) {
    const SmemLayout l = stage_layout(n_max, pair);
    const int bytes = l.offSFB + ((n_max + 127) / 128) * 512;
    return (bytes + 1023) & ~1023;
}

size_t gemm_smem_bytes(int n_max, int stages, int E, bool xbuf, bool pair) {
    return 1024 + static_cast<size_t>(stages) * gemm_stage_bytes(n_max, pair) + (xbuf ? kXbufBytes : 0) + kBarBytes +
           table_bytes(E);
}

int gemm_stages(int n_max, int groups, int E, bool xbuf, bool pair) {
    int s = kMaxStagesPerGroup * groups;
    while (s > 2 * groups && gemm_smem_bytes(n_max, s, E, xbuf, pair) > static_cast<size_t>(kSmemLimit)) --s;
    return s;
}


bool gemm_config_ok(int n_max, int groups, int ksplit, int acc_bufs) {
    if (groups < 1 || groups > kMaxGroups || acc_bufs < 1 || acc_bufs > 2) return false;
    if (ksplit < 1 || groups % ksplit) return false;
    if (n_max < 16 || n_max > kNMax || (n_max & 15)) return false;
    return groups * (acc_bufs * n_max + 24) <= kTmemCols;
}

namespace {

template <int KIND, int SET, bool PAIR = false>
cudaError_t raise_smem() {
    return cudaFuncSetAttribute(mx_gemm_kernel<KIND, SET, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemLimit);
}

// The kernel instance whose epilogue covers the launch's output modes: those
// of epi[0] (weight tiles below epi_split) and epi[1] (from epi_split on)
// that the launch's tiles use.
int epi_set(const GemmParams& p) {
    const bool use0 = !p.dense || p.epi_split > p.mt_base;
    const bool use1 = p.dense && p.epi_split < p.mt_base + p.m_tiles;
    const int m0 = p.epi[0].mode, m1 = p.epi[1].mode;
    const bool silu0 = m0 == EPI_SILU_QUANT || m0 == EPI_SILU_BF16, silu1 = m1 == EPI_SILU_QUANT || m1 == EPI_SILU_BF16;
    const bool s0 = use0 && silu0, s1 = use1 && silu1;          // SiLU outputs in use
    const bool n0 = use0 && !silu0, n1 = use1 && !silu1;        // other outputs in use
    if (!s0 && !s1) return ((n0 && m0 == EPI_QUANT) || (n1 && m1 == EPI_QUANT)) ? SET_QUANT : SET_F32;
    if (!n0 && !n1) return SET_SILU;
    if (s1 && n0 && !s0 && !n1) return SET_DUAL;
    return -1;
}

}  // namespace

bool gemm_needs_xbuf(const GemmParams& p) {
    const int set = epi_set(p);
    return set == SET_SILU || set == SET_DUAL || set == SET_QUANT;
}

cudaError_t gemm_setup() {
    cudaError_t err = raise_smem<KIND_MX, SET_F32>();
    if (err == cudaSuccess) err = raise_smem<KIND_MX, SET_QUANT>();
    if (err == cudaSuccess) err = raise_smem<KIND_MX, SET_SILU>();
    if (err == cudaSuccess) err = raise_smem<KIND_MX, SET_DUAL>();
    if (err == cudaSuccess) err = raise_smem<KIND_TF32, SET_F32>();
    if (err == cudaSuccess) err = raise_smem<KIND_BF16, SET_F32>();
    if (err == cudaSuccess) err = raise_smem<KIND_BF16, SET_DUAL>();
    if (err == cudaSuccess) err = raise_smem<KIND_MX, SET_F32, true>();
    if (err == cudaSuccess) err = raise_smem<KIND_MX, SET_QUANT, true>();
    if (err == cudaSuccess) err = raise_smem<KIND_MX, SET_SILU, true>();
    return err;
}

int gemm_pair_clusters() {
    static int device = -1, clusters = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev == device) return clusters;
    // the pair kernels run one CTA per SM (their shared memory): how many
    // two-CTA clusters of the largest configuration are resident at once
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3((2 + 4 * kEpiGroups + 1) * 32);
    cfg.dynamicSmemBytes = kSmemLimit;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (raise_smem<KIND_MX, SET_F32, true>() != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, mx_gemm_kernel<KIND_MX, SET_F32, true>, &cfg) != cudaSuccess)
        n = 0;
    device = dev;
    clusters = n;
    return clusters;
}

cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t s, bool pdl) {
    if (!gemm_config_ok(p.n_max, p.groups, p.ksplit, p.acc_bufs)) return cudaErrorInvalidValue;
    if (p.stages < 2 * p.groups || p.stages > kMaxStagesPerGroup * p.groups) return cudaErrorInvalidValue;
    const bool pair = p.pair != 0;
    const size_t smem = gemm_smem_bytes(p.n_max, p.stages, p.dense ? 0 : p.E, gemm_needs_xbuf(p), pair);
    if (smem > static_cast<size_t>(kSmemLimit)) return cudaErrorInvalidValue;
    if (p.stage_bytes != gemm_stage_bytes(p.n_max, pair)) return cudaErrorInvalidValue;
    if (p.kseg_tiles <= 0 || p.KT > 3 * p.kseg_tiles) return cudaErrorInvalidValue;
    if (!p.dense && (p.E <= 0 || p.E > 1024)) return cudaErrorInvalidValue;
    const int set = epi_set(p);
    if (set < 0) return cudaErrorInvalidValue;
    if (p.b_producer && p.groups != 1) return cudaErrorInvalidValue;
    if (p.dense && (p.mt_base < 0 || (p.mt_base + p.m_tiles) * kBlockM > p.a_rows)) return cudaErrorInvalidValue;
    const dim3 g(grid), b((2 * p.groups + 4 * kEpiGroups + (p.b_producer ? 1 : 0)) * 32);
    if (pair) {
        // one group of whole items fed by both producers, 16-row token boxes,
        // whole pairs of weight tiles, scale maps for the paired copies
        if (p.kind != KIND_MX || p.groups > 2 || p.ksplit != 1 || p.b_producer != (p.groups == 1 ? 1 : 0) ||
            p.b_box != pair_b_rows(p.n_max) || p.b_row1)
            return cudaErrorInvalidValue;
        if (grid < 2 || (grid & 1)) return cudaErrorInvalidValue;
        if (p.dense ? ((p.m_tiles & 1) || (p.mt_base & 1)) : (p.mt_per_e & 1)) return cudaErrorInvalidValue;
        if (set == SET_F32) return launch_ex_cluster(mx_gemm_kernel<KIND_MX, SET_F32, true>, g, b, smem, s, pdl, 2, p);
        if (set == SET_QUANT)
            return launch_ex_cluster(mx_gemm_kernel<KIND_MX, SET_QUANT, true>, g, b, smem, s, pdl, 2, p);
        if (set == SET_SILU) return launch_ex_cluster(mx_gemm_kernel<KIND_MX, SET_SILU, true>, g, b, smem, s, pdl, 2, p);
        return cudaErrorInvalidValue;
    }
    if (!(p.b_box == 16 || p.b_box == p.n_max)) return cudaErrorInvalidValue;   // boxes must tile the B rows
    if (p.kind == KIND_TF32) {
        if (set != SET_F32) return cudaErrorInvalidValue;
        return launch_ex(mx_gemm_kernel<KIND_TF32, SET_F32>, g, b, smem, s, pdl, p);
    }
    if (p.kind == KIND_BF16) {
        if (set == SET_F32) return launch_ex(mx_gemm_kernel<KIND_BF16, SET_F32>, g, b, smem, s, pdl, p);
        if (set == SET_DUAL) return launch_ex(mx_gemm_kernel<KIND_BF16, SET_DUAL>, g, b, smem, s, pdl, p);
        return cudaErrorInvalidValue;
    }
    if (set == SET_F32) return launch_ex(mx_gemm_kernel<KIND_MX, SET_F32>, g, b, smem, s, pdl, p);
    if (set == SET_QUANT) return launch_ex(mx_gemm_kernel<KIND_MX, SET_QUANT>, g, b, smem, s, pdl, p);
    if (set == SET_SILU) return launch_ex(mx_gemm_kernel<KIND_MX, SET_SILU>, g, b, smem, s, pdl, p);
    return launch_ex(mx_gemm_kernel<KIND_MX, SET_DUAL>, g, b, smem, s, pdl, p);
}

}  // namespace moe
