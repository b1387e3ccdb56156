// Router logits of decode-sized batches (up to 128 tokens), exact fp32:
//   logits[t][e] = sum_k z[t][k] R[e][k]
// ("Kimi K3 and the New Open-Weights Moat", section "How the router picks 16
// of 896": one score per expert from the token's router input).
//
// The work is 2 T E K FLOPs on fp32 CUDA cores while R (E x K fp32, 12.8 MB
// on the K3-shaped layer) streams from HBM once.  A CTA owns a tile of 128
// experts x 64 tokens and one contiguous range of the K dimension; the c CTAs
// of a thread-block cluster split K (c = 16 for up to 64 tokens, 8 above),
// so that about 112 SMs stream R at once.  A producer warp keeps up to eight
// 32-wide K chunks of R and z in flight (TMA, 128-byte swizzled tiles, one
// mbarrier per stage); the compute warps each own an equal share of the 128 experts x 64 tokens
// (lane l: tokens l and l + 32) and run one sequential FMA chain per output
// over the CTA's K range, as two interleaved chains (even and odd k) in the
// halves of packed fp32x2 FMAs.  The partial tiles are then summed across the
// cluster: every CTA owns 1/c of the tile and receives the other CTAs'
// partials of it by bulk copies into its shared memory (completion counted on
// its mbarrier), then adds the c partials in rank order: the logits do not
// depend on scheduling.
//
// Every wait is bounded; a wait that runs out records a status code.
#include <cooperative_groups.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace cg = cooperative_groups;

namespace {

constexpr int kRsE = 128;                  // experts per tile
constexpr int kRsT = 64;                   // tokens per tile
constexpr int kRsKC = 32;                  // K per chunk (one 128-byte row of fp32)
#ifndef MOE_RS_WARPS
#define MOE_RS_WARPS 16
#endif
#ifndef MOE_RS_UNROLL
#define MOE_RS_UNROLL 8
#endif
constexpr int kRsWarps = MOE_RS_WARPS;     // compute warps; warp kRsWarps produces
constexpr int kRsUnroll = MOE_RS_UNROLL;   // K steps of 4 unrolled in the compute loop
constexpr int kRsEpw = 128 / kRsWarps;     // experts per compute warp
constexpr int kRsStages = 8;
constexpr int kRsRBytes = kRsE * kRsKC * 4;             // 16 KB
constexpr int kRsStageBytes = kRsRBytes + kRsT * kRsKC * 4;   // + 8 KB of z
constexpr int kRsTile = kRsE * kRsT;                   // outputs of a tile: [expert][token]
// stages, then the receive area for the peers' partials (written by them at
// any time after this CTA's barriers exist), then the barriers
constexpr int kRsRecvOff = kRsStages * kRsStageBytes;
constexpr int kRsBarOff = kRsRecvOff + kRsTile * 4;
constexpr int kRsSmem = 1024 + kRsBarOff + 256;
static_assert(kRsTile * 4 <= kRsStages * kRsStageBytes, "the partial tile fits in the stage area");
static_assert(kRsSmem <= 227 * 1024, "shared memory per CTA");

struct RouterStreamParams {
    CUtensorMap tmR;    // fp32 [E][K], box {32, 128}, 128-byte swizzle
    CUtensorMap tmZ;    // fp32 [T_pad][K] (row pitch ld), box {32, 64}, 128-byte swizzle
    float* logits;      // [T][E]
    int T, E, K;
    int* status;
};

// Byte offset of elements (row, 4 c4 .. 4 c4 + 3) of a swizzled tile of
// 128-byte rows: 16-byte chunk c4 of row r sits at chunk position c4 ^ (r % 8).
__device__ __forceinline__ uint32_t swz(int row, int c4) {
    return static_cast<uint32_t>(row * 128 + ((c4 ^ (row & 7)) << 4));
}

// Shared-memory loads by 32-bit shared addresses (plain LDS, not generic
// loads), and loads from a peer CTA's shared memory in the cluster.  lds128
// is not volatile, so the compiler may schedule the loads of a step
// together; its address comes from an opaque copy made after the stage's
// barrier wait, so no load moves above the wait.
struct F2x2 {
    unsigned long long lo, hi;    // elements {0, 1} and {2, 3} of 16 bytes as packed fp32 pairs
};
__device__ __forceinline__ F2x2 lds128(uint32_t a) {
    F2x2 v;
    asm("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(v.lo), "=l"(v.hi) : "r"(a));
    return v;
}
// acc (two fp32 lanes) += a * b, lane by lane, each rounded once
__device__ __forceinline__ void ffma2(unsigned long long& acc, unsigned long long a, unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ float sum_pair(unsigned long long v) {
    return __uint_as_float(static_cast<uint32_t>(v)) + __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint32_t opaque(uint32_t v) {
    asm volatile("" : "+r"(v));
    return v;
}
// The values must exist before any later volatile statement (the release of
// the stage whose data they were computed from).
__device__ __forceinline__ void keep4(const unsigned long long* v) {
    asm volatile("" ::"l"(v[0]), "l"(v[1]), "l"(v[2]), "l"(v[3]));
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t a, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Bulk copy of `bytes` from this CTA's shared memory to a peer's (cluster
// addresses of the destination and of the peer's mbarrier), counted on that
// mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

__global__ void __launch_bounds__((kRsWarps + 1) * 32, 1) router_stream_kernel(const __grid_constant__ RouterStreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + kRsBarOff);
    uint64_t* empty = full + kRsStages;
    uint64_t* recv_bar = empty + kRsStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(recv_bar + 1);
    cg::cluster_group cluster = cg::this_cluster();
    const int c = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int e0 = blockIdx.y * kRsE, t0 = blockIdx.z * kRsT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = p.K / kRsKC;
    const int cb = chunks * rank / c, ce = chunks * (rank + 1) / c;
    const int n = ce - cb;
    const int S = n < kRsStages ? n : kRsStages;
    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRsStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRsWarps);
        }
        mbar_init(recv_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tmR);
        prefetch_tmap(&p.tmZ);
    }
    __syncthreads();
    pdl_wait();         // the router input and the logits belong to the kernels around this one
    // peers may copy into this CTA only once its barriers exist: arrive now,
    // wait just before the copies
    cluster_arrive();
    unsigned long long acc[kRsEpw][2];    // [expert][token l, l + 32]: even-k and odd-k partial sums
#pragma unroll
    for (int j = 0; j < kRsEpw; ++j) acc[j][0] = acc[j][1] = 0ull;
    if (warp == kRsWarps) {
        // producer: one elected lane issues, the warp stays converged
        int issued = 0;
        for (int i = 0; i < n; ++i) {
            const int s = i % S;
            const bool ok = mbar_wait(&empty[s], ((i / S) & 1) ^ 1, abort_flag, p.status, DEV_TIMEOUT_PRODUCER);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint8_t* st = base + s * kRsStageBytes;
            if (elect_one()) {
                mbar_arrive_expect_tx(&full[s], kRsStageBytes);
                tma_load_2d(st, &p.tmR, &full[s], (cb + i) * kRsKC, e0);
                tma_load_2d(st + kRsRBytes, &p.tmZ, &full[s], (cb + i) * kRsKC, t0);
            }
            __syncwarp();
            issued = i + 1;
        }
        if (*abort_flag && lane == 0) {
            // copies still in flight must land before the stage area is reused
            for (int i = (issued > S ? issued - S : 0); i < issued; ++i) {
                const uint64_t tstart = globaltimer_ns();
                while (!mbar_try_wait(&full[i % S], (i / S) & 1) && globaltimer_ns() - tstart < kWaitLimitNs) {
                }
            }
        }
        __syncwarp();
    } else {
        for (int i = 0; i < n; ++i) {
            const int s = i % S;
            const bool ok = mbar_wait(&full[s], (i / S) & 1, abort_flag, p.status, DEV_TIMEOUT_MMA);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint32_t Rt = opaque(smem_u32(base + s * kRsStageBytes));
            const uint32_t Zt = Rt + kRsRBytes;
#pragma unroll kRsUnroll
            for (int c4 = 0; c4 < kRsKC / 4; ++c4) {
                const F2x2 z0 = lds128(Zt + swz(lane, c4));
                const F2x2 z1 = lds128(Zt + swz(lane + 32, c4));
#pragma unroll
                for (int j = 0; j < kRsEpw; ++j) {
                    const F2x2 r = lds128(Rt + swz(kRsEpw * warp + j, c4));
                    ffma2(acc[j][0], z0.lo, r.lo);
                    ffma2(acc[j][0], z0.hi, r.hi);
                    ffma2(acc[j][1], z1.lo, r.lo);
                    ffma2(acc[j][1], z1.hi, r.hi);
                }
            }
#pragma unroll
            for (int j = 0; j < kRsEpw; j += 2) keep4(&acc[j][0]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    // the partial tile goes where the stages were (every chunk has been
    // consumed): [expert][token], so that each owner's share -- experts
    // [q E/c, (q + 1) E/c) of the tile -- is contiguous
    __syncthreads();
    float* part = reinterpret_cast<float*>(base);
    float* recv = reinterpret_cast<float*>(base + kRsRecvOff);  // [sender][share]
    if (warp < kRsWarps) {
#pragma unroll
        for (int j = 0; j < kRsEpw; ++j) {
            part[(kRsEpw * warp + j) * kRsT + lane] = sum_pair(acc[j][0]);
            part[(kRsEpw * warp + j) * kRsT + lane + 32] = sum_pair(acc[j][1]);
        }
    }
    fence_proxy_async_smem();                                   // visible to the bulk copies
    __syncthreads();
    cluster_wait();
    const int share = kRsTile / c;                              // floats per owner
    const uint32_t share_bytes = static_cast<uint32_t>(share) * 4u;
    const uint32_t part_s = smem_u32(part), recv_s = smem_u32(recv), bar_s = smem_u32(recv_bar);
    if (threadIdx.x == 0) mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(c - 1) * share_bytes);
    if (threadIdx.x < static_cast<unsigned>(c) && static_cast<int>(threadIdx.x) != rank) {
        const int q = static_cast<int>(threadIdx.x);
        bulk_to_peer(peer_addr(recv_s + static_cast<uint32_t>(rank) * share_bytes, q),
                     part_s + static_cast<uint32_t>(q) * share_bytes, share_bytes, peer_addr(bar_s, q));
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
    const bool got = mbar_wait(recv_bar, 0, abort_flag, p.status, DEV_TIMEOUT_EPILOGUE);
    if (got) {
        // this CTA's experts, summed over the senders in rank order;
        // consecutive threads take consecutive tokens of one expert
        for (int i = static_cast<int>(threadIdx.x); i < share; i += blockDim.x) {
            float v = 0.0f;
            for (int q = 0; q < c; ++q) v += (q == rank) ? part[rank * share + i] : recv[q * share + i];
            const int el = (rank * share + i) / kRsT, tl = (rank * share + i) % kRsT;
            const int t = t0 + tl, e = e0 + el;
            if (t < p.T && e < p.E) p.logits[static_cast<int64_t>(t) * p.E + e] = v;
        }
    }
    // the copies out of this CTA must have read their source before it exits
    if (threadIdx.x < static_cast<unsigned>(c) && static_cast<int>(threadIdx.x) != rank)
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

}  // namespace

bool router_stream_ok(int K) { return K % (kRsKC * 16) == 0 && K >= kRsKC * 16; }

cudaError_t router_stream_setup() {
    cudaError_t err = cudaFuncSetAttribute(router_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRsSmem);
    if (err == cudaSuccess) err = cudaFuncSetAttribute(router_stream_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return err;
}

// Clusters of `c` CTAs of the streaming router that can be resident at once
// (0: that cluster size cannot be scheduled on this device).
int router_stream_max_clusters(int c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1, 1);
    cfg.blockDim = dim3((kRsWarps + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = kRsSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_stream_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_router_stream(const CUtensorMap& tmR, const CUtensorMap& tmZ, float* logits, int T, int E, int K,
                                 int c, int* status, cudaStream_t s, bool pdl) {
    if (T < 1 || T > 2 * kRsT || E < 1 || (c != 8 && c != 16) || !router_stream_ok(K)) return cudaErrorInvalidValue;
    RouterStreamParams prm;
    prm.tmR = tmR;
    prm.tmZ = tmZ;
    prm.logits = logits;
    prm.T = T;
    prm.E = E;
    prm.K = K;
    prm.status = status;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, (E + kRsE - 1) / kRsE, (T + kRsT - 1) / kRsT);
    cfg.blockDim = dim3((kRsWarps + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = kRsSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, router_stream_kernel, prm);
}

}  // namespace moe
