// The non-GEMM kernels of the layer: MXFP8 quantisation of the input, the
// router GEMM, top-k selection with gate normalisation, the dispatch
// (per-expert counts, offsets, stable ranks, work lists, gather), the
// weighted combine with MXFP8 re-quantisation, the MXFP4 weight encoder, and
// plan-time repacking / debug export helpers.
#include <cooperative_groups.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

namespace cg = cooperative_groups;

namespace {

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ A1: x -> MXFP8
// One warp per (row, group of kQxSpans 256-wide column spans): the group's
// 16-byte loads are issued together, then each span is quantised; lane l owns
// elements 8l..8l+7 of a span, so 4 lanes form one 32-element block and
// lanes 0-15 / 16-31 the span's two 128-wide tiles.  Scales go to the
// item-atom planes of the GEMM that reads xq (token tiles of n_max rows;
// mx.cuh).  D is a multiple of 128; an odd last tile leaves lanes 16-31 idle.
constexpr int kQxSpans = 2;
__global__ void quant_x_kernel(const __nv_bfloat16* __restrict__ x, int T, int D, uint8_t* __restrict__ xq,
                               uint8_t* __restrict__ xsf, int64_t pitch, int n_max, float* __restrict__ xf,
                               uint32_t* __restrict__ zero, int64_t n_zero) {
    pdl_trigger();
    pdl_wait();
    // the forward's selection bitmaps start cleared (the first kernel of the
    // forward clears them, instead of a memset of its own)
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_zero;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        zero[i] = 0u;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles = D / 128;
    const int spans = (tiles + 1) / 2;
    const int groups = (spans + kQxSpans - 1) / kQxSpans;
    if (gw >= static_cast<int64_t>(T) * groups) return;
    const int64_t row = gw / groups;
    const int span0 = static_cast<int>(gw % groups) * kQxSpans;
    uint4 raw[kQxSpans];
#pragma unroll
    for (int j = 0; j < kQxSpans; ++j) {
        const int tile = 2 * (span0 + j) + (lane >> 4);
        if (tile < tiles)
            raw[j] = *reinterpret_cast<const uint4*>(x + row * D + static_cast<int64_t>(span0 + j) * 256 + lane * 8);
    }
    const int64_t b0 = (row / n_max) * n_max;
#pragma unroll
    for (int j = 0; j < kQxSpans; ++j) {
        if (span0 + j >= spans) break;
        const int tile = 2 * (span0 + j) + (lane >> 4);
        const bool valid = tile < tiles;                       // warp-uniform per half
        const int64_t off = row * D + static_cast<int64_t>(span0 + j) * 256 + lane * 8;
        float v[8];
        const uint32_t wd[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(wd[i] << 16);
            v[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
        }
        if (xf && valid) {                                    // x as fp32, exactly
            *reinterpret_cast<float4*>(xf + off) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(xf + off + 4) = make_float4(v[4], v[5], v[6], v[7]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const int e = mx8_exponent(amax);
        const float inv = exp2i(-e);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo |= static_cast<uint32_t>(f32_to_e4m3(v[i] * inv)) << (8 * i);
            hi |= static_cast<uint32_t>(f32_to_e4m3(v[4 + i] * inv)) << (8 * i);
        }
        if (valid) *reinterpret_cast<uint2*>(xq + off) = make_uint2(lo, hi);
        // gather each tile's 4 block scales (lanes 0, 4, 8, 12 and 16, 20, 24, 28) into one word
        const uint32_t sc = static_cast<uint32_t>(e + 127);
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) word |= __shfl_sync(0xffffffffu, sc, (lane & 16) + b * 4) << (8 * b);
        if ((lane & 15) == 0 && valid)
            *reinterpret_cast<uint32_t*>(xsf + sf_atom_offset(b0, static_cast<int>(row - b0), tile * 128, pitch)) = word;
    }
}

// ------------------------------------------------------------------ A3: router logits
// logits[t][e] = sum_l z[t][l] * R[e][l], fp32 with one sequential FMA chain
// per output (deterministic).  64 tokens x 64 experts per CTA, 16-wide K
// slices staged through shared memory, 4x4 outputs per thread.
constexpr int RT = 64, RE = 64, RK = 16;
__global__ void __launch_bounds__(256) router_kernel(const float* __restrict__ z, const float* __restrict__ R,
                                                     float* __restrict__ logits, int T, int E, int L, int ld, int lo) {
    pdl_trigger();
    pdl_wait();
    // z: rows of `ld` floats holding the router input (K = L) and, at offset
    // lo > 0, its exact remainder (the input is hi + lo); lo = 0: no remainder
    __shared__ float zs[RK][RT + 4];
    __shared__ float rs[RK][RE + 4];
    const int t0 = blockIdx.y * RT, e0 = blockIdx.x * RE;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < L; k0 += RK) {
        for (int i = threadIdx.x; i < RT * RK; i += 256) {
            const int r = i / RK, c = i % RK;
            const float* zr = z + static_cast<int64_t>(t0 + r) * ld + k0 + c;
            zs[c][r] = (t0 + r < T) ? zr[0] + (lo ? zr[lo] : 0.0f) : 0.0f;
            rs[c][r] = (e0 + r < E) ? R[static_cast<int64_t>(e0 + r) * L + k0 + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < RK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = zs[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = rs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) logits[static_cast<int64_t>(t) * E + e] = acc[i][j];
        }
    }
}

// Decode-sized batches (T <= 128): 64 experts x 64 tokens per output tile,
// its K range split over the kRouterSplit CTAs of a thread-block cluster, so
// that ~E/64 x 8 CTAs (one per SM) stream R from HBM in parallel while z
// (L2-resident) is re-read only E/64 times.  Each CTA accumulates its K range in registers
// (one sequential FMA chain per output, the next 32-wide K slice prefetched
// into registers during the current one), leaves its partial tile in shared
// memory, and after a cluster barrier reduces 1/8 of the tile by adding the 8
// partials, read through distributed shared memory, in split order -- a
// fixed order, so the logits are deterministic.
constexpr int RC_T = 64, RC_E = 64, RC_K = 32;
__global__ void __cluster_dims__(1, 1, kRouterSplit) __launch_bounds__(256)
    router_cluster_kernel(const float* __restrict__ z, const float* __restrict__ R, float* __restrict__ logits, int T,
                          int E, int L, int ld, int lo, int kper) {
    pdl_trigger();
    pdl_wait();
    __shared__ __align__(16) float zs[RC_K][RC_T + 4];     // [k][token]
    __shared__ __align__(16) float rs[RC_K][RC_E + 4];     // [k][expert]
    __shared__ float red[RC_T * RC_E];                     // this split's partial tile [token][expert]
    cg::cluster_group cluster = cg::this_cluster();
    const int t0 = blockIdx.y * RC_T, e0 = blockIdx.x * RC_E;
    const int ks = static_cast<int>(cluster.block_rank());
    const int kb = ks * kper, ke = min(L, kb + kper);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;   // experts 4tx..4tx+3; tokens 4ty..4ty+3
    float acc[4][4] = {};
    // one K slice: z rows t0..t0+63 (hi and lo, 2 float4 each per thread), R rows e0..e0+63 (2 float4)
    float4 zh[2], zl[2], rv[2];
    auto load = [&](int k0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = threadIdx.x + 256 * u;
            const int r = i >> 3, c = (i & 7) * 4;
            const float* zr = z + static_cast<int64_t>(t0 + r) * ld + k0 + c;
            const bool tv = t0 + r < T;
            zh[u] = tv ? *reinterpret_cast<const float4*>(zr) : make_float4(0.f, 0.f, 0.f, 0.f);
            zl[u] = (tv && lo) ? *reinterpret_cast<const float4*>(zr + lo) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = threadIdx.x + 256 * u;
            const int r = i >> 3, c = (i & 7) * 4;
            rv[u] = (e0 + r < E) ? *reinterpret_cast<const float4*>(R + static_cast<int64_t>(e0 + r) * L + k0 + c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    if (kb < ke) load(kb);
    for (int k0 = kb; k0 < ke; k0 += RC_K) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = threadIdx.x + 256 * u;
            const int r = i >> 3, c = (i & 7) * 4;
            zs[c][r] = zh[u].x + zl[u].x;
            zs[c + 1][r] = zh[u].y + zl[u].y;
            zs[c + 2][r] = zh[u].z + zl[u].z;
            zs[c + 3][r] = zh[u].w + zl[u].w;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = threadIdx.x + 256 * u;
            const int r = i >> 3, c = (i & 7) * 4;
            rs[c][r] = rv[u].x;
            rs[c + 1][r] = rv[u].y;
            rs[c + 2][r] = rv[u].z;
            rs[c + 3][r] = rv[u].w;
        }
        __syncthreads();
        if (k0 + RC_K < ke) load(k0 + RC_K);
#pragma unroll 8
        for (int kk = 0; kk < RC_K; ++kk) {
            const float4 a4 = *reinterpret_cast<const float4*>(&zs[kk][ty * 4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&rs[kk][tx * 4]);
            const float a[4] = {a4.x, a4.y, a4.z, a4.w};
            const float b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2)
#pragma unroll
                for (int j2 = 0; j2 < 4; ++j2) acc[i2][j2] = fmaf(a[i2], b[j2], acc[i2][j2]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2)
#pragma unroll
        for (int j2 = 0; j2 < 4; ++j2) red[(ty * 4 + i2) * RC_E + tx * 4 + j2] = acc[i2][j2];
    cluster.sync();
    // this CTA's eighth of the tile: 512 outputs, two per thread
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int o = ks * 512 + h * 256 + threadIdx.x;
        const int tt = o / RC_E, ee = o % RC_E;
        float v = 0.0f;
#pragma unroll
        for (int q = 0; q < kRouterSplit; ++q) v += cluster.map_shared_rank(red, q)[o];
        if (t0 + tt < T && e0 + ee < E) logits[static_cast<int64_t>(t0 + tt) * E + e0 + ee] = v;
    }
    cluster.sync();     // no CTA leaves while another still reads its tile
}

// ------------------------------------------------------------------ A4: top-k + gates
// One warp per token; lane l holds the keys of experts l, l+32, ... in
// registers (E <= 32 * kTopkPerLane).
//
// Selection key and its precision:
//  * no bias, or softmax gates: the fp32 logit.  sigmoid is strictly
//    increasing, so ranking logits ranks sigmoid(l) exactly (ties only where
//    the logits tie).
//  * with a bias: sigmoid(l) + b, decided in fp64.
// When the logits are approximate (tensor-core router) or keys need fp64,
// candidates are picked on the estimates.  Each key estimate k_e has a proven
// error bound d_e (the per-(token, expert) bound of TopkArgs for estimated
// logits; for sigmoid(l) + b that bound times the largest slope of sigmoid
// over the logit's interval, plus kKeyErr; kKeyErr alone for exact logits
// with a bias), so the exact key lies in [k_e - d_e, k_e + d_e].
// With theta = the k-th largest lower end, k experts have an exact key >=
// theta, and an expert whose upper end is below theta cannot be in the exact
// top-k: the candidates are the experts with k_e + d_e >= theta.  Their exact
// fp32 logits (recomputed from z and R when the logits were approximate) and
// keys give the final ranking; with more than 64 candidates every expert's
// logit and key are evaluated exactly instead.  Rounds take the largest
// remaining key, the lower expert id on a tie.
// Gates: sigmoid(l_j) / sum over the winners (fp32), or softmax over the
// winners' logits.  Each selection sets bit t of the expert's token bitmap.
#ifndef MOE_TOPK_WARPS
#define MOE_TOPK_WARPS 4
#endif
#ifndef MOE_TOPK_WIDE_TOKENS
#define MOE_TOPK_WIDE_TOKENS 512
#endif
constexpr int kTopkWarps = MOE_TOPK_WARPS;            // tokens (one warp each) per CTA of topk_kernel
constexpr int kTopkWideTokens = MOE_TOPK_WIDE_TOKENS;  // batches up to this size use one CTA per token (without refinement)
constexpr int kTopkPerLane = 32;     // E <= 1024
constexpr int kMaxE = 32 * kTopkPerLane;
constexpr int kMaxCand = 64;         // candidates ranked exactly per token (two per lane); more: exact pass over all
#ifndef MOE_TOPK_REFINE_GROUP
#define MOE_TOPK_REFINE_GROUP 9
#endif
// candidates whose exact logits share one pass over z: about 25 candidates
// a token take three passes in groups of 9 instead of four in groups of 8
// (8,192 tokens: top-k 294 -> 285 us; groups of 10: 297 us)
constexpr int kRefineGroup = MOE_TOPK_REFINE_GROUP;
static_assert(kRefineGroup >= 8 && kRefineGroup <= 10, "refinement groups of 8 to 10 candidates");
// Error bound of the fp32 estimate 1 / (1 + __expf(-l)) + b of sigmoid(l) + b
// for |b| <= 1: __expf errs by at most 2 + floor(1.173 |x|) ulp (CUDA's
// documented bound), which moves sigmoid by at most sigmoid (1 - sigmoid)
// times that relative error (below 1e-7 for every l); the IEEE division and
// the two additions add a few units of 2^-24.  Larger biases add |b| 2^-22
// (TopkArgs::bias_absmax).
constexpr float kKeyErr = 4.0e-6f;

// An upper bound of the slope sigmoid'(x) = sigmoid(x) (1 - sigmoid(x)) over
// [l - d, l + d], so that |sigmoid(l) - sigmoid(l')| <= bound * d for every l'
// in the interval (mean value theorem): 1/4 when the interval holds 0, else
// sigmoid'(m) <= 1 - sigmoid(m) = 1 / (1 + e^m) at the distance m of the
// interval from 0 (sigmoid' falls with |x|).  e^m comes from __expf, lowered
// by its documented error (2 + floor(1.173 m) units in the last place); every
// step rounds toward the safe side.
__device__ __forceinline__ float sigmoid_slope_ub(float l, float d) {
    const float lo = __fsub_rd(l, d), hi = __fadd_ru(l, d);
    if (!(lo > 0.0f || hi < 0.0f)) return 0.25f;          // holds 0 (or NaN)
    const float m = lo > 0.0f ? lo : -hi;                 // > 0
    const float rel = __fmul_ru(__fadd_ru(3.0f, __fmul_ru(1.174f, m)), 0x1p-23f);
    const float e_lo = __fmul_rd(__expf(m), __fsub_rd(1.0f, rel));
    const float s = __frcp_ru(__fadd_rd(1.0f, fmaxf(e_lo, 0.0f)));
    return fminf(fmaxf(s, 0x1p-126f), 0.25f);
}

// Keys as unsigned integers that order like the floats (larger key, larger
// integer; -inf above every "no entry" value 0), so that a selection round
// is two warp reductions: the largest key, then the lowest expert id among
// the lanes holding it.
__device__ __forceinline__ uint32_t key_bits(float k) {
    const uint32_t u = (k == 0.0f) ? 0u : __float_as_uint(k);     // -0 ties with +0, as the floats compare
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float bits_key(uint32_t b) {
    return __uint_as_float((b & 0x80000000u) ? (b & 0x7fffffffu) : ~b);
}
constexpr uint32_t kNoKey = 0u;

// The warp's best (key bits, id) pair: key desc, id asc.  Returns id
// 0x7fffffff when no lane holds an entry.
__device__ __forceinline__ int warp_best_id(uint32_t kb, int id, uint32_t& best) {
    best = __reduce_max_sync(0xffffffffu, kb);
    return __reduce_min_sync(0xffffffffu, (kb == best && kb != kNoKey) ? id : 0x7fffffff);
}

__device__ __forceinline__ double key64(float l, const float* bias, int e) {
    return 1.0 / (1.0 + exp(-static_cast<double>(l))) + static_cast<double>(bias[e]);
}

// Exact fp32 logits of NE experts e[0..NE) for the token whose router input
// row is zt (its fp32 values at offset lo, or at 0 when lo == 0):
// lane l runs one FMA chain per expert over elements 4l + 128j .. 4l + 128j
// + 3, j = 0, 1, ... in order, then a fixed butterfly sums the lanes; every
// lane returns the values.  The chain of an expert does not depend on NE or
// on the other experts, so every path gives the same logit.  16-byte loads,
// all NE rows of a step in flight together.  L % 128 == 0, 16-byte rows.
template <int NE>
__device__ __forceinline__ void exact_logits(const float* __restrict__ zt, int lo, const float* __restrict__ R,
                                             const int* e, int L, int lane, float* out) {
    const float* r[NE];
#pragma unroll
    for (int u = 0; u < NE; ++u) r[u] = R + static_cast<int64_t>(e[u]) * L;
    float acc[NE];
#pragma unroll
    for (int u = 0; u < NE; ++u) acc[u] = 0.0f;
    const float* zv = zt + lo;
    for (int i = 4 * lane; i < L; i += 128) {
        const float4 z4 = __ldg(reinterpret_cast<const float4*>(zv + i));
        float4 r4[NE];
#pragma unroll
        for (int u = 0; u < NE; ++u) r4[u] = __ldg(reinterpret_cast<const float4*>(r[u] + i));
#pragma unroll
        for (int u = 0; u < NE; ++u) {
            acc[u] = fmaf(z4.x, r4[u].x, acc[u]);
            acc[u] = fmaf(z4.y, r4[u].y, acc[u]);
            acc[u] = fmaf(z4.z, r4[u].z, acc[u]);
            acc[u] = fmaf(z4.w, r4[u].w, acc[u]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < NE; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
#pragma unroll
    for (int u = 0; u < NE; ++u) out[u] = acc[u];
}

// Second half of the top-k of token t, run by one warp.  cand[0..R) holds
// the candidate ids (R <= kMaxCand; overflow: more than that): exact keys of
// the candidates (their logits recomputed from z and R when the logits are
// estimates), their ranking, gates and token bitmaps.  Lane j owns
// candidates j and j + 32.  Without a band (exact logits, no bias) cand[0..k)
// is already the selection in slot order.  On overflow every expert's logit
// and key are evaluated exactly and k rounds select over all of them.
__device__ __noinline__ void topk_finish(const TopkArgs& a, int t, int lane, const int* cand, int R, bool overflow) {
    const int E = a.E, k = a.k;
    float* l = a.logits + static_cast<int64_t>(t) * E;
    const float* bias = a.bias;
    const bool use_bias = (bias != nullptr) && !a.softmax;
    const bool approx = a.refine != 0;
    const bool need_cand = use_bias || approx;
    const float* zt = a.z + static_cast<int64_t>(t) * a.z_ld;
    const int nper = (E + 31) / 32;
    int id0 = 0x7fffffff, id1 = 0x7fffffff;                   // this lane's candidates (0x7fffffff: none)
    float l0 = 0.0f, l1 = 0.0f;                               // their exact logits
    int slot0 = 64, slot1 = 64;                               // their final slots (>= k: not selected)
    if (!need_cand) {
        if (lane < k) {
            id0 = cand[lane];
            l0 = l[id0];
            slot0 = lane;
        }
    } else if (!overflow) {
        if (lane < R) id0 = cand[lane];
        if (lane + 32 < R) id1 = cand[lane + 32];
        if (approx) {
            // candidates in groups of up to kRefineGroup (z is read once per group)
            for (int c = 0; c < R; c += kRefineGroup) {
                const int m = min(kRefineGroup, R - c);
                int ids[kRefineGroup];
                float v[kRefineGroup];
#pragma unroll
                for (int u = 0; u < kRefineGroup; ++u) ids[u] = cand[min(c + u, R - 1)];
                if (m > 8)
                    exact_logits<kRefineGroup>(zt, a.z_lo, a.R, ids, a.L, lane, v);
                else if (m > 4)
                    exact_logits<8>(zt, a.z_lo, a.R, ids, a.L, lane, v);
                else if (m > 2)
                    exact_logits<4>(zt, a.z_lo, a.R, ids, a.L, lane, v);
                else if (m > 1)
                    exact_logits<2>(zt, a.z_lo, a.R, ids, a.L, lane, v);
                else
                    exact_logits<1>(zt, a.z_lo, a.R, ids, a.L, lane, v);
#pragma unroll
                for (int u = 0; u < kRefineGroup; ++u) {
                    if (u < m && c + u == lane) l0 = v[u];
                    if (u < m && c + u == lane + 32) l1 = v[u];
                }
            }
        } else {
            if (id0 != 0x7fffffff) l0 = l[id0];
            if (id1 != 0x7fffffff) l1 = l[id1];
        }
        // exact ranking of the R candidates: larger key first, lower id on a tie
        const double k0 = (id0 != 0x7fffffff) ? (use_bias ? key64(l0, bias, id0) : static_cast<double>(l0)) : -INFINITY;
        const double k1 = (id1 != 0x7fffffff) ? (use_bias ? key64(l1, bias, id1) : static_cast<double>(l1)) : -INFINITY;
        int r0 = 0, r1 = 0;
        for (int i = 0; i < R; ++i) {
            const double a0 = __shfl_sync(0xffffffffu, k0, i & 31), a1 = __shfl_sync(0xffffffffu, k1, i & 31);
            const int b0 = __shfl_sync(0xffffffffu, id0, i & 31), b1 = __shfl_sync(0xffffffffu, id1, i & 31);
            const double ki = (i < 32) ? a0 : a1;
            const int ii = (i < 32) ? b0 : b1;
            if (ii != id0 && (ki > k0 || (ki == k0 && ii < id0))) ++r0;
            if (ii != id1 && (ki > k1 || (ki == k1 && ii < id1))) ++r1;
        }
        if (id0 != 0x7fffffff) slot0 = r0;
        if (id1 != 0x7fffffff) slot1 = r1;
        if (approx) {                                          // export the exact candidate logits
            if (id0 != 0x7fffffff) l[id0] = l0;
            if (id1 != 0x7fffffff) l[id1] = l1;
        }
    } else {
        // rare: exact logits (written back to the logits row, eight experts
        // at a time) and keys of every expert, k rounds over all of them
        if (approx) {
            for (int c = 0; c < E; c += 8) {
                int ids[8];
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) ids[u] = min(c + u, E - 1);
                exact_logits<8>(zt, a.z_lo, a.R, ids, a.L, lane, v);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (c + u < E && lane == u) l[c + u] = v[u];
            }
            __syncwarp();
        }
        uint32_t taken = 0;
        for (int j = 0; j < k; ++j) {
            double bk = -INFINITY;
            int bid = 0x7fffffff;
            float bl = 0.0f;
            for (int i = 0; i < nper; ++i) {
                const int e = lane + 32 * i;
                if (e >= E || (taken & (1u << i))) continue;
                const float le = l[e];
                double kv = use_bias ? key64(le, bias, e) : static_cast<double>(le);
                if (kv != kv) kv = -INFINITY;
                if (bid == 0x7fffffff || kv > bk || (kv == bk && e < bid)) {
                    bk = kv;
                    bid = e;
                    bl = le;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double ob = __shfl_xor_sync(0xffffffffu, bk, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
                const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
                if (oi != 0x7fffffff && (bid == 0x7fffffff || ob > bk || (ob == bk && oi < bid))) {
                    bk = ob;
                    bid = oi;
                    bl = ol;
                }
            }
            if (bid < 0 || bid >= E) bid = 0;
            if (lane == j) {
                id0 = bid;
                l0 = bl;
                slot0 = j;
            }
            if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
        }
    }
    // gates over the k winners (candidates whose slot < k), from exact logits
    const bool w0 = slot0 < k, w1 = slot1 < k;
    float s0 = w0 ? l0 : 0.0f, s1 = w1 ? l1 : 0.0f;
    if (a.softmax) {
        float lmax = fmaxf(w0 ? s0 : -INFINITY, w1 ? s1 : -INFINITY);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
        s0 = w0 ? expf(s0 - lmax) : 0.0f;
        s1 = w1 ? expf(s1 - lmax) : 0.0f;
    } else {
        s0 = w0 ? 1.0f / (1.0f + expf(-s0)) : 0.0f;
        s1 = w1 ? 1.0f / (1.0f + expf(-s1)) : 0.0f;
    }
    float sum = s0 + s1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (w0) {
        a.idx[static_cast<int64_t>(t) * k + slot0] = id0;
        a.w[static_cast<int64_t>(t) * k + slot0] = s0 / sum;
        atomicOr(&a.sel[static_cast<int64_t>(id0) * a.W + (t >> 5)], 1u << (t & 31));
    }
    if (w1) {
        a.idx[static_cast<int64_t>(t) * k + slot1] = id1;
        a.w[static_cast<int64_t>(t) * k + slot1] = s1 / sum;
        atomicOr(&a.sel[static_cast<int64_t>(id1) * a.W + (t >> 5)], 1u << (t & 31));
    }
}

// Key interval ends as key_bits values: lower end rounded down, upper end
// rounded up; an end that is not a number widens to the infinity on its side.
__device__ __forceinline__ uint32_t lo_bits(float kv, float d) {
    const float v = __fsub_rd(kv, d);
    return key_bits(v != v ? -INFINITY : v);
}
__device__ __forceinline__ uint32_t hi_bits(float kv, float d) {
    const float v = __fadd_ru(kv, d);
    return key_bits(v != v ? INFINITY : v);
}

// Upper bounds of the 2-norms of the TF32 head (the first L values) and of
// the exact remainder z - head (the fp32 values z sit at offset lo; lo = 0:
// none, the row is then exactly TF32) of one router input row, from fp32 sums
// of squares scaled by `infl` (which covers their rounding).  Every lane
// returns both.
__device__ __forceinline__ void input_norms(const float* __restrict__ zt, int lo, int L, float infl, int lane,
                                            float& nhi, float& nlo) {
    float sh = 0.0f, sl = 0.0f;
    for (int i = 4 * lane; i < L; i += 128) {
        // with lo > 0 the head is recomputed from the values (the same
        // rounding that wrote it), so only the values are read
        const float4 z = __ldg(reinterpret_cast<const float4*>(zt + lo + i));
        const float4 h = lo ? make_float4(tf32_round(z.x), tf32_round(z.y), tf32_round(z.z), tf32_round(z.w)) : z;
        sh = fmaf(h.x, h.x, sh);
        sh = fmaf(h.y, h.y, sh);
        sh = fmaf(h.z, h.z, sh);
        sh = fmaf(h.w, h.w, sh);
        if (lo) {
            const float4 q = make_float4(z.x - h.x, z.y - h.y, z.z - h.z, z.w - h.w);   // exact
            sl = fmaf(q.x, q.x, sl);
            sl = fmaf(q.y, q.y, sl);
            sl = fmaf(q.z, q.z, sl);
            sl = fmaf(q.w, q.w, sl);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sh += __shfl_xor_sync(0xffffffffu, sh, o);
        sl += __shfl_xor_sync(0xffffffffu, sl, o);
    }
    nhi = __fsqrt_ru(__fmul_ru(sh, infl));
    nlo = lo ? __fsqrt_ru(__fmul_ru(sl, infl)) : 0.0f;
}

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(TopkArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_cand[kTopkWarps][kMaxCand];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= a.T) return;
    const int E = a.E, k = a.k;
    const float* l = a.logits + static_cast<int64_t>(t) * E;
    const float* bias = a.bias;
    const bool use_bias = (bias != nullptr) && !a.softmax;
    const bool approx = a.refine != 0;
    const int nper = (E + 31) / 32;
    if (!use_bias && !approx) {
        // exact logits ranked as they are: k rounds give the selection in slot order
        uint32_t key[kTopkPerLane];
#pragma unroll
        for (int i = 0; i < kTopkPerLane; ++i) {
            const int e = lane + 32 * i;
            float kv = (i < nper && e < E) ? l[e] : 0.0f;
            if (kv != kv) kv = -INFINITY;                     // NaN ranks last
            key[i] = (i < nper && e < E) ? key_bits(kv) : kNoKey;
        }
        uint32_t taken = 0;
        for (int j = 0; j < k; ++j) {
            uint32_t lb = kNoKey;
            int lid = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kTopkPerLane; ++i) {
                const uint32_t kv = (taken & (1u << i)) ? kNoKey : key[i];
                if (kv > lb) {
                    lb = kv;
                    lid = lane + 32 * i;
                }
            }
            uint32_t bb;
            int bid = warp_best_id(lb, lid, bb);
            if (bid < 0 || bid >= E) bid = 0;                 // unreachable while k <= E
            if (lane == 0) s_cand[warp][j] = bid;
            if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
        }
        __syncwarp();
        topk_finish(a, t, lane, s_cand[warp], k, false);
        return;
    }
    // error bound of each key estimate: d_e = A |R_lo_e| + B |R_e| for
    // tensor-core logit estimates (TopkArgs), times the largest slope of the
    // sigmoid over [l - d_e, l + d_e] (sigmoid_slope_ub), plus kKeyErr for
    // the fp32 evaluation of sigmoid(l) + b
    float A = 0.0f, B = 0.0f;
    if (approx) {
        float nhi, nlo;
        input_norms(a.z + static_cast<int64_t>(t) * a.z_ld, a.z_lo, a.L, a.sq_infl, lane, nhi, nlo);
        A = nhi;
        B = __fadd_ru(__fadd_ru(nlo, __fmul_ru(__fmul_ru(a.g_tc, 1.0f + 0x1p-11f), nhi)),
                      __fmul_ru(a.g_32, __fadd_ru(nhi, nlo)));
    }
    auto estimate = [&](int e, float& kv, float& d) {
        const float lv = l[e];
        d = approx ? __fmaf_ru(A, a.rnorm[E + e], __fmul_ru(B, a.rnorm[e])) : 0.0f;
        if (use_bias) {
            kv = 1.0f / (1.0f + __expf(-lv)) + bias[e];
            d = __fmaf_ru(sigmoid_slope_ub(lv, d), d, a.key_err);
        } else {
            kv = lv;
        }
        if (kv != kv) kv = -INFINITY;                         // NaN ranks last
    };
    // theta = the k-th largest lower end (k rounds over the lower ends)
    uint32_t lbk[kTopkPerLane];
#pragma unroll
    for (int i = 0; i < kTopkPerLane; ++i) {
        const int e = lane + 32 * i;
        lbk[i] = kNoKey;
        if (i < nper && e < E) {
            float kv, d;
            estimate(e, kv, d);
            lbk[i] = lo_bits(kv, d);
        }
    }
    uint32_t taken = 0, theta = kNoKey;
    for (int j = 0; j < k; ++j) {
        uint32_t lb = kNoKey;
        int lid = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kTopkPerLane; ++i) {
            const uint32_t kv = (taken & (1u << i)) ? kNoKey : lbk[i];
            if (kv > lb) {
                lb = kv;
                lid = lane + 32 * i;
            }
        }
        uint32_t bb;
        const int bid = warp_best_id(lb, lid, bb);
        theta = bb;
        if (bid >= 0 && bid < E && (bid & 31) == lane) taken |= 1u << (bid >> 5);
    }
    // candidates: every expert whose upper end reaches theta
    uint32_t mask = 0;
#pragma unroll
    for (int i = 0; i < kTopkPerLane; ++i) {
        const int e = lane + 32 * i;
        if (i < nper && e < E) {
            float kv, d;
            estimate(e, kv, d);
            if (hi_bits(kv, d) >= theta) mask |= 1u << i;
        }
    }
    const int c = __popc(mask);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const bool overflow = total > kMaxCand;
    if (!overflow) {
        int pos = incl - c;
        while (mask) {
            const int i = __ffs(mask) - 1;
            mask &= mask - 1;
            s_cand[warp][pos++] = lane + 32 * i;
        }
    }
    __syncwarp();
    topk_finish(a, t, lane, s_cand[warp], overflow ? 0 : total, overflow);
}

// Top-k of small batches: one CTA per token, one thread per expert.  The
// k-th largest key is found bit by bit with block-wide counts (the largest
// v with at least k keys >= v; without a band the search stops as soon as
// exactly k keys are >= v); the candidates are the keys >= v, or, with
// an error band, the keys >= the k-th estimate - 2 err (more than kMaxCand:
// overflow).  Each candidate's rank among the candidates (larger key, or
// equal key and lower id, first) orders them, and warp 0 finishes as
// topk_kernel.  Every step is a short chain: this batch size is latency-bound.
constexpr int kTopkWideThreads = kMaxE;
constexpr int kRankCap = kMaxCand + 1;
__global__ void __launch_bounds__(kTopkWideThreads) topk_wide_kernel(TopkArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ int s_cand[kMaxE];
    __shared__ uint32_t s_ckb[kMaxE];
    __shared__ int s_rank[kRankCap];
    __shared__ int s_n;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const int E = a.E, k = a.k;
    const int e = threadIdx.x;
    const bool use_bias = (a.bias != nullptr) && !a.softmax;
    const bool band = use_bias || a.refine != 0;
    uint32_t kb = kNoKey;
    if (e < E) {
        float kv = a.logits[static_cast<int64_t>(t) * E + e];
        if (use_bias) kv = 1.0f / (1.0f + __expf(-kv)) + a.bias[e];
        if (kv != kv) kv = -INFINITY;                         // NaN ranks last
        kb = key_bits(kv);
    }
    if (threadIdx.x == 0) s_n = 0;
    uint32_t v = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t tv = v | (1u << bit);
        const int c = __syncthreads_count(kb >= tv);
        if (c >= k) {
            v = tv;
            // exactly k keys >= v: they are the top k (without a band the
            // remaining bits cannot change the candidates)
            if (!band && c == k) break;
        }
    }
    uint32_t lo = v;
    if (band) lo = min(v, key_bits(__fsub_rd(bits_key(v), a.band_pad)));
    if (e < E && kb >= lo) {
        const int i = atomicAdd(&s_n, 1);
        s_cand[i] = e;
        s_ckb[i] = kb;
    }
    __syncthreads();
    const int n = s_n;
    for (int i = threadIdx.x; i < n; i += kTopkWideThreads) {
        const uint32_t ki = s_ckb[i];
        const int ei = s_cand[i];
        int r = 0;
        for (int j = 0; j < n; ++j) {
            const uint32_t kj = s_ckb[j];
            r += (kj > ki || (kj == ki && s_cand[j] < ei)) ? 1 : 0;
        }
        if (r < kRankCap) s_rank[r] = ei;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;
    const int R = band ? n : k;
    const bool over = R > kMaxCand;
    topk_finish(a, t, lane, s_rank, over ? 0 : R, over);
}

// ------------------------------------------------------------------ A5: per-expert scan
// One warp per expert: prefix popcounts of its token bitmap.  wpre[e][w] =
// number of tokens < 32w that selected e; counts[e] = total.
__global__ void expert_scan_kernel(const uint32_t* __restrict__ sel, int E, int W, int32_t* __restrict__ wpre,
                                   int32_t* __restrict__ counts) {
    pdl_trigger();
    pdl_wait();
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (e >= E) return;
    int running = 0;
    for (int w0 = 0; w0 < W; w0 += 32) {
        const int w = w0 + lane;
        const int c = (w < W) ? __popc(sel[static_cast<int64_t>(e) * W + w]) : 0;
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (w < W) wpre[static_cast<int64_t>(e) * W + w] = running + incl - c;
        running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[e] = running;
}

// Offsets (exact, and padded to 16 rows per expert) and the per-expert item
// offsets of the two grouped GEMMs, in one CTA of 1024 threads (E <= 1024:
// thread e owns expert e).  Expert e contributes ceil(n_e / n_max) token tiles
// x mt weight tiles to a GEMM; the GEMM derives each item from these tables.
__global__ void __launch_bounds__(1024) worklist_kernel(WorkListArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ int4 warp_tot[32];
    const int E = a.E;
    const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int n = 0;
    if (a.sel) {
        // expert e's prefix popcounts over its token bitmap (as expert_scan_kernel)
        if (e < E) {
            for (int w = 0; w < a.W; ++w) {
                a.wpre[static_cast<int64_t>(e) * a.W + w] = n;
                n += __popc(a.sel[static_cast<int64_t>(e) * a.W + w]);
            }
            a.counts_out[e] = n;
        }
    } else {
        n = (e < E) ? a.counts[e] : 0;
    }
    const int4 v = make_int4(n, (n + 15) & ~15, ceil_div(n, a.n_max1) * a.mt1, ceil_div(n, a.n_max2) * a.mt2);
    int4 inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, inc.x, o), y = __shfl_up_sync(0xffffffffu, inc.y, o);
        const int z = __shfl_up_sync(0xffffffffu, inc.z, o), w = __shfl_up_sync(0xffffffffu, inc.w, o);
        if (lane >= o) {
            inc.x += x;
            inc.y += y;
            inc.z += z;
            inc.w += w;
        }
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int4 tv = warp_tot[lane];
        int4 ti = tv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, ti.x, o), y = __shfl_up_sync(0xffffffffu, ti.y, o);
            const int z = __shfl_up_sync(0xffffffffu, ti.z, o), w = __shfl_up_sync(0xffffffffu, ti.w, o);
            if (lane >= o) {
                ti.x += x;
                ti.y += y;
                ti.z += z;
                ti.w += w;
            }
        }
        warp_tot[lane] = make_int4(ti.x - tv.x, ti.y - tv.y, ti.z - tv.z, ti.w - tv.w);
    }
    __syncthreads();
    const int4 base = warp_tot[warp];
    const int4 ex = make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z, base.w + inc.w - v.w);
    if (e < E) {
        a.offsets[e] = ex.x;
        a.seg[e] = ex.y;
        a.ioff1[e] = ex.z;
        a.ioff2[e] = ex.w;
    }
    if (e == E - 1) {
        a.offsets[E] = ex.x + v.x;
        a.seg[E] = ex.y + v.y;
        a.ioff1[E] = ex.z + v.z;
        a.ioff2[E] = ex.w + v.w;
    }
}

// ------------------------------------------------------------------ A5/A6: ranks + gather
// One warp per token and slots_per_warp of its slots.  The rank of token t
// inside expert e's segment is the number of tokens < t that selected e
// (bitmap prefix + popcount), so the resulting order is the stable sort of
// (token, slot) pairs by expert.  The token's codes and scale words are read
// once per warp and written to each of its slots' positions: large batches
// take 4 slots a warp (8,192 tokens: 134 -> 116 us; one warp per slot read
// each row from L2 once per slot), small ones one (64 tokens: 6.8 vs 8.9 us,
// the loads of more warps in flight).
#ifndef MOE_SCATTER_SLOTS
#define MOE_SCATTER_SLOTS 4
#endif
#ifndef MOE_SCATTER_SLOTS_FROM
#define MOE_SCATTER_SLOTS_FROM 1024
#endif
__global__ void scatter_kernel(ScatterArgs a) {
    pdl_trigger();
    pdl_wait();
    const int spw = a.slots_per_warp;
    const int groups = (a.k + spw - 1) / spw;
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= static_cast<int64_t>(a.T) * groups) return;
    const int t = static_cast<int>(gw / groups);
    const int j0 = static_cast<int>(gw - static_cast<int64_t>(t) * groups) * spw;
    const int j1 = min(j0 + spw, a.k);
    // the token's codes and scale words do not depend on where they go: their
    // loads are issued before the ranks' (up to 4096 codes a row from registers)
    constexpr int kRowRegs = 8;
    const int n16 = a.L / 16, n128 = a.L / 128;
    const bool in_regs = n16 <= 32 * kRowRegs;
    const uint4* src = reinterpret_cast<const uint4*>(a.zq + static_cast<int64_t>(t) * a.L);
    uint4 buf[kRowRegs];
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kRowRegs; ++j)
            if (lane + 32 * j < n16) buf[j] = src[lane + 32 * j];
    }
    const uint32_t* ssrc = reinterpret_cast<const uint32_t*>(a.zsf);
    const uint32_t sw = (lane < n128) ? ssrc[lane * a.zsf_pitch + t] : 0u;
    const int w = t >> 5;
    const uint32_t below = (1u << (t & 31)) - 1u;
    for (int j = j0; j < j1; ++j) {
        const int64_t slot = static_cast<int64_t>(t) * a.k + j;
        const int e = a.idx[slot];
        const int rank = a.wpre[static_cast<int64_t>(e) * a.W + w] + __popc(a.sel[static_cast<int64_t>(e) * a.W + w] & below);
        const int pos = a.seg[e] + rank;
        const int canon = a.offsets[e] + rank;
        if (lane == 0) {
            a.slot_pos[slot] = pos;
            a.canon_to_pad[canon] = pos;
            a.sorted_token[canon] = t;
        }
        uint4* dst = reinterpret_cast<uint4*>(a.zq_perm + static_cast<int64_t>(pos) * a.L);
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < kRowRegs; ++i)
                if (lane + 32 * i < n16) dst[lane + 32 * i] = buf[i];
        } else {
            for (int i = lane; i < n16; i += 32) dst[i] = src[i];
        }
        // scales: raw planes in, item-atom planes of the grouped GEMM's token tile out
        const int64_t b0 = a.seg[e] + (rank / a.n_max) * a.n_max;
        const int l = rank % a.n_max;
        if (lane < n128)
            *reinterpret_cast<uint32_t*>(a.zq_perm_sf + sf_atom_offset(b0, l, static_cast<int64_t>(lane) * 128, a.perm_pitch)) = sw;
        for (int kt = lane + 32; kt < n128; kt += 32)
            *reinterpret_cast<uint32_t*>(a.zq_perm_sf + sf_atom_offset(b0, l, static_cast<int64_t>(kt) * 128, a.perm_pitch)) =
                ssrc[kt * a.zsf_pitch + t];
    }
}

// ------------------------------------------------------------------ A9: combine + MXFP8
// c[t][l] = sum_j w[t][j] * o[slot_pos[t][j]][l], slots in order, then MXFP8
// along l.  CTA (t, chunk) covers kCombineWarps x 128 columns of token t; a
// warp owns 128 columns (4 MX blocks), lane i columns 4i..4i+3, so 8 lanes
// share one scale.  The slots' 16-byte loads are issued 8 at a time before
// their FMAs (each element's chain still runs j = 0, 1, ... in order); o is
// read once, with the streaming hint.  L % 128 == 0.  Measured at 8,192
// tokens: 332 us with a warp per 32 columns and 4-byte loads, 278 us with
// this layout (2 warps a CTA; 4 warps 279 us, 7 warps 638 us; 16 loads at a
// time 288 us).
#ifndef MOE_COMBINE_WARPS
#define MOE_COMBINE_WARPS 2
#endif
constexpr int kCombineWarps = MOE_COMBINE_WARPS;
#ifndef MOE_COMBINE_BATCH
#define MOE_COMBINE_BATCH 8
#endif
constexpr int kCombineBatch = MOE_COMBINE_BATCH;      // slots whose loads are issued together
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(
    const float* __restrict__ o, const int32_t* __restrict__ slot_pos, const float* __restrict__ w, int T, int k,
    int L, uint8_t* __restrict__ out_q, int64_t ld_q, uint8_t* __restrict__ out_sf, int64_t sf_pitch, int n_max,
    __nv_bfloat16* __restrict__ out_bf) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int pos_s[32];
    __shared__ float w_s[32];
    if (threadIdx.x < k) {
        pos_s[threadIdx.x] = slot_pos[static_cast<int64_t>(t) * k + threadIdx.x];
        w_s[threadIdx.x] = w[static_cast<int64_t>(t) * k + threadIdx.x];
    }
    __syncthreads();
    const int b4 = blockIdx.y * kCombineWarps + warp;
    if (b4 >= L / 128) return;
    const int col = b4 * 128 + lane * 4;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
        float4 v[kCombineBatch];
#pragma unroll
        for (int u = 0; u < kCombineBatch; ++u)
            if (j0 + u < k) v[u] = __ldcs(reinterpret_cast<const float4*>(o + static_cast<int64_t>(pos_s[j0 + u]) * L + col));
#pragma unroll
        for (int u = 0; u < kCombineBatch; ++u) {
            if (j0 + u < k) {
                const float wj = w_s[j0 + u];
                a0 = fmaf(wj, v[u].x, a0);
                a1 = fmaf(wj, v[u].y, a1);
                a2 = fmaf(wj, v[u].z, a2);
                a3 = fmaf(wj, v[u].w, a3);
            }
        }
    }
    if (out_bf) {                     // mixed precision: the up-projection reads c in bf16
        __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(out_bf + static_cast<int64_t>(t) * ld_q + col);
        d[0] = __floats2bfloat162_rn(a0, a1);
        d[1] = __floats2bfloat162_rn(a2, a3);
        return;
    }
    float amax = fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const int e = mx8_exponent(amax);
    const float inv = exp2i(-e);
    const uint32_t packed = static_cast<uint32_t>(f32_to_e4m3(a0 * inv)) | (static_cast<uint32_t>(f32_to_e4m3(a1 * inv)) << 8) |
                            (static_cast<uint32_t>(f32_to_e4m3(a2 * inv)) << 16) |
                            (static_cast<uint32_t>(f32_to_e4m3(a3 * inv)) << 24);
    *reinterpret_cast<uint32_t*>(out_q + static_cast<int64_t>(t) * ld_q + col) = packed;
    if ((lane & 7) == 0) {
        const int b0 = (t / n_max) * n_max;
        out_sf[sf_atom_offset(b0, t - b0, col, sf_pitch)] = static_cast<uint8_t>(e + 127);
    }
}

// ------------------------------------------------------------------ MXFP4 weight encoder
// One thread per 32-element block.  Shared exponent floor(log2 amax) - 2;
// level = number of grid midpoints {0.25,0.75,1.25,1.75,2.5,3.5,5} strictly
// below |v|/2^e (a value on a midpoint takes the smaller level; anything
// above 5 -- including beyond the clip at 6 -- takes level 7).
__global__ void mxfp4_encode_kernel(const float* __restrict__ w, int64_t rows, int64_t K,
                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    const int64_t nb = K / 32;
    const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= rows * nb) return;
    const int64_t r = b / nb, j = b % nb;
    const float* v = w + r * K + j * 32;
    float x[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 q = *reinterpret_cast<const float4*>(v + i);
        x[i] = q.x;
        x[i + 1] = q.y;
        x[i + 2] = q.z;
        x[i + 3] = q.w;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    uint8_t* c = codes + r * (K / 2) + j * 16;
    if (amax == 0.0f) {
        *reinterpret_cast<uint4*>(c) = make_uint4(0, 0, 0, 0);
        scales[b] = 0;
        return;
    }
    const uint32_t ab = __float_as_uint(amax);
    int fl;
    const int biased = static_cast<int>((ab >> 23) & 0xFFu);
    if (biased != 0) {
        fl = biased - 127;
    } else {
        const uint32_t m = ab & 0x7FFFFFu;             // subnormal: value = m * 2^-149
        fl = -149 + (31 - __clz(m));
    }
    int e = fl - 2;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    // |v| * 2^-e; split the power of two so each factor is a normal float
    const int ne = -e;
    const float s1 = exp2i(ne / 2), s2 = exp2i(ne - ne / 2);
    uint32_t packed[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float a = (fabsf(x[i]) * s1) * s2;
        const int lvl = (a > 0.25f) + (a > 0.75f) + (a > 1.25f) + (a > 1.75f) + (a > 2.5f) + (a > 3.5f) + (a > 5.0f);
        const uint32_t code = static_cast<uint32_t>(lvl) | ((__float_as_uint(x[i]) >> 31) << 3);
        packed[i / 8] |= code << (4 * (i % 8));
    }
    *reinterpret_cast<uint4*>(c) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    scales[b] = static_cast<uint8_t>(e + 127);
}

// ------------------------------------------------------------------ plan-time repacking
__global__ void copy_rows_kernel(uint8_t* __restrict__ dst, int64_t dst_stride, const uint8_t* const* src_rows,
                                 int64_t nrows, int64_t row_bytes) {
    const int64_t r = blockIdx.x;
    if (r >= nrows) return;
    const uint8_t* s = src_rows[r];
    uint8_t* d = dst + r * dst_stride;
    if (((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d) | row_bytes) & 15) == 0) {
        const uint4* s4 = reinterpret_cast<const uint4*>(s);
        uint4* d4 = reinterpret_cast<uint4*>(d);
        for (int64_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x) d4[i] = s4[i];
        return;
    }
    for (int64_t i = threadIdx.x; i < row_bytes; i += blockDim.x) d[i] = s[i];
}

// Row-major scales [rows][kb] -> MMA scale atoms [rows/128][kb/4][512]:
// atom byte 16*i + 4*c + j = scale of row 32*c + i, K-block j of the tile.
__global__ void sf_atoms_kernel(const uint8_t* __restrict__ rm, int64_t rows, int64_t kb, uint8_t* __restrict__ atoms) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * kb) return;
    const int64_t row = i / kb, b = i % kb;
    const int64_t rb = row / 128, rr = row % 128, kt = b / 4, j = b % 4;
    const int64_t KT = kb / 4;
    atoms[(rb * KT + kt) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + j] = rm[i];
}

__global__ void sf_item_planes_kernel(const uint8_t* __restrict__ rm, int64_t rows, int64_t kb,
                                      uint8_t* __restrict__ planes, int64_t pitch, int n_max) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * kb) return;
    const int64_t row = i / kb, b = i % kb;
    const int64_t b0 = (row / n_max) * n_max;
    planes[sf_atom_offset(b0, static_cast<int>(row - b0), b * 32, pitch)] = rm[i];
}

// [rows][K] fp32 -> [rows][2K]: nearest TF32 value, then the exact remainder.
__global__ void tf32_split_kernel(const float* __restrict__ src, int64_t rows, int64_t K, float* __restrict__ dst) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * K) return;
    const int64_t r = i / K, c = i % K;
    const float v = src[i];
    uint32_t hb;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hb) : "f"(v));
    const float hi = __uint_as_float(hb);
    dst[r * 2 * K + c] = hi;
    dst[r * 2 * K + K + c] = v - hi;
}

// Upper bounds of the 2-norms of router rows and of their TF32 remainders:
// one warp per row, fp64 sums of squares (relative error below 2^-40 for rows
// of up to 2^12 values per lane), square roots and the conversion to fp32
// rounded up.
__global__ void router_norms_kernel(const float* __restrict__ R, const float* __restrict__ Rs, int E, int K,
                                    float* __restrict__ out) {
    const int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (e >= E) return;
    double s = 0.0, sl = 0.0;
    for (int i = lane; i < K; i += 32) {
        const double v = R[static_cast<int64_t>(e) * K + i];
        const double q = Rs[static_cast<int64_t>(e) * 2 * K + K + i];
        s = fma(v, v, s);
        sl = fma(q, q, sl);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        sl += __shfl_xor_sync(0xffffffffu, sl, o);
    }
    if (lane == 0) {
        out[e] = __double2float_ru(__dsqrt_ru(__dmul_ru(s, 1.0 + 0x1p-40)));
        out[E + e] = __double2float_ru(__dsqrt_ru(__dmul_ru(sl, 1.0 + 0x1p-40)));
    }
}

// ------------------------------------------------------------------ debug export
__global__ void export_sf_kernel(const uint8_t* __restrict__ planes, int64_t pitch, const int32_t* __restrict__ row_map,
                                 int64_t rows, int64_t nblocks, int64_t col_block0, uint8_t* __restrict__ out,
                                 int item_n, const int32_t* __restrict__ seg, int E) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * nblocks) return;
    const int64_t r = i / nblocks, b = i % nblocks;
    const int64_t src_row = row_map ? row_map[r] : r;
    const int64_t cb = col_block0 + b;
    if (item_n == 0) {
        out[i] = planes[((cb / 4) * pitch + src_row) * 4 + (cb % 4)];
        return;
    }
    int64_t base = 0;                                   // first row of the segment holding src_row
    if (seg) {
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seg[mid] <= src_row) lo = mid;
            else hi = mid - 1;
        }
        base = seg[lo];
    }
    const int64_t b0 = base + ((src_row - base) / item_n) * item_n;
    out[i] = planes[sf_atom_offset(b0, static_cast<int>(src_row - b0), cb * 32, pitch)];
}

__global__ void gather_rows_kernel(const uint8_t* __restrict__ src, int64_t src_stride, const int32_t* __restrict__ row_map,
                                   int64_t rows, int64_t row_bytes, uint8_t* __restrict__ dst, int64_t dst_stride) {
    const int64_t r = blockIdx.x;
    if (r >= rows) return;
    const uint8_t* s = src + static_cast<int64_t>(row_map ? row_map[r] : r) * src_stride;
    uint8_t* d = dst + r * dst_stride;
    for (int64_t i = threadIdx.x; i < row_bytes; i += blockDim.x) d[i] = s[i];
}

}  // namespace

cudaError_t launch_quant_x(const __nv_bfloat16* x, int T, int D, uint8_t* xq, uint8_t* xsf, int64_t pitch, int n_max,
                           float* xf, uint32_t* zero, int64_t n_zero, cudaStream_t s, bool pdl) {
    if (n_max <= 0 || n_zero < 0 || (n_zero > 0 && !zero)) return cudaErrorInvalidValue;
    if (D % 128) return cudaErrorInvalidValue;
    const int64_t warps = static_cast<int64_t>(T) * (((D / 128 + 1) / 2 + kQxSpans - 1) / kQxSpans);
    const int blocks = static_cast<int>((warps * 32 + 255) / 256);
    return launch_ex(quant_x_kernel, dim3(blocks), dim3(256), 0, s, pdl, x, T, D, xq, xsf, pitch, n_max, xf, zero, n_zero);
}

cudaError_t launch_router(const float* z, int ld, int lo, const float* R, float* logits, int T, int E, int L,
                          cudaStream_t s, bool pdl) {
    if (L % 4 || ld % 4 || lo % 4) return cudaErrorInvalidValue;
    if (T <= kRouterSplitTokens && L % RC_K == 0) {
        static_assert(RC_T * RC_E == 512 * kRouterSplit, "two reduced outputs per thread");
        const int kper = ceil_div(L / RC_K, kRouterSplit) * RC_K;
        dim3 grid((E + RC_E - 1) / RC_E, (T + RC_T - 1) / RC_T, kRouterSplit);
        return launch_ex(router_cluster_kernel, grid, dim3(256), 0, s, pdl, z, R, logits, T, E, L, ld, lo, kper);
    }
    dim3 grid((E + RE - 1) / RE, (T + RT - 1) / RT);
    return launch_ex(router_kernel, grid, dim3(256), 0, s, pdl, z, R, logits, T, E, L, ld, lo);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, bool pdl) {
    if (a.E > kMaxE || a.k > 32 || a.k < 1 || a.k > a.E) return cudaErrorInvalidValue;
    // refinement reads router rows as 16-byte vectors, 128 values per warp step
    if (a.refine && (a.L <= 0 || a.L % 128 || a.z_ld % 4 || a.z_lo % 4)) return cudaErrorInvalidValue;
    if (a.refine && (!a.rnorm || !(a.g_tc >= 0.0f) || !(a.g_32 >= 0.0f) || !(a.sq_infl >= 1.0f)))
        return cudaErrorInvalidValue;
    // exact logits with a bias: the candidate band below the k-th key
    // estimate is twice the key's evaluation error, rounded up
    TopkArgs b = a;
    if (!(a.bias_absmax >= 0.0f)) return cudaErrorInvalidValue;
    const double key_err = kKeyErr + static_cast<double>(a.bias_absmax) * 0x1p-22;
    b.key_err = static_cast<float>(key_err);
    if (static_cast<double>(b.key_err) < key_err) b.key_err = nextafterf(b.key_err, INFINITY);
    b.band_pad = static_cast<float>(2.0 * static_cast<double>(b.key_err));
    if (static_cast<double>(b.band_pad) < 2.0 * static_cast<double>(b.key_err))
        b.band_pad = nextafterf(b.band_pad, INFINITY);
    // one CTA per token for small batches with exact logits; a batch whose
    // candidates need the exact refinement (one warp's work per token) runs a
    // warp per token, so that many tokens refine at once
    if (a.T <= kTopkWideTokens && !a.refine)
        return launch_ex(topk_wide_kernel, dim3(a.T), dim3(kTopkWideThreads), 0, s, pdl, b);
    return launch_ex(topk_kernel, dim3((a.T + kTopkWarps - 1) / kTopkWarps), dim3(kTopkWarps * 32), 0, s, pdl, b);
}

cudaError_t launch_router_norms(const float* R, const float* Rs, int E, int K, float* out, cudaStream_t s) {
    if (E <= 0 || K <= 0 || K > (1 << 17)) return cudaErrorInvalidValue;
    router_norms_kernel<<<(E * 32 + 255) / 256, 256, 0, s>>>(R, Rs, E, K, out);
    return cudaGetLastError();
}

cudaError_t launch_expert_scan(const uint32_t* sel, int E, int W, int32_t* wpre, int32_t* counts, cudaStream_t s,
                               bool pdl) {
    return launch_ex(expert_scan_kernel, dim3((E * 32 + 255) / 256), dim3(256), 0, s, pdl, sel, E, W, wpre, counts);
}

cudaError_t launch_worklist(const WorkListArgs& a, cudaStream_t s, bool pdl) {
    if (a.E > 1024) return cudaErrorInvalidValue;
    return launch_ex(worklist_kernel, dim3(1), dim3(1024), 0, s, pdl, a);
}

cudaError_t launch_scatter(const ScatterArgs& args, cudaStream_t s, bool pdl) {
    ScatterArgs a = args;
    a.slots_per_warp = (a.T >= MOE_SCATTER_SLOTS_FROM) ? MOE_SCATTER_SLOTS : 1;
    const int64_t warps = static_cast<int64_t>(a.T) * ((a.k + a.slots_per_warp - 1) / a.slots_per_warp);
    return launch_ex(scatter_kernel, dim3(static_cast<int>((warps * 32 + 255) / 256)), dim3(256), 0, s, pdl, a);
}

cudaError_t launch_combine(const float* o, const int32_t* slot_pos, const float* w, int T, int k, int L,
                           uint8_t* out_q, int64_t ld_q, uint8_t* out_sf, int64_t sf_pitch, int n_max,
                           __nv_bfloat16* out_bf, cudaStream_t s, bool pdl) {
    if (n_max <= 0 || L % 128 || k > 32 || (ld_q & 3)) return cudaErrorInvalidValue;
    dim3 grid(T, (L / 128 + kCombineWarps - 1) / kCombineWarps);
    return launch_ex(combine_kernel, grid, dim3(kCombineWarps * 32), 0, s, pdl, o, slot_pos, w, T, k, L, out_q, ld_q,
                     out_sf, sf_pitch, n_max, out_bf);
}

cudaError_t launch_mxfp4_encode(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                                cudaStream_t s) {
    const int64_t n = rows * (K / 32);
    if (n == 0) return cudaSuccess;
    mxfp4_encode_kernel<<<static_cast<unsigned>((n + 127) / 128), 128, 0, s>>>(w, rows, K, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_copy_rows(uint8_t* dst, int64_t dst_stride, const uint8_t* const* src_rows, int64_t nrows,
                             int64_t row_bytes, cudaStream_t s) {
    if (nrows == 0) return cudaSuccess;
    copy_rows_kernel<<<static_cast<unsigned>(nrows), 128, 0, s>>>(dst, dst_stride, src_rows, nrows, row_bytes);
    return cudaGetLastError();
}

cudaError_t launch_sf_atoms(const uint8_t* scales_rm, int64_t rows, int64_t kb, uint8_t* atoms, cudaStream_t s) {
    const int64_t n = rows * kb;
    sf_atoms_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(scales_rm, rows, kb, atoms);
    return cudaGetLastError();
}

cudaError_t kernels_setup() { return cudaSuccess; }

cudaError_t launch_tf32_split(const float* src, int64_t rows, int64_t K, float* dst, cudaStream_t s) {
    const int64_t n = rows * K;
    if (n == 0) return cudaSuccess;
    tf32_split_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(src, rows, K, dst);
    return cudaGetLastError();
}

cudaError_t launch_sf_item_planes(const uint8_t* scales_rm, int64_t rows, int64_t kb, uint8_t* planes, int64_t pitch,
                                  int n_max, cudaStream_t s) {
    const int64_t n = rows * kb;
    if (n == 0) return cudaSuccess;
    if (n_max <= 0) return cudaErrorInvalidValue;
    sf_item_planes_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(scales_rm, rows, kb, planes, pitch,
                                                                                 n_max);
    return cudaGetLastError();
}

cudaError_t launch_export_sf(const uint8_t* planes, int64_t pitch, const int32_t* row_map, int64_t rows,
                             int64_t nblocks, int64_t col_block0, uint8_t* out, int item_n, const int32_t* seg, int E,
                             cudaStream_t s) {
    const int64_t n = rows * nblocks;
    if (n == 0) return cudaSuccess;
    export_sf_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(planes, pitch, row_map, rows, nblocks,
                                                                          col_block0, out, item_n, seg, E);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint8_t* src, int64_t src_stride, const int32_t* row_map, int64_t rows,
                               int64_t row_bytes, uint8_t* dst, int64_t dst_stride, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    gather_rows_kernel<<<static_cast<unsigned>(rows), 128, 0, s>>>(src, src_stride, row_map, rows, row_bytes, dst,
                                                                   dst_stride);
    return cudaGetLastError();
}

}  // namespace moe
