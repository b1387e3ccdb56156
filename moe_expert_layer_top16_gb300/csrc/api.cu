// C ABI of libmoe (declared in include/moe.h): plan creation (validation,
// allocation, weight repacking, TMA descriptors), the forward pass as a fixed
// sequence of kernel launches on the caller's stream, and utilities.
//
// Forward pass (steps of the layer; see include/moe.h for the math):
//   1 quant_x       x bf16 -> MXFP8 codes + scale planes
//   2 GEMM (dense)  [P_down ; shared gate/up] x xq: z (fp32 + MXFP8) and the
//                   shared experts' SiLU-gated activation (MXFP8) in one pass
//   3 router        logits = z R^T (fp32)
//   4 top-k         expert ids, gates, per-expert token bitmaps
//   5 scan          per-expert counts / prefix popcounts
//   6 work lists    offsets (exact and 16-row padded) + grouped GEMM items
//   7 scatter       stable ranks -> permuted rows; gather zq rows
//   8 GEMM grouped  gate/up per expert segment, SiLU * up -> MXFP8
//   9 GEMM grouped  down per expert segment -> o (fp32)
//  10 combine       c = sum_j w_j o_j (slot order) -> MXFP8 into the
//                   concatenated [c | h_shared] activation buffer
//  11 GEMM (dense)  y = [cq | h_sq] [P_up | S_down]^T: the routed branch's
//                   up-projection and the shared experts' down-projection
//                   summed in one accumulator
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/moe.h"
#include "internal.h"

using namespace moe;

namespace {

// Bytes that one 128x128 MXFP4 TMA box (16U4_ALIGN16B) counts toward the
// mbarrier transaction: the packed size (128 rows x 64 B).  In shared memory
// the box occupies 16 KB -- each 16-byte chunk holds 8 bytes of packed
// elements and an 8-byte gap that the copy leaves unwritten.
// A single-group GEMM (wide items) issues its token-side copies from a warp
// of their own.
#ifndef MOE_B_PRODUCER
#define MOE_B_PRODUCER 1
#endif
// K-splits of the grouped GEMMs' narrow items (0: chosen from the items per CTA).
#ifndef MOE_GROUPED_NARROW_KS
#define MOE_GROUPED_NARROW_KS 0
#endif
// From this many tokens on, the shared experts' gate/up (the weight tiles of
// step 2 after the latent projection) runs on a stream of its own beside the
// routing steps, which leave the tensor cores idle; SMs kept free of it for
// the routing kernels.  Both parts then run on CTA pairs (the fused step 2
// has no paired instance): 1,024 tokens 0.858 -> 0.824 ms with graph replay,
// 0.872 -> 0.816 ms eager; from 512 tokens the split lost with graph replay.
#ifndef MOE_SPLIT_A2_TOKENS
#define MOE_SPLIT_A2_TOKENS 1024
#endif
#ifndef MOE_SPLIT_A2_FREE_SMS
#define MOE_SPLIT_A2_FREE_SMS 8
#endif
// Inside a stream capture (a CUDA graph) the shared experts' gate/up is
// forked after the routed down-projection instead, beside the combine (HBM-
// bound while the tensor cores idle), with this many SMs left free of it.
// Graph replay, 8,192 tokens: 2.346 -> 2.253 ms (8 free: 2.296); launched
// eagerly that order lost (2.33 -> 2.47 ms: the side kernel then started
// late), so eager forwards keep the early fork.
#ifndef MOE_SIDE_LATE_FREE_SMS
#define MOE_SIDE_LATE_FREE_SMS 32
#endif
#ifndef MOE_A_TX_BYTES
#define MOE_A_TX_BYTES 8192
#endif
// wide GEMMs of batches of at least this many tokens run on CTA pairs (0: never)
#ifndef MOE_PAIR_TOKENS
#define MOE_PAIR_TOKENS 1024
#endif
// tokens per work item at most when the GEMMs run on CTA pairs (a smaller
// item leaves room for one more shared-memory stage; 8,192 tokens: 240 2.72,
// 224 2.62, 208 2.65, 192 2.66 ms)
#ifndef MOE_PAIR_NMAX
#define MOE_PAIR_NMAX 224
#endif
// item lanes (groups) of a paired launch: step 2's dense GEMMs, step 11's,
// and the grouped ones (0: two lanes when each keeps two accumulators, else
// one); with two lanes a CTA streams two weight row blocks at once
#ifndef MOE_PAIR_GROUPS_DENSE
#define MOE_PAIR_GROUPS_DENSE 1
#endif
#ifndef MOE_PAIR_GROUPS_UP
#define MOE_PAIR_GROUPS_UP 2
#endif
#ifndef MOE_PAIR_GROUPS_GRP
#define MOE_PAIR_GROUPS_GRP 0
#endif
// the layer's step 11 runs on one lane (two K-half rings) from this many
// tokens on: 8,192 tokens 0.266 -> 0.258 ms, 32,768 1.029 -> 1.003; at 2,048
// two lanes stay ahead (0.075 vs 0.078 ms)
#ifndef MOE_PAIR_UP_ONE_LANE_FROM
#define MOE_PAIR_UP_ONE_LANE_FROM 8192
#endif
// grouped token tile of paired launches: the mean tokens per expert m plus
// this many tenths of sqrt(m) (a Poisson count's standard deviation), plus 8,
// at least 80 tokens (0: 3 m as unpaired)
#ifndef MOE_PAIR_GRP_SD10
#define MOE_PAIR_GRP_SD10 30
#endif

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// MXFP4 weights [rows][K] (packed codes), 128x128-element boxes.
bool map_mx4(CUtensorMap* m, const void* codes, int64_t rows, int64_t K) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(codes), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 matrix [rows][K] for the TF32 path: 32-wide (128-byte) x box_rows boxes.
bool map_f32(CUtensorMap* m, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 4)};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 rows of `pitch` floats viewed as [rows][K], 32-wide (128-byte) x
// box_rows boxes.
bool map_f32_view(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int64_t pitch, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch * 4)};
    cuuint32_t box[2] = {32, box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 matrix [rows][K] (rows of K elements), 64-wide (128-byte) x box_rows boxes.
bool map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MXFP8 activation codes [rows][K], 128-wide x 16-row boxes.
bool map_mx8(CUtensorMap* m, const void* codes, int64_t rows, int64_t K, int box_rows = 16) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Scale atoms or item-atom planes (bytes, a multiple of 256) as rows of 256
// bytes, boxes of box_rows rows (2 rows: one 512-byte atom): the paired GEMMs
// load their scales through these.
bool map_rows256(CUtensorMap* m, const void* base, int64_t bytes, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f || bytes % 256) return false;
    cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(bytes / 256)};
    cuuint64_t strides[1] = {256};
    cuuint32_t box[2] = {256, box_rows};
    cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int64_t rup(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

// Coefficients of the proven error bound of a tensor-core router estimate
// (TopkArgs in internal.h), for a router input of K values.
//  * Tensor-core accumulation: the products of TF32 operands are exact in
//    fp32; each one is added to the fp32 accumulator with an error of at most
//    two units in the last place of the running sum (one for aligning it to
//    the accumulator, one for rounding the sum, toward zero or to nearest),
//    and the K-split partials of the engine add a few more additions:
//    |est - sum z_hi R_hi| <= (K + 8) 2^-22 sum |z_hi| |R_hi|.
//  * The exact path's fp32 FMA chain (K/32 FMAs per lane, a 5-level
//    butterfly): at most (K/32 + 8) 2^-24 sum |z| |R|.
//  * Norms of the input rows come from fp32 sums of K squares, each chain
//    K/32 + 5 roundings long: the sums are scaled up by 2 (K/32 + 8) 2^-24.
float round_up_f(double v) {
    float f = static_cast<float>(v);
    if (static_cast<double>(f) < v) f = nextafterf(f, INFINITY);
    return f;
}
float tc_router_gamma(int K) { return round_up_f((K + 8) * 0x1p-22); }
float exact_router_gamma(int K) { return round_up_f((K / 32 + 8) * 0x1p-24); }
float router_norm_inflation(int K) { return round_up_f(1.0 + 2.0 * (K / 32 + 8) * 0x1p-24); }

// Token-bitmap words per expert up to which the work-list kernel also does the
// per-expert scan (batches of up to 128 tokens; above that one CTA scanning
// all experts costs more than the extra launch).
constexpr int kFusedScanWords = 4;

struct Plan {
    moe_config cfg;
    int device = 0, num_sms = 0;
    int D, L, E, k, I, Ip, S, Is, SIs, Kcat, rowsA2, T_max, T_pad, W_max;
    int64_t R_pad;
    size_t bytes = 0;
    std::vector<void*> allocs;
    // weights
    uint8_t *a2c, *a2sf, *w13c, *w13sf, *w2c, *w2sf, *a10c, *a10sf;
    float *router, *router2, *bias;   // router [E][RK]; router2: [E][2 RK] = TF32 high part | remainder
    float* rnorm;                     // [2][E] upper bounds of |R_e| and of |R_lo_e| (router2's remainder)
    float bias_absmax = 0.0f;
    bool has_bias = false;            // the selection bias is in use (bias holds E floats either way)
    double* qb_marg = nullptr;        // [E][T_max] margins of the Quantile Balancing update, made on first use
    int RK = 0;                       // router input width: L (latent routing) or D (hidden routing)
    bool route_hidden = false, out_bf16 = false;
    bool mixed = false;               // bf16 latent projections and shared experts (MOE_PRECISION_MIXED)
    uint16_t *a2b = nullptr, *a10b = nullptr;   // their bf16 operands, laid out as a2c / a10c
    __nv_bfloat16* act_bf = nullptr;  // [T_pad][Kcat] bf16: c | h_s (mixed precision)
    float* xr = nullptr;              // hidden routing: x as fp32 [T_pad][D]
    // workspace
    uint8_t *xq, *xsf, *zq, *zsf, *act, *actsf, *zqp, *zqpsf, *hq, *hqsf;
    float *z, *logits, *gw, *o;
    uint32_t* sel;
    int32_t *idx, *wpre, *counts, *offsets, *seg, *slot_pos, *canon_to_pad, *sorted_token;
    int32_t *ioff7, *ioff8;   // [E+1] per-expert item offsets of the grouped GEMMs
    int* status;
    void* x_stage;
    float* y_stage;
    int32_t* ep_inv;          // [T_max * k] wire row of each (token, slot) for the expert-parallel combine
    int last_T = 0;           // tokens of the last forward call (the expert-parallel dispatch reads its state)
    CUtensorMap tA2, tB2, tA7, tB7, tA8, tB8, tA10, tB10, tAR, tBR;
    // B maps with one box per wide work item (box height = that n_max),
    // re-encoded when a forward needs another height
    CUtensorMap tB2w, tB10w, tB7w, tB8w, tBRw;
    // the same MXFP8 token operands with one-row boxes (items of fewer than 16 tokens)
    CUtensorMap tB2r, tB7r, tB8r, tB10r;
    int wide_dense = 0, wide_grp = 0, wide_router = 0;
    bool tc_router;    // router logit estimates on the tensor cores (one TF32 product) above 128 tokens
    // streaming exact router of up to 128 tokens: R and router input maps,
    // and which cluster sizes this device schedules
    CUtensorMap tRS, tZS;
    bool rs16 = false, rs8 = false;
    // large batches: the shared experts' part of step 2 runs on a stream of
    // the plan's own, beside the routing steps (fork / join events)
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    // CTA pairs of the wide GEMMs: resident two-CTA clusters (0: pairs off)
    // and the scale maps of their paired copies (weights: atoms; tokens:
    // item-atom planes)
    int pair_clusters = 0;
    CUtensorMap tSA2, tSA7, tSA8, tSA10;
    // per token tile size (re-encoded when a forward needs another): each
    // CTA's half of an item's token rows, and all of the item's scale atoms
    CUtensorMap tPB2, tPB10, tPB7, tPB8, tPS2, tPS10, tPS7, tPS8;
    int pair_dense = 0, pair_grp = 0;
};

template <typename T>
cudaError_t palloc(Plan* p, T** out, size_t bytes) {
    void* ptr = nullptr;
    bytes = (bytes + 255) & ~size_t(255);
    if (bytes == 0) bytes = 256;
    cudaError_t err = cudaMalloc(&ptr, bytes);
    if (err != cudaSuccess) return err;
    err = cudaMemset(ptr, 0, bytes);
    if (err != cudaSuccess) {
        cudaFree(ptr);
        return err;
    }
    p->allocs.push_back(ptr);
    p->bytes += bytes;
    *out = static_cast<T*>(ptr);
    return cudaSuccess;
}

void plan_release(Plan* p) {
    if (!p) return;
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    for (void* a : p->allocs) cudaFree(a);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (p->ev_join) cudaEventDestroy(p->ev_join);
    if (p->side) cudaStreamDestroy(p->side);
    cudaSetDevice(cur);
    delete p;
}

struct DevGuard {
    int prev = -1;
    explicit DevGuard(int d) {
        cudaGetDevice(&prev);
        if (prev != d) cudaSetDevice(d);
    }
    ~DevGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

// Copy rows described by host-side source row pointers into dst (device).
cudaError_t copy_rows(uint8_t* dst, int64_t dst_stride, const std::vector<const uint8_t*>& rows, int64_t row_bytes) {
    if (rows.empty()) return cudaSuccess;
    const uint8_t** d_rows = nullptr;
    cudaError_t err = cudaMalloc(&d_rows, rows.size() * sizeof(void*));
    if (err != cudaSuccess) return err;
    err = cudaMemcpy(d_rows, rows.data(), rows.size() * sizeof(void*), cudaMemcpyHostToDevice);
    if (err == cudaSuccess)
        err = launch_copy_rows(dst, dst_stride, d_rows, static_cast<int64_t>(rows.size()), row_bytes, 0);
    if (err == cudaSuccess) err = cudaDeviceSynchronize();
    cudaFree(d_rows);
    return err;
}

// Repack one weight operand: `rows` destination rows, each filled from up to
// `nseg` K-segments (source row pointers for codes and scales, and the K
// width of the segment).  Produces packed codes [rows][Kp/2] and the scale
// atoms [rows/128][Kp/128][512]; columns not covered stay zero.
struct Segment {
    std::vector<const uint8_t*> code_rows, scale_rows;
    int64_t k_off, k_len;
};
cudaError_t repack(Plan* p, const std::vector<Segment>& segs, int64_t rows, int64_t Kp, uint8_t** codes_out,
                   uint8_t** atoms_out) {
    cudaError_t err = palloc(p, codes_out, static_cast<size_t>(rows * Kp / 2));
    if (err != cudaSuccess) return err;
    err = palloc(p, atoms_out, static_cast<size_t>(rows * Kp / 32));
    if (err != cudaSuccess) return err;
    uint8_t* rm = nullptr;
    err = cudaMalloc(&rm, static_cast<size_t>(rows * Kp / 32));
    if (err != cudaSuccess) return err;
    err = cudaMemset(rm, 0, static_cast<size_t>(rows * Kp / 32));
    for (const Segment& s : segs) {
        if (err != cudaSuccess) break;
        err = copy_rows(*codes_out + s.k_off / 2, Kp / 2, s.code_rows, s.k_len / 2);
        if (err == cudaSuccess) err = copy_rows(rm + s.k_off / 32, Kp / 32, s.scale_rows, s.k_len / 32);
    }
    if (err == cudaSuccess) err = launch_sf_atoms(rm, rows, Kp / 32, *atoms_out, 0);
    if (err == cudaSuccess) err = cudaDeviceSynchronize();
    cudaFree(rm);
    return err;
}

// bf16 variant of repack: rows of 2-byte elements, no scales.
cudaError_t repack_bf16(Plan* p, const std::vector<Segment>& segs, int64_t rows, int64_t Kp, uint16_t** out) {
    cudaError_t err = palloc(p, out, static_cast<size_t>(rows * Kp * 2));
    for (const Segment& s : segs) {
        if (err != cudaSuccess) break;
        err = copy_rows(reinterpret_cast<uint8_t*>(*out) + s.k_off * 2, Kp * 2, s.code_rows, s.k_len * 2);
    }
    return err;
}

moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    if (e == cudaErrorMemoryAllocation) return MOE_ERR_OOM;
    return MOE_ERR_CUDA;
}

GemmParams gemm_base(const CUtensorMap& A, const CUtensorMap& B, const uint8_t* sfa, const uint8_t* sfb,
                     int64_t sfb_pitch, int K, int n_max, int a_rows, int b_rows, int* status) {
    GemmParams g;
    std::memset(&g, 0, sizeof(g));
    g.tmA = A;
    g.tmB = B;
    g.sfa = sfa;
    g.sfb = sfb;
    g.sfb_pitch = sfb_pitch;
    g.KT = K / kBlockK;
    g.n_max = n_max;
    g.stage_bytes = gemm_stage_bytes(n_max);
    g.a_tx_bytes = MOE_A_TX_BYTES;
    g.kind = KIND_MX;
    g.kseg_tiles = g.KT;
    g.b_box = 16;
    g.a_rows = a_rows;
    g.b_rows = b_rows;
    g.status = status;
    return g;
}

// Tokens per dense work item: the batch split into equal 16-row multiples of
// at most `cap` rows.
int pick_n_max(int T, int cap = kNMax) {
    const int tiles = (T + cap - 1) / cap;
    const int per = (T + tiles - 1) / tiles;
    return static_cast<int>(rup(per, 16));
}

// Largest per-item token count at batch size T: small batches use narrow
// items (several groups, two TMEM buffers each), larger ones wide items.
int item_cap(int T) { return T <= 256 ? 48 : kNMax; }

// Groups / K-splits / accumulator buffers / stages of a GEMM launch whose
// items hold up to g.n_max tokens and span g.KT K tiles; about est_items
// items spread over `grid` CTAs; E > 0 for grouped items.
// Wide items (prefill) run one group with two accumulators: the tensor pipe
// is busy for a whole item and the epilogue overlaps the next one.  Narrow
// items are issue-bound, so four groups run side by side: as four item lanes
// when each CTA has 16 items or more, else as K-splits of fewer items (each
// split keeping at least 4 K tiles; two splits with 2..15 items per CTA
// measured faster than four lanes at 8 tokens); a CTA then takes a
// contiguous range of items, so that successive items mostly belong to one
// expert.
void shape_gemm(GemmParams& g, int E, int64_t est_items, int grid) {
    const bool narrow = g.n_max <= kNarrowMax;
    const bool xbuf = gemm_needs_xbuf(g);     // the output modes must be set before shaping
    const int64_t per_cta = std::max<int64_t>(1, (est_items + grid - 1) / std::max(grid, 1));
    int ks_max = 1;
    while (ks_max < 4 && g.KT >= 8 * ks_max) ks_max *= 2;
    for (int G = narrow ? 4 : 1; G >= 1; G >>= 1) {
        int KS = per_cta >= 16 ? 1 : (per_cta >= 2 ? 2 : 4);
        if (E > 0 && narrow && MOE_GROUPED_NARROW_KS > 0) KS = MOE_GROUPED_NARROW_KS;
        KS = std::min(std::min(KS, ks_max), G);
        for (int NB = 2; NB >= 1; --NB) {
            if (!gemm_config_ok(g.n_max, G, KS, NB)) continue;
            const int S = gemm_stages(g.n_max, G, E, xbuf);
            if (gemm_smem_bytes(g.n_max, S, E, xbuf) > static_cast<size_t>(kSmemLimit)) continue;
            g.groups = G;
            g.ksplit = KS;
            g.acc_bufs = NB;
            g.stages = S;
            g.contiguous = narrow ? 1 : 0;
            g.b_producer = (G == 1 && MOE_B_PRODUCER) ? 1 : 0;
            return;
        }
    }
    g.groups = 1;
    g.ksplit = 1;
    g.contiguous = 0;
    g.acc_bufs = 1;
    g.stages = gemm_stages(g.n_max, 1, E, xbuf);
}

// CTA pairs: an MX launch of wide items (one group, whole items, both
// producers) on two-CTA clusters whose CTAs share M = 256 MMAs, which halves
// the token rows each SM loads per weight tile.  g must carry the 16-row B map
// and its scale maps; E > 0 for grouped items.  Returns the grid (an even
// number of CTAs, at most max_grid), or 0 when the launch stays unpaired
// (g unchanged).
// Item lanes of a paired launch with items of n_max tokens.  One CTA
// streams its weights at about 24 GB/s from one 128-row block, whatever its
// stage count, and about twice that from two blocks at once; two lanes pay
// off unless each would be left with a single accumulator (the epilogue of a
// lane then stalls its MMAs), which the dense GEMMs' long items tolerate.
int pair_groups(int want, int n_max) {
    if (want > 0) return want;
    return gemm_config_ok(n_max, 2, 1, 2) ? 2 : 1;
}
// Accumulator buffers of a paired launch of G lanes with items of n_max
// tokens (0: its accumulators do not fit in TMEM).
int pair_acc_bufs(int n_max, int G) {
    for (int NB = 2; NB >= 1; --NB)
        if (gemm_config_ok(n_max, G, 1, NB)) return NB;
    return 0;
}

int shape_gemm_pair(GemmParams& g, int E, int64_t n_pairs, int max_grid, int clusters, int lanes) {
    if (clusters <= 0 || g.kind != KIND_MX || g.n_max <= kNarrowMax) return 0;
    if (g.dense ? ((g.m_tiles & 1) || (g.mt_base & 1)) : (g.mt_per_e & 1)) return 0;
    const int G = pair_groups(lanes, g.n_max);
    const int NB = pair_acc_bufs(g.n_max, G);
    if (NB == 0) return 0;
    const int64_t cl = std::min<int64_t>(std::min<int64_t>(clusters, max_grid / 2), std::max<int64_t>(n_pairs, 1));
    if (cl < 1) return 0;
    GemmParams t = g;
    t.pair = 1;
    t.groups = G;
    t.ksplit = 1;
    t.acc_bufs = NB;
    t.b_producer = G == 1 ? 1 : 0;
    t.b_box = pair_b_rows(t.n_max);
    t.b_row1 = 0;
    t.contiguous = 0;
    t.stage_bytes = gemm_stage_bytes(t.n_max, true);
    const bool xbuf = gemm_needs_xbuf(t);
    t.stages = gemm_stages(t.n_max, G, E, xbuf, true);
    if (gemm_smem_bytes(t.n_max, t.stages, E, xbuf, true) > static_cast<size_t>(kSmemLimit)) return 0;
    g = t;
    return static_cast<int>(2 * cl);
}

// The dense GEMM of the standalone entry points (moe_mx_gemm and its
// no-allocation form): items of nmax tokens, wide ones on CTA pairs where
// that applies.  The caller encodes B with dense_box_rows() rows per box and
// fills g's output description.
// Token tile of the standalone dense GEMM of N tokens and M weight rows, and
// the clusters its paired launch may use (*pair_cl = 0: unpaired).
int dense_nmax(int M, int N, int* pair_cl) {
    *pair_cl = 0;
    const int nmax = pick_n_max(N, item_cap(N));
    if (MOE_PAIR_TOKENS <= 0 || nmax <= kNarrowMax || (M / kBlockM) % 2) return nmax;
    const int pn = pick_n_max(N, std::min(item_cap(N), std::min(MOE_PAIR_NMAX, kNMax)));
    if (pn <= kNarrowMax || pair_acc_bufs(pn, pair_groups(MOE_PAIR_GROUPS_UP, pn)) == 0) return nmax;
    *pair_cl = gemm_pair_clusters();
    return *pair_cl > 0 ? pn : nmax;
}
int dense_box_rows(int nmax, int pair_cl) {
    return nmax <= kNarrowMax ? 16 : (pair_cl > 0 ? pair_b_rows(nmax) : nmax);
}
cudaError_t launch_dense_mx(GemmParams& g, int M, int N, int K, int64_t Np, int nmax, int pair_cl,
                            const uint8_t* atoms, const uint8_t* planes, int sms, cudaStream_t s) {
    if (nmax > kNarrowMax) g.b_box = dense_box_rows(nmax, pair_cl);
    g.dense = 1;
    g.m_tiles = M / kBlockM;
    g.n_tokens = N;
    g.epi_split = 1 << 30;
    const int items = g.m_tiles * ((N + nmax - 1) / nmax);
    int grid = 0;
    if (pair_cl > 0 && map_rows256(&g.tmSFA, atoms, static_cast<int64_t>(M) * K / 32, 2) &&
        map_rows256(&g.tmSFB, planes, static_cast<int64_t>(K / 128) * (Np + 32) * 16, 2 * ((nmax + 127) / 128)))
        grid = shape_gemm_pair(g, 0, items / 2, sms, pair_cl, MOE_PAIR_GROUPS_UP);
    if (!grid) {
        grid = std::min(items, sms);
        shape_gemm(g, 0, items, grid);
    }
    return launch_gemm(g, grid, s);
}

moe_status validate(const moe_config* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->d_model <= 0 || c->d_latent <= 0 || c->d_model % 128 || c->d_latent % 128) return MOE_ERR_INVALID_ARG;
    if (c->expert_inter <= 0 || c->expert_inter % 64) return MOE_ERR_INVALID_ARG;
    if (c->n_shared < 0 || (c->n_shared > 0 && (c->shared_inter <= 0 || c->shared_inter % 64)))
        return MOE_ERR_INVALID_ARG;
    if (c->n_experts < 1 || c->n_experts > 1024) return MOE_ERR_INVALID_ARG;
    if (c->top_k < 1 || c->top_k > 32 || c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
    if (c->max_tokens < 1 || c->max_tokens > 65536) return MOE_ERR_INVALID_ARG;
    if (c->score_fn != MOE_SCORE_SIGMOID_BIAS && c->score_fn != MOE_SCORE_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (c->route_input != MOE_ROUTE_ON_LATENT && c->route_input != MOE_ROUTE_ON_HIDDEN) return MOE_ERR_INVALID_ARG;
    if (c->out_dtype != MOE_OUT_F32 && c->out_dtype != MOE_OUT_BF16) return MOE_ERR_INVALID_ARG;
    if (c->precision != MOE_PRECISION_MX && c->precision != MOE_PRECISION_MIXED) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

bool mx_ok(const moe_mx4& m) { return m.codes && m.scales; }

}  // namespace

extern "C" {

const char* moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported";
        case MOE_ERR_OOM: return "out of device memory";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_TIMEOUT: return "device wait timed out";
        case MOE_ERR_DEVICE: return "device-side error";
    }
    return "unknown status";
}

moe_status moe_plan(const moe_config* cfg, const moe_weights* w, int device, void** plan_out) {
    if (!plan_out) return MOE_ERR_INVALID_ARG;
    *plan_out = nullptr;
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const bool mixed = cfg->precision == MOE_PRECISION_MIXED;
    if (!w || !mx_ok(w->w_gate) || !mx_ok(w->w_up) || !mx_ok(w->w_down) || !w->router_w) return MOE_ERR_INVALID_ARG;
    if (mixed ? (!w->p_down_bf16 || !w->p_up_bf16) : (!mx_ok(w->p_down) || !mx_ok(w->p_up))) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && (mixed ? (!w->s_gate_bf16 || !w->s_up_bf16 || !w->s_down_bf16)
                                    : (!mx_ok(w->s_gate) || !mx_ok(w->s_up) || !mx_ok(w->s_down))))
        return MOE_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_ERR_UNSUPPORTED;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MOE_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MOE_ERR_UNSUPPORTED;
    if (!encode_fn()) return MOE_ERR_UNSUPPORTED;

    DevGuard guard(device);
    Plan* p = new (std::nothrow) Plan();
    if (!p) return MOE_ERR_OOM;
    p->cfg = *cfg;
    p->device = device;
    p->num_sms = prop.multiProcessorCount;
    p->D = cfg->d_model;
    p->L = cfg->d_latent;
    p->E = cfg->n_experts;
    p->k = cfg->top_k;
    p->I = cfg->expert_inter;
    p->Ip = static_cast<int>(rup(p->I, 128));
    p->S = cfg->n_shared;
    p->Is = p->S > 0 ? cfg->shared_inter : 0;
    p->SIs = p->S * p->Is;
    p->Kcat = static_cast<int>(rup(p->L + p->SIs, 128));
    p->rowsA2 = p->L + 2 * p->SIs;
    p->T_max = cfg->max_tokens;
    p->T_pad = static_cast<int>(rup(p->T_max, 16));
    p->W_max = (p->T_max + 31) / 32;
    p->R_pad = rup(static_cast<int64_t>(p->T_max) * p->k + 15LL * p->E, 16);

    cudaError_t err = gemm_setup();
    if (err == cudaSuccess) err = kernels_setup();
    const int D = p->D, L = p->L, E = p->E, I = p->I, Ip = p->Ip, S = p->S, Is = p->Is;
    const int64_t Tp = p->T_pad, Rp = p->R_pad;
#define TRY(x)                          \
    do {                                \
        if (err == cudaSuccess) err = (x); \
    } while (0)
    // ---------------------------------------------------------------- weights
    p->mixed = mixed;
    if (mixed) {
        // the same row order in bf16: P_down, then per shared expert 128-row
        // tiles of 64 gate rows and the 64 matching up rows
        Segment s;
        s.k_off = 0;
        s.k_len = D;
        for (int r = 0; r < p->rowsA2; ++r) {
            const uint16_t* c;
            if (r < L) {
                c = w->p_down_bf16 + static_cast<int64_t>(r) * D;
            } else {
                const int rr = r - L, sh = rr / (2 * Is), within = rr % (2 * Is);
                const int t = within / 128, h = within % 128;
                const uint16_t* src = (h < 64) ? w->s_gate_bf16 : w->s_up_bf16;
                c = src + (static_cast<int64_t>(sh) * Is + 64 * t + (h % 64)) * D;
            }
            s.code_rows.push_back(reinterpret_cast<const uint8_t*>(c));
        }
        TRY(repack_bf16(p, {s}, p->rowsA2, D, &p->a2b));
    } else {
        // A2: rows [0, L) = P_down; then per shared expert, 128-row tiles of
        // 64 gate rows followed by the 64 matching up rows.
        Segment s;
        s.k_off = 0;
        s.k_len = D;
        for (int r = 0; r < p->rowsA2; ++r) {
            const uint8_t *c, *sc;
            if (r < L) {
                c = w->p_down.codes + static_cast<int64_t>(r) * (D / 2);
                sc = w->p_down.scales + static_cast<int64_t>(r) * (D / 32);
            } else {
                const int rr = r - L, sh = rr / (2 * Is), within = rr % (2 * Is);
                const int t = within / 128, h = within % 128;
                const moe_mx4& src = (h < 64) ? w->s_gate : w->s_up;
                const int64_t srow = static_cast<int64_t>(sh) * Is + 64 * t + (h % 64);
                c = src.codes + srow * (D / 2);
                sc = src.scales + srow * (D / 32);
            }
            s.code_rows.push_back(c);
            s.scale_rows.push_back(sc);
        }
        TRY(repack(p, {s}, p->rowsA2, D, &p->a2c, &p->a2sf));
    }
    {
        // W13: per expert, 128-row tiles of 64 gate rows + the 64 matching up rows.
        Segment s;
        s.k_off = 0;
        s.k_len = L;
        const int64_t rows = static_cast<int64_t>(E) * 2 * I;
        s.code_rows.reserve(rows);
        s.scale_rows.reserve(rows);
        for (int64_t r = 0; r < rows; ++r) {
            const int64_t e = r / (2 * I), within = r % (2 * I), t = within / 128, h = within % 128;
            const moe_mx4& src = (h < 64) ? w->w_gate : w->w_up;
            const int64_t srow = e * I + 64 * t + (h % 64);
            s.code_rows.push_back(src.codes + srow * (L / 2));
            s.scale_rows.push_back(src.scales + srow * (L / 32));
        }
        TRY(repack(p, {s}, rows, L, &p->w13c, &p->w13sf));
    }
    {
        // W2: [E*L][Ip], K zero-padded from I to a multiple of 128.
        Segment s;
        s.k_off = 0;
        s.k_len = I;
        const int64_t rows = static_cast<int64_t>(E) * L;
        for (int64_t r = 0; r < rows; ++r) {
            s.code_rows.push_back(w->w_down.codes + r * (I / 2));
            s.scale_rows.push_back(w->w_down.scales + r * (I / 32));
        }
        TRY(repack(p, {s}, rows, Ip, &p->w2c, &p->w2sf));
    }
    if (mixed) {
        // A10 in bf16: [D][Kcat] = [P_up | S_down[0] | S_down[1] | ...] along K
        std::vector<Segment> segs(1 + S);
        segs[0].k_off = 0;
        segs[0].k_len = L;
        for (int d = 0; d < D; ++d)
            segs[0].code_rows.push_back(reinterpret_cast<const uint8_t*>(w->p_up_bf16 + static_cast<int64_t>(d) * L));
        for (int sh = 0; sh < S; ++sh) {
            Segment& g = segs[1 + sh];
            g.k_off = L + static_cast<int64_t>(sh) * Is;
            g.k_len = Is;
            for (int d = 0; d < D; ++d)
                g.code_rows.push_back(
                    reinterpret_cast<const uint8_t*>(w->s_down_bf16 + (static_cast<int64_t>(sh) * D + d) * Is));
        }
        TRY(repack_bf16(p, segs, D, p->Kcat, &p->a10b));
    } else {
        // A10: [D][Kcat] = [P_up | S_down[0] | S_down[1] | ...] along K.
        std::vector<Segment> segs(1 + S);
        segs[0].k_off = 0;
        segs[0].k_len = L;
        for (int d = 0; d < D; ++d) {
            segs[0].code_rows.push_back(w->p_up.codes + static_cast<int64_t>(d) * (L / 2));
            segs[0].scale_rows.push_back(w->p_up.scales + static_cast<int64_t>(d) * (L / 32));
        }
        for (int sh = 0; sh < S; ++sh) {
            Segment& g = segs[1 + sh];
            g.k_off = L + static_cast<int64_t>(sh) * Is;
            g.k_len = Is;
            for (int d = 0; d < D; ++d) {
                const int64_t srow = static_cast<int64_t>(sh) * D + d;
                g.code_rows.push_back(w->s_down.codes + srow * (Is / 2));
                g.scale_rows.push_back(w->s_down.scales + srow * (Is / 32));
            }
        }
        TRY(repack(p, segs, D, p->Kcat, &p->a10c, &p->a10sf));
    }
    p->route_hidden = cfg->route_input == MOE_ROUTE_ON_HIDDEN;
    p->out_bf16 = cfg->out_dtype == MOE_OUT_BF16;
    p->RK = p->route_hidden ? D : L;
    const int RK = p->RK;
    TRY(palloc(p, &p->router, sizeof(float) * E * RK));
    TRY(cudaMemcpy(p->router, w->router_w, sizeof(float) * E * RK, cudaMemcpyDeviceToDevice));
    TRY(palloc(p, &p->router2, sizeof(float) * E * 2 * RK));
    TRY(launch_tf32_split(p->router, E, RK, p->router2, 0));
    TRY(palloc(p, &p->rnorm, sizeof(float) * 2 * E));
    TRY(launch_router_norms(p->router, p->router2, E, RK, p->rnorm, 0));
    TRY(cudaDeviceSynchronize());
    TRY(palloc(p, &p->bias, sizeof(float) * E));
    if (w->router_bias) {
        p->has_bias = true;
        TRY(cudaMemcpy(p->bias, w->router_bias, sizeof(float) * E, cudaMemcpyDeviceToDevice));
        std::vector<float> hb(E);
        TRY(cudaMemcpy(hb.data(), w->router_bias, sizeof(float) * E, cudaMemcpyDeviceToHost));
        if (err == cudaSuccess)
            for (float b : hb) p->bias_absmax = std::max(p->bias_absmax, b == b ? std::fabs(b) : INFINITY);
    }
    // ---------------------------------------------------------------- workspace
    TRY(palloc(p, &p->xq, Tp * D));
    // token-operand scales of the GEMMs: item-atom planes with 32 spare slots
    TRY(palloc(p, &p->xsf, (D / 128) * (Tp + 32) * 16));
    TRY(palloc(p, &p->z, sizeof(float) * Tp * 2 * L));     // TF32 high part | fp32 value (plain: the value first)
    if (p->route_hidden) TRY(palloc(p, &p->xr, sizeof(float) * Tp * D));
    TRY(palloc(p, &p->zq, Tp * L));
    TRY(palloc(p, &p->zsf, (L / 128) * Tp * 4));
    TRY(palloc(p, &p->act, Tp * p->Kcat));
    TRY(palloc(p, &p->actsf, (p->Kcat / 128) * (Tp + 32) * 16));
    if (mixed) TRY(palloc(p, &p->act_bf, Tp * p->Kcat * 2));
    TRY(palloc(p, &p->logits, sizeof(float) * p->T_max * E));
    TRY(palloc(p, &p->idx, sizeof(int32_t) * p->T_max * p->k));
    TRY(palloc(p, &p->gw, sizeof(float) * p->T_max * p->k));
    TRY(palloc(p, &p->sel, sizeof(uint32_t) * E * p->W_max));
    TRY(palloc(p, &p->wpre, sizeof(int32_t) * E * p->W_max));
    TRY(palloc(p, &p->counts, sizeof(int32_t) * E));
    TRY(palloc(p, &p->offsets, sizeof(int32_t) * (E + 1)));
    TRY(palloc(p, &p->seg, sizeof(int32_t) * (E + 1)));
    TRY(palloc(p, &p->slot_pos, sizeof(int32_t) * p->T_max * p->k));
    TRY(palloc(p, &p->canon_to_pad, sizeof(int32_t) * p->T_max * p->k));
    TRY(palloc(p, &p->sorted_token, sizeof(int32_t) * p->T_max * p->k));
    TRY(palloc(p, &p->zqp, Rp * L));
    TRY(palloc(p, &p->zqpsf, (L / 128) * (Rp + 32) * 16));
    TRY(palloc(p, &p->hq, Rp * Ip));
    TRY(palloc(p, &p->hqsf, (Ip / 128) * (Rp + 32) * 16));
    TRY(palloc(p, &p->o, sizeof(float) * Rp * L));
    TRY(palloc(p, &p->ioff7, sizeof(int32_t) * (E + 1)));
    TRY(palloc(p, &p->ioff8, sizeof(int32_t) * (E + 1)));
    TRY(palloc(p, &p->status, sizeof(int) * 4));
    TRY(palloc(p, &p->ep_inv, sizeof(int32_t) * p->T_max * p->k));
    TRY(palloc(p, &p->x_stage, sizeof(uint16_t) * p->T_max * D));
    TRY(palloc(p, &p->y_stage, sizeof(float) * p->T_max * D));
#undef TRY
    if (err != cudaSuccess) {
        st = cuda_status(err);
        plan_release(p);
        return st;
    }
    // ---------------------------------------------------------------- TMA descriptors
    bool ok = (mixed ? map_bf16(&p->tA2, p->a2b, p->rowsA2, D, 128)
                     : (map_mx4(&p->tA2, p->a2c, p->rowsA2, D) && map_mx8(&p->tB2, p->xq, Tp, D))) &&
              map_mx4(&p->tA7, p->w13c, static_cast<int64_t>(E) * 2 * I, L) && map_mx8(&p->tB7, p->zqp, Rp, L) &&
              map_mx4(&p->tA8, p->w2c, static_cast<int64_t>(E) * L, Ip) && map_mx8(&p->tB8, p->hq, Rp, Ip) &&
              (mixed ? (map_bf16(&p->tA10, p->a10b, D, p->Kcat, 128) && map_bf16(&p->tB10, p->act_bf, Tp, p->Kcat, 16))
                     : (map_mx4(&p->tA10, p->a10c, D, p->Kcat) && map_mx8(&p->tB10, p->act, Tp, p->Kcat))) &&
              map_mx8(&p->tB2r, p->xq, Tp, D, 1) && map_mx8(&p->tB7r, p->zqp, Rp, L, 1) &&
              map_mx8(&p->tB8r, p->hq, Rp, Ip, 1) && map_mx8(&p->tB10r, p->act, Tp, p->Kcat, 1) &&
              map_f32(&p->tAR, p->router2, E, 2 * p->RK, 128) &&
              (p->route_hidden ? map_f32(&p->tBR, p->xr, Tp, D, 16) : map_f32(&p->tBR, p->z, Tp, 2 * L, 16));
    p->tc_router = (E % 128 == 0) && (p->RK % 32 == 0);
    if (ok && !mixed && MOE_PAIR_TOKENS > 0 && p->T_max >= MOE_PAIR_TOKENS) {
        p->pair_clusters = gemm_pair_clusters();
        if (p->pair_clusters > 0)
            ok = map_rows256(&p->tSA2, p->a2sf, static_cast<int64_t>(p->rowsA2) * D / 32, 2) &&
                 map_rows256(&p->tSA7, p->w13sf, static_cast<int64_t>(E) * 2 * I * L / 32, 2) &&
                 map_rows256(&p->tSA8, p->w2sf, static_cast<int64_t>(E) * L * Ip / 32, 2) &&
                 map_rows256(&p->tSA10, p->a10sf, static_cast<int64_t>(D) * p->Kcat / 32, 2);
    }
    if (ok && router_stream_ok(p->RK) && router_stream_setup() == cudaSuccess) {
        ok = map_f32_view(&p->tRS, p->router, E, p->RK, p->RK, 128) &&
             (p->route_hidden ? map_f32_view(&p->tZS, p->xr, Tp, D, D, 64)
                              : map_f32_view(&p->tZS, p->z, Tp, L, 2 * L, 64));
        p->rs16 = router_stream_max_clusters(16) > 0;
        p->rs8 = router_stream_max_clusters(8) > 0;
    }
    if (ok && p->T_max >= MOE_SPLIT_A2_TOKENS && !mixed)
        ok = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        plan_release(p);
        return MOE_ERR_CUDA;
    }
    *plan_out = p;
    return MOE_OK;
}

moe_status moe_forward(void* plan, const void* x, int32_t T, void* y, void* stream, const moe_debug* dbg) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p || !x || !y) return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > p->T_max) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & (p->out_bf16 ? 1 : 3)))
        return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int D = p->D, L = p->L, E = p->E, k = p->k, I = p->I, Ip = p->Ip;
    const int W = (T + 31) / 32;
    const int64_t Tp = p->T_pad, Rp = p->R_pad;
    const int64_t Tps = Tp + 32, Rps = Rp + 32;   // slots per item-atom scale plane
    // dense GEMMs stream their weights once per token tile: a batch of up to
    // 64 tokens is one tile
    // wide GEMMs on CTA pairs from MOE_PAIR_TOKENS tokens on (their items
    // hold up to MOE_PAIR_NMAX tokens)
    const bool pair_on = p->pair_clusters > 0 && T >= MOE_PAIR_TOKENS;
    const int cap = pair_on ? std::min(MOE_PAIR_NMAX, kNMax) : kNMax;
    const int nmax_dense = (T <= 64) ? static_cast<int>(rup(T, 16)) : pick_n_max(T, std::min(item_cap(T), cap));
    // grouped token tile: about 3x the mean tokens per expert, 16..cap
    const int64_t per_expert = (static_cast<int64_t>(T) * k + E - 1) / E;
    int64_t grp_want = 3 * per_expert;
    if (pair_on && MOE_PAIR_GRP_SD10 > 0)
        grp_want = std::max<int64_t>(80, per_expert + 8 +
                                             static_cast<int64_t>(std::ceil(MOE_PAIR_GRP_SD10 * 0.1 *
                                                                            std::sqrt(static_cast<double>(per_expert)))));
    const int nmax_grp = static_cast<int>(std::min<int64_t>(std::min<int64_t>(std::max<int64_t>(rup(grp_want, 16), 16), cap),
                                                            rup(T, 16)));
    // experts expected to receive tokens (all of them once T * k >> E)
    const int64_t est_experts = std::min<int64_t>(E, static_cast<int64_t>(T) * k);
    // wide items load their token rows with one TMA box (height n_max)
    const bool wide_d = nmax_dense > kNarrowMax, wide_g = nmax_grp > kNarrowMax;
    if (wide_d && p->wide_dense != nmax_dense) {
        p->wide_dense = 0;
        const bool ok = p->mixed ? map_bf16(&p->tB10w, p->act_bf, Tp, p->Kcat, nmax_dense)
                                 : (map_mx8(&p->tB2w, p->xq, Tp, D, nmax_dense) &&
                                    map_mx8(&p->tB10w, p->act, Tp, p->Kcat, nmax_dense));
        if (!ok) return MOE_ERR_CUDA;
        p->wide_dense = nmax_dense;
    }
    // mixed precision: the down-projection and shared gate/up read x itself (bf16)
    CUtensorMap tx;
    if (p->mixed && !map_bf16(&tx, x, T, D, wide_d ? nmax_dense : 16)) return MOE_ERR_CUDA;
    if (wide_g && p->wide_grp != nmax_grp) {
        p->wide_grp = 0;
        if (!map_mx8(&p->tB7w, p->zqp, Rp, L, nmax_grp) || !map_mx8(&p->tB8w, p->hq, Rp, Ip, nmax_grp))
            return MOE_ERR_CUDA;
        p->wide_grp = nmax_grp;
    }
    // router estimate token tiles: 64 rows up to 1024 tokens (more work items
    // for the few expert tiles), else the dense tile with one B box per item
    const int nmax_router = (T <= 1024) ? 64 : nmax_dense;
    if (p->tc_router && T > 128 && nmax_router > kNarrowMax && p->wide_router != nmax_router) {
        p->wide_router = 0;
        const bool ok = p->route_hidden ? map_f32(&p->tBRw, p->xr, Tp, D, nmax_router)
                                        : map_f32(&p->tBRw, p->z, Tp, 2 * L, nmax_router);
        if (!ok) return MOE_ERR_CUDA;
        p->wide_router = nmax_router;
    }
    // above 128 tokens the router logits are tensor-core estimates from the
    // TF32 head of z (the rows keep the fp32 values beside it for the exact
    // refinement); smaller batches keep z plain
    const bool z_split = p->tc_router && T > 128;
    // large batches run step 2 as two GEMMs over the same x: the latent
    // projection, then the shared experts' gate/up.  The second runs on the
    // side stream beside the routing steps, or, while per-stage events are
    // recorded (which time the steps one by one), right after the first on
    // the caller's stream: the same kernels either way.
    const bool split_a2 = p->side != nullptr && T >= MOE_SPLIT_A2_TOKENS;
    const bool side_a2 = split_a2 && !(dbg && dbg->stage_events);
    cudaStreamCaptureStatus capst = cudaStreamCaptureStatusNone;
    const bool late_fork = side_a2 && cudaStreamIsCapturing(s, &capst) == cudaSuccess && capst == cudaStreamCaptureStatusActive;
    GemmParams a2s;
    int a2s_grid = 0;
    cudaError_t err = cudaSuccess;
#define TRY(x)                          \
    do {                                \
        if (err == cudaSuccess) err = (x); \
    } while (0)
    cudaEvent_t* ev = (dbg && dbg->stage_events) ? reinterpret_cast<cudaEvent_t*>(dbg->stage_events) : nullptr;
    auto mark = [&](int i) {
        if (ev && err == cudaSuccess) err = cudaEventRecord(ev[i], s);
    };
    // the selection bitmaps are cleared by the quantiser, the first kernel of
    // the forward; without it (bf16 projections, latent routing) by a memset
    const bool run_quant_x = !p->mixed || p->route_hidden;
    if (!run_quant_x) TRY(cudaMemsetAsync(p->sel, 0, sizeof(uint32_t) * E * W, s));
    // Kernels after the first are launched with programmatic serialization:
    // each may start while its predecessor drains and waits for it on the
    // device (pdl_wait).  Measured on GB300: every kernel gains up to 128
    // tokens; above that only the GEMMs do (their prologue is long and their
    // CTAs cannot share an SM with a running GEMM), while the small
    // many-CTA kernels launched early slowed the GEMMs they wait behind.  The
    // first kernel follows the memset with a plain launch; with per-stage
    // events every launch is plain.
    bool first_kernel = true;
    // wide GEMMs on CTA pairs: the copy of g with the pair's token and scale
    // maps, if it pairs; returns its grid or 0
    if (pair_on && wide_d && p->pair_dense != nmax_dense) {
        p->pair_dense = 0;
        const uint32_t sb = 2 * ((nmax_dense + 127) / 128);
        if (!map_mx8(&p->tPB2, p->xq, Tp, D, pair_b_rows(nmax_dense)) ||
            !map_mx8(&p->tPB10, p->act, Tp, p->Kcat, pair_b_rows(nmax_dense)) ||
            !map_rows256(&p->tPS2, p->xsf, static_cast<int64_t>(D / 128) * Tps * 16, sb) ||
            !map_rows256(&p->tPS10, p->actsf, static_cast<int64_t>(p->Kcat / 128) * Tps * 16, sb))
            return MOE_ERR_CUDA;
        p->pair_dense = nmax_dense;
    }
    if (pair_on && wide_g && p->pair_grp != nmax_grp) {
        p->pair_grp = 0;
        const uint32_t sb = 2 * ((nmax_grp + 127) / 128);
        if (!map_mx8(&p->tPB7, p->zqp, Rp, L, pair_b_rows(nmax_grp)) ||
            !map_mx8(&p->tPB8, p->hq, Rp, Ip, pair_b_rows(nmax_grp)) ||
            !map_rows256(&p->tPS7, p->zqpsf, static_cast<int64_t>(L / 128) * Rps * 16, sb) ||
            !map_rows256(&p->tPS8, p->hqsf, static_cast<int64_t>(Ip / 128) * Rps * 16, sb))
            return MOE_ERR_CUDA;
        p->pair_grp = nmax_grp;
    }
    auto try_pair = [&](GemmParams& g, const CUtensorMap& b16, const CUtensorMap& msfa, const CUtensorMap& msfb,
                        int E_tab, int64_t n_pairs, int max_grid, int lanes) -> int {
        if (!pair_on) return 0;
        GemmParams t = g;
        t.tmB = b16;
        t.tmSFA = msfa;
        t.tmSFB = msfb;
        const int grid = shape_gemm_pair(t, E_tab, n_pairs, max_grid, p->pair_clusters, lanes);
        if (grid) g = t;
        return grid;
    };
    auto pdl = [&](bool gemm) {
        const bool r = !first_kernel && ev == nullptr && (gemm || T <= 128);
        first_kernel = false;
        return r;
    };
    mark(0);
    // 1. x -> MXFP8 (and x as fp32 for hidden routing); mixed precision reads
    // x as it is, so only hidden routing needs this step
    if (run_quant_x)
        TRY(launch_quant_x(static_cast<const __nv_bfloat16*>(x), T, D, p->xq, p->xsf, Tps, nmax_dense, p->xr, p->sel,
                           static_cast<int64_t>(E) * W, s, pdl(false)));
    mark(1);
    // 2. latent down-projection + shared gate/up
    {
        GemmParams g = gemm_base(p->tA2, p->tB2, p->a2sf, p->xsf, Tps, D, nmax_dense, p->rowsA2, static_cast<int>(Tp),
                                 p->status);
        if (wide_d) {
            g.tmB = p->tB2w;
            g.b_box = nmax_dense;
        }
        if (!wide_d) {
            g.tmB1 = p->tB2r;
            g.b_row1 = 1;
        }
        if (p->mixed) {
            g.b_row1 = 0;
            g.tmB = tx;
            g.kind = KIND_BF16;
            g.KT = D / 64;
            g.kseg_tiles = g.KT;
            g.sfa = nullptr;
            g.sfb = nullptr;
        }
        g.dense = 1;
        g.m_tiles = split_a2 ? L / kBlockM : p->rowsA2 / kBlockM;
        g.n_tokens = T;
        g.epi_split = L / kBlockM;
        // z rows: for the TF32 router estimate the values' TF32 head, then the
        // values themselves at column L; else the values only
        g.epi[0] = EpiParams{EPI_QUANT, 0, 0, z_split ? L : 0, p->z, 2 * L, p->zq, L, p->zsf, Tp};
        g.epi[1] = p->mixed ? EpiParams{EPI_SILU_BF16, L / kBlockM, L, 0, nullptr, 0,
                                        reinterpret_cast<uint8_t*>(p->act_bf), p->Kcat, nullptr, 0, 0}
                            : EpiParams{EPI_SILU_QUANT, L / kBlockM, L, 0, nullptr, 0, p->act, p->Kcat, p->actsf, Tps, 1};
        if (split_a2) {
            // the shared experts' tiles, launched on the side stream after the router
            a2s = g;
            a2s.mt_base = L / kBlockM;
            a2s.m_tiles = p->rowsA2 / kBlockM - L / kBlockM;
            const int items_s = a2s.m_tiles * ((T + a2s.n_max - 1) / a2s.n_max);
            a2s_grid = std::max(1, std::min(items_s, p->num_sms - (late_fork ? MOE_SIDE_LATE_FREE_SMS : MOE_SPLIT_A2_FREE_SMS)));
            const int pg = try_pair(a2s, p->tPB2, p->tSA2, p->tPS2, 0, items_s / 2, a2s_grid, MOE_PAIR_GROUPS_DENSE);
            if (pg)
                a2s_grid = pg;
            else
                shape_gemm(a2s, 0, items_s, a2s_grid);
        }
        const int items = g.m_tiles * ((T + g.n_max - 1) / g.n_max);
        int grid = split_a2 ? try_pair(g, p->tPB2, p->tSA2, p->tPS2, 0, items / 2, p->num_sms, MOE_PAIR_GROUPS_DENSE) : 0;
        if (!grid) {
            grid = std::min(items, p->num_sms);
            shape_gemm(g, 0, items, grid);
        }
        TRY(launch_gemm(g, grid, s, pdl(true)));
        if (split_a2 && !side_a2) TRY(launch_gemm(a2s, a2s_grid, s, false));
    }
    // 3. router logits, 4. top-k + gates + bitmaps
    mark(2);
    const bool tc_logits = z_split;
    if (tc_logits) {
        // estimated logits = z_hi R_hi, one TF32 product on the tensor cores
        // (the high parts sit at the start of each row of z and router2; for
        // hidden routing x is bf16, so its TF32 value is x itself)
        const int RK = p->RK;
        GemmParams g = gemm_base(p->tAR, p->tBR, nullptr, nullptr, 0, RK * 4, nmax_router, E,
                                 static_cast<int>(Tp), p->status);
        if (nmax_router > kNarrowMax) {
            g.tmB = p->tBRw;
            g.b_box = nmax_router;
        }
        g.kind = KIND_TF32;
        g.KT = RK / 32;
        g.kseg_tiles = RK / 32;
        g.dense = 1;
        g.m_tiles = E / kBlockM;
        g.n_tokens = T;
        g.epi_split = 1 << 30;
        g.epi[0] = EpiParams{EPI_F32, 0, 0, 0, p->logits, E, nullptr, 0, nullptr, 0};
        const int items = g.m_tiles * ((T + g.n_max - 1) / g.n_max);
        shape_gemm(g, 0, items, std::min(items, p->num_sms));
        TRY(launch_gemm(g, std::min(items, p->num_sms), s, pdl(true)));
    } else if (T <= 128 && (T <= 64 ? p->rs16 : p->rs8)) {
        TRY(launch_router_stream(p->tRS, p->tZS, p->logits, T, E, p->RK, T <= 64 ? 16 : 8, p->status, s, pdl(false)));
    } else {
        if (p->route_hidden)
            TRY(launch_router(p->xr, D, 0, p->router, p->logits, T, E, D, s, pdl(false)));
        else
            TRY(launch_router(p->z, 2 * L, 0, p->router, p->logits, T, E, L, s, pdl(false)));
    }
    auto launch_a2s = [&]() {
        TRY(cudaStreamWaitEvent(p->side, p->ev_fork, 0));
        TRY(launch_gemm(a2s, a2s_grid, p->side, false));
        TRY(cudaEventRecord(p->ev_join, p->side));
    };
    if (side_a2 && !late_fork) {
        TRY(cudaEventRecord(p->ev_fork, s));
        launch_a2s();
    }
    mark(3);
    {
        TopkArgs a{};
        a.logits = p->logits;
        a.bias = p->has_bias ? p->bias : nullptr;
        a.T = T;
        a.E = E;
        a.k = k;
        a.softmax = p->cfg.score_fn == MOE_SCORE_SOFTMAX;
        a.refine = tc_logits ? 1 : 0;
        // hidden routing reads x, which is bf16 and so exactly TF32: no remainder
        a.z = p->route_hidden ? p->xr : p->z;
        a.z_ld = p->route_hidden ? D : 2 * L;
        a.z_lo = p->route_hidden ? 0 : L;
        a.R = p->router;
        a.rnorm = p->rnorm;
        a.g_tc = tc_router_gamma(p->RK);
        a.g_32 = exact_router_gamma(p->RK);
        a.sq_infl = router_norm_inflation(p->RK);
        a.bias_absmax = p->bias_absmax;
        a.L = p->RK;
        a.idx = p->idx;
        a.w = p->gw;
        a.sel = p->sel;
        a.W = W;
        TRY(launch_topk(a, s, pdl(false)));
    }
    // 5. per-expert prefix counts, 6. offsets + work lists
    mark(4);
    const bool fused_scan = W <= kFusedScanWords;     // small batches: one launch for scan + work lists
    if (!fused_scan) TRY(launch_expert_scan(p->sel, E, W, p->wpre, p->counts, s, pdl(false)));
    mark(5);
    {
        WorkListArgs a;
        a.counts = p->counts;
        a.E = E;
        a.sel = fused_scan ? p->sel : nullptr;
        a.W = W;
        a.wpre = p->wpre;
        a.counts_out = p->counts;
        a.offsets = p->offsets;
        a.seg = p->seg;
        a.ioff1 = p->ioff7;
        a.n_max1 = nmax_grp;
        a.mt1 = 2 * I / kBlockM;
        a.ioff2 = p->ioff8;
        a.n_max2 = nmax_grp;
        a.mt2 = L / kBlockM;
        TRY(launch_worklist(a, s, pdl(false)));
    }
    // 7. stable ranks, permuted rows, gather of zq
    mark(6);
    {
        ScatterArgs a;
        a.idx = p->idx;
        a.T = T;
        a.k = k;
        a.W = W;
        a.sel = p->sel;
        a.wpre = p->wpre;
        a.offsets = p->offsets;
        a.seg = p->seg;
        a.slot_pos = p->slot_pos;
        a.canon_to_pad = p->canon_to_pad;
        a.sorted_token = p->sorted_token;
        a.zq = p->zq;
        a.zsf = p->zsf;
        a.zsf_pitch = Tp;
        a.L = L;
        a.zq_perm = p->zqp;
        a.zq_perm_sf = p->zqpsf;
        a.perm_pitch = Rps;
        a.n_max = nmax_grp;
        TRY(launch_scatter(a, s, pdl(false)));
    }
    // 8. routed gate/up + SiLU -> MXFP8
    mark(7);
    {
        GemmParams g = gemm_base(p->tA7, p->tB7, p->w13sf, p->zqpsf, Rps, L, nmax_grp, E * 2 * I,
                                 static_cast<int>(Rp), p->status);
        if (wide_g) {
            g.tmB = p->tB7w;
            g.b_box = nmax_grp;
        } else {
            g.tmB1 = p->tB7r;
            g.b_row1 = 1;
        }
        g.dense = 0;
        g.ioff = p->ioff7;
        g.seg = p->seg;
        g.counts = p->counts;
        g.E = E;
        g.mt_per_e = 2 * I / kBlockM;
        g.rows_per_e = 2 * I;
        g.epi[0] = EpiParams{EPI_SILU_QUANT, 0, 0, 0, nullptr, 0, p->hq, Ip, p->hqsf, Rps, 1};
        int grid = try_pair(g, p->tPB7, p->tSA7, p->tPS7, E, est_experts * g.mt_per_e / 2, p->num_sms, MOE_PAIR_GROUPS_GRP);
        if (!grid) {
            grid = p->num_sms;
            shape_gemm(g, E, est_experts * g.mt_per_e, grid);
        }
        TRY(launch_gemm(g, grid, s, pdl(true)));
    }
    // 9. routed down -> o
    mark(8);
    {
        GemmParams g = gemm_base(p->tA8, p->tB8, p->w2sf, p->hqsf, Rps, Ip, nmax_grp, E * L, static_cast<int>(Rp),
                                 p->status);
        if (wide_g) {
            g.tmB = p->tB8w;
            g.b_box = nmax_grp;
        } else {
            g.tmB1 = p->tB8r;
            g.b_row1 = 1;
        }
        g.dense = 0;
        g.ioff = p->ioff8;
        g.seg = p->seg;
        g.counts = p->counts;
        g.E = E;
        g.mt_per_e = L / kBlockM;
        g.rows_per_e = L;
        g.epi[0] = EpiParams{EPI_F32, 0, 0, 0, p->o, L, nullptr, 0, nullptr, 0};
        int grid = try_pair(g, p->tPB8, p->tSA8, p->tPS8, E, est_experts * g.mt_per_e / 2, p->num_sms, MOE_PAIR_GROUPS_GRP);
        if (!grid) {
            grid = p->num_sms;
            shape_gemm(g, E, est_experts * g.mt_per_e, grid);
        }
        TRY(launch_gemm(g, grid, s, pdl(true)));
    }
    // 10. weighted combine -> MXFP8 into columns [0, L) of the concatenated activation
    if (late_fork) {
        TRY(cudaEventRecord(p->ev_fork, s));
        launch_a2s();
    }
    mark(9);
    TRY(launch_combine(p->o, p->slot_pos, p->gw, T, k, L, p->act, p->Kcat, p->actsf, Tps, nmax_dense, p->act_bf, s,
                       pdl(false)));
    // 11. y = [cq | h_sq] [P_up | S_down]^T
    mark(10);
    if (side_a2) TRY(cudaStreamWaitEvent(s, p->ev_join, 0));
    {
        GemmParams g = gemm_base(p->tA10, p->tB10, p->a10sf, p->actsf, Tps, p->Kcat, nmax_dense, D,
                                 static_cast<int>(Tp), p->status);
        if (wide_d) {
            g.tmB = p->tB10w;
            g.b_box = nmax_dense;
        }
        if (!wide_d && !p->mixed) {
            g.tmB1 = p->tB10r;
            g.b_row1 = 1;
        }
        if (p->mixed) {
            g.kind = KIND_BF16;
            g.KT = p->Kcat / 64;
            g.kseg_tiles = g.KT;
            g.sfa = nullptr;
            g.sfb = nullptr;
        }
        g.dense = 1;
        g.m_tiles = D / kBlockM;
        g.n_tokens = T;
        g.epi_split = 1 << 30;
        g.epi[0] = EpiParams{EPI_F32, 0, 0, 0, static_cast<float*>(y), D, nullptr, 0, nullptr, 0, 0, p->out_bf16 ? 1 : 0};
        const int items = g.m_tiles * ((T + g.n_max - 1) / g.n_max);
        int grid = try_pair(g, p->tPB10, p->tSA10, p->tPS10, 0, items / 2, p->num_sms,
                            T >= MOE_PAIR_UP_ONE_LANE_FROM ? 1 : MOE_PAIR_GROUPS_UP);
        if (!grid) {
            grid = std::min(items, p->num_sms);
            shape_gemm(g, 0, items, grid);
        }
        TRY(launch_gemm(g, grid, s, side_a2 ? false : pdl(true)));
    }
    mark(MOE_NUM_STAGES);
    if (err == cudaSuccess) p->last_T = T;
    // intermediate outputs on request
    if (dbg && err == cudaSuccess) {
        const int S = p->S, SIs = p->SIs;
        const int64_t TK = static_cast<int64_t>(T) * k;
        if (dbg->xq) TRY(cudaMemcpyAsync(dbg->xq, p->xq, static_cast<size_t>(T) * D, cudaMemcpyDeviceToDevice, s));
        if (dbg->xs) TRY(launch_export_sf(p->xsf, Tps, nullptr, T, D / 32, 0, dbg->xs, nmax_dense, nullptr, 0, s));
        if (dbg->z)         // split rows keep the fp32 values in their second half
            TRY(cudaMemcpy2DAsync(dbg->z, sizeof(float) * L, p->z + (z_split ? L : 0), sizeof(float) * 2 * L,
                                  sizeof(float) * L, T, cudaMemcpyDeviceToDevice, s));
        if (dbg->zq) TRY(cudaMemcpyAsync(dbg->zq, p->zq, static_cast<size_t>(T) * L, cudaMemcpyDeviceToDevice, s));
        if (dbg->zs) TRY(launch_export_sf(p->zsf, Tp, nullptr, T, L / 32, 0, dbg->zs, 0, nullptr, 0, s));
        if (S > 0 && dbg->hsq)
            TRY(cudaMemcpy2DAsync(dbg->hsq, SIs, p->act + L, p->Kcat, SIs, T, cudaMemcpyDeviceToDevice, s));
        if (S > 0 && dbg->hss)
            TRY(launch_export_sf(p->actsf, Tps, nullptr, T, SIs / 32, L / 32, dbg->hss, nmax_dense, nullptr, 0, s));
        if (dbg->logits)
            TRY(cudaMemcpyAsync(dbg->logits, p->logits, sizeof(float) * T * E, cudaMemcpyDeviceToDevice, s));
        if (dbg->topk_idx) TRY(cudaMemcpyAsync(dbg->topk_idx, p->idx, sizeof(int32_t) * TK, cudaMemcpyDeviceToDevice, s));
        if (dbg->topk_w) TRY(cudaMemcpyAsync(dbg->topk_w, p->gw, sizeof(float) * TK, cudaMemcpyDeviceToDevice, s));
        if (dbg->counts) TRY(cudaMemcpyAsync(dbg->counts, p->counts, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, s));
        if (dbg->offsets)
            TRY(cudaMemcpyAsync(dbg->offsets, p->offsets, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToDevice, s));
        if (dbg->sorted_token)
            TRY(cudaMemcpyAsync(dbg->sorted_token, p->sorted_token, sizeof(int32_t) * TK, cudaMemcpyDeviceToDevice, s));
        if (dbg->hq) TRY(launch_gather_rows(p->hq, Ip, p->canon_to_pad, TK, I, dbg->hq, I, s));
        if (dbg->hqs)
            TRY(launch_export_sf(p->hqsf, Rps, p->canon_to_pad, TK, I / 32, 0, dbg->hqs, nmax_grp, p->seg, E, s));
        if (dbg->o)
            TRY(launch_gather_rows(reinterpret_cast<const uint8_t*>(p->o), sizeof(float) * L, p->canon_to_pad, TK,
                                   sizeof(float) * L, reinterpret_cast<uint8_t*>(dbg->o), sizeof(float) * L, s));
        if (dbg->cq) TRY(cudaMemcpy2DAsync(dbg->cq, L, p->act, p->Kcat, L, T, cudaMemcpyDeviceToDevice, s));
        if (dbg->cs) TRY(launch_export_sf(p->actsf, Tps, nullptr, T, L / 32, 0, dbg->cs, nmax_dense, nullptr, 0, s));
    }
#undef TRY
    return cuda_status(err);
}

moe_status moe_forward_host(void* plan, const uint16_t* x_host, int32_t T, void* y_host, void* stream) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p || !x_host || !y_host) return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > p->T_max) return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err = cudaMemcpyAsync(p->x_stage, x_host, sizeof(uint16_t) * T * p->D, cudaMemcpyHostToDevice, s);
    if (err != cudaSuccess) return cuda_status(err);
    moe_status st = moe_forward(plan, p->x_stage, T, p->y_stage, stream, nullptr);
    if (st != MOE_OK) return st;
    err = cudaMemcpyAsync(y_host, p->y_stage, (p->out_bf16 ? 2 : 4) * static_cast<size_t>(T) * p->D,
                          cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    return cuda_status(err);
}

moe_status moe_quantile_balance(void* plan, int32_t T, int32_t target, double alpha, float* bias_out, void* stream) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p || !bias_out || T < 2 || T != p->last_T || p->cfg.score_fn != MOE_SCORE_SIGMOID_BIAS || p->k >= p->E ||
        !(alpha > 0.0 && alpha <= 1.0))
        return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(bias_out) & 3) return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    if (!p->qb_marg) {
        cudaError_t err = palloc(p, &p->qb_marg, sizeof(double) * p->E * p->T_max);
        if (err != cudaSuccess) return cuda_status(err);
    }
    if (target <= 0) target = static_cast<int32_t>((static_cast<int64_t>(T) * p->k + p->E / 2) / p->E);
    return cuda_status(launch_quantile_balance(p->logits, p->has_bias ? p->bias : nullptr, T, p->E, p->k, target, alpha,
                                               p->qb_marg, bias_out, static_cast<cudaStream_t>(stream)));
}

moe_status moe_set_bias(void* plan, const float* bias) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p || !bias || p->cfg.score_fn != MOE_SCORE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    std::vector<float> hb(p->E);
    cudaError_t err = cudaDeviceSynchronize();
    if (err == cudaSuccess) err = cudaMemcpy(hb.data(), bias, sizeof(float) * p->E, cudaMemcpyDeviceToHost);
    if (err != cudaSuccess) return cuda_status(err);
    float absmax = 0.0f;
    for (float b : hb) {
        if (!(b == b) || std::fabs(b) == INFINITY) return MOE_ERR_INVALID_ARG;
        absmax = std::max(absmax, std::fabs(b));
    }
    err = cudaMemcpy(p->bias, bias, sizeof(float) * p->E, cudaMemcpyDeviceToDevice);
    if (err != cudaSuccess) return cuda_status(err);
    p->bias_absmax = absmax;
    p->has_bias = true;
    return MOE_OK;
}

int64_t moe_ep_row_bytes(const void* plan) {
    const Plan* p = static_cast<const Plan*>(plan);
    return p ? ep_row_bytes(p->L) : 0;
}

moe_status moe_ep_dispatch(void* plan, int32_t T, int32_t ranks, uint8_t* wire, int64_t* rank_offsets, void* stream) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p || !wire || !rank_offsets || T < 1 || T != p->last_T || ranks < 1 || ranks > p->E)
        return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(wire) & 15 || reinterpret_cast<uintptr_t>(rank_offsets) & 7) return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    return cuda_status(launch_ep_pack(p->sorted_token, p->offsets, p->idx, p->gw, p->zq,
                                      reinterpret_cast<const uint32_t*>(p->zsf), p->T_pad, T, p->k, p->E, p->L, ranks,
                                      wire, rank_offsets, static_cast<cudaStream_t>(stream)));
}

moe_status moe_ep_combine(void* plan, int32_t T, const uint8_t* wire, const float* expert_out, float* c, void* stream) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p || !wire || !expert_out || !c || T < 1 || T > p->T_max) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(wire) & 15 || reinterpret_cast<uintptr_t>(expert_out) & 3 ||
        reinterpret_cast<uintptr_t>(c) & 3)
        return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    return cuda_status(launch_ep_combine(wire, expert_out, T, p->k, p->L, p->ep_inv, c, static_cast<cudaStream_t>(stream)));
}

moe_status moe_get_device_status(void* plan) {
    Plan* p = static_cast<Plan*>(plan);
    if (!p) return MOE_ERR_INVALID_ARG;
    DevGuard guard(p->device);
    int code = 0;
    if (cudaMemcpy(&code, p->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (code == 0) return MOE_OK;
    cudaMemset(p->status, 0, sizeof(int));
    return (code == DEV_BAD_WORK) ? MOE_ERR_DEVICE : MOE_ERR_TIMEOUT;
}

size_t moe_workspace_bytes(const void* plan) {
    const Plan* p = static_cast<const Plan*>(plan);
    return p ? p->bytes : 0;
}

void moe_free(void* plan) { plan_release(static_cast<Plan*>(plan)); }

moe_status moe_mxfp4_encode(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                            void* stream) {
    if (!w || !codes || !scales || rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(w) & 15 || reinterpret_cast<uintptr_t>(codes) & 15) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_mxfp4_encode(w, rows, K, codes, scales, static_cast<cudaStream_t>(stream)));
}

moe_status moe_mx_gemm(const uint8_t* a_codes, const uint8_t* a_scales, int32_t M, const uint8_t* b_codes,
                       const uint8_t* b_scales, int32_t N, int32_t K, float* out, int32_t* dev_status,
                       void* stream) {
    if (!a_codes || !a_scales || !b_codes || !b_scales || !out) return MOE_ERR_INVALID_ARG;
    if (M <= 0 || M % 128 || K <= 0 || K % 128 || N <= 0 || N > (1 << 24)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a_codes) & 31) || (reinterpret_cast<uintptr_t>(b_codes) & 15) ||
        (reinterpret_cast<uintptr_t>(out) & 3))
        return MOE_ERR_INVALID_ARG;
    if (!encode_fn()) return MOE_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess) err = gemm_setup();
    if (err != cudaSuccess) return cuda_status(err);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t Np = rup(N, 16);
    const size_t atom_bytes = static_cast<size_t>(M) * K / 32;
    const size_t plane_bytes = static_cast<size_t>(K / 128) * (Np + 32) * 16;    // item-atom planes
    CUtensorMap tA, tB, tB1;
    int pair_cl = 0;
    const int nmax = dense_nmax(M, N, &pair_cl);
    if (!map_mx4(&tA, a_codes, M, K) || !map_mx8(&tB, b_codes, N, K, dense_box_rows(nmax, pair_cl)) ||
        !map_mx8(&tB1, b_codes, N, K, 1))
        return MOE_ERR_INVALID_ARG;
    uint8_t* scratch = nullptr;
    err = cudaMallocAsync(reinterpret_cast<void**>(&scratch), atom_bytes + plane_bytes + 256, s);
    if (err != cudaSuccess) return cuda_status(err);
    uint8_t* atoms = scratch;
    uint8_t* planes = scratch + atom_bytes;
    int32_t* st = dev_status ? dev_status : reinterpret_cast<int32_t*>(scratch + atom_bytes + plane_bytes);
    err = cudaMemsetAsync(planes, 0, plane_bytes + 256, s);
    if (err == cudaSuccess) err = launch_sf_atoms(a_scales, M, K / 32, atoms, s);
    if (err == cudaSuccess) err = launch_sf_item_planes(b_scales, N, K / 32, planes, Np + 32, nmax, s);
    if (err == cudaSuccess) {
        GemmParams g = gemm_base(tA, tB, atoms, planes, Np + 32, K, nmax, M, static_cast<int>(Np), st);
        if (nmax <= kNarrowMax) {
            g.tmB1 = tB1;        // items of fewer than 16 tokens load their rows one by one
            g.b_row1 = 1;
        }
        g.epi[0] = EpiParams{EPI_F32, 0, 0, 0, out, M, nullptr, 0, nullptr, 0};
        err = launch_dense_mx(g, M, N, K, Np, nmax, pair_cl, atoms, planes, sms, s);
    }
    cudaError_t ferr = cudaFreeAsync(scratch, s);
    if (err == cudaSuccess) err = ferr;
    return cuda_status(err);
}

moe_status moe_mma_probe(int32_t kind, int32_t n, int32_t iters, int32_t* dev_status, double* flops_out,
                         void* stream) {
    if (!dev_status || !flops_out || kind < PROBE_MX_E2M1_E4M3 || kind > PROBE_BF16) return MOE_ERR_INVALID_ARG;
    if (n < 16 || n > (kind == PROBE_BF16 ? 256 : kNMax) || (n & 15) || iters < 1 || iters > (1 << 22))
        return MOE_ERR_INVALID_ARG;
    int dev = 0, sms = 0, major = 0, minor = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (err != cudaSuccess) return cuda_status(err);
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
    return cuda_status(launch_mma_probe(kind, n, iters, sms, dev_status, flops_out, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_mx_gemm_noalloc: the same block-scaled GEMM for callers that may not
// allocate device memory themselves or through us.  Its scratch (the
// re-arranged scale factors and a status word) lives in this fixed, file-scope
// device array instead of cudaMallocAsync memory.  Every device that loads
// the library holds the array until the process exits; all calls share it.
static __device__ __align__(256) uint8_t moe_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
constexpr int kNoAllocMaxDevices = 64;
uint8_t* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on `dev` (which must be current).  In
// host code the array's name is only a host-side stand-in, so the address is
// looked up once per device and cached.
cudaError_t noalloc_scratch(int dev, uint8_t** out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, moe_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}
}  // namespace

extern "C" moe_status moe_mx_gemm_noalloc(const uint8_t* a_codes, const uint8_t* a_scales, int32_t M,
                                          const uint8_t* b_codes, const uint8_t* b_scales, int32_t N, int32_t K,
                                          float* out, int32_t* dev_status, void* stream) {
    if (!a_codes || !a_scales || !b_codes || !b_scales || !out) return MOE_ERR_INVALID_ARG;
    if (M <= 0 || M % 128 || K <= 0 || K % 128 || N <= 0 || N > (1 << 24)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a_codes) & 31) || (reinterpret_cast<uintptr_t>(b_codes) & 15) ||
        (reinterpret_cast<uintptr_t>(out) & 3))
        return MOE_ERR_INVALID_ARG;
    const int64_t Np = rup(N, 16);
    const size_t atom_bytes = static_cast<size_t>(M) * K / 32;
    const size_t plane_bytes = static_cast<size_t>(K / 128) * (Np + 32) * 16;    // item-atom planes
    if (atom_bytes + plane_bytes + 256 > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_INVALID_ARG;
    if (!encode_fn()) return MOE_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess) err = gemm_setup();
    uint8_t* scratch = nullptr;
    if (err == cudaSuccess) err = noalloc_scratch(dev, &scratch);
    if (err != cudaSuccess) return cuda_status(err);
    CUtensorMap tA, tB;
    int pair_cl = 0;
    const int nmax = dense_nmax(M, N, &pair_cl);
    if (!map_mx4(&tA, a_codes, M, K) || !map_mx8(&tB, b_codes, N, K, dense_box_rows(nmax, pair_cl)))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* atoms = scratch;
    uint8_t* planes = scratch + atom_bytes;
    int32_t* st = dev_status ? dev_status : reinterpret_cast<int32_t*>(planes + plane_bytes);
    // the array keeps the previous call's contents: clear the scale planes
    // (their padding rows) and the internal status word
    err = cudaMemsetAsync(planes, 0, plane_bytes + 256, s);
    if (err == cudaSuccess) err = launch_sf_atoms(a_scales, M, K / 32, atoms, s);
    if (err == cudaSuccess) err = launch_sf_item_planes(b_scales, N, K / 32, planes, Np + 32, nmax, s);
    if (err == cudaSuccess) {
        GemmParams g = gemm_base(tA, tB, atoms, planes, Np + 32, K, nmax, M, static_cast<int>(Np), st);
        g.epi[0] = EpiParams{EPI_F32, 0, 0, 0, out, M, nullptr, 0, nullptr, 0};
        err = launch_dense_mx(g, M, N, K, Np, nmax, pair_cl, atoms, planes, sms, s);
    }
    return cuda_status(err);
}
