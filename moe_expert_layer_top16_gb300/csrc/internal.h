// Declarations shared by the translation units of libmoe (not installed).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// Programmatic dependent launch.  The forward's kernels after the first are
// launched with programmatic stream serialization (launch_ex with pdl): such
// a kernel may start while its predecessor in the stream drains, runs its
// prologue (barriers, TMEM allocation, descriptor prefetch), then waits in
// pdl_wait() until the predecessor has completed and its writes are visible,
// before it reads or writes any buffer.  Each of these kernels calls
// pdl_trigger() when it starts, so that its successor can launch as soon as
// every CTA of this grid is running.  Both are no-ops in a kernel launched
// without programmatic serialization.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The same with thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                     bool pdl, int cluster, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Device status codes (sticky; read by moe_get_device_status).
enum : int { DEV_OK = 0, DEV_TIMEOUT_PRODUCER = 1, DEV_TIMEOUT_MMA = 2, DEV_TIMEOUT_EPILOGUE = 3,
             DEV_TIMEOUT_TEARDOWN = 4, DEV_BAD_WORK = 5 };

// ------------------------------------------------------------------ GEMM engine
// Tiles: 128 weight rows (MMA M, the A operand, MXFP4) x up to kNMax tokens
// (MMA N, the B operand, MXFP8) x 128 along K per pipeline stage.
constexpr int kBlockM = 128;
constexpr int kBlockK = 128;
constexpr int kNMax = 240;        // tokens per work item at most (TMEM: accumulators + scale columns <= 512)
constexpr int kMaxGroups = 4;     // producer / MMA warp pairs per CTA
constexpr int kEpiGroups = 2;       // epilogue warpgroups of the GEMM engine
constexpr int kNarrowMax = 64;      // items of at most this many tokens are "narrow"
constexpr int kGemmMaxThreads = (2 * kMaxGroups + 4 * kEpiGroups) * 32;
constexpr int kSmemLimit = 227 * 1024;

enum EpiMode : int {
    EPI_F32 = 0,        // store fp32 accumulators
    EPI_QUANT = 1,      // optionally store fp32, and store MXFP8 of the row segment (blocks along M)
    EPI_SILU_QUANT = 2, // rows 0..63 gate, 64..127 up: store MXFP8 of SiLU(gate) * up
    EPI_SILU_BF16 = 3   // rows 0..63 gate, 64..127 up: store SiLU(gate) * up rounded to bf16 (out_q holds bf16)
};

// Where an epilogue region writes.  Output row = item.b_row0 + token index;
// output column = col0 + (item.mt - m_tile0) * cols_per_mtile + row-in-tile.
struct EpiParams {
    int mode;
    int m_tile0;
    int col0;
    int f32_split;      // > 0: store the fp32 output rounded to TF32 at col and as it is at col + f32_split
    float* out_f32;     // [rows][ld_f32]
    int64_t ld_f32;
    uint8_t* out_q;     // E4M3 codes [rows][ld_q]
    int64_t ld_q;
    uint8_t* out_sf;    // scale planes: uint32 word per (col/128, row), byte (col%128)/32
    int64_t sf_pitch;   // rows (raw planes) or 16-byte slots (item-atom planes) per plane
    int sf_item;        // 1: item-atom planes keyed by the output item's first row; 0: raw planes
    int out_bf16;       // EPI_F32: out_f32 points at bf16 storage (ld_f32 in elements), values rounded to nearest
};

enum GemmKind : int {
    KIND_MX = 0,        // MXFP4 A x MXFP8 B, block-scaled (kind::mxf8f6f4)
    KIND_TF32 = 1,      // fp32 A x fp32 B as TF32 (kind::tf32), no scales
    KIND_BF16 = 2       // bf16 A x bf16 B (kind::f16), fp32 accumulate, no scales
};

struct GemmParams {
    CUtensorMap tmA;        // MX: MXFP4 weights, 16U4_ALIGN16B, box {128, 128}; TF32: fp32, box {32, 128}
    CUtensorMap tmB;        // MX: MXFP8 activations, UINT8, box {128, 16}; TF32: fp32, box {32, 16}
    CUtensorMap tmB1;       // MX, b_row1 != 0: the same activations with a one-row box {128, 1}
    int b_row1;             // items of fewer than 16 tokens load only their own rows (tmB1) and scale slots
    int b_producer;         // groups == 1: a warp of its own issues the token-side copies (B rows, their scales)
    const uint8_t* sfa;     // weight scales, pre-arranged: [rows/128][KT][512]
    const uint8_t* sfb;     // activation scales, item-atom planes: [KT][sfb_pitch] 16-byte slots
    int64_t sfb_pitch;
    int KT;                 // 128-wide K tiles
    int n_max;              // tokens per work item (multiple of 16, <= kNMax)
    int groups;             // producer / MMA warp pairs = item lanes x ksplit
    int ksplit;             // groups per item; each takes a contiguous 1/ksplit of the item's K tiles
    int contiguous;         // 1: each CTA takes a contiguous range of items; 0: every gridDim.x-th item
    int b_box;              // token rows per TMA box of B (tmB's box height): 16, or n_max for wide items
    int acc_bufs;           // TMEM accumulator buffers per group (1 or 2)
    int stages;             // shared-memory stages of all groups together
    int stage_bytes;
    int a_tx_bytes;         // bytes a 128x128 MXFP4 TMA box delivers to the mbarrier
    int dense;              // 1: items = m_tiles x ceil(n_tokens / n_max); 0: item list
    int m_tiles;
    int mt_base;            // dense: the first of the m_tiles weight tiles (row block mt_base + i)
    int n_tokens;
    int a_rows;             // rows of A (bounds check of list items)
    int b_rows;             // rows of B / scale planes (bounds check)
    // grouped items (dense == 0): for expert e, ceil(counts[e] / n_max) token
    // tiles x mt_per_e weight tiles, numbered from ioff[e] (ioff[E] = total);
    // token tile j starts at permuted row seg[e] + j * n_max.
    const int* ioff;        // [E+1]
    const int* seg;         // [E+1]
    const int* counts;      // [E]
    int E;
    int mt_per_e;
    int rows_per_e;
    int epi_split;          // dense: m-tiles >= epi_split use epi[1]
    int kind;               // GemmKind
    int kseg_tiles;         // K tiles per K segment (K-concatenation through map coordinates)
    int a_seg_x[3];         // element offset along K of each segment in A's map
    int b_seg_x[3];         // element offset along K of each segment in B's map
    EpiParams epi[2];
    int* status;
    // CTA pairs (pair != 0): clusters of two CTAs share M = 256 MMAs; work
    // item i of the launch is the pair of engine items 2i (even CTA) and
    // 2i + 1 (odd CTA).  Needs one group without K-splits, the token-side
    // producer, B boxes of pair_b_rows(n_max) rows (each CTA loads half of
    // an item's token rows), an even grid, and an even number of weight tiles
    // per expert (grouped) or m_tiles and mt_base even (dense).  The scale
    // tiles then load through these maps of 256-byte rows: sfa as
    // [rows/128 * KT * 2][256] in 2-row boxes (one 512-byte atom), sfb as
    // [KT * sfb_pitch / 16][256] in boxes of 2 * ceil(n_max / 128) rows (all
    // atoms of an item; sfb_pitch and the items' first rows are multiples of
    // 16).
    int pair;
    CUtensorMap tmSFA;
    CUtensorMap tmSFB;
};

// Token rows of one CTA of a pair per stage (half of the largest item).
__host__ __device__ __forceinline__ int pair_b_rows(int n_max) { return ((n_max >> 1) + 15) & ~15; }
// Shared-memory bytes of one stage; pair: the stage of one CTA of a pair
// (half of the item's token rows, all of its token scales).
int gemm_stage_bytes(int n_max, bool pair = false);
// total shared-memory stages of a launch (all groups); E > 0: grouped items
// (per-expert tables in shared memory); xbuf: the SiLU exchange buffer and the
// per-warp staging of MXFP8 output codes (quantising epilogues)
int gemm_stages(int n_max, int groups, int E, bool xbuf, bool pair = false);
size_t gemm_smem_bytes(int n_max, int stages, int E, bool xbuf, bool pair = false);
// Clusters of two CTAs of the pair kernels that fit on the GPU at once (0: none).
int gemm_pair_clusters();
bool gemm_needs_xbuf(const GemmParams& p);
bool gemm_config_ok(int n_max, int groups, int ksplit, int acc_bufs);
cudaError_t gemm_setup();   // raise the dynamic shared memory limit once
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t s, bool pdl = false);

// ------------------------------------------------------------------ other kernels
// xsf: item-atom planes of a dense GEMM with token tiles of n_max
// xf (optional): x as fp32 [T][D]
// x -> MXFP8 codes and item-atom scales (and x as fp32 when xf is set);
// also clears zero[0, n_zero) (the forward's selection bitmaps)
cudaError_t launch_quant_x(const __nv_bfloat16* x, int T, int D, uint8_t* xq, uint8_t* xsf, int64_t pitch, int n_max,
                           float* xf, uint32_t* zero, int64_t n_zero,
                           cudaStream_t s, bool pdl = false);
// SIMT router on z = hi + lo ([T][2L]) writing logits [T][E]; batches of at
// most kRouterSplitTokens tokens split K kRouterSplit ways over a cluster.
constexpr int kRouterSplit = 8;
constexpr int kRouterSplitTokens = 128;
// z: router input rows of ld floats, K = L values, with their exact
// remainders at offset lo (lo = 0: none); R [E][L]
cudaError_t launch_router(const float* z, int ld, int lo, const float* R, float* logits, int T, int E, int L,
                          cudaStream_t s, bool pdl = false);
// Streaming exact fp32 router for up to 128 tokens (router.cu): tmR maps R
// [E][K] fp32 (box {32, 128}), tmZ the router input rows [T_pad][K] (box
// {32, 64}), both with the 128-byte swizzle; K split over clusters of c = 8
// or 16 CTAs.
bool router_stream_ok(int K);
cudaError_t router_stream_setup();
int router_stream_max_clusters(int c);
cudaError_t launch_router_stream(const CUtensorMap& tmR, const CUtensorMap& tmZ, float* logits, int T, int E, int K,
                                 int c, int* status, cudaStream_t s, bool pdl = false);
// top-k + gates (kernels.cu).  With refine, the logits are tensor-core
// estimates z_hi R_hi (both rounded to TF32) and the candidates' exact fp32
// logits are recomputed from z ([T][z_ld], z_hi | z) and R ([E][L]); the
// remainder z_lo = z - z_hi is exact in fp32 (Sterbenz).  The
// estimate of expert e for token t is within
//   delta_te = |z_hi_t| |R_lo_e| + (|z_lo_t| + g_tc (1 + 2^-11) |z_hi_t|
//              + g_32 (|z_hi_t| + |z_lo_t|)) |R_e|        (2-norms)
// of the exact logit: the first two terms bound the TF32 rounding of the
// operands (Cauchy-Schwarz), g_tc the tensor core's fp32 accumulation and g_32
// the exact path's FMA chain (both relative to sum |z| |R| <= |z| |R|).
struct TopkArgs {
    float* logits;
    const float* bias;
    int T, E, k, softmax;
    int refine;
    const float* z;         // router input rows (z_ld floats): L TF32 heads, the fp32 values at z_lo (0: the
    int z_ld, z_lo;         // rows are exactly TF32 and hold only the L values)
    const float* R;         // [E][L]
    const float* rnorm;     // refine: [2][E] upper bounds of |R_e| and |R_lo_e| (2-norms)
    float g_tc, g_32;       // refine: accumulation error coefficients (see above), rounded up
    float sq_infl;          // refine: factor covering the fp32 rounding of a sum of L squares
    int L;
    int32_t* idx;
    float* w;
    uint32_t* sel;
    int W;
    float bias_absmax;      // max |bias| (0 without a bias)
    float key_err;          // set by launch_topk: error bound of an fp32 sigmoid(l) + b evaluation
    float band_pad;         // set by launch_topk: twice key_err, rounded up
};
// upper bounds of the 2-norms of the rows of R [E][K] and of its TF32
// remainders (Rs [E][2K], hi | lo): out [0, E) = |R_e|, [E, 2E) = |R_lo_e|
cudaError_t launch_router_norms(const float* R, const float* Rs, int E, int K, float* out, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_expert_scan(const uint32_t* sel, int E, int W, int32_t* wpre, int32_t* counts, cudaStream_t s,
                               bool pdl = false);
struct WorkListArgs {
    const int32_t* counts;
    int E;
    // small batches: the per-expert scan of the token bitmaps happens here
    // too (sel [E][W] words in, wpre [E][W] and counts out); null = done before
    const uint32_t* sel;
    int W;
    int32_t* wpre;
    int32_t* counts_out;
    int32_t* offsets;    // [E+1] exclusive scan of counts
    int32_t* seg;        // [E+1] exclusive scan of counts rounded up to 16 (row starts in permuted buffers)
    int32_t* ioff1; int n_max1; int mt1;   // [E+1] item offsets of the gate/up GEMM
    int32_t* ioff2; int n_max2; int mt2;   // [E+1] item offsets of the down GEMM
};
cudaError_t launch_worklist(const WorkListArgs& a, cudaStream_t s, bool pdl = false);
struct ScatterArgs {
    const int32_t* idx; int T; int k; int W;
    const uint32_t* sel; const int32_t* wpre; const int32_t* offsets; const int32_t* seg;
    int32_t* slot_pos;        // [T*k] row of (t, j) in the permuted buffers
    int32_t* canon_to_pad;    // [T*k] sorted (unpadded) position -> permuted row
    int32_t* sorted_token;    // [T*k] token of each sorted position
    const uint8_t* zq; const uint8_t* zsf; int64_t zsf_pitch; int L;
    uint8_t* zq_perm; uint8_t* zq_perm_sf; int64_t perm_pitch;   // zq_perm_sf: item-atom planes
    int n_max;                // token tile of the grouped GEMM that reads zq_perm
    int slots_per_warp;       // set by launch_scatter
};
cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t s, bool pdl = false);
// out_sf: item-atom planes of a dense GEMM with token tiles of n_max
// out_bf (optional): write c rounded to bf16 at out_bf[t * ld_q + col] instead of MXFP8
cudaError_t launch_combine(const float* o, const int32_t* slot_pos, const float* w, int T, int k, int L,
                           uint8_t* out_q, int64_t ld_q, uint8_t* out_sf, int64_t sf_pitch, int n_max,
                           __nv_bfloat16* out_bf, cudaStream_t s, bool pdl = false);
cudaError_t launch_mxfp4_encode(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                                cudaStream_t s);
cudaError_t kernels_setup();   // per-device kernel attributes
// fp32 [rows][K] -> [rows][2K] = nearest TF32 | exact remainder
cudaError_t launch_tf32_split(const float* src, int64_t rows, int64_t K, float* dst, cudaStream_t s);
// [rows][2K] (hi | lo) -> [rows][K] = hi + lo
// row-major scales [rows][kb] -> item-atom planes [kb/4][pitch] of a dense
// GEMM with token tiles of n_max
cudaError_t launch_sf_item_planes(const uint8_t* scales_rm, int64_t rows, int64_t kb, uint8_t* planes, int64_t pitch,
                                  int n_max, cudaStream_t s);
// plan-time repacking
cudaError_t launch_copy_rows(uint8_t* dst, int64_t dst_stride, const uint8_t* const* src_rows, int64_t nrows,
                             int64_t row_bytes, cudaStream_t s);
cudaError_t launch_sf_atoms(const uint8_t* scales_rm, int64_t rows, int64_t kb, uint8_t* atoms, cudaStream_t s);
// debug export of scales to [rows][nblocks] bytes: raw planes (item_n == 0)
// or item-atom planes of token tiles of item_n (dense when seg is null, else
// tiles within the expert segments seg[0..E])
cudaError_t launch_export_sf(const uint8_t* planes, int64_t pitch, const int32_t* row_map, int64_t rows,
                             int64_t nblocks, int64_t col_block0, uint8_t* out, int item_n, const int32_t* seg, int E,
                             cudaStream_t s);
cudaError_t launch_gather_rows(const uint8_t* src, int64_t src_stride, const int32_t* row_map, int64_t rows,
                               int64_t row_bytes, uint8_t* dst, int64_t dst_stride, cudaStream_t s);

// ------------------------------------------------------------------ expert-parallel emulation (ep.cu)
int64_t ep_row_bytes(int L);
cudaError_t launch_ep_pack(const int32_t* sorted_token, const int32_t* offsets, const int32_t* idx, const float* gw,
                           const uint8_t* zq, const uint32_t* zsf, int64_t zsf_pitch, int T, int k, int E, int L,
                           int R, uint8_t* wire, int64_t* rank_offsets, cudaStream_t s);
cudaError_t launch_ep_combine(const uint8_t* wire, const float* out, int T, int k, int L, int32_t* inv, float* c,
                              cudaStream_t s);

// ------------------------------------------------------------------ Quantile Balancing (balance.cu)
// new bias [E] from logits [T][E] and the current bias (null: 0); marg: [E][T] fp64 workspace
cudaError_t launch_quantile_balance(const float* logits, const float* bias, int T, int E, int k, int target,
                                    double alpha, double* marg, float* bias_out, cudaStream_t s);

// ------------------------------------------------------------------ tensor-core rate probe (peak.cu)
enum ProbeKind : int { PROBE_MX_E2M1_E4M3 = 0, PROBE_MX_E4M3_E4M3 = 1, PROBE_BF16 = 2 };
// grid CTAs each issue iters x 4 MMAs of M = 128 x n; *flops = their FLOPs
cudaError_t launch_mma_probe(int kind, int n, int iters, int grid, int* status, double* flops, cudaStream_t s);

}  // namespace moe
