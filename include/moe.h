/*
 * moe.h -- C ABI of libmoe: the forward pass of a Kimi K3-style sparse MoE
 * layer (top-k of E routed experts in a latent space, plus always-on shared
 * experts) on one NVIDIA GB300 (sm_103a).
 *
 * What the layer computes, per token x (bf16, width D):
 *   xq  = MXFP8(x)                                   activations enter as MXFP8
 *   z   = xq P_down^T           (D -> L latent)      "Kimi K3 and the New
 *   l   = z R^T                 (router logits)       Open-Weights Moat",
 *   top-k on sigmoid(l) + bias; w = sigmoid(l_j) / sum over the winners
 *                                                     section "How the router
 *                                                     picks 16 of 896", Fig. 2
 *   for each winner e_j: h = SiLU(zq W_gate[e]^T) * (zq W_up[e]^T)
 *                        o_j = MXFP8(h) W_down[e]^T
 *   c   = sum_j w_j o_j                                weighted sum in the latent
 *   y   = MXFP8(c) P_up^T + sum_s MXFP8(h_s) S_down[s]^T
 *   h_s = SiLU(xq S_gate[s]^T) * (xq S_up[s]^T)       shared experts, full width
 * (section "Sparse computation: latent experts and routing": routed path in a
 * latent, shared experts at full width, branches summed).  All weights are
 * MXFP4 (E2M1 elements, one E8M0 scale per 32 along the reduction dim) and
 * every GEMM input activation is MXFP8 (E4M3, one E8M0 scale per 32):
 * section "Precision and deployment", Fig. 6.  The dispatch (stable sort of
 * (token, slot) pairs by expert, per-expert counts/offsets), one GEMM per
 * expert segment and the gate-weighted combine follow the one-page data path
 * of "Kimi K3: 2.8 Trillion Parameters, Four Bits at a Time", section "What
 * it takes to serve it".  With score_fn = MOE_SCORE_SOFTMAX the gates are the
 * softmax of the winners' logits instead (that page's toy router).
 *
 * With precision = MOE_PRECISION_MIXED the layer follows the scheme of
 * "Precision and deployment", Fig. 6 instead: only the routed experts'
 * weights are MXFP4 and their inputs MXFP8, while the latent projections and
 * the shared experts keep BF16 weights and read BF16 inputs (x as given,
 * h_s and c rounded to bf16, nearest even); z stays fp32 for the router.
 *
 * Byte layouts.  An MXFP4 matrix W[rows][K] is `codes` uint8 [rows][K/2]
 * (element 2i in the low nibble of byte i, bit 3 of a nibble = sign) plus
 * `scales` uint8 [rows][K/32] (E8M0, value 2^(code-127)); rows are output
 * features, K is the reduction dim.  MXFP8 activations are codes uint8
 * [T][K] (E4M3) plus scales uint8 [T][K/32].  All pointers in this header are
 * DEVICE pointers on the plan's device unless stated otherwise.
 *
 * Errors.  Every call validates its arguments before enqueuing anything and
 * returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED with nothing enqueued.
 * CUDA API failures return MOE_ERR_CUDA.  Kernels never trap: a device-side
 * failure (a bounded wait that ran out) is recorded in a sticky device status
 * word read by moe_get_device_status().
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad pointer, size or shape; nothing enqueued */
    MOE_ERR_UNSUPPORTED = 2,   /* valid config this build does not run (e.g. no sm_103a device) */
    MOE_ERR_OOM = 3,           /* device allocation failed inside moe_plan */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    MOE_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (device status) */
    MOE_ERR_DEVICE = 6         /* other device-side error (device status) */
} moe_status;

typedef enum {
    MOE_SCORE_SIGMOID_BIAS = 0, /* sigmoid score, top-k on score + bias, sum-normalised */
    MOE_SCORE_SOFTMAX = 1       /* top-k on the logit, softmax over the k winners */
} moe_score_fn;

/* What the router reads.  The pages route in the latent space ("Kimi K3: 2.8
 * Trillion Parameters, Four Bits at a Time", "The shape of the model"); "What
 * Kimi K3 asks of the hardware" leaves the latent part unspecified, so the
 * hidden state can be routed on instead. */
typedef enum {
    MOE_ROUTE_ON_LATENT = 0,    /* logits = z R^T, R [E][L] */
    MOE_ROUTE_ON_HIDDEN = 1     /* logits = x R^T (x exactly as given), R [E][D] */
} moe_route_input;

/* Number formats of the non-routed GEMMs. */
typedef enum {
    MOE_PRECISION_MX = 0,       /* every weight MXFP4, every GEMM input MXFP8 */
    MOE_PRECISION_MIXED = 1     /* bf16 latent projections and shared experts; MXFP4/MXFP8 routed experts */
} moe_precision;

/* Element type of the output y. */
typedef enum {
    MOE_OUT_F32 = 0,            /* fp32 [T][D] */
    MOE_OUT_BF16 = 1            /* bf16 [T][D], each value rounded to nearest even from fp32 */
} moe_out_dtype;

/* Layer shape.  Constraints (checked by moe_plan): d_model and d_latent
 * multiples of 128; expert_inter and shared_inter multiples of 64;
 * 1 <= top_k <= min(n_experts, 32); 1 <= n_experts <= 1024; n_shared >= 0;
 * 1 <= max_tokens <= 65536. */
typedef struct {
    int32_t d_model;       /* D */
    int32_t d_latent;      /* L */
    int32_t n_experts;     /* E */
    int32_t top_k;         /* k */
    int32_t expert_inter;  /* I: routed expert inner width */
    int32_t n_shared;      /* S */
    int32_t shared_inter;  /* Is: shared expert inner width */
    int32_t max_tokens;    /* largest T a forward call may pass */
    int32_t score_fn;      /* moe_score_fn */
    int32_t route_input;   /* moe_route_input */
    int32_t out_dtype;     /* moe_out_dtype */
    int32_t precision;     /* moe_precision */
} moe_config;

typedef struct {
    const uint8_t *codes;  /* [rows][K/2] */
    const uint8_t *scales; /* [rows][K/32] */
} moe_mx4;

/* Layer weights (device pointers; read only during moe_plan, which copies
 * and repacks them into plan-owned memory -- the caller may free them when
 * moe_plan returns). */
typedef struct {
    moe_mx4 p_down;           /* [L][D]       latent down-projection */
    moe_mx4 p_up;             /* [D][L]       latent up-projection   */
    moe_mx4 w_gate;           /* [E][I][L]    routed gate            */
    moe_mx4 w_up;             /* [E][I][L]    routed up              */
    moe_mx4 w_down;           /* [E][L][I]    routed down            */
    moe_mx4 s_gate;           /* [S][Is][D]   shared gate            */
    moe_mx4 s_up;             /* [S][Is][D]   shared up              */
    moe_mx4 s_down;           /* [S][D][Is]   shared down            */
    const float *router_w;    /* [E][L] fp32 router (latent routing), [E][D] (hidden routing) */
    const float *router_bias; /* [E] fp32 selection bias, or NULL (= 0) */
    /* MOE_PRECISION_MIXED only (the MXFP4 p_down, p_up and s_* above are then
     * not read): bf16 bit patterns */
    const uint16_t *p_down_bf16;  /* [L][D]     */
    const uint16_t *p_up_bf16;    /* [D][L]     */
    const uint16_t *s_gate_bf16;  /* [S][Is][D] */
    const uint16_t *s_up_bf16;    /* [S][Is][D] */
    const uint16_t *s_down_bf16;  /* [S][D][Is] */
} moe_weights;

/* Optional intermediate outputs of one forward call (device pointers; NULL
 * skips a field).  Row counts use the T of that call.  "Sorted order" is the
 * stable sort of the flat (token, slot) pairs by expert: row p of a sorted
 * tensor belongs to token sorted_token[p]. */
typedef struct {
    /* xq/xs, hsq/hss and cq/cs exist in MOE_PRECISION_MX only */
    uint8_t *xq, *xs;         /* [T][D], [T][D/32]           MXFP8 of x            */
    float *z;                 /* [T][L]                      latent, fp32          */
    uint8_t *zq, *zs;         /* [T][L], [T][L/32]           MXFP8 of z            */
    uint8_t *hsq, *hss;       /* [T][S*Is], [T][S*Is/32]     MXFP8 shared activation */
    float *logits;            /* [T][E]  router logits: fp32 up to 128 tokens; above that (E % 128 == 0)
                               * fp32 for each token's top-k candidates and a tensor-core
                               * estimate elsewhere, within a proven per-(token, expert)
                               * bound of the fp32 value and below the k-th selected logit */
    int32_t *topk_idx;        /* [T][k]   slot order: descending key, tie -> lower id */
    float *topk_w;            /* [T][k]                      gates                 */
    int32_t *counts;          /* [E]                         tokens per expert     */
    int32_t *offsets;         /* [E+1]                       exclusive scan        */
    int32_t *sorted_token;    /* [T*k]                       token of sorted row   */
    uint8_t *hq, *hqs;        /* [T*k][I], [T*k][I/32]       MXFP8 expert activation, sorted */
    float *o;                 /* [T*k][L]                    expert outputs, sorted */
    uint8_t *cq, *cs;         /* [T][L], [T][L/32]           MXFP8 of the combine  */
    /* Optional array of MOE_NUM_STAGES + 1 cudaEvent_t (created by the caller):
     * event i is recorded on the forward's stream before stage i, the last one
     * after the final stage, so the caller can time each stage. */
    void **stage_events;
} moe_debug;

/* Stages of moe_forward, in launch order (indices into stage_events):
 *  0 quantise x      1 down-projection + shared gate/up GEMM   2 router
 *  3 top-k + gates   4 per-expert counts   5 offsets + work lists
 *  6 dispatch (ranks, gather)   7 grouped gate/up GEMM   8 grouped down GEMM
 *  9 combine         10 up-projection + shared down GEMM */
#define MOE_NUM_STAGES 11

/* Validate `cfg`, allocate all device memory for up to cfg->max_tokens
 * tokens on `device`, copy and repack `w`, build TMA descriptors.
 * Host-synchronous; the only call that allocates.  On failure *plan_out is
 * NULL.  Needs a compute capability 10.3 device. */
MOE_API moe_status moe_plan(const moe_config *cfg, const moe_weights *w, int device, void **plan_out);

/* Forward pass: x bf16 [T][D] (device, rows 16-byte aligned) -> y [T][D]
 * (device; fp32 or bf16 as cfg->out_dtype says).  Enqueued on `stream` (a cudaStream_t; NULL = legacy
 * default stream); no host synchronisation, no allocation.  1 <= T <=
 * max_tokens.  `dbg` may be NULL.  One plan serves one stream at a time:
 * calls on different streams that overlap race on the plan's workspace.
 * From 1024 tokens on (MXFP4 plans), the shared experts' first GEMM runs
 * on a stream the plan owns, forked from `stream` by an event and joined
 * back into it before the last step, so the call stays one unit of work on
 * `stream` (and can be captured in a CUDA graph).  The fork follows the
 * router when the call is launched directly and the routed down-projection
 * when `stream` is being captured; the results are the same bit for bit. */
MOE_API moe_status moe_forward(void *plan, const void *x, int32_t T, void *y, void *stream,
                       const moe_debug *dbg);

/* Same as moe_forward with HOST buffers: copies x (host, bf16 [T][D]) to the
 * device, runs the layer and copies y back to host memory y_host ([T][D],
 * fp32 or bf16 as cfg->out_dtype says), all on `stream`, then synchronises
 * the stream.  Page-locked host
 * buffers make the copies asynchronous. */
MOE_API moe_status moe_forward_host(void *plan, const uint16_t *x_host, int32_t T, void *y_host,
                            void *stream);

/* Sticky device-side status of the plan (call after synchronising the stream
 * of the last forward): MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE.  Reading it
 * clears it. */
MOE_API moe_status moe_get_device_status(void *plan);

/* Bytes of device memory the plan owns (weights + workspace). */
MOE_API size_t moe_workspace_bytes(const void *plan);

/* Release everything the plan owns.  NULL-safe.  Synchronises the device. */
MOE_API void moe_free(void *plan);

/* Static string naming a status code. */
MOE_API const char *moe_status_str(moe_status s);

/* Weight preparation (not part of the forward pass): MXFP4-encode fp32
 * w[rows][K] (device) into codes [rows][K/2] and scales [rows][K/32]
 * (device), with the block encoder of "Kimi K3: 2.8 Trillion Parameters,
 * Four Bits at a Time", section "Four bits from the start": per 32-block,
 * shared exponent floor(log2 amax) - 2 (clamped to [-127, 127]; an all-zero
 * block gets codes 0 and scale code 0), elements |v|/2^e clipped to 6 and
 * rounded to the nearest E2M1 level, the smaller level on a tie.  K must be a
 * multiple of 32.  Enqueued on `stream` on the current device. */
MOE_API moe_status moe_mxfp4_encode(const float *w, int64_t rows, int64_t K, uint8_t *codes,
                            uint8_t *scales, void *stream);

/* One block-scaled GEMM on the layer's tcgen05 engine, for callers that
 * need the raw product:
 *   out[n][m] = sum_k dq(B[n][k]) * dq(A[m][k])      (fp32 accumulate)
 * A: MXFP4 [M][K] (a_codes [M][K/2], 32-byte aligned; a_scales [M][K/32]);
 * B: MXFP8 [N][K] (b_codes [N][K], 16-byte aligned; b_scales [N][K/32]);
 * out: fp32 [N][M].  All device pointers on the current device.  M and K
 * multiples of 128, 1 <= N <= 2^24.  The scale factors are re-arranged into
 * the engine's layouts in scratch memory that this call obtains with
 * cudaMallocAsync on `stream` and releases with cudaFreeAsync before it
 * returns.  dev_status (device int32, optional) receives a non-zero code if a
 * bounded wait inside the kernel ran out; it is the only way to learn of such
 * a time-out (out[] is then incomplete while the call still returns MOE_OK),
 * so pass it wherever a time-out matters.  Asynchronous on `stream`. */
MOE_API moe_status moe_mx_gemm(const uint8_t *a_codes, const uint8_t *a_scales, int32_t M, const uint8_t *b_codes,
                       const uint8_t *b_scales, int32_t N, int32_t K, float *out, int32_t *dev_status,
                       void *stream);

/* Quantile Balancing of the selection bias ("Kimi K3 and the New
 * Open-Weights Moat", section "How the router picks 16 of 896", Fig. 2: each
 * expert's bias is updated from the distribution of its score margins so
 * that its routed token count approaches the target load).  The pages give
 * no formula; this computes, from the logits of the last moe_forward call
 * (T must be its token count; enqueue on its stream after it) and the
 * plan's current bias b:
 *   key_te = sigmoid(l_te) + b_e (fp64);  m_te = key_te - the k-th largest
 *   key of token t among the other experts (positive exactly when e is
 *   selected, ties aside);  q_e = (m_(n) + m_(n+1)) / 2 over e's margins in
 *   descending order, n = target clamped to [1, T - 1] (target <= 0: the mean
 *   load round(T k / E));  bias_out[e] = b_e - alpha q_e  (0 < alpha <= 1).
 * With alpha = 1 an expert updated alone would get exactly n tokens.
 * bias_out: device fp32 [E].  Sigmoid scoring only.  The first call on a
 * plan allocates an [E][max_tokens] fp64 workspace (host-synchronous); later
 * calls are asynchronous and allocate nothing.  Above 128 tokens the logits
 * of experts outside a token's candidates are tensor-core estimates (see
 * moe_debug.logits), and the update reads them as they are. */
MOE_API moe_status moe_quantile_balance(void *plan, int32_t T, int32_t target, double alpha, float *bias_out,
                                        void *stream);

/* Replace the plan's selection bias with bias (device fp32 [E], finite);
 * later forward calls select on sigmoid(l) + bias.  Host-synchronous
 * (synchronises the device).  Sigmoid scoring only. */
MOE_API moe_status moe_set_bias(void *plan, const float *bias);

/* Expert-parallel dispatch, emulated on one GPU ("Kimi K3: 2.8 Trillion
 * Parameters, Four Bits at a Time", section "What it takes to serve it": each
 * token's vector ships to the devices owning its k experts and the k partial
 * outputs ship back; "What Kimi K3 asks of the hardware", section "Width: 896
 * experts and the interconnect").  The layer's routed experts read the MXFP8
 * latent, so that is the payload.  The E experts are split into `ranks`
 * contiguous slices (rank r owns experts [floor(E r / ranks),
 * floor(E (r + 1) / ranks))).  For the state of the last moe_forward call on
 * this plan (T must be its token count; enqueue on the same stream after
 * it), writes one wire row of moe_ep_row_bytes(plan) bytes per (token, slot)
 * into `wire` (device, T * k rows, 16-byte aligned): a 16-byte header of four
 * 32-bit fields {token, expert, slot, gate (fp32 bits)}, the token's L E4M3
 * codes of the latent, its L / 32 E8M0 scales, zero-padded to 16 bytes.  Rows
 * follow the layer's dispatch order, the stable sort of the (token, slot)
 * pairs by expert, so each rank's rows are contiguous: rank r sends rows
 * [rank_offsets[r], rank_offsets[r + 1]) (device int64 [ranks + 1]).
 * 1 <= ranks <= E.  Asynchronous on `stream`. */
MOE_API int64_t moe_ep_row_bytes(const void *plan);
MOE_API moe_status moe_ep_dispatch(void *plan, int32_t T, int32_t ranks, uint8_t *wire, int64_t *rank_offsets,
                                   void *stream);

/* The matching combine: expert_out (device fp32 [T * k][L]) holds the expert
 * outputs in wire-row order, as the owning ranks would return them; writes
 * c[t] = sum over the token's slots j, in slot order, of gate_j times its
 * row (device fp32 [T][L]) -- the layer's combine before its MXFP8
 * quantisation.  `wire` is the dispatch's output for the same T.
 * Asynchronous on `stream`. */
MOE_API moe_status moe_ep_combine(void *plan, int32_t T, const uint8_t *wire, const float *expert_out, float *c,
                                  void *stream);

/* Tensor-core rate probe (measurement, not part of the layer): enqueues on
 * `stream` one CTA per SM of the current device, each issuing iters x 4
 * back-to-back tcgen05.mma instructions of M = 128 x n on operand tiles held
 * in shared memory (no global memory traffic), and stores the FLOPs of the
 * launch in *flops_out (host).  Time it with events on `stream`.  kind:
 *   0  kind::mxf8f6f4, E2M1 x E4M3 with E8M0 scales (the layer's MMA), n <= 240
 *   1  kind::mxf8f6f4, E4M3 x E4M3 with E8M0 scales, n <= 240
 *   2  kind::f16, bf16 x bf16, fp32 accumulate, n <= 256
 * n a multiple of 16 (>= 16); 1 <= iters <= 2^22.  dev_status (device int32,
 * required) becomes non-zero if the final bounded wait ran out.  Needs a
 * compute capability 10.3 device (else MOE_ERR_UNSUPPORTED). */
MOE_API moe_status moe_mma_probe(int32_t kind, int32_t n, int32_t iters, int32_t *dev_status, double *flops_out,
                                 void *stream);

/* moe_mx_gemm without any allocation (the paper has no counterpart: this is
 * an entry point for callers that cannot allocate device memory -- e.g. code
 * whose device memory is owned by another allocator under a fixed budget, or
 * code that must not pay the device-wide synchronisation of cudaFree).
 * Arguments, layouts and the result are those of moe_mx_gemm.  Instead of
 * cudaMallocAsync it uses a fixed scratch array of MOE_NOALLOC_SCRATCH_BYTES
 * that lives in the library's device image: every GPU that loads the library
 * holds it until the process exits.  Limit: M*K/32 + (K/128)*(round16(N) +
 * 32)*16 + 256 <= MOE_NOALLOC_SCRATCH_BYTES (e.g. M = K = 4096 with N up to
 * about 7100);
 * larger calls return MOE_ERR_INVALID_ARG with nothing enqueued.  The first
 * call on a device looks up the array's device address (once per device, on
 * the current device); make that first call before any stream capture.  All
 * calls share the one array and it keeps the previous call's contents: calls
 * whose executions overlap on the GPU (other streams, other host threads)
 * race on it.  Makes no cudaMalloc / cudaFree call.  As with moe_mx_gemm, a
 * device time-out is reported only through dev_status. */
#define MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
MOE_API moe_status moe_mx_gemm_noalloc(const uint8_t *a_codes, const uint8_t *a_scales, int32_t M,
                                       const uint8_t *b_codes, const uint8_t *b_scales, int32_t N, int32_t K,
                                       float *out, int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
