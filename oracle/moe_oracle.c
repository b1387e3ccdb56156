/*
 * CPU oracle for the K3-style sparse MoE layer -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct restatement of what the layer computes,
 * in fp64.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the CUDA library never does, and this file shares no code,
 * header, table or constant with it.
 *
 * Sources (page title, then section / figure):
 *  - "Kimi K3 and the New Open-Weights Moat", section "Sparse computation:
 *    latent experts and routing": 16 of 896 routed experts plus two always-on
 *    shared experts; shared experts at the full 7168 width; routed path
 *    projected into a 3584-wide latent, experts run there, the combined result
 *    projected back ("Stable LatentMoE").
 *  - same page, section "How the router picks 16 of 896" and Fig. 2: a sigmoid
 *    score per expert, top-k on score + selection bias, raw sigmoid scores of
 *    the winners normalised by their sum; the bias is excluded from the
 *    weights; routed and shared branches are summed.
 *  - same page, section "Precision and deployment", Fig. 6: MX blocks of 32
 *    values sharing one 8-bit power-of-two scale; E2M1 (MXFP4) and E4M3
 *    (MXFP8) elements; element encodings per the OCP MX v1.0 specification
 *    that the page cites.
 *  - "Kimi K3: 2.8 Trillion Parameters, Four Bits at a Time", section "Four
 *    bits from the start": the MXFP4 block encoder (shared exponent =
 *    floor(log2 amax) - 2, magnitude clipped to 6, nearest grid level with the
 *    first level winning a tie) and the E2M1 grid {0,.5,1,1.5,2,3,4,6}.
 *  - same page, section "What it takes to serve it", the one-page MoE data
 *    path: route (top-k of logits, softmax over the k winners), dispatch
 *    (stable sort of the flattened (token, slot) pairs by expert, per-expert
 *    counts and offsets), one matrix product per expert segment, and a
 *    gate-weighted scatter-add back to [T, D].
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes):
 *  - MXFP8 shared exponent = floor(log2 amax) - 8 (8 = emax of E4M3, by
 *    analogy with "emax of E2M1 is 2"); elements rounded to nearest, ties to
 *    even, saturating at +-448; a block of zeros gets scale code 0.
 *  - Shared exponents are clamped to the E8M0 range [-127, 127].
 *  - MXFP4 zero block: all codes 0 and scale code 0 (the page writes zeros).
 *  - Sign bit of an encoded element = sign bit of the input value.
 *  - Expert FFN: h = SiLU(x W_gate^T) * (x W_up^T), out = h W_down^T; the
 *    activation is SiLU(g) = g / (1 + exp(-g)).
 *  - Every GEMM / activation output is rounded to fp32 before it is
 *    quantised or consumed; sums themselves run in fp64.
 *  - Router input is the fp32 latent z ("Kimi K3: 2.8 Trillion Parameters,
 *    Four Bits at a Time", section "The shape of the model": latent-space
 *    routing); "What Kimi K3 asks of the hardware" leaves the latent part
 *    unspecified, so routing on the hidden state x is kept as an option.
 *    Logits are summed in fp64.
 *  - Slot order within a token: descending key, tie -> lower expert id.
 *  - Combine accumulates the k slots of a token in slot order.
 *  - Mixed precision (the scheme of "Precision and deployment", Fig. 6: only
 *    the routed experts' weights are MXFP4 and their inputs MXFP8; the latent
 *    projections, the shared experts and the router stay at higher
 *    precision): "higher precision" is read as BF16 weights and BF16 inputs
 *    for the latent projections and the shared experts (the hidden state x is
 *    already bf16), fp32 for the router.  Values are rounded from fp32 to
 *    bf16 to nearest, ties to even; the latent z stays fp32 for the router
 *    and is MXFP8-quantised for the routed experts; the shared activation and
 *    the combine output are rounded to bf16 before the up-projection.
 *
 * Byte layouts (this file's own): an MX matrix [rows][K] is `codes`
 * [rows][K/2] (element 2i in the low nibble of byte i) for MXFP4 or
 * [rows][K] for MXFP8, plus `scales` [rows][K/32] E8M0 codes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Element decoding (OCP MX v1.0, cited by "Precision and deployment"). */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(int code)
{
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal; S.1111.111 is NaN; no infinities; largest normal 448. */
double orc_e4m3_decode(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10);     /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* E8M0: unsigned exponent, bias 127; code 255 is NaN. */
double orc_e8m0_decode(int code)
{
    if ((code & 255) == 255)
        return NAN;
    return ldexp(1.0, (code & 255) - 127);
}

/* floor(log2(a)) for finite a > 0, exactly (frexp gives a = f * 2^ex with
 * f in [0.5, 1)). */
static int floor_log2(double a)
{
    int ex;
    frexp(a, &ex);
    return ex - 1;
}

static int clamp_e8m0(int e) { return e < -127 ? -127 : (e > 127 ? 127 : e); }

/* ------------------------------------------------------------------ */
/* BF16: 1 sign, 8 exponent, 7 mantissa bits -- the upper half of an    */
/* fp32.                                                                */

double orc_bf16_decode(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* fp32 -> nearest bf16, ties to even; NaN stays a quiet NaN, infinities
 * and overflow to infinity follow from the rounding. */
uint16_t orc_bf16_round(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;                         /* carries into the exponent as it should */
    return (uint16_t)keep;
}

void orc_bf16_round_array(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_round(v[i]);
}

/* y[m] = fp32(sum_k a[k] * bf16(W[m][k])) for W bf16 [M][K]. */
static void bf16_gemv_f32(const double *a, const uint16_t *W, int64_t M, int64_t K, float *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += a[k] * orc_bf16_decode(W[m * K + k]);
        y[m] = (float)acc;
    }
}

/* ------------------------------------------------------------------ */
/* MXFP4 encoder: the block algorithm of "Four bits from the start".   */

void orc_mxfp4_encode_f64(const double *w, int64_t rows, int64_t K,
                          uint8_t *codes, uint8_t *scales)
{
    int64_t nb = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const double *v = w + r * K + b * 32;
            uint8_t *c = codes + r * (K / 2) + b * 16;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                if (fabs(v[i]) > amax)
                    amax = fabs(v[i]);
            if (amax == 0.0) {              /* the page writes zeros */
                memset(c, 0, 16);
                scales[r * nb + b] = 0;
                continue;
            }
            int e = clamp_e8m0(floor_log2(amax) - 2);   /* emax of E2M1 is 2 */
            double scale = ldexp(1.0, e);
            for (int i = 0; i < 32; ++i) {
                double x = fabs(v[i]) / scale;
                if (x > 6.0)
                    x = 6.0;                             /* clip to the grid max */
                int idx = 0;                             /* nearest level; the   */
                double best = fabs(x - E2M1_MAG[0]);     /* first one wins a tie */
                for (int l = 1; l < 8; ++l) {
                    double d = fabs(x - E2M1_MAG[l]);
                    if (d < best) {
                        best = d;
                        idx = l;
                    }
                }
                int code = idx | (signbit(v[i]) ? 8 : 0);
                if (i & 1)
                    c[i / 2] = (uint8_t)(c[i / 2] | (code << 4));
                else
                    c[i / 2] = (uint8_t)code;
            }
            scales[r * nb + b] = (uint8_t)(e + 127);
        }
    }
}

void orc_mxfp4_encode_f32(const float *w, int64_t rows, int64_t K,
                          uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel
    {
        double *tmp = (double *)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            for (int64_t i = 0; i < K; ++i)
                tmp[i] = (double)w[r * K + i];
            orc_mxfp4_encode_f64(tmp, 1, K, codes + r * (K / 2), scales + r * (K / 32));
        }
        free(tmp);
    }
}

/* ------------------------------------------------------------------ */
/* MXFP8 (E4M3) quantiser.                                              */

/* Nearest E4M3 value to v, ties to the even code, saturating at +-448.
 * Brute force over every finite magnitude code. */
static uint8_t e4m3_encode(double v)
{
    int s = signbit(v) ? 0x80 : 0;
    double a = fabs(v);
    if (!(a < 448.0))
        return (uint8_t)(s | 0x7E);
    int best = 0;
    double bd = a;
    for (int c = 1; c <= 126; ++c) {
        double d = fabs(a - orc_e4m3_decode(c));
        if (d < bd || (d == bd && (c & 1) == 0)) {
            bd = d;
            best = c;
        }
    }
    return (uint8_t)(s | best);
}

uint8_t orc_e4m3_encode(double v) { return e4m3_encode(v); }

/* One 32-block of fp32 values -> 32 E4M3 codes and one E8M0 scale code. */
static void mxfp8_block(const float *v, uint8_t *codes, uint8_t *scale)
{
    double amax = 0.0;
    for (int i = 0; i < 32; ++i)
        if (fabs((double)v[i]) > amax)
            amax = fabs((double)v[i]);
    int e = (amax == 0.0) ? -127 : clamp_e8m0(floor_log2(amax) - 8); /* emax of E4M3 is 8 */
    for (int i = 0; i < 32; ++i)
        codes[i] = e4m3_encode(ldexp((double)v[i], -e));
    *scale = (uint8_t)(e + 127);
}

void orc_mxfp8_quantize(const float *v, int64_t rows, int64_t K,
                        uint8_t *codes, uint8_t *scales)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < K / 32; ++b)
            mxfp8_block(v + r * K + b * 32, codes + r * K + b * 32, scales + r * (K / 32) + b);
}

/* ------------------------------------------------------------------ */
/* Block-scaled products.                                               */

typedef struct {
    const uint8_t *codes;   /* MXFP4 [rows][K/2] */
    const uint8_t *scales;  /* [rows][K/32] */
} orc_mx;

/* Decode an MXFP8 vector of length K into doubles. */
static void dq_mxfp8(const uint8_t *codes, const uint8_t *scales, int64_t K, double *out)
{
    for (int64_t i = 0; i < K; ++i)
        out[i] = orc_e4m3_decode(codes[i]) * orc_e8m0_decode(scales[i / 32]);
}

/* sum_k a[k] * dq(W[row][k]) in fp64, k ascending. */
static double mx4_row_dot(const double *a, const orc_mx *W, int64_t row, int64_t K)
{
    const uint8_t *c = W->codes + row * (K / 2);
    const uint8_t *s = W->scales + row * (K / 32);
    double acc = 0.0;
    for (int64_t b = 0; b < K / 32; ++b) {
        double sc = orc_e8m0_decode(s[b]);
        for (int64_t k = b * 32; k < b * 32 + 32; ++k) {
            int code = (k & 1) ? (c[k / 2] >> 4) : (c[k / 2] & 15);
            acc += a[k] * (orc_e2m1_decode(code) * sc);
        }
    }
    return acc;
}

/* out[n][m] = sum_k dq(B[n][k]) * dq(A[m][k]); A MXFP4 [M][K], B MXFP8 [N][K]. */
void orc_mx_matmul(const uint8_t *a_codes, const uint8_t *a_scales, int64_t M,
                   const uint8_t *b_codes, const uint8_t *b_scales, int64_t N,
                   int64_t K, double *out)
{
    orc_mx A = {a_codes, a_scales};
    double *bd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int64_t n = 0; n < N; ++n) {
        dq_mxfp8(b_codes + n * K, b_scales + n * (K / 32), K, bd);
        for (int64_t m = 0; m < M; ++m)
            out[n * M + m] = mx4_row_dot(bd, &A, m, K);
    }
    free(bd);
}

/* y[m] = fp32(sum_k a[k] * dq(W[m][k])) for m < M; rows split over threads. */
static void mx4_gemv_f32(const double *a, const orc_mx *W, int64_t M, int64_t K, float *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        y[m] = (float)mx4_row_dot(a, W, m, K);
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------------ */
/* Routing: "How the router picks 16 of 896" (sigmoid mode) and the     */
/* one-page data path (softmax-over-winners mode).                      */

void orc_route(const double *logits, const float *bias, int64_t T, int E, int k,
               int softmax, int32_t *idx, double *gates)
{
    double *key = (double *)malloc(sizeof(double) * (size_t)E);
    char *taken = (char *)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        const double *l = logits + t * E;
        /* Without a bias the key sigmoid(l) orders exactly as l (sigmoid is
         * strictly increasing); ranking l itself keeps that order where the
         * fp64 sigmoid rounds to 1 (l above about 37). */
        for (int e = 0; e < E; ++e) {
            key[e] = (softmax || !bias) ? l[e] : sigmoid(l[e]) + (double)bias[e];
            taken[e] = 0;
        }
        /* k rounds of "largest remaining key, lower id on a tie". */
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || key[e] > key[best]))
                    best = e;
            taken[best] = 1;
            idx[t * k + j] = best;
        }
        double sum = 0.0;
        if (softmax) {
            double lmax = l[idx[t * k]];
            for (int j = 1; j < k; ++j)
                if (l[idx[t * k + j]] > lmax)
                    lmax = l[idx[t * k + j]];
            for (int j = 0; j < k; ++j)
                sum += (gates[t * k + j] = exp(l[idx[t * k + j]] - lmax));
        } else {
            /* raw sigmoid scores of the winners; the bias is not part of them */
            for (int j = 0; j < k; ++j)
                sum += (gates[t * k + j] = sigmoid(l[idx[t * k + j]]));
        }
        for (int j = 0; j < k; ++j)
            gates[t * k + j] /= sum;
    }
    free(key);
    free(taken);
}

/* ------------------------------------------------------------------ */
/* Quantile Balancing ("Kimi K3 and the New Open-Weights Moat", section  */
/* "How the router picks 16 of 896", Fig. 2: each expert's selection     */
/* bias is updated from the distribution of its score margins so that    */
/* its routed token count approaches the target load; "What Kimi K3 asks */
/* of the hardware": allocation derived from quantiles of the router     */
/* scores).  The pages give no formula; the reading used here:           */
/*  - key_te = sigmoid(l_te) + b_e;                                      */
/*  - the margin of expert e for token t is key_te minus the key e must  */
/*    beat: the k-th largest key among the other experts (the (k+1)-th   */
/*    largest key of the token when e is among its top k, else the k-th) */
/*    -- e is selected exactly when its margin is positive (ties aside); */
/*  - with m_(1) >= m_(2) >= ... e's margins in descending order and n   */
/*    the target count (clamped to [1, T-1]), q_e = (m_(n) + m_(n+1))/2  */
/*    is the shift of e's bias that leaves exactly n positive margins    */
/*    when the other biases stay as they are;                            */
/*  - b_e <- b_e - alpha q_e (alpha in (0, 1]: the drift toward the      */
/*    target).                                                           */

static int cmp_desc(const void *a, const void *b)
{
    double x = *(const double *)a, y = *(const double *)b;
    return (x < y) - (x > y);
}

void orc_quantile_balance(const double *logits, const float *bias, int64_t T, int E, int k, int64_t target,
                          double alpha, double *bias_out)
{
    double *key = (double *)malloc(sizeof(double) * (size_t)E);
    double *srt = (double *)malloc(sizeof(double) * (size_t)E);
    double *marg = (double *)malloc(sizeof(double) * (size_t)(T * E));   /* [E][T] */
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            key[e] = sigmoid(logits[t * E + e]) + (bias ? (double)bias[e] : 0.0);
            srt[e] = key[e];
        }
        qsort(srt, (size_t)E, sizeof(double), cmp_desc);
        double kth = srt[k - 1], next = (k < E) ? srt[k] : -INFINITY;
        for (int e = 0; e < E; ++e) {
            /* e beats the k-th largest of the others: next when e is at or
             * above the k-th key, kth otherwise */
            double thr = (key[e] >= kth) ? next : kth;
            marg[(int64_t)e * T + t] = key[e] - thr;
        }
    }
    int64_t n = target < 1 ? 1 : (target > T - 1 ? T - 1 : target);
    for (int e = 0; e < E; ++e) {
        double *m = marg + (int64_t)e * T;
        qsort(m, (size_t)T, sizeof(double), cmp_desc);
        double q = 0.5 * (m[n - 1] + m[n]);
        bias_out[e] = (bias ? (double)bias[e] : 0.0) - alpha * q;
    }
    free(key);
    free(srt);
    free(marg);
}

/* Dispatch of the one-page data path: per-expert counts, exclusive offsets,
 * and the stable sort of flat indices f = t*k + j by expert. */
void orc_permute(const int32_t *idx, int64_t T, int k, int E,
                 int32_t *counts, int32_t *offsets, int32_t *order)
{
    int64_t n = T * k;
    memset(counts, 0, sizeof(int32_t) * (size_t)E);
    for (int64_t f = 0; f < n; ++f)
        counts[idx[f]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t f = 0; f < n; ++f) {       /* ascending f keeps the sort stable */
        int e = idx[f];
        order[offsets[e] + fill[e]++] = (int32_t)f;
    }
    free(fill);
}

/* Combine of the one-page data path: y[t] += gate[f] * rows[p] for the
 * permuted row p holding flat index f = order[p], t = f / k. */
void orc_combine(const double *rows, const int32_t *order, const double *gates,
                 int64_t T, int k, int64_t D, double *y)
{
    memset(y, 0, sizeof(double) * (size_t)(T * D));
    for (int64_t p = 0; p < T * k; ++p) {
        int64_t f = order[p], t = f / k;
        for (int64_t d = 0; d < D; ++d)
            y[t * D + d] += gates[f] * rows[p * D + d];
    }
}

/* ------------------------------------------------------------------ */
/* The layer.                                                           */

typedef struct {
    int32_t D, L, E, k, I, S, Is;
    int32_t softmax;        /* 1: softmax over winners (toy); 0: sigmoid + bias */
    int32_t route_hidden;   /* 1: the router reads the hidden state x ([E][D] weights); 0: the latent z */
    int32_t mixed;          /* 1: BF16 latent projections and shared experts (mixed scheme); 0: all MXFP4 */
} orc_cfg;

typedef struct {
    orc_mx p_down;          /* [L][D]  latent down-projection */
    orc_mx p_up;            /* [D][L]  latent up-projection   */
    const orc_mx *w_gate;   /* E x [I][L]  (codes NULL: expert not supplied) */
    const orc_mx *w_up;     /* E x [I][L] */
    const orc_mx *w_down;   /* E x [L][I] */
    const orc_mx *s_gate;   /* S x [Is][D] */
    const orc_mx *s_up;     /* S x [Is][D] */
    const orc_mx *s_down;   /* S x [D][Is] */
    const float *router;    /* [E][L] fp32 (latent routing) or [E][D] (hidden routing) */
    const float *bias;      /* [E] fp32 or NULL */
    /* mixed scheme only: BF16 weights of the latent projections and the
     * shared experts (the MXFP4 ones above are then unused) */
    const uint16_t *p_down_bf;   /* [L][D] */
    const uint16_t *p_up_bf;     /* [D][L] */
    const uint16_t *s_gate_bf;   /* [S][Is][D] */
    const uint16_t *s_up_bf;     /* [S][Is][D] */
    const uint16_t *s_down_bf;   /* [S][D][Is] */
} orc_weights;

/* Optional outputs, one row per processed token (NULL = not wanted). */
typedef struct {
    float *y;                       /* [n][D] */
    uint8_t *xq, *xs;               /* [n][D], [n][D/32] */
    float *z;                       /* [n][L] */
    uint8_t *zq, *zs;               /* [n][L], [n][L/32] */
    float *hs;                      /* [n][S*Is] shared-expert activation, fp32 */
    uint8_t *hsq, *hss;             /* [n][S*Is], [n][S*Is/32] */
    double *logits;                 /* [n][E] */
    int32_t *idx;                   /* [n][k] */
    double *gates;                  /* [n][k] */
    float *h;                       /* [n][k][I] */
    uint8_t *hq, *hqs;              /* [n][k][I], [n][k][I/32] */
    float *o;                       /* [n][k][L] */
    float *c;                       /* [n][L] */
    uint8_t *cq, *cs;               /* [n][L], [n][L/32] */
} orc_out;

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_MISSING_EXPERT = 2 };

/* Forward pass of the layer for n tokens x_bf16[n][D].
 * force_idx (optional, [n][k]) replaces the router's selection (the gates
 * are still the normalised scores of the forced experts).
 * route_only stops after the gates. */
int orc_moe_forward(const orc_cfg *cfg, const orc_weights *W, const uint16_t *x_bf16,
                    int64_t n, const int32_t *force_idx, int route_only, orc_out *out)
{
    const int64_t D = cfg->D, L = cfg->L, E = cfg->E, k = cfg->k, I = cfg->I,
                  S = cfg->S, Is = cfg->Is;
    if (D % 32 || L % 32 || I % 32 || Is % 32 || k < 1 || k > E)
        return ORC_ERR_ARG;
    const int64_t SIs = S * Is;
    size_t big = (size_t)(D > SIs ? D : SIs);
    if ((size_t)L > big) big = (size_t)L;
    if ((size_t)I > big) big = (size_t)I;
    float *xf = malloc(sizeof(float) * D);
    uint8_t *q = malloc(big), *qs = malloc(big / 32);
    double *a = malloc(sizeof(double) * big);
    float *z = malloc(sizeof(float) * L), *g = malloc(sizeof(float) * big), *u = malloc(sizeof(float) * big);
    float *hsh = malloc(sizeof(float) * SIs);
    uint8_t *zq = malloc(L), *zs = malloc(L / 32), *hsq = malloc(SIs), *hss = malloc(SIs / 32);
    double *lg = malloc(sizeof(double) * E), *gate = malloc(sizeof(double) * k);
    int32_t *sel = malloc(sizeof(int32_t) * k);
    float *o = malloc(sizeof(float) * k * L), *c = malloc(sizeof(float) * L);
    float *y = malloc(sizeof(float) * D);
    int rc = ORC_OK;

    for (int64_t t = 0; t < n && rc == ORC_OK; ++t) {
        /* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 */
        for (int64_t d = 0; d < D; ++d) {
            uint32_t bits = (uint32_t)x_bf16[t * D + d] << 16;
            memcpy(&xf[d], &bits, 4);
        }
        if (cfg->mixed) {
            /* mixed scheme: the projections and shared experts read x in bf16 */
            for (int64_t d = 0; d < D; ++d)
                a[d] = (double)xf[d];
        } else {
            /* A1: activations enter the GEMMs as MXFP8 */
            orc_mxfp8_quantize(xf, 1, D, q, qs);
            if (out->xq) memcpy(out->xq + t * D, q, D);
            if (out->xs) memcpy(out->xs + t * (D / 32), qs, D / 32);
            dq_mxfp8(q, qs, D, a);
        }

        /* latent down-projection z = x P_down^T */
        if (cfg->mixed)
            bf16_gemv_f32(a, W->p_down_bf, L, D, z);
        else
            mx4_gemv_f32(a, &W->p_down, L, D, z);
        orc_mxfp8_quantize(z, 1, L, zq, zs);
        if (out->z) memcpy(out->z + t * L, z, sizeof(float) * L);
        if (out->zq) memcpy(out->zq + t * L, zq, L);
        if (out->zs) memcpy(out->zs + t * (L / 32), zs, L / 32);

        /* shared experts at full width: h_s = SiLU(x S_gate^T) * (x S_up^T) */
        for (int64_t s = 0; s < S; ++s) {
            if (cfg->mixed) {
                bf16_gemv_f32(a, W->s_gate_bf + s * Is * D, Is, D, g);
                bf16_gemv_f32(a, W->s_up_bf + s * Is * D, Is, D, u);
            } else {
                mx4_gemv_f32(a, &W->s_gate[s], Is, D, g);
                mx4_gemv_f32(a, &W->s_up[s], Is, D, u);
            }
            for (int64_t i = 0; i < Is; ++i)
                hsh[s * Is + i] = (float)(silu((double)g[i]) * (double)u[i]);
        }
        if (out->hs) memcpy(out->hs + t * SIs, hsh, sizeof(float) * SIs);
        if (!cfg->mixed) {
            orc_mxfp8_quantize(hsh, 1, SIs, hsq, hss);
            if (out->hsq) memcpy(out->hsq + t * SIs, hsq, SIs);
            if (out->hss) memcpy(out->hss + t * (SIs / 32), hss, SIs / 32);
        }

        /* router logits, fp64 sum of fp32 products: on the latent z by
         * default, on the hidden state x (exactly its bf16 value) when the
         * router is configured to read the hidden state */
        {
            const float *rin = cfg->route_hidden ? xf : z;
            const int64_t RK = cfg->route_hidden ? D : L;
            for (int64_t e = 0; e < E; ++e) {
                double acc = 0.0;
                for (int64_t l = 0; l < RK; ++l)
                    acc += (double)rin[l] * (double)W->router[e * RK + l];
                lg[e] = acc;
            }
        }
        if (out->logits) memcpy(out->logits + t * E, lg, sizeof(double) * E);
        orc_route(lg, W->bias, 1, (int)E, (int)k, cfg->softmax, sel, gate);
        if (force_idx) {
            /* forced selection: gates are the normalised scores of these experts */
            double sum = 0.0, lmax = -INFINITY;
            for (int64_t j = 0; j < k; ++j) {
                sel[j] = force_idx[t * k + j];
                if (sel[j] < 0 || sel[j] >= E) { rc = ORC_ERR_ARG; break; }
                if (lg[sel[j]] > lmax) lmax = lg[sel[j]];
            }
            if (rc != ORC_OK) break;
            for (int64_t j = 0; j < k; ++j)
                sum += (gate[j] = cfg->softmax ? exp(lg[sel[j]] - lmax) : sigmoid(lg[sel[j]]));
            for (int64_t j = 0; j < k; ++j)
                gate[j] /= sum;
        }
        if (out->idx) memcpy(out->idx + t * k, sel, sizeof(int32_t) * k);
        if (out->gates) memcpy(out->gates + t * k, gate, sizeof(double) * k);
        if (route_only)
            continue;

        /* routed experts on the latent */
        double *za = malloc(sizeof(double) * L);
        dq_mxfp8(zq, zs, L, za);
        for (int64_t j = 0; j < k && rc == ORC_OK; ++j) {
            int e = sel[j];
            if (!W->w_gate[e].codes || !W->w_up[e].codes || !W->w_down[e].codes) {
                rc = ORC_ERR_MISSING_EXPERT;
                break;
            }
            mx4_gemv_f32(za, &W->w_gate[e], I, L, g);
            mx4_gemv_f32(za, &W->w_up[e], I, L, u);
            float *h = malloc(sizeof(float) * I);
            for (int64_t i = 0; i < I; ++i)
                h[i] = (float)(silu((double)g[i]) * (double)u[i]);
            orc_mxfp8_quantize(h, 1, I, q, qs);
            if (out->h) memcpy(out->h + (t * k + j) * I, h, sizeof(float) * I);
            if (out->hq) memcpy(out->hq + (t * k + j) * I, q, I);
            if (out->hqs) memcpy(out->hqs + (t * k + j) * (I / 32), qs, I / 32);
            dq_mxfp8(q, qs, I, a);
            mx4_gemv_f32(a, &W->w_down[e], L, I, o + j * L);
            free(h);
        }
        free(za);
        if (rc != ORC_OK)
            break;
        if (out->o) memcpy(out->o + t * k * L, o, sizeof(float) * k * L);

        /* gate-weighted sum of the k expert outputs, in slot order */
        for (int64_t l = 0; l < L; ++l) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j)
                acc += gate[j] * (double)o[j * L + l];
            c[l] = (float)acc;
        }
        if (out->c) memcpy(out->c + t * L, c, sizeof(float) * L);
        double *ca = malloc(sizeof(double) * L), *ha = malloc(sizeof(double) * (SIs > 0 ? SIs : 1));
        if (cfg->mixed) {
            /* the up-projection's inputs are rounded to bf16 */
            for (int64_t l = 0; l < L; ++l)
                ca[l] = orc_bf16_decode(orc_bf16_round(c[l]));
            for (int64_t i = 0; i < SIs; ++i)
                ha[i] = orc_bf16_decode(orc_bf16_round(hsh[i]));
        } else {
            orc_mxfp8_quantize(c, 1, L, q, qs);
            if (out->cq) memcpy(out->cq + t * L, q, L);
            if (out->cs) memcpy(out->cs + t * (L / 32), qs, L / 32);
            dq_mxfp8(q, qs, L, ca);
            dq_mxfp8(hsq, hss, SIs, ha);
        }

        /* y = c P_up^T + h_s S_down^T: routed branch up-projected, shared
         * branch summed, one fp64 sum per output */
#pragma omp parallel for schedule(static)
        for (int64_t d = 0; d < D; ++d) {
            double acc = 0.0;
            if (cfg->mixed) {
                for (int64_t l = 0; l < L; ++l)
                    acc += ca[l] * orc_bf16_decode(W->p_up_bf[d * L + l]);
                for (int64_t s = 0; s < S; ++s)
                    for (int64_t i = 0; i < Is; ++i)
                        acc += ha[s * Is + i] * orc_bf16_decode(W->s_down_bf[(s * D + d) * Is + i]);
            } else {
                acc = mx4_row_dot(ca, &W->p_up, d, L);
                for (int64_t s = 0; s < S; ++s)
                    acc += mx4_row_dot(ha + s * Is, &W->s_down[s], d, Is);
            }
            y[d] = (float)acc;
        }
        free(ca);
        free(ha);
        if (out->y) memcpy(out->y + t * D, y, sizeof(float) * D);
    }
    free(xf); free(q); free(qs); free(a); free(z); free(g); free(u); free(hsh);
    free(zq); free(zs); free(hsq); free(hss); free(lg); free(gate); free(sel);
    free(o); free(c); free(y);
    return rc;
}
