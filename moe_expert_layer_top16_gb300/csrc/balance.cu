// Quantile Balancing of the router's selection bias ("Kimi K3 and the New
// Open-Weights Moat", section "How the router picks 16 of 896", Fig. 2: each
// expert's bias is updated from the distribution of its score margins so that
// its routed token count approaches the target load; "What Kimi K3 asks of
// the hardware": expert allocation derived from quantiles of the router
// scores).  The pages give no formula; the reading implemented here:
//   key_te  = sigmoid(l_te) + b_e                      (fp64)
//   m_te    = key_te - (the k-th largest key of token t among the experts
//             other than e): positive exactly when e is selected (ties aside)
//   q_e     = (m_(n) + m_(n+1)) / 2 over e's margins in descending order,
//             n = the target count clamped to [1, T - 1]
//   b_e    <- b_e - alpha q_e
// It reads the logits the top-k stage used (the last forward's).
//
// Kernel 1, one warp per token: the token's k-th and (k+1)-th largest keys
// (k + 1 selection rounds), then every expert's margin into [E][T].
// Kernel 2, one CTA per expert: the n-th and (n+1)-th largest of its T
// margins by a most-significant-bit-first search over order-preserving
// 64-bit keys (block-wide counts), exact and independent of thread order.
#include "internal.h"

namespace moe {

namespace {

constexpr int kQbPerLane = 32;        // E <= 1024

__device__ __forceinline__ uint64_t dkey(double v) {
    const uint64_t u = static_cast<uint64_t>(__double_as_longlong(v == 0.0 ? 0.0 : v));
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double dval(uint64_t b) {
    return __longlong_as_double(static_cast<long long>((b & 0x8000000000000000ull) ? (b & 0x7fffffffffffffffull) : ~b));
}

__global__ void qb_margin_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                                 double* __restrict__ marg) {
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int nper = (E + 31) / 32;
    uint64_t key[kQbPerLane];
#pragma unroll
    for (int i = 0; i < kQbPerLane; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0;
        if (i < nper && e < E) {
            const double l = logits[static_cast<int64_t>(t) * E + e];
            double kv = 1.0 / (1.0 + exp(-l)) + (bias ? static_cast<double>(bias[e]) : 0.0);
            if (kv != kv) kv = -INFINITY;
            key[i] = dkey(kv);
        }
    }
    // the k-th and (k+1)-th largest keys: k + 1 rounds, each taking one entry
    uint32_t taken = 0;
    uint64_t kth = 0, next = 0;
    for (int j = 0; j <= k && j < E; ++j) {
        uint64_t best = 0;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < kQbPerLane; ++i)
            if (!(taken & (1u << i)) && i < nper && lane + 32 * i < E && (bi < 0 || key[i] > best)) {
                best = key[i];
                bi = i;
            }
        uint64_t m = best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t x = __shfl_xor_sync(0xffffffffu, m, o);
            m = x > m ? x : m;
        }
        // one lane holding the maximum gives it up (the lowest such lane)
        const uint32_t holders = __ballot_sync(0xffffffffu, bi >= 0 && best == m);
        if (holders && lane == __ffs(holders) - 1) taken |= 1u << bi;
        if (j == k - 1) kth = m;
        if (j == k) next = m;
    }
    const double kv = dval(kth), nv = (k < E) ? dval(next) : -INFINITY;
#pragma unroll
    for (int i = 0; i < kQbPerLane; ++i) {
        const int e = lane + 32 * i;
        if (i < nper && e < E) {
            const double ke = dval(key[i]);
            marg[static_cast<int64_t>(e) * T + t] = ke - ((key[i] >= kth) ? nv : kv);
        }
    }
}

constexpr int kQbThreads = 1024;

// Number of margins of this CTA's expert with key bits >= v (block-wide).
__device__ __forceinline__ int count_ge(const double* m, int T, uint64_t v, int* red) {
    int c = 0;
    for (int i = threadIdx.x; i < T; i += blockDim.x) c += dkey(m[i]) >= v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
    __syncthreads();
    int s = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
    return s;
}

__global__ void __launch_bounds__(kQbThreads) qb_update_kernel(const double* __restrict__ marg, const float* __restrict__ bias,
                                                               int T, int n, double alpha, float* __restrict__ bias_out) {
    __shared__ int red[32];
    __shared__ unsigned long long best_s;
    const int e = blockIdx.x;
    const double* m = marg + static_cast<int64_t>(e) * T;
    // v_n: the largest key bits v with at least n margins >= v
    uint64_t v = 0;
    for (int bit = 63; bit >= 0; --bit) {
        const uint64_t tv = v | (1ull << bit);
        if (count_ge(m, T, tv, red) >= n) v = tv;
    }
    double mn = dval(v), mn1;
    if (count_ge(m, T, v, red) >= n + 1) {
        mn1 = mn;                                  // a tie at the n-th place
    } else {
        // the largest margin below v_n
        if (threadIdx.x == 0) best_s = 0;
        __syncthreads();
        unsigned long long b = 0;
        for (int i = threadIdx.x; i < T; i += blockDim.x) {
            const uint64_t ki = dkey(m[i]);
            if (ki < v && ki > b) b = ki;
        }
        atomicMax(&best_s, b);
        __syncthreads();
        mn1 = dval(best_s);
    }
    if (threadIdx.x == 0) {
        const double b0 = bias ? static_cast<double>(bias[e]) : 0.0;
        bias_out[e] = static_cast<float>(b0 - alpha * 0.5 * (mn + mn1));
    }
}

}  // namespace

cudaError_t launch_quantile_balance(const float* logits, const float* bias, int T, int E, int k, int target,
                                    double alpha, double* marg, float* bias_out, cudaStream_t s) {
    if (T < 2 || E < 1 || E > 32 * kQbPerLane || k < 1 || k >= E || !(alpha > 0.0 && alpha <= 1.0))
        return cudaErrorInvalidValue;
    const int n = target < 1 ? 1 : (target > T - 1 ? T - 1 : target);
    qb_margin_kernel<<<(T * 32 + 255) / 256, 256, 0, s>>>(logits, bias, T, E, k, marg);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    qb_update_kernel<<<E, kQbThreads, 0, s>>>(marg, bias, T, n, alpha, bias_out);
    return cudaGetLastError();
}

}  // namespace moe
