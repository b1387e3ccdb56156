// Expert-parallel dispatch and combine, emulated on one GPU ("Kimi K3: 2.8
// Trillion Parameters, Four Bits at a Time", section "What it takes to serve
// it": each token's vector ships to the devices owning its k experts and the
// k partial outputs ship back, about 2 k d bytes per token at FP8; "What Kimi
// K3 asks of the hardware", section "Width: 896 experts and the
// interconnect": the two all-to-all exchanges of an expert-parallel layer).
//
// The E experts are split into R contiguous slices, one per (virtual) rank:
// rank r owns experts [floor(E r / R), floor(E (r + 1) / R)).  The dispatch
// writes one wire row per (token, slot): a 16-byte header {token, expert,
// slot, gate}, the token's MXFP8 latent codes (L bytes, E4M3) and its block
// scales (L / 32 bytes, E8M0), padded to 16 bytes.  Rows follow the layer's
// dispatch order -- the stable sort of the (token, slot) pairs by expert --
// so every rank's rows form one contiguous segment of the wire buffer, the
// send buffer of that rank in an all-to-all.  The combine takes the experts'
// fp32 outputs in wire-row order and forms c[t] = sum_j gate_j out_j in slot
// order (the layer's own combine).
#include "internal.h"

namespace moe {

namespace {

// One warp per wire row p (a sorted position).
__global__ void ep_pack_kernel(const int32_t* __restrict__ sorted_token, const int32_t* __restrict__ offsets,
                               const int32_t* __restrict__ idx, const float* __restrict__ gw,
                               const uint8_t* __restrict__ zq, const uint32_t* __restrict__ zsf, int64_t zsf_pitch,
                               int T, int k, int E, int L, uint8_t* __restrict__ wire, int64_t row_bytes) {
    const int64_t p = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (p >= static_cast<int64_t>(T) * k) return;
    const int t = sorted_token[p];
    // the expert of sorted position p: offsets[e] <= p < offsets[e + 1]
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    const int e = lo;
    // the token's slot holding that expert
    const int cand = (lane < k) ? idx[static_cast<int64_t>(t) * k + lane] : -1;
    const uint32_t hit = __ballot_sync(0xffffffffu, cand == e);
    const int j = hit ? __ffs(hit) - 1 : 0;
    uint8_t* row = wire + p * row_bytes;
    if (lane == 0) {
        int4 h;
        h.x = t;
        h.y = e;
        h.z = j;
        h.w = __float_as_int(gw[static_cast<int64_t>(t) * k + j]);
        *reinterpret_cast<int4*>(row) = h;
    }
    // payload: codes then scales (raw planes: word [col / 128][t], byte (col % 128) / 32)
    const uint4* src = reinterpret_cast<const uint4*>(zq + static_cast<int64_t>(t) * L);
    uint4* dst = reinterpret_cast<uint4*>(row + 16);
    for (int i = lane; i < L / 16; i += 32) dst[i] = src[i];
    uint32_t* sdst = reinterpret_cast<uint32_t*>(row + 16 + L);
    for (int w = lane; w < L / 128; w += 32) sdst[w] = zsf[static_cast<int64_t>(w) * zsf_pitch + t];
}

__global__ void ep_rank_offsets_kernel(const int32_t* __restrict__ offsets, int E, int R, int64_t* __restrict__ out) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r > R) return;
    out[r] = offsets[static_cast<int64_t>(E) * r / R];
}

// inverse of the dispatch order: inv[t * k + slot] = wire row
__global__ void ep_invert_kernel(const uint8_t* __restrict__ wire, int64_t row_bytes, int64_t rows, int k,
                                 int32_t* __restrict__ inv) {
    const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (p >= rows) return;
    const int4 h = *reinterpret_cast<const int4*>(wire + p * row_bytes);
    inv[static_cast<int64_t>(h.x) * k + h.z] = static_cast<int32_t>(p);
}

// c[t][l] = sum over slots j (in order) of gate_j * out[row(t, j)][l]; CTA
// (t, chunk of 256 columns), the gates from the wire headers.
__global__ void ep_combine_kernel(const uint8_t* __restrict__ wire, int64_t row_bytes, const int32_t* __restrict__ inv,
                                  const float* __restrict__ out, int k, int L, float* __restrict__ c) {
    __shared__ int rows_s[32];
    __shared__ float g_s[32];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        const int r = inv[static_cast<int64_t>(t) * k + threadIdx.x];
        rows_s[threadIdx.x] = r;
        g_s[threadIdx.x] = __int_as_float(reinterpret_cast<const int4*>(wire + static_cast<int64_t>(r) * row_bytes)->w);
    }
    __syncthreads();
    const int col = blockIdx.y * blockDim.x + threadIdx.x;
    if (col >= L) return;
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) acc = fmaf(g_s[j], out[static_cast<int64_t>(rows_s[j]) * L + col], acc);
    c[static_cast<int64_t>(t) * L + col] = acc;
}

}  // namespace

int64_t ep_row_bytes(int L) { return (16 + L + L / 32 + 15) / 16 * 16; }

cudaError_t launch_ep_pack(const int32_t* sorted_token, const int32_t* offsets, const int32_t* idx, const float* gw,
                           const uint8_t* zq, const uint32_t* zsf, int64_t zsf_pitch, int T, int k, int E, int L,
                           int R, uint8_t* wire, int64_t* rank_offsets, cudaStream_t s) {
    if (T < 1 || k < 1 || k > 32 || E < 1 || R < 1 || R > E || L % 128) return cudaErrorInvalidValue;
    const int64_t warps = static_cast<int64_t>(T) * k;
    ep_pack_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, s>>>(
        sorted_token, offsets, idx, gw, zq, zsf, zsf_pitch, T, k, E, L, wire, ep_row_bytes(L));
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    ep_rank_offsets_kernel<<<(R + 1 + 127) / 128, 128, 0, s>>>(offsets, E, R, rank_offsets);
    return cudaGetLastError();
}

cudaError_t launch_ep_combine(const uint8_t* wire, const float* out, int T, int k, int L, int32_t* inv, float* c,
                              cudaStream_t s) {
    if (T < 1 || k < 1 || k > 32 || L < 1) return cudaErrorInvalidValue;
    const int64_t rows = static_cast<int64_t>(T) * k;
    const int64_t rb = ep_row_bytes(L);
    ep_invert_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, s>>>(wire, rb, rows, k, inv);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    dim3 grid(T, (L + 255) / 256);
    ep_combine_kernel<<<grid, 256, 0, s>>>(wire, rb, inv, out, k, L, c);
    return cudaGetLastError();
}

}  // namespace moe
