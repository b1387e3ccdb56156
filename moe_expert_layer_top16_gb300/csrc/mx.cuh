// Device-side MX format helpers: E8M0 shared exponents, E4M3 conversion,
// and the scale-plane byte layout used by every activation buffer.
//
// MXFP8 quantisation of a 32-element block (blocks of 32 sharing one 8-bit
// power-of-two scale: "Kimi K3 and the New Open-Weights Moat", section
// "Precision and deployment", Fig. 6):
//   e     = floor(log2(amax)) - 8   (8 = largest exponent of E4M3), clamped to
//           the E8M0 range [-127, 127]; an all-zero block gets e = -127
//   code  = E4M3(v * 2^-e), round to nearest even, saturating at +-448
//   scale = e + 127
#pragma once
#include <cstdint>

namespace moe {

// Shared exponent of an MXFP8 block with absolute maximum `amax` (finite).
__device__ __forceinline__ int mx8_exponent(float amax) {
    const uint32_t b = __float_as_uint(amax);
    const int biased = static_cast<int>((b >> 23) & 0xFFu);
    if (biased == 0) return -127;                 // zero or subnormal: floor(log2) <= -127
    const int e = biased - 127 - 8;
    return e < -127 ? -127 : e;
}

// 2^n for -126 <= n <= 127 as an exact float.
__device__ __forceinline__ float exp2i(int n) { return __uint_as_float(static_cast<uint32_t>(n + 127) << 23); }

// E4M3 code of v: round to nearest even, saturate to +-448 (the hardware
// conversion; the low byte of the packed pair holds the second operand).
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return static_cast<uint8_t>(r & 0xFFu);
}

// Maximum over the warp of a non-negative float (its bit pattern orders like
// an unsigned integer), in one warp reduction.
__device__ __forceinline__ float warp_max32(float v) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// Quantise one value per lane of a full warp (the 32 lanes form one MX
// block).  Returns this lane's code; *scale_code gets the block's E8M0 code.
__device__ __forceinline__ uint8_t warp_mx8_quant(float v, uint8_t* scale_code) {
    const float amax = warp_max32(fabsf(v));
    const int e = mx8_exponent(amax);
    *scale_code = static_cast<uint8_t>(e + 127);
    return f32_to_e4m3(v * exp2i(-e));
}

// Scale planes: the scale of element (row, col) lives in byte (col%128)/32 of
// the uint32 word [col/128][row] of a [K/128][pitch] word array.
__device__ __forceinline__ int64_t sf_byte_offset(int64_t row, int64_t col, int64_t pitch) {
    return ((col >> 7) * pitch + row) * 4 + ((col & 127) >> 5);
}

// Item-atom scale planes (a GEMM's token-operand scales): per 128-wide K tile
// a plane of `pitch` 16-byte slots.  The tokens of a GEMM work item that
// starts at row b0 are placed so that the bytes from slot b0 on are the image
// of the 32x128b tensor-memory copy: token l of the item (row b0 + l), K-block
// (col % 128) / 32, lives in slot b0 + 32 * (l / 128) + l % 32, at byte
// 4 * ((l / 32) % 4) + K-block of that slot.  An item of n <= 240 tokens uses
// only slots of its own rows; planes carry 32 spare slots so that the copy of
// a short item's atom stays inside the plane.
__host__ __device__ __forceinline__ int64_t sf_atom_offset(int64_t b0, int l, int64_t col, int64_t pitch) {
    return ((col >> 7) * pitch + b0 + 32 * (l >> 7) + (l & 31)) * 16 + ((l >> 5) & 3) * 4 + ((col & 127) >> 5);
}

}  // namespace moe
