// formats.cuh -- device helpers for the number formats of the layer:
// bf16 <-> fp32, the UE8M0 shared scale of an MX block, and E4M3 casts.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace moe {

// UE8M0 scale byte of a block for E4M3 codes: the smallest e with
// amax <= 448 * 2^e, clamped to [-126, 127], returned biased (e + 127).
// Read off the bits of amax = f * 2^q (f in [1,2)):  448 = 1.75 * 2^8, so
// e = q - 8 when f <= 1.75 and q - 7 otherwise.  amax == 0 gives 127; a
// subnormal amax is far below 448 * 2^-126 and gives the floor byte 1.
__device__ __forceinline__ uint32_t ue8m0_scale_e4m3(float amax) {
    const uint32_t bits = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (bits == 0) return 127u;
    const int ex = static_cast<int>(bits >> 23);
    if (ex == 0) return 1u;
    int e = (ex - 127) - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = max(-126, min(127, e));
    return static_cast<uint32_t>(e + 127);
}

// The OCP MX v1.0 rule instead: X = 2^(floor(log2 amax) - 8) (8 = the
// exponent of E4M3's largest normal, 448 = 1.75 * 2^8); scaled values beyond
// 448 saturate in the cast.  floor(log2 amax) is the unbiased exponent field
// of a normal amax; a subnormal amax gives the floor byte 1, 0 gives 127.
__device__ __forceinline__ uint32_t ue8m0_scale_e4m3_floor(float amax) {
    const uint32_t bits = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (bits == 0) return 127u;
    const int ex = static_cast<int>(bits >> 23);
    if (ex == 0) return 1u;
    const int e = max(-126, min(127, (ex - 127) - 8));
    return static_cast<uint32_t>(e + 127);
}

// Scale byte by rule (0 = ceil, 1 = OCP floor).
__device__ __forceinline__ uint32_t ue8m0_scale_e4m3_rule(float amax, int rule) {
    return rule ? ue8m0_scale_e4m3_floor(amax) : ue8m0_scale_e4m3(amax);
}

// 2^(127 - byte) for a scale byte in [1, 253] (always a normal float).
__device__ __forceinline__ float inv_scale_from_byte(uint32_t byte) {
    return __uint_as_float((254u - byte) << 23);
}

// Two floats -> two E4M3 codes (round to nearest even, saturate to +-448);
// the first argument lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> packed bf16x2 (round to nearest even), first in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// True when amax lies within `ulps` of the E4M3 scale boundary (mantissa
// 1.75, where ue8m0_scale_e4m3 changes exponent).
__device__ __forceinline__ bool near_e4m3_scale_boundary(float amax, uint32_t ulps) {
    const uint32_t m = __float_as_uint(amax) & 0x7FFFFFu;
    const uint32_t d = m > 0x600000u ? m - 0x600000u : 0x600000u - m;
    return d <= ulps;
}

// True when amax lies within `ulps` of a power of two (where the floor
// rule's scale changes exponent).
__device__ __forceinline__ bool near_pow2(float amax, uint32_t ulps) {
    const uint32_t m = __float_as_uint(amax) & 0x7FFFFFu;
    return m <= ulps || 0x800000u - m <= ulps;
}

}  // namespace moe
