// dispatch.cu -- gather of token-major bf16 activations into the expert-major
// pool with MXFP8 quantisation (page "Dispatch/Combine in the DeepGEMM Mega
// MoE kernel", section 3.1: the token pull into l1_token_buffer; Appendix A.1
// for the FP8 token buffer with its scale buffer; recipe (1,1,32) of the
// "Normal vs Low-Latency" page, section 2).
//
// The pages quantise upstream and move FP8 rows with 1-D TMA copies.  Here
// the quantisation is fused into the gather: each token row is read once,
// quantised once (E4M3 codes, one UE8M0 byte per 32 elements), and written to
// each of its k pool rows (or, when layer 1 gathers its rows by token, once
// to a token-major copy, the pool rows getting only their scales).  One warp
// handles a 1024-element segment of one token; a lane owns 16 consecutive elements (two 16-byte loads, one 16-byte
// store per pool row), two lanes one 32-block.
// Scales are written directly in the tensor-core layout the GEMM consumes:
// chunk (row/128, col/128) of 512 bytes, byte 16*(row%32) + 4*((row%128)/32)
// + (col/32)%4.
#include <cuda_runtime.h>

#include "formats.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSeg = 1024;  // elements per warp work item
constexpr int kHalves = kSeg / 512;
constexpr int kThreads = 256;

// x_q != nullptr: the token's codes go once to x_q[t] (token-major) and the
// pool rows get only their scales; otherwise every pool row gets the codes.
__global__ void __launch_bounds__(kThreads) dispatch_quant_kernel(const uint16_t* __restrict__ x, int T, int H, int k,
                                                                   const int* __restrict__ slot_of,
                                                                   uint8_t* __restrict__ pool_q,
                                                                   uint8_t* __restrict__ pool_sf, int scale_rule,
                                                                   uint8_t* __restrict__ x_q, int64_t p_cap,
                                                                   int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int nseg = (H + kSeg - 1) / kSeg;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int t = static_cast<int>(item / nseg);
    if (t >= T) return;
    const int seg = static_cast<int>(item % nseg);
    const int my_slot = lane < k ? __ldg(slot_of + static_cast<size_t>(t) * k + lane) : -1;
    const int s_begin = seg * kSeg, s_end = min(s_begin + kSeg, H);
    const int sf_cols = H / 128;
    // both 512-element halves of the segment are loaded before either is
    // quantised (four 16-byte loads in flight per lane)
    uint4 raw[kHalves][2];
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
        raw[h][0] = make_uint4(0, 0, 0, 0);
        raw[h][1] = make_uint4(0, 0, 0, 0);
        const int col = s_begin + h * 512 + lane * 16;
        if (col < s_end) {
            const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H + col);
            raw[h][0] = __ldg(src);
            raw[h][1] = __ldg(src + 1);
        }
    }
#pragma unroll
    for (int h = 0; h < kHalves; ++h) {
        const int col = s_begin + h * 512 + lane * 16;
        const bool active = col < s_end;  // H is a multiple of 128: a lane's 16 columns are all in or all out
        const uint4 raw0 = raw[h][0], raw1 = raw[h][1];
        float f[16] = {bf16_lo(raw0.x), bf16_hi(raw0.x), bf16_lo(raw0.y), bf16_hi(raw0.y),
                       bf16_lo(raw0.z), bf16_hi(raw0.z), bf16_lo(raw0.w), bf16_hi(raw0.w),
                       bf16_lo(raw1.x), bf16_hi(raw1.x), bf16_lo(raw1.y), bf16_hi(raw1.y),
                       bf16_lo(raw1.z), bf16_hi(raw1.z), bf16_lo(raw1.w), bf16_hi(raw1.w)};
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const uint32_t sbyte = ue8m0_scale_e4m3_rule(amax, scale_rule);
        const float inv = inv_scale_from_byte(sbyte);
        uint4 codes;
        codes.x = e4m3x2(f[0] * inv, f[1] * inv) | (e4m3x2(f[2] * inv, f[3] * inv) << 16);
        codes.y = e4m3x2(f[4] * inv, f[5] * inv) | (e4m3x2(f[6] * inv, f[7] * inv) << 16);
        codes.z = e4m3x2(f[8] * inv, f[9] * inv) | (e4m3x2(f[10] * inv, f[11] * inv) << 16);
        codes.w = e4m3x2(f[12] * inv, f[13] * inv) | (e4m3x2(f[14] * inv, f[15] * inv) << 16);
        // scale word of the 128-column group owned by lanes 8g..8g+7 (two lanes per 32-block)
        const int g = lane & 24;
        const uint32_t sw = __shfl_sync(0xffffffffu, sbyte, g) | (__shfl_sync(0xffffffffu, sbyte, g + 2) << 8) |
                            (__shfl_sync(0xffffffffu, sbyte, g + 4) << 16) |
                            (__shfl_sync(0xffffffffu, sbyte, g + 6) << 24);
        if (x_q && active) *reinterpret_cast<uint4*>(x_q + static_cast<size_t>(t) * H + col) = codes;
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_slot, j);
            if (r < 0) continue;
            if (!moe_dcheck(r, 0, p_cap, err, kWhereDispatch)) continue;
            if (active) {
                if (!x_q) *reinterpret_cast<uint4*>(pool_q + static_cast<size_t>(r) * H + col) = codes;
                if ((lane & 7) == 0) {
                    const size_t chunk = static_cast<size_t>(r / kBlockM) * sf_cols + col / 128;
                    const int m = r % kBlockM;
                    *reinterpret_cast<uint32_t*>(pool_sf + chunk * kSfChunkBytes + 16 * (m % 32) + 4 * (m / 32)) =
                        sw;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch(const Layout& L, uint8_t* ws, const void* x, int scale_rule, bool gather,
                            cudaStream_t s) {
    if (L.T == 0) return cudaSuccess;
    const int nseg = (L.H + kSeg - 1) / kSeg;
    const int64_t items = static_cast<int64_t>(L.T) * nseg;
    const int64_t blocks = (items + kThreads / 32 - 1) / (kThreads / 32);
    dispatch_quant_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        static_cast<const uint16_t*>(x), L.T, L.H, L.k, reinterpret_cast<const int*>(ws + L.slot_of),
        ws + L.pool_q, ws + L.pool_sf, scale_rule, gather ? ws + L.x_q : nullptr, L.p_cap,
        reinterpret_cast<int*>(ws + L.err));
    return cudaGetLastError();
}

}  // namespace moe
