// combine.cu -- top-k reduction back to token-major bf16 (page "DeepEP ->
// Mega MoE", combine_utils.cuh snippet: fp32 accumulation of bf16 rows,
// __float22bfloat162_rn at the end; page "Dispatch/Combine in the DeepGEMM
// Mega MoE kernel", section 5.1, phase B).
//
// y[t] = bf16( sum over ascending j of the valid entries' L2 rows ), summed
// in fp32 starting from 0, one rounding at the end; tokens without a valid
// entry get +0.  The top-k weight was applied once, in the L1 epilogue.
// One warp handles a 1024-element segment of one token; a lane owns four
// 8-element chunks of it (one 16-byte load per chunk and source row).  The
// warp reads only the rows of the token's valid entries (a bit mask of them,
// taken in ascending j), two rows per round with all their chunks loaded
// before they are added, so a warp keeps 8 loads in flight whether the token
// has one valid entry (an expert-parallel shard) or all k.
#include <cuda_runtime.h>

#include "formats.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSeg = 1024;
constexpr int kChunks = kSeg / 256;
constexpr int kThreads = 256;

__device__ __forceinline__ void add8(float (&acc)[8], uint4 v) {
    acc[0] += bf16_lo(v.x);
    acc[1] += bf16_hi(v.x);
    acc[2] += bf16_lo(v.y);
    acc[3] += bf16_hi(v.y);
    acc[4] += bf16_lo(v.z);
    acc[5] += bf16_hi(v.z);
    acc[6] += bf16_lo(v.w);
    acc[7] += bf16_hi(v.w);
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const uint16_t* __restrict__ rows,
                                                            const int* __restrict__ slot_of, int T, int H, int k,
                                                            uint16_t* __restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int nseg = (H + kSeg - 1) / kSeg;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int t = static_cast<int>(item / nseg);
    if (t >= T) return;
    const int seg = static_cast<int>(item % nseg);
    const int my_slot = lane < k ? __ldg(slot_of + static_cast<size_t>(t) * k + lane) : -1;
    // the token's valid entries, bit j for entry j: only those rows are read,
    // in ascending j (the order of the sum)
    const uint32_t valid = __ballot_sync(0xffffffffu, my_slot >= 0);
    const int s_begin = seg * kSeg, s_end = min(s_begin + kSeg, H);
    // chunk c of the segment: elements s_begin + 256c + 8*lane .. +7
    bool active[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) active[c] = s_begin + c * 256 + lane * 8 < s_end;
    const size_t base = static_cast<size_t>(s_begin) + lane * 8;
    float acc[kChunks][8];
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[c][i] = 0.0f;
    // two valid entries per round, all chunks of both rows loaded before they
    // are added (8 loads in flight), the earlier entry added first
    uint32_t m = valid;
    while (m) {
        const int j0 = __ffs(m) - 1;
        m &= m - 1;
        const int j1 = __ffs(m) - 1;  // -1: no second entry this round
        if (m) m &= m - 1;
        const bool two = j1 >= 0;
        const uint16_t* r0 = rows + static_cast<size_t>(__shfl_sync(0xffffffffu, my_slot, j0)) * H + base;
        const uint16_t* r1 = rows + static_cast<size_t>(max(__shfl_sync(0xffffffffu, my_slot, j1 & 31), 0)) * H + base;
        uint4 v0[kChunks], v1[kChunks];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            v0[c] = make_uint4(0, 0, 0, 0);
            v1[c] = make_uint4(0, 0, 0, 0);
            if (active[c]) v0[c] = __ldg(reinterpret_cast<const uint4*>(r0 + c * 256));
            if (active[c] && two) v1[c] = __ldg(reinterpret_cast<const uint4*>(r1 + c * 256));
        }
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
            add8(acc[c], v0[c]);
            if (two) add8(acc[c], v1[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        if (active[c]) {
            uint4 o;
            o.x = bf16x2_rn(acc[c][0], acc[c][1]);
            o.y = bf16x2_rn(acc[c][2], acc[c][3]);
            o.z = bf16x2_rn(acc[c][4], acc[c][5]);
            o.w = bf16x2_rn(acc[c][6], acc[c][7]);
            *reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * H + base + c * 256) = o;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const Layout& L, const uint8_t* ws, void* y, cudaStream_t s) {
    if (L.T == 0) return cudaSuccess;
    const int nseg = (L.H + kSeg - 1) / kSeg;
    const int64_t items = static_cast<int64_t>(L.T) * nseg;
    const int64_t blocks = (items + kThreads / 32 - 1) / (kThreads / 32);
    combine_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        reinterpret_cast<const uint16_t*>(ws + L.l2_out), reinterpret_cast<const int*>(ws + L.slot_of), L.T, L.H,
        L.k, static_cast<uint16_t*>(y));
    return cudaGetLastError();
}

}  // namespace moe
