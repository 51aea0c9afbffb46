// combine.cu -- top-k reduction back to token-major bf16 (page "DeepEP ->
// Mega MoE", combine_utils.cuh snippet: fp32 accumulation of bf16 rows,
// __float22bfloat162_rn at the end; page "Dispatch/Combine in the DeepGEMM
// Mega MoE kernel", section 5.1, phase B).
//
// y[t] = bf16( sum over ascending j of the valid entries' L2 rows ), summed
// in fp32 starting from 0, one rounding at the end; tokens without a valid
// entry get +0.  The top-k weight was applied once, in the L1 epilogue.
// One warp handles a 1024-element segment of one token; a lane owns 8
// consecutive elements (one 16-byte load per source row), and up to 8 source
// rows are loaded before they are added, so the loads overlap.
#include <cuda_runtime.h>

#include "formats.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kSeg = 1024;
constexpr int kThreads = 256;

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
    const int s_begin = seg * kSeg, s_end = min(s_begin + kSeg, H);
    for (int s0 = s_begin; s0 < s_end; s0 += 256) {
        const int col = s0 + lane * 8;
        const bool active = col < s_end;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += 8) {
            int r[8];
            uint4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) r[jj] = __shfl_sync(0xffffffffu, my_slot, (j0 + jj) & 31);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                v[jj] = make_uint4(0, 0, 0, 0);
                if (j0 + jj < k && r[jj] >= 0 && active)
                    v[jj] = __ldg(reinterpret_cast<const uint4*>(rows + static_cast<size_t>(r[jj]) * H + col));
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (j0 + jj < k && r[jj] >= 0) {
                    acc[0] += bf16_lo(v[jj].x);
                    acc[1] += bf16_hi(v[jj].x);
                    acc[2] += bf16_lo(v[jj].y);
                    acc[3] += bf16_hi(v[jj].y);
                    acc[4] += bf16_lo(v[jj].z);
                    acc[5] += bf16_hi(v[jj].z);
                    acc[6] += bf16_lo(v[jj].w);
                    acc[7] += bf16_hi(v[jj].w);
                }
            }
        }
        if (active) {
            uint4 o;
            o.x = bf16x2_rn(acc[0], acc[1]);
            o.y = bf16x2_rn(acc[2], acc[3]);
            o.z = bf16x2_rn(acc[4], acc[5]);
            o.w = bf16x2_rn(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * H + col) = o;
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
