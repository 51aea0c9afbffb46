// combine.cu -- top-k reduction back to token-major bf16 (page "DeepEP ->
// Mega MoE", combine_utils.cuh snippet: fp32 accumulation of bf16 rows,
// __float22bfloat162_rn at the end; page "Dispatch/Combine in the DeepGEMM
// Mega MoE kernel", section 5.1, phase B).
//
// y[t] = bf16( sum over ascending j of the valid entries' L2 rows ), summed
// in fp32 starting from 0, one rounding at the end; tokens without a valid
// entry get +0.  The top-k weight was applied once, in the L1 epilogue.
// One warp handles a segment of one token (1024 elements, or 256 for
// decode-sized batches); a lane owns one 8-element piece of every 256-element
// chunk of it (one 16-byte load per chunk and source row).  The warp reads
// only the rows of the token's valid entries (a bit mask of them, taken in
// ascending j), 8 / chunks rows per round with all their chunks loaded before
// they are added, so a warp keeps 8 loads in flight whether the token has one
// valid entry (an expert-parallel shard) or all k.  The L2 rows are read and y
// is written with streaming cache hints (each byte is touched once): full
// workload 160 -> 153 us, mid 24.6 -> 20.6 us.
#include <cuda_runtime.h>

#include "formats.cuh"
#include "internal.h"

namespace moe {
namespace {

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

// kChunks 256-element chunks per warp (a segment of 256 * kChunks elements of
// one token) and 8 / kChunks valid entries per round, so a warp always has up
// to 8 loads in flight.
template <int kChunks>
__global__ void __launch_bounds__(kThreads) combine_kernel(const uint16_t* __restrict__ rows,
                                                            const int* __restrict__ slot_of, int T, int H, int k,
                                                            uint16_t* __restrict__ y, int64_t p_cap,
                                                            int* __restrict__ err) {
    constexpr int kSeg = 256 * kChunks, kRows = 8 / kChunks;
    const int lane = threadIdx.x & 31;
    const int nseg = (H + kSeg - 1) / kSeg;
    const int64_t item = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
    const int t = static_cast<int>(item / nseg);
    if (t >= T) return;
    const int seg = static_cast<int>(item % nseg);
    int my_slot = lane < k ? __ldg(slot_of + static_cast<size_t>(t) * k + lane) : -1;
    if (my_slot >= 0 && seg == 0 && !moe_dcheck(my_slot, 0, p_cap, err, kWhereCombine)) my_slot = -1;
#ifdef MOE_DEBUG
    if (my_slot >= p_cap) my_slot = -1;  // the other segments skip it too (reported once, above)
#endif
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
    // kRows valid entries per round, every chunk of them loaded before any is
    // added; within a chunk the entries are added in ascending j
    uint32_t m = valid;
    while (m) {
        const uint16_t* r[kRows];
        bool has[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int j = __ffs(m) - 1;  // -1 once m is empty
            has[q] = m != 0;
            r[q] = rows + static_cast<size_t>(max(__shfl_sync(0xffffffffu, my_slot, j & 31), 0)) * H + base;
            if (m) m &= m - 1;
        }
        uint4 v[kRows][kChunks];
#pragma unroll
        for (int q = 0; q < kRows; ++q)
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                v[q][c] = make_uint4(0, 0, 0, 0);
                if (has[q] && active[c]) v[q][c] = __ldcs(reinterpret_cast<const uint4*>(r[q] + c * 256));
            }
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
#pragma unroll
            for (int q = 0; q < kRows; ++q)
                if (has[q]) add8(acc[c], v[q][c]);
    }
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        if (active[c]) {
            uint4 o;
            o.x = bf16x2_rn(acc[c][0], acc[c][1]);
            o.y = bf16x2_rn(acc[c][2], acc[c][3]);
            o.z = bf16x2_rn(acc[c][4], acc[c][5]);
            o.w = bf16x2_rn(acc[c][6], acc[c][7]);
            __stcs(reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * H + base + c * 256), o);
        }
    }
}

template <int kChunks>
cudaError_t launch_combine_chunks(const Layout& L, uint8_t* ws, void* y, cudaStream_t s) {
    constexpr int kSeg = 256 * kChunks;
    const int nseg = (L.H + kSeg - 1) / kSeg;
    const int64_t items = static_cast<int64_t>(L.T) * nseg;
    const int64_t blocks = (items + kThreads / 32 - 1) / (kThreads / 32);
    combine_kernel<kChunks><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        reinterpret_cast<const uint16_t*>(ws + L.l2_out), reinterpret_cast<const int*>(ws + L.slot_of), L.T, L.H,
        L.k, static_cast<uint16_t*>(y), L.p_cap, reinterpret_cast<int*>(ws + L.err));
    return cudaGetLastError();
}

}  // namespace

// Decode-sized batches (at most kSmallBatchWarps warps of 1024-element
// segments, well under one wave) take 256-element segments with up to 8 rows
// a round: four times the warps, each with fewer rounds (decode, 1024 entries:
// 11.9 -> 8.8 us).  Larger batches keep 1024-element segments with 2 rows a
// round, which keeps 8 loads in flight per warp also when a token has only one
// or two valid entries (one expert-parallel shard: 47 us, against 69 us with
// 256-element segments; all 8 entries valid: 160 against 153 us).
constexpr int64_t kSmallBatchWarps = 1024;

cudaError_t launch_combine(const Layout& L, uint8_t* ws, void* y, cudaStream_t s) {
    if (L.T == 0) return cudaSuccess;
    if (static_cast<int64_t>(L.T) * ((L.H + 1023) / 1024) <= kSmallBatchWarps)
        return launch_combine_chunks<1>(L, ws, y, s);
    return launch_combine_chunks<4>(L, ws, y, s);
}

}  // namespace moe
