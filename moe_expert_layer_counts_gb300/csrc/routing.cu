// routing.cu -- dispatch plan: per-expert counts, prefix sums and a stable
// slot per top-k entry (page "DeepEP -> Mega MoE", dispatch.cuh snippet:
// expert counting with block-scope atomics, do_psum prefix sum, slot
// assignment; page "Dispatch/Combine in the DeepGEMM Mega MoE kernel",
// section 3.1 and Appendix A.2 for the expert-major pool padded to the row
// block).
//
// The pages assign slots with a global atomicAdd, so the order of tokens
// inside an expert is not reproducible.  Here the slot of entry i = t*k+j is
// its expert's padded offset plus the number of entries of the same expert
// with a smaller flat index -- a stable counting sort -- computed with three
// kernels and no atomics on the result:
//   route_count  one CTA per chunk of kRouteChunk entries: shared-memory
//                histogram, warp-aggregated (one atomic per distinct expert
//                per warp, via __match_any_sync)
//   route_scan   one CTA: per-expert prefix over chunks, exclusive scans of
//                counts and of counts padded to MOE_BLOCK_M, the row-block ->
//                expert table, the number of row blocks, and the inverse maps
//                of the padding rows (one warp per expert)
//   route_slot   one CTA per chunk: ranks inside the chunk in flat order
//                (rank in warp from the match mask, plus same-expert counts of
//                lower warps), inverse maps of every routed pool row
// A batch of at most kRouteChunk entries (decode-sized) takes one kernel
// instead, route_small: the same three steps in one CTA, so the plan is a
// single launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "internal.h"

namespace moe {
namespace {

constexpr int kCountThreads = 1024;
constexpr int kScanThreads = 1024;
// route_small runs as many warps (up to 32) as keep its shared memory, E x
// (3 + warps) ints, within 47 KB (under the 48 KB default): 32 warps up to E = 343, 8 at
// E = 1024.
constexpr int kSmallMaxThreads = 1024;
constexpr int kSmallMinThreads = 256;
constexpr int kSmallSmemInts = 47 * 1024 / 4;  // leaves room for the static shared arrays
constexpr int kSmallPerThread = (kMaxExperts + kSmallMinThreads - 1) / kSmallMinThreads;  // experts per thread
__host__ __device__ constexpr int small_threads(int E) {
    return E * (3 + kSmallMaxThreads / 32) <= kSmallSmemInts
               ? kSmallMaxThreads
               : (kSmallSmemInts / E - 3) * 32 < kSmallMinThreads ? kSmallMinThreads : (kSmallSmemInts / E - 3) * 32;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int ld_acquire_gpu_int(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Expert id of entry i, or -1 for skipped / out-of-range entries.
__device__ __forceinline__ int entry_expert(const int64_t* idx, int64_t i, int64_t end, int E, bool* bad) {
    if (i >= end) return -1;
    const int64_t v = __ldg(idx + i);
    if (v < -1 || v >= E) {
        *bad = true;
        return -1;
    }
    return static_cast<int>(v);
}

// Histogram of chunk `chunk` (kRouteChunk entries) into hist[chunk][E].
__device__ __forceinline__ void count_chunk(const int64_t* __restrict__ topk_idx, int64_t n_entries, int E, int chunk,
                                            int* __restrict__ hist, int* __restrict__ err, int* s_hist) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t base = static_cast<int64_t>(chunk) * kRouteChunk;
    const int64_t end = min(base + kRouteChunk, n_entries);
    bool bad = false;
    for (int64_t i0 = base; i0 < end; i0 += blockDim.x) {
        const int e = entry_expert(topk_idx, i0 + threadIdx.x, end, E, &bad);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(same) - 1) atomicAdd(&s_hist[e], __popc(same));
    }
    if (bad) atomicOr(err, kDevErrBadExpert);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<size_t>(chunk) * E + e] = s_hist[e];
}

__global__ void __launch_bounds__(kCountThreads) route_count_kernel(const int64_t* __restrict__ topk_idx,
                                                                     int64_t n_entries, int E,
                                                                     int* __restrict__ hist, int* __restrict__ err) {
    extern __shared__ int s_hist[];
    count_chunk(topk_idx, n_entries, E, blockIdx.x, hist, err, s_hist);
}

// Block-wide inclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_inclusive_scan(int v, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += o;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? s_warp[warp - 1] : 0);
    __syncthreads();
    return r;
}

// The prefix sums over chunks and experts (one thread per expert; blockDim.x ==
// kScanThreads): counts, exclusive scans of counts and of padded counts, each
// chunk's base per expert, the row-block tables, the largest count and the
// padding rows' inverse maps.
__device__ __forceinline__ void scan_body(const int* __restrict__ hist, int chunks, int E,
                                                                   int* __restrict__ count, int* __restrict__ off,
                                                                   int* __restrict__ poff,
                                                                   int* __restrict__ chunk_base,
                                                                   int* __restrict__ block_expert,
                                                                   int* __restrict__ block_rows,
                                                                   int* __restrict__ n_blocks,
                                                                   int* __restrict__ max_count,
                                                                   int* __restrict__ row_token,
                                                                   int* __restrict__ row_topk,
                                                                   float* __restrict__ row_weight) {
    __shared__ int s_warp[32];
    __shared__ int s_max;
    __shared__ int s_pad[2][kScanThreads];  // padding rows [begin, end) of each expert
    __shared__ int s_cnt[kScanThreads];     // count of each expert
    const int e = threadIdx.x;
    int c_e = 0;
    if (e == 0) s_max = 0;
    __syncthreads();
    if (e < E) {
#pragma unroll 8
        for (int c = 0; c < chunks; ++c) {
            const int v = hist[static_cast<size_t>(c) * E + e];
            chunk_base[static_cast<size_t>(c) * E + e] = c_e;
            c_e += v;
        }
        count[e] = c_e;
        if (max_count && c_e > 0) atomicMax(&s_max, c_e);
    }
    const int padded = (c_e + kBlockM - 1) / kBlockM * kBlockM;
    const int inc_c = block_inclusive_scan(c_e, s_warp);
    const int inc_p = block_inclusive_scan(padded, s_warp);
    if (e < E) {
        off[e] = inc_c - c_e;
        poff[e] = inc_p - padded;
        if (e == E - 1) {
            off[E] = inc_c;
            poff[E] = inc_p;
            *n_blocks = inc_p / kBlockM;
        }
        // s_max is final: the scans above passed block-wide barriers
        if (e == 0 && max_count) *max_count = s_max;
        s_pad[0][e] = inc_p - padded + c_e;
        s_pad[1][e] = inc_p;
        s_cnt[e] = c_e;
    }
    __syncthreads();
    // the row-block tables and the padding rows' inverse maps: one warp per expert
    const int lane = threadIdx.x & 31;
    for (int x = threadIdx.x >> 5; x < E; x += kScanThreads / 32) {
        const int c_x = s_cnt[x], end = s_pad[1][x];
        const int nb = (c_x + kBlockM - 1) / kBlockM;
        const int b0 = end / kBlockM - nb;
        for (int b = lane; b < nb; b += 32) {
            block_expert[b0 + b] = x;
            if (block_rows) block_rows[b0 + b] = min(kBlockM, c_x - b * kBlockM);
        }
        if (row_token) {
            for (int r = s_pad[0][x] + lane; r < end; r += 32) {
                row_token[r] = -1;
                row_topk[r] = -1;
                row_weight[r] = 0.0f;
            }
        }
    }
}

__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(const int* __restrict__ hist, int chunks, int E,
                                                                   int* __restrict__ count, int* __restrict__ off,
                                                                   int* __restrict__ poff,
                                                                   int* __restrict__ chunk_base,
                                                                   int* __restrict__ block_expert,
                                                                   int* __restrict__ block_rows,
                                                                   int* __restrict__ n_blocks,
                                                                   int* __restrict__ max_count,
                                                                   int* __restrict__ row_token,
                                                                   int* __restrict__ row_topk,
                                                                   float* __restrict__ row_weight) {
    scan_body(hist, chunks, E, count, off, poff, chunk_base, block_expert, block_rows, n_blocks, max_count, row_token,
              row_topk, row_weight);
}

// Stable slots of chunk `chunk`: ranks inside the chunk in flat order (rank in
// warp from the match mask, plus same-expert counts of lower warps) on top of
// the expert's padded offset and the chunk's base; inverse maps of every
// routed pool row.  s_mem: E * (1 + warps) ints.
__device__ __forceinline__ void slot_chunk(const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                                           int64_t n_entries, int k, int E, int chunk, const int* __restrict__ poff,
                                           const int* __restrict__ chunk_base, int* __restrict__ slot_of,
                                           int* __restrict__ row_token, int* __restrict__ row_topk,
                                           float* __restrict__ row_weight, int* s_mem) {
    const int nwarps = blockDim.x / 32;
    int* s_next = s_mem;        // [E] next free slot of each expert for this chunk
    int* s_wcnt = s_mem + E;    // [nwarps][E] same-expert counts per warp, this round
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        s_next[e] = poff[e] + chunk_base[static_cast<size_t>(chunk) * E + e];
        for (int w = 0; w < nwarps; ++w) s_wcnt[w * E + e] = 0;
    }
    __syncthreads();
    const int64_t base = static_cast<int64_t>(chunk) * kRouteChunk;
    const int64_t end = min(base + kRouteChunk, n_entries);
    bool bad = false;
    for (int64_t i0 = base; i0 < end; i0 += blockDim.x) {
        const int64_t i = i0 + threadIdx.x;
        const int e = entry_expert(topk_idx, i, end, E, &bad);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const bool leader = lane == __ffs(same) - 1;
        if (e >= 0 && leader) s_wcnt[warp * E + e] = __popc(same);
        __syncthreads();
        int slot = -1;
        if (e >= 0) {
            int before = __popc(same & lanemask_lt());
            for (int w = 0; w < warp; ++w) before += s_wcnt[w * E + e];
            slot = s_next[e] + before;
        }
        __syncthreads();
        if (e >= 0 && leader) {
            atomicAdd(&s_next[e], __popc(same));
            s_wcnt[warp * E + e] = 0;
        }
        __syncthreads();
        if (i < end) {
            slot_of[i] = slot;
            if (slot >= 0) {
                row_token[slot] = static_cast<int>(i / k);
                row_topk[slot] = static_cast<int>(i % k);
                row_weight[slot] = __ldg(topk_w + i);
            }
        }
    }
}

__global__ void __launch_bounds__(kSmallMaxThreads) route_slot_kernel(
    const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t n_entries, int k, int E,
    const int* __restrict__ poff, const int* __restrict__ chunk_base,
    int* __restrict__ slot_of, int* __restrict__ row_token, int* __restrict__ row_topk,
    float* __restrict__ row_weight) {
    extern __shared__ int s_mem[];
    slot_chunk(topk_idx, topk_w, n_entries, k, E, blockIdx.x, poff, chunk_base, slot_of, row_token, row_topk,
               row_weight, s_mem);
}

// The whole plan in ONE multi-CTA launch for batches of more than one chunk
// and at most kFusedMaxExperts experts.  Three phases over the chunks, each
// chunk taken from a work counter (sync[0], sync[1]):
//   1. histograms of chunks; the CTA that counts the last chunk done (sync[2])
//   2. runs the scans (as route_scan) and releases a flag (sync[3]);
//   3. every CTA then takes chunks for the stable slots (as route_slot).
// A CTA waits for the flag only once no chunk of phase 1 is left to take, so
// every chunk of phase 1 is held by a running CTA: no co-residency is needed.
// The wait is bounded (1 s of global time; the error record gets
// MOE_ERR_TIMEOUT).  sync[0..3] must be zero at launch.
constexpr int kFusedMaxExperts = 256;
constexpr uint64_t kRouteWaitNs = 1000000000ull;

__global__ void __launch_bounds__(kScanThreads) route_fused_kernel(
    const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t n_entries, int k, int E,
    int chunks, int* __restrict__ sync, int* __restrict__ hist, int* __restrict__ count, int* __restrict__ off,
    int* __restrict__ poff, int* __restrict__ chunk_base, int* __restrict__ block_expert,
    int* __restrict__ block_rows, int* __restrict__ n_blocks, int* __restrict__ max_count,
    int* __restrict__ slot_of, int* __restrict__ row_token, int* __restrict__ row_topk,
    float* __restrict__ row_weight, int* __restrict__ err) {
    extern __shared__ int s_mem[];
    __shared__ int s_chunk, s_last;
    // 1. counts
    while (true) {
        if (threadIdx.x == 0) s_chunk = atomicAdd(&sync[0], 1);
        __syncthreads();
        const int c = s_chunk;
        __syncthreads();
        if (c >= chunks) break;
        count_chunk(topk_idx, n_entries, E, c, hist, err, s_mem);
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();  // this chunk's histogram before the count of finished chunks
            s_last = atomicAdd(&sync[2], 1) == chunks - 1;
        }
        __syncthreads();
        if (s_last) {
            // 2. the last chunk is in: every histogram is visible
            __threadfence();
            scan_body(hist, chunks, E, count, off, poff, chunk_base, block_expert, block_rows, n_blocks, max_count,
                      row_token, row_topk, row_weight);
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                atomicExch(&sync[3], 1);
            }
        }
    }
    // 3. stable slots, once the scans are released
    if (threadIdx.x == 0) {
        const uint64_t deadline = globaltimer_ns() + kRouteWaitNs;
        bool ok = true;
        while (ld_acquire_gpu_int(&sync[3]) == 0) {
            if (globaltimer_ns() > deadline) {
                ok = false;
                break;
            }
            __nanosleep(256);
        }
        if (!ok) {
            atomicOr(err, kDevErrTimeout);
            atomicCAS(err + 1, 0, 1 + 99);
        }
        s_last = ok;
    }
    __syncthreads();
    if (!s_last) return;
    while (true) {
        if (threadIdx.x == 0) s_chunk = atomicAdd(&sync[1], 1);
        __syncthreads();
        const int c = s_chunk;
        __syncthreads();
        if (c >= chunks) break;
        slot_chunk(topk_idx, topk_w, n_entries, k, E, c, poff, chunk_base, slot_of, row_token, row_topk, row_weight,
                   s_mem);
        __syncthreads();
    }
}

// All of routing for n <= kRouteChunk entries in one CTA: counts (shared
// histogram), exclusive scans of the counts and of the counts padded to
// MOE_BLOCK_M (thread t owns experts [t*per, t*per + per)), the row-block
// tables, the padding rows, then the stable slots exactly as route_slot ranks
// them (chunk base 0).  Also zeroes the error record and sets the bad-id bit.
__global__ void __launch_bounds__(kSmallMaxThreads) route_small_kernel(
    const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int n, int k, int E,
    int* __restrict__ count, int* __restrict__ off, int* __restrict__ poff, int* __restrict__ block_expert,
    int* __restrict__ block_rows, int* __restrict__ n_blocks, int* __restrict__ max_count, int* __restrict__ slot_of,
    int* __restrict__ row_token, int* __restrict__ row_topk, float* __restrict__ row_weight, int* __restrict__ err) {
    extern __shared__ int s_mem[];
    const int nthreads = blockDim.x, nwarps = nthreads / 32;
    int* s_cnt = s_mem;                      // [E] counts, later the next free slot of each expert
    int* s_wcnt = s_mem + E;                 // [nwarps][E] same-expert counts per warp, this round
    int* s_pad = s_mem + E * (1 + nwarps);   // [2][E] padding rows [begin, end) of each expert
    __shared__ int s_warp[32];
    __shared__ int s_max, s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += nthreads) {
        s_cnt[e] = 0;
        for (int w = 0; w < nwarps; ++w) s_wcnt[w * E + e] = 0;
    }
    if (tid == 0) {
        s_max = 0;
        s_bad = 0;
    }
    __syncthreads();
    // 1. counts
    bool bad = false;
    for (int i0 = 0; i0 < n; i0 += nthreads) {
        const int e = entry_expert(topk_idx, i0 + tid, n, E, &bad);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(same) - 1) atomicAdd(&s_cnt[e], __popc(same));
    }
    if (bad) s_bad = 1;
    __syncthreads();
    // 2. scans over experts, per-thread runs of kSmallPerThread
    const int per = (E + nthreads - 1) / nthreads;
    int c[kSmallPerThread];
    int sum_c = 0, sum_p = 0, mx = 0;
#pragma unroll
    for (int q = 0; q < kSmallPerThread; ++q) {
        const int e = tid * per + q;
        c[q] = (q < per && e < E) ? s_cnt[e] : 0;
        sum_c += c[q];
        sum_p += (c[q] + kBlockM - 1) / kBlockM * kBlockM;
        mx = max(mx, c[q]);
    }
    if (mx > 0) atomicMax(&s_max, mx);
    const int inc_c = block_inclusive_scan(sum_c, s_warp);
    const int inc_p = block_inclusive_scan(sum_p, s_warp);
    int o_c = inc_c - sum_c, o_p = inc_p - sum_p;
#pragma unroll
    for (int q = 0; q < kSmallPerThread; ++q) {
        const int e = tid * per + q;
        if (q < per && e < E) {
            const int padded = (c[q] + kBlockM - 1) / kBlockM * kBlockM;
            count[e] = c[q];
            off[e] = o_c;
            poff[e] = o_p;
            for (int b = 0; b < padded / kBlockM; ++b) {
                block_expert[o_p / kBlockM + b] = e;
                block_rows[o_p / kBlockM + b] = min(kBlockM, c[q] - b * kBlockM);
            }
            s_pad[e] = o_p + c[q];
            s_pad[E + e] = o_p + padded;
            s_cnt[e] = o_p;  // next free slot (the chunk base is 0)
            o_c += c[q];
            o_p += padded;
            if (e == E - 1) {
                off[E] = o_c;
                poff[E] = o_p;
                *n_blocks = o_p / kBlockM;
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        *max_count = s_max;
        err[0] = s_bad ? kDevErrBadExpert : 0;
        err[1] = 0;
    }
    // padding rows: one warp per expert
    for (int x = warp; x < E; x += nwarps) {
        for (int r = s_pad[x] + lane; r < s_pad[E + x]; r += 32) {
            row_token[r] = -1;
            row_topk[r] = -1;
            row_weight[r] = 0.0f;
        }
    }
    // 3. stable slots, in rounds of blockDim entries in flat order
    for (int i0 = 0; i0 < n; i0 += nthreads) {
        const int i = i0 + tid;
        bool unused = false;
        const int e = entry_expert(topk_idx, i, n, E, &unused);
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const bool leader = lane == __ffs(same) - 1;
        if (e >= 0 && leader) s_wcnt[warp * E + e] = __popc(same);
        __syncthreads();
        int slot = -1;
        if (e >= 0) {
            int before = __popc(same & lanemask_lt());
            for (int w = 0; w < warp; ++w) before += s_wcnt[w * E + e];
            slot = s_cnt[e] + before;
        }
        __syncthreads();
        if (e >= 0 && leader) {
            atomicAdd(&s_cnt[e], __popc(same));
            s_wcnt[warp * E + e] = 0;
        }
        __syncthreads();
        if (i < n) {
            slot_of[i] = slot;
            if (slot >= 0) {
                row_token[slot] = i / k;
                row_topk[slot] = i % k;
                row_weight[slot] = __ldg(topk_w + i);
            }
        }
    }
}

}  // namespace

cudaError_t launch_route(const Layout& L, uint8_t* ws, const int64_t* topk_idx, const float* topk_w,
                         cudaStream_t s) {
    const int64_t n = static_cast<int64_t>(L.T) * L.k;
    int* err = reinterpret_cast<int*>(ws + L.err);
    int* hist = reinterpret_cast<int*>(ws + L.hist);
    int* count = reinterpret_cast<int*>(ws + L.count);
    int* off = reinterpret_cast<int*>(ws + L.off);
    int* poff = reinterpret_cast<int*>(ws + L.poff);
    int* chunk_base = reinterpret_cast<int*>(ws + L.chunk_base);
    if (L.chunks == 1) {  // one kernel for a decode-sized batch
        const int threads = small_threads(L.E);
        const size_t smem = static_cast<size_t>(L.E) * (3 + threads / 32) * sizeof(int);
        route_small_kernel<<<1, threads, smem, s>>>(
            topk_idx, topk_w, static_cast<int>(n), L.k, L.E, count, off, poff,
            reinterpret_cast<int*>(ws + L.block_expert), reinterpret_cast<int*>(ws + L.block_rows),
            reinterpret_cast<int*>(ws + L.n_blocks), reinterpret_cast<int*>(ws + L.max_count),
            reinterpret_cast<int*>(ws + L.slot_of), reinterpret_cast<int*>(ws + L.row_token),
            reinterpret_cast<int*>(ws + L.row_topk), reinterpret_cast<float*>(ws + L.row_weight), err);
        return cudaGetLastError();
    }
    // the error record and the fused plan's four scheduling words start at zero
    cudaError_t st = cudaMemsetAsync(err, 0, kErrWords * sizeof(int), s);
    if (st != cudaSuccess) return st;
    if (L.E <= kFusedMaxExperts && L.chunks > 0) {  // the whole plan in one launch
        const size_t smem = static_cast<size_t>(L.E) * (1 + kScanThreads / 32) * sizeof(int);
        route_fused_kernel<<<std::min(L.chunks, 512), kScanThreads, smem, s>>>(
            topk_idx, topk_w, n, L.k, L.E, L.chunks, err + kErrSyncOff, hist, count, off, poff, chunk_base,
            reinterpret_cast<int*>(ws + L.block_expert), reinterpret_cast<int*>(ws + L.block_rows),
            reinterpret_cast<int*>(ws + L.n_blocks), reinterpret_cast<int*>(ws + L.max_count),
            reinterpret_cast<int*>(ws + L.slot_of), reinterpret_cast<int*>(ws + L.row_token),
            reinterpret_cast<int*>(ws + L.row_topk), reinterpret_cast<float*>(ws + L.row_weight), err);
        return cudaGetLastError();
    }
    if (L.chunks > 0) {
        route_count_kernel<<<L.chunks, kCountThreads, L.E * sizeof(int), s>>>(topk_idx, n, L.E, hist, err);
        if ((st = cudaGetLastError()) != cudaSuccess) return st;
    }
    route_scan_kernel<<<1, kScanThreads, 0, s>>>(hist, L.chunks, L.E, count, off, poff, chunk_base,
                                                 reinterpret_cast<int*>(ws + L.block_expert),
                                                 reinterpret_cast<int*>(ws + L.block_rows),
                                                 reinterpret_cast<int*>(ws + L.n_blocks),
                                                 reinterpret_cast<int*>(ws + L.max_count),
                                                 reinterpret_cast<int*>(ws + L.row_token),
                                                 reinterpret_cast<int*>(ws + L.row_topk),
                                                 reinterpret_cast<float*>(ws + L.row_weight));
    if ((st = cudaGetLastError()) != cudaSuccess) return st;
    if (L.chunks > 0) {
        const int threads = small_threads(L.E);  // its shared memory, E x (1 + warps) ints, fits as well
        const size_t smem = static_cast<size_t>(L.E) * (1 + threads / 32) * sizeof(int);
        route_slot_kernel<<<L.chunks, threads, smem, s>>>(
            topk_idx, topk_w, n, L.k, L.E, poff, chunk_base, reinterpret_cast<int*>(ws + L.slot_of),
            reinterpret_cast<int*>(ws + L.row_token), reinterpret_cast<int*>(ws + L.row_topk),
            reinterpret_cast<float*>(ws + L.row_weight));
        if ((st = cudaGetLastError()) != cudaSuccess) return st;
    }
    return cudaSuccess;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Expert counts and offsets without a caller workspace.  The scratch of the
// count and scan kernels lives in one fixed device array of this file; its
// device address is looked up once per device (host code may not use the
// array's name as an address).
namespace moe {
namespace {

constexpr int64_t kStaticMaxEntries = 262144;   // T * k
constexpr int kStaticMaxChunkExperts = 32768;   // ceil(T*k / kRouteChunk) * E
constexpr int kStaticBlockCap = 4096;           // row blocks: (262144 + 1024*127) / 128 < 4096
constexpr int kStaticHist = 0;
constexpr int kStaticBase = kStaticMaxChunkExperts;
constexpr int kStaticBlocks = 2 * kStaticMaxChunkExperts;
constexpr int kStaticNBlocks = kStaticBlocks + kStaticBlockCap;
constexpr int kStaticErr = kStaticNBlocks + 32;
constexpr int kStaticInts = kStaticErr + 32;

static __device__ __align__(256) int g_offsets_scratch[kStaticInts];

// Device address of the array on device `dev` (which must be current),
// looked up on the first call for that device and cached.  The cache is one
// atomic pointer per device: two host threads that make the first call at
// the same time both look the address up and store the same value.  A cached
// address belongs to the context it was looked up in; after cudaDeviceReset()
// it is stale, so the entry point must not be called on that device again in
// the same process (stated in moe.h).
std::atomic<int*> g_static_ptrs[64];

int* static_scratch_ptr(int dev) {
    if (dev < 0 || dev >= 64) return nullptr;
    int* p = g_static_ptrs[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_offsets_scratch) != cudaSuccess) return nullptr;
    p = static_cast<int*>(a);
    g_static_ptrs[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace
}  // namespace moe

extern "C" int moe_expert_offsets_static(const int64_t* topk_idx, int T, int k, int E, int32_t* count,
                                         int32_t* offsets, int32_t* padded_offsets, void* stream) {
    using namespace moe;
    if (T < 0 || k < 1 || k > kMaxTopk || E < 1) return MOE_ERR_INVALID_ARG;
    if (!count || !offsets || !padded_offsets || (T > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
    const int64_t n = static_cast<int64_t>(T) * k;
    const int chunks = static_cast<int>((n + kRouteChunk - 1) / kRouteChunk);
    if (E > kMaxExperts || n > kStaticMaxEntries || static_cast<int64_t>(chunks) * E > kStaticMaxChunkExperts)
        return MOE_ERR_TOO_LARGE;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return MOE_ERR_UNSUPPORTED;
    int* scratch = static_scratch_ptr(dev);
    if (!scratch) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Nothing needs clearing: the count kernel writes every histogram cell the
    // scan reads, and the scan writes every base and table cell.  The count
    // kernel's bad-id flag lands in a word that nothing reads (this entry point
    // skips ids outside [-1, E) without reporting them).
    if (chunks > 0) {
        route_count_kernel<<<chunks, kCountThreads, E * sizeof(int), s>>>(topk_idx, n, E, scratch + kStaticHist,
                                                                          scratch + kStaticErr);
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
    route_scan_kernel<<<1, kScanThreads, 0, s>>>(scratch + kStaticHist, chunks, E, count, offsets, padded_offsets,
                                                 scratch + kStaticBase, scratch + kStaticBlocks, nullptr,
                                                 scratch + kStaticNBlocks, nullptr, nullptr, nullptr, nullptr);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
