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
// with a smaller flat index -- a stable counting sort -- with no atomics on
// the result.  Three steps over chunks of kRouteChunk entries:
//   count  shared-memory histogram per chunk, warp-aggregated (one atomic
//          per distinct expert per warp, via __match_any_sync)
//   scan   per-expert prefix over chunks, exclusive scans of counts and of
//          counts padded to MOE_BLOCK_M, the row-block -> expert table, the
//          number of row blocks, and the inverse maps of the padding rows
//   slot   ranks inside each chunk in flat order (rank in warp from the match
//          mask, plus same-expert counts of lower warps), inverse maps of
//          every routed pool row
// Up to kFusedMaxExperts experts the whole plan is ONE multi-CTA launch,
// route_fused (described where it is defined).  Beyond that, a batch of at
// most kRouteChunk entries takes one single-CTA kernel, route_small, and
// larger ones the three kernels route_count (one CTA per chunk), route_scan
// (one CTA) and route_slot (one CTA per chunk).
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

// One round of stable ranks: the slot of this thread's entry (expert e, -1
// for none) is s_next[e] + the same-expert entries of lower lanes of its warp
// (match mask) + those of lower warps (s_wcnt, zero on entry and on exit);
// s_next then advances past the round.  All threads of the CTA take part.
__device__ __forceinline__ int rank_round(int e, int E, int* s_next, int* s_wcnt) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
    return slot;
}

// The slot of entry i and the inverse maps of its pool row.
__device__ __forceinline__ void write_slot(int64_t i, int slot, float w, int k, int* __restrict__ slot_of,
                                           int* __restrict__ row_token, int* __restrict__ row_topk,
                                           float* __restrict__ row_weight) {
    slot_of[i] = slot;
    if (slot >= 0) {
        const int t = static_cast<int>(i) / k;  // plans hold at most 2^28 entries
        row_token[slot] = t;
        row_topk[slot] = static_cast<int>(i) - t * k;
        row_weight[slot] = w;
    }
}

// Stable slots of chunk `chunk`: ranks inside the chunk in flat order on top
// of s_next[e] (the expert's padded offset plus the chunk's base, set by the
// caller, with s_wcnt zeroed); inverse maps of every routed pool row.
// s_wcnt: [warps][E] same-expert counts per warp of the entries being ranked.
__device__ __forceinline__ void slot_rank(const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                                          int64_t n_entries, int k, int E, int chunk, int* s_next, int* s_wcnt,
                                          int* __restrict__ slot_of, int* __restrict__ row_token,
                                          int* __restrict__ row_topk, float* __restrict__ row_weight) {
    const int64_t base = static_cast<int64_t>(chunk) * kRouteChunk;
    const int64_t end = min(base + kRouteChunk, n_entries);
    bool bad = false;
    for (int64_t i0 = base; i0 < end; i0 += blockDim.x) {
        const int64_t i = i0 + threadIdx.x;
        const int e = entry_expert(topk_idx, i, end, E, &bad);
        const int slot = rank_round(e, E, s_next, s_wcnt);
        if (i < end) write_slot(i, slot, __ldg(topk_w + i), k, slot_of, row_token, row_topk, row_weight);
    }
}

// slot_rank of chunk `chunk` with the bases from the scan's tables.
// s_mem: E * (1 + warps) ints.
__device__ __forceinline__ void slot_chunk(const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                                           int64_t n_entries, int k, int E, int chunk, const int* __restrict__ poff,
                                           const int* __restrict__ chunk_base, int* __restrict__ slot_of,
                                           int* __restrict__ row_token, int* __restrict__ row_topk,
                                           float* __restrict__ row_weight, int* s_mem) {
    const int nwarps = blockDim.x / 32;
    int* s_next = s_mem;        // [E] next free slot of each expert for this chunk
    int* s_wcnt = s_mem + E;    // [nwarps][E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        s_next[e] = poff[e] + chunk_base[static_cast<size_t>(chunk) * E + e];
        for (int w = 0; w < nwarps; ++w) s_wcnt[w * E + e] = 0;
    }
    __syncthreads();
    slot_rank(topk_idx, topk_w, n_entries, k, E, chunk, s_next, s_wcnt, slot_of, row_token, row_topk, row_weight);
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

// The whole plan in ONE multi-CTA launch, for at most kFusedMaxExperts
// experts and any number of entries:
//   1. every CTA takes a chunk number from a counter (sync[0]) and counts that
//      chunk, keeping its ids and weights in registers; a counted chunk is
//      added to sync[2] (release).  A CTA then waits until sync[2] reaches the
//      number of chunks (acquire), and while it waits it takes any chunk still
//      untaken from the same counter and counts it from memory (sync[3]
//      counts those) -- a chunk is taken only by a running CTA and a waiting
//      CTA keeps taking chunks, so every chunk is counted whether or not all
//      CTAs are resident;
//   2. EVERY CTA sums the histogram rows itself (the per-expert totals and the
//      base of its own chunk) and scans the totals, so no CTA waits for
//      another's scan; CTA 0 writes the count / offset tables, and the
//      row-block tables and padding rows are shared out one expert per warp
//      over the whole grid;
//   3. every CTA ranks the chunk it holds in registers; chunks counted from
//      memory (marked in chunk_kind) are ranked from memory, taken from a
//      second counter (sync[1]).
// The wait is bounded (1 s of global time; the error record gets
// MOE_ERR_TIMEOUT).  sync[0..3] must be zero at launch.
constexpr int kFusedMaxExperts = 256;
constexpr int kFusedMinCtas = 16;  // CTAs that share the tables and padding rows of a small batch
constexpr uint64_t kRouteWaitNs = 1000000000ull;

// Per-expert sums of the histogram rows of all chunks (s_tot) and of chunks
// [0, upto) (s_base).  min(blockDim.x / E, 32) threads share an expert, each
// summing a stride of the chunks; rows written by other CTAs are read at L2.
// s_part: 2 * blockDim.x ints.
__device__ __forceinline__ void chunk_sums(const int* __restrict__ hist, int chunks, int E, int upto, int* s_part,
                                           int* s_tot, int* s_base) {
    const int parts = min(static_cast<int>(blockDim.x) / E, 32);
    const int e = threadIdx.x % E, part = threadIdx.x / E;
    if (part < parts) {
        int tot = 0, base = 0;
#pragma unroll 8
        for (int c = part; c < chunks; c += parts) {
            const int v = __ldcg(hist + static_cast<size_t>(c) * E + e);
            tot += v;
            base += c < upto ? v : 0;
        }
        s_part[part * E + e] = tot;
        s_part[(parts + part) * E + e] = base;
    }
    __syncthreads();
    if (threadIdx.x < E) {
        int tot = 0, base = 0;
        for (int q = 0; q < parts; ++q) {
            tot += s_part[q * E + threadIdx.x];
            base += s_part[(parts + q) * E + threadIdx.x];
        }
        s_tot[threadIdx.x] = tot;
        s_base[threadIdx.x] = base;
    }
    __syncthreads();
}

// Inclusive scans of two ints per thread at once (blockDim.x == 1024): packed
// into one 64-bit sum, which cannot carry from the low half while the low
// values sum to less than 2^32.
__device__ __forceinline__ void block_inclusive_scan2(int a, int b, int* s_warp2, int& inc_a, int& inc_b) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t v = (static_cast<uint64_t>(static_cast<uint32_t>(b)) << 32) | static_cast<uint32_t>(a);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint64_t o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    uint64_t* s_w = reinterpret_cast<uint64_t*>(s_warp2);
    if (lane == 31) s_w[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = s_w[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint64_t o = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += o;
        }
        s_w[lane] = w;
    }
    __syncthreads();
    const uint64_t r = v + (warp > 0 ? s_w[warp - 1] : 0ull);
    inc_a = static_cast<int>(static_cast<uint32_t>(r));
    inc_b = static_cast<int>(r >> 32);
}

constexpr int kFusedPer = kRouteChunk / kScanThreads;  // entries of a chunk per thread
static_assert(kFusedPer * kScanThreads == kRouteChunk, "a chunk is whole rounds of the plan CTA");

__global__ void __launch_bounds__(kScanThreads) route_fused_kernel(
    const int64_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int64_t n_entries, int k, int E,
    int chunks, int* __restrict__ sync, int* __restrict__ hist, int* __restrict__ chunk_kind,
    int* __restrict__ count, int* __restrict__ off, int* __restrict__ poff, int* __restrict__ block_expert,
    int* __restrict__ block_rows, int* __restrict__ n_blocks, int* __restrict__ max_count,
    int* __restrict__ slot_of, int* __restrict__ row_token, int* __restrict__ row_topk,
    float* __restrict__ row_weight, int* __restrict__ err) {
    extern __shared__ int s_mem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x / 32;
    int* s_next = s_mem;                       // [E] histogram (phase 1), next free slot (phase 3)
    int* s_wcnt = s_mem + E;                   // [nwarps][E]
    int* s_part = s_mem + E * (1 + nwarps);    // [2 * blockDim.x]
    int* s_tot = s_part + 2 * blockDim.x;      // [E] count of each expert
    int* s_base = s_tot + E;                   // [E] base of the current slot chunk
    int* s_poff = s_base + E;                  // [E] padded offset of each expert
    __shared__ __align__(8) int s_warp2[64];
    __shared__ int s_chunk, s_state, s_max;
    constexpr int kDone = -1, kWait = -2, kTimedOut = -3;
    int e_r[kFusedPer];
    float w_r[kFusedPer];
    if (tid == 0) {
        s_max = 0;
        s_chunk = atomicAdd(&sync[0], 1);
    }
    for (int e = tid; e < E; e += blockDim.x) s_next[e] = 0;
    __syncthreads();
    // 1. the chunk this CTA holds in registers
    const int c0 = s_chunk;
    if (c0 < chunks) {
        const int64_t base = static_cast<int64_t>(c0) * kRouteChunk;
        const int64_t end = min(base + kRouteChunk, n_entries);
        bool bad = false;
#pragma unroll
        for (int q = 0; q < kFusedPer; ++q) {
            const int64_t i = base + q * kScanThreads + tid;
            e_r[q] = entry_expert(topk_idx, i, end, E, &bad);
            w_r[q] = i < end ? __ldg(topk_w + i) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < kFusedPer; ++q) {
            const uint32_t same = __match_any_sync(0xffffffffu, e_r[q]);
            if (e_r[q] >= 0 && lane == __ffs(same) - 1) atomicAdd(&s_next[e_r[q]], __popc(same));
        }
        if (bad) atomicOr(err, kDevErrBadExpert);
        __syncthreads();
        for (int e = tid; e < E; e += blockDim.x) hist[static_cast<size_t>(c0) * E + e] = s_next[e];
        __syncthreads();
        if (tid == 0) {
            chunk_kind[c0] = 1;  // ranked from registers by this CTA
            __threadfence();     // the histogram row and the mark before the count of finished chunks
            atomicAdd(&sync[2], 1);
        }
    }
    // wait until every chunk is counted, counting untaken chunks meanwhile
    const uint64_t deadline = globaltimer_ns() + kRouteWaitNs;
    while (true) {
        if (tid == 0) {
            int state = kWait;
            if (ld_acquire_gpu_int(&sync[2]) >= chunks) {
                state = kDone;
            } else if (*reinterpret_cast<volatile int*>(&sync[0]) < chunks) {
                const int c = atomicAdd(&sync[0], 1);
                if (c < chunks) state = c;
            } else if (globaltimer_ns() > deadline) {
                state = kTimedOut;
            } else {
                __nanosleep(128);
            }
            s_state = state;
        }
        __syncthreads();
        const int state = s_state;
        __syncthreads();
        if (state == kDone) break;
        if (state == kTimedOut) {
            if (tid == 0) {
                atomicOr(err, kDevErrTimeout);
                atomicCAS(err + 1, 0, 1 + 99);
            }
            return;
        }
        if (state >= 0) {
            count_chunk(topk_idx, n_entries, E, state, hist, err, s_mem);
            __syncthreads();
            if (tid == 0) {
                chunk_kind[state] = 2;  // ranked from memory in phase 3
                atomicAdd(&sync[3], 1);
                __threadfence();
                atomicAdd(&sync[2], 1);
            }
        }
    }
    // 2. totals and this CTA's chunk base, then the scans, in every CTA
    chunk_sums(hist, chunks, E, min(c0, chunks), s_part, s_tot, s_base);
    const int c_e = tid < E ? s_tot[tid] : 0;
    const int padded = (c_e + kBlockM - 1) / kBlockM * kBlockM;
    int inc_c, inc_p;
    block_inclusive_scan2(c_e, padded, s_warp2, inc_c, inc_p);
    if (tid < E) {
        s_poff[tid] = inc_p - padded;
        if (blockIdx.x == 0) {
            count[tid] = c_e;
            off[tid] = inc_c - c_e;
            poff[tid] = inc_p - padded;
            if (c_e > 0) atomicMax(&s_max, c_e);
            if (tid == E - 1) {
                off[E] = inc_c;
                poff[E] = inc_p;
                *n_blocks = inc_p / kBlockM;
            }
        }
    }
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0) *max_count = s_max;
    // the row-block tables and the padding rows: one expert per warp of the grid
    for (int x = blockIdx.x * nwarps + warp; x < E; x += gridDim.x * nwarps) {
        const int c_x = s_tot[x], p_x = s_poff[x];
        const int nb = (c_x + kBlockM - 1) / kBlockM;
        for (int b = lane; b < nb; b += 32) {
            block_expert[p_x / kBlockM + b] = x;
            block_rows[p_x / kBlockM + b] = min(kBlockM, c_x - b * kBlockM);
        }
        for (int r = p_x + c_x + lane; r < p_x + nb * kBlockM; r += 32) {
            row_token[r] = -1;
            row_topk[r] = -1;
            row_weight[r] = 0.0f;
        }
    }
    // 3. stable slots: the chunk held in registers
    if (c0 < chunks) {
        for (int e = tid; e < E; e += blockDim.x) {
            s_next[e] = s_poff[e] + s_base[e];
            for (int w = 0; w < nwarps; ++w) s_wcnt[w * E + e] = 0;
        }
        __syncthreads();
        const int64_t base = static_cast<int64_t>(c0) * kRouteChunk;
        const int64_t end = min(base + kRouteChunk, n_entries);
#pragma unroll
        for (int q = 0; q < kFusedPer; ++q) {
            if (base + q * kScanThreads >= end) break;  // a short last chunk has fewer rounds (uniform)
            const int64_t i = base + q * kScanThreads + tid;
            const int slot = rank_round(e_r[q], E, s_next, s_wcnt);
            if (i < end) write_slot(i, slot, w_r[q], k, slot_of, row_token, row_topk, row_weight);
        }
    }
    // then the chunks counted from memory (final: counted before sync[2] was)
    if (__ldcg(&sync[3]) == 0) return;
    while (true) {
        __syncthreads();
        if (tid == 0) {
            int c = atomicAdd(&sync[1], 1);
            while (c < chunks && __ldcg(&chunk_kind[c]) != 2) c = atomicAdd(&sync[1], 1);
            s_chunk = c;
        }
        __syncthreads();
        const int c = s_chunk;
        if (c >= chunks) break;
        chunk_sums(hist, chunks, E, c, s_part, s_tot, s_base);
        for (int e = tid; e < E; e += blockDim.x) {
            s_next[e] = s_poff[e] + s_base[e];
            for (int w = 0; w < nwarps; ++w) s_wcnt[w * E + e] = 0;
        }
        __syncthreads();
        slot_rank(topk_idx, topk_w, n_entries, k, E, c, s_next, s_wcnt, slot_of, row_token, row_topk, row_weight);
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
    int* s_wcnt = s_mem + E;                 // [nwarps][E] same-expert counts per warp of the entries being ranked
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
    if (L.E <= kFusedMaxExperts) {  // the whole plan in one launch
        // the error record and the plan's four scheduling words start at zero
        cudaError_t st = cudaMemsetAsync(err, 0, kErrWords * sizeof(int), s);
        if (st != cudaSuccess) return st;
        const int ctas = std::min(std::max(L.chunks, kFusedMinCtas), 512);
        const size_t smem = (static_cast<size_t>(L.E) * (4 + kScanThreads / 32) + 2 * kScanThreads) * sizeof(int);
        route_fused_kernel<<<ctas, kScanThreads, smem, s>>>(
            topk_idx, topk_w, n, L.k, L.E, L.chunks, err + kErrSyncOff, hist, chunk_base, count, off, poff,
            reinterpret_cast<int*>(ws + L.block_expert), reinterpret_cast<int*>(ws + L.block_rows),
            reinterpret_cast<int*>(ws + L.n_blocks), reinterpret_cast<int*>(ws + L.max_count),
            reinterpret_cast<int*>(ws + L.slot_of), reinterpret_cast<int*>(ws + L.row_token),
            reinterpret_cast<int*>(ws + L.row_topk), reinterpret_cast<float*>(ws + L.row_weight), err);
        return cudaGetLastError();
    }
    if (L.chunks == 1) {  // one kernel for a decode-sized batch of many experts
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
    cudaError_t st = cudaMemsetAsync(err, 0, kErrWords * sizeof(int), s);
    if (st != cudaSuccess) return st;
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
