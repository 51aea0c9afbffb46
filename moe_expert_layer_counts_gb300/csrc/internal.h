// internal.h -- workspace layout and the launchers shared by the C-ABI
// translation unit and the kernel translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kBlockM = MOE_BLOCK_M;   // pool rows per MMA tile
constexpr int kBlockK = 128;           // K per pipeline stage (one scale chunk)
constexpr int kSfVec = 32;             // elements per UE8M0 scale
constexpr int kSfChunkBytes = 512;     // 128 rows x 4 scales, tensor-core layout
constexpr int kRouteChunk = 2048;      // top-k entries per routing CTA
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopk = 32;
constexpr int kSchedWords = 4;         // work counters at the head of the scheduler region

// Device-side error bits recorded in the workspace (word 0); word 1 records
// where a bounded wait expired.
constexpr int kDevErrBadExpert = 1;
constexpr int kDevErrTimeout = 2;
constexpr int kDevErrBounds = 4;  // a bounds check of a debug build fired (MOE_DEBUG)

// Bounds checks of debug builds (compiled with -DMOE_DEBUG; the release build
// has none and no cost).  moe_dcheck(v, lo, hi, err, where) is true when
// lo <= v < hi; otherwise it records kDevErrBounds in err[0] and, if no
// earlier failure is recorded, 200 + where in err[1], and returns false so
// the caller skips (or clamps) the access.  Places: 1 dispatch (pool row of
// a slot), 2 combine (L2 row of a slot), 3 expert kernel (a row block's
// expert and valid rows).
constexpr int kWhereDispatch = 1, kWhereCombine = 2, kWhereExpertBlock = 3;
#if defined(__CUDACC__)
__device__ __forceinline__ bool moe_dcheck(int64_t v, int64_t lo, int64_t hi, int* err, int where) {
#ifdef MOE_DEBUG
    if (v >= lo && v < hi) return true;
    atomicOr(err, kDevErrBounds);
    atomicCAS(err + 1, 0, 200 + where);
    return false;
#else
    (void)v, (void)lo, (void)hi, (void)err, (void)where;
    return true;
#endif
}
#endif
// The error record's region: words 0-1 the record, words 4-7 the scheduling
// words of the one-launch plan kernel (zeroed together before each plan).
constexpr int kErrWords = 8;
constexpr int kErrSyncOff = 4;

// Byte offsets of every array inside the caller's workspace.
struct Layout {
    int T, k, E, H, I;
    int chunks;        // routing chunks (CTAs of the count / slot kernels)
    int64_t p_cap;     // pool row capacity (multiple of kBlockM)
    size_t err, n_blocks, max_count, count, off, poff, hist, chunk_base, block_expert, block_rows;
    size_t slot_of, row_token, row_topk, row_weight;
    size_t pool_q, pool_sf, h_q, h_sf, l2_out;
    size_t x_q;        // token-major MXFP8 codes of x [T, H] (layer 1 gathers its rows from here)
    size_t sched;      // expert kernels: work counters (L1, L2, fused), then per row block the
                       // layer-1 epilogue warps done (fused kernel's readiness counters)
    size_t total;
};

bool make_layout(int T, int k, int E, int H, int I, Layout* L);

// Plan storage behind moe_plan_t.
struct PlanState {
    uint64_t magic;
    uint8_t* ws;
    size_t ws_bytes;
    int32_t T, k, E, H, I, device;
};
static_assert(sizeof(PlanState) <= sizeof(moe_plan_t), "plan storage too small");
constexpr uint64_t kPlanMagic = 0x4D6F45506C616E31ull;  // "MoEPlan1"

// Launchers (enqueue only; return cudaError_t of the launch).
cudaError_t launch_route(const Layout& L, uint8_t* ws, const int64_t* topk_idx, const float* topk_w,
                         cudaStream_t s);
// gather: write each token's codes once, token-major, instead of the pool rows
// (the pool's scales are written either way).
cudaError_t launch_dispatch(const Layout& L, uint8_t* ws, const void* x, int scale_rule, bool gather,
                            cudaStream_t s);
cudaError_t launch_combine(const Layout& L, uint8_t* ws, void* y, cudaStream_t s);
cudaError_t launch_prepare_sf(const uint8_t* sf, int E, int N, int K, int halves, uint8_t* out, size_t out_bytes,
                              cudaStream_t s);

cudaError_t launch_bounded_wait_selftest(int arrive, uint64_t timeout_ns, int32_t* out, cudaStream_t s);
cudaError_t launch_mma_rate_selftest(int kblocks, int ctas, int32_t* status, cudaStream_t s);
cudaError_t launch_stream_rate_selftest(const void* a, const void* b, const void* sfa, const void* sfb, int kblocks,
                                        int ctas, int32_t* status, cudaStream_t s);
// The layer-1 GEMM's operand maps: A as 128-row boxes of a [rows, K] E4M3
// matrix, B as the 3-D two-plane E2M1 map [2][rows][K] (256 weight rows per
// request), both as the expert kernel builds them.
bool make_layer1_operand_maps(CUtensorMap* a_map, const void* a, CUtensorMap* b_map, const void* b, uint64_t K,
                              uint64_t rows);

struct GemmLaunch {
    const void* w_q;      // packed e2m1 weights [E, N, K/2]
    const void* w_sf;     // tensor-core scale layout
    int E, N, K;
    float clamp;          // layer 1: limit of the bf16 gate/up values (0 = none)
    int scale_rule;       // layer 1: MOE_SCALE_CEIL or MOE_SCALE_OCP_FLOOR for h
    int fast_math;        // layer 1: 1 = fast SwiGLU with exact decisions, 0 = exact everywhere
    bool a_gather;        // layer 1: A rows gathered by token from token-major x (tile::gather4)
};
// layer 1: pool x W1 -> requantised h; layer 2: h x W2 -> bf16 rows.
cudaError_t launch_expert_gemm(int layer, const Layout& L, uint8_t* ws, const GemmLaunch& g, int num_sms,
                               cudaStream_t s);
// Both layers in one persistent launch (layer-2 tiles of a row block start once
// that block's layer-1 tiles have stored h).
// publish == false is the failure-detection self-test: no row block ever
// becomes ready, so every layer-2 tile's bounded wait expires.
cudaError_t launch_expert_fused(const Layout& L, uint8_t* ws, const GemmLaunch& g1, const GemmLaunch& g2, int num_sms,
                                cudaStream_t s, bool publish = true);

}  // namespace moe
