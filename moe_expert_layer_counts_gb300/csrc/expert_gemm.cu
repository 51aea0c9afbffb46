// expert_gemm.cu -- persistent grouped GEMM over the expert-major pool on the
// 5th-generation tensor cores: A = pool rows (E4M3), B = expert weights
// (E2M1), UE8M0 scales per 32 along K, fp32 accumulation in tensor memory
// (page "DeepEP -> Mega MoE", sm100_fp8_fp4_mega_moe.cuh snippets: the
// block-scaled MXF8F6F4 MMA, the TMA-A / TMA-B / MMA / epilogue warp roles,
// the SwiGLU + amax + FP8 requant epilogue; "Normal vs Low-Latency" page
// sections 3 and 5: one persistent CTA per SM, pipeline depth set by shared
// memory).
//
// Layer 1: a work item is (pool row block b, intermediate tile j of 128).  The
//   MMA has N = 256: weight rows gate [j*128, +128) and up [I + j*128, +128)
//   arrive in one 3-D TMA box (expert-half as the outer dimension) into one B
//   tile, so SwiGLU is tile-local.
//   Epilogue per pool row: g = bf16(acc_gate), u = bf16(acc_up),
//   h = (g / (1 + exp(-g))) * u * topk_weight in fp32, requantised per 32 to
//   E4M3 + UE8M0 (scales written in the tensor-core layout L2 reads).
// Layer 2: a work item is (pool row block b, output tile j of 256 columns);
//   epilogue rounds the fp32 accumulators to bf16 rows in pool order.  Each
//   epilogue warp stages 32 rows x 32 columns at a time in shared memory and
//   writes them with a TMA tensor store: per-thread row stores (32 rows x 16
//   bytes per instruction) held up the next tile's operand loads.
//
// Warp roles (352 threads, one CTA per SM, persistent over work items):
//   warp 0   TMA producer: A box, the B tile, the two scale copies per stage
//   warp 1   tensor-memory owner and MMA issuer (one elected thread)
//   warps 2-9 epilogue; warp w reads tensor-memory lanes 32*(w%4)..+31 and
//            one half of the accumulator columns ((w-2)/4), so two warps
//            share each lane quadrant
//   warp 10  scale copies (shared memory -> tensor memory) for each stage,
//            so that the MMA thread issues only MMAs and stage releases
// Every wait is bounded (a global-timer deadline); on expiry the CTA records
// an error in the workspace, waits for its own copies in flight, releases
// tensor memory and exits.
#include <atomic>
#include <limits>

#include <cuda.h>
#include <cuda_runtime.h>

#include "formats.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBN = 256;                       // MMA N: 256 weight rows (gate|up halves for layer 1)
constexpr int kABytes = kBlockM * kBlockK;     // 16 KB of E4M3
constexpr int kBBytes = kBN * kBlockK;         // 32 KB in smem: E2M1 unpacked to one byte per element
constexpr int kBTxBytes = kBN * kBlockK / 2;   // a FP4 box's transaction count is its packed size
// A stage: the A box, the whole B tile in one request (a 3-D map for layer 1
// brings the gate and up rows together; a 256-row box for layer 2), and two
// scale copies (SFA chunk 512 B, SFB chunk pair 1 KB) after A and B.
constexpr int kStageTxBytes = kABytes + kBTxBytes + 3 * kSfChunkBytes;
// The operand ring has one of two shapes, chosen per launch from the plan:
//   wide:   4 stages of 50 KB (A 16 KB for 128 rows, B 32 KB, scales 2 KB)
//   narrow: 6 stages of 36 KB (A 2 KB for 16 rows, B, scales), used when no
//           expert has more than 16 rows (decode-sized batches): the stream is
//           then weight bytes from HBM, and 6 stages keep 50% more of them in
//           flight.  The MMA still reads a 16 KB A window from the stage start;
//           beyond the 16 loaded rows it covers the stage's own B bytes, which
//           feed only accumulator rows that are never stored.
constexpr int kMaxStages = 6;
constexpr int kWideStages = 4, kWideStride = 51200, kWideABytes = kABytes;
constexpr int kNarrowStages = 6, kNarrowStride = 36864, kNarrowABytes = 16 * kBlockK;
constexpr int kNarrowRows = 16;
static_assert(kWideABytes + kBBytes + 3 * kSfChunkBytes <= kWideStride && kWideStride % 1024 == 0, "wide stage");
static_assert(kNarrowABytes + kBBytes + 3 * kSfChunkBytes <= kNarrowStride && kNarrowStride % 1024 == 0,
              "narrow stage");
static_assert(kNarrowABytes + kBBytes >= kABytes, "the MMA's A window stays inside a narrow stage");
// A row block that is not full (an expert's last block, or decode-sized
// batches) loads only the first 16, 32 or 64 rows of A that hold its valid
// rows: the MMA still multiplies 128 rows, the others hold stale shared memory
// and their accumulator rows are never stored.
constexpr int kABoxLevels = 4;  // A boxes of 16, 32, 64 and 128 rows

struct Maps {
    CUtensorMap box[kABoxLevels];  // A: boxes of 16, 32, 64 and 128 rows
    CUtensorMap out;               // layer 2 output: bf16 [P_cap][H], box 32 x 32, 64-byte swizzle
    CUtensorMap gather;            // layer 1, gathered A: token-major x codes [T][H], box 128 K x 1 row
};

__device__ __forceinline__ int a_box_level(int rows) {
    return rows <= 16 ? 0 : rows <= 32 ? 1 : rows <= 64 ? 2 : 3;
}
// Shared memory: barriers (1 KB), the ring, and (wide ring only) the layer-2
// output staging, which a narrow ring overlaps: with at most 16 rows per
// block no epilogue warp ever holds 32 routed rows, the staged path's condition.
constexpr int kRingOff = 1024;
constexpr int kOutStageBytes = 2048;           // layer 2: 32 rows x 32 bf16 per epilogue warp
constexpr int kOutStageOff = kRingOff + kWideStages * kWideStride;
constexpr int kTmemCols = 512;
constexpr int kSfTmemCol = 256;                // scale slots: 16 columns per stage
constexpr int kThreads = 352;                  // 11 warps: TMA, MMA, 8 epilogue, scale copies
constexpr int kEpiWarps = 8;
constexpr int kScaleWarp = 10;
constexpr int kSmemEnd = kOutStageOff + kEpiWarps * kOutStageBytes;
static_assert(kRingOff + kNarrowStages * kNarrowStride <= kSmemEnd, "narrow ring inside the allocation");
constexpr int kSmemBytes = kSmemEnd + 1024;    // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kSfTmemCol + 16 * kMaxStages <= kTmemCols, "scale slots");
// Bounded waits: 1 s for the producer thread, whose waits are the only ones
// that depend on anything outside the CTA (its copies, the work counter and,
// fused, other CTAs' layer-1 tiles); 2 s for every wait downstream of it, so
// that when something outside stalls, the producer's wait expires first and
// the error record names the root cause.
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr uint64_t kReaderWaitNs = 2 * kWaitNs;

struct GemmParams {
    const int* n_blocks;
    const int* block_expert;
    const int* row_token;
    const float* row_weight;
    const uint8_t* sfa;     // activation scales, chunks [P_cap/128][K/128]
    const uint8_t* sfb;     // weight scales, [E][N/256 pairs][K/128][2][512]
    uint8_t* out_q;         // layer 1: E4M3 h [P_cap, I]
    uint8_t* out_sf;        // layer 1: scales of h, chunks [P_cap/128][I/128]
    uint16_t* out_bf16;     // layer 2: bf16 rows [P_cap, H]
    int K;                  // reduction length
    int N;                  // weight rows per expert
    int n_tiles;            // work items per pool row block
    int I;                  // layer 1: intermediate size
    int H;                  // layer 2: output columns
    int* err;
    float clamp;            // layer 1: gate/up limit, +inf for none
    int scale_rule;         // layer 1: 0 = ceil, 1 = OCP floor (scales of h)
    int fast_math;          // layer 1: 0 = every SwiGLU value by the exact formula
    const int* block_rows;  // valid rows of each pool row block (plan)
    const int* max_count;   // largest expert count (plan): selects the ring shape
    const uint8_t* a_rows;  // A operand rows (pool or h), K bytes each
    int a_gather;           // layer 1: A rows gathered by token (tile::gather4 from maps.gather)
    int E;                  // experts (the range of block_expert; checked in debug builds)
};

// Work items are handed out by a global counter (dynamic scheduling: a CTA
// takes its next item when it starts the current one).  The producer thread
// takes them and passes each item number to the MMA thread, the scale warp
// and the epilogue warps through a small queue in shared memory; a number at
// or beyond the item count ends the CTA's loop.
constexpr int kQueue = 4;
constexpr int kItemReaders = 2 + kEpiWarps;   // MMA thread, scale warp, epilogue warps

struct Shared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t sf_ready[kMaxStages];   // the stage's scales are in tensor memory
    uint64_t sf_drain;
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint64_t item_full[kQueue];
    uint64_t item_empty[kQueue];
    int item[kQueue];
    uint32_t tmem_base;
    int abort;
};

// On expiry the first CTA to give up records where: err[1] = 1 + where, with
// where = stage (producer waiting on empty), 16 (MMA on tmem_empty),
// 32 + stage (MMA on the stage's operands and scales), 48 (epilogue on
// tmem_full), 64 + stage (scale warp on the stage's operands), 80 (fused: a
// layer-2 tile on its row block's layer-1 tiles), 96 (producer on a queue
// slot), 97 (a reader on the next item number).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, Shared* sh, int* err, int where,
                                              uint64_t wait_ns = kReaderWaitNs) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::mbar_wait(bar, parity, ptx::globaltimer() + wait_ns)) return true;
    atomicOr(err, kDevErrTimeout);
    atomicCAS(err + 1, 0, 1 + where);
    *reinterpret_cast<volatile int*>(&sh->abort) = 1;
    return false;
}
__device__ __forceinline__ bool aborted(Shared* sh) { return *reinterpret_cast<volatile int*>(&sh->abort) != 0; }

// Producer side of the item queue: the seq-th item number of this CTA into
// slot seq % kQueue, once every reader has taken the item kQueue before it.
__device__ __forceinline__ bool put_item(Shared* sh, int seq, int w, int* err) {
    const int slot = seq & (kQueue - 1);
    if (seq >= kQueue &&
        !wait_or_abort(ptx::smem_addr(&sh->item_empty[slot]), ((seq / kQueue) - 1) & 1, sh, err, 96, kWaitNs))
        return false;
    sh->item[slot] = w;
    ptx::mbar_arrive(ptx::smem_addr(&sh->item_full[slot]));  // release: the number is visible to the readers
    return true;
}
// Reader side: the seq-th item number (one thread per reader); -1 if the
// wait expired.
__device__ __forceinline__ int get_item(Shared* sh, int seq, int* err) {
    const int slot = seq & (kQueue - 1);
    if (!wait_or_abort(ptx::smem_addr(&sh->item_full[slot]), (seq / kQueue) & 1, sh, err, 97)) return -1;
    const int w = sh->item[slot];
    ptx::mbar_arrive(ptx::smem_addr(&sh->item_empty[slot]));
    return w;
}

// SwiGLU of one value by the exact definition, (float)(g / (1 + exp(-g))) in
// double; kept out of line so the rare callers stay small.
__device__ __noinline__ float silu_exact(float g) {
    return static_cast<float>(static_cast<double>(g) / (1.0 + exp(-static_cast<double>(g))));
}

// SwiGLU * topk weight and MXFP8 requantisation of 32 intermediate columns
// of one pool row ("DeepEP -> Mega MoE" page, SwiGLU / amax / FP8 cast
// snippets).  gu holds (bf16 gate, bf16 up) pairs.  The fast path uses
// __expf and an approximate divide (error well below kDecisionUlps for
// |gate| <= 16).  Wherever that could change an integer decision under the
// exact formula, the exact value is used instead: an element with
// |gate| > 16, or with a rounding boundary of the E4M3 grid within
// kDecisionUlps of it, is recomputed alone; if the block maximum lies that
// close to the UE8M0 scale boundary, the whole block is recomputed.  So every
// code and scale byte is the one the exact definition gives.  The fast path is branch-free (it only collects
// bit masks), so the 32 values are computed with full instruction-level
// parallelism.  Writes 32 E4M3 codes to dst (16-byte aligned) and returns the
// scale byte.
constexpr uint32_t kDecisionUlps = 64;

// The optional activation clamp: the bf16 gate / up value limited to
// [-c, c] (c = +inf when off, which leaves every finite value unchanged).
__device__ __forceinline__ float clamp_act(float v, float c) { return fminf(fmaxf(v, -c), c); }

// Replace h[i] by its exact value for every bit i set in `mask` (rare; a
// local copy keeps dynamic indexing off the fast path).
__device__ __noinline__ void exact_fixup(const uint32_t* gu, float wgt, float clamp, float* h, uint32_t mask) {
    while (mask) {
        const int i = __ffs(mask) - 1;
        mask &= mask - 1;
        h[i] = (silu_exact(clamp_act(bf16_lo(gu[i]), clamp)) * clamp_act(bf16_hi(gu[i]), clamp)) * wgt;
    }
}

__device__ __forceinline__ void fixup(const uint32_t* gu, float wgt, float clamp, float (&h)[32], uint32_t mask) {
    uint32_t gl[32];
    float hl[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        gl[i] = gu[i];
        hl[i] = h[i];
    }
    exact_fixup(gl, wgt, clamp, hl, mask);
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = hl[i];
}

// kClamp: the optional activation clamp is on (a kernel instantiation of its
// own, so the default path carries no clamp arithmetic: layer 1 ran 2-3%
// faster without it).
template <bool kClamp>
__device__ __forceinline__ uint32_t requant_block(const uint32_t* gu, float wgt, uint8_t* dst, float clamp,
                                                  int scale_rule, int fast_math) {
    // 1. fast path, straight-line: values, block maximum, values it cannot decide
    float h[32];
    uint32_t big = fast_math ? 0u : 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float g = kClamp ? clamp_act(bf16_lo(gu[i]), clamp) : bf16_lo(gu[i]);
        const float u = kClamp ? clamp_act(bf16_hi(gu[i]), clamp) : bf16_hi(gu[i]);
        h[i] = (__fdividef(g, 1.0f + __expf(-g)) * u) * wgt;
        big |= static_cast<uint32_t>(fabsf(g) > 16.0f) << i;
    }
    if (big) fixup(gu, wgt, clamp, h, big);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
    // 2. the scale: if the maximum sits near the rule's boundary, the whole block goes exact
    if (scale_rule ? near_pow2(amax, kDecisionUlps) : near_e4m3_scale_boundary(amax, kDecisionUlps)) {
        fixup(gu, wgt, clamp, h, 0xFFFFFFFFu);
        amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
    }
    const uint32_t sbyte = ue8m0_scale_e4m3_rule(amax, scale_rule);
    const float inv = inv_scale_from_byte(sbyte);
    // 3. the codes.  The E4M3 codes of q*(1-eps) and q*(1+eps), eps = kDecisionUlps
    // * 2^-23 (at least kDecisionUlps ulps of q), are equal unless a rounding
    // boundary of the E4M3 grid (normal or subnormal) lies within the band;
    // then the fast value could round differently from the exact one and goes
    // exact.  Otherwise either code is the exact value's code.
    constexpr float kLo = 1.0f - static_cast<float>(kDecisionUlps) * 0x1p-23f;
    constexpr float kHi = 1.0f + static_cast<float>(kDecisionUlps) * 0x1p-23f;
    uint32_t near = 0;
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float q0 = h[2 * i] * inv, q1 = h[2 * i + 1] * inv;
        const uint32_t a = e4m3x2(q0 * kLo, q1 * kLo), c = e4m3x2(q0 * kHi, q1 * kHi);
        const uint32_t d = a ^ c;
        near |= (static_cast<uint32_t>((d & 0xFFu) != 0u) | (static_cast<uint32_t>((d & 0xFF00u) != 0u) << 1)) << (2 * i);
        if (i & 1)
            q[i >> 1] |= a << 16;
        else
            q[i >> 1] = a;
    }
    if (near) {
        fixup(gu, wgt, clamp, h, near);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            q[i] = e4m3x2(h[4 * i] * inv, h[4 * i + 1] * inv) | (e4m3x2(h[4 * i + 2] * inv, h[4 * i + 3] * inv) << 16);
    }
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(q[0], q[1], q[2], q[3]);
    d[1] = make_uint4(q[4], q[5], q[6], q[7]);
    return sbyte;
}

// Drain this warp's half of one accumulator row block from tensor memory
// (32 lanes = 32 rows, 128 of the 256 columns) with wide loads, signal that the
// accumulator may be overwritten (release(), once the loads have landed), and
// pack the values as bf16 pairs: layer 1 (gate, up) of one intermediate
// column, layer 2 two adjacent output columns.
template <int kLayer, typename Release>
__device__ __forceinline__ void drain_accumulator(uint32_t t_row, int half, uint32_t (&pk)[64], Release release) {
    if (kLayer == 1) {
        uint32_t g[64], u[64];
        ptx::tmem_ld_32x32b_x64(t_row + 64 * half, g);
        ptx::tmem_ld_32x32b_x64(t_row + 128 + 64 * half, u);
        ptx::tc_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        release();
        // gate/up rounded to bf16 (the reading of the pages' bf16 gate/up)
#pragma unroll
        for (int i = 0; i < 64; ++i) pk[i] = bf16x2_rn(__uint_as_float(g[i]), __uint_as_float(u[i]));
    } else {
        uint32_t v[128];
        ptx::tmem_ld_32x32b_x128(t_row + 128 * half, v);
        ptx::tc_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        release();
#pragma unroll
        for (int i = 0; i < 64; ++i) pk[i] = bf16x2_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    }
}

// Layer 1: requantise one pool row's 64 intermediate columns of a finished
// tile (columns j*128 + 64*half + [0, 64), two 32-blocks) to E4M3 + scales.
// The two blocks go through one copy of the unrolled requant code (a loop
// that is not unrolled, the block selected without dynamic indexing): with
// two copies the kernel's code is twice as large, and on short-K shapes
// (K = 2048) layer 1 ran 12% slower.
template <bool kClamp>
__device__ __forceinline__ void store_h_row(const GemmParams& p, int b, int j, int r, int quad, int half, int lane,
                                            float wgt, const uint32_t (&pk)[64]) {
    uint8_t* dst = p.out_q + static_cast<size_t>(r) * p.I + j * 128 + 64 * half;
    uint32_t s0 = 0, s1 = 0;
#pragma unroll 1
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t cur[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) cur[i] = blk ? pk[32 + i] : pk[i];
        const uint32_t sb = requant_block<kClamp>(cur, wgt, dst + 32 * blk, p.clamp, p.scale_rule, p.fast_math);
        if (blk)
            s1 = sb;
        else
            s0 = sb;
    }
    const size_t chunk = static_cast<size_t>(b) * (p.I / 128) + j;
    *reinterpret_cast<uint16_t*>(p.out_sf + chunk * kSfChunkBytes + 16 * lane + 4 * quad + 2 * half) =
        static_cast<uint16_t>(s0 | (s1 << 8));
}

// Layer 2, partly filled row groups (an expert's last block; decode-sized
// batches): each routed row's 128 bf16 columns straight from its lane.
__device__ __forceinline__ void store_out_rows_direct(const GemmParams& p, int r, int col0, const uint32_t (&pk)[64]) {
    uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + static_cast<size_t>(r) * p.H + col0);
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// Layer 2: one warp's 32 rows x 128 bf16 columns of a finished tile (lane =
// row, columns col0 + [0, 128)) go out in four 32 x 32 blocks through the
// warp's 2 KB staging buffer and a TMA tensor store each.  The buffer uses the
// map's 64-byte swizzle (16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)),
// which also makes the row-per-lane writes free of bank conflicts.  Before a
// buffer is rewritten, lane 0 waits until its previous store has read it.
// Used when all 32 rows hold routed entries; a warp with padding rows writes
// its routed rows directly (store_out_rows_direct).
__device__ __forceinline__ void store_out_rows(const CUtensorMap* map, uint8_t* stg, int col0, int row0, int lane,
                                               const uint32_t (&pk)[64]) {
    const uint32_t stg_addr = ptx::smem_addr(stg);
    const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t* v = pk + 16 * blk + 4 * c;
            *reinterpret_cast<uint4*>(stg + lane * 64 + 16 * (c ^ sw)) = make_uint4(v[0], v[1], v[2], v[3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            ptx::tma_store_2d(map, col0 + 32 * blk, row0, stg_addr);
            ptx::bulk_commit_group();
        }
    }
}

// Everything a launch needs, for both layers: the tensor maps (grid constants,
// which the TMA unit reads in parameter space) and each layer's parameters.
// A one-layer launch uses entry layer-1; the fused launch uses both.
struct KernelArgs {
    Maps maps[2];            // A boxes of each layer (+ layer 2's output map)
    CUtensorMap tmap_b[2];   // W1 as a 3-D map (expert-half, row, K), W2 as a 2-D map
    GemmParams p[2];
    int* l1_done;            // fused: per pool row block, epilogue warps done with its h rows
    int* blocks_done;        // fused: row blocks whose layer-1 tiles are all done
    int* work_ctr;           // items handed out (zero at launch)
};

// Work item w -> (layer, pool row block, tile).  kMode 1 or 2: that layer's
// items, block-major.  kMode 3 (fused): all of layer 1's items first, then
// all of layer 2's, so an item only ever waits on items before it.
template <int kMode>
__device__ __forceinline__ void decode_item(const KernelArgs& ka, int w, int n_work1, int& layer, int& b, int& j) {
    if (kMode == 3) {
        layer = w < n_work1 ? 1 : 2;
        if (layer == 2) w -= n_work1;
    } else {
        layer = kMode;
    }
    const int nt = ka.p[layer - 1].n_tiles;
    b = w / nt;
    j = w % nt;
}

// Fused launch: the layer-2 items of row block b wait until every epilogue
// warp of every layer-1 tile of b has stored its h rows and scales (release
// on the writer side: each lane fences, then one lane counts the warp in).
// The warp that completes a block also counts the block in `blocks_done`;
// once the producer has seen every block counted (one acquire), it skips the
// per-block check for the rest of the launch.
// Bounded: past the deadline the error is recorded and the CTA aborts.  The
// proxy fence orders the acquired generic-proxy view of h before the TMA
// (async-proxy) loads that follow.
__device__ __forceinline__ bool wait_l1_block(const int* counter, int target, Shared* sh, int* err) {
    if (ptx::ld_acquire_gpu(counter) < target) {
        const uint64_t deadline = ptx::globaltimer() + kWaitNs;
        while (ptx::ld_acquire_gpu(counter) < target) {
            if (aborted(sh)) return false;
            if (ptx::globaltimer() > deadline) {
                atomicOr(err, kDevErrTimeout);
                atomicCAS(err + 1, 0, 1 + 80);
                *reinterpret_cast<volatile int*>(&sh->abort) = 1;
                return false;
            }
            __nanosleep(128);
        }
    }
    ptx::fence_proxy_async_global();
    return true;
}

// kMode 1 / 2: one layer; kMode 3: both layers in one persistent launch.
// kGather: layer 1 gathers its A rows by token (the whole producer warp runs
// the producer loop); otherwise one thread runs it alone (the broadcasts a
// warp-wide loop needs cost 17% on the latency-bound operand stream).
template <int kMode, bool kClamp, bool kGather>
__global__ void __launch_bounds__(kThreads, 1) expert_gemm_kernel(const __grid_constant__ KernelArgs ka) {
#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ >= 1000)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared* sh = reinterpret_cast<Shared*>(smem);
    uint8_t* ring = smem + kRingOff;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // fields both layers share (the plan's tables, the error record)
    const GemmParams& p0 = ka.p[kMode == 2 ? 1 : 0];

    const int n_blocks = *p0.n_blocks;
    const int n_work1 = kMode == 2 ? 0 : n_blocks * ka.p[0].n_tiles;
    const int n_work = kMode == 1 ? n_work1
                       : kMode == 2 ? n_blocks * ka.p[1].n_tiles
                                    : n_work1 + n_blocks * ka.p[1].n_tiles;
    if (static_cast<int>(blockIdx.x) >= n_work) return;  // uniform for the CTA
    // ring shape (uniform for the launch)
    const bool narrow = *p0.max_count <= kNarrowRows;
    const int n_stages = narrow ? kNarrowStages : kWideStages;
    const int stride = narrow ? kNarrowStride : kWideStride;
    const int a_bytes = narrow ? kNarrowABytes : kWideABytes;
    const int sf_off = a_bytes + kBBytes;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&sh->full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh->empty[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh->sf_ready[s]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&sh->sf_drain), 1);
        ptx::mbar_init(ptx::smem_addr(&sh->tmem_full), 1);
        ptx::mbar_init(ptx::smem_addr(&sh->tmem_empty), kEpiWarps);
        ptx::mbar_init(ptx::smem_addr(&sh->drain), 1);
        for (int q = 0; q < kQueue; ++q) {
            ptx::mbar_init(ptx::smem_addr(&sh->item_full[q]), 1);
            ptx::mbar_init(ptx::smem_addr(&sh->item_empty[q]), kItemReaders);
        }
        sh->abort = 0;
        ptx::fence_mbar_init();
        for (int l = (kMode == 2 ? 1 : 0); l < (kMode == 1 ? 1 : 2); ++l) {
            for (int i = 0; i < kABoxLevels; ++i) ptx::prefetch_tensormap(&ka.maps[l].box[i]);
            ptx::prefetch_tensormap(&ka.tmap_b[l]);
        }
        if (kMode != 1) ptx::prefetch_tensormap(&ka.maps[1].out);
        if (kGather) ptx::prefetch_tensormap(&ka.maps[0].gather);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(&sh->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&sh->tmem_base);

    if (warp == 0 && (kGather || lane == 0)) {
        // ------------------------------------------------ TMA producer
        // Lane 0 takes every decision (waits, the work counter, the queue, all
        // copies but one kind).  With gathered A rows the whole warp runs the
        // loop in step, the decisions are broadcast, and lane l fetches rows
        // 4l..4l+3 of a layer-1 block with one tile::gather4 load; otherwise
        // lane 0 runs it alone and the broadcasts vanish.
        const bool leader = lane == 0;
        auto bcast = [&](int v) { return kGather ? __shfl_sync(0xffffffffu, v, 0) : v; };
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        bool ok;
        // Item numbers all come from the work counter, the first one too, so an
        // item is only ever held by a running CTA: a layer-2 tile's wait on
        // layer-1 tiles of lower numbers ends even when not every CTA of the
        // launch is resident (another stream's kernels on some SMs).  The next
        // item is taken when the current one starts, so its block metadata is
        // loaded one item ahead and never stalls the copies at a tile boundary.
        int seq = 0;
        int w = 0;
        if (leader) w = min(n_work, atomicAdd(ka.work_ctr, 1));
        w = bcast(w);
        int layer = 1, b = 0, j = 0, e = 0, rows = kBlockM;
        if (w < n_work) {
            decode_item<kMode>(ka, w, n_work1, layer, b, j);
            e = __ldg(p0.block_expert + b);
            rows = __ldg(p0.block_rows + b);
            // debug builds: a plan table out of range is reported and clamped, so
            // no copy leaves its tensor (release builds trust the plan kernel)
            if (!moe_dcheck(e, 0, p0.E, p0.err, kWhereExpertBlock)) e = 0;
            if (!moe_dcheck(rows, 1, kBlockM + 1, p0.err, kWhereExpertBlock)) rows = kBlockM;
        }
        bool all_l1_done = false;  // fused: every row block's layer-1 tiles seen complete
        ok = bcast(leader ? put_item(sh, seq, w, p0.err) : true);
        ++seq;
        while (ok && w < n_work) {
            int wn = 0;
            if (leader) wn = min(n_work, atomicAdd(ka.work_ctr, 1));
            wn = bcast(wn);
            if (!bcast(leader ? put_item(sh, seq, wn, p0.err) : true)) {
                ok = false;
                break;
            }
            ++seq;
            int next_layer = 0, next_b = 0, next_j = 0, next_e = 0, next_rows = 0;
            if (wn < n_work) {
                decode_item<kMode>(ka, wn, n_work1, next_layer, next_b, next_j);
                next_e = __ldg(p0.block_expert + next_b);
                next_rows = __ldg(p0.block_rows + next_b);
                if (!moe_dcheck(next_e, 0, p0.E, p0.err, kWhereExpertBlock)) next_e = 0;
                if (!moe_dcheck(next_rows, 1, kBlockM + 1, p0.err, kWhereExpertBlock)) next_rows = kBlockM;
            }
            const GemmParams& P = ka.p[layer - 1];
            const int kb_count = P.K / kBlockK;
            const int pairs = (P.N + 255) / 256;
            if (kMode == 3 && layer == 2 && !all_l1_done) {
                int st = 1;  // 1 ready, 2 all blocks done, 0 failed
                if (leader) {
                    if (ptx::ld_acquire_gpu(ka.blocks_done) >= n_blocks) {
                        st = 2;
                        ptx::fence_proxy_async_global();
                    } else if (!wait_l1_block(ka.l1_done + b, kEpiWarps * ka.p[0].n_tiles, sh, p0.err)) {
                        st = 0;
                    }
                }
                st = bcast(st);
                if (st == 0) {
                    ok = false;
                    break;
                }
                all_l1_done = st == 2;
            }
            // layer 1: gate|up halves of expert e, rows j*128 of each (3-D map: K, row, expert-half)
            // layer 2: rows e*H + 256*j .. +256 (2-D map)
            const int b_y = layer == 1 ? j * 128 : e * P.N + j * kBN;
            const int b_z = layer == 1 ? 2 * e : 0;
            const uint8_t* sfa = P.sfa + static_cast<size_t>(b) * kb_count * kSfChunkBytes;
            const uint8_t* sfb = P.sfb + (static_cast<size_t>(e) * pairs + j) * kb_count * 2 * kSfChunkBytes;
            const bool gather = kGather && layer == 1;
            // gathered A: groups of 4 rows covering the block's valid rows; the
            // token of a row (a padding row's token is -1: row 0 stands in, its
            // accumulator row is never stored)
            const int groups = (rows + 3) / 4;
            int t0 = 0, t1 = 0, t2 = 0, t3 = 0;
            if (gather && lane < groups) {
                const int4 tk = __ldg(reinterpret_cast<const int4*>(p0.row_token + b * kBlockM) + lane);
                t0 = max(tk.x, 0);
                t1 = max(tk.y, 0);
                t2 = max(tk.z, 0);
                t3 = max(tk.w, 0);
            }
            const int level = a_box_level(rows);  // the A box that covers the block's valid rows
            const uint32_t a_tx = gather ? groups * 4 * kBlockK : (16u << level) * kBlockK;
            const uint32_t tx = kStageTxBytes - kABytes + a_tx;
            const CUtensorMap* map_a = &ka.maps[layer - 1].box[level];
            const CUtensorMap* map_b = &ka.tmap_b[layer - 1];
            for (int kb = 0; kb < kb_count; ++kb) {
                bool go = true;
                if (leader)
                    go = !aborted(sh) &&
                         wait_or_abort(ptx::smem_addr(&sh->empty[stage]), phase ^ 1, sh, p0.err, stage, kWaitNs);
                if (!bcast(go)) {
                    ok = false;
                    break;
                }
                uint8_t* st = ring + stage * stride;
                const uint32_t full = ptx::smem_addr(&sh->full[stage]);
                if (leader) {
                    ptx::mbar_arrive_expect_tx(full, tx);
                    if (!gather) ptx::tma_load_2d(ptx::smem_addr(st), map_a, kb * kBlockK, b * kBlockM, full);
                    if (layer == 1)
                        ptx::tma_load_3d(ptx::smem_addr(st + a_bytes), map_b, kb * kBlockK, b_y, b_z, full);
                    else
                        ptx::tma_load_2d(ptx::smem_addr(st + a_bytes), map_b, kb * kBlockK, b_y, full);
                    ptx::bulk_load(ptx::smem_addr(st + sf_off), sfa + kb * kSfChunkBytes, kSfChunkBytes, full);
                    ptx::bulk_load(ptx::smem_addr(st + sf_off + kSfChunkBytes), sfb + kb * 2 * kSfChunkBytes,
                                   2 * kSfChunkBytes, full);
                }
                if (kGather) __syncwarp();
                if (gather && lane < groups)
                    ptx::tma_gather4(ptx::smem_addr(st + lane * 4 * kBlockK), &ka.maps[0].gather, kb * kBlockK, t0, t1,
                                     t2, t3, full);
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == n_stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok || wn >= n_work) break;
            w = wn;
            layer = next_layer;
            b = next_b;
            j = next_j;
            e = next_e;
            rows = next_rows;
        }
        if (!ok && leader) {
            // let this CTA's copies in flight land before the CTA may exit
            for (int s = 0; s < n_stages; ++s)
                if (issued_mask & (1u << s))
                    ptx::mbar_wait(ptx::smem_addr(&sh->full[s]), (issued_parity >> s) & 1u,
                                   ptx::globaltimer() + kWaitNs);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        // The issue rate of one thread bounds the MMA rate (each tcgen05
        // instruction takes tens of cycles to issue), so this thread issues
        // only the MMAs and the stage release; the scale copies come from the
        // scale warp, and everything that does not change with the k-block is
        // computed once.  A stage's shared-memory descriptors are those of
        // stage 0 plus the stage offset in 16-byte units (the start-address
        // field); a 32-wide K step adds 2.
        constexpr uint32_t idesc = ptx::idesc_e4m3_e2m1(kBlockM, kBN);
        const uint32_t st0 = ptx::smem_addr(ring);
        const uint64_t a_desc0 = ptx::desc_kmajor_sw128(st0);
        const uint64_t b_desc0 = ptx::desc_kmajor_sw128(st0 + a_bytes);
        const uint32_t ready0 = ptx::smem_addr(&sh->sf_ready[0]);
        const uint32_t empty0 = ptx::smem_addr(&sh->empty[0]);
        const uint32_t tsf0 = tmem + kSfTmemCol;
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true;
        for (int seq = 0; ok; ++seq) {
            const int w = get_item(sh, seq, p0.err);
            if (w < 0 || w >= n_work) break;
            const int kb_count = ka.p[(kMode == 3 ? (w < n_work1 ? 1 : 2) : kMode) - 1].K / kBlockK;
            if (aborted(sh) || !wait_or_abort(ptx::smem_addr(&sh->tmem_empty), acc_phase ^ 1, sh, p0.err, 16)) break;
            ptx::tc_fence_after();
            for (int kb = 0; kb < kb_count; ++kb) {
                // the stage's operands have landed and its scales are in tensor memory
                if (!wait_or_abort(ready0 + 8 * stage, phase, sh, p0.err, 32 + stage)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t so = static_cast<uint64_t>(stage * (stride >> 4));
                const uint32_t tsf = tsf0 + 16 * stage;
#pragma unroll
                for (int kk = 0; kk < kBlockK / 32; ++kk)
                    ptx::mma_mxf8f6f4(tmem, a_desc0 + so + 2 * kk, b_desc0 + so + 2 * kk,
                                      ptx::idesc_with_sf_id(idesc, kk), tsf + 0, tsf + 4, (kb | kk) != 0);
                ptx::tc_commit(empty0 + 8 * stage);
                if (++stage == n_stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            ptx::tc_commit(ptx::smem_addr(&sh->tmem_full));
            acc_phase ^= 1;
        }
        // all tensor-core work of this CTA done before tensor memory is freed
        ptx::tc_commit(ptx::smem_addr(&sh->drain));
        ptx::mbar_wait(ptx::smem_addr(&sh->drain), 0, ptx::globaltimer() + kWaitNs);
    } else if (warp == kScaleWarp && lane == 0) {
        // ------------------------------------------------ scale copies
        // Per k-block, once the stage has landed: the A scale chunk and the
        // B scale pair into the stage's tensor-memory slot, then an ordered
        // hand-off to the MMA thread (fence before the arrive here, fence
        // after the wait there), so the MMAs queue behind the copies without
        // waiting for them to complete.  The slot is free by then: the stage
        // was refilled only after the MMAs that last read the slot had
        // completed.
        const uint64_t sf_desc0 = ptx::desc_sf_32x16(ptx::smem_addr(ring) + sf_off);
        const uint32_t full0 = ptx::smem_addr(&sh->full[0]);
        const uint32_t ready0 = ptx::smem_addr(&sh->sf_ready[0]);
        const uint32_t tsf0 = tmem + kSfTmemCol;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int seq = 0; ok; ++seq) {
            const int w = get_item(sh, seq, p0.err);
            if (w < 0 || w >= n_work) break;
            const int kb_count = ka.p[(kMode == 3 ? (w < n_work1 ? 1 : 2) : kMode) - 1].K / kBlockK;
            for (int kb = 0; kb < kb_count; ++kb) {
                if (!wait_or_abort(full0 + 8 * stage, phase, sh, p0.err, 64 + stage)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t so = static_cast<uint64_t>(stage * (stride >> 4));
                const uint32_t tsf = tsf0 + 16 * stage;
                ptx::tc_cp_32x128b_warpx4(tsf + 0, sf_desc0 + so);
                ptx::tc_cp_32x128b_warpx4(tsf + 4, sf_desc0 + so + (kSfChunkBytes >> 4));
                ptx::tc_cp_32x128b_warpx4(tsf + 8, sf_desc0 + so + (2 * kSfChunkBytes >> 4));
                // ordered hand-off: the MMAs the MMA thread issues after it has
                // seen this arrive (and fenced) execute after these copies
                ptx::tc_fence_before();
                ptx::mbar_arrive(ready0 + 8 * stage);
                if (++stage == n_stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // its copies complete before tensor memory is freed
        ptx::tc_commit(ptx::smem_addr(&sh->sf_drain));
        ptx::mbar_wait(ptx::smem_addr(&sh->sf_drain), 0, ptx::globaltimer() + kWaitNs);
    } else if (warp >= 2 && warp < 2 + kEpiWarps) {
        // ------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int half = (warp - 2) / 4;                // which half of the accumulator columns
        const int m = quad * 32 + lane;                 // row of the tile = tensor-memory lane
        const uint32_t t_row = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        uint32_t acc_phase = 0;
        for (int seq = 0;; ++seq) {
            int w = 0;
            if (lane == 0) w = get_item(sh, seq, p0.err);
            w = __shfl_sync(0xffffffffu, w, 0);
            if (w < 0 || w >= n_work) break;
            int layer, b, j;
            decode_item<kMode>(ka, w, n_work1, layer, b, j);
            const int r = b * kBlockM + m;
            const int tok = __ldg(p0.row_token + r);
            const float wgt = __ldg(p0.row_weight + r);
            // tcgen05.ld is warp-collective: the whole warp goes on or stops together
            const bool go = !aborted(sh) && wait_or_abort(ptx::smem_addr(&sh->tmem_full), acc_phase, sh, p0.err, 48);
            if (!__all_sync(0xffffffffu, go)) break;
            ptx::tc_fence_after();
            uint32_t pk[64];
            if (kMode != 2 && layer == 1) {
                drain_accumulator<1>(t_row, half, pk, [&] {
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sh->tmem_empty));
                });
                if (tok >= 0) store_h_row<kClamp>(ka.p[0], b, j, r, quad, half, lane, wgt, pk);
                if (kMode == 3) {
                    // this warp's h codes and scale bytes are stored: count it in for block b
                    // (and the block in blocks_done when this warp completes it)
                    ptx::fence_proxy_async_global();
                    __threadfence();
                    __syncwarp();
                    if (lane == 0 &&
                        ptx::atom_add_acq_rel_gpu(ka.l1_done + b, 1) == kEpiWarps * ka.p[0].n_tiles - 1)
                        ptx::atom_add_acq_rel_gpu(ka.blocks_done, 1);  // acq_rel: a chain through every block
                }
            } else {
                drain_accumulator<2>(t_row, half, pk, [&] {
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&sh->tmem_empty));
                });
                const GemmParams& P = ka.p[1];
                const int col0 = j * kBN + 128 * half;  // H is a multiple of 128: a half is all in or all out
                const uint32_t routed = __ballot_sync(0xffffffffu, tok >= 0);
                if (col0 < P.H) {
                    if (!narrow && routed == 0xffffffffu)
                        store_out_rows(&ka.maps[1].out, smem + kOutStageOff + (warp - 2) * kOutStageBytes, col0,
                                       b * kBlockM + quad * 32, lane, pk);
                    else if (tok >= 0)
                        store_out_rows_direct(P, r, col0, pk);
                }
            }
            acc_phase ^= 1;
        }
        // this warp's tensor stores complete before the CTA exits
        if (kMode != 1 && lane == 0) ptx::bulk_wait_all();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
#else
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(ka.p[0].err, kDevErrTimeout);
#endif
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda directly.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once; concurrent first calls from several host threads look it up
// alike and store the same pointer.
EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> cached{nullptr};
    EncodeTiledFn fn = cached.load(std::memory_order_acquire);
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<EncodeTiledFn>(p);
            cached.store(fn, std::memory_order_release);
        }
    }
    return fn;
}

// 2-D K-major tile map: rows x K, box box_rows x 128 K elements, 128-byte swizzle.
bool make_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t k_elems, uint64_t rows,
              uint64_t row_bytes, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {k_elems, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D FP4 map [planes][rows][K] (K-major), box 128 K x 128 rows x 2 planes:
// one request brings the same 128 rows of two consecutive planes.
bool make_map_3d_fp4(CUtensorMap* map, const void* base, uint64_t k_elems, uint64_t rows, uint64_t planes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {k_elems, rows, planes};
    cuuint64_t strides[2] = {k_elems / 2, rows * (k_elems / 2)};
    cuuint32_t box[3] = {128, 128, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-major E4M3 rows [rows][cols] for tile::gather4 loads: box 128 columns x
// 1 row, 128-byte swizzle (four gathered rows land as rows of the K-major,
// 128-byte-swizzled A tile that the MMA reads).
bool make_gather_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows][cols] output map for tensor stores: box 32 columns x 32 rows,
// 64-byte swizzle (the staging layout of store_out_rows).
bool make_out_map(CUtensorMap* map, void* base, uint64_t cols, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_layer1_operand_maps(CUtensorMap* a_map, const void* a, CUtensorMap* b_map, const void* b, uint64_t K,
                              uint64_t rows) {
    return make_map(a_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, K, rows, K, kBlockM) &&
           make_map_3d_fp4(b_map, b, K, rows, 2);
}

namespace {

// Opt a kernel into its dynamic shared memory once per device (a repeated
// call from another host thread sets the same attribute again, harmlessly).
template <typename Kernel>
cudaError_t smem_attr_once(Kernel kernel, int slot, int bytes) {
    static std::atomic<int> done[9][64] = {};
    int dev = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st != cudaSuccess) return st;
    if (dev < 64 && done[slot][dev].load(std::memory_order_acquire)) return cudaSuccess;
    st = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (st == cudaSuccess && dev < 64) done[slot][dev].store(1, std::memory_order_release);
    return st;
}

}  // namespace

namespace {

// The maps and parameters of one layer (index layer-1 of the launch's args).
bool fill_layer(int layer, const Layout& L, uint8_t* ws, const GemmLaunch& g, KernelArgs* ka) {
    GemmParams& p = ka->p[layer - 1];
    p = GemmParams{};
    p.n_blocks = reinterpret_cast<const int*>(ws + L.n_blocks);
    p.block_expert = reinterpret_cast<const int*>(ws + L.block_expert);
    p.row_token = reinterpret_cast<const int*>(ws + L.row_token);
    p.row_weight = reinterpret_cast<const float*>(ws + L.row_weight);
    p.sfb = static_cast<const uint8_t*>(g.w_sf);
    p.K = g.K;
    p.N = g.N;
    p.E = L.E;
    p.I = L.I;
    p.H = L.H;
    p.err = reinterpret_cast<int*>(ws + L.err);
    p.block_rows = reinterpret_cast<const int*>(ws + L.block_rows);
    p.max_count = reinterpret_cast<const int*>(ws + L.max_count);
    p.clamp = g.clamp > 0.0f ? g.clamp : std::numeric_limits<float>::infinity();  // no clamp
    p.scale_rule = g.scale_rule;
    p.fast_math = g.fast_math;
    Maps& maps = ka->maps[layer - 1];
    bool ok = true;
    maps.gather = CUtensorMap{};  // used by layer 1 with gathered A rows only
    if (layer == 1) {
        p.a_rows = ws + L.pool_q;
        p.sfa = ws + L.pool_sf;
        p.out_q = ws + L.h_q;
        p.out_sf = ws + L.h_sf;
        p.n_tiles = L.I / 128;
        p.a_gather = g.a_gather ? 1 : 0;
        if (g.a_gather && !make_gather_map(&maps.gather, ws + L.x_q, L.H, L.T)) return false;
        maps.out = CUtensorMap{};  // unused by layer 1
        // W1 as [2E expert-halves][I rows][H]: 128 gate rows + the matching 128 up rows
        ok = make_map_3d_fp4(&ka->tmap_b[0], g.w_q, g.K, g.N / 2, 2 * static_cast<uint64_t>(g.E));
    } else {
        p.a_rows = ws + L.h_q;
        p.sfa = ws + L.h_sf;
        p.out_bf16 = reinterpret_cast<uint16_t*>(ws + L.l2_out);
        p.n_tiles = (L.H + kBN - 1) / kBN;
        ok = make_out_map(&maps.out, p.out_bf16, L.H, L.p_cap) &&
             make_map(&ka->tmap_b[1], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, g.w_q, g.K,
                      static_cast<uint64_t>(g.E) * g.N, g.K / 2, kBN);
    }
    for (int i = 0; i < kABoxLevels; ++i)
        ok = ok && make_map(&maps.box[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a_rows, g.K, L.p_cap, g.K, 16u << i);
    return ok;
}

template <int kMode, bool kClamp, bool kGather>
cudaError_t launch_mode(const KernelArgs& ka, int slot, int num_sms, cudaStream_t s) {
    cudaError_t st = smem_attr_once(expert_gemm_kernel<kMode, kClamp, kGather>, slot, kSmemBytes);
    if (st != cudaSuccess) return st;
    if (kMode != 3 && (st = cudaMemsetAsync(ka.work_ctr, 0, sizeof(int), s)) != cudaSuccess) return st;
    expert_gemm_kernel<kMode, kClamp, kGather><<<num_sms, kThreads, kSmemBytes, s>>>(ka);
    return cudaGetLastError();
}

// Layer 1 alone (kMode 1) or fused (kMode 3): the instantiation for the clamp
// and the A operand's source.
template <int kMode>
cudaError_t launch_layer1_mode(const KernelArgs& ka, int slot0, int num_sms, cudaStream_t s) {
    const bool clamp = ka.p[0].clamp != std::numeric_limits<float>::infinity();
    if (ka.p[0].a_gather)
        return clamp ? launch_mode<kMode, true, true>(ka, slot0 + 3, num_sms, s)
                     : launch_mode<kMode, false, true>(ka, slot0 + 2, num_sms, s);
    return clamp ? launch_mode<kMode, true, false>(ka, slot0 + 1, num_sms, s)
                 : launch_mode<kMode, false, false>(ka, slot0, num_sms, s);
}

}  // namespace

cudaError_t launch_expert_gemm(int layer, const Layout& L, uint8_t* ws, const GemmLaunch& g, int num_sms,
                               cudaStream_t s) {
    if (L.T == 0) return cudaSuccess;
    KernelArgs ka{};
    if (!fill_layer(layer, L, ws, g, &ka)) return cudaErrorInvalidValue;
    ka.work_ctr = reinterpret_cast<int*>(ws + L.sched) + (layer - 1);
    if (layer == 1) return launch_layer1_mode<1>(ka, 0, num_sms, s);
    return launch_mode<2, false, false>(ka, 4, num_sms, s);
}

cudaError_t launch_expert_fused(const Layout& L, uint8_t* ws, const GemmLaunch& g1, const GemmLaunch& g2, int num_sms,
                                cudaStream_t s, bool publish) {
    if (L.T == 0) return cudaSuccess;
    KernelArgs ka{};
    if (!fill_layer(1, L, ws, g1, &ka) || !fill_layer(2, L, ws, g2, &ka)) return cudaErrorInvalidValue;
    // The work counter and the readiness counters start at zero for every
    // launch.  (Self-test only: with publish == false the readiness counters
    // start at 0x80808080, a large negative count that the layer-1 tiles can
    // never raise to the target, so every layer-2 tile's bounded wait runs out.)
    ka.work_ctr = reinterpret_cast<int*>(ws + L.sched) + 2;
    ka.blocks_done = reinterpret_cast<int*>(ws + L.sched) + 3;
    ka.l1_done = reinterpret_cast<int*>(ws + L.sched) + kSchedWords;
    const size_t blocks = static_cast<size_t>(L.p_cap / kBlockM);
    cudaError_t st = cudaMemsetAsync(ws + L.sched, 0, sizeof(int) * (kSchedWords + blocks), s);
    if (st != cudaSuccess) return st;
    if (!publish && (st = cudaMemsetAsync(ka.l1_done, 0x80, sizeof(int) * blocks, s)) != cudaSuccess) return st;
    return launch_layer1_mode<3>(ka, 5, num_sms, s);
}

}  // namespace moe
