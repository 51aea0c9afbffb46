/*
 * moe.h -- C ABI of the single-GPU fused Mixture-of-Experts layer forward
 * (GB300, sm_103a).
 *
 * What the layer computes (the DeepGEMM "Mega MoE" forward as analysed in the
 * pages "DeepEP -> Mega MoE: the boundary evolution of communication and
 * compute" and "Dispatch/Combine in the DeepGEMM Mega MoE kernel"), with every
 * expert local to one GPU:
 *
 *   dispatch  per-expert counts of the top-k entries, exclusive prefix sums,
 *             a deterministic slot per entry in an expert-major pool whose
 *             expert segments are padded to MOE_BLOCK_M rows, then a gather of
 *             token-major bf16 x into that pool with MXFP8 quantisation
 *             (E4M3 codes, one UE8M0 scale per 32 hidden elements);
 *   expert    L1 = pool x W1^T (FP8 x FP4 block-scaled, fp32 accumulate),
 *             gate/up rounded to bf16, h = silu(gate) * up * topk_weight,
 *             requantised to MXFP8 along I; L2 = h x W2^T rounded to bf16;
 *   combine   y[t] = bf16( fp32 sum over ascending j of the valid entries'
 *             L2 rows ); 0 for tokens with no valid entry.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, except
 *     where a comment says "host".  The library allocates no device memory;
 *     every scratch buffer lives in the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).  All
 *     work is enqueued on it; no call synchronises the host except
 *     moe_plan_check().
 *   - Every call returns a moe_status (0 = MOE_OK).  Nothing is thrown across
 *     the ABI and no kernel traps: errors found on the device (bad expert id,
 *     a bounded wait that expired) are recorded in the workspace and reported
 *     by moe_plan_check().
 *   - Shapes: x, y are [T, H] bf16 row-major; topk_idx [T, k] int64 with -1
 *     meaning "not routed here"; topk_w [T, k] float32.  Requirements:
 *     H % 128 == 0, I % 128 == 0, 1 <= k <= 32, 1 <= E <= 1024, T >= 0.
 */
#ifndef MOE_GB300_MOE_H_
#define MOE_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape, plan mismatch */
    MOE_ERR_UNSUPPORTED = 2,   /* shape outside the requirements above, or not an sm_103 device */
    MOE_ERR_WORKSPACE = 3,     /* workspace smaller than moe_plan_workspace_bytes() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    MOE_ERR_BAD_EXPERT_ID = 5, /* device saw topk_idx outside [-1, E); those entries were skipped */
    MOE_ERR_TIMEOUT = 6,       /* a bounded device-side wait expired; outputs are invalid */
    MOE_ERR_NO_KERNEL = 7,     /* the library holds no code for this device */
    MOE_ERR_TOO_LARGE = 8,     /* sizes exceed the fixed scratch of moe_expert_offsets_static() */
    MOE_ERR_DEBUG_BOUNDS = 9   /* debug build only (-DMOE_DEBUG): a device bounds check on a plan table
                                  fired and the access was skipped; outputs are invalid */
} moe_status;

/* Rows of one MMA tile; every expert's pool segment is padded to a whole
 * number of such row blocks (Dispatch/Combine page, Appendix A.2, where the
 * block is BLOCK_M). */
#define MOE_BLOCK_M 128

/* Plan: caller-owned opaque storage, filled by moe_plan().  It records the
 * shapes and the workspace pointer; all device state lives in the
 * workspace.  It may be copied by value. */
typedef struct moe_plan_t {
    uint64_t opaque[24];
} moe_plan_t;

/* One MXFP4 weight tensor [E, N, K].
 *   q       e2m1 codes, two per byte, the even K index in the low nibble,
 *           bit 3 of a nibble = sign; [E][N][K/2] bytes, 32-byte aligned.
 *   sf_mma  UE8M0 scales (biased exponents, one per 32 along K) in the
 *           tensor-core layout written by moe_prepare_weight_scales()
 *           (MOE_SF_PAIRS_HALVES for W1, MOE_SF_PAIRS_ADJACENT for W2).
 * W1 has N = 2I (gate rows 0..I-1, then up rows I..2I-1), K = H.
 * W2 has N = H, K = I. */
typedef struct moe_weights_t {
    const void* q;
    const void* sf_mma;
    int32_t E, N, K;
} moe_weights_t;

/* Bytes of device workspace that moe_plan() needs for these shapes: routing
 * tables, the expert-major MXFP8 pool, the requantised L1 output and the L2
 * output.  Returns 0 if the shapes are unsupported.  Host-only, no CUDA. */
size_t moe_plan_workspace_bytes(int T, int k, int E, int H, int I);

/* Bytes of the tensor-core scale layout for an [E, N, K] weight:
 * E * ceil(N/256) * (K/128) * 1024.  0 if N % 128 or K % 128 is nonzero.
 * Host-only. */
size_t moe_weight_scales_bytes(int E, int N, int K);

/* How moe_prepare_weight_scales pairs 128-row chunks: the expert GEMMs read
 * one pair per 256-row weight tile, so both chunks of a pair, for every 128-K
 * step, are stored side by side. */
enum {
    MOE_SF_PAIRS_ADJACENT = 0, /* pair p = rows [256p, 256p+256) (W2) */
    MOE_SF_PAIRS_HALVES = 1    /* pair p = rows [128p, +128) and [N/2 + 128p, +128) (W1: gate | up) */
};

/* One-time relayout of weight scales (not part of the per-batch path; the
 * pages' "transformed_l1_weights" plays the same role).
 *   sf       UE8M0 bytes [E][N][K/32] (device, row-major)
 *   pairing  MOE_SF_PAIRS_HALVES for W1, MOE_SF_PAIRS_ADJACENT for W2
 *   sf_mma   output, moe_weight_scales_bytes(E,N,K) bytes (device); layout
 *            [E][pair][K/128][2][512], each 512-byte chunk holding 128 rows x
 *            4 scales at byte 16*(row%32) + 4*(row/32) + (k/32)%4
 * Errors: MOE_ERR_INVALID_ARG (null pointers, small buffer, bad pairing, N/2
 * not a multiple of 128 for MOE_SF_PAIRS_HALVES), MOE_ERR_UNSUPPORTED (N or K
 * not multiples of 128), MOE_ERR_CUDA. */
int moe_prepare_weight_scales(const void* sf, int E, int N, int K, int pairing, void* sf_mma,
                              size_t sf_mma_bytes, void* stream);

/* Dispatch plan (DeepEP -> Mega MoE page, dispatch.cuh snippet: expert count,
 * prefix sum, slot assignment; Dispatch/Combine page section 3.1).
 * Computes per-chunk expert histograms (2048 entries a chunk; warp-aggregated
 * shared-memory atomics), prefix sums over chunks and experts (offsets,
 * row-block-padded offsets, the tile table), and a stable slot per entry:
 * slot = padded offset of its expert + number of earlier (smaller flat index
 * t*k+j) entries of the same expert.  Enqueues a memset of the workspace's
 * error region and ONE kernel for E <= 256 (or E > 256 with T*k <= 2048),
 * otherwise three kernels; none of them needs its CTAs to be co-resident.  Entries with id -1 are skipped; ids
 * outside [-1, E) are skipped and flagged (MOE_ERR_BAD_EXPERT_ID, via
 * moe_plan_check).
 *   plan       out (host): filled on success
 *   topk_idx   [T, k] int64, device; read only by this call
 *   topk_w     [T, k] float32, device; copied into the workspace
 *   workspace  >= moe_plan_workspace_bytes(T,k,E,H,I) bytes, device,
 *              256-byte aligned; owned by the caller, must stay alive and
 *              untouched while the plan is used
 * No host synchronisation.  T == 0 is a valid empty plan. */
int moe_plan(moe_plan_t* plan, const int64_t* topk_idx, const float* topk_w, int T, int k, int E,
             int H, int I, void* workspace, size_t workspace_bytes, void* stream);

/* Layer options (the activation_clamp and fast_math arguments of the API on
 * the Normal-vs-Low-Latency page; the pages define neither, so the readings
 * are stated here).  Pass NULL for the defaults {0, MOE_SCALE_CEIL, 1, MOE_A_POOL}.
 *   activation_clamp  > 0: the bf16-rounded gate and up values are limited to
 *                     [-c, c] before SwiGLU; 0 or +inf: no clamp (NaN and
 *                     negative values are MOE_ERR_INVALID_ARG)
 *   scale_rule        UE8M0 rule of the activation scales (x in dispatch, h in
 *                     the L1 epilogue): MOE_SCALE_CEIL = the smallest 2^e with
 *                     amax <= 448 * 2^e; MOE_SCALE_OCP_FLOOR = OCP MX v1.0,
 *                     2^(floor(log2 amax) - 8), values beyond 448 saturate
 *   fast_math         1: SwiGLU with __expf and an approximate divide, every
 *                     value recomputed exactly where that could change an E4M3
 *                     code or a scale (so the result equals the exact
 *                     formula's); 0: every value by the exact formula.  Both
 *                     give the same bytes; 0 is slower. */
enum {
    MOE_SCALE_CEIL = 0,
    MOE_SCALE_OCP_FLOOR = 1
};
/* Where layer 1 takes its FP8 operand rows from (moe_options_t.a_operand):
 *   MOE_A_POOL    moe_dispatch writes every valid entry's row into the
 *                 expert-major pool (k copies of a token); layer 1 loads
 *                 128-row boxes of the pool
 *   MOE_A_GATHER  moe_dispatch writes each token's MXFP8 row once,
 *                 token-major, and the pool's scales only; layer 1 gathers
 *                 the rows of each pool row block by token index with TMA
 *                 tile::gather4 loads (the "skip the pool" collapse of the
 *                 Dispatch/Combine page, section 7.2).  Same results, bit
 *                 for bit; fewer bytes written by dispatch, more TMA requests
 *                 per layer-1 stage.
 * moe_dispatch and the layer-1 call (moe_expert_l1 / moe_expert_fused) of one
 * forward must be given the same a_operand; moe_forward passes one options
 * value to both. */
enum {
    MOE_A_POOL = 0,
    MOE_A_GATHER = 1
};
typedef struct moe_options_t {
    float activation_clamp;
    int32_t scale_rule;
    int32_t fast_math;
    int32_t a_operand;   /* MOE_A_POOL (default) or MOE_A_GATHER */
    int32_t reserved[4]; /* must be zero */
} moe_options_t;

/* Dispatch gather (Dispatch/Combine page section 3.1, token pull into the
 * expert pool; recipe (1,1,32) of the Normal-vs-Low-Latency page section 2):
 * for each valid entry, pool row slot = MXFP8(x[t]) with opts->scale_rule.
 * x [T, H] bf16; opts may be NULL. */
int moe_dispatch(const moe_plan_t* plan, const void* x, const moe_options_t* opts, void* stream);

/* Expert L1 (DeepEP -> Mega MoE page, sm100_fp8_fp4_mega_moe.cuh snippets:
 * block-scaled FP8 x FP4 MMA, SwiGLU, amax, FP8 requant): for every pool row
 * block, tcgen05 block-scaled MMA over H, then the epilogue
 * h = silu(bf16(gate)) * bf16(up) * topk_weight, requantised to MXFP8
 * (gate and up clamped, the scale rule and fast_math as in moe_options_t;
 * opts may be NULL).
 * W1: E, N = 2I, K = H must match the plan. */
int moe_expert_l1(const moe_plan_t* plan, const moe_weights_t* W1, const moe_options_t* opts, void* stream);

/* Expert L2: pool rows of h x W2^T, fp32 accumulate, rounded to bf16 rows in
 * pool order (Dispatch/Combine page section 5.1, the unweighted bf16
 * combine buffer).  W2: E, N = H, K = I must match the plan. */
int moe_expert_l2(const moe_plan_t* plan, const moe_weights_t* W2, void* stream);

/* Both expert layers in ONE persistent launch (the single-kernel design of
 * the pages: DeepEP -> Mega MoE page, the sm100_fp8_fp4_mega_moe.cuh
 * compute pipeline and its on-chip L1 -> L2 hand-off; Normal-vs-Low-Latency
 * page sections 6.2-6.3, the scheduler's block phases and the wait of an L2
 * block on its L1 arrival count).  Computes exactly what moe_expert_l1 +
 * moe_expert_l2 compute (the same bytes of h and of the L2 rows).  Work items
 * are all layer-1 tiles (pool row block x 128 intermediate columns), then all
 * layer-2 tiles (row block x 256 output columns), spread over one CTA per
 * SM; a layer-2 tile of row block b starts once every layer-1 tile of b has
 * stored its h rows (a per-block counter in the workspace, zeroed by this
 * call).  So the last layer-1 wave is filled with layer-2 work and the
 * second launch disappears.  The wait is bounded: if a block is not ready
 * within 1 s of global time the launch records MOE_ERR_TIMEOUT (error word 1
 * = 81, see MOE_EXPORT_ERROR) and its CTAs exit; the wait needs every CTA of
 * the launch resident at once (one per SM), so it may time out if other work
 * holds SMs for that long.  W1, W2 and opts as for moe_expert_l1 /
 * moe_expert_l2. */
int moe_expert_fused(const moe_plan_t* plan, const moe_weights_t* W1, const moe_weights_t* W2,
                     const moe_options_t* opts, void* stream);

/* Combine (DeepEP -> Mega MoE page, combine_utils.cuh snippet; Dispatch/
 * Combine page section 5.1): y[t] = bf16(fp32 sum over ascending j of the
 * valid entries' L2 rows), y[t] = 0 if token t has no valid entry.
 * y [T, H] bf16. */
int moe_combine(const moe_plan_t* plan, void* y, void* stream);

/* The whole layer after moe_plan(): moe_dispatch + moe_expert_fused +
 * moe_combine, in stream order; opts may be NULL. */
int moe_forward(const void* x, const moe_weights_t* W1, const moe_weights_t* W2,
                const moe_plan_t* plan, void* y, const moe_options_t* opts, void* stream);

/* Synchronises `stream`, then returns the first device-side error recorded
 * in the plan's workspace (MOE_ERR_DEBUG_BOUNDS, MOE_ERR_TIMEOUT,
 * MOE_ERR_BAD_EXPERT_ID, in that order of precedence) or
 * MOE_OK.  The record is cleared by the next moe_plan() on that workspace. */
int moe_plan_check(const moe_plan_t* plan, void* stream);

/* Where an internal array of the plan lives inside the workspace, for tests
 * and tools: byte offset and size.  `what` is one of MOE_EXPORT_*. */
enum {
    MOE_EXPORT_COUNT = 0,        /* int32 [E] */
    MOE_EXPORT_OFFSETS = 1,      /* int32 [E+1] exclusive scan of counts */
    MOE_EXPORT_POFFSETS = 2,     /* int32 [E+1] exclusive scan of counts padded to MOE_BLOCK_M */
    MOE_EXPORT_SLOT_OF = 3,      /* int32 [T*k] pool row of entry (t,j), -1 if skipped */
    MOE_EXPORT_ROW_TOKEN = 4,    /* int32 [P_cap] token of a pool row, -1 on padding */
    MOE_EXPORT_ROW_TOPK = 5,     /* int32 [P_cap] j of a pool row, -1 on padding */
    MOE_EXPORT_ROW_WEIGHT = 6,   /* float [P_cap] topk weight of a pool row */
    MOE_EXPORT_BLOCK_EXPERT = 7, /* int32 [P_cap/128] expert of each pool row block */
    MOE_EXPORT_NUM_BLOCKS = 8,   /* int32 [1] number of pool row blocks in use */
    MOE_EXPORT_POOL_Q = 9,       /* uint8 [P_cap, H] E4M3 pool */
    MOE_EXPORT_POOL_SF = 10,     /* uint8 [P_cap/128][H/128][512] UE8M0, tensor-core layout */
    MOE_EXPORT_H_Q = 11,         /* uint8 [P_cap, I] E4M3 requantised L1 output */
    MOE_EXPORT_H_SF = 12,        /* uint8 [P_cap/128][I/128][512] UE8M0, tensor-core layout */
    MOE_EXPORT_L2_OUT = 13,      /* bf16 [P_cap, H] L2 output rows in pool order */
    MOE_EXPORT_ERROR = 14,       /* int32 [2] device error record: bits, then 1 + where a wait expired
                                  * (0-15 producer on a stage, 16 MMA on the accumulator, 32-47 MMA on a
                                  * stage, 48 epilogue, 64-79 scale copies, 80 a fused layer-2 tile on
                                  * its row block's layer-1 tiles, 96 producer on its work-item queue,
                                  * 97 a warp waiting for its next work item) */
    MOE_EXPORT_POOL_ROWS = 15,   /* (size only) P_cap, the pool row capacity, in the size field */
    MOE_EXPORT_MAX_COUNT = 16,   /* int32 [1] largest expert count (0 when nothing is routed) */
    MOE_EXPORT_X_Q = 17          /* uint8 [T, H] token-major E4M3 x (written by dispatch with MOE_A_GATHER) */
};
int moe_plan_export(const moe_plan_t* plan, int what, size_t* offset, size_t* bytes);

/* Expert counts and offsets for callers that cannot allocate device memory.
 * The analysed pages have no counterpart of this entry point.
 *
 * Some callers cannot call cudaMalloc at all: a plugin that runs inside a
 * host framework which owns every byte of device memory, or a serving loop
 * whose memory budget is frozen after start-up (an allocation there may also
 * synchronise the device).  Such callers can still pass their inputs and
 * outputs, but not a workspace.  This entry point runs the same counting and
 * prefix-sum kernels as moe_plan(), with their scratch (per-chunk
 * histograms, per-chunk bases, the row-block table) in a fixed array inside
 * the library: about 280 KB of device memory that every GPU which loads the
 * library keeps until the process exits.  Nothing is allocated per call.
 *   topk_idx        [T, k] int64 (device); -1 = not routed; other ids outside
 *                   [-1, E) are skipped (not reported here)
 *   count           out [E] int32 (device): entries per expert
 *   offsets         out [E+1] int32 (device): exclusive scan of count
 *   padded_offsets  out [E+1] int32 (device): exclusive scan of count rounded
 *                   up to MOE_BLOCK_M
 * Limits: T*k <= 262144, E <= 1024, ceil(T*k / 2048) * E <= 32768, 1 <= k <= 32;
 * larger sizes return MOE_ERR_TOO_LARGE before anything is enqueued.
 * The first call on a device looks up the array's device address (a CUDA
 * runtime query, no allocation) and keeps it for the life of the process;
 * make that first call before any stream capture, and do not call this entry
 * point on a device again after cudaDeviceReset() on it (the kept address
 * would belong to the destroyed context).  Concurrent first calls from
 * several host threads are safe.  All calls share the one array and it keeps
 * the last call's contents, so calls whose kernels overlap on the GPU
 * (different streams without ordering) race and give wrong results; order
 * them on one stream. */
int moe_expert_offsets_static(const int64_t* topk_idx, int T, int k, int E, int32_t* count, int32_t* offsets,
                              int32_t* padded_offsets, void* stream);

/* Self-test of the device-side bounded wait that every pipeline barrier of
 * the library uses (no counterpart on the pages; it exists so that failure
 * detection can be exercised on a GPU without a fault).  One CTA waits on an
 * mbarrier that `arrive` = 1 completes after about 20 us and `arrive` = 0
 * leaves incomplete, giving up after timeout_ns of global time.
 *   out  device int32[2], written by the kernel: {MOE_OK or MOE_ERR_TIMEOUT,
 *        elapsed microseconds}
 * Errors: MOE_ERR_INVALID_ARG (null out, timeout_ns of 0 or above 2 s),
 * MOE_ERR_UNSUPPORTED (not an sm_103 device), MOE_ERR_CUDA.  The kernel never
 * traps; after a time-out the context stays usable. */
int moe_selftest_bounded_wait(int arrive, uint64_t timeout_ns, int32_t* out, void* stream);

/* Tensor-pipe ceiling of the block-scaled MMA that the expert GEMMs issue
 * (no counterpart on the pages; a calibration for the roofline of the GEMMs).
 * Launches one CTA per SM; in each, one thread issues kblocks x 4
 * tcgen05.mma.kind::mxf8f6f4.block_scale instructions (M = 128, N = 256,
 * K = 32: E4M3 x E2M1 with UE8M0 scales, the GEMMs' instruction) back to back
 * on fixed shared-memory operands, then waits for them.  No global memory is
 * touched except `status`.  The caller times the launch (e.g. CUDA events on
 * `stream`): the work is ctas * kblocks * 2*128*256*128 FLOP.
 *   kblocks  1 .. 2^20 (about 260 ns each per SM at the full tensor rate)
 *   status   device int32, written: MOE_OK, or MOE_ERR_TIMEOUT if the MMAs did
 *            not complete within 2 s of global time
 *   ctas     out (host): the number of CTAs launched (the SM count)
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED (not sm_103), MOE_ERR_CUDA. */
int moe_selftest_mma_rate(int kblocks, int32_t* status, int* ctas, void* stream);

/* Operand-stream ceiling of the layer-1 GEMM tile (no counterpart on the
 * pages; a second calibration for the roofline of the GEMMs).  The MMAs of
 * moe_selftest_mma_rate, fed as the expert kernel feeds them: one CTA per SM,
 * a 4-stage ring of 50 KB stages filled by TMA (a 128-row E4M3 box of A, the
 * 256-row two-plane E2M1 box of B expanded to one byte per element, the A
 * scale chunk and the B scale pair), a thread copying each stage's scales
 * into tensor memory and the MMA thread; no epilogue.  CTA c reads row block
 * (c / 16) % 16 of A and weight rows 128 * (c % 16) .. +128 of both planes of
 * B, cycling through the 56 k-blocks of K = 7168.  The values only need to be
 * finite codes; the product is discarded.
 *   a        device E4M3 codes [2048][7168] (row-major, 16-byte aligned)
 *   b        device E2M1 codes [2][2048][7168/2] (two per byte, 16-byte aligned)
 *   sfa      device UE8M0 scale chunks [16][56][512] (tensor-core layout)
 *   sfb      device UE8M0 scale chunk pairs [16][56][1024]
 *   kblocks  k-blocks per CTA, 1 .. 2^20; the work is ctas * kblocks *
 *            2*128*256*128 FLOP
 *   status   device int32, written: MOE_OK, or MOE_ERR_TIMEOUT if a stage
 *            wait gave up after 2 s of global time (the kernel then returns)
 *   ctas     out (host): the number of CTAs launched (the SM count)
 * Errors: MOE_ERR_INVALID_ARG (null or unaligned pointers, kblocks out of
 * range), MOE_ERR_UNSUPPORTED (not sm_103), MOE_ERR_CUDA.  The caller owns
 * every buffer and times the launch on `stream`. */
int moe_selftest_stream_rate(const void* a, const void* b, const void* sfa, const void* sfb, int kblocks,
                             int32_t* status, int* ctas, void* stream);

/* Failure-detection self-test of moe_expert_fused (no counterpart on the
 * pages): runs the fused launch with its readiness counters set so that no
 * row block ever becomes ready, so every layer-2 tile's bounded wait expires
 * after 1 s.  The launch then records MOE_ERR_TIMEOUT in the plan's
 * workspace (read it with moe_plan_check) and exits without a fault or a
 * trap; the context stays usable.  Layer-1 outputs are written as usual,
 * layer-2 outputs are invalid.  Arguments as for moe_expert_fused. */
int moe_selftest_fused_wait(const moe_plan_t* plan, const moe_weights_t* W1, const moe_weights_t* W2, void* stream);

/* Static text for a status code. */
const char* moe_error_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H_ */
