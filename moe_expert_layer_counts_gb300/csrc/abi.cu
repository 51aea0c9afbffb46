// abi.cu -- the extern "C" boundary of libmoe: argument checks, the
// workspace layout, the one-time weight-scale relayout and the per-stage
// launches.  No entry point allocates device memory; none synchronises the
// host except moe_plan_check().
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cmath>
#include <cstring>

#include "internal.h"

namespace moe {
namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-device facts, filled on first use.
struct DeviceInfo {
    int ready;
    int sms;
    int supported;
};
DeviceInfo g_dev[64];

int device_info(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        d.sms = n;
        d.supported = (major == 10 && minor == 3);
        d.ready = 1;
    }
    if (!d.supported) return MOE_ERR_UNSUPPORTED;
    if (sms) *sms = d.sms;
    return MOE_OK;
}

// Scale relayout: canonical [E][N][K/32] -> [E][pair][K/128][2][512]; within
// a 512-byte chunk (128 rows x 4 scales) byte 16*(n%32) + 4*((n%128)/32) +
// (k/32)%4.  Pairs: adjacent 128-row chunks (2p, 2p+1), or the chunk p of
// each half of N (gate | up).  The second chunk of a last, odd adjacent pair
// stays zero.
__global__ void prepare_sf_kernel(const uint8_t* __restrict__ sf, int64_t total, int N, int K, int halves,
                                  uint8_t* __restrict__ out) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int kq_n = K / kSfVec;
    const int64_t row = i / kq_n;  // e*N + n
    const int kq = static_cast<int>(i % kq_n);
    const int64_t e = row / N;
    const int n = static_cast<int>(row % N);
    const int pairs = (N + 255) / 256;
    int pair, half, m;
    if (halves) {
        half = n >= N / 2;
        const int nh = n - half * (N / 2);
        pair = nh / 128;
        m = nh % 128;
    } else {
        pair = n / 256;
        half = (n / 128) % 2;
        m = n % 128;
    }
    const int kb = kq / 4, sub = kq % 4;
    const size_t chunk = ((static_cast<size_t>(e) * pairs + pair) * (K / 128) + kb) * 2 + half;
    out[chunk * kSfChunkBytes + 16 * (m % 32) + 4 * (m / 32) + sub] = sf[i];
}

const PlanState* plan_state(const moe_plan_t* plan) {
    if (!plan) return nullptr;
    const PlanState* ps = reinterpret_cast<const PlanState*>(plan);
    return ps->magic == kPlanMagic ? ps : nullptr;
}

int check_weights(const moe_weights_t* w, int E, int N, int K) {
    if (!w || !w->q || !w->sf_mma) return MOE_ERR_INVALID_ARG;
    if (w->E != E || w->N != N || w->K != K) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(w->q) & 31u) || (reinterpret_cast<uintptr_t>(w->sf_mma) & 15u))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Options with defaults filled in; false if a field is out of range.
bool read_options(const moe_options_t* opts, moe_options_t* o) {
    *o = moe_options_t{0.0f, MOE_SCALE_CEIL, 1, MOE_A_POOL, {0, 0, 0, 0}};
    if (!opts) return true;
    if (std::isnan(opts->activation_clamp) || opts->activation_clamp < 0.0f) return false;
    if (opts->scale_rule != MOE_SCALE_CEIL && opts->scale_rule != MOE_SCALE_OCP_FLOOR) return false;
    if (opts->fast_math != 0 && opts->fast_math != 1) return false;
    if (opts->a_operand != MOE_A_POOL && opts->a_operand != MOE_A_GATHER) return false;
    for (int r : opts->reserved)
        if (r != 0) return false;
    *o = *opts;
    if (std::isinf(o->activation_clamp)) o->activation_clamp = 0.0f;
    return true;
}

}  // namespace

bool make_layout(int T, int k, int E, int H, int I, Layout* L) {
    if (T < 0 || k < 1 || k > kMaxTopk || E < 1 || E > kMaxExperts) return false;
    if (H < 128 || I < 128 || H % 128 || I % 128) return false;
    const int64_t n = static_cast<int64_t>(T) * k;
    if (n > (int64_t(1) << 28)) return false;
    L->T = T;
    L->k = k;
    L->E = E;
    L->H = H;
    L->I = I;
    L->chunks = static_cast<int>((n + kRouteChunk - 1) / kRouteChunk);
    int64_t cap = n + std::min<int64_t>(E, n) * (kBlockM - 1);
    cap = std::max<int64_t>(kBlockM, (cap + kBlockM - 1) / kBlockM * kBlockM);
    L->p_cap = cap;
    const int chunks = std::max(L->chunks, 1);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align_up(o + bytes, 1024);
        return at;
    };
    L->err = take(kErrWords * sizeof(int));
    L->n_blocks = take(sizeof(int));
    L->max_count = take(sizeof(int));  // largest expert count (selects the GEMM's operand ring)
    L->count = take(sizeof(int) * E);
    L->off = take(sizeof(int) * (E + 1));
    L->poff = take(sizeof(int) * (E + 1));
    L->hist = take(sizeof(int) * static_cast<size_t>(chunks) * E);
    L->chunk_base = take(sizeof(int) * static_cast<size_t>(chunks) * E);
    L->block_expert = take(sizeof(int) * static_cast<size_t>(cap / kBlockM));
    L->block_rows = take(sizeof(int) * static_cast<size_t>(cap / kBlockM));
    L->slot_of = take(sizeof(int) * static_cast<size_t>(std::max<int64_t>(n, 1)));
    L->row_token = take(sizeof(int) * static_cast<size_t>(cap));
    L->row_topk = take(sizeof(int) * static_cast<size_t>(cap));
    L->row_weight = take(sizeof(float) * static_cast<size_t>(cap));
    L->pool_q = take(static_cast<size_t>(cap) * H);
    L->pool_sf = take(static_cast<size_t>(cap / kBlockM) * (H / 128) * kSfChunkBytes);
    L->h_q = take(static_cast<size_t>(cap) * I);
    L->h_sf = take(static_cast<size_t>(cap / kBlockM) * (I / 128) * kSfChunkBytes);
    L->l2_out = take(static_cast<size_t>(cap) * H * 2);
    L->x_q = take(static_cast<size_t>(std::max(T, 1)) * H);  // token-major MXFP8 x (MOE_A_GATHER)
    L->sched = take(sizeof(int) * (kSchedWords + static_cast<size_t>(cap / kBlockM)));
    L->total = o;
    return true;
}

cudaError_t launch_prepare_sf(const uint8_t* sf, int E, int N, int K, int halves, uint8_t* out, size_t out_bytes,
                              cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(E) * N * (K / kSfVec);
    if (total == 0) return cudaSuccess;
    cudaError_t st = cudaMemsetAsync(out, 0, out_bytes, s);  // zero the unused half of an odd last pair
    if (st != cudaSuccess) return st;
    const int threads = 256;
    prepare_sf_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, s>>>(sf, total, N, K,
                                                                                                 halves, out);
    return cudaGetLastError();
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_plan_workspace_bytes(int T, int k, int E, int H, int I) {
    Layout L;
    return make_layout(T, k, E, H, I, &L) ? L.total : 0;
}

size_t moe_weight_scales_bytes(int E, int N, int K) {
    if (E < 1 || N < 128 || K < 128 || N % 128 || K % 128) return 0;
    return static_cast<size_t>(E) * ((N + 255) / 256) * (K / 128) * 2 * kSfChunkBytes;
}

int moe_prepare_weight_scales(const void* sf, int E, int N, int K, int pairing, void* sf_mma,
                              size_t sf_mma_bytes, void* stream) {
    if (!sf || !sf_mma) return MOE_ERR_INVALID_ARG;
    if (pairing != MOE_SF_PAIRS_ADJACENT && pairing != MOE_SF_PAIRS_HALVES) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_weight_scales_bytes(E, N, K);
    if (need == 0) return MOE_ERR_UNSUPPORTED;
    if (pairing == MOE_SF_PAIRS_HALVES && (N / 2) % 128) return MOE_ERR_INVALID_ARG;
    if (sf_mma_bytes < need) return MOE_ERR_INVALID_ARG;
    int rc = device_info(nullptr);
    if (rc) return rc;
    return cuda_status(launch_prepare_sf(static_cast<const uint8_t*>(sf), E, N, K, pairing == MOE_SF_PAIRS_HALVES,
                                         static_cast<uint8_t*>(sf_mma), need, static_cast<cudaStream_t>(stream)));
}

int moe_plan(moe_plan_t* plan, const int64_t* topk_idx, const float* topk_w, int T, int k, int E, int H, int I,
             void* workspace, size_t workspace_bytes, void* stream) {
    if (!plan || !workspace) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MOE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(T, k, E, H, I, &L)) return MOE_ERR_UNSUPPORTED;
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    int rc = device_info(nullptr);
    if (rc) return rc;
    PlanState ps{};
    ps.magic = kPlanMagic;
    ps.ws = static_cast<uint8_t*>(workspace);
    ps.ws_bytes = workspace_bytes;
    ps.T = T;
    ps.k = k;
    ps.E = E;
    ps.H = H;
    ps.I = I;
    cudaGetDevice(&ps.device);
    std::memset(plan, 0, sizeof(*plan));
    std::memcpy(plan, &ps, sizeof(ps));
    return cuda_status(launch_route(L, ps.ws, topk_idx, topk_w, static_cast<cudaStream_t>(stream)));
}

int moe_dispatch(const moe_plan_t* plan, const void* x, const moe_options_t* opts, void* stream) {
    const PlanState* ps = plan_state(plan);
    moe_options_t o;
    if (!ps || (ps->T > 0 && !x) || (reinterpret_cast<uintptr_t>(x) & 15u)) return MOE_ERR_INVALID_ARG;
    if (!read_options(opts, &o)) return MOE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(ps->T, ps->k, ps->E, ps->H, ps->I, &L)) return MOE_ERR_INVALID_ARG;  // a valid plan always has one
    int rc = device_info(nullptr);
    if (rc) return rc;
    return cuda_status(
        launch_dispatch(L, ps->ws, x, o.scale_rule, o.a_operand == MOE_A_GATHER, static_cast<cudaStream_t>(stream)));
}

static int expert_layer(int layer, const moe_plan_t* plan, const moe_weights_t* W, const moe_options_t* opts,
                        void* stream) {
    const PlanState* ps = plan_state(plan);
    moe_options_t o;
    if (!ps || !read_options(opts, &o)) return MOE_ERR_INVALID_ARG;
    const int N = layer == 1 ? 2 * ps->I : ps->H;
    const int K = layer == 1 ? ps->H : ps->I;
    int rc = check_weights(W, ps->E, N, K);
    if (rc) return rc;
    int sms = 0;
    if ((rc = device_info(&sms))) return rc;
    Layout L;
    if (!make_layout(ps->T, ps->k, ps->E, ps->H, ps->I, &L)) return MOE_ERR_INVALID_ARG;  // a valid plan always has one
    GemmLaunch g{W->q, W->sf_mma, W->E, W->N, W->K, o.activation_clamp, o.scale_rule, o.fast_math,
                 layer == 1 && o.a_operand == MOE_A_GATHER};
    return cuda_status(launch_expert_gemm(layer, L, ps->ws, g, sms, static_cast<cudaStream_t>(stream)));
}

int moe_expert_l1(const moe_plan_t* plan, const moe_weights_t* W1, const moe_options_t* opts, void* stream) {
    return expert_layer(1, plan, W1, opts, stream);
}

int moe_expert_l2(const moe_plan_t* plan, const moe_weights_t* W2, void* stream) {
    return expert_layer(2, plan, W2, nullptr, stream);
}

static int expert_fused(const moe_plan_t* plan, const moe_weights_t* W1, const moe_weights_t* W2,
                        const moe_options_t* opts, void* stream, bool publish) {
    const PlanState* ps = plan_state(plan);
    moe_options_t o;
    if (!ps || !read_options(opts, &o)) return MOE_ERR_INVALID_ARG;
    int rc = check_weights(W1, ps->E, 2 * ps->I, ps->H);
    if (rc) return rc;
    if ((rc = check_weights(W2, ps->E, ps->H, ps->I))) return rc;
    int sms = 0;
    if ((rc = device_info(&sms))) return rc;
    Layout L;
    if (!make_layout(ps->T, ps->k, ps->E, ps->H, ps->I, &L)) return MOE_ERR_INVALID_ARG;  // a valid plan always has one
    GemmLaunch g1{W1->q, W1->sf_mma, W1->E, W1->N, W1->K, o.activation_clamp, o.scale_rule, o.fast_math,
                  o.a_operand == MOE_A_GATHER};
    GemmLaunch g2{W2->q, W2->sf_mma, W2->E, W2->N, W2->K, 0.0f, MOE_SCALE_CEIL, 1, false};
    return cuda_status(launch_expert_fused(L, ps->ws, g1, g2, sms, static_cast<cudaStream_t>(stream), publish));
}

int moe_expert_fused(const moe_plan_t* plan, const moe_weights_t* W1, const moe_weights_t* W2,
                     const moe_options_t* opts, void* stream) {
    return expert_fused(plan, W1, W2, opts, stream, true);
}

int moe_selftest_fused_wait(const moe_plan_t* plan, const moe_weights_t* W1, const moe_weights_t* W2, void* stream) {
    return expert_fused(plan, W1, W2, nullptr, stream, false);
}

int moe_combine(const moe_plan_t* plan, void* y, void* stream) {
    const PlanState* ps = plan_state(plan);
    if (!ps || (ps->T > 0 && !y) || (reinterpret_cast<uintptr_t>(y) & 15u)) return MOE_ERR_INVALID_ARG;
    int rc = device_info(nullptr);
    if (rc) return rc;
    Layout L;
    if (!make_layout(ps->T, ps->k, ps->E, ps->H, ps->I, &L)) return MOE_ERR_INVALID_ARG;  // a valid plan always has one
    return cuda_status(launch_combine(L, ps->ws, y, static_cast<cudaStream_t>(stream)));
}

int moe_forward(const void* x, const moe_weights_t* W1, const moe_weights_t* W2, const moe_plan_t* plan, void* y,
                const moe_options_t* opts, void* stream) {
    int rc;
    moe_options_t o;
    if (!read_options(opts, &o)) return MOE_ERR_INVALID_ARG;
    if ((rc = moe_dispatch(plan, x, &o, stream))) return rc;
    if ((rc = moe_expert_fused(plan, W1, W2, &o, stream))) return rc;
    return moe_combine(plan, y, stream);
}

int moe_plan_check(const moe_plan_t* plan, void* stream) {
    const PlanState* ps = plan_state(plan);
    if (!ps) return MOE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(ps->T, ps->k, ps->E, ps->H, ps->I, &L)) return MOE_ERR_INVALID_ARG;  // a valid plan always has one
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
    int err = 0;
    if (cudaMemcpy(&err, ps->ws + L.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (err & kDevErrBounds) return MOE_ERR_DEBUG_BOUNDS;
    if (err & kDevErrTimeout) return MOE_ERR_TIMEOUT;
    if (err & kDevErrBadExpert) return MOE_ERR_BAD_EXPERT_ID;
    return MOE_OK;
}

int moe_plan_export(const moe_plan_t* plan, int what, size_t* offset, size_t* bytes) {
    const PlanState* ps = plan_state(plan);
    if (!ps || !offset || !bytes) return MOE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(ps->T, ps->k, ps->E, ps->H, ps->I, &L)) return MOE_ERR_INVALID_ARG;  // a valid plan always has one
    const size_t cap = static_cast<size_t>(L.p_cap);
    const size_t n = static_cast<size_t>(ps->T) * ps->k;
    switch (what) {
        case MOE_EXPORT_COUNT: *offset = L.count; *bytes = 4 * ps->E; break;
        case MOE_EXPORT_OFFSETS: *offset = L.off; *bytes = 4 * (ps->E + 1); break;
        case MOE_EXPORT_POFFSETS: *offset = L.poff; *bytes = 4 * (ps->E + 1); break;
        case MOE_EXPORT_SLOT_OF: *offset = L.slot_of; *bytes = 4 * n; break;
        case MOE_EXPORT_ROW_TOKEN: *offset = L.row_token; *bytes = 4 * cap; break;
        case MOE_EXPORT_ROW_TOPK: *offset = L.row_topk; *bytes = 4 * cap; break;
        case MOE_EXPORT_ROW_WEIGHT: *offset = L.row_weight; *bytes = 4 * cap; break;
        case MOE_EXPORT_BLOCK_EXPERT: *offset = L.block_expert; *bytes = 4 * (cap / kBlockM); break;
        case MOE_EXPORT_NUM_BLOCKS: *offset = L.n_blocks; *bytes = 4; break;
        case MOE_EXPORT_POOL_Q: *offset = L.pool_q; *bytes = cap * ps->H; break;
        case MOE_EXPORT_POOL_SF: *offset = L.pool_sf; *bytes = (cap / kBlockM) * (ps->H / 128) * kSfChunkBytes; break;
        case MOE_EXPORT_H_Q: *offset = L.h_q; *bytes = cap * ps->I; break;
        case MOE_EXPORT_H_SF: *offset = L.h_sf; *bytes = (cap / kBlockM) * (ps->I / 128) * kSfChunkBytes; break;
        case MOE_EXPORT_L2_OUT: *offset = L.l2_out; *bytes = cap * ps->H * 2; break;
        case MOE_EXPORT_ERROR: *offset = L.err; *bytes = 8; break;
        case MOE_EXPORT_POOL_ROWS: *offset = 0; *bytes = cap; break;
        case MOE_EXPORT_MAX_COUNT: *offset = L.max_count; *bytes = 4; break;
        case MOE_EXPORT_X_Q: *offset = L.x_q; *bytes = static_cast<size_t>(ps->T) * ps->H; break;
        default: return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

int moe_selftest_bounded_wait(int arrive, uint64_t timeout_ns, int32_t* out, void* stream) {
    if (!out || timeout_ns == 0 || timeout_ns > 2000000000ull || (arrive != 0 && arrive != 1))
        return MOE_ERR_INVALID_ARG;
    int rc = device_info(nullptr);
    if (rc) return rc;
    return cuda_status(launch_bounded_wait_selftest(arrive, timeout_ns, out, static_cast<cudaStream_t>(stream)));
}

int moe_selftest_mma_rate(int kblocks, int32_t* status, int* ctas, void* stream) {
    if (!status || !ctas || kblocks < 1 || kblocks > (1 << 20)) return MOE_ERR_INVALID_ARG;
    int sms = 0;
    int rc = device_info(&sms);
    if (rc) return rc;
    *ctas = sms;
    return cuda_status(launch_mma_rate_selftest(kblocks, sms, status, static_cast<cudaStream_t>(stream)));
}

int moe_selftest_stream_rate(const void* a, const void* b, const void* sfa, const void* sfb, int kblocks,
                             int32_t* status, int* ctas, void* stream) {
    if (!a || !b || !sfa || !sfb || !status || !ctas || kblocks < 1 || kblocks > (1 << 20)) return MOE_ERR_INVALID_ARG;
    for (const void* p : {a, b, sfa, sfb})
        if (reinterpret_cast<uintptr_t>(p) & 15u) return MOE_ERR_INVALID_ARG;
    int sms = 0;
    int rc = device_info(&sms);
    if (rc) return rc;
    *ctas = sms;
    return cuda_status(launch_stream_rate_selftest(a, b, sfa, sfb, kblocks, sms, status, static_cast<cudaStream_t>(stream)));
}

const char* moe_error_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or device (needs sm_103, H%128==0, I%128==0, k<=32, E<=1024)";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA call failed";
        case MOE_ERR_BAD_EXPERT_ID: return "topk_idx held an expert id outside [-1, E); those entries were skipped";
        case MOE_ERR_TIMEOUT: return "a bounded device-side wait expired; outputs are invalid";
        case MOE_ERR_NO_KERNEL: return "no kernel image for this device";
        case MOE_ERR_DEBUG_BOUNDS:
            return "a bounds check of the debug build fired on a plan table (access skipped; outputs invalid)";
        case MOE_ERR_TOO_LARGE:
            return "sizes exceed the fixed scratch of moe_expert_offsets_static (T*k <= 262144, E <= 1024, "
                   "ceil(T*k/2048)*E <= 32768)";
        default: return "unknown status";
    }
}

}  // extern "C"
