/*
 * moe_oracle.c -- plain CPU oracle for the fused MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU product path
 * never links or calls it, and this file shares no code, header, table or
 * helper with the CUDA sources.
 *
 * It is written to be read against the pages it follows, not to be fast:
 * sequential loops, double-precision accumulation, codecs that search the
 * format's value table instead of manipulating bits.  The only concession to
 * speed is an OpenMP "parallel for" over independent output rows.
 *
 * Sources (page titles of the analysed web pages):
 *   [P1] "DeepEP -> Mega MoE: the boundary evolution of communication and
 *        compute" -- dispatch.cuh snippet (expert counting, prefix sum, slot
 *        assignment), sm100_fp8_fp4_mega_moe.cuh snippets (SwiGLU, amax,
 *        FP8 requant), combine_utils.cuh snippet (fp32 top-k reduction).
 *   [P2] "Normal vs Low-Latency" section 2 (recipe (1,1,32), fast_math).
 *   [P3] "Dispatch/Combine in the DeepGEMM Mega MoE kernel" sections 3.1
 *        (count / offset / pool layout), 4.1 (skip of negative expert ids),
 *        4.2 (weight applied in the L1 epilogue; the 0.73/0.27 example),
 *        5.1 (combine: fp32 sum of bf16 rows), Appendix A.1/A.2 (buffers,
 *        expert pool aligned to the row block).
 * Number formats: OCP 8-bit floating point (OFP8) E4M3, and the OCP
 * Microscaling (MX) v1.0 formats E2M1 and the UE8M0 shared scale.
 *
 * Readings taken where the pages are silent (each is restated in the
 * design notes):
 *   - UE8M0 scale = smallest power of two 2^e with amax <= maxnorm * 2^e,
 *     e clamped to [-126, 127]; amax == 0 gives e = 0.
 *   - FP8 / FP4 casts round to nearest, ties to even, saturate to +-max.
 *   - Slots inside an expert follow ascending flat index t*k+j.
 *   - gate = rows [0, I) of W1, up = rows [I, 2I).
 *   - gate/up accumulators are rounded fp32 -> bf16 before SwiGLU.
 *   - The top-k weight multiplies the SwiGLU output once; combine is an
 *     unweighted fp32 sum over ascending j, rounded once to bf16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_BLOCK_M 128 /* expert pool rows are aligned to one MMA row block */
#define OR_SF_VEC 32   /* one UE8M0 scale per 32 elements (recipe 1,1,32)  */
#define OR_RULE_CEIL 0      /* activation scale rule: smallest 2^e with amax <= max * 2^e */
#define OR_RULE_OCP_FLOOR 1 /* activation scale rule: 2^(floor(log2 amax) - emax), saturating */

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* OFP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits.  Exponent field
 * 15 with mantissa 7 is NaN; there is no infinity.  Subnormals: field 0. */
double or_e4m3_decode(int code) {
    int s = (code >> 7) & 1, ex = (code >> 3) & 15, m = code & 7;
    double mag;
    if (ex == 15 && m == 7) return NAN;
    if (ex == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, ex - 7);
    return s ? -mag : mag;
}

/* Round to nearest representable E4M3 value, ties to the even code,
 * saturating to +-448 (the largest finite value).  Positive codes 0..126 are
 * monotone in value, so a binary search over them finds the two neighbours. */
int or_e4m3_encode(double v) {
    int sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x80 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7F;
    if (a >= 448.0) return sign | 0x7E;
    int lo = 0, hi = 126; /* invariant: value(lo) <= a < value(hi) or hi==lo */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (or_e4m3_decode(mid) <= a) lo = mid; else hi = mid;
    }
    double vlo = or_e4m3_decode(lo), vhi = or_e4m3_decode(hi);
    int pick;
    if (a - vlo < vhi - a) pick = lo;
    else if (a - vlo > vhi - a) pick = hi;
    else pick = (lo % 2 == 0) ? lo : hi; /* tie: even mantissa */
    return sign | pick;
}

/* MX E2M1: 1 sign (bit 3), 2 exponent, 1 mantissa; magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
static const double kE2m1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double or_e2m1_decode(int nibble) {
    double mag = kE2m1Mag[nibble & 7];
    return (nibble & 8) ? -mag : mag;
}

int or_e2m1_encode(double v) {
    int sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 8 : 0;
    double a = fabs(v);
    if (a >= 6.0) return sign | 7;
    int lo = 0;
    while (lo < 7 && kE2m1Mag[lo + 1] <= a) lo++;
    int hi = lo + 1;
    double dlo = a - kE2m1Mag[lo], dhi = kE2m1Mag[hi] - a;
    int pick = dlo < dhi ? lo : (dlo > dhi ? hi : ((lo % 2 == 0) ? lo : hi));
    return sign | pick;
}

/* UE8M0 shared scale, "ceil" rule: the smallest integer e with
 * amax <= maxnorm * 2^e, clamped to [-126, 127]; returns the biased byte
 * e + 127.  amax == 0 gives byte 127 (scale 1).  Found by stepping e, all
 * products exact in double. */
int or_ue8m0_ceil(double amax, double maxnorm) {
    if (!(amax > 0.0)) return 127;
    int q;
    frexp(amax, &q);            /* amax in [2^(q-1), 2^q) */
    int e = q - 16;             /* certainly too small for maxnorm >= 1 */
    while (amax > ldexp(maxnorm, e)) e++;
    if (e < -126) e = -126;
    if (e > 127) e = 127;
    return e + 127;
}

/* UE8M0 shared scale, OCP MX "floor" rule (OCP Microscaling Formats v1.0,
 * section 6.3): X = 2^(floor(log2(amax)) - emax_elem), emax_elem = 8 for
 * E4M3 (448 = 1.75 * 2^8) and 2 for E2M1 (6 = 1.5 * 2^2); scaled values
 * beyond the largest normal saturate in the cast.  e clamped to [-126, 127];
 * amax == 0 gives byte 127.  frexp gives amax = f * 2^q with f in [0.5, 1),
 * so floor(log2(amax)) = q - 1 exactly. */
int or_ue8m0_floor(double amax, int emax_elem) {
    if (!(amax > 0.0)) return 127;
    int q;
    frexp(amax, &q);
    int e = (q - 1) - emax_elem;
    if (e < -126) e = -126;
    if (e > 127) e = 127;
    return e + 127;
}

double or_ue8m0_value(int byte) { return ldexp(1.0, byte - 127); }

/* bfloat16: upper half of an IEEE binary32.  Round to nearest even on the
 * bit pattern (NaN kept as a quiet NaN). */
float or_bf16_decode(uint16_t h) {
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return f;
}

uint16_t or_bf16_encode(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    if (isnan(f)) return (uint16_t)((b >> 16) | 0x40);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

/* MX quantisation of n values (n a multiple of 32) to E4M3 codes with one
 * UE8M0 byte per 32 ([P1] amax reduction + __nv_fp8x4_e4m3 cast; recipe
 * (1,1,32) of [P2] section 2). */
void or_quant_mx_e4m3_rule(const float* v, int n, uint8_t* codes, uint8_t* sf, int rule) {
    for (int b = 0; b < n / OR_SF_VEC; ++b) {
        double amax = 0.0;
        for (int i = 0; i < OR_SF_VEC; ++i) amax = fmax(amax, fabs((double)v[b * OR_SF_VEC + i]));
        int byte = rule == OR_RULE_OCP_FLOOR ? or_ue8m0_floor(amax, 8) : or_ue8m0_ceil(amax, 448.0);
        sf[b] = (uint8_t)byte;
        double inv = ldexp(1.0, 127 - byte);
        for (int i = 0; i < OR_SF_VEC; ++i)
            codes[b * OR_SF_VEC + i] = (uint8_t)or_e4m3_encode((double)v[b * OR_SF_VEC + i] * inv);
    }
}

void or_quant_mx_e4m3(const float* v, int n, uint8_t* codes, uint8_t* sf) {
    or_quant_mx_e4m3_rule(v, n, codes, sf, OR_RULE_CEIL);
}

/* Same for E2M1 (maxnorm 6); nibbles returned one per byte. */
void or_quant_mx_e2m1(const float* v, int n, uint8_t* nibbles, uint8_t* sf) {
    for (int b = 0; b < n / OR_SF_VEC; ++b) {
        double amax = 0.0;
        for (int i = 0; i < OR_SF_VEC; ++i) amax = fmax(amax, fabs((double)v[b * OR_SF_VEC + i]));
        int byte = or_ue8m0_ceil(amax, 6.0);
        sf[b] = (uint8_t)byte;
        double inv = ldexp(1.0, 127 - byte);
        for (int i = 0; i < OR_SF_VEC; ++i)
            nibbles[b * OR_SF_VEC + i] = (uint8_t)or_e2m1_encode((double)v[b * OR_SF_VEC + i] * inv);
    }
}

/* ------------------------------------------------------------------------ */
/* Dispatch plan: counts -> offsets -> slots ([P1] dispatch.cuh snippet;     */
/* [P3] section 3.1 and Appendix A.2)                                        */
/* ------------------------------------------------------------------------ */

/* Returns 0, or 1 if an expert id outside [-1, E) was seen (it is skipped).
 * count[E]; off[E+1] exclusive scan of count; poff[E+1] exclusive scan of
 * count rounded up to the row block; slot_of[T*k] (-1 for skipped entries);
 * row_token/row_topk/row_weight[p_cap] with -1/-1/0 on padding rows.
 * Slot order inside an expert = ascending flat index (stable counting sort). */
int or_plan(const int64_t* topk_idx, const float* topk_w, int T, int k, int E, int64_t p_cap,
            int32_t* count, int32_t* off, int32_t* poff, int32_t* slot_of,
            int32_t* row_token, int32_t* row_topk, float* row_weight) {
    int bad = 0;
    int64_t n = (int64_t)T * k;
    for (int e = 0; e < E; ++e) count[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t e = topk_idx[i];
        if (e < -1 || e >= E) { bad = 1; continue; }
        if (e >= 0) count[e]++;
    }
    off[0] = 0;
    poff[0] = 0;
    for (int e = 0; e < E; ++e) {
        off[e + 1] = off[e] + count[e];
        int padded = (count[e] + OR_BLOCK_M - 1) / OR_BLOCK_M * OR_BLOCK_M;
        poff[e + 1] = poff[e] + padded;
    }
    if (poff[E] > p_cap) return 2;
    for (int64_t r = 0; r < p_cap; ++r) { row_token[r] = -1; row_topk[r] = -1; row_weight[r] = 0.0f; }
    int32_t* fill = (int32_t*)calloc((size_t)(E > 0 ? E : 1), sizeof(int32_t));
    for (int64_t i = 0; i < n; ++i) {
        int64_t e = topk_idx[i];
        if (e < 0 || e >= E) { slot_of[i] = -1; continue; }
        int32_t s = poff[e] + fill[e]++;
        slot_of[i] = s;
        row_token[s] = (int32_t)(i / k);
        row_topk[s] = (int32_t)(i % k);
        row_weight[s] = topk_w[i];
    }
    free(fill);
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN ([P1] SwiGLU / amax / FP8 requant snippets; [P3] 4.2, 5.1)     */
/* ------------------------------------------------------------------------ */

/* Dequantised weights of one expert: w[n*K + kk] = e2m1 * 2^(sf-127).
 * q is packed two nibbles per byte, the even index in the low nibble. */
static void dequant_expert(const uint8_t* q, const uint8_t* sf, int e, int N, int K, float* out) {
    const uint8_t* qe = q + (size_t)e * N * (K / 2);
    const uint8_t* se = sf + (size_t)e * N * (K / OR_SF_VEC);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int kk = 0; kk < K; ++kk) {
            uint8_t byte = qe[(size_t)n * (K / 2) + kk / 2];
            int nib = (kk % 2 == 0) ? (byte & 15) : (byte >> 4);
            double s = or_ue8m0_value(se[(size_t)n * (K / OR_SF_VEC) + kk / OR_SF_VEC]);
            out[(size_t)n * K + kk] = (float)(or_e2m1_decode(nib) * s);
        }
    }
}

/* The optional activation clamp ("activation_clamp" of the API on the
 * "Normal vs Low-Latency" page, whose meaning the pages do not spell out):
 * c > 0 limits the bf16-rounded gate and up values to [-c, c] before
 * SwiGLU; c <= 0 leaves them unchanged. */
static float clamp_act(float v, float c) {
    if (!(c > 0.0f)) return v;
    if (v > c) return c;
    if (v < -c) return -c;
    return v;
}

/* L1 of one (token, expert) row: gate/up accumulators (double sum -> fp32
 * -> bf16), SwiGLU * top-k weight in fp32, requantised to MXFP8 along I.
 *   xq/xsf : the token's E4M3 codes [H] and UE8M0 bytes [H/32]
 *   w1d    : dequantised W1 of the expert [2I, H]   (gate rows 0..I-1, up I..2I-1)
 *   weight : the top-k weight of this (token, j) entry
 * Outputs: h[I] (fp32 SwiGLU*w), hq[I] / hsf[I/32] (its MXFP8 form). */
static void l1_row(const uint8_t* xq, const uint8_t* xsf, const float* w1d, int H, int I, float weight,
                   float clamp, int rule, double* xd, float* h, uint8_t* hq, uint8_t* hsf) {
    for (int c = 0; c < H; ++c) xd[c] = or_e4m3_decode(xq[c]) * or_ue8m0_value(xsf[c / OR_SF_VEC]);
    for (int n = 0; n < I; ++n) {
        double ag = 0.0, au = 0.0;
        const float* wg = w1d + (size_t)n * H;
        const float* wu = w1d + (size_t)(I + n) * H;
        for (int c = 0; c < H; ++c) { ag += xd[c] * (double)wg[c]; au += xd[c] * (double)wu[c]; }
        float g = clamp_act(or_bf16_decode(or_bf16_encode((float)ag)), clamp);
        float u = clamp_act(or_bf16_decode(or_bf16_encode((float)au)), clamp);
        /* SwiGLU in fp32: (gate * 1/(1+exp(-gate))) * up, then * topk weight */
        float silu = (float)((double)g / (1.0 + exp(-(double)g)));
        float hu = silu * u;
        h[n] = hu * weight;
    }
    or_quant_mx_e4m3_rule(h, I, hq, hsf, rule);
}

/* L2 of one row: o[c] = bf16(double sum over i of deq(hq)*deq(W2[c])), unweighted.
 *   w2d : dequantised W2 of the expert [H, I] */
static void l2_row(const uint8_t* hq, const uint8_t* hsf, const float* w2d, int H, int I, double* hd, uint16_t* o) {
    for (int i = 0; i < I; ++i) hd[i] = or_e4m3_decode(hq[i]) * or_ue8m0_value(hsf[i / OR_SF_VEC]);
    for (int c = 0; c < H; ++c) {
        double acc = 0.0;
        const float* w = w2d + (size_t)c * I;
        for (int i = 0; i < I; ++i) acc += hd[i] * (double)w[i];
        o[c] = or_bf16_encode((float)acc);
    }
}

/* One (token, expert) row of the FFN: l1_row then l2_row. */
static void ffn_row(const uint8_t* xq, const uint8_t* xsf, const float* w1d, const float* w2d,
                    int H, int I, float weight, float clamp, int rule, double* xd, double* hd, float* h,
                    uint8_t* hq, uint8_t* hsf, uint16_t* o) {
    l1_row(xq, xsf, w1d, H, I, weight, clamp, rule, xd, h, hq, hsf);
    l2_row(hq, hsf, w2d, H, I, hd, o);
}

/* Token-major MXFP8 quantisation of x (bf16 bits [T,H]). */
void or_quant_x(const uint16_t* x, int T, int H, int rule, uint8_t* q, uint8_t* sf, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            for (int c = 0; c < H; ++c) row[c] = or_bf16_decode(x[(size_t)t * H + c]);
            or_quant_mx_e4m3_rule(row, H, q + (size_t)t * H, sf + (size_t)t * (H / OR_SF_VEC), rule);
        }
        free(row);
    }
}

/* Forward pass.  tokens == NULL computes every token; otherwise only the
 * ntok listed tokens, with y rows written in list order ([ntok, H]).
 * Optional per-pool-row outputs (may be NULL), written for the pool rows of
 * the computed tokens only (other rows are left as they are):
 *   hq_pool [p_cap, I], hsf_pool [p_cap, I/32], o_pool [p_cap, H] (bf16 bits),
 *   h_pool [p_cap, I] (fp32 SwiGLU*w before requantisation).
 * Work is done expert by expert over the expert-major pool, each expert's
 * weights dequantised once.  Returns the or_plan status (0 ok). */
int or_forward(const uint16_t* x, const int64_t* topk_idx, const float* topk_w,
               int T, int k, int E, int H, int I,
               const uint8_t* w1q, const uint8_t* w1sf, const uint8_t* w2q, const uint8_t* w2sf,
               const int32_t* tokens, int ntok, uint16_t* y,
               uint8_t* hq_pool, uint8_t* hsf_pool, uint16_t* o_pool, float* h_pool, int64_t p_cap,
               float clamp, int rule, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int64_t n = (int64_t)T * k;
    int32_t* count = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* off = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* poff = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* slot_of = (int32_t*)malloc(sizeof(int32_t) * (n > 0 ? n : 1));
    int32_t* row_token = (int32_t*)malloc(sizeof(int32_t) * (p_cap > 0 ? p_cap : 1));
    int32_t* row_topk = (int32_t*)malloc(sizeof(int32_t) * (p_cap > 0 ? p_cap : 1));
    float* row_weight = (float*)malloc(sizeof(float) * (p_cap > 0 ? p_cap : 1));
    int st = or_plan(topk_idx, topk_w, T, k, E, p_cap, count, off, poff, slot_of, row_token, row_topk, row_weight);
    if (st > 1) goto done;

    /* which tokens are wanted, and where their y row goes */
    int32_t* want = (int32_t*)malloc(sizeof(int32_t) * (T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) want[t] = tokens ? -1 : t;
    if (tokens) for (int i = 0; i < ntok; ++i) want[tokens[i]] = i;
    int nout = tokens ? ntok : T;

    /* quantise the wanted tokens of x (token-major; pool rows are copies) */
    uint8_t* xq = (uint8_t*)malloc((size_t)T * H + 1);
    uint8_t* xsf = (uint8_t*)malloc((size_t)T * (H / OR_SF_VEC) + 1);
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            if (want[t] < 0) continue;
            for (int c = 0; c < H; ++c) row[c] = or_bf16_decode(x[(size_t)t * H + c]);
            or_quant_mx_e4m3_rule(row, H, xq + (size_t)t * H, xsf + (size_t)t * (H / OR_SF_VEC), rule);
        }
        free(row);
    }

    /* per-entry L2 outputs of wanted tokens, indexed by output row and j */
    uint16_t* o_ent = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)nout * k * H + 2);
    float* w1d = (float*)malloc(sizeof(float) * (size_t)2 * I * H + 4);
    float* w2d = (float*)malloc(sizeof(float) * (size_t)H * I + 4);
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (p_cap > 0 ? p_cap : 1));

    for (int e = 0; e < E; ++e) {
        int nr = 0;
        for (int32_t r = poff[e]; r < poff[e] + count[e]; ++r)
            if (want[row_token[r]] >= 0) rows[nr++] = r;
        if (nr == 0) continue;
        dequant_expert(w1q, w1sf, e, 2 * I, H, w1d);
        dequant_expert(w2q, w2sf, e, H, I, w2d);
#pragma omp parallel
        {
            double* xd = (double*)malloc(sizeof(double) * (size_t)H);
            double* hd = (double*)malloc(sizeof(double) * (size_t)I);
            float* h = (float*)malloc(sizeof(float) * (size_t)I);
            uint8_t* hq = (uint8_t*)malloc((size_t)I);
            uint8_t* hsf = (uint8_t*)malloc((size_t)I / OR_SF_VEC + 1);
            uint16_t* o = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
            for (int ir = 0; ir < nr; ++ir) {
                int32_t r = rows[ir];
                int t = row_token[r], j = row_topk[r];
                ffn_row(xq + (size_t)t * H, xsf + (size_t)t * (H / OR_SF_VEC), w1d, w2d, H, I,
                        row_weight[r], clamp, rule, xd, hd, h, hq, hsf, o);
                memcpy(o_ent + ((size_t)want[t] * k + j) * H, o, sizeof(uint16_t) * H);
                if (hq_pool) memcpy(hq_pool + (size_t)r * I, hq, (size_t)I);
                if (hsf_pool) memcpy(hsf_pool + (size_t)r * (I / OR_SF_VEC), hsf, (size_t)I / OR_SF_VEC);
                if (o_pool) memcpy(o_pool + (size_t)r * H, o, sizeof(uint16_t) * H);
                if (h_pool) memcpy(h_pool + (size_t)r * I, h, sizeof(float) * I);
            }
            free(xd); free(hd); free(h); free(hq); free(hsf); free(o);
        }
    }

    /* combine ([P1] combine_utils.cuh; [P3] 5.1): fp32 sum over ascending j
     * of the valid entries' bf16 rows, one final round to bf16; +0 if none */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        int oi = want[t];
        if (oi < 0) continue;
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                if (slot_of[(size_t)t * k + j] < 0) continue;
                acc = acc + or_bf16_decode(o_ent[((size_t)oi * k + j) * H + c]);
            }
            y[(size_t)oi * H + c] = or_bf16_encode(acc);
        }
    }
    free(want); free(xq); free(xsf); free(o_ent); free(w1d); free(w2d); free(rows);
done:
    free(count); free(off); free(poff); free(slot_of); free(row_token); free(row_topk); free(row_weight);
    return st;
}

/* L2 and combine of the listed tokens from GIVEN requantised L1 outputs
 * hq_pool [p_cap, I] / hsf_pool [p_cap, I/32] (row-major, indexed by the
 * plan's pool rows): the second half of or_forward (the same l2_row and the
 * same combine), used to replay the layer from another implementation's h.
 * y [ntok, H] in list order.  Returns the or_plan status. */
int or_l2_combine(const int64_t* topk_idx, const float* topk_w, int T, int k, int E, int H, int I,
                  const uint8_t* w2q, const uint8_t* w2sf, const uint8_t* hq_pool, const uint8_t* hsf_pool,
                  int64_t p_cap, const int32_t* tokens, int ntok, uint16_t* y, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int64_t n = (int64_t)T * k;
    int32_t* count = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* off = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* poff = (int32_t*)malloc(sizeof(int32_t) * (E + 1));
    int32_t* slot_of = (int32_t*)malloc(sizeof(int32_t) * (n > 0 ? n : 1));
    int32_t* row_token = (int32_t*)malloc(sizeof(int32_t) * (p_cap > 0 ? p_cap : 1));
    int32_t* row_topk = (int32_t*)malloc(sizeof(int32_t) * (p_cap > 0 ? p_cap : 1));
    float* row_weight = (float*)malloc(sizeof(float) * (p_cap > 0 ? p_cap : 1));
    int st = or_plan(topk_idx, topk_w, T, k, E, p_cap, count, off, poff, slot_of, row_token, row_topk, row_weight);
    if (st > 1) goto done;
    int32_t* want = (int32_t*)malloc(sizeof(int32_t) * (T > 0 ? T : 1));
    for (int t = 0; t < T; ++t) want[t] = -1;
    for (int i = 0; i < ntok; ++i) want[tokens[i]] = i;
    uint16_t* o_ent = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)ntok * k * H + 2);
    float* w2d = (float*)malloc(sizeof(float) * (size_t)H * I + 4);
    int32_t* rows = (int32_t*)malloc(sizeof(int32_t) * (p_cap > 0 ? p_cap : 1));
    for (int e = 0; e < E; ++e) {
        int nr = 0;
        for (int32_t r = poff[e]; r < poff[e] + count[e]; ++r)
            if (want[row_token[r]] >= 0) rows[nr++] = r;
        if (nr == 0) continue;
        dequant_expert(w2q, w2sf, e, H, I, w2d);
#pragma omp parallel
        {
            double* hd = (double*)malloc(sizeof(double) * (size_t)I);
            uint16_t* o = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
            for (int ir = 0; ir < nr; ++ir) {
                int32_t r = rows[ir];
                l2_row(hq_pool + (size_t)r * I, hsf_pool + (size_t)r * (I / OR_SF_VEC), w2d, H, I, hd, o);
                memcpy(o_ent + ((size_t)want[row_token[r]] * k + row_topk[r]) * H, o, sizeof(uint16_t) * H);
            }
            free(hd); free(o);
        }
    }
    for (int i = 0; i < ntok; ++i) {
        int t = tokens[i];
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                if (slot_of[(size_t)t * k + j] < 0) continue;
                acc = acc + or_bf16_decode(o_ent[((size_t)i * k + j) * H + c]);
            }
            y[(size_t)i * H + c] = or_bf16_encode(acc);
        }
    }
    free(want); free(o_ent); free(w2d); free(rows);
done:
    free(count); free(off); free(poff); free(slot_of); free(row_token); free(row_topk); free(row_weight);
    return st;
}

/* Combine alone, over given per-pool-row bf16 outputs o_pool [p_cap, H] and
 * the slot map; used to check the GPU combine on identical inputs. */
void or_combine(const uint16_t* o_pool, const int32_t* slot_of, int T, int k, int H, uint16_t* y) {
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int32_t s = slot_of[(size_t)t * k + j];
                if (s < 0) continue;
                acc = acc + or_bf16_decode(o_pool[(size_t)s * H + c]);
            }
            y[(size_t)t * H + c] = or_bf16_encode(acc);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Brute force: one token at a time, no pool, no grouping, every weight      */
/* decoded where it is used.  Same quantisation points as or_forward.        */
/* ------------------------------------------------------------------------ */
int or_bruteforce_token(const uint16_t* x_row, const int64_t* idx_row, const float* w_row, int k, int E,
                        int H, int I, const uint8_t* w1q, const uint8_t* w1sf,
                        const uint8_t* w2q, const uint8_t* w2sf, float clamp, int rule, uint16_t* y_row) {
    float* xf = (float*)calloc(H > 0 ? H : 1, sizeof(float));
    uint8_t* xq = (uint8_t*)malloc(H);
    uint8_t* xsf = (uint8_t*)malloc(H / OR_SF_VEC + 1);
    float* h = (float*)malloc(sizeof(float) * I);
    uint8_t* hq = (uint8_t*)malloc(I);
    uint8_t* hsf = (uint8_t*)malloc(I / OR_SF_VEC + 1);
    float* acc_y = (float*)calloc(H, sizeof(float));
    int bad = 0;
    for (int c = 0; c < H; ++c) xf[c] = or_bf16_decode(x_row[c]);
    or_quant_mx_e4m3_rule(xf, H, xq, xsf, rule);
    for (int j = 0; j < k; ++j) {
        int64_t e = idx_row[j];
        if (e < -1 || e >= E) { bad = 1; continue; }
        if (e < 0) continue;
        for (int n = 0; n < I; ++n) {
            double ag = 0.0, au = 0.0;
            for (int c = 0; c < H; ++c) {
                double a = or_e4m3_decode(xq[c]) * or_ue8m0_value(xsf[c / OR_SF_VEC]);
                size_t rg = (size_t)e * 2 * I + n, ru = (size_t)e * 2 * I + I + n;
                uint8_t bg = w1q[rg * (H / 2) + c / 2], bu = w1q[ru * (H / 2) + c / 2];
                int ng = (c % 2 == 0) ? (bg & 15) : (bg >> 4);
                int nu = (c % 2 == 0) ? (bu & 15) : (bu >> 4);
                ag += a * or_e2m1_decode(ng) * or_ue8m0_value(w1sf[rg * (H / OR_SF_VEC) + c / OR_SF_VEC]);
                au += a * or_e2m1_decode(nu) * or_ue8m0_value(w1sf[ru * (H / OR_SF_VEC) + c / OR_SF_VEC]);
            }
            float g = clamp_act(or_bf16_decode(or_bf16_encode((float)ag)), clamp);
            float u = clamp_act(or_bf16_decode(or_bf16_encode((float)au)), clamp);
            float silu = (float)((double)g / (1.0 + exp(-(double)g)));
            float hu = silu * u;
            h[n] = hu * w_row[j];
        }
        or_quant_mx_e4m3_rule(h, I, hq, hsf, rule);
        for (int c = 0; c < H; ++c) {
            double acc = 0.0;
            size_t r2 = (size_t)e * H + c;
            for (int i = 0; i < I; ++i) {
                uint8_t b = w2q[r2 * (I / 2) + i / 2];
                int nb = (i % 2 == 0) ? (b & 15) : (b >> 4);
                acc += or_e4m3_decode(hq[i]) * or_ue8m0_value(hsf[i / OR_SF_VEC]) * or_e2m1_decode(nb) *
                       or_ue8m0_value(w2sf[r2 * (I / OR_SF_VEC) + i / OR_SF_VEC]);
            }
            float o = or_bf16_decode(or_bf16_encode((float)acc));
            acc_y[c] = acc_y[c] + o;
        }
    }
    for (int c = 0; c < H; ++c) y_row[c] = or_bf16_encode(acc_y[c]);
    free(xf); free(xq); free(xsf); free(h); free(hq); free(hsf); free(acc_y);
    return bad;
}

int or_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
