/*
 * moe_oracle.c -- plain, slow CPU oracle of the block-FP8 mixture-of-experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file:
 * only tests/, __graft_entry__.smoke() and bench.py (its CPU-baseline leg and its
 * reference arm) use it.  It shares no code, header, table or constant generator with the
 * CUDA library; the two meet only through the seeded input generators.
 *
 * Every function restates one step of the method as the pages state it, with scalar loops and
 * no blocking, fusion or reordering beyond that statement:
 *
 *   route preparation  -- lmdeploy PR #4857 "optimize compact blocked FP8 MoE and route
 *                         preparation", section "Changes" (sorted indices, compact blocks) and
 *                         its review note on local-expert slices;
 *   activation quant   -- vLLM PR #53875 "Fuse clamped MoE activation and UE8M0 FP8 block
 *                         quantization", section "Purpose" (clamp, BF16 SiLU*mul, per-128 E4M3
 *                         quantisation, UE8M0 scales, expert filter); lmdeploy PR #4956
 *                         "Perf/pytorch block fp8 moe decode", section "Fused SwiGLU and FP8
 *                         quantization";
 *   grouped GEMM       -- lmdeploy PR #4956, section "Active-expert block scheduling" and
 *                         vLLM PR #53875 "Purpose" ("FP8 W8A8 block shape [128, 128]");
 *   moe_reduce         -- lmdeploy PR #4228 "Moe Reduce kernel", Copilot overview (weighted
 *                         top-k sum moved into a dedicated reduction; fp32 accumulation).
 *
 * Readings where the pages are silent:
 *   E4M3 is OCP e4m3fn (bias 7, max 448, no infinities); encoding rounds to nearest even and
 *   saturates finite values to +-448; the fp32 group scale is max(amax, 1e-10) / 448; UE8M0
 *   rounds that scale up to a power of two; the quantised value is an IEEE fp32 division; the
 *   SiLU exponential is one fixed fp32 algorithm (Cody-Waite reduction by ln 2, degree-7
 *   Taylor polynomial in Horner form with fused multiply-adds); the gate is the first N columns
 *   of the gate/up output and the up half the last N; BF16 rounding is to nearest even at each
 *   materialisation point; the GEMM K-block partial is summed exactly (double holds it exactly)
 *   and scales are applied and accumulated in double, rounded once to BF16; the reduce
 *   accumulates w*z in fp32 with fused multiply-adds in top-k order.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (optionally -fopenmp).  Contraction
 * must stay off: the pages' fp32 steps are separate roundings unless stated otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_SLICE 2

/* act codes: identity (input quantisation), SiLU(gate)*up with symmetric clamp on both halves,
 * SiLU(gate)*up with the gate clamped from above only and the up half clamped symmetrically. */
#define ORC_ACT_IDENTITY 0
#define ORC_ACT_SILU_MUL 1
#define ORC_ACT_SILU_MUL_GATE_UPPER 2

#define ORC_SCALE_F32 0
#define ORC_SCALE_UE8M0 1

/* ------------------------------------------------------------------------------------------ */
/* bit helpers                                                                                */
/* ------------------------------------------------------------------------------------------ */
static uint32_t f2u(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float u2f(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* 2^n as an fp32 value for n in [-126, 127] (normal range only). */
static float pow2i(int n) { return u2f((uint32_t)(n + 127) << 23); }

/* ------------------------------------------------------------------------------------------ */
/* E4M3 (OCP e4m3fn) codec                                                                    */
/* ------------------------------------------------------------------------------------------ */
/* Closed-form decode: sign s, exponent field e (4 bits, bias 7), mantissa m (3 bits).
 * e = 0 -> subnormal m * 2^-9;  e = 15, m = 7 -> NaN;  otherwise (1 + m/8) * 2^(e-7). */
float orc_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = (float)m * pow2i(-9);
    else v = (1.0f + (float)m / 8.0f) * pow2i(e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even encode with saturation of finite values (and infinities) to +-448;
 * NaN encodes as 0x7F with the sign kept; the sign of zero is kept. */
uint8_t orc_e4m3_encode(float x)
{
    uint8_t sign = (f2u(x) >> 31) ? 0x80 : 0x00;
    float a = fabsf(x);
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    if (a > 448.0f) return (uint8_t)(sign | 0x7E);
    if (a < 0.015625f) {                     /* below the smallest normal 2^-6: grid of 2^-9 */
        float q = rintf(a * 512.0f);         /* exact scaling, then round half to even      */
        return (uint8_t)(sign | (uint8_t)q); /* q == 8 is the code of 2^-6, as it should be */
    }
    int e = (int)((f2u(a) >> 23) & 0xFF) - 127;   /* a is a normal fp32 here, e in [-6, 8] */
    float frac = a / pow2i(e);                    /* exact, in [1, 2)                       */
    float t = rintf((frac - 1.0f) * 8.0f);        /* exact products, RNE on the 3-bit grid  */
    int m = (int)t;
    if (m == 8) { m = 0; e += 1; }
    int code = ((e + 7) << 3) | m;
    if (code > 0x7E) code = 0x7E;                 /* 0x7F would be NaN: saturate            */
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------------------------ */
/* BF16 round-to-nearest-even                                                                 */
/* ------------------------------------------------------------------------------------------ */
uint16_t orc_bf16_from_f32(float x)
{
    uint32_t u = f2u(x);
    if (isnan(x)) return (uint16_t)(((u >> 16) & 0x8000) | 0x7FC0);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float orc_f32_from_bf16(uint16_t h) { return u2f((uint32_t)h << 16); }

static uint16_t bf16_from_double(double x)
{
    /* Direct RNE from double to bf16 (one rounding): scale into the fp32 bit pattern exactly
     * when possible.  BF16 has the fp32 exponent range, so round the double to 8 significant
     * bits with ties to even, then convert (exactly) to fp32 and take the top half. */
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    int e;
    frexp(a, &e);                      /* a = f * 2^e, f in [0.5, 1)                          */
    int ulp_exp = e - 8;               /* 8 significant bits: ulp = 2^(e-8)                   */
    if (ulp_exp < -133) ulp_exp = -133;/* bf16 subnormal grid (fp32 subnormal step 2^-149,
                                          bf16 keeps 7 explicit bits: step 2^-133)            */
    double q = ldexp(a, -ulp_exp);     /* exact                                               */
    double r = nearbyint(q);           /* ties to even in the default rounding mode           */
    double v = ldexp(r, ulp_exp);
    float f = (float)v;                /* exact unless it overflows, which gives inf          */
    if (v > 3.3895313892515355e38) f = INFINITY;
    uint16_t h = (uint16_t)(f2u(f) >> 16);
    return (uint16_t)(x < 0 ? (h | 0x8000) : h);
}

/* ------------------------------------------------------------------------------------------ */
/* fp32 exponential used by SiLU                                                              */
/* ------------------------------------------------------------------------------------------ */
/* Cody & Waite argument reduction (W. J. Cody, W. Waite, "Software Manual for the Elementary
 * Functions", 1980): n = rint(x * log2 e), r = x - n*ln2 with ln 2 split into a high fp32 part
 * and the fp32 remainder, both subtractions as fused multiply-adds.  e^r comes from the degree-7
 * Taylor polynomial (coefficients 1/i! rounded to fp32) evaluated in Horner form with fused
 * multiply-adds; the result is scaled by 2^n in two exact power-of-two steps so that the only
 * rounding of the scaling is the last one.  |r| <= ln2/2 keeps the truncation error near
 * 2^-27 relative.  Outside [-104, 89] the result is 0 or +inf. */
float orc_exp_f32(float x)
{
    if (isnan(x)) return x;
    if (x > 89.0f) return INFINITY;
    if (x < -104.0f) return 0.0f;
    const float log2e = (float)1.44269504088896340736;
    const float ln2_hi = (float)0.69314718055994530942;
    const float ln2_lo = (float)(0.69314718055994530942 - (double)(float)0.69314718055994530942);
    float n = rintf(x * log2e);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float p = (float)(1.0 / 5040.0);
    p = fmaf(p, r, (float)(1.0 / 720.0));
    p = fmaf(p, r, (float)(1.0 / 120.0));
    p = fmaf(p, r, (float)(1.0 / 24.0));
    p = fmaf(p, r, (float)(1.0 / 6.0));
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ni = (int)n;
    int n1 = ni / 2, n2 = ni - n1;
    return (p * pow2i(n1)) * pow2i(n2);
}

/* SiLU(g) = g / (1 + e^-g): fp32 add, IEEE fp32 division. */
float orc_silu_f32(float g)
{
    float e = orc_exp_f32(-g);
    return g / (1.0f + e);
}

/* ------------------------------------------------------------------------------------------ */
/* group scale and quantised value                                                            */
/* ------------------------------------------------------------------------------------------ */
/* fp32 scale s = max(amax, 1e-10) / 448 (one IEEE division).  UE8M0: the same s rounded up to
 * 2^ceil(log2 s), taken exactly from its bits (non-zero mantissa -> next exponent). */
float orc_group_scale(float amax, int fmt)
{
    float s = fmaxf(amax, 1e-10f) / 448.0f;
    if (fmt == ORC_SCALE_UE8M0) {
        uint32_t b = f2u(s);
        uint32_t e = (b >> 23) & 0xFFu;
        if (b & 0x7FFFFFu) e += 1u;
        s = u2f(e << 23);
    }
    return s;
}

/* ------------------------------------------------------------------------------------------ */
/* activation value before quantisation                                                       */
/* ------------------------------------------------------------------------------------------ */
/* The value that is materialised in BF16 and then quantised:
 *   identity:  the BF16 input itself;
 *   SiLU*mul:  clamp (if finite), a = bf16( SiLU(g) * u ), fp32 product, one rounding. */
static float act_value(int act, float g, float u, float L)
{
    if (act == ORC_ACT_IDENTITY) return g;
    if (isfinite(L)) {
        if (act == ORC_ACT_SILU_MUL) g = fminf(fmaxf(g, -L), L);
        else g = fminf(g, L);
        u = fminf(fmaxf(u, -L), L);
    }
    float a = orc_silu_f32(g) * u;
    return orc_f32_from_bf16(orc_bf16_from_f32(a));
}

static int row_kept(int row, const int32_t* row_expert, const int32_t* expert_map, int E)
{
    if (!row_expert) return 1;
    int id = row_expert[row];
    if (id < 0 || id >= E) return 0;
    if (expert_map && expert_map[id] < 0) return 0;
    return 1;
}

/* Per row, per 128-wide group: optional SiLU*mul, BF16 materialisation, amax, scale, divide,
 * E4M3 encode.  in: BF16 [rows, N] (identity) or [rows, 2N] (gate | up).  Rows whose expert id
 * is invalid or maps to no local expert are skipped and their outputs left untouched.  out_a
 * (optional) receives the BF16 activation that was quantised. */
int orc_act_quant(int act, const uint16_t* in, int rows, int N, float clamp_limit, int fmt,
                  const int32_t* row_expert, const int32_t* expert_map, int E,
                  uint8_t* out_q, float* out_s, uint16_t* out_a)
{
    if (rows < 0 || N <= 0 || N % 128) return ORC_ERR_ARG;
    int W = act == ORC_ACT_IDENTITY ? N : 2 * N;
    int G = N / 128;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int row = 0; row < rows; ++row) {
        if (!row_kept(row, row_expert, expert_map, E)) continue;
        const uint16_t* x = in + (size_t)row * W;
        for (int g = 0; g < G; ++g) {
            float a[128];
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                int c = g * 128 + i;
                float gv = orc_f32_from_bf16(x[c]);
                float uv = act == ORC_ACT_IDENTITY ? 0.0f : orc_f32_from_bf16(x[N + c]);
                a[i] = act_value(act, gv, uv, clamp_limit);
                amax = fmaxf(amax, fabsf(a[i]));
            }
            float s = orc_group_scale(amax, fmt);
            for (int i = 0; i < 128; ++i) {
                size_t o = (size_t)row * N + g * 128 + i;
                out_q[o] = orc_e4m3_encode(a[i] / s);
                if (out_a) out_a[o] = orc_bf16_from_f32(a[i]);
            }
            out_s[(size_t)row * G + g] = s;
        }
    }
    return ORC_OK;
}

/* The unfused first half of the two-kernel path: BF16 SiLU*mul written out (no quantisation). */
int orc_silu_and_mul(int act, const uint16_t* in, int rows, int N, float clamp_limit,
                     uint16_t* out)
{
    if (rows < 0 || N <= 0 || act == ORC_ACT_IDENTITY) return ORC_ERR_ARG;
    for (int row = 0; row < rows; ++row)
        for (int c = 0; c < N; ++c) {
            float gv = orc_f32_from_bf16(in[(size_t)row * 2 * N + c]);
            float uv = orc_f32_from_bf16(in[(size_t)row * 2 * N + N + c]);
            out[(size_t)row * N + c] = orc_bf16_from_f32(act_value(act, gv, uv, clamp_limit));
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* route preparation                                                                          */
/* ------------------------------------------------------------------------------------------ */
/* Local expert of a route: invalid global ids (< 0 or >= E) and ids the expert map sends to -1
 * are dropped (-1).  A map entry outside [-1, E_loc) is an invalid slice. */
static int local_expert(int id, int E, const int32_t* expert_map, int E_loc, int* bad)
{
    if (id < 0 || id >= E) return -1;
    int e = expert_map ? expert_map[id] : id;
    if (e < -1 || e >= E_loc) { *bad = 1; return -1; }
    return e;
}

/* Block capacity: ceil(R / bm) + min(E_loc, R) blocks always hold every active expert's
 * blocks, because sum_e ceil(c_e / bm) <= R / bm + (#active experts). */
int orc_block_capacity(int R, int E_loc, int bm)
{
    return (R + bm - 1) / bm + (E_loc < R ? E_loc : R);
}

/* Stable counting sort of the routes by local expert (experts ascending, flat route id t*k+j
 * ascending inside an expert), each expert's run padded to a multiple of block_m with -1, one
 * block record per block_m chunk of an expert that received routes.  Slots and blocks past the
 * last block are -1.  expert_offset is the exclusive scan of the padded counts (E_loc+1). */
int orc_route_prepare(const int32_t* topk_ids, int M, int k, int E, const int32_t* expert_map,
                      int E_loc, int bm, int32_t* sorted_idx, int32_t* block_expert,
                      int32_t* num_blocks, int32_t* expert_count, int32_t* expert_offset)
{
    if (M < 0 || k <= 0 || E <= 0 || E_loc <= 0 || bm <= 0) return ORC_ERR_ARG;
    if (!expert_map && E_loc != E) return ORC_ERR_SLICE;
    int R = M * k, bad = 0;
    int B_cap = orc_block_capacity(R, E_loc, bm);
    int* loc = (int*)malloc(sizeof(int) * (size_t)(R > 0 ? R : 1));
    for (int r = 0; r < R; ++r) loc[r] = local_expert(topk_ids[r], E, expert_map, E_loc, &bad);
    if (bad) { free(loc); return ORC_ERR_SLICE; }
    for (int e = 0; e < E_loc; ++e) expert_count[e] = 0;
    for (int r = 0; r < R; ++r) if (loc[r] >= 0) expert_count[loc[r]] += 1;
    expert_offset[0] = 0;
    for (int e = 0; e < E_loc; ++e) {
        int padded = (expert_count[e] + bm - 1) / bm * bm;
        expert_offset[e + 1] = expert_offset[e] + padded;
    }
    int nb = expert_offset[E_loc] / bm;
    *num_blocks = nb;
    for (int i = 0; i < B_cap * bm; ++i) sorted_idx[i] = -1;
    for (int b = 0; b < B_cap; ++b) block_expert[b] = -1;
    for (int e = 0; e < E_loc; ++e)
        for (int b = expert_offset[e] / bm; b < expert_offset[e + 1] / bm; ++b) block_expert[b] = e;
    int* fill = (int*)calloc((size_t)E_loc, sizeof(int));
    for (int r = 0; r < R; ++r) {
        int e = loc[r];
        if (e < 0) continue;
        sorted_idx[expert_offset[e] + fill[e]] = r;
        fill[e] += 1;
    }
    free(fill);
    free(loc);
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* block-scaled FP8 GEMM, one output row per route                                            */
/* ------------------------------------------------------------------------------------------ */
static float g_dec[256];
static int g_dec_ready = 0;
static void dec_table(void)
{
    if (g_dec_ready) return;
    for (int c = 0; c < 256; ++c) g_dec[c] = orc_e4m3_decode((uint8_t)c);
    g_dec_ready = 1;
}

/* y[r, n] = sum_kb ( sum_{i in kb} aq[row(r), i] * W[e(r), n, i] ) * as[row(r), kb] * sW[e(r), n/128, kb]
 * The inner 128-term sum of FP8 products is exact in double (products have at most 8
 * significant bits and lie in [2^-18, 2^18]); the two scales multiply it and the K-blocks are
 * accumulated in double, rounded once to BF16.  Routes with route_row[r] < 0 are skipped. */
int orc_route_gemm(const uint8_t* aq, const float* as, int a_rows, int K, const uint8_t* wq,
                   const float* ws, int E_loc, int N_out, const int32_t* route_row,
                   const int32_t* route_expert, int R, uint16_t* out)
{
    if (K <= 0 || K % 128 || N_out <= 0 || N_out % 128) return ORC_ERR_ARG;
    dec_table();
    int KB = K / 128, NB = N_out / 128;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic)
#endif
    for (int r = 0; r < R; ++r) {
        int row = route_row[r], e = route_expert[r];
        if (row < 0 || row >= a_rows || e < 0 || e >= E_loc) continue;
        const uint8_t* a = aq + (size_t)row * K;
        for (int n = 0; n < N_out; ++n) {
            const uint8_t* w = wq + ((size_t)e * N_out + n) * K;
            double acc = 0.0;
            for (int kb = 0; kb < KB; ++kb) {
                double part = 0.0;
                for (int i = kb * 128; i < kb * 128 + 128; ++i)
                    part += (double)g_dec[a[i]] * (double)g_dec[w[i]];
                double sa = as[(size_t)row * KB + kb];
                double sw = ws[((size_t)e * NB + n / 128) * KB + kb];
                acc += part * sa * sw;
            }
            out[(size_t)r * N_out + n] = bf16_from_double(acc);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* moe_reduce                                                                                 */
/* ------------------------------------------------------------------------------------------ */
/* out[t, h] = bf16( sum over kept j, in order j = 0..k-1, of w[t, j] * z[t*k + j, h] ), the
 * sum held in fp32 and each term added with one fused multiply-add.  Dropped routes add 0. */
int orc_moe_reduce(const uint16_t* z, const float* topk_w, const int32_t* topk_ids,
                   const int32_t* expert_map, int M, int k, int E, int H, uint16_t* out)
{
    if (M < 0 || k <= 0 || H <= 0) return ORC_ERR_ARG;
    for (int t = 0; t < M; ++t)
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int id = topk_ids[t * k + j];
                if (id < 0 || id >= E) continue;
                if (expert_map && expert_map[id] < 0) continue;
                acc = fmaf(topk_w[t * k + j], orc_f32_from_bf16(z[((size_t)t * k + j) * H + h]), acc);
            }
            out[(size_t)t * H + h] = orc_bf16_from_f32(acc);
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* whole layer                                                                                */
/* ------------------------------------------------------------------------------------------ */
/* Sparse evaluation in the method's order: input quantisation per token, gate/up GEMM per kept
 * route, SiLU*mul + quantisation per kept route, down GEMM per kept route, weighted reduce.
 * token_list (optional, n_tokens entries) restricts the work to those tokens: every token's
 * output depends only on its own routes, so a sample is computed exactly as in the full run.
 * Output rows of tokens not in the list are left untouched. */
static int forward_impl(const uint16_t* x, const int32_t* topk_ids, const float* topk_w, int M,
                        int k, int E, const int32_t* expert_map, int E_loc, int H, int N,
                        const uint8_t* wgu_q, const float* wgu_s, const uint8_t* wd_q,
                        const float* wd_s, int act, float clamp_limit, int fmt,
                        const int32_t* token_list, int n_tokens, int dense, uint16_t* out)
{
    if (M < 0 || k <= 0 || E <= 0 || E_loc <= 0 || H % 128 || N % 128 || H <= 0 || N <= 0)
        return ORC_ERR_ARG;
    if (!expert_map && E_loc != E) return ORC_ERR_SLICE;
    int T = token_list ? n_tokens : M;
    int rc = ORC_OK, bad = 0;
    int HB = H / 128, NB = N / 128;
    /* per sampled token: quantised input row */
    uint8_t* xq = (uint8_t*)malloc((size_t)T * H + 1);
    float* xs = (float*)malloc(sizeof(float) * ((size_t)T * HB + 1));
    int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * ((size_t)T + 1));
    for (int i = 0; i < T; ++i) tok[i] = token_list ? token_list[i] : i;
    for (int i = 0; i < T; ++i) {
        if (tok[i] < 0 || tok[i] >= M) { rc = ORC_ERR_ARG; goto done; }
        orc_act_quant(ORC_ACT_IDENTITY, x + (size_t)tok[i] * H, 1, H, INFINITY, fmt, NULL, NULL, 0,
                      xq + (size_t)i * H, xs + (size_t)i * HB, NULL);
    }
    /* the (sample-token, expert) pairs to evaluate: the kept routes (sparse), or every local
     * expert for every token (dense brute force, masked by the routing afterwards) */
    int P = dense ? T * E_loc : T * k;
    int32_t* p_row = (int32_t*)malloc(sizeof(int32_t) * ((size_t)P + 1));
    int32_t* p_exp = (int32_t*)malloc(sizeof(int32_t) * ((size_t)P + 1));
    for (int i = 0; i < T; ++i) {
        if (dense) {
            for (int e = 0; e < E_loc; ++e) { p_row[i * E_loc + e] = i; p_exp[i * E_loc + e] = e; }
        } else {
            for (int j = 0; j < k; ++j) {
                int e = local_expert(topk_ids[tok[i] * k + j], E, expert_map, E_loc, &bad);
                p_row[i * k + j] = e >= 0 ? i : -1;
                p_exp[i * k + j] = e;
            }
        }
    }
    if (bad) { rc = ORC_ERR_SLICE; goto done2; }
    {
        uint16_t* gu = (uint16_t*)malloc(sizeof(uint16_t) * ((size_t)P * 2 * N + 1));
        uint8_t* aq = (uint8_t*)malloc((size_t)P * N + 1);
        float* as = (float*)malloc(sizeof(float) * ((size_t)P * NB + 1));
        uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * ((size_t)P * H + 1));
        int32_t* p_self = (int32_t*)malloc(sizeof(int32_t) * ((size_t)P + 1));
        int32_t* p_keep = (int32_t*)malloc(sizeof(int32_t) * ((size_t)P + 1));
        for (int p = 0; p < P; ++p) { p_self[p] = p_row[p] >= 0 ? p : -1; p_keep[p] = p_row[p] >= 0 ? 0 : -1; }
        orc_route_gemm(xq, xs, T, H, wgu_q, wgu_s, E_loc, 2 * N, p_row, p_exp, P, gu);
        orc_act_quant(act, gu, P, N, clamp_limit, fmt, p_keep, NULL, 1, aq, as, NULL);
        orc_route_gemm(aq, as, P, N, wd_q, wd_s, E_loc, H, p_self, p_exp, P, z);
        for (int i = 0; i < T; ++i) {
            int t = tok[i];
            for (int h = 0; h < H; ++h) {
                float acc = 0.0f;
                for (int j = 0; j < k; ++j) {
                    int e = local_expert(topk_ids[t * k + j], E, expert_map, E_loc, &bad);
                    if (e < 0) continue;
                    size_t p = dense ? (size_t)i * E_loc + e : (size_t)i * k + j;
                    acc = fmaf(topk_w[t * k + j], orc_f32_from_bf16(z[p * H + h]), acc);
                }
                out[(size_t)t * H + h] = orc_bf16_from_f32(acc);
            }
        }
        free(gu); free(aq); free(as); free(z); free(p_self); free(p_keep);
    }
done2:
    free(p_row); free(p_exp);
done:
    free(xq); free(xs); free(tok);
    return rc;
}

int orc_moe_forward(const uint16_t* x, const int32_t* topk_ids, const float* topk_w, int M, int k,
                    int E, const int32_t* expert_map, int E_loc, int H, int N,
                    const uint8_t* wgu_q, const float* wgu_s, const uint8_t* wd_q,
                    const float* wd_s, int act, float clamp_limit, int fmt,
                    const int32_t* token_list, int n_tokens, uint16_t* out)
{
    return forward_impl(x, topk_ids, topk_w, M, k, E, expert_map, E_loc, H, N, wgu_q, wgu_s,
                        wd_q, wd_s, act, clamp_limit, fmt, token_list, n_tokens, 0, out);
}

/* Brute force: every sampled token through every local expert, then masked by the routing and
 * summed with the routing weights in top-k order. */
int orc_moe_forward_dense(const uint16_t* x, const int32_t* topk_ids, const float* topk_w, int M,
                          int k, int E, const int32_t* expert_map, int E_loc, int H, int N,
                          const uint8_t* wgu_q, const float* wgu_s, const uint8_t* wd_q,
                          const float* wd_s, int act, float clamp_limit, int fmt, uint16_t* out)
{
    return forward_impl(x, topk_ids, topk_w, M, k, E, expert_map, E_loc, H, N, wgu_q, wgu_s,
                        wd_q, wd_s, act, clamp_limit, fmt, NULL, 0, 1, out);
}

/* ------------------------------------------------------------------------------------------ */
/* array helpers for tests                                                                    */
/* ------------------------------------------------------------------------------------------ */
void orc_e4m3_encode_array(const float* x, uint8_t* q, long n)
{ for (long i = 0; i < n; ++i) q[i] = orc_e4m3_encode(x[i]); }
void orc_e4m3_decode_array(const uint8_t* q, float* x, long n)
{ for (long i = 0; i < n; ++i) x[i] = orc_e4m3_decode(q[i]); }
void orc_bf16_round_array(const float* x, uint16_t* h, long n)
{ for (long i = 0; i < n; ++i) h[i] = orc_bf16_from_f32(x[i]); }
void orc_bf16_round_double_array(const double* x, uint16_t* h, long n)
{ for (long i = 0; i < n; ++i) h[i] = bf16_from_double(x[i]); }
void orc_exp_array(const float* x, float* y, long n)
{ for (long i = 0; i < n; ++i) y[i] = orc_exp_f32(x[i]); }
void orc_silu_array(const float* x, float* y, long n)
{ for (long i = 0; i < n; ++i) y[i] = orc_silu_f32(x[i]); }
void orc_group_scale_array(const float* amax, float* s, long n, int fmt)
{ for (long i = 0; i < n; ++i) s[i] = orc_group_scale(amax[i], fmt); }

int orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
