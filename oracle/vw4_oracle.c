/*
 * vw4_oracle.c -- the CPU oracle for speculative-decoding verification with
 * 4-bit weights.  TEST INFRASTRUCTURE ONLY: nothing in the product path may
 * link, load or call this file.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.
 *
 * Plain, slow, obviously correct.  Floating point in fp64 unless the method
 * fixes the precision (the integer-mass acceptance rule below is fixed to fp32
 * + integers on purpose, so that committed ids are bit-exact).  Build with
 * -O2 -ffp-contract=off so that the compiler never fuses a*b+c on its own.
 *
 * What each function follows (page titles and sections of the source pages):
 *  - "Faster Gemma 4 on MLX with multi-token prediction", verification
 *    paragraph: the verify pass multiplies a block-quantized (nvfp4) weight
 *    matrix by a batch of 2-8 token rows with "identical computation" to the
 *    per-row product.  The oracle is that product written out: dequantize each
 *    weight, multiply, sum over k in fp64.
 *  - Qiita roofline article on MTP in llama.cpp, PART 2 sections 2-3 / 2-4:
 *    verify turns the matrix-vector product into a skinny matrix product over
 *    the same weights; the longest agreeing prefix is accepted and the target's
 *    own token at the first mismatch is always committed.
 *  - Ollama commit log for x/mlxrunner/mtp.go, "Greedy is a special case of
 *    sampled decoding" and "rework the MLX sampler": greedy is the temperature-0
 *    point mass; the distribution pipeline order is top-k -> temperature/
 *    softmax -> top-p -> min-p -> normalize -> categorical (penalties, the
 *    first stage there, are left to the caller); acceptance, residual and bonus draws
 *    reuse the same draft/target distributions; the seed makes it reproducible.
 *  - "Your model may already ship a speculative decoder", section "Why it is
 *    interesting on a Mac specifically": Leviathan/Chen rejection sampling with
 *    residual correction at temperature 0.6, top_p 0.95.
 *  - Qiita article PART 3 (expert scattering) and the mtp.go log on the
 *    segmented-gather path for MoE heads: each routed (token, expert) pair is a
 *    dense product with that expert's weights; the combine is the gate-weighted
 *    sum over a token's experts.
 *
 * Formats (no page defines the bit layouts; they are the standard ones):
 *  - E2M1 (OCP Microscaling v1.0): bits s e1 e0 m; e=0 -> m*0.5, else
 *    2^(e-1)*(1+m/2).
 *  - E4M3 "fn" (OCP 8-bit float): bits s eeee mmm, bias 7, subnormals, codes
 *    0x7F/0xFF are NaN, no infinity.
 *  - nvfp4 tensor: Wq u8[N][K/2] (element 2i = LOW nibble of byte i),
 *    S e4m3[N][K/16] (one scale per 16 consecutive k), one fp32 tensor scale.
 *  - Q4_0: qs u8[N][K/2] and d f16[N][K/32]; in 32-element block b of a row,
 *    byte j of the block holds element 32b+j (low nibble) and 32b+j+16 (high
 *    nibble); w = (nibble - 8) * d.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ formats */

ORACLE_API double oracle_e2m1(uint32_t code) {
    uint32_t s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

ORACLE_API double oracle_e4m3(uint32_t code) {
    uint32_t s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

ORACLE_API double oracle_f16(uint32_t bits) {
    uint32_t s = (bits >> 15) & 1u, e = (bits >> 10) & 31u, m = bits & 1023u;
    double mag;
    if (e == 31u) mag = (m == 0) ? INFINITY : NAN;
    else if (e == 0) mag = ldexp((double)m / 1024.0, -14);
    else mag = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return s ? -mag : mag;
}

/* bf16 is the upper half of an IEEE binary32. */
ORACLE_API double oracle_bf16(uint32_t bits) {
    uint32_t u = (bits & 0xFFFFu) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

enum { ORACLE_FMT_NVFP4 = 1, ORACLE_FMT_Q4_0 = 2 };

/* Dequantized weight w[n][k] of either format, in fp64. */
static double weight_at(int fmt, int K, const uint8_t* q, const void* scales,
                        double tensor_scale, int64_t n, int64_t k) {
    const uint8_t* row = q + n * (int64_t)(K / 2);
    if (fmt == ORACLE_FMT_NVFP4) {
        uint32_t byte = row[k / 2];
        uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
        const uint8_t* s = (const uint8_t*)scales + n * (int64_t)(K / 16);
        return oracle_e2m1(code) * oracle_e4m3(s[k / 16]) * tensor_scale;
    } else {
        int64_t blk = k / 32, j = k % 32;
        uint32_t byte = row[blk * 16 + (j & 15)];
        uint32_t nib = (j < 16) ? (byte & 15u) : (byte >> 4);
        const uint16_t* d = (const uint16_t*)scales + n * (int64_t)(K / 32);
        return ((double)nib - 8.0) * oracle_f16(d[blk]);
    }
}

ORACLE_API void oracle_dequant(int fmt, int N, int K, const uint8_t* q, const void* scales,
                               double tensor_scale, double* w /* [N][K] */) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = weight_at(fmt, K, q, scales, tensor_scale, n, k);
}

/* ------------------------------------------------------------------- GEMM */
/*
 * out[m][j] = sum_k a[m][k] * w[cols[j]][k]     (fp64, k ascending)
 * bound[m][j] = sum_k |a[m][k] * w[cols[j]][k]|
 * cols == NULL means all N columns (j == n).  A is bf16 (raw bits) [M][lda].
 * Each weight is dequantized once and used for all M rows: the definition
 * does not depend on how often it is decoded.
 */
ORACLE_API void oracle_gemm_w4(int fmt, int N, int K, const uint8_t* q, const void* scales,
                               double tensor_scale, const uint16_t* A, int M, int lda,
                               const int32_t* cols, int ncols, double* out, double* bound) {
    int64_t nc = cols ? ncols : N;
    double* a = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) a[m * K + k] = oracle_bf16(A[m * (int64_t)lda + k]);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t j = 0; j < nc; ++j) {
        int64_t n = cols ? cols[j] : j;
        double acc[8], mag[8];
        double* accv = M <= 8 ? acc : (double*)malloc(sizeof(double) * (size_t)M * 2);
        double* magv = M <= 8 ? mag : accv + M;
        for (int m = 0; m < M; ++m) { accv[m] = 0.0; magv[m] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            double w = weight_at(fmt, K, q, scales, tensor_scale, n, k);
            for (int m = 0; m < M; ++m) {
                double p = a[m * K + k] * w;
                accv[m] += p;
                magv[m] += fabs(p);
            }
        }
        for (int m = 0; m < M; ++m) {
            out[m * nc + j] = accv[m];
            if (bound) bound[m * nc + j] = magv[m];
        }
        if (M > 8) free(accv);
    }
    free(a);
}

/* ------------------------------------------------------------------- MoE */
/*
 * Routed pairs p = m*topk + j use expert e = expert_ids[p].  The expert
 * weights are stacked: expert e's rows are rows e*N .. e*N+N-1 of a [E*N][K]
 * tensor of the given format.  Activation row of pair p is A[m] when
 * rows_are_pairs == 0, else A[p].
 *   combine == 0: out[p][n]  = sum_k a_p[k] * w_e[n][k]        (out is [M*topk][N])
 *   combine == 1: out[m][n]  = sum_j gates[m][j] * pair(m,j)[n] (out is [M][N]),
 *                 the pair products in fp64, then summed over j ascending.
 * bound is the matching sum of |.| terms (|gate| times the pair bound).
 */
ORACLE_API void oracle_moe_w4(int fmt, int E, int N, int K, const uint8_t* q, const void* scales,
                              double tensor_scale, const uint16_t* A, int lda, int rows_are_pairs,
                              const int32_t* expert_ids, const float* gates, int M, int topk,
                              int combine, double* out, double* bound) {
    int64_t P = (int64_t)M * topk;
    int64_t per_expert_q = (int64_t)N * (K / 2);
    int64_t per_expert_s = (fmt == ORACLE_FMT_NVFP4) ? (int64_t)N * (K / 16) : (int64_t)N * (K / 32) * 2;
    double* pair_out = (double*)calloc((size_t)(P * N), sizeof(double));
    double* pair_bnd = (double*)calloc((size_t)(P * N), sizeof(double));
    for (int64_t p = 0; p < P; ++p) {
        int e = expert_ids[p];
        if (e < 0 || e >= E) continue; /* an invalid expert contributes nothing */
        const uint16_t* arow = A + (rows_are_pairs ? p : p / topk) * (int64_t)lda;
        oracle_gemm_w4(fmt, N, K, q + e * per_expert_q, (const uint8_t*)scales + e * per_expert_s,
                       tensor_scale, arow, 1, lda, NULL, 0, pair_out + p * N, pair_bnd + p * N);
    }
    if (!combine) {
        memcpy(out, pair_out, sizeof(double) * (size_t)(P * N));
        if (bound) memcpy(bound, pair_bnd, sizeof(double) * (size_t)(P * N));
    } else {
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                double s = 0.0, b = 0.0;
                for (int64_t j = 0; j < topk; ++j) {
                    double g = (double)gates[m * topk + j];
                    s += g * pair_out[(m * topk + j) * N + n];
                    b += fabs(g) * pair_bnd[(m * topk + j) * N + n];
                }
                out[m * N + n] = s;
                if (bound) bound[m * N + n] = b;
            }
    }
    free(pair_out);
    free(pair_bnd);
}

/* Stable counting sort of the routed pairs by expert: order[] receives pair
 * indices grouped by ascending expert, ties in pair order; seg_start[e] is the
 * first position of expert e (size E+1).  Invalid experts are dropped. */
ORACLE_API int oracle_route_sort(const int32_t* expert_ids, int P, int E, int32_t* order,
                                 int32_t* seg_start) {
    int n = 0;
    for (int e = 0; e < E; ++e) {
        seg_start[e] = n;
        for (int p = 0; p < P; ++p)
            if (expert_ids[p] == e) order[n++] = p;
    }
    seg_start[E] = n;
    return n;
}

/* ---------------------------------------------------------------- argmax */
/* Ties go to the lowest index; NaN compares as -infinity (so it never beats a
 * number, and an all-NaN or all -inf row returns index 0). */
static float nan_low(float v) { return (v != v) ? -INFINITY : v; }

ORACLE_API int32_t oracle_argmax_f32(const float* row, int64_t V) {
    int64_t best = 0;
    float bv = nan_low(row[0]);
    for (int64_t v = 1; v < V; ++v) {
        float x = nan_low(row[v]);
        if (x > bv) { bv = x; best = v; }
    }
    return (int32_t)best;
}

/* --------------------------------------------------------- greedy accept */
/*
 * For each sequence b: g_i = argmax of target row (b, i), i = 0..Kd.
 * n = first i < Kd with drafts[b][i] != g_i (n = Kd if none).
 * tokens[b] = drafts[b][0..n-1], then g_n, then -1 up to Kd+1 entries;
 * len[b] = n + 1.  Returns the number of out-of-range draft ids seen (they
 * never match, so they count as rejections).
 */
ORACLE_API int oracle_accept_greedy(const float* target, int64_t ld_b, const int32_t* drafts,
                                    int B, int Kd, int64_t V, int32_t* tokens, int32_t* len) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        const float* tb = target + (int64_t)b * ld_b;
        int n = 0;
        int32_t g = 0;
        for (int i = 0; i <= Kd; ++i) {
            g = oracle_argmax_f32(tb + (int64_t)i * V, V);
            if (i == Kd) break;
            int32_t x = drafts[(int64_t)b * Kd + i];
            if (x < 0 || x >= V) { bad++; break; }
            if (x != g) break;
            n++;
        }
        for (int i = 0; i <= Kd; ++i) {
            int32_t t = -1;
            if (i < n) t = drafts[(int64_t)b * Kd + i];
            else if (i == n) t = g;
            tokens[(int64_t)b * (Kd + 1) + i] = t;
        }
        len[b] = n + 1;
    }
    return bad;
}

/* ------------------------------------------------------------- Philox */
/*
 * Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers: as easy
 * as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
 * published multipliers and a Weyl-sequence key schedule.
 */
ORACLE_API void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                                     uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Counter layout: (position i, sequence b, offset lo, offset hi); key = seed. */
static void philox_at(uint64_t seed, uint64_t offset, uint32_t i, uint32_t b, uint32_t r[4]) {
    uint32_t ctr[4] = {i, b, (uint32_t)offset, (uint32_t)(offset >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    oracle_philox4x32_10(ctr, key, r);
}

/* ------------------------------------------------------------- own exp */
/*
 * exp on [-32, 0] from a Cody-Waite argument reduction (Cody & Waite,
 * "Software Manual for the Elementary Functions", 1980) and the degree-7
 * Taylor polynomial of e^r on |r| <= ln2/2, all in fp32 with explicit fused
 * multiply-adds, so that an implementation that performs the same IEEE
 * operations in the same order gets the same bits.
 *   n  = rint(x * log2(e))
 *   r  = (x - n*LN2_HI) - n*LN2_LO           (two fmas)
 *   p  = 1 + r + r^2/2! + ... + r^7/7!       (Horner, fmas)
 *   e  = p * 2^n                              (exact, result is normal)
 * LN2_HI is ln 2 rounded to 15 significant bits (n*LN2_HI is exact for
 * |n| < 512); LN2_LO is the fp32 rounding of ln2 - LN2_HI.  Inputs below -32
 * (and NaN) give 0: such terms weigh less than 2^-40 and vanish in the integer
 * mass below anyway.
 */
ORACLE_API float oracle_own_exp(float x) {
    const float LOG2E = 1.44269504088896340736f;
    const float LN2_HI = 0.693145751953125f;
    const float LN2_LO = 1.42860682030941723212e-6f;
    if (!(x >= -32.0f)) return 0.0f;
    float t = x * LOG2E;
    float n = rintf(t);
    float r = fmaf(-n, LN2_HI, x);
    r = fmaf(-n, LN2_LO, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ni = (int)n;
    uint32_t bits = (uint32_t)(ni + 127) << 23;
    float two_n;
    memcpy(&two_n, &bits, 4);
    return p * two_n;
}

ORACLE_API void oracle_own_exp_array(const float* x, float* y, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_own_exp(x[i]);
}

/* ------------------------------------------------- integer-mass sampler */
/*
 * Temperature / softmax / top-p / normalize, made exact with integers:
 *   mx  = max_v l_v
 *   x_v = fp32((fp32(l_v - mx)) * invT)
 *   W_v = floor(own_exp(x_v) * 2^40)                 (u64; exact scaling)
 *   S   = sum_v W_v
 * top-p keeps the shortest prefix, in order (W desc, index asc), whose mass
 * cum satisfies cum * 2^32 >= P * S, P = round(top_p * 2^32).  P >= 2^32
 * (top_p >= 1) keeps everything.  Dropped entries get W = 0; the kept sum is
 * returned.  The normalized distribution is W_v / S_kept.
 */
typedef unsigned __int128 u128;

typedef struct { uint64_t w; int64_t idx; } wi_t;

static int cmp_wdesc_iasc(const void* a, const void* b) {
    const wi_t* x = (const wi_t*)a;
    const wi_t* y = (const wi_t*)b;
    if (x->w != y->w) return (x->w > y->w) ? -1 : 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/* Order of the top-k stage: logit descending (NaN as -infinity, -0 equal to
 * +0, as in the argmax), then index ascending. */
typedef struct { float l; int64_t idx; } li_t;

static int cmp_ldesc_iasc(const void* a, const void* b) {
    const li_t* x = (const li_t*)a;
    const li_t* y = (const li_t*)b;
    if (x->l != y->l) return (x->l > y->l) ? -1 : 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/*
 * The whole pipeline of "rework the MLX sampler" (penalties are not part of
 * it here): top-k on the logits, temperature/softmax as the integer masses W,
 * top-p, min-p, normalize.
 *   top_k:  0 or >= V = off; else only the top_k first entries in (logit
 *           desc, index asc) order keep a mass, every other W is 0.
 *   P:      top-p as above, over the masses left by top-k.
 *   MP:     min-p, MP = round(min_p * 2^32), 0 = off: of the entries top-p
 *           keeps, those with W * 2^32 < MP * W_top are dropped too, W_top the
 *           largest mass.  (Both stages keep a prefix of the (W desc, index
 *           asc) order, so the result is the shorter of the two prefixes.)
 * Returns the kept sum.
 */
ORACLE_API uint64_t oracle_row_mass_ex(const float* logits, int64_t V, float invT, uint64_t P,
                                       int64_t top_k, uint64_t MP, uint64_t* W) {
    float mx = logits[0];
    for (int64_t v = 1; v < V; ++v)
        if (logits[v] > mx) mx = logits[v];
    unsigned char* in_k = (unsigned char*)malloc((size_t)V);
    memset(in_k, 1, (size_t)V);
    if (top_k > 0 && top_k < V) {
        li_t* o = (li_t*)malloc(sizeof(li_t) * (size_t)V);
        for (int64_t v = 0; v < V; ++v) { o[v].l = nan_low(logits[v]); o[v].idx = v; }
        qsort(o, (size_t)V, sizeof(li_t), cmp_ldesc_iasc);
        memset(in_k, 0, (size_t)V);
        for (int64_t j = 0; j < top_k; ++j) in_k[o[j].idx] = 1;
        free(o);
    }
    uint64_t S = 0;
    for (int64_t v = 0; v < V; ++v) {
        W[v] = 0;
        if (!in_k[v]) continue;
        float d = logits[v] - mx;
        float x = d * invT;
        float e = oracle_own_exp(x);
        float scaled = e * 1099511627776.0f; /* 2^40, exact */
        W[v] = (uint64_t)scaled;
        S += W[v];
    }
    free(in_k);
    if (P >= ((uint64_t)1 << 32) && MP == 0) return S;
    wi_t* srt = (wi_t*)malloc(sizeof(wi_t) * (size_t)V);
    for (int64_t v = 0; v < V; ++v) { srt[v].w = W[v]; srt[v].idx = v; }
    qsort(srt, (size_t)V, sizeof(wi_t), cmp_wdesc_iasc);
    int64_t keep = V;
    if (P < ((uint64_t)1 << 32)) {
        u128 target = (u128)P * (u128)S;
        uint64_t cum = 0;
        for (int64_t j = 0; j < V; ++j) {
            cum += srt[j].w;
            if (((u128)cum << 32) >= target) { keep = j + 1; break; }
        }
    }
    if (MP > 0) {
        const uint64_t Wtop = srt[0].w;
        int64_t j = 0;
        while (j < keep && ((u128)srt[j].w << 32) >= (u128)MP * Wtop) ++j;
        keep = j;
    }
    uint64_t kept = 0;
    for (int64_t j = 0; j < V; ++j) {
        if (j < keep) kept += srt[j].w;
        else W[srt[j].idx] = 0;
    }
    free(srt);
    return kept;
}

ORACLE_API uint64_t oracle_row_mass(const float* logits, int64_t V, float invT, uint64_t P,
                                    uint64_t* W) {
    return oracle_row_mass_ex(logits, V, invT, P, 0, 0, W);
}

/* Inverse CDF: first v (ascending) whose running sum of weights exceeds
 * t = floor(u64 * total / 2^64).  weights are u128 here so that the residual
 * products fit; total must be > 0. */
static int64_t categorical_u128(const u128* wts, int64_t V, u128 total, uint64_t u64) {
    /* t = floor(u64 * total / 2^64) with a 64x128 -> 192-bit product */
    uint64_t tlo = (uint64_t)total, thi = (uint64_t)(total >> 64);
    u128 lo = (u128)u64 * tlo;           /* bits 0..127 */
    u128 hi = (u128)u64 * thi;           /* bits 64..191 */
    u128 mid = (lo >> 64) + hi;          /* bits 64..191 of the product */
    u128 t = mid;                        /* floor(product / 2^64) */
    u128 run = 0;
    for (int64_t v = 0; v < V; ++v) {
        run += wts[v];
        if (run > t) return v;
    }
    return V - 1; /* not reached when total > 0 */
}

static int64_t categorical_u64(const uint64_t* W, int64_t V, uint64_t total, uint64_t u64) {
    u128 t = ((u128)u64 * (u128)total) >> 64;
    u128 run = 0;
    for (int64_t v = 0; v < V; ++v) {
        run += W[v];
        if (run > t) return v;
    }
    return V - 1;
}

/*
 * Rejection-sampling accept (Leviathan et al. / Chen et al.), exact integers.
 * target [B][ld_tb] with rows (b, i) at b*ld_tb + i*V, i = 0..Kd;
 * draft  [B][ld_db] with rows (b, i) at b*ld_db + i*V, i = 0..Kd-1.
 * Both go through the same transform (invT, P).  For i = 0..Kd-1, with
 * x = drafts[b][i] and Philox block (i, b, offset): U = r0 >> 8;
 * accept iff U * Wq(x) * Sp < 2^24 * Wp(x) * Sq (u128).  At the first
 * rejection draw from r_v = max(0, Wp_v*Sq - Wq_v*Sp) with U64 = r2:r1 of the
 * same block (if every r_v is 0, draw from p instead).  If all Kd are
 * accepted, draw the bonus from p_Kd with U64 of block (Kd, b).
 * temperature == 0 routes to the greedy rule and draws nothing.
 * Sequence b of this call uses Philox counter index b_base + b (so a slice of
 * a batch can be checked on its own).
 * Returns the number of out-of-range draft ids (counted as rejections).
 */
/* P = round(p * 2^32) of a probability threshold, saturating at 2^32. */
static uint64_t fixed32(float p) {
    double pd = (double)p * 4294967296.0;
    return (pd >= 4294967296.0) ? ((uint64_t)1 << 32) : (uint64_t)llround(pd);
}

/* With top_k and min_p (the rest of the sampler pipeline, oracle_row_mass_ex)
 * applied to the target and the draft rows alike; top_k = 0 and min_p = 0 is
 * oracle_accept_rejection. */
ORACLE_API int oracle_accept_rejection_ex(const float* target, int64_t ld_tb, const float* draft,
                                          int64_t ld_db, const int32_t* drafts, int B, int Kd,
                                          int64_t V, float temperature, float top_p,
                                          int64_t top_k, float min_p, uint64_t seed,
                                          uint64_t offset, uint32_t b_base, int32_t* tokens,
                                          int32_t* len) {
    if (temperature == 0.0f)
        return oracle_accept_greedy(target, ld_tb, drafts, B, Kd, V, tokens, len);
    float invT = (float)(1.0 / (double)temperature);
    const uint64_t P = fixed32(top_p);
    const uint64_t MP = min_p > 0.0f ? fixed32(min_p) : 0;
    int bad = 0;
    uint64_t* Wp = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
    uint64_t* Wq = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
    u128* r = (u128*)malloc(sizeof(u128) * (size_t)V);
    for (int b = 0; b < B; ++b) {
        const float* tb = target + (int64_t)b * ld_tb;
        const float* db = draft + (int64_t)b * ld_db;
        int n = 0;
        int64_t last = -1;
        for (int i = 0; i < Kd; ++i) {
            uint64_t Sp = oracle_row_mass_ex(tb + (int64_t)i * V, V, invT, P, top_k, MP, Wp);
            uint64_t Sq = oracle_row_mass_ex(db + (int64_t)i * V, V, invT, P, top_k, MP, Wq);
            int32_t x = drafts[(int64_t)b * Kd + i];
            uint32_t rr[4];
            philox_at(seed, offset, (uint32_t)i, b_base + (uint32_t)b, rr);
            uint64_t U = rr[0] >> 8;
            uint64_t u64 = ((uint64_t)rr[2] << 32) | rr[1];
            int ok = 0;
            if (x >= 0 && x < V) {
                u128 lhs = (u128)U * Wq[x] * Sp;
                u128 rhs = ((u128)Wp[x] * Sq) << 24;
                ok = lhs < rhs;
            } else {
                bad++;
            }
            if (ok) { n++; continue; }
            u128 R = 0;
            for (int64_t v = 0; v < V; ++v) {
                u128 a = (u128)Wp[v] * Sq, c = (u128)Wq[v] * Sp;
                r[v] = a > c ? a - c : 0;
                R += r[v];
            }
            if (R > 0) last = categorical_u128(r, V, R, u64);
            else last = categorical_u64(Wp, V, Sp, u64);
            break;
        }
        if (n == Kd) {
            uint64_t Sp = oracle_row_mass_ex(tb + (int64_t)Kd * V, V, invT, P, top_k, MP, Wp);
            uint32_t rr[4];
            philox_at(seed, offset, (uint32_t)Kd, b_base + (uint32_t)b, rr);
            uint64_t u64 = ((uint64_t)rr[2] << 32) | rr[1];
            last = categorical_u64(Wp, V, Sp, u64);
        }
        for (int i = 0; i <= Kd; ++i) {
            int32_t t = -1;
            if (i < n) t = drafts[(int64_t)b * Kd + i];
            else if (i == n) t = (int32_t)last;
            tokens[(int64_t)b * (Kd + 1) + i] = t;
        }
        len[b] = n + 1;
    }
    free(Wp);
    free(Wq);
    free(r);
    return bad;
}

ORACLE_API int oracle_accept_rejection(const float* target, int64_t ld_tb, const float* draft,
                                       int64_t ld_db, const int32_t* drafts, int B, int Kd,
                                       int64_t V, float temperature, float top_p, uint64_t seed,
                                       uint64_t offset, uint32_t b_base, int32_t* tokens,
                                       int32_t* len) {
    return oracle_accept_rejection_ex(target, ld_tb, draft, ld_db, drafts, B, Kd, V, temperature,
                                      top_p, 0, 0.0f, seed, offset, b_base, tokens, len);
}

/*
 * Draws x_i ~ q_i for every sequence and draft position with the same
 * transform and inverse-CDF rule, using Philox blocks (i, b, offset) -- the
 * caller passes an offset disjoint from the acceptance offset (e.g. +2^32).
 * Used only to make test inputs whose drafts really come from q.
 */
ORACLE_API void oracle_sample_drafts_ex(const float* draft, int64_t ld_db, int B, int Kd,
                                        int64_t V, float temperature, float top_p, int64_t top_k,
                                        float min_p, uint64_t seed, uint64_t offset,
                                        uint32_t b_base, int32_t* drafts) {
    float invT = (float)(1.0 / (double)temperature);
    const uint64_t P = fixed32(top_p);
    const uint64_t MP = min_p > 0.0f ? fixed32(min_p) : 0;
    uint64_t* Wq = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < Kd; ++i) {
            uint64_t Sq = oracle_row_mass_ex(draft + (int64_t)b * ld_db + (int64_t)i * V, V, invT,
                                             P, top_k, MP, Wq);
            uint32_t rr[4];
            philox_at(seed, offset, (uint32_t)i, b_base + (uint32_t)b, rr);
            uint64_t u64 = ((uint64_t)rr[2] << 32) | rr[1];
            drafts[(int64_t)b * Kd + i] = (int32_t)categorical_u64(Wq, V, Sq, u64);
        }
    free(Wq);
}

ORACLE_API void oracle_sample_drafts(const float* draft, int64_t ld_db, int B, int Kd, int64_t V,
                                     float temperature, float top_p, uint64_t seed,
                                     uint64_t offset, uint32_t b_base, int32_t* drafts) {
    oracle_sample_drafts_ex(draft, ld_db, B, Kd, V, temperature, top_p, 0, 0.0f, seed, offset,
                            b_base, drafts);
}
