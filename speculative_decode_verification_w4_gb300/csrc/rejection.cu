// rejection.cu -- rejection-sampling accept with residual correction.
//
// Defined by "Your model may already ship a speculative decoder", section
// "Why it is interesting on a Mac specifically" (Leviathan and Chen rejection
// sampling with residual correction at temperature 0.6, top_p 0.95 reproduces
// plain decoding) and the Ollama mtp.go commit log paragraphs "Greedy is a
// special case of sampled decoding" and "rework the MLX sampler" (temperature
// / softmax -> top-p -> normalize -> categorical; acceptance, residual and
// bonus draws reuse the same draft and target distributions; seeded).
//
// Exact integer form, identical to the oracle, so committed ids are
// bit-exact:
//   W_v  = floor(own_exp(fp32(fp32(l_v - max l) * invT)) * 2^40)
//   top-p keeps the shortest prefix of (W desc, index asc) with
//         cum * 2^32 >= P * sum W,  P = round(top_p * 2^32)
//   accept draft x at position i iff  U * q(x) * Sp < 2^24 * p(x) * Sq
//   residual  r_v = max(0, p_v * Sq - q_v * Sp), inverse CDF with a 64-bit
//   uniform; bonus from p_Kd when every draft is accepted.
//
// Kernel 1 (row_kernel), one 512-thread CTA per logits row (two per SM) --
// every target row (b, i <= Kd) and every draft row (b, i < Kd)
// independently; the row is streamed three times:
//   * the max, and the max of every 128-entry segment (to the workspace);
//   * own_exp, sum W, and a log-scale histogram of the mass of the entries
//     at or above c0 = floor((2^32 - P) * 2^40 / (V * 2^32)) -- every entry
//     below it lies in the dropped tail, because all of them together weigh
//     less than (1 - P/2^32) * S (S >= 2^40, the top entry's own mass) -- in
//     one private copy per warp; the merged suffix sums give the bucket where
//     the kept prefix ends;
//   * that bucket's members (a scaled-logit window, then the exact test;
//     only the segments whose max reaches the window are read), sorted by
//     (W desc, index asc) and scanned, which gives the exact cut (an exact
//     radix search is the fallback when the bucket is crowded);
//   * (max, tau, cut, kept sum) of the row go to the workspace.
// Kernel 2 (seq_kernel), one CTA per sequence: the acceptance tests in
// order (Philox block (i, b)), then one ordered draw over the row it needs --
// the residual at the first rejection, or the bonus from p_Kd -- and the
// committed run.  Every entry whose scaled logit lies below a bound under the
// cut (a 1e-3 margin in the exponent) weighs 0, and so does every segment
// whose max does: the draw reads only the other segments, sums each of them
// (to the workspace), finds the segment that holds the draw point by a block
// scan of those sums and rescans that one segment.
#include <cmath>
#include <cstddef>

#include "ptx.cuh"
#include "vw4.h"
#include "vw4_internal.cuh"

namespace vw4 {

namespace {

constexpr uint32_t kStatusBadDraft = 0x1u;
constexpr uint32_t kStatusZeroResidual = 0x8u;
constexpr uint32_t kStatusBadListId = 0x10u;
constexpr int kThreads = 512;  // the sequence kernel
constexpr int kWarps = kThreads / 32;
constexpr int kLogBuckets = 16 + 37 * 8;  // exact 0..15, then 8 per binade up to 2^40
constexpr int kLinBuckets = 256;
constexpr int kCandTotal = 1024;   // top-k candidates a row may gather
// crossing-bucket members a row may gather before the radix fallback: the
// flat distributions of wide vocabularies (an LM head's 262144 logits of
// spread ~1.5 at T = 0.6) put a few thousand entries in the bucket where the
// top-p cut falls
constexpr int kCutCand = 4096;
constexpr int kRankSortMax = 128;  // up to this many: sort by counting ranks
constexpr unsigned long long kKeepAll = 1ull << 32;
static_assert(kThreads >= kMaxRows + 1, "one thread per acceptance test");

typedef unsigned __int128 u128;

struct RowInfo {
    float mx;
    int cut;                 // largest kept index among W == tau
    unsigned long long tau;  // kept: W > tau, or W == tau and v <= cut
    unsigned long long S;    // kept sum
    uint32_t tk_key;         // top-k: an entry takes part iff its logit key > tk_key,
    int tk_idx;              //   or == tk_key and its index <= tk_idx (off: 0, max int)
};

// The top-k order of a logit (the argmax's): NaN as -infinity, -0 as +0,
// then an order-preserving unsigned key.
__device__ __forceinline__ uint32_t logit_key(float l) {
    if (l != l) l = -INFINITY;
    if (l == 0.0f) l = 0.0f;
    const uint32_t b = __float_as_uint(l);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ------------------------------------------------------------- own exp
// Cody-Waite reduction + degree-7 Taylor polynomial in fp32 with explicit
// fmas; the same operations in the same order as the oracle's own_exp.
__device__ __forceinline__ float own_exp(float x) {
    if (!(x >= -32.0f)) return 0.0f;
    const float t = __fmul_rn(x, 1.44269504088896340736f);
    const float n = rintf(t);
    float r = __fmaf_rn(-n, 0.693145751953125f, x);
    r = __fmaf_rn(-n, 1.42860682030941723212e-6f, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    // n is an integer in [-47, 1]: adding 1.5 * 2^23 puts it in the low
    // mantissa bits (exact), which avoids a float-to-int conversion
    const int ni = __float_as_int(__fadd_rn(n, 12582912.0f)) - 0x4B400000;
    return __fmul_rn(p, __uint_as_float(static_cast<uint32_t>(ni + 127) << 23));
}

// own_exp(x) * 2^40 as the row statistics need it: the same reduction and
// polynomial, with the final power of two taken as 2^(n + 40).  The value is
// __fmul_rn(own_exp(x), 2^40) exactly wherever own_exp(x) > 0 (both are
// p * 2^(n + 40), in the normal range).  Below -32 (and for NaN) x is clamped
// to -32, where own_exp is 0 and this gives less than 1: the integer mass
// floor() of either is 0.
__device__ __forceinline__ float own_exp_2_40(float x) {
    x = fmaxf(x, -32.0f);
    const float t = __fmul_rn(x, 1.44269504088896340736f);
    const float n = rintf(t);
    float r = __fmaf_rn(-n, 0.693145751953125f, x);
    r = __fmaf_rn(-n, 1.42860682030941723212e-6f, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    // the bits of n + 1.5 * 2^23 are 0x4B400000 + n; the exponent field of
    // 2^(n + 40) is n + 167
    const uint32_t nb = __float_as_uint(__fadd_rn(n, 12582912.0f));
    return __fmul_rn(p, __uint_as_float((nb - (0x4B400000u - 167u)) << 23));
}

// own_exp_2_40 of two scaled logits with packed fp32-pair operations: each
// half is the same IEEE operation, rounding included, as in own_exp_2_40
// (x - n c equals x + n (-c)).  n = rint(t) is taken per half with rintf: a
// packed add and subtract of 1.5 * 2^23 was measured to round some exact
// ties (t = -9.5) away from the even integer, which moves the reduction by
// ln 2 and the result by an ulp.  n + 1.5 * 2^23 is then exact.
__device__ __forceinline__ float2 own_exp_2_40_x2(float2 x) {
    x.x = fmaxf(x.x, -32.0f);
    x.y = fmaxf(x.y, -32.0f);
    const float2 t = __fmul2_rn(x, make_float2(1.44269504088896340736f, 1.44269504088896340736f));
    const float2 n = make_float2(rintf(t.x), rintf(t.y));
    const float2 m = __fadd2_rn(n, make_float2(12582912.0f, 12582912.0f));
    float2 r = __ffma2_rn(n, make_float2(-0.693145751953125f, -0.693145751953125f), x);
    r = __ffma2_rn(n, make_float2(-1.42860682030941723212e-6f, -1.42860682030941723212e-6f), r);
    float2 p = make_float2(1.0f / 5040.0f, 1.0f / 5040.0f);
    p = __ffma2_rn(p, r, make_float2(1.0f / 720.0f, 1.0f / 720.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f / 120.0f, 1.0f / 120.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f / 24.0f, 1.0f / 24.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f / 6.0f, 1.0f / 6.0f));
    p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    const uint32_t bx = __float_as_uint(m.x), by = __float_as_uint(m.y);
    return __fmul2_rn(p, make_float2(__uint_as_float((bx - (0x4B400000u - 167u)) << 23),
                                     __uint_as_float((by - (0x4B400000u - 167u)) << 23)));
}

// The two exact 20-bit halves of W = floor(f), 0 <= f <= 2^40, as the bit
// patterns of 2^23 + hi and 2^23 + lo (a sum of them loses the 2^23 terms
// once, at the end): adding 2^23 rounding down is floor() below 2^23, and
// f - hi * 2^20 is exact (a multiple of ulp(f) below 2^20).
__device__ __forceinline__ void mass_bits(float f, uint32_t& hib, uint32_t& lob) {
    const float t1 = __fadd_rd(__fmul_rn(f, 9.5367431640625e-07f), 8388608.0f);
    const float fh = __fsub_rn(t1, 8388608.0f);
    const float t2 = __fadd_rd(__fmaf_rn(-fh, 1048576.0f, f), 8388608.0f);
    hib = __float_as_uint(t1);
    lob = __float_as_uint(t2);
}

__device__ __forceinline__ float scaled_x(float l, float mx, float invT) {
    return __fmul_rn(__fsub_rn(l, mx), invT);
}

// floor(e * 2^40) for 0 <= e <= 1 with 32-bit float operations only: f =
// e * 2^40 is exact; fh = floor(f / 2^20) < 2^21 and d = f - fh * 2^20 in
// [0, 2^20) are exact in fp32 (d is a multiple of ulp(f)); each integer part
// is read from the mantissa after adding 2^23.
__device__ __forceinline__ unsigned long long mass_of(float e) {
    const float f = __fmul_rn(e, 1099511627776.0f);
    const float fh = floorf(__fmul_rn(f, 9.5367431640625e-07f));
    const float d = __fmaf_rn(-fh, 1048576.0f, f);
    const float dl = floorf(d);
    const uint32_t hi = __float_as_uint(__fadd_rn(fh, 8388608.0f)) - 0x4B000000u;
    const uint32_t lo = __float_as_uint(__fadd_rn(dl, 8388608.0f)) - 0x4B000000u;
    return (static_cast<unsigned long long>(hi) << 20) | lo;
}

__device__ __forceinline__ bool in_top_k(float l, int v, const RowInfo& s) {
    const uint32_t k = logit_key(l);
    return k > s.tk_key || (k == s.tk_key && v <= s.tk_idx);
}

// The kept mass of entry v (logit l, mass W) of a row.
__device__ __forceinline__ unsigned long long kept(unsigned long long W, float l, int v,
                                                   const RowInfo& s) {
    return ((W > s.tau || (W == s.tau && v <= s.cut)) && in_top_k(l, v, s)) ? W : 0ull;
}

// Log-scale bucket of W = floor(f) >= 1, f = e * 2^40: W itself below 16,
// then 16 + 8 * (binade - 4) + the 3 bits after the leading one.  Computed
// from the float's bits: every bucket edge at or above 16 is an integer, so
// floor() never crosses one.
__device__ __forceinline__ int log_bucket_f(float f) {
    if (f < 16.0f) return static_cast<int>(f);
    const uint32_t bits = __float_as_uint(f);
    const int msb = static_cast<int>((bits >> 23) & 0xFFu) - 127;
    return 16 + (msb - 4) * 8 + static_cast<int>((bits >> 20) & 7u);
}

// The e range [lo, hi) of log bucket beta (exact: the edges have at most 4
// significant bits, and the 2^-40 scaling is exact).
__device__ __forceinline__ void bucket_e_range(int beta, float& lo, float& hi) {
    unsigned long long a, b;
    if (beta < 16) {
        a = static_cast<unsigned long long>(beta);
        b = a + 1ull;
    } else {
        const int msb = 4 + (beta - 16) / 8, j = (beta - 16) % 8;
        a = static_cast<unsigned long long>(8 + j) << (msb - 3);
        b = static_cast<unsigned long long>(9 + j) << (msb - 3);
    }
    lo = __fmul_rn(__ull2float_rn(a), 9.094947017729282379e-13f);  // * 2^-40
    hi = __fmul_rn(__ull2float_rn(b), 9.094947017729282379e-13f);
}

// ------------------------------------------------------------- Philox
__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1, uint32_t out[4]) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

// --------------------------------------------------------------- helpers
__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int o) {
    const unsigned long long lo = __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v), o);
    const unsigned long long hi =
        __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v >> 64), o);
    return (static_cast<u128>(hi) << 64) | lo;
}

__device__ __forceinline__ u128 shfl_up_u128(u128 v, int o) {
    const unsigned long long lo = __shfl_up_sync(0xffffffffu, static_cast<unsigned long long>(v), o);
    const unsigned long long hi =
        __shfl_up_sync(0xffffffffu, static_cast<unsigned long long>(v >> 64), o);
    return (static_cast<u128>(hi) << 64) | lo;
}

__device__ __forceinline__ u128 warp_sum_u128(u128 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += shfl_xor_u128(v, o);
    return v;
}

// floor(u * R / 2^64) for a 64-bit u and a 128-bit R (< 2^120 here)
__device__ __forceinline__ u128 scale_u64(unsigned long long u, u128 R) {
    const u128 lo = static_cast<u128>(u) * static_cast<unsigned long long>(R);
    const u128 hi = static_cast<u128>(u) * static_cast<unsigned long long>(R >> 64);
    return (lo >> 64) + hi;
}

// Scratch of the block-wide reductions (up to 32 warps; loops use the
// block's own warp count).
struct Red {
    unsigned long long w[32];
    unsigned long long w2[32];
    float f[32];
};

__device__ __forceinline__ float block_max(float v, Red& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sm.f[wid] = v;
    __syncthreads();
    float m = -INFINITY;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, sm.f[w]);
    __syncthreads();
    return m;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, Red& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sm.w[wid] = v;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += sm.w[w];
    __syncthreads();
    return t;
}

// Exclusive prefix over the block of a u128 value per thread; also returns the total.
__device__ __forceinline__ u128 block_excl_u128(u128 v, Red& sm, u128& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    u128 incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u128 y = shfl_up_u128(incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) {
        sm.w[wid] = static_cast<unsigned long long>(incl);
        sm.w2[wid] = static_cast<unsigned long long>(incl >> 64);
    }
    __syncthreads();
    u128 base = 0, t = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        const u128 x = (static_cast<u128>(sm.w2[w]) << 64) | sm.w[w];
        if (w < wid) base += x;
        t += x;
    }
    __syncthreads();
    total = t;
    return base + incl - v;
}

// ----------------------------------------------------------- row statistics
// Exact 64-bit add into shared memory with two native 32-bit atomics: the
// low word's carry goes to the high word (the value reads back as one u64).
__device__ __forceinline__ void atomic_add_u64_split(unsigned long long* a, unsigned long long v) {
    uint32_t* w = reinterpret_cast<uint32_t*>(a);  // little endian: w[0] low, w[1] high
    const uint32_t lo = static_cast<uint32_t>(v);
    const uint32_t hi = static_cast<uint32_t>(v >> 32);
    const uint32_t old = atomicAdd(&w[0], lo);
    const uint32_t carry = (old + lo < old) ? 1u : 0u;
    if (hi + carry) atomicAdd(&w[1], hi + carry);
}

// One 512-thread CTA per logits row, two per SM.  The row is streamed three
// times (the second and third partly from L2): the max and the segment
// maxima; own_exp, sum W and the mass histogram of the entries >= c0; the
// members of the crossing bucket, in the segments that can hold them.
constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kHistQ = 24;       // queue slots per lane (MassPass)
constexpr int kSegCache = 2048;  // segment maxima kept in shared memory (V <= 262144)
constexpr int kHistGroup = 16;   // entries a lane may push between two checks
static_assert(kRowThreads >= kLogBuckets, "one thread per log bucket in the suffix scan");

struct RowSmem {
    Red red;
    unsigned long long whist[kRowWarps][kLogBuckets];  // per-warp mass histograms
    unsigned long long mass[kLogBuckets];             // merged
    unsigned int cnt[kLinBuckets];                    // radix fallback: counts
    unsigned long long lmass[kLinBuckets];            //                 masses
    union {
        struct {
            unsigned long long cw[kCutCand];  // crossing-bucket members
            int ci[kCutCand];
        };
        float hq[kRowWarps][kHistQ][32];  // the mass pass's histogram queues
    };
    unsigned int ncand;
    int beta, wbits, cut_found;
    unsigned long long above, lo, width, n_eq, count_eq;
    RowInfo info;
    float segc[kSegCache];  // the row's segment maxima, when it has at most kSegCache
};

// f(k, l) for every entry of the row, each thread taking entries in
// coalesced float4 groups (four loads in flight).
template <class F>
__device__ __forceinline__ void stream_row(const float* __restrict__ row, int V, bool vec, F&& f) {
    const int tid = threadIdx.x;
    if (vec) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int V4 = V >> 2;
        int i = tid;
        for (; i + 3 * kRowThreads < V4; i += 4 * kRowThreads) {
            const float4 a = __ldg(r4 + i), b = __ldg(r4 + i + kRowThreads),
                         c = __ldg(r4 + i + 2 * kRowThreads), d = __ldg(r4 + i + 3 * kRowThreads);
            f(4 * i, a.x); f(4 * i + 1, a.y); f(4 * i + 2, a.z); f(4 * i + 3, a.w);
            const int j = i + kRowThreads, m = i + 2 * kRowThreads, q = i + 3 * kRowThreads;
            f(4 * j, b.x); f(4 * j + 1, b.y); f(4 * j + 2, b.z); f(4 * j + 3, b.w);
            f(4 * m, c.x); f(4 * m + 1, c.y); f(4 * m + 2, c.z); f(4 * m + 3, c.w);
            f(4 * q, d.x); f(4 * q + 1, d.y); f(4 * q + 2, d.z); f(4 * q + 3, d.w);
        }
        for (; i < V4; i += kRowThreads) {
            const float4 a = __ldg(r4 + i);
            f(4 * i, a.x); f(4 * i + 1, a.y); f(4 * i + 2, a.z); f(4 * i + 3, a.w);
        }
    } else {
        for (int k = tid; k < V; k += kRowThreads) f(k, __ldg(row + k));
    }
}

// Segments: the row's entries in runs of kSegLen = 128 (one warp's float4
// group).  The max pass records each segment's largest logit; a later pass
// that only wants entries with scaled logit >= xa skips every segment whose
// max falls below (scaled_x is monotone, so no entry of it can qualify; an
// entry that is NaN never qualifies either, and fmaxf passes it over).
constexpr int kSegLen = 128;

__device__ __forceinline__ int n_segments(int V) { return (V + kSegLen - 1) / kSegLen; }

// Order-preserving int key of a float (for a warp max by integer reduction).
__device__ __forceinline__ int float_key(float x) {
    const int k = __float_as_int(x);
    return k ^ ((k >> 31) & 0x7fffffff);
}

// A segment max written by this CTA in its max pass: from its shared-memory
// copy, or from the workspace through L2 (which the writes reached; L1 may
// hold an older line).
__device__ __forceinline__ float seg_load(const float* p) {
    return __isShared(p) ? *p : __ldcg(p);
}

// f(k, l) for every entry of the segments whose max passes the window test
// (vec rows with a segment table; otherwise every entry, as stream_row).
// (need(m): whether a segment whose largest logit is m can hold a wanted
// entry.)  A warp loads up to kDepth of its wanted segments before it hands
// any entry on (1 where f is heavy: its inlined copies would crowd the loop).
template <int kDepth = 4, class N, class F>
__device__ __forceinline__ void stream_segments(const float* __restrict__ row, int V, bool vec,
                                                const float* seg, N&& need_of, F&& f) {
    if (seg == nullptr) {
        stream_row(row, V, vec, f);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int V4 = V >> 2, nk = (V4 + kRowThreads - 1) / kRowThreads, nseg = n_segments(V);
    for (int k0 = 0; k0 < nk; k0 += 32) {
        // lane j tests the segment of step k0 + j that this warp streams
        const int k = k0 + lane, sg = k * kRowWarps + wid;
        bool need = false;
        if (k < nk && sg < nseg) need = need_of(seg_load(seg + sg));
        unsigned int m = __ballot_sync(0xffffffffu, need);  // the same in every lane
        while (m) {
            int ks[kDepth];
            float4 v[kDepth];
#pragma unroll
            for (int q = 0; q < kDepth; ++q) {
                ks[q] = -1;
                if (m) {
                    ks[q] = k0 + __ffs(m) - 1;
                    m &= m - 1;
                }
                const int i = ks[q] * kRowThreads + tid;
                v[q] = (ks[q] >= 0 && i < V4) ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kDepth; ++q) {
                const int i = ks[q] * kRowThreads + tid;
                if (ks[q] >= 0 && i < V4) {
                    f(4 * i, v[q].x); f(4 * i + 1, v[q].y); f(4 * i + 2, v[q].z);
                    f(4 * i + 3, v[q].w);
                }
            }
        }
    }
}

template <int kDepth = 4, class F>
__device__ __forceinline__ void stream_window(const float* __restrict__ row, int V, bool vec,
                                              const float* seg, float mx, float invT, float xa,
                                              F&& f) {
    stream_segments<kDepth>(row, V, vec, seg,
                    [&](float m) { return !(scaled_x(m, mx, invT) < xa); }, f);
}

// How many entries stream_row hands to this thread.
__device__ __forceinline__ uint32_t stream_count(int V, bool vec) {
    const int tid = threadIdx.x;
    if (vec) {
        const int V4 = V >> 2;
        return tid < V4 ? 4u * static_cast<uint32_t>((V4 - 1 - tid) / kRowThreads + 1) : 0u;
    }
    return tid < V ? static_cast<uint32_t>((V - 1 - tid) / kRowThreads + 1) : 0u;
}

// mass_bits of two entries with packed operations: the halves' bit patterns
// are 2^23 + floor(f / 2^20) (t1) and 2^23 + floor(f mod 2^20) (t2).
__device__ __forceinline__ void mass_bits_x2(float2 f, float2& t1, float2& t2) {
    const float2 k20 = make_float2(9.5367431640625e-07f, 9.5367431640625e-07f);
    const float2 m20 = make_float2(-1048576.0f, -1048576.0f);
    const float2 b23 = make_float2(8388608.0f, 8388608.0f);
    const float2 nb23 = make_float2(-8388608.0f, -8388608.0f);
    t1 = __fadd2_rd(__fmul2_rn(f, k20), b23);
    t2 = __fadd2_rd(__ffma2_rn(__fadd2_rn(t1, nb23), m20, f), b23);
}

// The mass pass over a lane's entries, two at a time with packed fp32-pair
// operations: the integer masses W = floor(own_exp(x) 2^40) summed exactly
// (as the two 20-bit halves' 2^23-biased bit patterns, mod 2^32; the true
// sums stay below 2^32), and every W >= cmin added to the warp's mass
// histogram.  Only a few entries reach cmin, so a lane does not add them as
// it meets them (the whole warp would step through the insertion for the one
// lane that has one): it queues their f = own_exp(x) 2^40 in its own column of
// a shared-memory queue, and the warp empties all its lanes' queues together
// when one of them runs full, recomputing each W from f bit for bit.
struct MassPass {
    float2 nmx, it2;
    float f_lo;               // f < f_lo proves W < cmin (cmin rounded down)
    unsigned long long cmin;
    unsigned long long* hist; // the warp's histogram [kLogBuckets]
    float* q0;                // this lane's queue column: slot s at q0[32 s]
    float* qp;                // next free slot
    uint32_t sum_hib, sum_lob, n;

    __device__ __forceinline__ void init(float mx, float invT, unsigned long long cmin_,
                                         float f_lo_, unsigned long long* hist_, float* col) {
        nmx = make_float2(-mx, -mx);
        it2 = make_float2(invT, invT);
        cmin = cmin_;
        f_lo = f_lo_;
        hist = hist_;
        q0 = col;
        qp = col;
        sum_hib = sum_lob = n = 0u;
    }
    __device__ __forceinline__ void pair(float la, float lb) {
        const float2 f = own_exp_2_40_x2(__fmul2_rn(__fadd2_rn(make_float2(la, lb), nmx), it2));
        float2 t1, t2;
        mass_bits_x2(f, t1, t2);
        sum_hib += __float_as_uint(t1.x) + __float_as_uint(t1.y);
        sum_lob += __float_as_uint(t2.x) + __float_as_uint(t2.y);
        n += 2u;
        if (f.x >= f_lo) { *qp = f.x; qp += 32; }
        if (f.y >= f_lo) { *qp = f.y; qp += 32; }
    }
    __device__ __forceinline__ void quad(const float4& v) {
        pair(v.x, v.y);
        pair(v.z, v.w);
    }
    // empties the warp's queues into the histogram (every lane calls it)
    __device__ __forceinline__ void drain() {
        const int mine = static_cast<int>((qp - q0) >> 5);
        const int rounds = __reduce_max_sync(0xffffffffu, mine);
        for (int r = 0; r < rounds; ++r) {
            if (r < mine) {
                const float f = q0[32 * r];
                uint32_t hib, lob;
                mass_bits(f, hib, lob);
                const unsigned long long W =
                    (static_cast<unsigned long long>(hib - 0x4B000000u) << 20) |
                    (lob - 0x4B000000u);
                if (W >= cmin) atomic_add_u64_split(&hist[log_bucket_f(f)], W);
            }
        }
        qp = q0;
    }
    // after at most kHistGroup entries per lane since the last call
    __device__ __forceinline__ void check() {
        if (__any_sync(0xffffffffu, (qp - q0) > 32 * (kHistQ - kHistGroup))) drain();
    }
    // the lane's exact sum of W (its entries' halves, with the bias removed)
    __device__ __forceinline__ unsigned long long sum() const {
        const uint32_t bias = n * 0x4B000000u;
        return (static_cast<unsigned long long>(sum_hib - bias) << 20) + (sum_lob - bias);
    }
};

// The scaled-logit window [xa, xb) that holds every entry with wlo <= W <
// whi (1 <= wlo): own_exp is monotone and within 2 ulp of exp, so a margin of
// 1e-3 in the exponent is far wider than any rounding.
__device__ __forceinline__ void x_window(unsigned long long wlo, unsigned long long whi, float& xa,
                                         float& xb) {
    const float ln2_40 = 27.725887222397812f;
    xa = __logf(static_cast<float>(wlo)) - ln2_40 - 1e-3f;
    xb = __logf(static_cast<float>(whi)) - ln2_40 + 1e-3f;
}

// Blocks of the maxima that a verify GEMM can hand over with its logits: the
// largest of every 16 consecutive entries of a row (NaN read as -infinity).
constexpr int kBlockLen = 16;
static_assert(kSegLen % kBlockLen == 0, "a segment is whole blocks");

// The row's max and segment maxima from its block maxima bm[ceil(V / 16)]
// instead of the row itself: the same values as the max pass for any row
// whose NaN entries (which weigh 0) lie elsewhere than index 0.
__device__ float row_max_from_blocks(const float* __restrict__ bm, int V, float* seg,
                                     RowSmem& sm) {
    const int nb = (V + kBlockLen - 1) / kBlockLen;
    float lmax = -INFINITY;
    if (seg != nullptr) {
        constexpr int kPer = kSegLen / kBlockLen;
        const int nseg = n_segments(V);
        for (int sg = threadIdx.x; sg < nseg; sg += kRowThreads) {
            float m = -INFINITY;
            const int b0 = sg * kPer, b1 = min(b0 + kPer, nb);
            for (int bk = b0; bk < b1; ++bk) m = fmaxf(m, __ldg(bm + bk));
            seg[sg] = m;
            if (sg < kSegCache) sm.segc[sg] = m;
            lmax = fmaxf(lmax, m);
        }
    } else {
        for (int bk = threadIdx.x; bk < nb; bk += kRowThreads) lmax = fmaxf(lmax, __ldg(bm + bk));
    }
    return block_max(lmax, sm.red);
}

// The row's max (valid in every thread), and its segment maxima into seg
// (vec rows), or null.
__device__ float row_max(const float* __restrict__ row, int V, bool vec, float* seg, RowSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    // 1. max, and the segment maxima: at step k warp w streams float4 groups
    //    kRowThreads k + 32 w + lane, i.e. segment kRowWarps k + w
    float lmax = -INFINITY;
    if (seg != nullptr) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int V4 = V >> 2, nk = (V4 + kRowThreads - 1) / kRowThreads, nseg = n_segments(V);
        const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        for (int k0 = 0; k0 < nk; k0 += 4) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = (k0 + j) * kRowThreads + tid;
                v[j] = (k0 + j < nk && i < V4) ? __ldg(r4 + i) : ninf;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (k0 + j >= nk) break;  // the same for the whole warp
                const float m = fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w));
                lmax = fmaxf(lmax, m);
                const int key = __reduce_max_sync(0xffffffffu, float_key(m));
                const int sg = (k0 + j) * kRowWarps + wid;
                if (lane == 0 && sg < nseg) {
                    const float sm_ = __int_as_float(key ^ ((key >> 31) & 0x7fffffff));
                    seg[sg] = sm_;
                    if (sg < kSegCache) sm.segc[sg] = sm_;
                }
            }
        }
    } else {
        stream_row(row, V, vec, [&](int, float l) { lmax = fmaxf(lmax, l); });
    }
    return block_max(lmax, sm.red);
}

// The top-k cut from the segment maxima.  Any L at or below the k-th largest
// segment max bounds the k-th largest entry from below (the k largest maxima
// are k distinct entries >= L), so every top-k entry has a key >= L and lies
// in a segment whose max reaches L.  L is the lower edge of the 16-bit key
// bucket holding the k-th largest maximum (two 256-bucket histograms of the
// maxima); the entries >= L are gathered (each as the packed key (logit key,
// ~index), all distinct) and the k-th of them found by counting ranks.
// Returns false -- nothing decided -- when the row has too many segments, k
// is larger than the gather holds, or too many entries reach L.
__device__ bool top_k_cut_segments(const float* __restrict__ row, int V, const float* seg,
                                   int top_k, RowSmem& sm, uint32_t& K, int& I) {
    constexpr int kMaxSegs = 2048;
    const int nseg = n_segments(V);
    if (nseg > kMaxSegs || nseg < top_k || top_k > kCandTotal) return false;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t* sk = reinterpret_cast<uint32_t*>(&sm.whist[0][0]);  // [kMaxSegs] maxima keys
    uint32_t* hist = sk + kMaxSegs;                                // [256]
    for (int t = tid; t < nseg; t += kRowThreads) sk[t] = logit_key(seg_load(seg + t));
    uint32_t prefix = 0u;
    unsigned int need = static_cast<unsigned int>(top_k);
    for (int shift = 24; shift >= 16; shift -= 8) {
        const uint32_t hmask = shift == 24 ? 0u : 0xFF000000u;
        if (tid < 256) hist[tid] = 0u;
        __syncthreads();
        for (int t0 = 0; t0 < nseg; t0 += kRowThreads) {  // the whole warp in step
            const int t = t0 + tid;
            const bool in = t < nseg && (sk[t] & hmask) == prefix;
            const unsigned int d = in ? ((sk[t] >> shift) & 255u) : 256u;
            const unsigned int peers = __match_any_sync(0xffffffffu, d);
            if (in && __ffs(peers) - 1 == lane) atomicAdd(&hist[d], __popc(peers));
        }
        __syncthreads();
        if (wid == 0) {
            // lane j holds buckets 255 - 8j .. 248 - 8j, counted from the top
            unsigned int c8[8], sum = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c8[i] = hist[255 - 8 * lane - i];
                sum += c8[i];
            }
            unsigned int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            unsigned int run = incl - sum;
            if (run < need && need <= incl) {
                for (int i = 0; i < 8; ++i) {
                    if (run + c8[i] >= need) {
                        sm.beta = 255 - 8 * lane - i;
                        sm.above = run;
                        break;
                    }
                    run += c8[i];
                }
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sm.beta) << shift;
        need -= static_cast<unsigned int>(sm.above);
        __syncthreads();
    }
    const uint32_t L = prefix;  // the 16-bit bucket's lower edge
    if (tid == 0) sm.ncand = 0;
    __syncthreads();
    stream_segments(row, V, true, seg, [&](float m) { return logit_key(m) >= L; },
                    [&](int k, float l) {
                        const uint32_t key = logit_key(l);
                        if (key >= L) {
                            const unsigned int slot = atomicAdd(&sm.ncand, 1u);
                            if (slot < static_cast<unsigned int>(kCandTotal))
                                sm.cw[slot] = (static_cast<unsigned long long>(key) << 32) |
                                              (0xFFFFFFFFu - static_cast<uint32_t>(k));
                        }
                    });
    __syncthreads();
    const unsigned int C = sm.ncand;
    if (C > static_cast<unsigned int>(kCandTotal)) return false;  // the same in every thread
    // the candidate with exactly top_k - 1 larger ones
    for (unsigned int i = tid; i < C; i += kRowThreads) {
        const unsigned long long ki = sm.cw[i];
        unsigned int rank = 0u;
        for (unsigned int j = 0; j < C; ++j) rank += sm.cw[j] > ki ? 1u : 0u;
        if (rank == static_cast<unsigned int>(top_k - 1)) sm.lo = ki;
    }
    __syncthreads();
    const unsigned long long kk = sm.lo;
    K = static_cast<uint32_t>(kk >> 32);
    I = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
    __syncthreads();
    return true;
}

// The top-k cut of a row: the key K and index I of its top_k-th entry in
// (logit key desc, index asc) order, so that an entry is among the first
// top_k iff its key > K, or == K and its index <= I.  A radix select on the
// 32-bit keys, eight bits a level: each level counts the entries whose higher
// bits match so far (warp-aggregated counts into per-warp histograms),
// skipping the segments whose largest logit lies below the level's range;
// then, when K is shared by more entries than the cut takes, the index cut
// among them in index order.
__device__ void top_k_cut(const float* __restrict__ row, int V, bool vec, const float* seg,
                          int top_k, RowSmem& sm, uint32_t& K, int& I) {
    if (seg != nullptr && top_k_cut_segments(row, V, seg, top_k, sm, K, I)) return;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t* hist = reinterpret_cast<uint32_t*>(&sm.whist[0][0]);  // [kRowWarps][256]
    uint32_t prefix = 0u;
    unsigned long long need = static_cast<unsigned long long>(top_k);
    unsigned long long n_at = 0ull;  // entries with the final key
    for (int shift = 24; shift >= 0; shift -= 8) {
        const uint32_t hmask = shift == 24 ? 0u : (0xFFFFFFFFu << (shift + 8));
        const uint32_t lo_key = prefix & hmask;  // the smallest key of this level's range
        for (int t = tid; t < kRowWarps * 256; t += kRowThreads) hist[t] = 0u;
        __syncthreads();
        uint32_t* h = hist + wid * 256;
        stream_segments(row, V, vec, seg, [&](float m) { return logit_key(m) >= lo_key; },
                        [&](int, float l) {
                            const uint32_t k = logit_key(l);
                            const bool in = (k & hmask) == lo_key;
                            const unsigned int d = in ? ((k >> shift) & 255u) : 256u;
                            const unsigned int peers = __match_any_sync(__activemask(), d);
                            if (in && __ffs(peers) - 1 == lane) atomicAdd(&h[d], __popc(peers));
                        });
        __syncthreads();
        // thread t holds digit 255 - t: the digit where the count from the
        // top first reaches `need`
        const int dg = 255 - tid;
        unsigned long long c = 0ull;
        if (dg >= 0)
            for (int w = 0; w < kRowWarps; ++w) c += hist[w * 256 + dg];
        u128 tot_unused;
        const u128 incl = block_excl_u128(static_cast<u128>(c), sm.red, tot_unused) + c;
        if (dg >= 0 && incl >= need && incl - c < need) {
            sm.beta = dg;
            sm.above = static_cast<unsigned long long>(incl - c);
            sm.count_eq = c;
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sm.beta) << shift;
        need -= sm.above;
        n_at = sm.count_eq;
        __syncthreads();
    }
    K = prefix;
    I = 0x7fffffff;
    if (need < n_at) {
        // the need-th entry with key K in index order: each thread counts its
        // contiguous chunk, a block scan orders the chunks
        const int chunk = (V + kRowThreads - 1) / kRowThreads;
        const int k0 = tid * chunk < V ? tid * chunk : V, k1 = k0 + chunk < V ? k0 + chunk : V;
        unsigned int mine = 0u;
        for (int k = k0; k < k1; ++k) mine += logit_key(__ldg(row + k)) == prefix ? 1u : 0u;
        u128 ctot;
        const unsigned long long excl = static_cast<unsigned long long>(
            block_excl_u128(static_cast<u128>(mine), sm.red, ctot));
        if (tid == 0) sm.cut_found = V - 1;
        __syncthreads();
        if (excl < need && need <= excl + mine) {
            unsigned long long seen = excl;
            for (int k = k0; k < k1; ++k)
                if (logit_key(__ldg(row + k)) == prefix && ++seen == need) {
                    sm.cut_found = k;
                    break;
                }
        }
        __syncthreads();
        I = sm.cut_found;
        __syncthreads();
    }
}

// The integer masses of log bucket beta: [wlo, wlo + 2^wbits).
__device__ __forceinline__ void bucket_w_range(int beta, unsigned long long& wlo, int& wbits) {
    if (beta < 16) {
        wlo = static_cast<unsigned long long>(beta);
        wbits = 0;
    } else {
        const int msb = 4 + (beta - 16) / 8, j = (beta - 16) % 8;
        wbits = msb - 3;
        wlo = static_cast<unsigned long long>(8 + j) << wbits;
    }
}

// The cut of cut_from_candidates without sorting the members: their masses
// lie in [wlo, wlo + 2^wbits); each level histograms the members still in
// play by the next 8 bits of the mass (counts and exact masses), and the
// sub-bucket where the running mass from the top crosses the target narrows
// the range, until one mass tau is left.  The cut is then the jneed-th member
// of mass tau in index order (jneed the fewest such entries whose mass
// reaches the target), found by a radix selection on the indices: the entry
// the sorted scan stops at.
__device__ void cut_by_radix(RowSmem& sm, unsigned int total, unsigned long long wlo, int wbits,
                             unsigned long long above_in, u128 TGT, RowInfo& info) {
    const int tid = threadIdx.x;
    unsigned long long lo = wlo, above = above_in, n_eq = total;
    int wb = wbits;
    while (wb > 0) {
        const int bits = wb < 8 ? wb : 8;
        const int shift = wb - bits;
        const unsigned long long hi = lo + (1ull << wb);
        for (int t = tid; t < kLinBuckets; t += kRowThreads) {
            sm.cnt[t] = 0u;
            sm.lmass[t] = 0ull;
        }
        __syncthreads();
        for (unsigned int t = tid; t < total; t += kRowThreads) {
            const unsigned long long W = sm.cw[t];
            if (W >= lo && W < hi) {
                const int bk = static_cast<int>((W - lo) >> shift);
                atomicAdd(&sm.cnt[bk], 1u);
                atomic_add_u64_split(&sm.lmass[bk], W);
            }
        }
        __syncthreads();
        const int t = (1 << bits) - 1 - tid;  // thread tid holds sub-bucket t, masses descending
        const unsigned long long mt = t >= 0 ? sm.lmass[t] : 0ull;
        u128 tot2;
        const u128 inc = block_excl_u128(static_cast<u128>(mt), sm.red, tot2) + mt;
        if (t >= 0 && ((above + inc) << 32) >= TGT && ((above + inc - mt) << 32) < TGT) {
            sm.lo = lo + (static_cast<unsigned long long>(t) << shift);
            sm.above = static_cast<unsigned long long>(above + inc - mt);
            sm.n_eq = sm.cnt[t];
        }
        __syncthreads();
        lo = sm.lo;
        above = sm.above;
        n_eq = sm.n_eq;
        wb = shift;
        __syncthreads();
    }
    const unsigned long long tau = lo;
    const u128 num = TGT - (static_cast<u128>(above) << 32);
    const u128 den = static_cast<u128>(tau) << 32;
    unsigned long long jneed = static_cast<unsigned long long>((num + den - 1) / den);
    if (jneed > n_eq) jneed = n_eq;  // (not reached: the crossing lies in this mass)
    // the jneed-th index among the members of mass tau: 8 bits a level
    unsigned int prefix = 0u;
    unsigned long long need = jneed;
    for (int sh = 16; sh >= 0; sh -= 8) {
        for (int t = tid; t < kLinBuckets; t += kRowThreads) sm.cnt[t] = 0u;
        __syncthreads();
        for (unsigned int t = tid; t < total; t += kRowThreads) {
            const unsigned int ix = static_cast<unsigned int>(sm.ci[t]);
            if (sm.cw[t] == tau && (ix >> (sh + 8)) == (prefix >> (sh + 8)))
                atomicAdd(&sm.cnt[(ix >> sh) & 255u], 1u);
        }
        __syncthreads();
        const unsigned long long ct = tid < kLinBuckets ? sm.cnt[tid] : 0u;  // ascending
        u128 tot3;
        const unsigned long long ex =
            static_cast<unsigned long long>(block_excl_u128(static_cast<u128>(ct), sm.red, tot3));
        if (tid < kLinBuckets && ex < need && need <= ex + ct) {
            sm.cut_found = tid;
            sm.count_eq = need - ex;
        }
        __syncthreads();
        prefix |= static_cast<unsigned int>(sm.cut_found) << sh;
        need = sm.count_eq;
        __syncthreads();
    }
    info.tau = tau;
    info.S = above + jneed * tau;
    info.cut = static_cast<int>(prefix);
}

// The cut inside the crossing bucket from its gathered members sm.cw / sm.ci
// (total <= kCutCand, in any order): sorted by (W desc, index asc), then the
// running mass from `above_in` down the list; the first entry whose running
// mass reaches TGT / 2^32 is the cut.  Sets info.tau, info.cut, info.S (valid
// in every thread).
__device__ void cut_from_candidates(RowSmem& sm, unsigned int total, unsigned long long above_in,
                                    u128 TGT, RowInfo& info, int beta) {
    const int tid = threadIdx.x;
    if (total > static_cast<unsigned int>(kRankSortMax)) {
        // many members: select the cut by radix instead of sorting them
        unsigned long long wlo;
        int wbits;
        bucket_w_range(beta, wlo, wbits);
        cut_by_radix(sm, total, wlo, wbits, above_in, TGT, info);
        return;
    }
    {
        // few: each candidate's place is the number that precede it
        unsigned long long wt = 0ull;
        int it = 0x7fffffff;
        unsigned int place = 0;
        if (static_cast<unsigned int>(tid) < total) {
            wt = sm.cw[tid];
            it = sm.ci[tid];
            for (unsigned int u = 0; u < total; ++u) {
                const unsigned long long wu = sm.cw[u];
                const int iu = sm.ci[u];
                place += (wu > wt || (wu == wt && iu < it)) ? 1u : 0u;
            }
        }
        __syncthreads();
        if (static_cast<unsigned int>(tid) < total) {
            sm.cw[place] = wt;
            sm.ci[place] = it;
        }
        __syncthreads();
    }
    // running mass down the sorted list; the first crossing is the cut
    constexpr int kCutPer = kCutCand / kRowThreads;  // candidates per thread
    const unsigned int t0 = kCutPer * tid;
    u128 part = 0;
    for (int j = 0; j < kCutPer; ++j)
        if (t0 + j < total) part += sm.cw[t0 + j];
    u128 tot;
    const u128 ex = block_excl_u128(part, sm.red, tot);
    const u128 above = above_in;
    u128 run = above + ex;
    for (int j = 0; j < kCutPer; ++j) {
        if (t0 + j >= total) break;
        const unsigned long long w = sm.cw[t0 + j];
        const u128 nxt = run + w;
        if ((nxt << 32) >= TGT && (run << 32) < TGT) {
            sm.info.tau = w;
            sm.info.cut = sm.ci[t0 + j];
            sm.info.S = static_cast<unsigned long long>(nxt);
        }
        run = nxt;
    }
    __syncthreads();
    info.tau = sm.info.tau;
    info.cut = sm.info.cut;
    info.S = sm.info.S;
}

// The row's (tau, cut, kept sum) after top-p, over the entries the top-k
// stage of info keeps (n_keep of them); valid in every thread.
__device__ RowInfo row_cut(const float* __restrict__ row, int V, bool vec, float invT,
                           unsigned long long P, const float* seg, RowInfo info, int n_keep,
                           RowSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float mx = info.mx;
    const bool topk = n_keep < V;

    // 2. sum W, and the mass histogram of the entries with W >= c0 (each warp
    //    its own copy).  The entries below c <= (1 - P/2^32) S / V weigh less
    //    than (1 - P/2^32) S together, so they all lie in the dropped tail;
    //    c0 uses a lower bound Slb of S in place of S, so c0 <= c and the
    //    histogram holds every bucket the cut can be in.  Slb is 2^40 (the top
    //    entry's own mass), or, with the segment maxima at hand and no top-k
    //    stage, the masses of the segment maxima (distinct entries) summed.
    const bool want_hist = P < kKeepAll;
    unsigned long long c0 = 0ull;
    if (want_hist) {
        unsigned long long Slb = 1ull << 40;
        if (seg != nullptr && !topk) {
            unsigned long long part = 0ull;
            for (int j = tid; j < n_segments(V); j += kRowThreads) {
                uint32_t hib, lob;
                mass_bits(own_exp_2_40(scaled_x(seg_load(seg + j), mx, invT)), hib, lob);
                part += (static_cast<unsigned long long>(hib - 0x4B000000u) << 20) +
                        (lob - 0x4B000000u);
            }
            const unsigned long long sum = block_sum_u64(part, sm.red);
            Slb = sum > Slb ? sum : Slb;  // (a non-finite max: every W is 0)
        }
        c0 = static_cast<unsigned long long>(static_cast<u128>(kKeepAll - P) * Slb /
                                             (static_cast<u128>(n_keep) << 32));
    }
    const unsigned long long cmin = c0 > 1ull ? c0 : 1ull;
    // f < f_lo proves W < cmin with one compare (f_lo is cmin rounded down)
    const float f_lo = want_hist ? __ull2float_rd(cmin) : INFINITY;
    unsigned long long* hist = sm.whist[wid];
    for (int t = lane; t < kLogBuckets; t += 32) hist[t] = 0ull;
    __syncwarp();
    // the two exact 20-bit halves of each W, summed as 2^23-biased bit
    // patterns (mod 2^32; the true sums stay below 2^32)
    uint32_t sum_hib = 0u, sum_lob = 0u;
    auto to_hist = [&](float f, uint32_t hib, uint32_t lob) {
        const unsigned long long W =
            (static_cast<unsigned long long>(hib - 0x4B000000u) << 20) | (lob - 0x4B000000u);
        if (W >= cmin) atomic_add_u64_split(&hist[log_bucket_f(f)], W);
    };
    uint32_t n_mine = 0u;  // entries this thread summed (the top-k path)
    if (topk) {
        // only the top-k entries carry mass: the segments that can hold one
        stream_segments<1>(row, V, vec, seg,
                        [&](float m) { return logit_key(m) >= info.tk_key; },
                        [&](int k, float l) {
                            if (!in_top_k(l, k, info)) return;
                            const float f = own_exp_2_40(scaled_x(l, mx, invT));
                            uint32_t hib, lob;
                            mass_bits(f, hib, lob);
                            sum_hib += hib;
                            sum_lob += lob;
                            ++n_mine;
                            if (f >= f_lo) to_hist(f, hib, lob);
                        });
    } else if (vec) {
        // two entries per packed operation; the histogram through the queues
        // (they share the candidate arrays, which are unused until step 3)
        __syncthreads();
        MassPass mp;
        mp.init(mx, invT, cmin, f_lo, hist, &sm.hq[wid][0][lane]);
        // float4 group k of this thread is r4[k * kRowThreads + tid]; the last
        // groups first: they left L2 least long ago in the max pass.  The
        // loop runs over k, the same for every lane of a warp.
        const float4* r4 = reinterpret_cast<const float4*>(row);
        const int V4 = V >> 2;
        const int nk = (V4 + kRowThreads - 1) / kRowThreads;
        static_assert(kHistGroup >= 16, "four float4 groups between checks");
        int k = nk - 1;
        {
            // the top group may be partial: entries past V4 are skipped
            const int i = k * kRowThreads + tid;
            if (i < V4) mp.quad(__ldg(r4 + i));
            mp.check();
            --k;
        }
        for (; k >= 3; k -= 4) {
            const int i = k * kRowThreads + tid;
            if (k >= 7) {  // the next four groups towards L2 while these are computed
                prefetch_l2(r4 + i - 4 * kRowThreads);
                prefetch_l2(r4 + i - 5 * kRowThreads);
                prefetch_l2(r4 + i - 6 * kRowThreads);
                prefetch_l2(r4 + i - 7 * kRowThreads);
            }
            const float4 a = __ldg(r4 + i), b = __ldg(r4 + i - kRowThreads),
                         c = __ldg(r4 + i - 2 * kRowThreads), d = __ldg(r4 + i - 3 * kRowThreads);
            mp.quad(a); mp.quad(b); mp.quad(c); mp.quad(d);
            mp.check();
        }
        for (; k >= 0; --k) {
            mp.quad(__ldg(r4 + k * kRowThreads + tid));
            mp.check();
        }
        mp.drain();
        sum_hib = mp.sum_hib;
        sum_lob = mp.sum_lob;
    } else {
        stream_row(row, V, vec, [&](int, float l) {
            const float f = own_exp_2_40(scaled_x(l, mx, invT));
            uint32_t hib, lob;
            mass_bits(f, hib, lob);
            sum_hib += hib;
            sum_lob += lob;
            if (f >= f_lo) to_hist(f, hib, lob);
        });
    }
    const uint32_t bias = (topk ? n_mine : stream_count(V, vec)) * 0x4B000000u;
    const unsigned long long S = block_sum_u64(
        (static_cast<unsigned long long>(sum_hib - bias) << 20) + (sum_lob - bias), sm.red);
    if (!want_hist) {
        info.cut = V - 1;
        info.tau = 0;
        info.S = S;
        return info;
    }
    if (S == 0ull) {
        // every W is 0 (the row's max is not finite: all -inf, or a +inf):
        // the kept prefix is the first entry in (W desc, index asc) order,
        // with mass 0
        info.cut = 0;
        info.tau = 0;
        info.S = 0;
        return info;
    }
    const u128 TGT = static_cast<u128>(P) * S;
    // merged bucket masses, then a block-wide suffix sum: the crossing bucket
    // beta is the highest bucket whose suffix mass reaches the target
    const int tb = kLogBuckets - 1 - tid;  // thread tid holds bucket 311 - tid
    unsigned long long m = 0;
    if (tb >= 1)
        for (int w = 0; w < kRowWarps; ++w) m += sm.whist[w][tb];
    u128 tot_unused;
    const u128 incl = block_excl_u128(static_cast<u128>(m), sm.red, tot_unused) + m;
    if (tid == 0) {
        sm.ncand = 0;
        sm.beta = -1;
    }
    __syncthreads();
    if (tb >= 1 && (incl << 32) >= TGT && ((incl - m) << 32) < TGT) {
        sm.beta = tb;
        sm.above = static_cast<unsigned long long>(incl - m);
    }
    __syncthreads();

    // 3. the members of the crossing bucket.  Members below c0 are not in the
    //    histogram but are gathered too; they are below the cut and sort
    //    after it, so the scan below never reaches them.
    const int beta = sm.beta;
    if (beta < 0) {  // not reached: the entries >= c0 hold at least P/2^32 of S
        info.cut = V - 1;
        info.tau = 0;
        info.S = S;
        return info;
    }
    float b_lo, b_hi;  // members of bucket beta: b_lo <= e < b_hi
    bucket_e_range(beta, b_lo, b_hi);
    {
        unsigned long long wlo, whi;
        if (beta < 16) {
            wlo = static_cast<unsigned long long>(beta);
            whi = wlo + 1ull;
        } else {
            const int msb = 4 + (beta - 16) / 8, j = (beta - 16) % 8;
            wlo = static_cast<unsigned long long>(8 + j) << (msb - 3);
            whi = static_cast<unsigned long long>(9 + j) << (msb - 3);
        }
        float xa, xb;
        x_window(wlo, whi, xa, xb);
        stream_window(row, V, vec, seg, mx, invT, xa, [&](int k, float l) {
            const float x = scaled_x(l, mx, invT);
            if (x >= xa && x < xb && in_top_k(l, k, info)) {
                const float e = own_exp(x);
                if (e >= b_lo && e < b_hi) {
                    const unsigned int slot = atomicAdd(&sm.ncand, 1u);
                    if (slot < static_cast<unsigned int>(kCutCand)) {
                        sm.cw[slot] = mass_of(e);
                        sm.ci[slot] = k;
                    }
                }
            }
        });
    }
    __syncthreads();
    const unsigned int total = sm.ncand;
    if (total <= static_cast<unsigned int>(kCutCand)) {
        cut_from_candidates(sm, total, sm.above, TGT, info, beta);
        return info;
    }

    // 4. fallback (a crowded bucket): exact radix search inside the bucket
    if (tid == 0) {
        if (beta < 16) {
            sm.lo = static_cast<unsigned long long>(beta);
            sm.width = 1;
            sm.wbits = 0;
            sm.n_eq = total;  // every member of an exact bucket has W == beta
        } else {
            const int msb = 4 + (beta - 16) / 8, j = (beta - 16) % 8;
            sm.wbits = msb - 3;
            sm.lo = static_cast<unsigned long long>(8 + j) << sm.wbits;
            sm.width = 1ull << sm.wbits;
            sm.n_eq = 0;
        }
    }
    __syncthreads();
    while (sm.width > 1ull) {
        const int wbits = sm.wbits;
        const int bits = wbits < 8 ? wbits : 8;
        const int shift = wbits - bits;
        const unsigned long long rlo = sm.lo, rhi = sm.lo + sm.width;
        for (int t = tid; t < kLinBuckets; t += kRowThreads) {
            sm.cnt[t] = 0u;
            sm.lmass[t] = 0ull;
        }
        __syncthreads();
        float xa, xb;
        x_window(rlo, rhi, xa, xb);
        stream_window(row, V, vec, seg, mx, invT, xa, [&](int k, float l) {
            const float x = scaled_x(l, mx, invT);
            if (x >= xa && x < xb && in_top_k(l, k, info)) {
                const unsigned long long W = mass_of(own_exp(x));
                if (W >= rlo && W < rhi) {
                    const int bk = static_cast<int>((W - rlo) >> shift);
                    atomicAdd(&sm.cnt[bk], 1u);
                    atomic_add_u64_split(&sm.lmass[bk], W);
                }
            }
        });
        __syncthreads();
        {
            const int nb = 1 << bits;
            const int t = nb - 1 - tid;  // thread tid holds sub-bucket nb - 1 - tid
            const unsigned long long mt = t >= 0 ? sm.lmass[t] : 0ull;
            u128 tot2;
            const u128 inc = block_excl_u128(static_cast<u128>(mt), sm.red, tot2) + mt;
            const u128 ab = static_cast<u128>(sm.above);
            if (t >= 0 && ((ab + inc) << 32) >= TGT && ((ab + inc - mt) << 32) < TGT) {
                sm.beta = t;
                sm.lo = rlo + (static_cast<unsigned long long>(t) << shift);
                sm.n_eq = sm.cnt[t];
                sm.count_eq = static_cast<unsigned long long>(ab + inc - mt);
            }
            __syncthreads();
            if (tid == 0) {
                sm.above = sm.count_eq;
                sm.width = 1ull << shift;
                sm.wbits = shift;
            }
            __syncthreads();
        }
    }
    const unsigned long long tau = sm.lo, above = sm.above, n_eq = sm.n_eq;
    // smallest j >= 1 with (above + j*tau) * 2^32 >= P*S
    const u128 num = TGT - (static_cast<u128>(above) << 32);
    const u128 den = static_cast<u128>(tau) << 32;
    const unsigned long long jneed = static_cast<unsigned long long>((num + den - 1) / den);
    info.tau = tau;
    info.S = above + jneed * tau;
    info.cut = V - 1;
    if (jneed < n_eq) {
        // the jneed-th entry with W == tau in index order sets the cut: each
        // thread counts its contiguous chunk, a block scan orders the chunks
        const int chunk = (V + kRowThreads - 1) / kRowThreads;
        const int k0 = tid * chunk, k1 = (k0 + chunk < V) ? k0 + chunk : V;
        float xa, xb;
        x_window(tau, tau + 1ull, xa, xb);
        auto is_tau = [&](int k) {
            const float l = __ldg(row + k);
            const float x = scaled_x(l, mx, invT);
            return x >= xa && x < xb && mass_of(own_exp(x)) == tau && in_top_k(l, k, info);
        };
        unsigned int mine = 0;
        for (int k = k0; k < k1; ++k) mine += is_tau(k) ? 1u : 0u;
        u128 ctot;
        const unsigned long long excl = static_cast<unsigned long long>(
            block_excl_u128(static_cast<u128>(mine), sm.red, ctot));
        if (tid == 0) sm.cut_found = -1;
        __syncthreads();
        if (excl < jneed && jneed <= excl + mine) {
            unsigned long long seen = excl;
            for (int k = k0; k < k1; ++k)
                if (is_tau(k) && ++seen == jneed) {
                    sm.cut_found = k;
                    break;
                }
        }
        __syncthreads();
        info.cut = sm.cut_found;
    }
    return info;
}

// The row's RowInfo through the whole pipeline: max, top-k (0 or >= V: off),
// the integer masses, top-p, min-p (MP = round(min_p 2^32), 0: off);
// valid in every thread.  seg: this row's segment maxima (vec rows), or null.
__device__ RowInfo row_stats(const float* __restrict__ row, int V, bool vec, float invT,
                             unsigned long long P, int top_k, unsigned long long MP, float* seg,
                             const float* bm, RowSmem& sm) {
    RowInfo info;
    info.mx = bm != nullptr ? row_max_from_blocks(bm, V, seg, sm) : row_max(row, V, vec, seg, sm);
    info.tk_key = 0u;
    info.tk_idx = 0x7fffffff;
    info.tau = 0ull;
    info.cut = V - 1;
    info.S = 0ull;
    const bool topk = top_k > 0 && top_k < V;
    // the later passes read the segment maxima from shared memory when the
    // row has few enough segments (the max pass wrote both copies)
    const float* segr = (seg != nullptr && n_segments(V) <= kSegCache) ? sm.segc : seg;
    if (topk) top_k_cut(row, V, vec, segr, top_k, sm, info.tk_key, info.tk_idx);
    RowInfo r = row_cut(row, V, vec, invT, P, segr, info, topk ? top_k : V, sm);
    // min-p: of what top-p keeps, only W * 2^32 >= MP * W_top, W_top = 2^40
    // (the max entry's own mass), i.e. W >= MP * 2^8.  Both keep a prefix of
    // the (W desc, index asc) order: when min-p's is the shorter, it is every
    // entry with W >= MP 2^8, ties included.
    if (MP > 0ull && r.S > 0ull) {
        const unsigned long long Wmin = MP << 8;
        if (Wmin > r.tau) {
            float xa, xb;
            x_window(Wmin, Wmin + 1ull, xa, xb);
            const float mx = r.mx;
            unsigned long long part = 0ull;
            stream_window<1>(row, V, vec, segr, mx, invT, xa, [&](int k, float l) {
                const float x = scaled_x(l, mx, invT);
                if (x >= xa && in_top_k(l, k, r)) {
                    const unsigned long long W = mass_of(own_exp(x));
                    if (W >= Wmin) part += W;
                }
            });
            r.S = block_sum_u64(part, sm.red);
            r.tau = Wmin;
            r.cut = V - 1;
        }
    }
    return r;
}

// ------------------------------------------------------------- row kernel
// Rows 0 .. B(Kd+1)-1 are the target rows (b, i) in order, then the B*Kd
// draft rows (b, i).
__global__ void __launch_bounds__(kRowThreads, 2) row_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, long long n_target_rows,
    int V, int vec_ok, float invT, unsigned long long P, int top_k, unsigned long long MP,
    RowInfo* __restrict__ info, float* __restrict__ segmax, const float* __restrict__ tbm,
    const float* __restrict__ dbm) {
    extern __shared__ float4 dyn[];
    RowSmem& sm = *reinterpret_cast<RowSmem*>(dyn);
    const long long row = blockIdx.x;
    const float* src = row < n_target_rows
                           ? target + row * static_cast<long long>(V)
                           : draft + (row - n_target_rows) * static_cast<long long>(V);
    // block maxima handed over by the GEMM that wrote the logits, if any
    const long long nb = (V + kBlockLen - 1) / kBlockLen;
    const float* bm = row < n_target_rows ? (tbm ? tbm + row * nb : nullptr)
                                          : (dbm ? dbm + (row - n_target_rows) * nb : nullptr);
    float* seg = vec_ok ? segmax + row * static_cast<long long>(n_segments(V)) : nullptr;
    const RowInfo r = row_stats(src, V, vec_ok != 0, invT, P, top_k, MP, seg, bm, sm);
    if (threadIdx.x == 0) info[row] = r;
}

// ------------------------------------------------------- split rows
// With few logits rows (a handful of sequences, e.g. one sequence of an
// LM-head verify) one CTA per row leaves most SMs idle, and each CTA streams
// its whole row several times.  Then every row is cut into C chunks of whole
// 128-entry segments, one CTA per (row, chunk), and the row statistics are
// taken in five launches: the chunk maxima; the chunks' integer mass sums and
// mass histograms (exact integers, so their sums over the chunks are exact
// and order-free); the crossing bucket of the top-p cut per row; the members
// of that bucket gathered from every chunk; and the cut among them.  The
// records are exactly those of the one-CTA row kernel (same masses, same
// cut); a bucket with more than kCutCand members falls back to that kernel's
// code for its row.
// Chained launches: a kernel launched with launch_dependent() is a
// programmatic dependent of the work before it on the stream, launched as
// that grid's blocks exit rather than after the whole grid has retired.
// pdl_start(), the first statement of every such kernel, waits until the
// previous grid has finished and its writes are visible, so nothing is read
// or written early.  (Launched the ordinary way, the wait returns at once.)
// Releasing the next kernel earlier, at the start of each kernel, measured
// slower (one sequence, 7 drafts, V = 262144: 100.8 us against 92.6).
__device__ __forceinline__ void pdl_start() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kSplitRowsMax = 152;   // more rows than this: one CTA per row
constexpr int kSplitMinV = 16384;    // shorter rows: one CTA per row
constexpr int kSplitSlots = 304;     // (row, chunk) CTAs per call

struct SplitState {
    int beta;                 // crossing bucket, or -1 when the record is final
    int pad;
    unsigned long long above; // kept mass above the bucket
    unsigned long long S;     // the row's whole mass (top-p off: the kept sum)
    unsigned long long pad2;
};

__host__ __device__ inline int split_chunks(long long rows) {
    const long long c = kSplitSlots / (rows > 0 ? rows : 1);
    return static_cast<int>(c < 2 ? 2 : (c > 64 ? 64 : c));
}

struct SplitWs {
    float* chunkmax;               // [rows][C]
    unsigned long long* pS;        // [rows][C]
    unsigned long long* phist;     // [rows][C][kLogBuckets]
    SplitState* state;             // [rows]
    uint32_t* ncand;               // [rows]
    unsigned long long* cw;        // [rows][kCutCand]
    int* ci;                       // [rows][kCutCand]
    ulonglong2* chunk_tot;         // [sequences][C] draw weight of each chunk (u128)
    size_t bytes;
};

static size_t r256(size_t x) { return (x + 255) / 256 * 256; }

static SplitWs split_layout(char* base, long long rows) {
    SplitWs w{};
    const int C = split_chunks(rows);
    size_t off = 0;
    auto take = [&](size_t b) {
        char* p = base ? base + off : nullptr;
        off += r256(b);
        return p;
    };
    w.chunkmax = reinterpret_cast<float*>(take(rows * C * sizeof(float)));
    w.pS = reinterpret_cast<unsigned long long*>(take(rows * C * 8));
    w.phist = reinterpret_cast<unsigned long long*>(take(rows * C * kLogBuckets * 8));
    w.state = reinterpret_cast<SplitState*>(take(rows * sizeof(SplitState)));
    w.ncand = reinterpret_cast<uint32_t*>(take(rows * 4));
    w.cw = reinterpret_cast<unsigned long long*>(take(rows * kCutCand * 8));
    w.ci = reinterpret_cast<int*>(take(rows * kCutCand * 4));
    w.chunk_tot = reinterpret_cast<ulonglong2*>(take(rows * 64 * sizeof(ulonglong2)));
    w.bytes = off;
    return w;
}

// Row r's logits: the target rows (b, i <= Kd) first, then the draft rows.
__device__ __forceinline__ const float* split_row(const float* target, const float* draft,
                                                  long long n_target_rows, long long r, int V) {
    return r < n_target_rows ? target + r * static_cast<long long>(V)
                             : draft + (r - n_target_rows) * static_cast<long long>(V);
}

// Segments [s0, s1) of chunk c of a row of nseg segments.
__device__ __forceinline__ void split_span(int nseg, int C, int c, int& s0, int& s1) {
    const int spc = (nseg + C - 1) / C;
    s0 = c * spc;
    s1 = min(s0 + spc, nseg);
    if (s0 > nseg) s0 = nseg;
}

// 1. Chunk maxima and the maxima of the chunk's segments (the max pass of
//    row_max, segment by segment: a warp takes a segment, a lane one float4
//    group); with block maxima given, from those.
__global__ void __launch_bounds__(kRowThreads) split_max_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, long long n_target_rows,
    int V, int C, const float* __restrict__ tbm, const float* __restrict__ dbm,
    float* __restrict__ segmax, float* __restrict__ chunkmax) {
    pdl_start();
    __shared__ Red red;
    const long long r = blockIdx.x / C;
    const int c = blockIdx.x % C;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nseg = n_segments(V), V4 = V >> 2;
    int s0, s1;
    split_span(nseg, C, c, s0, s1);
    float* seg = segmax + r * nseg;
    const long long nb = (V + kBlockLen - 1) / kBlockLen;
    const float* bm = r < n_target_rows ? (tbm ? tbm + r * nb : nullptr)
                                        : (dbm ? dbm + (r - n_target_rows) * nb : nullptr);
    float lmax = -INFINITY;
    if (bm != nullptr) {
        constexpr int kPer = kSegLen / kBlockLen;
        for (int sg = s0 + tid; sg < s1; sg += kRowThreads) {
            float m = -INFINITY;
            const int b1 = min((sg + 1) * kPer, static_cast<int>(nb));
            for (int bk = sg * kPer; bk < b1; ++bk) m = fmaxf(m, __ldg(bm + bk));
            seg[sg] = m;
            lmax = fmaxf(lmax, m);
        }
    } else {
        const float4* r4 = reinterpret_cast<const float4*>(split_row(target, draft, n_target_rows,
                                                                     r, V));
        const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        for (int sg0 = s0 + wid; sg0 < s1; sg0 += 4 * kRowWarps) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int sg = sg0 + j * kRowWarps, i = sg * 32 + lane;
                v[j] = (sg < s1 && i < V4) ? __ldg(r4 + i) : ninf;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int sg = sg0 + j * kRowWarps;
                if (sg >= s1) break;  // the same for the whole warp
                const float m = fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w));
                lmax = fmaxf(lmax, m);
                const int key = __reduce_max_sync(0xffffffffu, float_key(m));
                if (lane == 0) seg[sg] = __int_as_float(key ^ ((key >> 31) & 0x7fffffff));
            }
        }
    }
    const float m = block_max(lmax, red);
    if (tid == 0) chunkmax[r * C + c] = m;
}

// 2. The chunk's mass sum and mass histogram: the integer masses W of
//    row_cut's second pass, entry for entry the same operations; the sums are
//    exact, so the row's are their sums over the chunks.
__global__ void __launch_bounds__(kRowThreads, 2) split_mass_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, long long n_target_rows,
    int V, int C, float invT, unsigned long long P, const float* __restrict__ chunkmax,
    unsigned long long* __restrict__ pS, unsigned long long* __restrict__ phist) {
    pdl_start();
    extern __shared__ float4 dyn[];
    RowSmem& sm = *reinterpret_cast<RowSmem*>(dyn);
    const long long r = blockIdx.x / C;
    const int c = blockIdx.x % C;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nseg = n_segments(V), V4 = V >> 2;
    int s0, s1;
    split_span(nseg, C, c, s0, s1);
    float mx = -INFINITY;
    for (int j = 0; j < C; ++j) mx = fmaxf(mx, __ldg(chunkmax + r * C + j));
    const bool want_hist = P < kKeepAll;
    const unsigned long long c0 =
        want_hist ? ((kKeepAll - P) << 8) / static_cast<unsigned long long>(V) : 0ull;
    const unsigned long long cmin = c0 > 1ull ? c0 : 1ull;
    const float f_lo = want_hist ? __ull2float_rd(cmin) : INFINITY;
    unsigned long long* hist = sm.whist[wid];
    for (int t = lane; t < kLogBuckets; t += 32) hist[t] = 0ull;
    __syncwarp();
    MassPass mp;
    mp.init(mx, invT, cmin, f_lo, hist, &sm.hq[wid][0][lane]);
    const float4* r4 = reinterpret_cast<const float4*>(split_row(target, draft, n_target_rows, r, V));
    static_assert(kHistGroup >= 16, "four float4 groups between checks");
    for (int sg0 = s0 + wid; sg0 < s1; sg0 += 4 * kRowWarps) {  // the same for a warp's lanes
        float4 v[4];
        bool in[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int sg = sg0 + j * kRowWarps, i = sg * 32 + lane;
            in[j] = sg < s1 && i < V4;
            v[j] = in[j] ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (in[j]) mp.quad(v[j]);
        mp.check();
    }
    mp.drain();
    const unsigned long long S = block_sum_u64(mp.sum(), sm.red);
    __syncthreads();  // every warp's histogram is complete
    unsigned long long* out = phist + (r * C + c) * kLogBuckets;
    for (int t = tid; t < kLogBuckets; t += kRowThreads) {
        unsigned long long m = 0ull;
        for (int w = 0; w < kRowWarps; ++w) m += sm.whist[w][t];
        out[t] = m;
    }
    if (tid == 0) pS[r * C + c] = S;
}

// 3. Per row: the mass S, the merged histogram and the bucket where the
//    top-p cut falls, as row_cut finds them; a row whose record is already
//    decided (top-p off, all masses 0, or the cut at the last entry) gets it.
__global__ void __launch_bounds__(kRowThreads, 2) split_beta_kernel(
    int V, int C, unsigned long long P, const float* __restrict__ chunkmax,
    const unsigned long long* __restrict__ pS, const unsigned long long* __restrict__ phist,
    RowInfo* __restrict__ info_out, SplitState* __restrict__ state, uint32_t* __restrict__ ncand) {
    pdl_start();
    extern __shared__ float4 dyn[];
    RowSmem& sm = *reinterpret_cast<RowSmem*>(dyn);
    const long long r = blockIdx.x;
    const int tid = threadIdx.x;
    float mx = -INFINITY;
    for (int j = 0; j < C; ++j) mx = fmaxf(mx, __ldg(chunkmax + r * C + j));
    unsigned long long s = 0ull;
    for (int j = tid; j < C; j += kRowThreads) s += pS[r * C + j];
    const unsigned long long S = block_sum_u64(s, sm.red);
    RowInfo info;
    info.mx = mx;
    info.tk_key = 0u;
    info.tk_idx = 0x7fffffff;
    info.tau = 0ull;
    info.cut = V - 1;
    info.S = S;
    int beta = -1;
    unsigned long long above = 0ull;
    if (P < kKeepAll && S == 0ull) {
        info.cut = 0;  // every W is 0: the prefix is the first entry, mass 0
    } else if (P < kKeepAll) {
        const u128 TGT = static_cast<u128>(P) * S;
        const int tb = kLogBuckets - 1 - tid;
        unsigned long long m = 0ull;
        if (tb >= 1)
            for (int j = 0; j < C; ++j) m += phist[(r * C + j) * kLogBuckets + tb];
        u128 tot_unused;
        const u128 incl = block_excl_u128(static_cast<u128>(m), sm.red, tot_unused) + m;
        if (tid == 0) sm.beta = -1;
        __syncthreads();
        if (tb >= 1 && (incl << 32) >= TGT && ((incl - m) << 32) < TGT) {
            sm.beta = tb;
            sm.above = static_cast<unsigned long long>(incl - m);
        }
        __syncthreads();
        beta = sm.beta;
        above = sm.above;
    }
    if (tid == 0) {
        SplitState st{};
        st.beta = beta;
        st.above = above;
        st.S = S;
        state[r] = st;
        ncand[r] = 0u;
        if (beta < 0) info_out[r] = info;
    }
}

// 4. The members of the crossing bucket, from every chunk (the window pass
//    of row_cut, over the chunk's segments whose max reaches the window).
__global__ void __launch_bounds__(kRowThreads) split_gather_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, long long n_target_rows,
    int V, int C, float invT, const float* __restrict__ segmax, const float* __restrict__ chunkmax,
    const SplitState* __restrict__ state, uint32_t* __restrict__ ncand,
    unsigned long long* __restrict__ cw, int* __restrict__ ci) {
    pdl_start();
    const long long r = blockIdx.x / C;
    const int c = blockIdx.x % C;
    const int beta = state[r].beta;
    if (beta < 0) return;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nseg = n_segments(V), V4 = V >> 2;
    int s0, s1;
    split_span(nseg, C, c, s0, s1);
    float mx = -INFINITY;
    for (int j = 0; j < C; ++j) mx = fmaxf(mx, __ldg(chunkmax + r * C + j));
    float b_lo, b_hi;
    bucket_e_range(beta, b_lo, b_hi);
    unsigned long long wlo, whi;
    if (beta < 16) {
        wlo = static_cast<unsigned long long>(beta);
        whi = wlo + 1ull;
    } else {
        const int msb = 4 + (beta - 16) / 8, j = (beta - 16) % 8;
        wlo = static_cast<unsigned long long>(8 + j) << (msb - 3);
        whi = static_cast<unsigned long long>(9 + j) << (msb - 3);
    }
    float xa, xb;
    x_window(wlo, whi, xa, xb);
    const float* seg = segmax + r * nseg;
    const float4* r4 = reinterpret_cast<const float4*>(split_row(target, draft, n_target_rows, r, V));
    // four segments of the warp at a time, their loads first (a segment whose
    // max lies below the window holds no member)
    for (int sg0 = s0 + wid; sg0 < s1; sg0 += 4 * kRowWarps) {
        float4 v[4];
        bool in[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int sg = sg0 + j * kRowWarps, i = sg * 32 + lane;
            in[j] = sg < s1 && i < V4 && !(scaled_x(__ldcg(seg + sg), mx, invT) < xa);
            v[j] = in[j] ? __ldg(r4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (!in[j]) continue;
            const int i = (sg0 + j * kRowWarps) * 32 + lane;
            const float lv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x = scaled_x(lv[q], mx, invT);
                if (x >= xa && x < xb) {
                    const float e = own_exp(x);
                    if (e >= b_lo && e < b_hi) {
                        const unsigned int slot = atomicAdd(&ncand[r], 1u);
                        if (slot < static_cast<unsigned int>(kCutCand)) {
                            cw[r * kCutCand + slot] = mass_of(e);
                            ci[r * kCutCand + slot] = 4 * i + q;
                        }
                    }
                }
            }
        }
    }
}

// 5. Per row: the cut among the gathered members (or, for a bucket with more
//    than kCutCand members, the one-CTA row statistics of that row).
__global__ void __launch_bounds__(kRowThreads, 2) split_cut_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, long long n_target_rows,
    int V, int C, float invT, unsigned long long P, float* __restrict__ segmax,
    const float* __restrict__ chunkmax, const SplitState* __restrict__ state,
    const uint32_t* __restrict__ ncand, const unsigned long long* __restrict__ cw,
    const int* __restrict__ ci, RowInfo* __restrict__ info_out) {
    pdl_start();
    extern __shared__ float4 dyn[];
    RowSmem& sm = *reinterpret_cast<RowSmem*>(dyn);
    const long long r = blockIdx.x;
    const SplitState st = state[r];
    if (st.beta < 0) return;
    const int tid = threadIdx.x;
    const unsigned int total = ncand[r];
    RowInfo info;
    if (total <= static_cast<unsigned int>(kCutCand)) {
        float mx = -INFINITY;
        for (int j = 0; j < C; ++j) mx = fmaxf(mx, __ldg(chunkmax + r * C + j));
        for (unsigned int t = tid; t < total; t += kRowThreads) {
            sm.cw[t] = cw[r * kCutCand + t];
            sm.ci[t] = ci[r * kCutCand + t];
        }
        __syncthreads();
        info.mx = mx;
        info.tk_key = 0u;
        info.tk_idx = 0x7fffffff;
        const u128 TGT = static_cast<u128>(P) * st.S;
        cut_from_candidates(sm, total, st.above, TGT, info, st.beta);
    } else {
        const float* row = split_row(target, draft, n_target_rows, r, V);
        info = row_stats(row, V, true, invT, P, 0, 0ull, segmax + r * n_segments(V), nullptr, sm);
    }
    if (tid == 0) info_out[r] = info;
}

// --------------------------------------------------------- sequence kernel
// Weight of entry v in the draw: the kept target mass (p), or the residual
// max(0, p_v * Sq - q_v * Sp).  Entries whose scaled logit is below xth have
// a kept target mass of 0 (own_exp is monotone and within 2 ulp of exp, and
// xth sits 1e-3 below log(max(tau, 1) / 2^40)), so they cost two flops.
struct DrawRow {
    const float* lp;
    const float* lq;  // null: draw from p
    const float* sp;  // segment maxima of the p row (vec rows), or null
    RowInfo ip, iq;
    float invT, xth;
    int V;
    bool vec;
    __device__ __forceinline__ u128 weight(int v, float lpv, float lqv) const {
        const float xp = scaled_x(lpv, ip.mx, invT);
        if (xp < xth) return 0;
        const unsigned long long wp = kept(mass_of(own_exp(xp)), lpv, v, ip);
        if (lq == nullptr || wp == 0ull) return static_cast<u128>(wp);
        const unsigned long long wq =
            kept(mass_of(own_exp(scaled_x(lqv, iq.mx, invT))), lqv, v, iq);
        const u128 a = static_cast<u128>(wp) * iq.S, c = static_cast<u128>(wq) * ip.S;
        return a > c ? a - c : static_cast<u128>(0);
    }
    // The logits of entries v .. v+3 (v % 4 == 0; entries >= V read as -inf,
    // which weighs 0).
    __device__ __forceinline__ void load4(int v, float4& p, float4& q) const {
        const float ninf = -INFINITY;
        q = make_float4(ninf, ninf, ninf, ninf);
        if (vec) {  // V % 4 == 0 and 16-byte aligned rows
            p = v < V ? __ldg(reinterpret_cast<const float4*>(lp + v)) : q;
            if (lq != nullptr && v < V) q = __ldg(reinterpret_cast<const float4*>(lq + v));
            return;
        }
        p = make_float4(v < V ? __ldg(lp + v) : ninf, v + 1 < V ? __ldg(lp + v + 1) : ninf,
                        v + 2 < V ? __ldg(lp + v + 2) : ninf, v + 3 < V ? __ldg(lp + v + 3) : ninf);
        if (lq != nullptr)
            q = make_float4(v < V ? __ldg(lq + v) : ninf, v + 1 < V ? __ldg(lq + v + 1) : ninf,
                            v + 2 < V ? __ldg(lq + v + 2) : ninf,
                            v + 3 < V ? __ldg(lq + v + 3) : ninf);
    }
    __device__ __forceinline__ void weights4(int v, const float4& p, const float4& q,
                                             u128 w[4]) const {
        w[0] = weight(v, p.x, q.x);
        w[1] = weight(v + 1, p.y, q.y);
        w[2] = weight(v + 2, p.z, q.z);
        w[3] = weight(v + 3, p.w, q.w);
    }
    // false: every entry of segment s weighs 0 (its max is below xth)
    __device__ __forceinline__ bool may_weigh(int s) const {
        return sp == nullptr || !(scaled_x(__ldg(sp + s), ip.mx, invT) < xth);
    }
};

// A warp's queue of the entries of one batch of segments that may weigh
// (scaled logit >= xth): a few per batch, so their weights are computed one
// per lane instead of in divergent per-slot passes.
constexpr int kQueue = 64;
struct WarpQueue {
    int v[kQueue];
    float lp[kQueue], lq[kQueue];
    unsigned char slot[kQueue];
    unsigned long long acc[4][2];  // the batch's segment sums (lo, hi)
};

struct SeqSmem {
    WarpQueue q[kWarps];
    Red red;
    unsigned long long tot_lo[kWarps], tot_hi[kWarps];
    unsigned long long u64s[kMaxRows + 1];
    int ok[kMaxRows + 1];
    int n_acc, rowp, rowq, sel, token, seg;
    unsigned long long u64;
    unsigned long long t_lo, t_hi;  // the draw point, then its offset inside segment seg
};

// Exact 128-bit add into shared memory: 64-bit atomics, the low word's carry
// to the high word.
__device__ __forceinline__ void atomic_add_u128(unsigned long long* a, u128 x) {
    const unsigned long long lo = static_cast<unsigned long long>(x);
    const unsigned long long hi = static_cast<unsigned long long>(x >> 64);
    const unsigned long long old = atomicAdd(&a[0], lo);
    const unsigned long long h = hi + (old + lo < old ? 1ull : 0ull);
    if (h) atomicAdd(&a[1], h);
}

// Level 1 of the draw: warp wid sums the weights of each segment of its run
// of segments into ssum[] (zero for the segments that cannot weigh) and
// returns the run's total (in lane 0).
// (Segments [s_begin, s_end) of the row; the whole row by default.)
__device__ __forceinline__ u128 segment_sums(const DrawRow& w, ulonglong2* ssum, WarpQueue& wq,
                                             int wid, int lane, int s_begin = 0,
                                             int s_end = -1) {
    if (s_end < 0) s_end = n_segments(w.V);
    const long long span = s_end - s_begin;
    const int s_lo = s_begin + static_cast<int>(static_cast<long long>(wid) * span / kWarps);
    const int s_hi = s_begin + static_cast<int>(static_cast<long long>(wid + 1) * span / kWarps);
    u128 tot = 0;
    for (int s0 = s_lo; s0 < s_hi; s0 += 32) {
        const int s = s0 + lane;
        const bool need = s < s_hi && w.may_weigh(s);
        if (s < s_hi && !need) __stcg(ssum + s, make_ulonglong2(0ull, 0ull));
        unsigned int m = __ballot_sync(0xffffffffu, need);
        while (m) {
            // up to four marked segments at a time, their loads first
            const int n = __popc(m) < 4 ? __popc(m) : 4;
            int sj[4];
            float4 p[4], q[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                sj[j] = s0 + static_cast<int>(__fns(m, 0, j < n ? j + 1 : 1));
                w.load4(sj[j] * kSegLen + 4 * lane, p[j], q[j]);
            }
            // the entries that may weigh: bit 4 j + e of fl for entry e of segment j
            uint32_t fl = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < n) {
                    fl |= (scaled_x(p[j].x, w.ip.mx, w.invT) < w.xth ? 0u : 1u) << (4 * j);
                    fl |= (scaled_x(p[j].y, w.ip.mx, w.invT) < w.xth ? 0u : 2u) << (4 * j);
                    fl |= (scaled_x(p[j].z, w.ip.mx, w.invT) < w.xth ? 0u : 4u) << (4 * j);
                    fl |= (scaled_x(p[j].w, w.ip.mx, w.invT) < w.xth ? 0u : 8u) << (4 * j);
                }
            }
            const int c = __popc(fl);
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int K = __shfl_sync(0xffffffffu, incl, 31);
            if (K <= kQueue) {
                int pos = incl - c;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float pv[4] = {p[j].x, p[j].y, p[j].z, p[j].w};
                    const float qv[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if ((fl >> (4 * j + e)) & 1u) {
                            wq.v[pos] = sj[j] * kSegLen + 4 * lane + e;
                            wq.lp[pos] = pv[e];
                            wq.lq[pos] = qv[e];
                            wq.slot[pos] = static_cast<unsigned char>(j);
                            ++pos;
                        }
                    }
                }
                if (lane < 8) (&wq.acc[0][0])[lane] = 0ull;
                __syncwarp();
                for (int r = lane; r < K; r += 32)
                    atomic_add_u128(wq.acc[wq.slot[r]], w.weight(wq.v[r], wq.lp[r], wq.lq[r]));
                __syncwarp();
            } else {
                // a crowded batch: every entry through the slot-by-slot path
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j >= n) break;
                    u128 e[4];
                    w.weights4(sj[j] * kSegLen + 4 * lane, p[j], q[j], e);
                    const u128 seg = warp_sum_u128(e[0] + e[1] + e[2] + e[3]);
                    if (lane == 0) {
                        wq.acc[j][0] = static_cast<unsigned long long>(seg);
                        wq.acc[j][1] = static_cast<unsigned long long>(seg >> 64);
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j >= n) break;
                    const unsigned long long lo = wq.acc[j][0], hi = wq.acc[j][1];
                    __stcg(ssum + sj[j], make_ulonglong2(lo, hi));
                    tot += (static_cast<u128>(hi) << 64) | lo;
                }
            }
            __syncwarp();
            for (int j = 0; j < n; ++j) m &= m - 1;
        }
    }
    return tot;
}

// One CTA per sequence: acceptance tests in order, then one ordered draw and
// the committed run.
// (Two CTAs per SM: 256 sequences fit one wave.)
// The sequence's acceptance tests (thread i < Kd takes draft i, in
// parallel) and the run they decide: sm.n_acc accepted drafts, the rows of
// the draw (sm.rowp, and sm.rowq for a residual, -1 for the bonus) and its
// 64-bit uniform sm.u64.  Every thread of the block calls it.
__device__ void seq_decide(const float* __restrict__ target, const float* __restrict__ draft,
                           const int32_t* __restrict__ drafts, int Kd, int V, float invT,
                           unsigned long long seed, unsigned long long offset,
                           long long n_target_rows, const RowInfo* __restrict__ info, int b,
                           uint32_t* status, SeqSmem& sm) {
    const int tid = threadIdx.x;
    if (tid <= Kd) {
        const int i = tid;
        uint32_t rr[4];
        philox4x32_10(static_cast<uint32_t>(i), static_cast<uint32_t>(b),
                      static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
                      static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), rr);
        sm.u64s[i] = (static_cast<unsigned long long>(rr[2]) << 32) | rr[1];
        int ok = 1;  // position Kd: the bonus
        if (i < Kd) {
            const long long rp = static_cast<long long>(b) * (Kd + 1) + i;
            const long long rq = n_target_rows + static_cast<long long>(b) * Kd + i;
            const RowInfo ip = info[rp], iq = info[rq];
            const int32_t x = drafts[static_cast<long long>(b) * Kd + i];
            ok = 0;
            if (x >= 0 && x < V) {
                const float lpx = target[rp * V + x];
                const float lqx = draft[(rq - n_target_rows) * V + x];
                const unsigned long long Wp =
                    kept(mass_of(own_exp(scaled_x(lpx, ip.mx, invT))), lpx, x, ip);
                const unsigned long long Wq =
                    kept(mass_of(own_exp(scaled_x(lqx, iq.mx, invT))), lqx, x, iq);
                const unsigned long long U = rr[0] >> 8;
                const u128 lhs = static_cast<u128>(U * Wq) * ip.S;
                const u128 rhs = (static_cast<u128>(Wp) * iq.S) << 24;
                ok = lhs < rhs ? 1 : 0;
            } else {
                atomicOr(status, kStatusBadDraft);
            }
        }
        sm.ok[i] = ok;
    }
    __syncthreads();
    if (tid == 0) {  // the first rejection decides the run
        int n = 0;
        while (n < Kd && sm.ok[n]) ++n;
        sm.n_acc = n;
        sm.rowp = b * (Kd + 1) + n;
        sm.rowq = n < Kd ? static_cast<int>(n_target_rows + static_cast<long long>(b) * Kd + n) : -1;
        sm.u64 = sm.u64s[n];
        sm.token = -1;
        sm.seg = -1;
    }
    __syncthreads();
}

// The row the draw weighs: the kept target masses p (the bonus), or the
// residual max(0, p Sq - q Sp) at the first rejection.
__device__ DrawRow seq_draw_row(const float* __restrict__ target, const float* __restrict__ draft,
                                int V, int vec_ok, float invT, long long n_target_rows,
                                const RowInfo* __restrict__ info,
                                const float* __restrict__ segmax, const SeqSmem& sm) {
    const int rowp = sm.rowp, rowq = sm.rowq;
    const int nseg = n_segments(V);
    DrawRow w;
    w.ip = info[rowp];
    w.lp = target + static_cast<long long>(rowp) * V;
    w.sp = vec_ok ? segmax + static_cast<long long>(rowp) * nseg : nullptr;
    w.lq = nullptr;
    if (rowq >= 0) {
        w.iq = info[rowq];
        w.lq = draft + (rowq - n_target_rows) * static_cast<long long>(V);
    }
    w.invT = invT;
    w.V = V;
    w.vec = vec_ok != 0;
    const unsigned long long tm = w.ip.tau > 1ull ? w.ip.tau : 1ull;
    w.xth = static_cast<float>(log(static_cast<double>(tm)) - 40.0 * 0.69314718055994530942 -
                               1e-3);
    return w;
}

// Sums the warps' level-1 totals (lane 0 of each) into one u128 in every
// thread.
__device__ __forceinline__ u128 seq_block_total(u128 wt, SeqSmem& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (lane == 0) {
        sm.tot_lo[wid] = static_cast<unsigned long long>(wt);
        sm.tot_hi[wid] = static_cast<unsigned long long>(wt >> 64);
    }
    __syncthreads();
    u128 R = 0;
    for (int k = 0; k < kWarps; ++k) R += (static_cast<u128>(sm.tot_hi[k]) << 64) | sm.tot_lo[k];
    __syncthreads();
    return R;
}

// Given every segment's weight in ssum[] and their total R: the draw point,
// the segment that holds it (a block scan), the entry inside it (warp 0
// rescans the segment), and the committed run.
__device__ void seq_finish(DrawRow& w, u128 R, ulonglong2* ssum, const int32_t* __restrict__ drafts,
                           int Kd, int b, int32_t* __restrict__ tokens, int32_t* __restrict__ len,
                           uint32_t* status, SeqSmem& sm) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int V = w.V, nseg = n_segments(V), rowq = sm.rowq;
    if (tid == 0) {
        sm.sel = 0;
        if (rowq >= 0 && R == 0) {  // only reachable through an invalid draft id
            atomicOr(status, kStatusZeroResidual);
            sm.sel = 1;
        }
        const u128 total = rowq >= 0 && R != 0 ? R : static_cast<u128>(w.ip.S);
        const u128 t = scale_u64(sm.u64, total);
        sm.t_lo = static_cast<unsigned long long>(t);
        sm.t_hi = static_cast<unsigned long long>(t >> 64);
    }
    __syncthreads();
    if (sm.sel) {  // the residual is empty: draw from p
        w.lq = nullptr;
        segment_sums(w, ssum, sm.q[wid], wid, lane);
        __syncthreads();
    }
    // level 2: the segment whose inclusive prefix first exceeds t (each
    // thread sums a run of consecutive segments; a block scan orders the runs)
    const u128 t = (static_cast<u128>(sm.t_hi) << 64) | sm.t_lo;
    {
        const int c = (nseg + kThreads - 1) / kThreads;
        const int a = tid * c < nseg ? tid * c : nseg, e = a + c < nseg ? a + c : nseg;
        u128 run = 0;
        for (int s = a; s < e; ++s) {
            const ulonglong2 x = __ldcg(ssum + s);
            run += (static_cast<u128>(x.y) << 64) | x.x;
        }
        u128 all;
        const u128 excl = block_excl_u128(run, sm.red, all);
        if (excl <= t && t < excl + run) {
            u128 acc = excl;
            for (int s = a; s < e; ++s) {
                const ulonglong2 x = __ldcg(ssum + s);
                const u128 xs = (static_cast<u128>(x.y) << 64) | x.x;
                if (t < acc + xs) {
                    sm.seg = s;
                    const u128 rem = t - acc;
                    sm.t_lo = static_cast<unsigned long long>(rem);
                    sm.t_hi = static_cast<unsigned long long>(rem >> 64);
                    break;
                }
                acc += xs;
            }
        }
    }
    __syncthreads();
    // level 3: warp 0 rescans that segment in index order
    if (wid == 0) {
        const int s = sm.seg;
        int tok = -1;
        if (s >= 0) {
            const u128 tt = (static_cast<u128>(sm.t_hi) << 64) | sm.t_lo;
            const int v = s * kSegLen + 4 * lane;
            float4 p, q;
            w.load4(v, p, q);
            u128 e[4];
            w.weights4(v, p, q, e);
            const u128 mine = e[0] + e[1] + e[2] + e[3];
            u128 incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const u128 y = shfl_up_u128(incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned int hit = __ballot_sync(0xffffffffu, incl > tt);
            if (hit) {
                const int L = __ffs(hit) - 1;
                if (lane == L) {
                    u128 cum = incl - mine;
                    for (int j = 0; j < 4; ++j) {
                        cum += e[j];
                        if (cum > tt) {
                            tok = v + j;
                            break;
                        }
                    }
                }
                tok = __shfl_sync(0xffffffffu, tok, L);
            }
        }
        if (lane == 0) {
            if (tok >= 0) check(tok < V, status);  // the drawn entry lies in the row
            sm.token = tok >= 0 ? tok : V - 1;
        }
    }
    __syncthreads();
    if (tid <= Kd) {
        const int n = sm.n_acc;
        int32_t tk = -1;
        if (tid < n) tk = drafts[static_cast<long long>(b) * Kd + tid];
        else if (tid == n) tk = sm.token;
        tokens[static_cast<long long>(b) * (Kd + 1) + tid] = tk;
    }
    if (tid == 0) len[b] = sm.n_acc + 1;
}

__global__ void __launch_bounds__(kThreads, 2) seq_kernel(
    const float* __restrict__ target, const float* __restrict__ draft,
    const int32_t* __restrict__ drafts, int Kd, int V, int vec_ok, float invT,
    unsigned long long seed, unsigned long long offset, long long n_target_rows,
    const RowInfo* __restrict__ info, const float* __restrict__ segmax, ulonglong2* segsum,
    int32_t* __restrict__ tokens, int32_t* __restrict__ len, uint32_t* status) {
    __shared__ SeqSmem sm;
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    seq_decide(target, draft, drafts, Kd, V, invT, seed, offset, n_target_rows, info, b, status,
               sm);
    DrawRow w = seq_draw_row(target, draft, V, vec_ok, invT, n_target_rows, info, segmax, sm);
    ulonglong2* ssum = segsum + static_cast<long long>(b) * n_segments(V);
    // level 1: the weight of every segment, and the total
    const u128 R = seq_block_total(segment_sums(w, ssum, sm.q[wid], wid, lane), sm);
    seq_finish(w, R, ssum, drafts, Kd, b, tokens, len, status, sm);
}

// The draw of a split call: (sequence, chunk) CTAs weigh the chunk's
// segments of the sequence's draw row (level 1) ...
__global__ void __launch_bounds__(kThreads, 2) split_seq_sums_kernel(
    const float* __restrict__ target, const float* __restrict__ draft,
    const int32_t* __restrict__ drafts, int Kd, int V, int C, float invT,
    unsigned long long seed, unsigned long long offset, long long n_target_rows,
    const RowInfo* __restrict__ info, const float* __restrict__ segmax, ulonglong2* segsum,
    ulonglong2* chunk_tot, uint32_t* status) {
    pdl_start();
    __shared__ SeqSmem sm;
    const int b = blockIdx.x / C, c = blockIdx.x % C;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    seq_decide(target, draft, drafts, Kd, V, invT, seed, offset, n_target_rows, info, b, status,
               sm);
    DrawRow w = seq_draw_row(target, draft, V, 1, invT, n_target_rows, info, segmax, sm);
    int s0, s1;
    split_span(n_segments(V), C, c, s0, s1);
    ulonglong2* ssum = segsum + static_cast<long long>(b) * n_segments(V);
    const u128 R = seq_block_total(segment_sums(w, ssum, sm.q[wid], wid, lane, s0, s1), sm);
    if (threadIdx.x == 0)
        chunk_tot[static_cast<long long>(b) * C + c] =
            make_ulonglong2(static_cast<unsigned long long>(R), static_cast<unsigned long long>(R >> 64));
}

// ... then one CTA per sequence sums the chunk totals and finishes the draw.
__global__ void __launch_bounds__(kThreads, 2) split_seq_finish_kernel(
    const float* __restrict__ target, const float* __restrict__ draft,
    const int32_t* __restrict__ drafts, int Kd, int V, int C, float invT,
    unsigned long long seed, unsigned long long offset, long long n_target_rows,
    const RowInfo* __restrict__ info, const float* __restrict__ segmax, ulonglong2* segsum,
    const ulonglong2* __restrict__ chunk_tot, int32_t* __restrict__ tokens,
    int32_t* __restrict__ len, uint32_t* status) {
    pdl_start();
    __shared__ SeqSmem sm;
    const int b = blockIdx.x;
    seq_decide(target, draft, drafts, Kd, V, invT, seed, offset, n_target_rows, info, b, status,
               sm);
    DrawRow w = seq_draw_row(target, draft, V, 1, invT, n_target_rows, info, segmax, sm);
    u128 R = 0;
    for (int c = 0; c < C; ++c) {
        const ulonglong2 x = chunk_tot[static_cast<long long>(b) * C + c];
        R += (static_cast<u128>(x.y) << 64) | x.x;
    }
    seq_finish(w, R, segsum + static_cast<long long>(b) * n_segments(V), drafts, Kd, b, tokens,
               len, status, sm);
}

// ------------------------------------------------------ top-k lists
// The accept over sparse rows: every row is given as Kt (id, logit) pairs,
// the entries a top-k stage kept, in any order; every other entry of the
// vocabulary reads as -infinity.  The kept masses are those of the dense
// pipeline on that row, so the committed ids equal the dense accept's on
// rows holding the listed logits and -infinity elsewhere.
constexpr int kListMax = 1024;  // longest list

// Row kernel shapes: NT threads for lists of up to NMAX entries (NMAX / NT
// sorted positions per thread in the prefix scan).  Short lists take small
// blocks with small arrays, so that many rows run per SM.
template <int NT, int NMAX>
struct ListSmem {
    unsigned long long key[NMAX];
    unsigned long long W[NMAX];
    int id[NMAX];
    float l[NMAX];
    Red red;
    int nan0, cut_p, cut_mp;
};

// Sorts a[0 .. n) (n a power of two) in descending order across the block.
__device__ void list_sort_desc(unsigned long long* a, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = threadIdx.x; t < n; t += blockDim.x) {
                const int u = t ^ j;
                if (u > t) {
                    const unsigned long long x = a[t], y = a[u];
                    if ((t & k) == 0 ? (x < y) : (x > y)) {
                        a[t] = y;
                        a[u] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Inclusive prefix over the block of one u64 per thread (the block's
// threads in order).
__device__ __forceinline__ unsigned long long block_incl_u64(unsigned long long v, Red& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm.w[wid] = incl;
    __syncthreads();
    unsigned long long base = 0;
    for (int w = 0; w < wid; ++w) base += sm.w[w];
    __syncthreads();
    return base + incl;
}

// One CTA per list row: rows (b, j) for j = 0..Kd are target rows, j =
// Kd+1..2Kd draft rows.  Writes the row's entries sorted by id with their
// kept masses (0 for the dropped ones) and the kept sum.
template <int NT, int NMAX>
__global__ void __launch_bounds__(NT) list_row_kernel(
    const int32_t* __restrict__ t_ids, const float* __restrict__ t_vals,
    const int32_t* __restrict__ d_ids, const float* __restrict__ d_vals, int Kd, int Kt, int V,
    float invT, unsigned long long P, int top_k, unsigned long long MP, int32_t* __restrict__ o_ids,
    unsigned long long* __restrict__ o_W, unsigned long long* __restrict__ o_S, uint32_t* status) {
    constexpr int kListThreads = NT;
    constexpr int kListPer = NMAX / NT;
    static_assert(NMAX % NT == 0 && NT % 32 == 0, "list row kernel shape");
    __shared__ ListSmem<NT, NMAX> sm;
    const int tid = threadIdx.x;
    const long long r = blockIdx.x;
    const int per_seq = 2 * Kd + 1;
    const long long b = r / per_seq;
    const int j = static_cast<int>(r % per_seq);
    const long long src = j <= Kd ? (b * (Kd + 1) + j) * Kt : (b * Kd + (j - Kd - 1)) * Kt;
    const int32_t* ids = j <= Kd ? t_ids : d_ids;
    const float* vals = j <= Kd ? t_vals : d_vals;
    int n = 1;
    while (n < Kt) n <<= 1;

    // (1) load; an id outside [0, V) is dropped (its logit read as -inf)
    if (tid == 0) sm.nan0 = 0;
    __syncthreads();
    float m = -INFINITY;
    int bad = 0;
    for (int t = tid; t < Kt; t += kListThreads) {
        int id = __ldg(ids + src + t);
        float l = __ldg(vals + src + t);
        if (id < 0 || id >= V) {
            bad = 1;
            id = V + t;  // past every real id: sorts last, never looked up
            l = -INFINITY;
        }
        if (id == 0 && l != l) sm.nan0 = 1;
        m = fmaxf(m, l);  // NaN never raises the max
        sm.id[t] = id;
        sm.l[t] = l;
    }
    if (bad) atomicOr(status, kStatusBadListId);
    // The dense row's max is taken from index 0 upwards with ">": a NaN at
    // index 0 makes it NaN (then every mass is 0); elsewhere NaN is skipped.
    m = block_max(m, sm.red);
    const float mx = sm.nan0 ? __int_as_float(0x7fc00000) : m;

    // (2) top-k: the first top_k entries in (logit desc, id asc) order take
    // part; -inf and NaN entries weigh 0 whether they take part or not
    const bool tk_on = top_k > 0 && top_k < V && top_k < Kt;
    unsigned long long tk_cut = 0ull;
    if (tk_on) {
        for (int t = tid; t < n; t += kListThreads)
            sm.key[t] = t < Kt ? (static_cast<unsigned long long>(logit_key(sm.l[t])) << 32) |
                                     (0xFFFFFFFFu - static_cast<uint32_t>(sm.id[t]))
                               : 0ull;
        __syncthreads();
        list_sort_desc(sm.key, n);
        tk_cut = sm.key[top_k - 1];
        __syncthreads();
    }
    // (3) masses
    unsigned long long part = 0ull;
    for (int t = tid; t < Kt; t += kListThreads) {
        const float l = sm.l[t];
        bool in = true;
        if (tk_on)
            in = ((static_cast<unsigned long long>(logit_key(l)) << 32) |
                  (0xFFFFFFFFu - static_cast<uint32_t>(sm.id[t]))) >= tk_cut;
        const unsigned long long W = in ? mass_of(own_exp(scaled_x(l, mx, invT))) : 0ull;
        sm.W[t] = W;
        part += W;
    }
    const unsigned long long S = block_sum_u64(part, sm.red);

    // (4) top-p and min-p: both keep a prefix of the (W desc, id asc) order.
    // Key: W (2^40 read as 2^40 - 1: no other mass lies above 2^40 - 2^16),
    // then the low 24 bits of ~id (ids below 2^24; only dropped ids collide,
    // and they weigh 0).
    if (P < kKeepAll || MP > 0) {
        for (int t = tid; t < n; t += kListThreads) {
            unsigned long long key = 0ull;
            if (t < Kt) {
                const unsigned long long W = sm.W[t];
                const unsigned long long w40 = W >= (1ull << 40) ? (1ull << 40) - 1ull : W;
                key = (w40 << 24) | (0xFFFFFFull - (static_cast<uint32_t>(sm.id[t]) & 0xFFFFFFu));
            }
            sm.key[t] = key;
        }
        if (tid == 0) {
            sm.cut_p = Kt;
            sm.cut_mp = Kt;
        }
        __syncthreads();
        list_sort_desc(sm.key, n);
        // each thread takes kListPer consecutive sorted positions
        const int p0 = tid * kListPer;
        unsigned long long w[kListPer], run = 0ull;
#pragma unroll
        for (int q = 0; q < kListPer; ++q) {
            const int p = p0 + q;
            unsigned long long W = 0ull;
            if (p < Kt) {
                W = sm.key[p] >> 24;
                if (W == (1ull << 40) - 1ull) W = 1ull << 40;
            }
            w[q] = W;
            run += W;
        }
        const unsigned long long incl = block_incl_u64(run, sm.red);
        const unsigned long long w_top = sm.key[0] >> 24 == (1ull << 40) - 1ull
                                             ? (1ull << 40)
                                             : sm.key[0] >> 24;
        unsigned long long cum = incl - run;
        const u128 target = static_cast<u128>(P) * S;
#pragma unroll
        for (int q = 0; q < kListPer; ++q) {
            const int p = p0 + q;
            if (p >= Kt) break;
            cum += w[q];
            if (P < kKeepAll && (static_cast<u128>(cum) << 32) >= target)
                atomicMin(&sm.cut_p, p + 1);  // the shortest prefix reaching P
            if (MP > 0 && (static_cast<u128>(w[q]) << 32) < static_cast<u128>(MP) * w_top)
                atomicMin(&sm.cut_mp, p);     // the first entry below min-p
        }
        __syncthreads();
        const int keep = min(sm.cut_p, sm.cut_mp);
        // the kept entries are the sorted positions below keep; keep >= 1
        // unless min-p drops the top entry itself (then nothing is kept)
        const unsigned long long kcut = keep > 0 ? sm.key[keep - 1] : ~0ull;
        __syncthreads();
        for (int t = tid; t < Kt; t += kListThreads) {
            const unsigned long long W = sm.W[t];
            const unsigned long long w40 = W >= (1ull << 40) ? (1ull << 40) - 1ull : W;
            const unsigned long long key =
                (w40 << 24) | (0xFFFFFFull - (static_cast<uint32_t>(sm.id[t]) & 0xFFFFFFu));
            if (keep == 0 || key < kcut) sm.W[t] = 0ull;
        }
        __syncthreads();
    }
    unsigned long long kpart = 0ull;
    for (int t = tid; t < Kt; t += kListThreads) kpart += sm.W[t];
    const unsigned long long S_kept = block_sum_u64(kpart, sm.red);

    // (5) the row sorted by id (ascending), with its kept masses
    for (int t = tid; t < n; t += kListThreads)
        sm.key[t] = t < Kt ? ((static_cast<unsigned long long>(0x7FFFFFFF - sm.id[t]) << 32) |
                              static_cast<uint32_t>(t))
                           : 0ull;
    __syncthreads();
    list_sort_desc(sm.key, n);  // descending in 0x7FFFFFFF - id: ascending in id
    for (int p = tid; p < Kt; p += kListThreads) {
        const int t = static_cast<int>(sm.key[p] & 0xFFFFFFFFu);
        o_ids[r * Kt + p] = sm.id[t];
        o_W[r * Kt + p] = sm.W[t];
    }
    if (tid == 0) o_S[r] = S_kept;
}

// ------------------------------------------------ top-k lists, warp rows
// Lists of at most 256 entries: one warp per list row, the same steps as
// list_row_kernel with the row in registers -- lane l holds positions
// l + 32 r, r < R (R = 2, 4, 8 for up to 64, 128, 256 entries) -- and every
// sort a bitonic network over the 32 R positions: partners less than 32
// apart are exchanged by shuffles, the others are in the same lane.  No step
// waits on a block barrier.
constexpr int kListWarpMax = 256;
constexpr int kListWarpRows = 4;  // rows (warps) per CTA

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int o) {
    return __shfl_xor_sync(0xffffffffu, v, o);
}

// Sorts the 32 R keys a[r] at positions lane + 32 r in descending order.
template <int R>
__device__ __forceinline__ void warp_sort_desc(unsigned long long (&a)[R]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32 * R; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 32) {
                // partners in the same lane: registers r and r ^ (j / 32)
                const int jr = j >> 5;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r & jr) continue;  // (the pair is handled from its lower register)
                    const int p = lane + 32 * r;
                    const unsigned long long x = a[r], y = a[r | jr];
                    const bool desc = (p & k) == 0;  // the lower position keeps the larger
                    const bool swap = desc ? x < y : x > y;
                    a[r] = swap ? y : x;
                    a[r | jr] = swap ? x : y;
                }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int p = lane + 32 * r;
                    const unsigned long long y = shfl_xor_u64(a[r], j);
                    // in a block sorted descending ((p & k) == 0) the lower
                    // position keeps the larger key; in an ascending one the smaller
                    const bool keep_max = ((p & j) == 0) == ((p & k) == 0);
                    a[r] = keep_max ? (a[r] > y ? a[r] : y) : (a[r] < y ? a[r] : y);
                }
            }
        }
    }
}

// Register r of an array (r the same in every lane, or not: no local memory).
template <int R, class T>
__device__ __forceinline__ T reg_at(const T (&a)[R], int r) {
    T v = a[0];
#pragma unroll
    for (int q = 1; q < R; ++q)
        if (q == r) v = a[q];
    return v;
}

// The key at sorted position p (the same p in every lane).
template <int R>
__device__ __forceinline__ unsigned long long warp_at(const unsigned long long (&a)[R], int p) {
    return __shfl_sync(0xffffffffu, reg_at<R>(a, p >> 5), p & 31);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += shfl_xor_u64(v, o);
    return v;
}

template <int R>
__global__ void __launch_bounds__(kListWarpRows * 32) list_row_warp_kernel(
    const int32_t* __restrict__ t_ids, const float* __restrict__ t_vals,
    const int32_t* __restrict__ d_ids, const float* __restrict__ d_vals, int Kd, int Kt, int V,
    long long rows, float invT, unsigned long long P, int top_k, unsigned long long MP,
    int32_t* __restrict__ o_ids, unsigned long long* __restrict__ o_W,
    unsigned long long* __restrict__ o_S, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const long long r = static_cast<long long>(blockIdx.x) * kListWarpRows + (threadIdx.x >> 5);
    if (r >= rows) return;  // (whole warps)
    const int per_seq = 2 * Kd + 1;
    const long long b = r / per_seq;
    const int j = static_cast<int>(r % per_seq);
    const long long src = j <= Kd ? (b * (Kd + 1) + j) * Kt : (b * Kd + (j - Kd - 1)) * Kt;
    const int32_t* ids = j <= Kd ? t_ids : d_ids;
    const float* vals = j <= Kd ? t_vals : d_vals;

    // (1) load; an id outside [0, V) is dropped (its logit read as -inf)
    int id[R];
    float l[R];
    float m = -INFINITY;
    bool bad = false, nan0 = false;
#pragma unroll
    for (int q = 0; q < R; ++q) {
        const int t = lane + 32 * q;
        id[q] = V + t;  // positions past Kt: never real, sort last
        l[q] = -INFINITY;
        if (t < Kt) {
            int i = __ldg(ids + src + t);
            float v = __ldg(vals + src + t);
            if (i < 0 || i >= V) {
                bad = true;
                i = V + t;
                v = -INFINITY;
            }
            if (i == 0 && v != v) nan0 = true;
            m = fmaxf(m, v);  // NaN never raises the max
            id[q] = i;
            l[q] = v;
        }
    }
    if (bad) atomicOr(status, kStatusBadListId);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // the dense row's max: NaN when id 0 holds a NaN, else NaN is skipped
    const float mx = __any_sync(0xffffffffu, nan0) ? __int_as_float(0x7fc00000) : m;

    // (2) top-k: the first top_k entries in (logit desc, id asc) order
    const bool tk_on = top_k > 0 && top_k < V && top_k < Kt;
    unsigned long long tkey[R];
#pragma unroll
    for (int q = 0; q < R; ++q)
        tkey[q] = lane + 32 * q < Kt ? (static_cast<unsigned long long>(logit_key(l[q])) << 32) |
                                           (0xFFFFFFFFu - static_cast<uint32_t>(id[q]))
                                     : 0ull;
    unsigned long long tk_cut = 0ull;
    if (tk_on) {
        unsigned long long srt[R];
#pragma unroll
        for (int q = 0; q < R; ++q) srt[q] = tkey[q];
        warp_sort_desc<R>(srt);
        tk_cut = warp_at<R>(srt, top_k - 1);
    }
    // (3) masses
    unsigned long long W[R];
    unsigned long long part = 0ull;
#pragma unroll
    for (int q = 0; q < R; ++q) {
        const bool in = lane + 32 * q < Kt && (!tk_on || tkey[q] >= tk_cut);
        W[q] = in ? mass_of(own_exp(scaled_x(l[q], mx, invT))) : 0ull;
        part += W[q];
    }
    const unsigned long long S = warp_sum_u64(part);

    // (4) top-p and min-p: both keep a prefix of the (W desc, id asc) order
    // (keys as in list_row_kernel)
    auto wkey = [&](int q) -> unsigned long long {
        if (lane + 32 * q >= Kt) return 0ull;
        const unsigned long long w40 = W[q] >= (1ull << 40) ? (1ull << 40) - 1ull : W[q];
        return (w40 << 24) | (0xFFFFFFull - (static_cast<uint32_t>(id[q]) & 0xFFFFFFu));
    };
    if (P < kKeepAll || MP > 0) {
        unsigned long long srt[R];
#pragma unroll
        for (int q = 0; q < R; ++q) srt[q] = wkey(q);
        warp_sort_desc<R>(srt);
        unsigned long long ws[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const unsigned long long w = srt[q] >> 24;
            ws[q] = lane + 32 * q < Kt ? (w == (1ull << 40) - 1ull ? (1ull << 40) : w) : 0ull;
        }
        const unsigned long long w_top = __shfl_sync(0xffffffffu, ws[0], 0);
        const u128 target = static_cast<u128>(P) * S;
        int keep = Kt;
        unsigned long long base = 0ull;  // the mass of positions 0 .. 32 q - 1
#pragma unroll
        for (int q = 0; q < R; ++q) {
            // inclusive prefix over positions 32 q + 0 .. 31
            unsigned long long cum = ws[q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, cum, o);
                if (lane >= o) cum += y;
            }
            cum += base;
            base = __shfl_sync(0xffffffffu, cum, 31);
            const bool valid = lane + 32 * q < Kt;
            // the shortest prefix reaching P; the first entry below min-p
            const unsigned int hp = __ballot_sync(
                0xffffffffu, valid && P < kKeepAll && (static_cast<u128>(cum) << 32) >= target);
            const unsigned int hm = __ballot_sync(
                0xffffffffu,
                valid && MP > 0 && (static_cast<u128>(ws[q]) << 32) < static_cast<u128>(MP) * w_top);
            if (hp) keep = min(keep, 32 * q + __ffs(hp));
            if (hm) keep = min(keep, 32 * q + __ffs(hm) - 1);
        }
        // the kept entries are the sorted positions below keep (keep >= 1
        // unless min-p drops the top entry itself)
        const unsigned long long kcut = keep > 0 ? warp_at<R>(srt, keep - 1) : ~0ull;
#pragma unroll
        for (int q = 0; q < R; ++q)
            if (keep == 0 || wkey(q) < kcut) W[q] = 0ull;
    }
    unsigned long long kpart = 0ull;
#pragma unroll
    for (int q = 0; q < R; ++q) kpart += W[q];
    const unsigned long long S_kept = warp_sum_u64(kpart);

    // (5) the row sorted by id (ascending), with its kept masses
    unsigned long long srt[R];
#pragma unroll
    for (int q = 0; q < R; ++q) {
        const int t = lane + 32 * q;
        srt[q] = t < Kt ? ((static_cast<unsigned long long>(0x7FFFFFFF - id[q]) << 32) |
                           static_cast<uint32_t>(t))
                        : 0ull;
    }
    warp_sort_desc<R>(srt);  // descending in 0x7FFFFFFF - id: ascending in id
#pragma unroll
    for (int q = 0; q < R; ++q) {
        const int p = lane + 32 * q;
        const int t = static_cast<int>(srt[q] & 0xFFFFFFFFu);
        // entry t's mass from the lane that holds it (every lane shuffles)
        unsigned long long wt = 0ull;
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const unsigned long long x = __shfl_sync(0xffffffffu, W[u], t & 31);
            if (u == (t >> 5)) wt = x;
        }
        if (p < Kt) {
            o_ids[r * Kt + p] = 0x7FFFFFFF - static_cast<int>(srt[q] >> 32);
            o_W[r * Kt + p] = wt;
        }
    }
    if (lane == 0) o_S[r] = S_kept;
}

// The kept mass of id x in a row sorted by id (0 when absent).
__device__ __forceinline__ unsigned long long list_mass(const int32_t* ids,
                                                        const unsigned long long* W, int Kt,
                                                        int x) {
    int lo = 0, hi = Kt;  // first position with id >= x
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(ids + mid) < x) lo = mid + 1;
        else hi = mid;
    }
    return lo < Kt && __ldg(ids + lo) == x ? __ldg(W + lo) : 0ull;
}

// One warp per sequence: the acceptance tests in order, then one ordered
// draw over the rejected position's list (the residual against the draft's
// list, or p itself), or the bonus from the last target list.
constexpr int kListSeqWarps = 4;

__global__ void __launch_bounds__(kListSeqWarps * 32) list_seq_kernel(
    const int32_t* __restrict__ drafts, int B, int Kd, int Kt, int V, unsigned long long seed,
    unsigned long long offset, const int32_t* __restrict__ l_ids,
    const unsigned long long* __restrict__ l_W, const unsigned long long* __restrict__ l_S,
    int32_t* __restrict__ tokens, int32_t* __restrict__ len, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kListSeqWarps + (threadIdx.x >> 5);
    if (b >= B) return;
    const long long per_seq = 2 * Kd + 1;
    auto row = [&](int j) { return static_cast<long long>(b) * per_seq + j; };  // list row
    // the acceptance tests, lane i taking position i (Kd < 32), all at once;
    // the first rejection decides the run, and position n's uniform the draw
    static_assert(kMaxRows < 32, "one lane per position");
    unsigned long long u64 = 0ull;
    bool ok = true;
    if (lane <= Kd) {
        const int i = lane;
        uint32_t rr[4];
        philox4x32_10(static_cast<uint32_t>(i), static_cast<uint32_t>(b),
                      static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
                      static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), rr);
        u64 = (static_cast<unsigned long long>(rr[2]) << 32) | rr[1];
        if (i < Kd) {
            const int32_t x = drafts[static_cast<long long>(b) * Kd + i];
            ok = false;
            if (x >= 0 && x < V) {
                const long long rp = row(i), rq = row(Kd + 1 + i);
                const unsigned long long Wp = list_mass(l_ids + rp * Kt, l_W + rp * Kt, Kt, x);
                const unsigned long long Wq = list_mass(l_ids + rq * Kt, l_W + rq * Kt, Kt, x);
                const unsigned long long U = rr[0] >> 8;
                const u128 lhs = static_cast<u128>(U * Wq) * l_S[rp];
                const u128 rhs = (static_cast<u128>(Wp) * l_S[rq]) << 24;
                ok = lhs < rhs;
            }
        }
    }
    const unsigned int rej = __ballot_sync(0xffffffffu, lane < Kd && !ok);
    const int n = rej ? __ffs(rej) - 1 : Kd;  // accepted drafts before the first rejection
    u64 = __shfl_sync(0xffffffffu, u64, n);
    // an invalid draft id counts as a rejection; flagged when it is reached
    // (the tests after the first rejection are not part of the run)
    if (lane == n && n < Kd) {
        const int32_t x = drafts[static_cast<long long>(b) * Kd + n];
        if (x < 0 || x >= V) atomicOr(status, kStatusBadDraft);
    }
    // the draw: over target list n in id order, weights the residual
    // max(0, Wp Sq - Wq Sp) at a rejection, else (the bonus, or an empty
    // residual) Wp itself
    const long long rp = row(n);
    const int32_t* pid = l_ids + rp * Kt;
    const unsigned long long* pW = l_W + rp * Kt;
    const unsigned long long Sp = l_S[rp];
    const bool rejected = n < Kd;
    const long long rq = rejected ? row(Kd + 1 + n) : -1;
    const unsigned long long Sq = rejected ? l_S[rq] : 0ull;
    const int c = (Kt + 31) / 32;
    const int a = min(lane * c, Kt), e = min(a + c, Kt);
    auto weight = [&](int p, bool resid) -> u128 {
        const unsigned long long Wp = __ldg(pW + p);
        if (!resid) return Wp;
        const unsigned long long Wq =
            Wp ? list_mass(l_ids + rq * Kt, l_W + rq * Kt, Kt, __ldg(pid + p)) : 0ull;
        const u128 x = static_cast<u128>(Wp) * Sq, y = static_cast<u128>(Wq) * Sp;
        return x > y ? x - y : 0;
    };
    bool resid = rejected;
    // up to two positions a lane (lists of at most 64): both weights at once
    // (their searches overlap), kept for the rescan below
    u128 w2[2] = {0, 0};
    auto weigh_all = [&]() -> u128 {
        if (c <= 2) {
            w2[0] = a < e ? weight(a, resid) : 0;
            w2[1] = a + 1 < e ? weight(a + 1, resid) : 0;
            return w2[0] + w2[1];
        }
        u128 m = 0;
        for (int p = a; p < e; ++p) m += weight(p, resid);
        return m;
    };
    u128 mine = weigh_all();
    u128 R = warp_sum_u128(mine);
    if (resid && R == 0) {  // only reachable through an invalid draft id
        if (lane == 0) atomicOr(status, kStatusZeroResidual);
        resid = false;
        mine = weigh_all();
        R = warp_sum_u128(mine);
    }
    int tok = V - 1;  // an empty row: as the dense draw
    if (R > 0) {
        const u128 t = scale_u64(u64, R);
        u128 incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const u128 y = shfl_up_u128(incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned int hit = __ballot_sync(0xffffffffu, incl > t);
        const int L = __ffs(hit) - 1;  // R > t, so some lane's prefix exceeds t
        int found = -1;
        if (lane == L) {
            u128 cum = incl - mine;
            for (int p = a; p < e; ++p) {
                cum += c <= 2 ? (p == a ? w2[0] : w2[1]) : weight(p, resid);
                if (cum > t) {
                    found = __ldg(pid + p);
                    break;
                }
            }
        }
        tok = __shfl_sync(0xffffffffu, found, L);
    }
    if (lane == 0) check(tok >= 0 && tok < V, status);  // the drawn id lies in the vocabulary
    for (int i = lane; i <= Kd; i += 32) {
        int32_t tk = -1;
        if (i < n) tk = drafts[static_cast<long long>(b) * Kd + i];
        else if (i == n) tk = tok;
        tokens[static_cast<long long>(b) * (Kd + 1) + i] = tk;
    }
    if (lane == 0) len[b] = n + 1;
}

__global__ void own_exp_kernel(const float* __restrict__ x, float* __restrict__ y, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        y[i] = own_exp(x[i]);
}

// W = floor(own_exp(x) 2^40) of scaled logits x by the packed-pair path of
// the mass passes (entries 2j and 2j + 1 in one pair; an odd tail paired
// with -inf).
__global__ void own_mass_pairs_kernel(const float* __restrict__ x,
                                      unsigned long long* __restrict__ W, long long n) {
    const long long np = (n + 1) / 2;
    for (long long j = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; j < np;
         j += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long i = 2 * j;
        const bool two = i + 1 < n;
        const float2 f = own_exp_2_40_x2(make_float2(x[i], two ? x[i + 1] : -INFINITY));
        float2 t1, t2;
        mass_bits_x2(f, t1, t2);
        W[i] = (static_cast<unsigned long long>(__float_as_uint(t1.x) - 0x4B000000u) << 20) +
               (__float_as_uint(t2.x) - 0x4B000000u);
        if (two)
            W[i + 1] = (static_cast<unsigned long long>(__float_as_uint(t1.y) - 0x4B000000u) << 20) +
                       (__float_as_uint(t2.y) - 0x4B000000u);
    }
}


}  // namespace

cudaError_t launch_own_mass_pairs(const float* x, unsigned long long* W, long long n,
                                  cudaStream_t s) {
    long long blocks = ((n + 1) / 2 + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    if (blocks < 1) blocks = 1;
    own_mass_pairs_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, W, n);
    return cudaGetLastError();
}

cudaError_t launch_own_exp(const float* x, float* y, long long n, cudaStream_t s) {
    long long blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    if (blocks < 1) blocks = 1;
    own_exp_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, y, n);
    return cudaGetLastError();
}

// [rows] RowInfo, then [rows][segments] float segment maxima.
static size_t info_bytes(size_t rows) { return ((rows * sizeof(RowInfo) + 255) / 256) * 256; }

// ... then [B][segments] 128-bit segment weights of the draw.
static size_t segmax_bytes(size_t rows, int V) {
    const size_t seg = rows * static_cast<size_t>((V + kSegLen - 1) / kSegLen) * sizeof(float);
    return ((seg + 255) / 256) * 256;
}

// ... then, for few rows of a wide vocabulary, the split-row arrays.
static size_t base_bytes(size_t rows, int B, int V) {
    const size_t draw = static_cast<size_t>(B) * ((V + kSegLen - 1) / kSegLen) * 16;
    return info_bytes(rows) + segmax_bytes(rows, V) + r256(draw);
}

static bool split_sized(long long rows, int V) { return rows <= kSplitRowsMax && V >= kSplitMinV; }

size_t rejection_workspace_bytes(int B, int Kd, int V) {
    const size_t rows = static_cast<size_t>(B) * (2 * static_cast<size_t>(Kd) + 1);
    size_t b = base_bytes(rows, B, V);
    if (split_sized(static_cast<long long>(rows), V))
        b += split_layout(nullptr, static_cast<long long>(rows)).bytes;
    return b;
}

cudaError_t launch_accept_rejection(const float* target, const float* draft,
                                    const int32_t* drafts, int B, int Kd, int V, float invT,
                                    uint64_t P, int top_k, uint64_t MP, uint64_t seed,
                                    uint64_t offset, int32_t* tokens,
                                    int32_t* len, void* ws, size_t ws_bytes, uint32_t* status,
                                    unsigned long long wait_ns, cudaStream_t s,
                                    const float* target_bmax, const float* draft_bmax) {
    const long long n_target_rows = static_cast<long long>(B) * (Kd + 1);
    const long long rows = n_target_rows + static_cast<long long>(B) * Kd;
    if (rows > 0x7fffffffll) return cudaErrorNotSupported;
    if (rejection_workspace_bytes(B, Kd, V) > ws_bytes) return cudaErrorInvalidValue;
    RowInfo* info = static_cast<RowInfo*>(ws);
    float* segmax = reinterpret_cast<float*>(static_cast<char*>(ws) + info_bytes(rows));
    ulonglong2* segsum = reinterpret_cast<ulonglong2*>(static_cast<char*>(ws) + info_bytes(rows) +
                                                       segmax_bytes(rows, V));
    (void)wait_ns;

    const size_t smem = sizeof(RowSmem);
    cudaError_t e = cudaFuncSetAttribute(row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int vec_ok = (V % 4 == 0 && (reinterpret_cast<uintptr_t>(target) & 15u) == 0 &&
                        (reinterpret_cast<uintptr_t>(draft) & 15u) == 0)
                           ? 1
                           : 0;
    // few rows of a wide vocabulary (and no top-k or min-p stage): each row
    // in chunks over many CTAs
    const bool split = split_sized(rows, V) && vec_ok && (top_k <= 0 || top_k >= V) && MP == 0;
    if (split) {
        const int C = split_chunks(rows);
        const SplitWs sw = split_layout(static_cast<char*>(ws) + base_bytes(rows, B, V), rows);
        const unsigned long long Pu = static_cast<unsigned long long>(P);
        for (const void* k : {reinterpret_cast<const void*>(split_mass_kernel),
                              reinterpret_cast<const void*>(split_beta_kernel),
                              reinterpret_cast<const void*>(split_cut_kernel)}) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        // seven chained launches (each a programmatic dependent of the one before)
        const unsigned grid = static_cast<unsigned>(rows * C), nrows = static_cast<unsigned>(rows);
        e = launch_dependent(split_max_kernel, grid, kRowThreads, 0, s, target, draft,
                             n_target_rows, V, C, target_bmax, draft_bmax, segmax, sw.chunkmax);
        if (e == cudaSuccess)
            e = launch_dependent(split_mass_kernel, grid, kRowThreads, smem, s, target, draft,
                                 n_target_rows, V, C, invT, Pu, sw.chunkmax, sw.pS, sw.phist);
        if (e == cudaSuccess)
            e = launch_dependent(split_beta_kernel, nrows, kRowThreads, smem, s, V, C, Pu,
                                 sw.chunkmax, sw.pS, sw.phist, info, sw.state, sw.ncand);
        if (e == cudaSuccess)
            e = launch_dependent(split_gather_kernel, grid, kRowThreads, 0, s, target, draft,
                                 n_target_rows, V, C, invT, segmax, sw.chunkmax, sw.state,
                                 sw.ncand, sw.cw, sw.ci);
        if (e == cudaSuccess)
            e = launch_dependent(split_cut_kernel, nrows, kRowThreads, smem, s, target, draft,
                                 n_target_rows, V, C, invT, Pu, segmax, sw.chunkmax, sw.state,
                                 sw.ncand, sw.cw, sw.ci, info);
        // the draw: every sequence's draw row weighed in chunks, then finished
        const int Cs = split_chunks(B);
        const unsigned long long seed_u = static_cast<unsigned long long>(seed);
        const unsigned long long offset_u = static_cast<unsigned long long>(offset);
        if (e == cudaSuccess)
            e = launch_dependent(split_seq_sums_kernel, static_cast<unsigned>(B * Cs), kThreads, 0,
                                 s, target, draft, drafts, Kd, V, Cs, invT, seed_u, offset_u,
                                 n_target_rows, info, segmax, segsum, sw.chunk_tot, status);
        if (e == cudaSuccess)
            e = launch_dependent(split_seq_finish_kernel, static_cast<unsigned>(B), kThreads, 0, s,
                                 target, draft, drafts, Kd, V, Cs, invT, seed_u, offset_u,
                                 n_target_rows, info, segmax, segsum, sw.chunk_tot, tokens, len,
                                 status);
        return e != cudaSuccess ? e : cudaGetLastError();
    } else {
        row_kernel<<<static_cast<unsigned>(rows), kRowThreads, smem, s>>>(
            target, draft, n_target_rows, V, vec_ok, invT, static_cast<unsigned long long>(P),
            top_k, static_cast<unsigned long long>(MP), info, segmax, target_bmax, draft_bmax);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    seq_kernel<<<B, kThreads, 0, s>>>(target, draft, drafts, Kd, V, vec_ok, invT,
                                      static_cast<unsigned long long>(seed),
                                      static_cast<unsigned long long>(offset), n_target_rows,
                                      info, segmax, segsum, tokens, len, status);
    return cudaGetLastError();
}

// The records are vw4_row_record in the public header: the same fields at
// the same offsets.
static_assert(sizeof(RowInfo) == sizeof(vw4_row_record), "row record size");
static_assert(offsetof(RowInfo, mx) == offsetof(vw4_row_record, max) &&
                  offsetof(RowInfo, cut) == offsetof(vw4_row_record, cut) &&
                  offsetof(RowInfo, tau) == offsetof(vw4_row_record, tau) &&
                  offsetof(RowInfo, S) == offsetof(vw4_row_record, kept_sum) &&
                  offsetof(RowInfo, tk_key) == offsetof(vw4_row_record, topk_key) &&
                  offsetof(RowInfo, tk_idx) == offsetof(vw4_row_record, topk_idx),
              "row record layout");

cudaError_t copy_rejection_row_records(const void* ws, long long rows, void* out,
                                       cudaStream_t s) {
    // the records are the first part of the workspace (info_bytes)
    return cudaMemcpyAsync(out, ws,
                           static_cast<size_t>(rows) * sizeof(RowInfo),
                           cudaMemcpyDeviceToDevice, s);
}

static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

size_t rejection_topk_workspace_bytes(int B, int Kd, int Kt) {
    const size_t rows = static_cast<size_t>(B) * (2 * static_cast<size_t>(Kd) + 1);
    return round256(rows * Kt * 4) + round256(rows * Kt * 8) + round256(rows * 8);
}

cudaError_t launch_accept_rejection_topk(const int32_t* t_ids, const float* t_vals,
                                         const int32_t* d_ids, const float* d_vals,
                                         const int32_t* drafts, int B, int Kd, int Kt, int V,
                                         float invT, uint64_t P, int top_k, uint64_t MP,
                                         uint64_t seed, uint64_t offset, int32_t* tokens,
                                         int32_t* len, void* ws, size_t ws_bytes,
                                         uint32_t* status, cudaStream_t s) {
    if (Kt < 1 || Kt > kListMax) return cudaErrorNotSupported;
    static_assert(kListMax == 1024, "the row kernel shapes cover lists up to 1024");
    const long long rows = static_cast<long long>(B) * (2 * Kd + 1);
    if (rows > 0x7fffffffll) return cudaErrorNotSupported;
    if (rejection_topk_workspace_bytes(B, Kd, Kt) > ws_bytes) return cudaErrorInvalidValue;
    char* w = static_cast<char*>(ws);
    int32_t* l_ids = reinterpret_cast<int32_t*>(w);
    w += round256(static_cast<size_t>(rows) * Kt * 4);
    unsigned long long* l_W = reinterpret_cast<unsigned long long*>(w);
    w += round256(static_cast<size_t>(rows) * Kt * 8);
    unsigned long long* l_S = reinterpret_cast<unsigned long long*>(w);
    const unsigned wgrid = static_cast<unsigned>((rows + kListWarpRows - 1) / kListWarpRows);
    const unsigned long long Pu = static_cast<unsigned long long>(P);
    const unsigned long long MPu = static_cast<unsigned long long>(MP);
    static_assert(kListWarpMax == 256, "three warp shapes: 64, 128 and 256 entries");
    if (Kt <= 64)
        list_row_warp_kernel<2><<<wgrid, kListWarpRows * 32, 0, s>>>(
            t_ids, t_vals, d_ids, d_vals, Kd, Kt, V, rows, invT, Pu, top_k, MPu, l_ids, l_W,
            l_S, status);
    else if (Kt <= 128)
        list_row_warp_kernel<4><<<wgrid, kListWarpRows * 32, 0, s>>>(
            t_ids, t_vals, d_ids, d_vals, Kd, Kt, V, rows, invT, Pu, top_k, MPu, l_ids, l_W,
            l_S, status);
    else if (Kt <= kListWarpMax)
        list_row_warp_kernel<8><<<wgrid, kListWarpRows * 32, 0, s>>>(
            t_ids, t_vals, d_ids, d_vals, Kd, Kt, V, rows, invT, Pu, top_k, MPu, l_ids, l_W,
            l_S, status);
    else
        list_row_kernel<256, 1024><<<static_cast<unsigned>(rows), 256, 0, s>>>(
            t_ids, t_vals, d_ids, d_vals, Kd, Kt, V, invT, Pu, top_k, MPu, l_ids, l_W, l_S,
            status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    list_seq_kernel<<<(B + kListSeqWarps - 1) / kListSeqWarps, kListSeqWarps * 32, 0, s>>>(
        drafts, B, Kd, Kt, V, static_cast<unsigned long long>(seed),
        static_cast<unsigned long long>(offset), l_ids, l_W, l_S, tokens, len, status);
    return cudaGetLastError();
}

}  // namespace vw4
