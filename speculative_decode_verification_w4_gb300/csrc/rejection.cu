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
// Three kernels:
//  1. row statistics, one thread-block cluster per logits row: the row is
//     held in the cluster's shared memory (a slice per CTA); max and sum are
//     combined through distributed shared memory, and the top-p cut is found
//     by an exact radix search on W (a log-scale histogram, then 8-bit
//     digits inside the crossing bucket), histograms merged over DSMEM.
//     Output per row: max, threshold tau, cut index among W == tau, kept sum.
//  2. accept decisions, one thread per sequence (Philox4x32-10 uniforms).
//  3. the residual or bonus draw, one CTA per sequence: an exact u128 total,
//     then an ordered scan in 4096-element tiles.
#include <cooperative_groups.h>

#include "vw4_internal.cuh"

namespace cg = cooperative_groups;

namespace vw4 {

namespace {

constexpr uint32_t kStatusBadDraft = 0x1u;
constexpr uint32_t kStatusZeroResidual = 0x8u;
constexpr int kStatThreads = 512;
constexpr int kSampleThreads = 1024;
constexpr int kLogBuckets = 16 + 37 * 8;  // exact 0..15, then 8 per binade up to 2^40
constexpr int kLinBuckets = 256;
constexpr int kMaxSlice = 49152;  // floats per CTA (192 KB)
constexpr unsigned long long kKeepAll = 1ull << 32;

typedef unsigned __int128 u128;

struct RowStat {
    float mx;
    int cut;                 // largest kept index among W == tau
    unsigned long long tau;  // kept: W > tau, or W == tau and v <= cut
    unsigned long long S;    // kept sum
    unsigned long long pad;
};

struct SeqState {
    int mode;  // 0 residual at pos, 1 bonus from target row Kd, 2 residual forced (bad id)
    int pos;
    int n;
    int pad;
    unsigned long long u64;
};

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
    const int ni = static_cast<int>(n);
    return __fmul_rn(p, __uint_as_float(static_cast<uint32_t>(ni + 127) << 23));
}

__device__ __forceinline__ float scaled_x(float l, float mx, float invT) {
    return __fmul_rn(__fsub_rn(l, mx), invT);
}

__device__ __forceinline__ unsigned long long mass_of(float e) {
    return __float2ull_rz(__fmul_rn(e, 1099511627776.0f));  // e * 2^40 is exact
}

__device__ __forceinline__ unsigned long long mass_at(float l, float mx, float invT) {
    return mass_of(own_exp(scaled_x(l, mx, invT)));
}

__device__ __forceinline__ unsigned long long kept(unsigned long long W, int v, const RowStat& s) {
    return (W > s.tau || (W == s.tau && v <= s.cut)) ? W : 0ull;
}

// Log-scale bucket of W > 0: exact below 16, then the binade and 3 more bits.
__device__ __forceinline__ int log_bucket(unsigned long long W) {
    if (W < 16ull) return static_cast<int>(W);
    const int msb = 63 - __clzll(static_cast<long long>(W));
    return 16 + (msb - 4) * 8 + static_cast<int>((W >> (msb - 3)) & 7ull);
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

__device__ __forceinline__ void philox_at(unsigned long long seed, unsigned long long offset,
                                          uint32_t i, uint32_t b, uint32_t r[4]) {
    philox4x32_10(i, b, static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), r);
}

// ------------------------------------------------------- block reductions
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int o) {
    const unsigned long long lo = static_cast<unsigned long long>(v);
    const unsigned long long hi = static_cast<unsigned long long>(v >> 64);
    const unsigned long long l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    const unsigned long long h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    return (static_cast<u128>(h2) << 64) | l2;
}

__device__ __forceinline__ u128 shfl_up_u128(u128 v, int o) {
    const unsigned long long lo = static_cast<unsigned long long>(v);
    const unsigned long long hi = static_cast<unsigned long long>(v >> 64);
    const unsigned long long l2 = __shfl_up_sync(0xffffffffu, lo, o);
    const unsigned long long h2 = __shfl_up_sync(0xffffffffu, hi, o);
    return (static_cast<u128>(h2) << 64) | l2;
}

// floor(u * R / 2^64) for a 64-bit u and a 128-bit R (< 2^120 here)
__device__ __forceinline__ u128 scale_u64(unsigned long long u, u128 R) {
    const unsigned long long rlo = static_cast<unsigned long long>(R);
    const unsigned long long rhi = static_cast<unsigned long long>(R >> 64);
    const u128 lo = static_cast<u128>(u) * rlo;
    const u128 hi = static_cast<u128>(u) * rhi;
    return (lo >> 64) + hi;
}

// ------------------------------------------------------ kernel 1: row stats
struct StatSmem {
    unsigned int cnt[2][kLogBuckets];
    unsigned long long mass[2][kLogBuckets];
    unsigned int mcnt[kLogBuckets];
    unsigned long long mmass[kLogBuckets];
    float fred[kStatThreads / 32];
    unsigned long long ured[kStatThreads / 32];
    float lmax;               // this CTA's max (read by peers)
    unsigned long long lsum;  // this CTA's sum of W (read by peers)
    unsigned int lcnt;        // this CTA's count of W == tau (read by peers)
    // broadcast from thread 0
    unsigned long long lo, width, above, n_eq;
    int wbits, done, cut_found;
};

__global__ void __launch_bounds__(kStatThreads) row_stats_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, int Kd, int V, int slice,
    float invT, unsigned long long P, RowStat* __restrict__ stats) {
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ float s_e[];
    __shared__ StatSmem sm;
    const int C = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const long long row = blockIdx.x / C;
    const int per = 2 * Kd + 1;
    const long long b = row / per;
    const int i = static_cast<int>(row % per);
    const float* src = (i <= Kd) ? target + (b * (Kd + 1) + i) * static_cast<long long>(V)
                                 : draft + (b * Kd + (i - Kd - 1)) * static_cast<long long>(V);
    const int lo = rank * slice;
    const int n = (lo < V) ? ((V - lo < slice) ? V - lo : slice) : 0;

    // 1. load the slice and reduce the max over the cluster
    float lmax = -INFINITY;
    for (int k = tid; k < n; k += kStatThreads) {
        const float v = __ldg(src + lo + k);
        s_e[k] = v;
        lmax = fmaxf(lmax, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    if (lane == 0) sm.fred[wid] = lmax;
    __syncthreads();
    if (tid == 0) {
        float m = -INFINITY;
        for (int w = 0; w < kStatThreads / 32; ++w) m = fmaxf(m, sm.fred[w]);
        sm.lmax = m;
    }
    cl.sync();
    float mx = -INFINITY;
    for (int r = 0; r < C; ++r) mx = fmaxf(mx, *cl.map_shared_rank(&sm.lmax, r));

    // 2. e_v and the total mass
    unsigned long long lsum = 0;
    for (int k = tid; k < n; k += kStatThreads) {
        const float e = own_exp(scaled_x(s_e[k], mx, invT));
        s_e[k] = e;
        lsum += mass_of(e);
    }
    lsum = warp_sum_u64(lsum);
    if (lane == 0) sm.ured[wid] = lsum;
    for (int t = tid; t < kLogBuckets; t += kStatThreads) {
        sm.cnt[0][t] = 0u;
        sm.mass[0][t] = 0ull;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < kStatThreads / 32; ++w) s += sm.ured[w];
        sm.lsum = s;
    }
    cl.sync();
    unsigned long long S = 0;
    for (int r = 0; r < C; ++r) S += *cl.map_shared_rank(&sm.lsum, r);

    RowStat out;
    out.mx = mx;
    out.pad = 0;
    if (P >= kKeepAll) {
        if (rank == 0 && tid == 0) {
            out.tau = 0;
            out.cut = V - 1;
            out.S = S;
            stats[row] = out;
        }
        cl.sync();
        return;
    }
    const u128 TGT = static_cast<u128>(P) * S;

    // 3. log-scale histogram of W > 0
    for (int k = tid; k < n; k += kStatThreads) {
        const unsigned long long W = mass_of(s_e[k]);
        if (W == 0ull) continue;
        const int bk = log_bucket(W);
        atomicAdd(&sm.cnt[0][bk], 1u);
        atomicAdd(&sm.mass[0][bk], W);
    }
    __syncthreads();
    cl.sync();
    for (int t = tid; t < kLogBuckets; t += kStatThreads) {
        unsigned int c = 0;
        unsigned long long m = 0;
        for (int r = 0; r < C; ++r) {
            c += cl.map_shared_rank(&sm.cnt[0][0], r)[t];
            m += cl.map_shared_rank(&sm.mass[0][0], r)[t];
        }
        sm.mcnt[t] = c;
        sm.mmass[t] = m;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long above = 0;
        int beta = 1;
        for (int t = kLogBuckets - 1; t >= 1; --t) {
            if ((static_cast<u128>(above + sm.mmass[t]) << 32) >= TGT) {
                beta = t;
                break;
            }
            above += sm.mmass[t];
        }
        sm.above = above;
        if (beta < 16) {
            sm.lo = static_cast<unsigned long long>(beta);
            sm.width = 1;
            sm.wbits = 0;
            sm.n_eq = sm.mcnt[beta];
        } else {
            const int msb = 4 + (beta - 16) / 8, j = (beta - 16) % 8;
            sm.wbits = msb - 3;
            sm.lo = static_cast<unsigned long long>(8 + j) << sm.wbits;
            sm.width = 1ull << sm.wbits;
            sm.n_eq = 0;
        }
    }
    __syncthreads();

    // 4. refine inside the crossing bucket, 8 bits at a time
    int buf = 0;
    while (sm.width > 1ull) {
        buf ^= 1;
        const int wbits = sm.wbits;
        const int bits = wbits < 8 ? wbits : 8;
        const int shift = wbits - bits;
        const unsigned long long rlo = sm.lo, rhi = sm.lo + sm.width;
        for (int t = tid; t < kLinBuckets; t += kStatThreads) {
            sm.cnt[buf][t] = 0u;
            sm.mass[buf][t] = 0ull;
        }
        __syncthreads();
        for (int k = tid; k < n; k += kStatThreads) {
            const unsigned long long W = mass_of(s_e[k]);
            if (W < rlo || W >= rhi) continue;
            const int bk = static_cast<int>((W - rlo) >> shift);
            atomicAdd(&sm.cnt[buf][bk], 1u);
            atomicAdd(&sm.mass[buf][bk], W);
        }
        __syncthreads();
        cl.sync();
        for (int t = tid; t < (1 << bits); t += kStatThreads) {
            unsigned int c = 0;
            unsigned long long m = 0;
            for (int r = 0; r < C; ++r) {
                c += cl.map_shared_rank(&sm.cnt[buf][0], r)[t];
                m += cl.map_shared_rank(&sm.mass[buf][0], r)[t];
            }
            sm.mcnt[t] = c;
            sm.mmass[t] = m;
        }
        __syncthreads();
        if (tid == 0) {
            unsigned long long above = sm.above;
            int sb = 0;
            for (int t = (1 << bits) - 1; t >= 0; --t) {
                if ((static_cast<u128>(above + sm.mmass[t]) << 32) >= TGT) {
                    sb = t;
                    break;
                }
                above += sm.mmass[t];
            }
            sm.above = above;
            sm.lo = rlo + (static_cast<unsigned long long>(sb) << shift);
            sm.width = 1ull << shift;
            sm.wbits = shift;
            if (shift == 0) sm.n_eq = sm.mcnt[sb];
        }
        __syncthreads();
    }
    const unsigned long long tau = sm.lo, above = sm.above, n_eq = sm.n_eq;
    // smallest j >= 1 with (above + j*tau) * 2^32 >= P*S
    const u128 num = TGT - (static_cast<u128>(above) << 32);
    const u128 den = static_cast<u128>(tau) << 32;
    const unsigned long long jneed = static_cast<unsigned long long>((num + den - 1) / den);
    out.tau = tau;
    out.S = above + jneed * tau;
    if (jneed >= n_eq) {
        if (rank == 0 && tid == 0) {
            out.cut = V - 1;
            stats[row] = out;
        }
        cl.sync();
        return;
    }

    // 5. the jneed-th element with W == tau in index order sets the cut
    const int chunk = (n + kStatThreads - 1) / kStatThreads;
    const int k0 = tid * chunk, k1 = (k0 + chunk < n) ? k0 + chunk : n;
    unsigned int mine = 0;
    for (int k = k0; k < k1; ++k) mine += (mass_of(s_e[k]) == tau) ? 1u : 0u;
    // block exclusive scan of mine
    unsigned int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm.ured[wid] = incl;
    __syncthreads();
    if (tid == 0) {
        unsigned long long run = 0;
        for (int w = 0; w < kStatThreads / 32; ++w) {
            const unsigned long long x = sm.ured[w];
            sm.ured[w] = run;
            run += x;
        }
        sm.lcnt = static_cast<unsigned int>(run);
    }
    __syncthreads();
    const unsigned long long excl = sm.ured[wid] + (incl - mine);
    cl.sync();
    unsigned long long before = 0;
    for (int r = 0; r < rank; ++r) before += *cl.map_shared_rank(&sm.lcnt, r);
    const unsigned long long need = jneed - before;  // 1-based within this CTA
    if (before < jneed && jneed <= before + sm.lcnt && excl < need && need <= excl + mine) {
        unsigned long long seen = excl;
        for (int k = k0; k < k1; ++k) {
            if (mass_of(s_e[k]) == tau && ++seen == need) {
                out.cut = lo + k;
                stats[row] = out;
                break;
            }
        }
    }
    cl.sync();
}

// ---------------------------------------------------- kernel 2: decisions
__global__ void decide_kernel(const float* __restrict__ target, const float* __restrict__ draft,
                              const int32_t* __restrict__ drafts, int B, int Kd, int V,
                              float invT, unsigned long long seed, unsigned long long offset,
                              const RowStat* __restrict__ stats, SeqState* __restrict__ seq,
                              int32_t* __restrict__ tokens, int32_t* __restrict__ len,
                              uint32_t* status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int per = 2 * Kd + 1;
    int n = 0;
    SeqState st;
    st.mode = 1;
    st.pos = Kd;
    st.pad = 0;
    uint32_t r[4];
    for (int i = 0; i < Kd; ++i) {
        const int32_t x = drafts[static_cast<long long>(b) * Kd + i];
        philox_at(seed, offset, static_cast<uint32_t>(i), static_cast<uint32_t>(b), r);
        const unsigned long long u64 = (static_cast<unsigned long long>(r[2]) << 32) | r[1];
        bool ok = false;
        if (x >= 0 && x < V) {
            const RowStat sp = stats[static_cast<long long>(b) * per + i];
            const RowStat sq = stats[static_cast<long long>(b) * per + Kd + 1 + i];
            const float lp = target[(static_cast<long long>(b) * (Kd + 1) + i) * V + x];
            const float lq = draft[(static_cast<long long>(b) * Kd + i) * V + x];
            const unsigned long long Wp = kept(mass_at(lp, sp.mx, invT), x, sp);
            const unsigned long long Wq = kept(mass_at(lq, sq.mx, invT), x, sq);
            const unsigned long long U = r[0] >> 8;
            const u128 lhs = static_cast<u128>(U * Wq) * sp.S;
            const u128 rhs = (static_cast<u128>(Wp) * sq.S) << 24;
            ok = lhs < rhs;
        } else {
            atomicOr(status, kStatusBadDraft);
        }
        if (ok) {
            ++n;
            continue;
        }
        st.mode = 0;
        st.pos = i;
        st.u64 = u64;
        break;
    }
    if (n == Kd) {
        philox_at(seed, offset, static_cast<uint32_t>(Kd), static_cast<uint32_t>(b), r);
        st.u64 = (static_cast<unsigned long long>(r[2]) << 32) | r[1];
    }
    st.n = n;
    seq[b] = st;
    for (int i = 0; i <= Kd; ++i) {
        if (i < n) tokens[static_cast<long long>(b) * (Kd + 1) + i] = drafts[static_cast<long long>(b) * Kd + i];
        else if (i > n) tokens[static_cast<long long>(b) * (Kd + 1) + i] = -1;
    }
    len[b] = n + 1;
}

// ----------------------------------------------------- kernel 3: the draw
struct SampleSmem {
    unsigned long long lo[kSampleThreads / 32];
    unsigned long long hi[kSampleThreads / 32];
    int found;
};

__device__ __forceinline__ u128 block_sum_u128(u128 v, SampleSmem& sm, int lane, int wid) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += shfl_xor_u128(v, o);
    if (lane == 0) {
        sm.lo[wid] = static_cast<unsigned long long>(v);
        sm.hi[wid] = static_cast<unsigned long long>(v >> 64);
    }
    __syncthreads();
    u128 t = 0;
    for (int w = 0; w < kSampleThreads / 32; ++w)
        t += (static_cast<u128>(sm.hi[w]) << 64) | sm.lo[w];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(
    const float* __restrict__ target, const float* __restrict__ draft, int Kd, int V, float invT,
    const RowStat* __restrict__ stats, const SeqState* __restrict__ seq,
    int32_t* __restrict__ tokens, uint32_t* status) {
    __shared__ SampleSmem sm;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const SeqState st = seq[b];
    const int per = 2 * Kd + 1;
    const int pos = st.pos;
    const RowStat sp = stats[static_cast<long long>(b) * per + pos];
    const float* lp = target + (static_cast<long long>(b) * (Kd + 1) + pos) * V;
    bool residual = (st.mode == 0);
    RowStat sq{};
    const float* lq = nullptr;
    if (residual) {
        sq = stats[static_cast<long long>(b) * per + Kd + 1 + pos];
        lq = draft + (static_cast<long long>(b) * Kd + pos) * V;
    }
    // weight of token v under the chosen rule
    auto weight = [&](int v, bool res) -> u128 {
        const unsigned long long wp = kept(mass_at(__ldg(lp + v), sp.mx, invT), v, sp);
        if (!res) return static_cast<u128>(wp);
        const unsigned long long wq = kept(mass_at(__ldg(lq + v), sq.mx, invT), v, sq);
        const u128 a = static_cast<u128>(wp) * sq.S, c = static_cast<u128>(wq) * sp.S;
        return a > c ? a - c : static_cast<u128>(0);
    };
    u128 total;
    if (residual) {
        u128 part = 0;
        for (int v = tid; v < V; v += kSampleThreads) part += weight(v, true);
        total = block_sum_u128(part, sm, lane, wid);
        if (total == 0) {  // only reachable through an invalid draft id
            residual = false;
            if (tid == 0) atomicOr(status, kStatusZeroResidual);
        }
    }
    if (!residual) total = static_cast<u128>(sp.S);
    const u128 t = scale_u64(st.u64, total);
    // ordered scan, 4 consecutive tokens per thread per tile
    if (tid == 0) sm.found = -1;
    __syncthreads();
    u128 run = 0;
    constexpr int kTile = 4 * kSampleThreads;
    for (int base = 0; base < V; base += kTile) {
        const int v0 = base + 4 * tid;
        u128 w[4];
        u128 mine = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[q] = (v0 + q < V) ? weight(v0 + q, residual) : static_cast<u128>(0);
            mine += w[q];
        }
        u128 incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const u128 y = shfl_up_u128(incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) {
            sm.lo[wid] = static_cast<unsigned long long>(incl);
            sm.hi[wid] = static_cast<unsigned long long>(incl >> 64);
        }
        __syncthreads();
        u128 wbase = 0, tile_total = 0;
        for (int w2 = 0; w2 < kSampleThreads / 32; ++w2) {
            const u128 x = (static_cast<u128>(sm.hi[w2]) << 64) | sm.lo[w2];
            if (w2 < wid) wbase += x;
            tile_total += x;
        }
        __syncthreads();
        const u128 excl = run + wbase + (incl - mine);
        if (excl <= t && t < excl + mine) {
            u128 c = excl;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                c += w[q];
                if (c > t) {
                    sm.found = v0 + q;
                    break;
                }
            }
        }
        __syncthreads();
        if (sm.found >= 0) break;
        run += tile_total;
    }
    if (tid == 0) {
        const int tok = sm.found >= 0 ? sm.found : V - 1;
        tokens[static_cast<long long>(b) * (Kd + 1) + st.n] = tok;
    }
}

__global__ void own_exp_kernel(const float* __restrict__ x, float* __restrict__ y, long long n) {
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        y[i] = own_exp(x[i]);
}

int cluster_for(int V) {
    int c = (V + 16383) / 16384;
    return c < 1 ? 1 : (c > 8 ? 8 : c);
}

}  // namespace

cudaError_t launch_own_exp(const float* x, float* y, long long n, cudaStream_t s) {
    long long blocks = (n + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    if (blocks < 1) blocks = 1;
    own_exp_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(x, y, n);
    return cudaGetLastError();
}

size_t rejection_workspace_bytes(int B, int Kd, int V) {
    (void)V;
    const size_t rows = static_cast<size_t>(B) * (2 * Kd + 1);
    return ((rows * sizeof(RowStat) + 255) / 256) * 256 + ((B * sizeof(SeqState) + 255) / 256) * 256;
}

cudaError_t launch_accept_rejection(const float* target, const float* draft,
                                    const int32_t* drafts, int B, int Kd, int V, float invT,
                                    uint64_t P, uint64_t seed, uint64_t offset, int32_t* tokens,
                                    int32_t* len, void* ws, size_t ws_bytes, uint32_t* status,
                                    cudaStream_t s) {
    const int C = cluster_for(V);
    int slice = (V + C - 1) / C;
    slice = (slice + 3) & ~3;
    if (slice > kMaxSlice) return cudaErrorNotSupported;
    const size_t rows = static_cast<size_t>(B) * (2 * Kd + 1);
    if (rows * C > 0x7fffffffull) return cudaErrorNotSupported;
    char* base = static_cast<char*>(ws);
    RowStat* stats = reinterpret_cast<RowStat*>(base);
    SeqState* seq = reinterpret_cast<SeqState*>(base + ((rows * sizeof(RowStat) + 255) / 256) * 256);
    if (rejection_workspace_bytes(B, Kd, V) > ws_bytes) return cudaErrorInvalidValue;

    const size_t smem = static_cast<size_t>(slice) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(row_stats_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(rows * C));
    cfg.blockDim = dim3(kStatThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, row_stats_kernel, target, draft, Kd, V, slice, invT,
                           static_cast<unsigned long long>(P), stats);
    if (e != cudaSuccess) return e;
    decide_kernel<<<(B + 127) / 128, 128, 0, s>>>(target, draft, drafts, B, Kd, V, invT, seed,
                                                   offset, stats, seq, tokens, len, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sample_kernel<<<B, kSampleThreads, 0, s>>>(target, draft, Kd, V, invT, stats, seq, tokens,
                                               status);
    return cudaGetLastError();
}

}  // namespace vw4
