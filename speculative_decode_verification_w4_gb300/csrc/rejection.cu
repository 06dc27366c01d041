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
// Kernel 1, one thread-block cluster per (sequence b, position i):
//   * the target row (b, i) and, for i < Kd, the draft row (b, i) are loaded
//     once into the cluster's shared memory, a slice per CTA;
//   * per row: max and sum W over the cluster (DSMEM), a log-scale histogram
//     of W finds the bucket where the top-p prefix ends; its members are
//     gathered to rank 0, sorted by (W desc, index asc) and scanned, which
//     gives the exact cut (an exact radix search over the slices is the
//     fallback when that bucket is too crowded);
//   * the acceptance test of draft i (Philox block (i, b)), and, only if it
//     is rejected, the residual draw -- or, for i = Kd, the bonus draw --
//     from the rows already on chip: an exact u128 total, then an ordered
//     search across the cluster's slices.
// Kernel 2, one thread per sequence: the first rejected position decides the
// committed run.  Rows after the first rejection are evaluated in parallel
// and discarded.
#include <cooperative_groups.h>

#include "ptx.cuh"
#include "vw4_internal.cuh"

namespace cg = cooperative_groups;

namespace vw4 {

namespace {

constexpr uint32_t kStatusBadDraft = 0x1u;
constexpr uint32_t kStatusZeroResidual = 0x8u;
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kLogBuckets = 16 + 37 * 8;  // exact 0..15, then 8 per binade up to 2^40
constexpr int kLinBuckets = 256;
constexpr int kCandLocal = 512;   // candidates one CTA may hold per row
constexpr int kCandTotal = 2048;  // candidates the cluster may gather per row
constexpr int kMaxSlice = 20480;  // floats per CTA per row (two rows on chip)
constexpr unsigned long long kKeepAll = 1ull << 32;

typedef unsigned __int128 u128;

struct RowInfo {
    float mx;
    int cut;                 // largest kept index among W == tau
    unsigned long long tau;  // kept: W > tau, or W == tau and v <= cut
    unsigned long long S;    // kept sum
};

struct PairOut {
    int accept;  // 1: draft i accepted (or the bonus row)
    int token;   // residual draw at a rejection; bonus draw for i == Kd
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

__device__ __forceinline__ unsigned long long kept(unsigned long long W, int v, const RowInfo& s) {
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

// floor(u * R / 2^64) for a 64-bit u and a 128-bit R (< 2^120 here)
__device__ __forceinline__ u128 scale_u64(unsigned long long u, u128 R) {
    const u128 lo = static_cast<u128>(u) * static_cast<unsigned long long>(R);
    const u128 hi = static_cast<u128>(u) * static_cast<unsigned long long>(R >> 64);
    return (lo >> 64) + hi;
}

struct Smem {
    unsigned int cnt[kLogBuckets];         // this CTA's histogram (read by peers)
    unsigned long long mass[kLogBuckets];
    unsigned int mcnt[kLogBuckets];        // the cluster's merged histogram
    unsigned long long mmass[kLogBuckets];
    unsigned long long cw[kCandLocal];     // this CTA's candidates (read by rank 0)
    int ci[kCandLocal];
    unsigned long long gw[kCandTotal];     // rank 0: gathered, sorted candidates
    int gi[kCandTotal];
    unsigned long long wred[kWarps];
    unsigned long long wred2[kWarps];
    float fred[kWarps];
    // values peers read over DSMEM
    float lmax;
    unsigned long long lsum;
    unsigned int ncand;
    int overflow;
    unsigned long long part_lo, part_hi;   // this CTA's u128 partial total
    RowInfo info;                          // rank 0's result for the current row
    int decision;
    // broadcast inside the CTA
    int beta, wbits;
    unsigned long long lo, width, above, n_eq, count_eq;
    int cut_found;
};

__device__ __forceinline__ float block_max(float v, Smem& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) sm.fred[wid] = v;
    __syncthreads();
    float m = -INFINITY;
    for (int w = 0; w < kWarps; ++w) m = fmaxf(m, sm.fred[w]);
    __syncthreads();
    return m;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, Smem& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sm.wred[wid] = v;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < kWarps; ++w) t += sm.wred[w];
    __syncthreads();
    return t;
}

__device__ __forceinline__ u128 block_sum_u128(u128 v, Smem& sm) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += shfl_xor_u128(v, o);
    if (lane == 0) {
        sm.wred[wid] = static_cast<unsigned long long>(v);
        sm.wred2[wid] = static_cast<unsigned long long>(v >> 64);
    }
    __syncthreads();
    u128 t = 0;
    for (int w = 0; w < kWarps; ++w) t += (static_cast<u128>(sm.wred2[w]) << 64) | sm.wred[w];
    __syncthreads();
    return t;
}

// Exclusive prefix over the block of a u128 value per thread; also returns the total.
__device__ __forceinline__ u128 block_excl_u128(u128 v, Smem& sm, u128& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    u128 incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u128 y = shfl_up_u128(incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) {
        sm.wred[wid] = static_cast<unsigned long long>(incl);
        sm.wred2[wid] = static_cast<unsigned long long>(incl >> 64);
    }
    __syncthreads();
    u128 base = 0, t = 0;
    for (int w = 0; w < kWarps; ++w) {
        const u128 x = (static_cast<u128>(sm.wred2[w]) << 64) | sm.wred[w];
        if (w < wid) base += x;
        t += x;
    }
    __syncthreads();
    total = t;
    return base + incl - v;
}

// ----------------------------------------------------------- row statistics
// s holds this CTA's slice [lo, lo + n) of the row's logits on entry and the
// own_exp values on exit.  Every CTA of the cluster returns the same RowInfo.
__device__ RowInfo row_stats(cg::cluster_group& cl, float* s, int n, int lo, int V, float invT,
                             unsigned long long P, Smem& sm) {
    const int C = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;

    // 1. max over the cluster
    float lmax = -INFINITY;
    for (int k = tid; k < n; k += kThreads) lmax = fmaxf(lmax, s[k]);
    lmax = block_max(lmax, sm);
    if (tid == 0) sm.lmax = lmax;
    for (int t = tid; t < kLogBuckets; t += kThreads) {
        sm.cnt[t] = 0u;
        sm.mass[t] = 0ull;
    }
    cl.sync();
    float mx = -INFINITY;
    for (int r = 0; r < C; ++r) mx = fmaxf(mx, *cl.map_shared_rank(&sm.lmax, r));

    // 2. e_v, the total mass and the log-scale histogram in one pass
    unsigned long long lsum = 0;
    for (int k = tid; k < n; k += kThreads) {
        const float e = own_exp(scaled_x(s[k], mx, invT));
        s[k] = e;
        const unsigned long long W = mass_of(e);
        lsum += W;
        if (W != 0ull && P < kKeepAll) atomicAdd(&sm.mass[log_bucket(W)], W);
    }
    lsum = block_sum_u64(lsum, sm);
    if (tid == 0) sm.lsum = lsum;
    cl.sync();
    unsigned long long S = 0;
    for (int r = 0; r < C; ++r) S += *cl.map_shared_rank(&sm.lsum, r);
    RowInfo info;
    info.mx = mx;
    if (P >= kKeepAll) {
        info.cut = V - 1;
        info.tau = 0;
        info.S = S;
        cl.sync();  // peers are done reading this CTA's values
        return info;
    }
    const u128 TGT = static_cast<u128>(P) * S;
    // merged bucket masses, then a block-wide suffix sum: the crossing bucket
    // beta is the highest bucket whose suffix mass reaches the target
    unsigned long long m = 0;
    const int tb = kLogBuckets - 1 - tid;  // thread tid holds bucket 311 - tid
    if (tb >= 1) {
        for (int r = 0; r < C; ++r) m += cl.map_shared_rank(&sm.mass[0], r)[tb];
        sm.mmass[tb] = m;
    }
    u128 tot_unused;
    const u128 incl = block_excl_u128(static_cast<u128>(m), sm, tot_unused) + m;  // mass of >= tb
    if (tid == 0) {
        sm.ncand = 0;
        sm.overflow = 0;
    }
    if (tb >= 1 && (incl << 32) >= TGT && ((incl - m) << 32) < TGT) {
        sm.beta = tb;
        sm.above = static_cast<unsigned long long>(incl - m);
    }
    __syncthreads();

    // 3. gather the members of the crossing bucket
    const int beta = sm.beta;
    const int lane = tid & 31;
    for (int k0 = tid - lane; k0 < n; k0 += kThreads) {  // warp-uniform trip count
        const int k = k0 + lane;
        const unsigned long long W = k < n ? mass_of(s[k]) : 0ull;
        const bool hit = W != 0ull && log_bucket(W) == beta;
        const unsigned int ball = __ballot_sync(0xffffffffu, hit);
        if (ball == 0u) continue;
        unsigned int base = 0;
        if (lane == 0) base = atomicAdd(&sm.ncand, static_cast<unsigned int>(__popc(ball)));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (hit) {
            const unsigned int slot = base + __popc(ball & ((1u << lane) - 1u));
            if (slot < static_cast<unsigned int>(kCandLocal)) {
                sm.cw[slot] = W;
                sm.ci[slot] = lo + k;
            } else {
                sm.overflow = 1;
            }
        }
    }
    __syncthreads();
    cl.sync();
    unsigned int total = 0;
    int overflow = 0;
    for (int r = 0; r < C; ++r) {
        total += *cl.map_shared_rank(&sm.ncand, r);
        overflow |= *cl.map_shared_rank(&sm.overflow, r);
    }
    if (!overflow && total <= static_cast<unsigned int>(kCandTotal)) {
        if (rank == 0) {
            // gather, pad to a power of two, bitonic sort by (W desc, index asc)
            unsigned int pw = 1;
            while (pw < total) pw <<= 1;
            unsigned int base = 0;
            for (int r = 0; r < C; ++r) {
                const unsigned int cr = *cl.map_shared_rank(&sm.ncand, r);
                const unsigned long long* rw = cl.map_shared_rank(&sm.cw[0], r);
                const int* ri = cl.map_shared_rank(&sm.ci[0], r);
                for (unsigned int t = tid; t < cr; t += kThreads) {
                    sm.gw[base + t] = rw[t];
                    sm.gi[base + t] = ri[t];
                }
                base += cr;
            }
            for (unsigned int t = total + tid; t < pw; t += kThreads) {
                sm.gw[t] = 0ull;
                sm.gi[t] = 0x7fffffff;
            }
            __syncthreads();
            for (unsigned int kk = 2; kk <= pw; kk <<= 1) {
                for (unsigned int j = kk >> 1; j > 0; j >>= 1) {
                    for (unsigned int t = tid; t < pw; t += kThreads) {
                        const unsigned int u = t ^ j;
                        if (u > t) {
                            const unsigned long long wa = sm.gw[t], wb = sm.gw[u];
                            const int ia = sm.gi[t], ib = sm.gi[u];
                            const bool a_first = wa > wb || (wa == wb && ia < ib);
                            const bool up = (t & kk) == 0;
                            if (up != a_first) {
                                sm.gw[t] = wb;
                                sm.gw[u] = wa;
                                sm.gi[t] = ib;
                                sm.gi[u] = ia;
                            }
                        }
                    }
                    __syncthreads();
                }
            }
            // running mass down the sorted list; the first crossing is the cut
            const unsigned int t0 = 2 * tid;
            const unsigned long long w0 = t0 < total ? sm.gw[t0] : 0ull;
            const unsigned long long w1 = t0 + 1 < total ? sm.gw[t0 + 1] : 0ull;
            u128 tot;
            const u128 ex = block_excl_u128(static_cast<u128>(w0) + w1, sm, tot);
            const u128 above = sm.above;
            const u128 c0 = above + ex + w0, c1 = c0 + w1;
            if (t0 < total && (c0 << 32) >= TGT && ((above + ex) << 32) < TGT) {
                sm.info.tau = w0;
                sm.info.cut = sm.gi[t0];
                sm.info.S = static_cast<unsigned long long>(c0);
            } else if (t0 + 1 < total && (c1 << 32) >= TGT && (c0 << 32) < TGT) {
                sm.info.tau = w1;
                sm.info.cut = sm.gi[t0 + 1];
                sm.info.S = static_cast<unsigned long long>(c1);
            }
        }
        cl.sync();
        const RowInfo* r0 = cl.map_shared_rank(&sm.info, 0);
        info.tau = r0->tau;
        info.cut = r0->cut;
        info.S = r0->S;
        cl.sync();  // rank 0's result stays until everyone has it
        return info;
    }

    // 4. fallback: exact radix search over the slices inside the bucket
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
        cl.sync();  // peers finished reading this CTA's previous histogram
        for (int t = tid; t < kLinBuckets; t += kThreads) {
            sm.cnt[t] = 0u;
            sm.mass[t] = 0ull;
        }
        __syncthreads();
        for (int k = tid; k < n; k += kThreads) {
            const unsigned long long W = mass_of(s[k]);
            if (W < rlo || W >= rhi) continue;
            const int bk = static_cast<int>((W - rlo) >> shift);
            atomicAdd(&sm.cnt[bk], 1u);
            atomicAdd(&sm.mass[bk], W);
        }
        cl.sync();
        for (int t = tid; t < (1 << bits); t += kThreads) {
            unsigned int c = 0;
            unsigned long long m = 0;
            for (int r = 0; r < C; ++r) {
                c += cl.map_shared_rank(&sm.cnt[0], r)[t];
                m += cl.map_shared_rank(&sm.mass[0], r)[t];
            }
            sm.mcnt[t] = c;
            sm.mmass[t] = m;
        }
        __syncthreads();
        {
            const int nb = 1 << bits;
            const int t = nb - 1 - tid;  // thread tid holds sub-bucket nb - 1 - tid
            const unsigned long long mt = t >= 0 ? sm.mmass[t] : 0ull;
            u128 tot2;
            const u128 inc = block_excl_u128(static_cast<u128>(mt), sm, tot2) + mt;
            const u128 ab = static_cast<u128>(sm.above);
            if (t >= 0 && ((ab + inc) << 32) >= TGT && ((ab + inc - mt) << 32) < TGT) {
                sm.beta = t;
                sm.lo = rlo + (static_cast<unsigned long long>(t) << shift);
                sm.n_eq = sm.mcnt[t];
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
    // the jneed-th element with W == tau in index order sets the cut
    const int chunk = (n + kThreads - 1) / kThreads;
    const int k0 = tid * chunk, k1 = (k0 + chunk < n) ? k0 + chunk : n;
    unsigned int mine = 0;
    for (int k = k0; k < k1; ++k) mine += (mass_of(s[k]) == tau) ? 1u : 0u;
    u128 ctot;
    const unsigned long long excl =
        static_cast<unsigned long long>(block_excl_u128(static_cast<u128>(mine), sm, ctot));
    if (tid == 0) {
        sm.count_eq = static_cast<unsigned long long>(ctot);
        sm.cut_found = -1;
    }
    cl.sync();
    unsigned long long before = 0;
    for (int r = 0; r < rank; ++r) before += *cl.map_shared_rank(&sm.count_eq, r);
    const unsigned long long need = jneed - before;  // 1-based inside this CTA
    if (jneed < n_eq && before < jneed && jneed <= before + sm.count_eq && excl < need &&
        need <= excl + mine) {
        unsigned long long seen = excl;
        for (int k = k0; k < k1; ++k)
            if (mass_of(s[k]) == tau && ++seen == need) {
                sm.cut_found = lo + k;
                break;
            }
    }
    cl.sync();
    if (jneed < n_eq) {
        int cut = -1;
        for (int r = 0; r < C; ++r) {
            const int x = *cl.map_shared_rank(&sm.cut_found, r);
            if (x >= 0) cut = x;
        }
        info.cut = cut;
    }
    cl.sync();
    return info;
}

// --------------------------------------------------- ordered categorical draw
// Weight of slice element k: the residual r_v (res) or the kept target mass.
struct Weights {
    const float* ep;
    const float* eq;
    RowInfo ip, iq;
    bool res;
    int lo;
    __device__ __forceinline__ u128 at(int k) const {
        const int v = lo + k;
        const unsigned long long wp = kept(mass_of(ep[k]), v, ip);
        if (!res) return static_cast<u128>(wp);
        const unsigned long long wq = kept(mass_of(eq[k]), v, iq);
        const u128 a = static_cast<u128>(wp) * iq.S, c = static_cast<u128>(wq) * ip.S;
        return a > c ? a - c : static_cast<u128>(0);
    }
};

// Sum of the weights of this CTA's slice (every thread gets it).
__device__ __forceinline__ u128 slice_total(const Weights& w, int n, Smem& sm) {
    u128 part = 0;
    for (int k = threadIdx.x; k < n; k += kThreads) part += w.at(k);
    return block_sum_u128(part, sm);
}

// Returns (to every CTA) the first index whose running weight sum exceeds
// floor(u64 * total / 2^64); `mine` is this CTA's slice total.
__device__ int ordered_draw(cg::cluster_group& cl, const Weights& w, int n, u128 mine, u128 total,
                            unsigned long long u64, Smem& sm) {
    const int C = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    const u128 t = scale_u64(u64, total);
    if (tid == 0) {
        sm.part_lo = static_cast<unsigned long long>(mine);
        sm.part_hi = static_cast<unsigned long long>(mine >> 64);
        sm.cut_found = -1;
    }
    cl.sync();
    u128 before = 0;
    for (int r = 0; r < rank; ++r)
        before += (static_cast<u128>(*cl.map_shared_rank(&sm.part_hi, r)) << 64) |
                  *cl.map_shared_rank(&sm.part_lo, r);
    if (before <= t && t < before + mine) {  // the draw lands in this CTA's slice
        const int chunk = (n + kThreads - 1) / kThreads;
        const int k0 = tid * chunk, k1 = (k0 + chunk < n) ? k0 + chunk : n;
        u128 own = 0;
        for (int k = k0; k < k1; ++k) own += w.at(k);
        u128 tot;
        const u128 ex = before + block_excl_u128(own, sm, tot);
        if (ex <= t && t < ex + own) {
            u128 run = ex;
            for (int k = k0; k < k1; ++k) {
                run += w.at(k);
                if (run > t) {
                    sm.cut_found = w.lo + k;
                    break;
                }
            }
        }
    }
    cl.sync();
    int tok = -1;
    for (int r = 0; r < C; ++r) {
        const int x = *cl.map_shared_rank(&sm.cut_found, r);
        if (x >= 0) tok = x;
    }
    cl.sync();
    return tok;
}

__device__ __forceinline__ void load_slice(float* dst, const float* src, int n, bool vec) {
    if (vec) {
        const int n4 = n >> 2;
        const float4* s4 = reinterpret_cast<const float4*>(src);
        float4* d4 = reinterpret_cast<float4*>(dst);
        for (int k = threadIdx.x; k < n4; k += kThreads) d4[k] = __ldg(s4 + k);
        for (int k = 4 * n4 + threadIdx.x; k < n; k += kThreads) dst[k] = __ldg(src + k);
    } else {
        for (int k = threadIdx.x; k < n; k += kThreads) dst[k] = __ldg(src + k);
    }
}

__global__ void __launch_bounds__(kThreads, 1) pair_kernel(
    const float* __restrict__ target, const float* __restrict__ draft,
    const int32_t* __restrict__ drafts, int Kd, int V, int slice, int vec_ok, float invT,
    unsigned long long P, unsigned long long seed, unsigned long long offset,
    PairOut* __restrict__ out, uint32_t* status) {
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ float4 dyn[];
    __shared__ Smem sm;
    float* sp = reinterpret_cast<float*>(dyn);
    float* sq = sp + slice;
    const int C = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const long long pid = blockIdx.x / C;
    const long long b = pid / (Kd + 1);
    const int i = static_cast<int>(pid % (Kd + 1));
    const bool has_q = i < Kd;
    const int lo = rank * slice;
    const int n = (lo < V) ? ((V - lo < slice) ? V - lo : slice) : 0;
    const float* lp = target + (b * (Kd + 1) + i) * static_cast<long long>(V);
    const float* lq = has_q ? draft + (b * Kd + i) * static_cast<long long>(V) : nullptr;
    const bool vec = vec_ok != 0;  // rows start on 16-byte boundaries
    load_slice(sp, lp + lo, n, vec);
    if (has_q) load_slice(sq, lq + lo, n, vec);
    __syncthreads();

    const RowInfo ip = row_stats(cl, sp, n, lo, V, invT, P, sm);
    RowInfo iq{};
    if (has_q) iq = row_stats(cl, sq, n, lo, V, invT, P, sm);

    uint32_t rr[4];
    philox4x32_10(static_cast<uint32_t>(i), static_cast<uint32_t>(b),
                  static_cast<uint32_t>(offset), static_cast<uint32_t>(offset >> 32),
                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), rr);
    const unsigned long long u64 = (static_cast<unsigned long long>(rr[2]) << 32) | rr[1];

    Weights w{sp, sq, ip, iq, false, lo};
    if (!has_q) {  // the bonus row
        const u128 mine = slice_total(w, n, sm);
        const int tok = ordered_draw(cl, w, n, mine, static_cast<u128>(ip.S), u64, sm);
        if (rank == 0 && threadIdx.x == 0) out[pid] = PairOut{1, tok};
        return;
    }
    // the acceptance test of draft i
    if (rank == 0 && threadIdx.x == 0) {
        const int32_t x = drafts[b * Kd + i];
        int ok = 0;
        if (x >= 0 && x < V) {
            const unsigned long long Wp = kept(mass_of(own_exp(scaled_x(lp[x], ip.mx, invT))), x, ip);
            const unsigned long long Wq = kept(mass_of(own_exp(scaled_x(lq[x], iq.mx, invT))), x, iq);
            const unsigned long long U = rr[0] >> 8;
            const u128 lhs = static_cast<u128>(U * Wq) * ip.S;
            const u128 rhs = (static_cast<u128>(Wp) * iq.S) << 24;
            ok = lhs < rhs ? 1 : 0;
        } else {
            atomicOr(status, kStatusBadDraft);
        }
        sm.decision = ok;
    }
    cl.sync();
    const int ok = *cl.map_shared_rank(&sm.decision, 0);
    if (ok) {
        cl.sync();
        if (rank == 0 && threadIdx.x == 0) out[pid] = PairOut{1, -1};
        return;
    }
    // rejected: residual max(0, p*Sq - q*Sp) from the rows on chip
    w.res = true;
    u128 mine = slice_total(w, n, sm);
    if (threadIdx.x == 0) {
        sm.part_lo = static_cast<unsigned long long>(mine);
        sm.part_hi = static_cast<unsigned long long>(mine >> 64);
    }
    cl.sync();
    u128 R = 0;
    for (int r = 0; r < C; ++r)
        R += (static_cast<u128>(*cl.map_shared_rank(&sm.part_hi, r)) << 64) |
             *cl.map_shared_rank(&sm.part_lo, r);
    cl.sync();
    if (R == 0) {  // only reachable through an invalid draft id: draw from p
        if (rank == 0 && threadIdx.x == 0) atomicOr(status, kStatusZeroResidual);
        w.res = false;
        mine = slice_total(w, n, sm);
        R = static_cast<u128>(ip.S);
    }
    const int tok = ordered_draw(cl, w, n, mine, R, u64, sm);
    if (rank == 0 && threadIdx.x == 0) out[pid] = PairOut{0, tok};
}

// One thread per sequence: the first rejection decides the committed run.
__global__ void commit_kernel(const int32_t* __restrict__ drafts, const PairOut* __restrict__ pairs,
                              int B, int Kd, int32_t* __restrict__ tokens,
                              int32_t* __restrict__ len) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const PairOut* pr = pairs + static_cast<long long>(b) * (Kd + 1);
    int n = 0;
    while (n < Kd && pr[n].accept) ++n;
    for (int i = 0; i <= Kd; ++i) {
        int32_t t = -1;
        if (i < n) t = drafts[static_cast<long long>(b) * Kd + i];
        else if (i == n) t = pr[n].token;
        tokens[static_cast<long long>(b) * (Kd + 1) + i] = t;
    }
    len[b] = n + 1;
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
    const size_t pairs = static_cast<size_t>(B) * (Kd + 1);
    return ((pairs * sizeof(PairOut) + 255) / 256) * 256;
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
    const size_t pairs = static_cast<size_t>(B) * (Kd + 1);
    if (pairs * C > 0x7fffffffull) return cudaErrorNotSupported;
    if (rejection_workspace_bytes(B, Kd, V) > ws_bytes) return cudaErrorInvalidValue;
    PairOut* out = static_cast<PairOut*>(ws);

    const size_t smem = static_cast<size_t>(2) * slice * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(pairs * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int vec_ok = (V % 4 == 0 && (reinterpret_cast<uintptr_t>(target) & 15u) == 0 &&
                        (reinterpret_cast<uintptr_t>(draft) & 15u) == 0)
                           ? 1
                           : 0;
    e = cudaLaunchKernelEx(&cfg, pair_kernel, target, draft, drafts, Kd, V, slice, vec_ok, invT,
                           static_cast<unsigned long long>(P), static_cast<unsigned long long>(seed),
                           static_cast<unsigned long long>(offset), out, status);
    if (e != cudaSuccess) return e;
    commit_kernel<<<(B + 127) / 128, 128, 0, s>>>(drafts, out, B, Kd, tokens, len);
    return cudaGetLastError();
}

}  // namespace vw4
