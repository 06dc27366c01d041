// gemm_w4.cu -- the verification pass's skinny 4-bit-weight GEMM on sm_103a.
//
// What it computes ("Faster Gemma 4 on MLX with multi-token prediction",
// paragraph on the verify kernel; Qiita roofline article on MTP, PART 2 section
// 2-3): out[m][n] = sum_k A[m][k] * w[n][k] for M <= 8 verify rows, where each
// block-quantized weight is streamed from HBM and unpacked exactly once and
// then reused by all M rows.
//
// How (GB300 design):
//  * A persistent stream-K grid (2 CTAs per SM).  The work is the list of
//    units (tile of 128 weight rows, 256-wide k slice); CTA i owns the
//    contiguous unit range [i*U/G, (i+1)*U/G), so every CTA streams the same
//    number of weight bytes to within one unit.  A tile split across CTAs is
//    finished by whichever contributing warp arrives last (atomic ticket, no
//    waiting), summing the partial tiles in k order: deterministic.
//  * One producer warp moves each unit into a 4-deep shared-memory ring with
//    TMA: a 128x128-byte 2-D tensor copy of the packed nibbles (128-byte
//    swizzle, so the consumers' 16-byte reads are bank-conflict free), a
//    128x16-byte copy of the scales, and a 4 KB bulk copy of the unit's
//    fp16 activations; one mbarrier per slot counts the bytes in.
//  * Four consumer warps each own 32 rows.  They unpack nibbles to fp16 in
//    registers (hardware e2m1x2 -> f16x2 conversion; exact), apply the E4M3
//    block scale with an exact f16x2 multiply (nvfp4) or keep the integer
//    (q - 8) and apply the fp16 scale in fp32 after the block's two MMAs
//    (Q4_0, exact products), and multiply on the tensor cores with
//    mma.m16n8k16 (weights as the 16-row operand, the <= 8 verify rows as
//    the n = 8 operand, fp32 accumulation).
//  * Activations are pre-converted once per call to fp16 times a per-row
//    power of two (so any bf16 magnitude fits fp16 without overflow); the
//    epilogue multiplies the inverse back exactly.
//  * Optional fused argmax over n for every verify row (ties to the lowest
//    index, NaN never wins) via 64-bit atomic max on (ordered value, ~index).
// Every wait is bounded (global timer); a wait that runs out sets a status
// bit, the producer drains its in-flight copies, and the kernel returns.
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "vw4_internal.cuh"

namespace vw4 {

constexpr uint32_t kStatusTimeout = 0x4u;
constexpr uint32_t kStatusBadExpert = 0x2u;

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

GemmWorkspace gemm_workspace_layout(void* base, int n_seg_max, int N, int K, int grid,
                                    int pair_rows) {
    GemmWorkspace w{};
    char* b = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void* {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return b ? static_cast<void*>(b + o) : nullptr;
    };
    const int T = K / kStageK;
    const int n_tiles = (N + kTileRows - 1) / kTileRows;
    w.seg = static_cast<SegTable*>(take(sizeof(SegTable)));
    w.inv_scale = static_cast<float*>(take(sizeof(float) * kMaxSeg * kMaxRows));
    w.act16 = static_cast<__half*>(take((size_t)n_seg_max * T * kMaxRows * kStageK * 2));
    w.partials = static_cast<float*>(take((size_t)2 * grid * kPartialFloats * sizeof(float)));
    w.tile_cnt = static_cast<uint32_t*>(take((size_t)n_seg_max * n_tiles * 4));
    w.am_key = static_cast<unsigned long long*>(take(sizeof(unsigned long long) * kMaxRows));
    w.am_cnt = static_cast<uint32_t*>(take(4));
    w.pair_out = pair_rows ? static_cast<float*>(take((size_t)pair_rows * N * sizeof(float)))
                           : nullptr;
    w.bytes = off;
    return w;
}

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float pow2f(int n) {  // exact 2^n, n in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(n + 127) << 23);
}

// Position, in halves, of element e (0..255) of verify row r inside one
// stage's [8][256] fp16 block.  The order puts each consumer lane's B
// operand of consecutive MMAs in one 16-byte chunk, and the XOR keeps the
// eight lanes of a quarter-warp on distinct bank groups.
__device__ __forceinline__ int act_pos(int fmt, int r, int e) {
    if (fmt == 1) {  // nvfp4: lane c covers elements [64c, 64c+64), 8 chunks
        const int c = e >> 6, i = (e >> 3) & 7, j = e & 7;
        const int sw = ((r & 1) << 2) | c;
        return r * 256 + c * 64 + ((i ^ sw) << 3) + j;
    } else {  // Q4_0: chunk (block, lane) = elements 4c+{0,2,1,3} and 16+4c+{0,2,1,3}
        const int beta = e >> 5, ee = e & 31, half = ee >> 4, e2 = ee & 15, c = e2 >> 2,
                  q = e2 & 3;
        const int perm = (q == 0) ? 0 : (q == 1) ? 2 : (q == 2) ? 1 : 3;
        const int chunk = ((beta << 2) | c) ^ ((r & 1) << 2);
        return r * 256 + chunk * 8 + half * 4 + perm;
    }
}

// ------------------------------------------------------------- prep kernel
// One block per (segment, verify row).  Dense mode (dense_M > 0) writes the
// one-segment table itself; MoE mode reads the table written by the router.
// Also resets the tickets of this call.
__global__ void __launch_bounds__(256) prep_act_kernel(
    const uint16_t* __restrict__ A, int lda, int K, int fmt, int dense_M, int rows_are_pairs,
    int topk, SegTable* seg, float* inv_scale, __half* act16, uint32_t* tile_cnt, int n_cnt,
    unsigned long long* am_key, uint32_t* am_cnt) {
    const int s = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const int T = K / kStageK;
    if (s == 0 && r == 0) {
        for (int i = tid; i < n_cnt; i += blockDim.x) tile_cnt[i] = 0u;
        if (tid < kMaxRows) am_key[tid] = 0ull;
        if (tid == 0) *am_cnt = 0u;
    }
    int n_seg, count, src_row = 0;
    if (dense_M > 0) {
        n_seg = 1;
        count = dense_M;
        if (s == 0 && r == 0 && tid == 0) {
            seg->n_seg = 1;
            seg->expert[0] = 0;
            seg->count[0] = dense_M;
            for (int j = 0; j < kMaxRows; ++j) seg->dest[0][j] = j;
        }
        src_row = r;
    } else {
        n_seg = seg->n_seg;
        if (s >= n_seg) return;
        count = seg->count[s];
        if (r < count) {
            const int pr = seg->dest[s][r];
            src_row = rows_are_pairs ? pr : pr / topk;
        }
    }
    if (s >= n_seg) return;
    __half* dst = act16 + (size_t)s * T * (kMaxRows * kStageK);
    if (r >= count) {
        for (int k = tid; k < K; k += blockDim.x)
            dst[(size_t)(k >> 8) * (kMaxRows * kStageK) + act_pos(fmt, r, k & 255)] =
                __float2half_rn(0.0f);
        if (tid == 0) inv_scale[s * kMaxRows + r] = 0.0f;
        return;
    }
    const uint16_t* a = A + (size_t)src_row * lda;
    float amax = 0.0f;
    int bad = 0;
    for (int k = tid; k < K; k += blockDim.x) {
        const float v = fabsf(bf16_to_f32(a[k]));
        if (!(v <= 3.4e38f)) bad = 1;
        else amax = fmaxf(amax, v);
    }
    __shared__ float s_max[8];
    __shared__ int s_bad[8];
    for (int o = 16; o > 0; o >>= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if ((tid & 31) == 0) {
        s_max[tid >> 5] = amax;
        s_bad[tid >> 5] = bad;
    }
    __syncthreads();
    amax = 0.0f;
    bad = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        amax = fmaxf(amax, s_max[w]);
        bad |= s_bad[w];
    }
    int n = 0;
    if (!bad && amax > 0.0f) {
        int e;
        frexpf(amax, &e);  // amax in [2^(e-1), 2^e)
        n = 15 - e;        // scaled max in [2^14, 2^15)
        n = n < -125 ? -125 : (n > 125 ? 125 : n);
    }
    const float sc = pow2f(n);
    for (int k = tid; k < K; k += blockDim.x)
        dst[(size_t)(k >> 8) * (kMaxRows * kStageK) + act_pos(fmt, r, k & 255)] =
            __float2half_rn(bf16_to_f32(a[k]) * sc);
    if (tid == 0) inv_scale[s * kMaxRows + r] = pow2f(-n);
}

// ------------------------------------------------------------ MoE router
// Stable counting sort of the routed pairs by expert into segments of at
// most 8 rows (one thread; at most 64 pairs).  Pairs with an invalid expert
// are dropped, flagged, and their direct output rows zeroed.
__global__ void route_kernel(const int32_t* __restrict__ ids, int P, int E, SegTable* seg,
                             uint32_t* status, float* out_zero, int ldo, int N) {
    __shared__ int s_ids[kMaxSeg];
    __shared__ int s_bad[kMaxSeg];
    __shared__ int s_nbad;
    const int tid = threadIdx.x;
    if (tid < P) s_ids[tid] = ids[tid];
    __syncthreads();
    if (tid == 0) {
        int order[kMaxSeg];
        int cnt = 0, nbad = 0;
        for (int p = 0; p < P; ++p) {
            const int e = s_ids[p];
            if (e < 0 || e >= E) {
                s_bad[nbad++] = p;
                continue;
            }
            int j = cnt++;
            while (j > 0 && s_ids[order[j - 1]] > e) {  // stable insertion
                order[j] = order[j - 1];
                --j;
            }
            order[j] = p;
        }
        int ns = 0;
        for (int i = 0; i < cnt;) {
            const int e = s_ids[order[i]];
            int c = 0;
            while (i < cnt && s_ids[order[i]] == e && c < kMaxRows) {
                seg->dest[ns][c++] = order[i++];
            }
            for (int j = c; j < kMaxRows; ++j) seg->dest[ns][j] = 0;
            seg->expert[ns] = e;
            seg->count[ns] = c;
            ++ns;
        }
        seg->n_seg = ns;
        s_nbad = nbad;
        if (nbad) atomicOr(status, kStatusBadExpert);
    }
    __syncthreads();
    if (out_zero != nullptr) {
        for (int b = 0; b < s_nbad; ++b) {
            float* row = out_zero + (size_t)s_bad[b] * ldo;
            for (int n = tid; n < N; n += blockDim.x) row[n] = 0.0f;
        }
    }
}

// ------------------------------------------------------------ GEMM pieces
__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    return *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ uint32_t lds32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

// four FP4 E2M1 pairs (the four bytes of w) -> four f16x2, low nibble -> low half
__device__ __forceinline__ void cvt_e2m1x8(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                           uint32_t& h3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

// four E4M3 bytes -> (bytes 0,1) and (bytes 2,3) as f16x2
__device__ __forceinline__ void cvt_e4m3x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Q4_0 nibble pairs -> f16x2 of (q - 8): 0x6400|q is 1024 + q exactly.
__device__ __forceinline__ uint32_t q4pair(uint32_t x) {
    return hsub2((x & 0x000F000Fu) | 0x64006400u, 0x64086408u);
}

// One 256-wide k slice of the warp's 32 rows, nvfp4.
//   lane (g, c): rows g and g+8 of each 16-row half; its k range is
//   [64c, 64c+64) of the slice, i.e. 16-byte chunks 2c and 2c+1 of a row.
//   MMA j takes elements 64c+4j .. 64c+4j+3 from every lane: the A operand
//   pairs (k 2c,2c+1) and (k 2c+8,2c+9) of the mma fragment are mapped to
//   these four consecutive elements, and the B operand uses the same map, so
//   the sum over the slice is unchanged.
__device__ __forceinline__ void stage_nvfp4(const uint8_t* __restrict__ W,
                                            const uint8_t* __restrict__ S,
                                            const uint8_t* __restrict__ Ab, int warp, int lane,
                                            float (&acc)[2][4]) {
    const int g = lane >> 2, c = lane & 3;
    uint4 bf[8];
    const uint8_t* ab = Ab + g * 512 + c * 128;
    const int sw = ((g & 1) << 2) | c;
#pragma unroll
    for (int i = 0; i < 8; ++i) bf[i] = lds128(ab + ((i ^ sw) << 4));
#pragma unroll
    for (int t2 = 0; t2 < 2; ++t2) {
        const int r0 = warp * 32 + t2 * 16 + g;
        const uint8_t* w0 = W + r0 * 128;
        const uint8_t* w1 = w0 + 8 * 128;
        const int x0 = ((2 * c) ^ g) << 4, x1 = ((2 * c + 1) ^ g) << 4;  // 128-byte swizzle
        const uint4 p00 = lds128(w0 + x0), p01 = lds128(w0 + x1);
        const uint4 p10 = lds128(w1 + x0), p11 = lds128(w1 + x1);
        uint32_t sa0, sb0, sa1, sb1;
        cvt_e4m3x4(lds32(S + r0 * 16 + 4 * c), sa0, sb0);
        cvt_e4m3x4(lds32(S + (r0 + 8) * 16 + 4 * c), sa1, sb1);
        const uint32_t sc0[4] = {__byte_perm(sa0, sa0, 0x1010), __byte_perm(sa0, sa0, 0x3232),
                                 __byte_perm(sb0, sb0, 0x1010), __byte_perm(sb0, sb0, 0x3232)};
        const uint32_t sc1[4] = {__byte_perm(sa1, sa1, 0x1010), __byte_perm(sa1, sa1, 0x3232),
                                 __byte_perm(sb1, sb1, 0x1010), __byte_perm(sb1, sb1, 0x3232)};
        const uint32_t wr0[8] = {p00.x, p00.y, p00.z, p00.w, p01.x, p01.y, p01.z, p01.w};
        const uint32_t wr1[8] = {p10.x, p10.y, p10.z, p10.w, p11.x, p11.y, p11.z, p11.w};
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            uint32_t h0, h1, h2, h3, q0, q1, q2, q3;
            cvt_e2m1x8(wr0[wi], h0, h1, h2, h3);
            cvt_e2m1x8(wr1[wi], q0, q1, q2, q3);
            const uint32_t s0 = sc0[wi >> 1], s1 = sc1[wi >> 1];
            const uint32_t* b = reinterpret_cast<const uint32_t*>(&bf[wi]);
            mma16816(acc[t2], hmul2(h0, s0), hmul2(q0, s1), hmul2(h1, s0), hmul2(q1, s1), b[0],
                     b[1]);
            mma16816(acc[t2], hmul2(h2, s0), hmul2(q2, s1), hmul2(h3, s0), hmul2(q3, s1), b[2],
                     b[3]);
        }
    }
}

// One 256-wide k slice of the warp's 32 rows, Q4_0 (eight 32-element blocks).
//   For block beta, lane (g, c) reads bytes 4c..4c+3 of the block: low
//   nibbles are elements 4c..4c+3, high nibbles 4c+16..4c+19.  The two MMAs
//   of a block run on exact integers (q - 8) into a zeroed temporary, and the
//   block's fp16 scale is applied to the fp32 result.
__device__ __forceinline__ void stage_q4_0(const uint8_t* __restrict__ W,
                                           const uint8_t* __restrict__ S,
                                           const uint8_t* __restrict__ Ab, int warp, int lane,
                                           float (&acc)[2][4]) {
    const int g = lane >> 2, c = lane & 3;
    uint4 bf[8];
    const uint8_t* ab = Ab + g * 512;
#pragma unroll
    for (int beta = 0; beta < 8; ++beta)
        bf[beta] = lds128(ab + ((((beta << 2) | c) ^ ((g & 1) << 2)) << 4));
#pragma unroll
    for (int t2 = 0; t2 < 2; ++t2) {
        const int r0 = warp * 32 + t2 * 16 + g;
        const uint8_t* w0 = W + r0 * 128 + 4 * c;
        const uint8_t* w1 = w0 + 8 * 128;
        const uint4 d0 = lds128(S + r0 * 16), d1 = lds128(S + (r0 + 8) * 16);
        const uint32_t dw0[4] = {d0.x, d0.y, d0.z, d0.w};
        const uint32_t dw1[4] = {d1.x, d1.y, d1.z, d1.w};
#pragma unroll
        for (int beta = 0; beta < 8; ++beta) {
            const uint32_t x0 = lds32(w0 + ((beta ^ g) << 4));
            const uint32_t x1 = lds32(w1 + ((beta ^ g) << 4));
            const uint32_t* b = reinterpret_cast<const uint32_t*>(&bf[beta]);
            float t[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(t, q4pair(x0), q4pair(x1), q4pair(x0 >> 8), q4pair(x1 >> 8), b[0], b[1]);
            mma16816(t, q4pair(x0 >> 4), q4pair(x1 >> 4), q4pair(x0 >> 12), q4pair(x1 >> 12),
                     b[2], b[3]);
            const __half2 dh0 = *reinterpret_cast<const __half2*>(&dw0[beta >> 1]);
            const __half2 dh1 = *reinterpret_cast<const __half2*>(&dw1[beta >> 1]);
            const float e0 = (beta & 1) ? __high2float(dh0) : __low2float(dh0);
            const float e1 = (beta & 1) ? __high2float(dh1) : __low2float(dh1);
            acc[t2][0] = fmaf(e0, t[0], acc[t2][0]);
            acc[t2][1] = fmaf(e0, t[1], acc[t2][1]);
            acc[t2][2] = fmaf(e1, t[2], acc[t2][2]);
            acc[t2][3] = fmaf(e1, t[3], acc[t2][3]);
        }
    }
}

// Packed argmax key: larger key = larger value, then smaller index.  NaN is
// ordered as -inf and -0 as +0, matching the oracle's scan.
__device__ __forceinline__ unsigned long long am_key(float v, uint32_t idx) {
    if (v != v) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - idx);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a,
                                                     unsigned long long b) {
    return a > b ? a : b;
}

struct Range {
    unsigned long long U, G;
    __device__ __forceinline__ unsigned long long start(unsigned long long i) const {
        return i * U / G;
    }
    // the CTA whose range holds unit u
    __device__ __forceinline__ unsigned long long owner(unsigned long long u) const {
        return ((u + 1) * G + U - 1) / U - 1;
    }
};

// Called by the warp that completes the fused argmax bookkeeping.
__device__ void argmax_finish(const GemmParams& p, int lane) {
    __threadfence();
    if (lane < p.argmax_M) {
        const unsigned long long k = atomicAdd(&p.am_key[lane], 0ull);
        p.row_argmax[lane] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k));
    }
}

template <int FMT>
__global__ void __launch_bounds__(kGemmThreads, 2)
    gemm_w4_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                   const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmS);
    }
    __syncthreads();

    const int T = p.T, n_tiles = p.n_tiles;
    const int n_seg = p.seg->n_seg;
    // Effective grid: never more CTAs than units, so every active CTA owns at
    // least one unit (the contributor arithmetic of split tiles relies on it).
    const unsigned long long U = static_cast<unsigned long long>(n_seg) * n_tiles * T;
    const unsigned long long G = U < gridDim.x ? U : gridDim.x;
    if (blockIdx.x >= G) return;
    const Range R{U, G};
    const unsigned long long u_begin = R.start(blockIdx.x), u_end = R.start(blockIdx.x + 1);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_a = policy_evict_last();
        uint32_t it = 0;
        bool ok = true;
        for (unsigned long long u = u_begin; u < u_end; ++u, ++it) {
            const int s = it % kStages;
            if (it >= (uint32_t)kStages &&
                !mbar_wait_bounded(&empty[s], ((it / kStages) - 1) & 1, p.wait_ns, abort_flag)) {
                ok = false;
                break;
            }
            const unsigned long long tg = u / T;
            const int st = static_cast<int>(u % T);
            const int sg = static_cast<int>(tg / n_tiles), tile = static_cast<int>(tg % n_tiles);
            const int row0 = p.seg->expert[sg] * p.N + tile * kTileRows;
            uint8_t* slot = smem + s * kStageBytes;
            mbar_arrive_expect_tx(&full[s], kStageBytes);
            tma_load_2d(slot, &tmW, st * (kStageK / 2), row0, &full[s], pol_w);
            tma_load_2d(slot + kWBytes, &tmS, st * 16, row0, &full[s], pol_w);
            bulk_load(slot + kWBytes + kSBytes,
                      p.act16 + (static_cast<size_t>(sg) * T + st) * (kMaxRows * kStageK),
                      kABytes, &full[s], pol_a);
        }
        if (!ok) {
            atomicOr(p.status, kStatusTimeout);
            *abort_flag = 1;
        }
        // Drain: every issued copy must land before this CTA may exit.
        const uint64_t drain_ns = p.wait_ns > 2000000000ull ? p.wait_ns : 2000000000ull;
        for (uint32_t j = (it > (uint32_t)kStages ? it - kStages : 0u); j < it; ++j)
            mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1, drain_ns, nullptr);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    uint32_t it = 0;
    const unsigned long long my_first_tile = u_begin / T;
    for (unsigned long long u = u_begin; u < u_end;) {
        const unsigned long long tg = u / T;
        const int st0 = static_cast<int>(u % T);
        const unsigned long long left = u_end - u;
        const int st_end = (left < static_cast<unsigned long long>(T - st0))
                               ? st0 + static_cast<int>(left)
                               : T;
        float acc[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
        for (int st = st0; st < st_end; ++st, ++it) {
            const int s = it % kStages;
            if (!mbar_wait_bounded(&full[s], (it / kStages) & 1, p.wait_ns, abort_flag)) {
                if (lane == 0) atomicOr(p.status, kStatusTimeout);
                *abort_flag = 1;
                return;
            }
            const uint8_t* slot = smem + s * kStageBytes;
            if (FMT == 1)
                stage_nvfp4(slot, slot + kWBytes, slot + kWBytes + kSBytes, warp, lane, acc);
            else
                stage_q4_0(slot, slot + kWBytes, slot + kWBytes + kSBytes, warp, lane, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        u += static_cast<unsigned long long>(st_end - st0);

        // ------------------------------------------------------ epilogue
        const int sg = static_cast<int>(tg / n_tiles), tile = static_cast<int>(tg % n_tiles);
        const int count = p.seg->count[sg];
        const float sc0 = p.tensor_scale * p.inv_scale[sg * kMaxRows + 2 * c];
        const float sc1 = p.tensor_scale * p.inv_scale[sg * kMaxRows + 2 * c + 1];
        float v[2][4];
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
            v[t2][0] = acc[t2][0] * sc0;
            v[t2][1] = acc[t2][1] * sc1;
            v[t2][2] = acc[t2][2] * sc0;
            v[t2][3] = acc[t2][3] * sc1;
        }
        const int n0 = tile * kTileRows;
        const bool whole = (st0 == 0 && st_end == T);
        if (whole) {
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tok = 2 * c + (q & 1);
                    const int n = n0 + warp * 32 + t2 * 16 + g + ((q & 2) ? 8 : 0);
                    if (tok < count && n < p.N)
                        p.out[static_cast<size_t>(p.seg->dest[sg][tok]) * p.ldo + n] = v[t2][q];
                }
            if (p.argmax_M > 0) {
                unsigned long long k0 = 0ull, k1 = 0ull;  // tokens 2c, 2c+1
#pragma unroll
                for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int n = n0 + warp * 32 + t2 * 16 + g + ((q & 2) ? 8 : 0);
                        if (n < p.N) {
                            const unsigned long long k = am_key(v[t2][q], static_cast<uint32_t>(n));
                            if (q & 1) k1 = umax64(k1, k);
                            else k0 = umax64(k0, k);
                        }
                    }
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    k0 = umax64(k0, __shfl_xor_sync(0xffffffffu, k0, o));
                    k1 = umax64(k1, __shfl_xor_sync(0xffffffffu, k1, o));
                }
                if (g == 0) {
                    if (2 * c < p.argmax_M && k0) atomicMax(&p.am_key[2 * c], k0);
                    if (2 * c + 1 < p.argmax_M && k1) atomicMax(&p.am_key[2 * c + 1], k1);
                }
                __threadfence();
                __syncwarp();
                uint32_t old = 0;
                if (lane == 0) old = atomicAdd(p.am_cnt, 1u);
                old = __shfl_sync(0xffffffffu, old, 0);
                if (old + 1 == 4u * static_cast<uint32_t>(n_tiles)) argmax_finish(p, lane);
            }
            continue;
        }
        // partial tile: publish my slice, then the last contributing warp sums
        const unsigned long long tile_u0 = tg * static_cast<unsigned long long>(T);
        const unsigned long long i_lo = R.owner(tile_u0), i_hi = R.owner(tile_u0 + T - 1);
        const uint32_t n_contrib = static_cast<uint32_t>(i_hi - i_lo + 1);
        const unsigned long long my_slot =
            2ull * blockIdx.x + ((my_first_tile == tg) ? 0ull : 1ull);
        float* part = p.partials + my_slot * kPartialFloats;
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int tok = 2 * c + (q & 1);
                const int r = warp * 32 + t2 * 16 + g + ((q & 2) ? 8 : 0);
                __stcg(&part[tok * kTileRows + r], v[t2][q]);
            }
        __threadfence();
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atomicAdd(&p.tile_cnt[tg], 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + 1 != static_cast<uint32_t>(kConsumerWarps) * n_contrib) continue;
        __threadfence();
        // This warp sums the 8 x 128 values in contributor (= k) order.  Every
        // contributor after the first starts inside this tile, so its slot is
        // its "first tile" slot; only the first may end in it instead.
        const unsigned long long slot_lo =
            2ull * i_lo + ((R.start(i_lo) / T == tg) ? 0ull : 1ull);
        float4 sum[kMaxRows];
#pragma unroll
        for (int tok = 0; tok < kMaxRows; ++tok) sum[tok] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (unsigned long long i = i_lo; i <= i_hi; ++i) {
            const unsigned long long slot = (i == i_lo) ? slot_lo : 2ull * i;
            const float4* src =
                reinterpret_cast<const float4*>(p.partials + slot * kPartialFloats) + lane;
            float4 x[kMaxRows];
#pragma unroll
            for (int tok = 0; tok < kMaxRows; ++tok) x[tok] = __ldcg(src + tok * (kTileRows / 4));
#pragma unroll
            for (int tok = 0; tok < kMaxRows; ++tok) {
                sum[tok].x += x[tok].x;
                sum[tok].y += x[tok].y;
                sum[tok].z += x[tok].z;
                sum[tok].w += x[tok].w;
            }
        }
        unsigned long long kbest[kMaxRows];
#pragma unroll
        for (int tok = 0; tok < kMaxRows; ++tok) {
            kbest[tok] = 0ull;
            if (tok >= count) continue;
            const float sv[4] = {sum[tok].x, sum[tok].y, sum[tok].z, sum[tok].w};
            float* orow = p.out + static_cast<size_t>(p.seg->dest[sg][tok]) * p.ldo;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + 4 * lane + j;
                if (n < p.N) {
                    orow[n] = sv[j];
                    kbest[tok] = umax64(kbest[tok], am_key(sv[j], static_cast<uint32_t>(n)));
                }
            }
        }
        if (p.argmax_M > 0) {
#pragma unroll
            for (int tok = 0; tok < kMaxRows; ++tok) {
                unsigned long long k = kbest[tok];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) k = umax64(k, __shfl_xor_sync(0xffffffffu, k, o));
                if (lane == 0 && tok < p.argmax_M && k) atomicMax(&p.am_key[tok], k);
            }
            __threadfence();
            __syncwarp();
            uint32_t o2 = 0;
            if (lane == 0) o2 = atomicAdd(p.am_cnt, static_cast<uint32_t>(kConsumerWarps));
            o2 = __shfl_sync(0xffffffffu, o2, 0);
            if (o2 + kConsumerWarps == 4u * static_cast<uint32_t>(n_tiles)) argmax_finish(p, lane);
        }
    }
}

// ------------------------------------------------------------ MoE combine
__global__ void combine_kernel(const float* __restrict__ pair_out, const float* __restrict__ gates,
                               const int32_t* __restrict__ ids, int E, int M, int topk, int N,
                               float* __restrict__ out, int ldo) {
    const int m = blockIdx.y;
    for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
        float s = 0.0f;
        for (int j = 0; j < topk; ++j) {
            const int e = ids[m * topk + j];
            if (e < 0 || e >= E) continue;
            s = fmaf(gates[m * topk + j], pair_out[static_cast<size_t>(m * topk + j) * N + n], s);
        }
        out[static_cast<size_t>(m) * ldo + n] = s;
    }
}

// --------------------------------------------------- Q4_0 18-byte records
__global__ void q4_0_split_kernel(const uint8_t* __restrict__ blocks, int N, int K,
                                  uint8_t* __restrict__ q, __half* __restrict__ d) {
    const long long nb = static_cast<long long>(N) * (K / 32);
    for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nb;
         b += static_cast<long long>(gridDim.x) * blockDim.x) {
        const uint8_t* src = blocks + b * 18;
        const uint16_t dbits = static_cast<uint16_t>(src[0] | (src[1] << 8));
        d[b] = __ushort_as_half(dbits);
        uint8_t* dst = q + b * 16;
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[j] = src[2 + j];
    }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_prep_act(const uint16_t* A, int lda, int K, int fmt, int dense_M,
                            int rows_are_pairs, int topk, int n_seg_grid, const GemmWorkspace& ws,
                            int n_counters, cudaStream_t s) {
    dim3 grid(n_seg_grid, kMaxRows);
    prep_act_kernel<<<grid, 256, 0, s>>>(A, lda, K, fmt, dense_M, rows_are_pairs, topk, ws.seg,
                                         ws.inv_scale, ws.act16, ws.tile_cnt, n_counters,
                                         ws.am_key, ws.am_cnt);
    return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_gemm_t(const CUtensorMap& tmW, const CUtensorMap& tmS,
                                 const GemmParams& p, int grid, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(gemm_w4_kernel<FMT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    gemm_w4_kernel<FMT><<<grid, kGemmThreads, kGemmSmem, s>>>(tmW, tmS, p);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int fmt, const CUtensorMap& tmW, const CUtensorMap& tmS,
                        const GemmParams& p, int grid, cudaStream_t s) {
    return fmt == 1 ? launch_gemm_t<1>(tmW, tmS, p, grid, s) : launch_gemm_t<2>(tmW, tmS, p, grid, s);
}

int gemm_blocks_per_sm(int fmt) {
    int n = 0;
    if (fmt == 1) {
        cudaFuncSetAttribute(gemm_w4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemmSmem);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemm_w4_kernel<1>, kGemmThreads, kGemmSmem);
    } else {
        cudaFuncSetAttribute(gemm_w4_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemmSmem);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemm_w4_kernel<2>, kGemmThreads, kGemmSmem);
    }
    return n > 0 ? n : 1;
}

cudaError_t launch_combine(const float* pair_out, const float* gates, const int32_t* ids,
                               int E, int M, int topk, int N, float* out, int ldo, cudaStream_t s) {
    dim3 grid((N + 255) / 256, M);
    combine_kernel<<<grid, 256, 0, s>>>(pair_out, gates, ids, E, M, topk, N, out, ldo);
    return cudaGetLastError();
}

cudaError_t launch_route(const int32_t* expert_ids, int M, int topk, int E,
                              const GemmWorkspace& ws, uint32_t* status, float* out_zero, int ldo,
                              int N, cudaStream_t s) {
    route_kernel<<<1, 64, 0, s>>>(expert_ids, M * topk, E, ws.seg, status, out_zero, ldo, N);
    return cudaGetLastError();
}

cudaError_t launch_q4_0_split(const uint8_t* blocks, int N, int K, uint8_t* q, __half* d,
                              cudaStream_t s) {
    const long long nb = static_cast<long long>(N) * (K / 32);
    int grid = static_cast<int>((nb + 255) / 256);
    if (grid > 65535) grid = 65535;
    if (grid < 1) grid = 1;
    q4_0_split_kernel<<<grid, 256, 0, s>>>(blocks, N, K, q, d);
    return cudaGetLastError();
}

}  // namespace vw4
