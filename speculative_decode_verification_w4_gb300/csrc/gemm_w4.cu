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
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "vw4_internal.cuh"

namespace cg = cooperative_groups;

namespace vw4 {

constexpr uint32_t kStatusTimeout = 0x4u;
constexpr uint32_t kStatusBadDraft = 0x1u;
constexpr uint32_t kStatusBadExpert = 0x2u;

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

GemmWorkspace gemm_workspace_layout(void* base, int n_seg_max, int N, int K, int grid,
                                    int pair_rows, int nr, int pad_rows) {
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
    w.act = static_cast<uint8_t*>(take((size_t)n_seg_max * T * act_stride(nr)));
    w.partials = static_cast<float*>(take((size_t)2 * grid * nr * kTileRows * sizeof(float)));
    w.tile_cnt = static_cast<uint32_t*>(take((size_t)n_seg_max * n_tiles * kConsumerWarps * 4));
    w.am_key = static_cast<unsigned long long*>(take(sizeof(unsigned long long) * kMaxVerifyRows));
    w.am_cnt = static_cast<uint32_t*>(take(4));
    w.pair_out = pair_rows ? static_cast<float*>(take((size_t)pair_rows * N * sizeof(float)))
                           : nullptr;
    w.wpad = pad_rows ? static_cast<uint8_t*>(take((size_t)pad_rows * (K / 2))) : nullptr;
    w.spad = pad_rows ? static_cast<uint8_t*>(take((size_t)pad_rows * (K / 16))) : nullptr;
    w.bytes = off;
    return w;
}

// ------------------------------------------------------------ padded weights
// A matrix whose K is a multiple of the block but not of 256 (row pitches of
// K/2 and K/16 bytes that TMA cannot address) is copied into rows of Kp/2
// nibble bytes and Kp/16 scale bytes (Kp = K rounded up to 256), zero past K:
// zero nibbles and zero scales are weights of exactly 0 in both formats.
// Both formats keep K/16 scale bytes per row (nvfp4: one E4M3 per 16; Q4_0:
// one fp16 per 32).
__global__ void pad_weights_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sc,
                                   int N, int K, int Kp, uint8_t* __restrict__ qo,
                                   uint8_t* __restrict__ so) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long t0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    // nibbles in 8-byte units (K / 2 is a multiple of 8, rows start 8-byte aligned)
    const int in8 = K / 16, out8 = Kp / 16;
    const unsigned long long* q8 = reinterpret_cast<const unsigned long long*>(q);
    unsigned long long* qo8 = reinterpret_cast<unsigned long long*>(qo);
    for (long long i = t0; i < static_cast<long long>(N) * out8; i += stride) {
        const long long row = i / out8;
        const int j = static_cast<int>(i % out8);
        qo8[i] = j < in8 ? q8[row * in8 + j] : 0ull;
    }
    // scales, byte by byte (K / 16 bytes a row, any alignment)
    const int ins = K / 16, outs = Kp / 16;
    for (long long i = t0; i < static_cast<long long>(N) * outs; i += stride) {
        const long long row = i / outs;
        const int j = static_cast<int>(i % outs);
        so[i] = j < ins ? sc[row * ins + j] : static_cast<uint8_t>(0);
    }
}

cudaError_t launch_pad_weights(const void* q, const void* sc, int N, int K, int Kp, uint8_t* qo,
                               uint8_t* so, cudaStream_t s) {
    pad_weights_kernel<<<1216, 256, 0, s>>>(static_cast<const uint8_t*>(q),
                                             static_cast<const uint8_t*>(sc), N, K, Kp, qo, so);
    return cudaGetLastError();
}

// ------------------------------------------------------------ small helpers
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float pow2f(int n) {  // exact 2^n, n in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(n + 127) << 23);
}

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- prep kernel
// One warp per (segment, 256-wide k stage, verify row); each lane owns one
// 16-byte chunk of the stage's fp16 block.  The row's values in the stage are
// multiplied by 2^s so that their max lies in [2^14, 2^15) (exact; any bf16
// magnitude then fits fp16), and 2^-s is stored after the block for the
// GEMM's per-stage rescale.  Dense mode (dense_M > 0) writes the one-segment
// table itself; MoE mode reads the table written by the router.  Block 0 also
// resets the tickets of this call.
__device__ __forceinline__ void load8_bf16(const uint16_t* a, bool vec, float (&x)[8]) {
    if (vec) {
        const uint4 u = *reinterpret_cast<const uint4*>(a);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            x[2 * j] = __uint_as_float(w[j] << 16);
            x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = bf16_to_f32(a[j]);
    }
}

__device__ __forceinline__ void load4_bf16(const uint16_t* a, bool vec, float* x) {
    if (vec) {
        const uint2 u = *reinterpret_cast<const uint2*>(a);
        x[0] = __uint_as_float(u.x << 16);
        x[1] = __uint_as_float(u.x & 0xFFFF0000u);
        x[2] = __uint_as_float(u.y << 16);
        x[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = bf16_to_f32(a[j]);
    }
}

// ------------------------------------------------------------ MoE router
// Stable counting sort of the routed pairs by expert into segments of at
// most 8 rows, one thread per pair (at most 64): a pair's segment is the
// number of segments of the smaller expert ids plus its rank among the pairs
// of its own expert, divided by 8.  Segments come out ordered by expert id,
// and inside an expert by pair index.  Computed by threads 0 .. P-1 of a
// block into a table in its shared memory; pairs with an invalid expert id
// join no segment and are listed in bad[0 .. nbad).
struct RouteScratch {
    int ids[kMaxSeg];
    int cnt[kMaxSeg];    // pairs of this pair's expert
    int first[kMaxSeg];  // this pair is its expert's first
    int bad[kMaxSeg];
    int nbad, nseg;
};

__device__ void route_pairs(const int32_t* __restrict__ ids, int P, int E, SegTable& seg,
                            RouteScratch& rs) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        rs.nbad = 0;
        rs.nseg = 0;
    }
    if (tid < P) rs.ids[tid] = ids[tid];
    __syncthreads();
    int e = -1, rank = 0, valid = 0;
    if (tid < P) {
        e = rs.ids[tid];
        valid = (e >= 0 && e < E) ? 1 : 0;
        int cnt = 0;
        for (int q = 0; q < P; ++q) {
            const int same = rs.ids[q] == e ? 1 : 0;
            cnt += same;
            rank += (same && q < tid) ? 1 : 0;
        }
        rs.cnt[tid] = cnt;
        rs.first[tid] = (valid && rank == 0) ? 1 : 0;
        if (!valid) rs.bad[atomicAdd(&rs.nbad, 1)] = tid;
    }
    __syncthreads();
    if (tid < P && valid) {
        int base = 0;  // segments of the smaller expert ids
        for (int q = 0; q < P; ++q)
            if (rs.first[q] && rs.ids[q] < e) base += (rs.cnt[q] + kMaxRows - 1) / kMaxRows;
        const int sgi = base + rank / kMaxRows, slot = rank % kMaxRows;
        seg.dest[sgi][slot] = tid;
        if (slot == 0) {
            const int c = min(kMaxRows, rs.cnt[tid] - rank);
            seg.expert[sgi] = e;
            seg.count[sgi] = c;
            for (int j = c; j < kMaxRows; ++j) seg.dest[sgi][j] = 0;
        }
        if (rs.first[tid]) atomicAdd(&rs.nseg, (rs.cnt[tid] + kMaxRows - 1) / kMaxRows);
    }
    __syncthreads();
    if (tid == 0) seg.n_seg = rs.nseg;
    __syncthreads();
}

// MoE calls (dense_M == 0) route the pairs here too: every block computes the
// (tiny) routing into its own shared memory and block 0 publishes it for the
// GEMM, marks invalid expert ids in the status word and zeroes their output
// rows (out_zero, when the pair rows are the output).
// One warp per verify row: 256 threads (8 rows) or 512 (16 rows, dense only).
__global__ void __launch_bounds__(512) prep_act_kernel(
    const uint16_t* __restrict__ A, int lda, int vec_ok, int K, int K_true, int fmt, int nr,
    int dense_M,
    int rows_are_pairs, int topk, SegTable* seg, uint8_t* act, uint32_t* tile_cnt, int n_cnt,
    unsigned long long* am_key, uint32_t* am_cnt, const int32_t* __restrict__ ids, int P, int E,
    uint32_t* status, float* out_zero, int ldo, int N, int stage_ctas) {
    __shared__ SegTable lt;
    __shared__ RouteScratch rs;
    // The GEMM may start streaming weights now; it waits for this grid before
    // touching the activations or the tickets.  This grid itself may have
    // been launched while its predecessor (the previous GEMM, or the router)
    // still runs: nothing is read or written before that grid has finished.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // CTA (sgi, st0) converts stages st0, st0 + stage_ctas, ... of segment
    // sgi: one CTA per stage for dense calls; for MoE calls a few per
    // segment, so that each CTA's routing (below) serves several stages
    const int T = K / kStageK;
    const int sgi = blockIdx.x / stage_ctas, st0 = blockIdx.x % stage_ctas;
    const int r = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) tile_cnt[i] = 0u;
        if (threadIdx.x < kMaxVerifyRows) am_key[threadIdx.x] = 0ull;
        if (threadIdx.x == 0) *am_cnt = 0u;
    }
    int count, src_row = 0;
    if (dense_M > 0) {
        count = dense_M;
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            seg->n_seg = 1;
            seg->expert[0] = 0;
            seg->count[0] = dense_M;
            for (int j = 0; j < kMaxRows; ++j) seg->dest[0][j] = j;
        }
        src_row = r;
    } else {
        route_pairs(ids, P, E, lt, rs);
        if (blockIdx.x == 0) {
            for (int i = threadIdx.x; i < static_cast<int>(sizeof(SegTable) / 4); i += blockDim.x)
                reinterpret_cast<int*>(seg)[i] = reinterpret_cast<const int*>(&lt)[i];
            if (threadIdx.x == 0 && rs.nbad) atomicOr(status, kStatusBadExpert);
            if (out_zero != nullptr)
                for (int bq = 0; bq < rs.nbad; ++bq) {
                    float* row = out_zero + static_cast<size_t>(rs.bad[bq]) * ldo;
                    for (int n = threadIdx.x; n < N; n += blockDim.x) row[n] = 0.0f;
                }
        }
        if (sgi >= lt.n_seg) return;
        count = lt.count[sgi];
        if (r < count) {
            const int pr = lt.dest[sgi][r];
            if (check(pr >= 0 && pr < P, status)) src_row = rows_are_pairs ? pr : pr / topk;
            else count = r;  // this row and the ones after it stay zero
        }
    }
    for (int st = st0; st < T; st += stage_ctas) {
        uint8_t* blk = act + (static_cast<size_t>(sgi) * T + st) * act_stride(nr);
        __half* dst = reinterpret_cast<__half*>(blk);
        float* inv = reinterpret_cast<float*>(blk + act_bytes(nr));
        // Where this lane's 16-byte chunk goes in the stage's [nr][256] block (16
        // rows: two [8][256] halves, one per mma n-tile, laid out alike).  The
        // order puts a consumer lane's B operands of consecutive MMAs in one chunk
        // and the XOR keeps a quarter-warp's reads on distinct bank groups.
        //  nvfp4: lane holds elements 8*lane .. 8*lane+7 (consumer lane c = lane/8
        //         covers [64c, 64c+64) of the stage);
        //  Q4_0:  lane = 4*beta + c holds elements 4c+{0,2,1,3} and 16+4c+{0,2,1,3}
        //         of 32-element block beta.
        int pos;
        if (fmt == 1) {
            const int c = lane >> 3, i = lane & 7;
            pos = r * 256 + c * 64 + ((i ^ (((r & 1) << 2) | c)) << 3);
        } else {
            pos = r * 256 + ((lane ^ ((r & 1) << 2)) << 3);
        }
        if (r >= count) {
            *reinterpret_cast<uint4*>(dst + pos) = make_uint4(0u, 0u, 0u, 0u);
            if (lane == 0) inv[r] = 0.0f;
            continue;
        }
        const uint16_t* a = A + static_cast<size_t>(src_row) * lda + st * kStageK;
        float x[8];
        // past K_true (a K padded to whole stages) the activations are zero; a
        // lane's 8 (nvfp4) or 32-block (Q4_0) elements lie wholly on one side
        const int k_lane = st * kStageK + (fmt == 1 ? 8 * lane : 32 * (lane >> 2));
        if (k_lane >= K_true) {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = 0.0f;
        } else if (fmt == 1) {
            load8_bf16(a + 8 * lane, vec_ok != 0, x);
        } else {
            const int beta = lane >> 2, c = lane & 3;
            float lo4[4], hi4[4];
            load4_bf16(a + 32 * beta + 4 * c, vec_ok != 0, lo4);
            load4_bf16(a + 32 * beta + 16 + 4 * c, vec_ok != 0, hi4);
            x[0] = lo4[0]; x[1] = lo4[2]; x[2] = lo4[1]; x[3] = lo4[3];
            x[4] = hi4[0]; x[5] = hi4[2]; x[6] = hi4[1]; x[7] = hi4[3];
        }
        float amax = 0.0f;
        int bad = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float v = fabsf(x[j]);
            if (!(v <= 3.4e38f)) bad = 1;
            else amax = fmaxf(amax, v);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            bad |= __shfl_xor_sync(0xffffffffu, bad, o);
        }
        int n = 0;
        if (!bad && amax > 0.0f) {
            int ex;
            frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
            n = 15 - ex;        // scaled max in [2^14, 2^15)
            n = n < -125 ? -125 : (n > 125 ? 125 : n);
        }
        const float sc = pow2f(n);
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 v = __floats2half2_rn(x[2 * j] * sc, x[2 * j + 1] * sc);
            h[j] = *reinterpret_cast<const uint32_t*>(&v);
        }
        *reinterpret_cast<uint4*>(dst + pos) = make_uint4(h[0], h[1], h[2], h[3]);
        if (lane == 0) inv[r] = pow2f(-n);
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

__device__ __forceinline__ __half2 as_half2(uint32_t u) {
    __half2 h;
    memcpy(&h, &u, 4);
    return h;
}
__device__ __forceinline__ uint32_t as_u32(__half2 h) {
    uint32_t u;
    memcpy(&u, &h, 4);
    return u;
}
// a * s, s one block scale in both halves.  Written as an f16x2 multiply by
// a half broadcast (not a byte-permuted register) so that the broadcast
// becomes the multiply's operand selection: 16 fewer instructions a warp and
// stage, and 1-3 % off the call time.
__device__ __forceinline__ uint32_t hmul2_bcast(uint32_t a, __half2 s) {
    return as_u32(__hmul2(as_half2(a), s));
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

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Q4_0 nibble pairs -> f16x2 of (q - 8).  Nibbles at bits 0..3 and 16..19:
// 0x6400 | q is 1024 + q exactly, minus 1032.  Nibbles at bits 4..7 and
// 20..23 (no shift needed): 0x6400 | q << 4 is 1024 + 16 q exactly, and one
// fma with 1/16 and -72 gives q - 8 exactly.
__device__ __forceinline__ uint32_t q4pair(uint32_t x) {
    return hsub2((x & 0x000F000Fu) | 0x64006400u, 0x64086408u);
}
__device__ __forceinline__ uint32_t q4pair_hi(uint32_t x) {
    return hfma2((x & 0x00F000F0u) | 0x64006400u, 0x2C002C00u, 0xD480D480u);
}

// One 256-wide k slice of the warp's 32 rows, as two 16-row MMA blocks that
// share the activation fragments.  Each stage is split into a load phase,
// which copies everything the warp needs out of the ring slot into registers
// (after which the slot is released to the producer), and a compute phase
// that works on registers only.  Row block rb of warp w covers tile rows
// 32w + 16rb + [0, 16); lane (g, c) holds rows g and g+8 of the block.  The
// 128-byte swizzle XORs the 16-byte chunk index with the row mod 8, which is
// g for every row a lane touches.
//
// nvfp4 -- lane c's k range is [64c, 64c+64) of the slice, i.e. 16-byte
//   chunks 2c and 2c+1 of a row.  MMA j takes elements 64c+4j .. 64c+4j+3
//   from every lane: the A operand pairs (k 2c,2c+1) and (k 2c+8,2c+9) of the
//   mma fragment are mapped to these four consecutive elements, and the B
//   operand uses the same map, so the sum over the slice is unchanged.  Even
//   and odd MMAs accumulate into two independent chains.
struct ActRegs {
    uint4 bf[8];  // B operand: this lane's 64 activations
    float2 inv;   // 2^-s of verify rows 2c, 2c+1
};

struct WRegsNv {
    uint4 w00, w01, w10, w11;  // rows g and g+8: chunks 2c, 2c+1
    uint32_t s0, s1;           // four e4m3 block scales of rows g and g+8
};

// Ab: the n-tile's [8][256] activation block; Ai: its eight 2^-s factors.
__device__ __forceinline__ void load_act_nvfp4(const uint8_t* __restrict__ Ab,
                                               const uint8_t* __restrict__ Ai, int lane,
                                               ActRegs& a) {
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* ab = Ab + g * 512 + c * 128;
    const int sw = ((g & 1) << 2) | c;
#pragma unroll
    for (int i = 0; i < 8; ++i) a.bf[i] = lds128(ab + ((i ^ sw) << 4));
    a.inv = *reinterpret_cast<const float2*>(Ai + 8 * c);
}

// W: the stage's weight slot; Sr: this stage's 16 bytes inside the scale
// slot row of tile row r0 (rows are spitch bytes apart: the box width).
__device__ __forceinline__ void load_w_nvfp4(const uint8_t* __restrict__ W,
                                             const uint8_t* __restrict__ Sr, int spitch, int r0,
                                             int lane, WRegsNv& r) {
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* w0 = W + r0 * 128;
    const uint8_t* w1 = w0 + 8 * 128;
    const int x0 = ((2 * c) ^ g) << 4, x1 = ((2 * c + 1) ^ g) << 4;
    r.w00 = lds128(w0 + x0);
    r.w01 = lds128(w0 + x1);
    r.w10 = lds128(w1 + x0);
    r.w11 = lds128(w1 + x1);
    r.s0 = lds32(Sr + 4 * c);
    r.s1 = lds32(Sr + 8 * spitch + 4 * c);
}

// NT n-tiles (8 verify rows each) share every unpacked weight fragment.
// Accumulator chains per n-tile: two (even and odd MMAs) for one n-tile; one
// for two n-tiles, whose chains are already independent of each other.
template <int NT>
struct Chains {
    static constexpr int kN = NT == 1 ? 2 : 1;
};

template <int NT>
__device__ __forceinline__ void compute_nvfp4(const ActRegs (&a)[NT], const WRegsNv& r,
                                              float (&acc)[NT][Chains<NT>::kN][4]) {
    constexpr int C1 = Chains<NT>::kN - 1;
    uint32_t sa0, sb0, sa1, sb1;
    cvt_e4m3x4(r.s0, sa0, sb0);
    cvt_e4m3x4(r.s1, sa1, sb1);
    const __half2 A0 = as_half2(sa0), B0 = as_half2(sb0), A1 = as_half2(sa1), B1 = as_half2(sb1);
    const __half2 sc0[4] = {__low2half2(A0), __high2half2(A0), __low2half2(B0), __high2half2(B0)};
    const __half2 sc1[4] = {__low2half2(A1), __high2half2(A1), __low2half2(B1), __high2half2(B1)};
    const uint32_t wr0[8] = {r.w00.x, r.w00.y, r.w00.z, r.w00.w, r.w01.x, r.w01.y, r.w01.z, r.w01.w};
    const uint32_t wr1[8] = {r.w10.x, r.w10.y, r.w10.z, r.w10.w, r.w11.x, r.w11.y, r.w11.z, r.w11.w};
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        uint32_t h0, h1, h2, h3, q0, q1, q2, q3;
        cvt_e2m1x8(wr0[wi], h0, h1, h2, h3);
        cvt_e2m1x8(wr1[wi], q0, q1, q2, q3);
        const __half2 s0 = sc0[wi >> 1], s1 = sc1[wi >> 1];
        const uint32_t e0 = hmul2_bcast(h0, s0), e1 = hmul2_bcast(q0, s1),
                       e2 = hmul2_bcast(h1, s0), e3 = hmul2_bcast(q1, s1);
        const uint32_t o0 = hmul2_bcast(h2, s0), o1 = hmul2_bcast(q2, s1),
                       o2 = hmul2_bcast(h3, s0), o3 = hmul2_bcast(q3, s1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4& b = a[nt].bf[wi];
            mma16816(acc[nt][0], e0, e1, e2, e3, b.x, b.y);
            mma16816(acc[nt][C1], o0, o1, o2, o3, b.z, b.w);
        }
    }
}

// Q4_0 (eight 32-element blocks per slice) -- for block beta, lane (g, c)
//   reads bytes 4c..4c+3 of the block: low nibbles are elements 4c..4c+3,
//   high nibbles 4c+16..4c+19.  The two MMAs of a block run on exact integers
//   (q - 8) into a zeroed temporary, and the block's fp16 scale is applied to
//   the fp32 result.
struct WRegsQ4 {
    uint32_t x0[8], x1[8];  // rows g and g+8, bytes 4c..4c+3 of each block
    uint4 d0, d1;           // the eight fp16 scales of rows g and g+8
};

__device__ __forceinline__ void load_act_q4_0(const uint8_t* __restrict__ Ab,
                                              const uint8_t* __restrict__ Ai, int lane,
                                              ActRegs& a) {
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* ab = Ab + g * 512;
#pragma unroll
    for (int beta = 0; beta < 8; ++beta)
        a.bf[beta] = lds128(ab + ((((beta << 2) | c) ^ ((g & 1) << 2)) << 4));
    a.inv = *reinterpret_cast<const float2*>(Ai + 8 * c);
}

__device__ __forceinline__ void load_w_q4_0(const uint8_t* __restrict__ W,
                                            const uint8_t* __restrict__ Sr, int spitch, int r0,
                                            int lane, WRegsQ4& r) {
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* w0 = W + r0 * 128 + 4 * c;
    const uint8_t* w1 = w0 + 8 * 128;
#pragma unroll
    for (int beta = 0; beta < 8; ++beta) {
        r.x0[beta] = lds32(w0 + ((beta ^ g) << 4));
        r.x1[beta] = lds32(w1 + ((beta ^ g) << 4));
    }
    r.d0 = lds128(Sr);
    r.d1 = lds128(Sr + 8 * spitch);
}

template <int NT>
__device__ __forceinline__ void compute_q4_0(const ActRegs (&a)[NT], const WRegsQ4& r,
                                             float (&acc)[NT][Chains<NT>::kN][4]) {
    constexpr int C1 = Chains<NT>::kN - 1;
    const uint32_t dw0[4] = {r.d0.x, r.d0.y, r.d0.z, r.d0.w};
    const uint32_t dw1[4] = {r.d1.x, r.d1.y, r.d1.z, r.d1.w};
#pragma unroll
    for (int beta = 0; beta < 8; ++beta) {
        const uint32_t x0 = r.x0[beta], x1 = r.x1[beta];
        const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
        const uint32_t l0 = q4pair(x0), l1 = q4pair(x1), l2 = q4pair(y0), l3 = q4pair(y1);
        const uint32_t u0 = q4pair_hi(x0), u1 = q4pair_hi(x1), u2 = q4pair_hi(y0),
                       u3 = q4pair_hi(y1);
        const __half2 dh0 = *reinterpret_cast<const __half2*>(&dw0[beta >> 1]);
        const __half2 dh1 = *reinterpret_cast<const __half2*>(&dw1[beta >> 1]);
        const float e0 = (beta & 1) ? __high2float(dh0) : __low2float(dh0);
        const float e1 = (beta & 1) ? __high2float(dh1) : __low2float(dh1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4& b = a[nt].bf[beta];
            float t[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(t, l0, l1, l2, l3, b.x, b.y);
            mma16816(t, u0, u1, u2, u3, b.z, b.w);
            float(&ac)[4] = (beta & 1) ? acc[nt][C1] : acc[nt][0];
            ac[0] = fmaf(e0, t[0], ac[0]);
            ac[1] = fmaf(e0, t[1], ac[1]);
            ac[2] = fmaf(e1, t[2], ac[2]);
            ac[3] = fmaf(e1, t[3], ac[3]);
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

// The value of the high half of a key: the value ordered by am_key (NaN
// read as -inf, -0 as +0).
__device__ __forceinline__ float key_value(unsigned long long k) {
    const uint32_t ord = static_cast<uint32_t>(k >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

constexpr int kFinishBatch = 8;

__device__ __forceinline__ unsigned long long umax64(unsigned long long a,
                                                     unsigned long long b) {
    return a > b ? a : b;
}

// The unit range of each CTA.  Stream-K (S == 0): CTA i owns units
// [iU/G, (i+1)U/G) of the (tile, stage) order, whatever the tile boundaries.
// Tile-aligned split-K (S > 0, G = tiles * S): CTA tS + p owns stages
// [pT/S, (p+1)T/S) of tile t, so no CTA spans two tiles.  Whole tiles
// (S < 0): CTA i owns tiles [i TT/G, (i+1) TT/G) of the TT = U / T tiles.
struct Range {
    unsigned long long U, G;
    int T, S;
    __device__ __forceinline__ unsigned long long start(unsigned long long i) const {
        if (S > 0) {
            const unsigned long long t = i / S, q = i % S;
            return t * T + q * T / S;
        }
        if (S < 0) return i * (U / T) / G * T;
        return i * U / G;
    }
    // the CTA whose range holds unit u
    __device__ __forceinline__ unsigned long long owner(unsigned long long u) const {
        if (S > 0) {
            const unsigned long long t = u / T, st = u % T;
            return t * S + ((st + 1) * S - 1) / T;
        }
        if (S < 0) {
            const unsigned long long TT = U / T;
            return ((u / T + 1) * G + TT - 1) / TT - 1;
        }
        return ((u + 1) * G + U - 1) / U - 1;
    }
};

// Called by the warp that completes the fused argmax bookkeeping.
// The last warp of the grid: each verify row's argmax out of its key, then,
// with greedy_B > 0, the greedy accept of every sequence (the longest draft
// prefix equal to the row argmaxes, then the argmax at the first mismatch or
// the bonus; a draft id outside [0, N) stops the prefix and is flagged).
__device__ void argmax_finish(const GemmParams& p, int lane) {
    __threadfence();
    int32_t am = 0;
    if (lane < p.argmax_M) {
        const unsigned long long k = atomicAdd(&p.am_key[lane], 0ull);
        am = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k));
        if (p.row_argmax != nullptr) p.row_argmax[lane] = am;
    }
    if (p.greedy_B > 0) {
        int32_t g[kMaxVerifyRows];
#pragma unroll
        for (int i = 0; i < kMaxVerifyRows; ++i) g[i] = __shfl_sync(0xffffffffu, am, i);
        const int Kd = p.greedy_Kd, b = lane;
        if (b < p.greedy_B) {
            const int32_t* d = p.drafts + b * Kd;
            const int r0 = b * (Kd + 1);
            int n = 0;
            bool bad = false;
            for (int i = 0; i < Kd; ++i) {
                const int32_t x = d[i];
                if (x < 0 || x >= p.N) {
                    bad = true;
                    break;
                }
                if (x != g[r0 + i]) break;
                ++n;
            }
            check(g[r0 + n] >= 0 && g[r0 + n] < p.N, p.status);  // the argmax was found
            for (int i = 0; i <= Kd; ++i)
                p.tokens[r0 + i] = i < n ? d[i] : (i == n ? g[r0 + n] : -1);
            p.len[b] = n + 1;
            if (bad) atomicOr(p.status, kStatusBadDraft);
        }
    }
}

// NR verify rows per activation block: 8 (one mma n-tile; dense or MoE) or
// 16 (two n-tiles over the same unpacked weights; dense calls of 9..16 rows).
template <int FMT, int NR>
__global__ void __launch_bounds__(kGemmThreads, 2)
    gemm_w4_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                   const GemmParams p) {
    using Sh = GemmShape<NR>;
    constexpr int NT = Sh::kNT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::kSmemBar);
    uint64_t* empty = full + Sh::kStages;
    uint64_t* never = empty + Sh::kStages;  // completed by nothing (the stall test)
    volatile int* abort_flag = reinterpret_cast<volatile int*>(never + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The next call's kernels may become resident now: they touch nothing
    // this grid uses before it has finished, and prefetch only weights.
    grid_dependents_launch();
    if (threadIdx.x == 0) {
        for (int s = 0; s < Sh::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(never, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmS);
    }
    __syncthreads();

    const int T = p.T, n_tiles = p.n_tiles;
    // Dense calls pass the one-segment shape directly.  MoE calls read the
    // routing table that the activation prep (this grid's predecessor)
    // writes: wait for that grid first.
    if (p.dense_M == 0) grid_dependency_wait();
    const int n_seg = p.dense_M > 0 ? 1 : p.seg->n_seg;
    // Effective grid: never more CTAs than units, so every active CTA owns at
    // least one unit (the contributor arithmetic of split tiles relies on it).
    const unsigned long long U = static_cast<unsigned long long>(n_seg) * n_tiles * T;
    // (whole-tile mode: never more CTAs than tiles)
    const unsigned long long n_items = p.split < 0 ? U / T : U;
    const unsigned long long G = n_items < gridDim.x ? n_items : gridDim.x;
    if (blockIdx.x >= G) return;
    const Range R{U, G, T, p.split};
    const unsigned long long u_begin = R.start(blockIdx.x), u_end = R.start(blockIdx.x + 1);
    // The split parts of a tile form one cluster and combine over DSMEM.
    // Every thread of such a CTA must reach both cluster barriers at the end,
    // so nothing below returns early in this mode (all waits are bounded).
    const bool cluster_mode = p.cluster != 0 && p.split > 1;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        // Lane 0 issues the copies and waits on the ring.
        if (lane != 0) {
            if (!cluster_mode) return;
            goto combine;
        }
        const uint64_t pol_w = policy_evict_first();   // nibbles: read exactly once
        const uint64_t pol_s = policy_evict_normal();  // scale sectors span two stages
        const uint64_t pol_a = policy_evict_last();    // activations: reread by every tile
        uint32_t it = 0;
        bool ok = true;
        // Scale boxes: a unit that starts a group of kScaleGroup stages (or
        // this CTA's range) loads one box into the next scale slot.  Before
        // reusing a slot, every stage that read the previous box must have
        // been released; the stage ring implies it unless that was less than
        // Sh::kStages units ago, in which case wait for that release explicitly.
        uint32_t n_sbox = 0;
        static_assert(kSSlots == 2, "two scale slots");
        uint32_t slot_last0 = 0xffffffffu, slot_last1 = 0xffffffffu;  // last unit per slot
        const int sg_n = p.sgroup;
        const int smask = sg_n == kScaleGroup ? kScaleGroup - 1 : 0x7fffffff;
        // Position of a unit: k stage, row tile, segment; advanced one unit at
        // a time so that the loop does no division.
        struct Cursor {
            int st, tile, sg, row0;
        };
        auto cursor_at = [&](unsigned long long u) {
            const unsigned long long tg = u / T;
            Cursor c{static_cast<int>(u % T), static_cast<int>(tg % n_tiles),
                     static_cast<int>(tg / n_tiles), 0};
            const int expert = p.dense_M > 0 ? 0 : p.seg->expert[c.sg];
            c.row0 = expert * p.N + c.tile * kTileRows;
            return c;
        };
        auto advance = [&](Cursor& c) {
            if (++c.st < T) return;
            c.st = 0;
            c.row0 += kTileRows;
            if (++c.tile < n_tiles) return;
            c.tile = 0;
            ++c.sg;
            if (c.sg < n_seg) {
                const int expert = p.dense_M > 0 ? 0 : p.seg->expert[c.sg];
                c.row0 = expert * p.N;
            }
        };
        // Returns 1 when issued, 0 when a wait ran out, -1 when the unit would
        // have to wait but may not (then nothing was changed).
        // with_act: also copy the stage's activation block now (it is ready).
        auto issue = [&](const Cursor& c, bool first, uint32_t it_u, bool with_act,
                         bool may_wait) -> int {
            const int s = it_u % Sh::kStages;
            const bool new_box = first || (c.st & smask) == 0;
            // the activation copy of a unit issued before the prep wait is
            // added later, but its bytes are expected here already
            uint32_t bytes = kWBytes + Sh::kAStride;
            int sslot = (n_sbox + kSSlots - 1) % kSSlots;
            if (new_box) {
                sslot = n_sbox % kSSlots;
                const uint32_t last = sslot ? slot_last1 : slot_last0;
                if (last != 0xffffffffu && it_u - last < static_cast<uint32_t>(Sh::kStages)) {
                    if (!may_wait) return -1;
                    if (!mbar_wait_bounded(&empty[last % Sh::kStages], (last / Sh::kStages) & 1, p.wait_ns,
                                           abort_flag))
                        return 0;
                }
                bytes += kTileRows * 16 * sg_n;
                ++n_sbox;
            }
            if (sslot) slot_last1 = it_u;
            else slot_last0 = it_u;
            mbar_arrive_expect_tx(&full[s], bytes);
            tma_load_2d(smem + s * kWBytes, &tmW, c.st * (kStageK / 2), c.row0, &full[s], pol_w);
            if (new_box) {  // box start: this stage, moved back to fit inside the row
                const int st_box = c.st < T - sg_n ? c.st : T - sg_n;
                tma_load_2d(smem + Sh::kSmemS + sslot * kSSlotBytes, &tmS, st_box * 16, c.row0,
                            &full[s], pol_s);
            }
            if (with_act)
                bulk_load(smem + Sh::kSmemA + s * Sh::kAStride,
                          p.act + (static_cast<size_t>(c.sg) * T + c.st) * Sh::kAStride, Sh::kAStride,
                          &full[s], pol_a);
            return 1;
        };
        // The weights and scales do not depend on the activation prep: start
        // streaming up to Sh::kStages units before waiting for it (stopping early
        // rather than waiting on consumers, who need the activations first).
        const Cursor c0 = cursor_at(u_begin);
        Cursor cur = c0;
        const unsigned long long n_units = u_end - u_begin;
        while (it < n_units && it < static_cast<uint32_t>(Sh::kStages)) {
            if (issue(cur, it == 0, it, false, false) != 1) break;
            ++it;
            advance(cur);
        }
        const uint32_t n_pre = it;
        grid_dependency_wait();
        {
            Cursor a = c0;
            for (uint32_t j = 0; j < n_pre; ++j, advance(a))
                bulk_load(smem + Sh::kSmemA + j * Sh::kAStride,
                          p.act + (static_cast<size_t>(a.sg) * T + a.st) * Sh::kAStride, Sh::kAStride,
                          &full[j], pol_a);
        }
        for (; it < n_units; ++it, advance(cur)) {
            const int s = it % Sh::kStages;
            if ((it >= static_cast<uint32_t>(Sh::kStages) &&
                 !mbar_wait_bounded(&empty[s], ((it / Sh::kStages) - 1) & 1, p.wait_ns,
                                    abort_flag)) ||
                issue(cur, it == 0, it, true, true) != 1) {
                ok = false;
                break;
            }
        }
        if (!ok) {
            atomicOr(p.status, kStatusTimeout);
            *abort_flag = 1;
        }
        // Drain: every issued copy must land before this CTA may exit.
        const uint64_t drain_ns = p.wait_ns > 2000000000ull ? p.wait_ns : 2000000000ull;
        for (uint32_t j = (it > (uint32_t)Sh::kStages ? it - Sh::kStages : 0u); j < it; ++j)
            mbar_wait_bounded(&full[j % Sh::kStages], (j / Sh::kStages) & 1, drain_ns, nullptr);
        if (!cluster_mode) return;
        goto combine;
    }

    // ---------------------------------------------------------- consumers
    {
    grid_dependency_wait();  // activations, scales of this call, tickets reset
    if (p.stall_test && !mbar_wait_bounded(never, 0u, p.wait_ns, abort_flag)) {
        if (lane == 0) atomicOr(p.status, kStatusTimeout);
        *abort_flag = 1;
        if (cluster_mode) goto combine;
        return;
    }
    const int g = lane >> 2, c = lane & 3;
    const int wrow = warp * kWarpRows;  // first tile row of this warp
    uint32_t it = 0;
    uint32_t n_sbox = 0;  // scale boxes seen, in the producer's order
    // scale slot of the current box, offset back by the box's first stage
    const uint8_t* s_base = smem + Sh::kSmemS;
    const int sg_n = p.sgroup;
    const int spitch = 16 * sg_n;
    const int smask = sg_n == kScaleGroup ? kScaleGroup - 1 : 0x7fffffff;
    const unsigned long long my_first_tile = u_begin / T;
    // fused argmax: this warp's running key of verify row lane / 4 (held in
    // the lanes with lane % 4 == 0), published once when the warp is done
    unsigned long long am_run[NT] = {};
    for (unsigned long long u = u_begin; u < u_end;) {
        const unsigned long long tg = u / T;
        const int st0 = static_cast<int>(u % T);
        const unsigned long long left = u_end - u;
        const int st_end = (left < static_cast<unsigned long long>(T - st0))
                               ? st0 + static_cast<int>(left)
                               : T;
        float tot[kRowBlocks][NT][4] = {};
        for (int st = st0; st < st_end; ++st, ++it) {
            const int s = it % Sh::kStages;
            if (!mbar_wait_bounded(&full[s], (it / Sh::kStages) & 1, p.wait_ns, abort_flag)) {
                if (lane == 0) atomicOr(p.status, kStatusTimeout);
                *abort_flag = 1;
                if (cluster_mode) goto combine;
                return;
            }
            if (it == 0 || (st & smask) == 0) {
                ++n_sbox;
                const int sbox_st = st < T - sg_n ? st : T - sg_n;
                s_base = smem + Sh::kSmemS + ((n_sbox - 1) % kSSlots) * kSSlotBytes - sbox_st * 16;
            }
            const uint8_t* Ws = smem + s * kWBytes;
            const uint8_t* Ss = s_base + st * 16 + (wrow + g) * spitch;
            const uint8_t* As = smem + Sh::kSmemA + s * Sh::kAStride;
            constexpr int NC = Chains<NT>::kN;
            float acc[kRowBlocks][NT][NC][4] = {};
            ActRegs ar[NT];
            if (FMT == 1) {
                WRegsNv wr[kRowBlocks];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    load_act_nvfp4(As + nt * act_bytes(8), As + Sh::kABytes + nt * 32, lane, ar[nt]);
#pragma unroll
                for (int rb = 0; rb < kRowBlocks; ++rb)
                    load_w_nvfp4(Ws, Ss + rb * 16 * spitch, spitch, wrow + rb * 16 + g, lane,
                                 wr[rb]);
                __syncwarp();  // every lane's reads of the slot are done:
                if (lane == 0) mbar_arrive(&empty[s]);  // the producer may refill it
#pragma unroll
                for (int rb = 0; rb < kRowBlocks; ++rb)
                    compute_nvfp4<NT>(ar, wr[rb], acc[rb]);
            } else {
                // Q4_0: one 16-row block loaded and computed at a time, the
                // slot released after both (fewer registers live at once:
                // gate_up 28.3 against 29.0 us, down 19.6 against 20.6)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    load_act_q4_0(As + nt * act_bytes(8), As + Sh::kABytes + nt * 32, lane, ar[nt]);
#pragma unroll
                for (int rb = 0; rb < kRowBlocks; ++rb) {
                    WRegsQ4 wr;
                    load_w_q4_0(Ws, Ss + rb * 16 * spitch, spitch, wrow + rb * 16 + g, lane, wr);
                    compute_q4_0<NT>(ar, wr, acc[rb]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // this stage's activations were scaled by 2^s per verify row
#pragma unroll
            for (int rb = 0; rb < kRowBlocks; ++rb)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 iv = ar[nt].inv;
                    float(&t)[4] = tot[rb][nt];
                    const float(&a0)[4] = acc[rb][nt][0];
                    const float(&a1)[4] = acc[rb][nt][NC - 1];
                    if (NC == 2) {
                        t[0] = fmaf(iv.x, a0[0] + a1[0], t[0]);
                        t[1] = fmaf(iv.y, a0[1] + a1[1], t[1]);
                        t[2] = fmaf(iv.x, a0[2] + a1[2], t[2]);
                        t[3] = fmaf(iv.y, a0[3] + a1[3], t[3]);
                    } else {
                        t[0] = fmaf(iv.x, a0[0], t[0]);
                        t[1] = fmaf(iv.y, a0[1], t[1]);
                        t[2] = fmaf(iv.x, a0[2], t[2]);
                        t[3] = fmaf(iv.y, a0[3], t[3]);
                    }
                }
        }
        u += static_cast<unsigned long long>(st_end - st0);

        // ------------------------------------------------------ epilogue
        // Lane (g, c) holds, per row block rb and n-tile nt, rows
        // r = wrow + 16rb + g (+8 for q & 2) and verify rows 8nt + 2c + (q & 1).
        const int sg = static_cast<int>(tg / n_tiles), tile = static_cast<int>(tg % n_tiles);
        const int count = p.dense_M > 0 ? p.dense_M : p.seg->count[sg];
        // output row of verify row tok (16-row blocks are dense-only)
        auto dest_of = [&](int tok) {
            return (NR > kMaxRows || p.dense_M > 0) ? tok : p.seg->dest[sg][tok];
        };
        float v[kRowBlocks][NT][4];
#pragma unroll
        for (int rb = 0; rb < kRowBlocks; ++rb)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) v[rb][nt][q] = tot[rb][nt][q] * p.tensor_scale;
        const int n0 = tile * kTileRows;
        const bool whole = (st0 == 0 && st_end == T);
        if (whole) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // argmax keys of verify rows 8nt + 2c and 8nt + 2c + 1, per
                // 16-row block and over the warp's 32 rows
                unsigned long long k0 = 0ull, k1 = 0ull;
                unsigned long long kr0[kRowBlocks], kr1[kRowBlocks];
#pragma unroll
                for (int rb = 0; rb < kRowBlocks; ++rb) {
                    kr0[rb] = kr1[rb] = 0ull;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tok = 8 * nt + 2 * c + (q & 1);
                        const int n = n0 + wrow + rb * 16 + g + ((q & 2) ? 8 : 0);
                        if (n < p.N) {
                            if (tok < count && p.out != nullptr) {
                                const int dr = dest_of(tok);
                                if (check(dr >= 0 && dr < p.out_rows, p.status))
                                    p.out[static_cast<size_t>(dr) * p.ldo + n] = v[rb][nt][q];
                            }
                            const unsigned long long k =
                                am_key(v[rb][nt][q], static_cast<uint32_t>(n));
                            if (q & 1) kr1[rb] = umax64(kr1[rb], k);
                            else kr0[rb] = umax64(kr0[rb], k);
                        }
                    }
                    k0 = umax64(k0, kr0[rb]);
                    k1 = umax64(k1, kr1[rb]);
                }
                if (p.bmax != nullptr) {
                    // the largest of each 16 outputs: one block per row block
#pragma unroll
                    for (int rb = 0; rb < kRowBlocks; ++rb) {
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) {
                            kr0[rb] = umax64(kr0[rb], __shfl_xor_sync(0xffffffffu, kr0[rb], o));
                            kr1[rb] = umax64(kr1[rb], __shfl_xor_sync(0xffffffffu, kr1[rb], o));
                        }
                        const int nb0 = n0 + wrow + rb * 16;
                        const int t0 = 8 * nt + 2 * c;
                        if (lane < 4 && nb0 < p.N) {  // lane c holds rows 2c, 2c + 1
                            float* bm = p.bmax + nb0 / kBlockMaxRows;
                            if (t0 < count) bm[static_cast<size_t>(t0) * p.ldb] = key_value(kr0[rb]);
                            if (t0 + 1 < count)
                                bm[static_cast<size_t>(t0 + 1) * p.ldb] = key_value(kr1[rb]);
                        }
                    }
                }
                if (p.argmax_M > 0) {
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        k0 = umax64(k0, __shfl_xor_sync(0xffffffffu, k0, o));
                        k1 = umax64(k1, __shfl_xor_sync(0xffffffffu, k1, o));
                    }
                    // lane c (< 4) holds rows 2c and 2c + 1 of the n-tile;
                    // row t goes to lanes 4t .. 4t + 3
                    const int t = lane >> 2;
                    const unsigned long long a = __shfl_sync(0xffffffffu, k0, t >> 1);
                    const unsigned long long b = __shfl_sync(0xffffffffu, k1, t >> 1);
                    am_run[nt] = umax64(am_run[nt], (t & 1) ? b : a);
                }
            }
            continue;
        }
        if (cluster_mode) {  // leave this part's slice in shared memory
            float* part = reinterpret_cast<float*>(smem + Sh::kSmemPart);
#pragma unroll
            for (int rb = 0; rb < kRowBlocks; ++rb)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int tok = 8 * nt + 2 * c + (q & 1);
                        const int r = wrow + rb * 16 + g + ((q & 2) ? 8 : 0);
                        part[tok * kTileRows + r] = v[rb][nt][q];
                    }
            continue;
        }
        // Partial tile: publish this warp's 32-row slice; the last of the
        // tile's contributors to arrive for this slice sums it in k order.
        const unsigned long long tile_u0 = tg * static_cast<unsigned long long>(T);
        const unsigned long long i_lo = R.owner(tile_u0), i_hi = R.owner(tile_u0 + T - 1);
        const uint32_t n_contrib = static_cast<uint32_t>(i_hi - i_lo + 1);
        const unsigned long long my_slot =
            2ull * blockIdx.x + ((my_first_tile == tg) ? 0ull : 1ull);
        float* part = p.partials + my_slot * Sh::kPartialFloats;
#pragma unroll
        for (int rb = 0; rb < kRowBlocks; ++rb)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int tok = 8 * nt + 2 * c + (q & 1);
                    const int r = wrow + rb * 16 + g + ((q & 2) ? 8 : 0);
                    __stcg(&part[tok * kTileRows + r], v[rb][nt][q]);
                }
        // The warp barrier orders every lane's partial stores before lane 0's
        // release; the last arriver's acquire orders the reads after them.
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = atom_add_acq_rel_gpu(&p.tile_cnt[tg * kConsumerWarps + warp], 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old + 1 != n_contrib) continue;
        // Every contributor after the first starts inside this tile, so its
        // slot is its "first tile" slot; only the first may end in it instead.
        const unsigned long long slot_lo =
            2ull * i_lo + ((R.start(i_lo) / T == tg) ? 0ull : 1ull);
        // lane: verify row 8nt + tok of each n-tile, rows rr .. rr+3 and
        // rr+16 .. rr+19 of the slice
        const int rr = wrow + 4 * (lane & 3);
        auto slot_of = [&](unsigned long long i) { return i == i_lo ? slot_lo : 2ull * i; };
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int tok = 8 * nt + (lane >> 2);
            const size_t off = static_cast<size_t>(tok) * kTileRows + rr;
            auto ld4 = [&](unsigned long long i, int h) {
                return __ldcg(reinterpret_cast<const float4*>(
                    p.partials + slot_of(i) * Sh::kPartialFloats + off + 16 * h));
            };
            float4 sa = make_float4(0.f, 0.f, 0.f, 0.f), sb = sa;
            // up to kFinishBatch contributors' loads in flight, then summed in order
            for (unsigned long long i0 = i_lo; i0 <= i_hi; i0 += kFinishBatch) {
                float4 xa[kFinishBatch], xb[kFinishBatch];
#pragma unroll
                for (int j = 0; j < kFinishBatch; ++j) {  // past the end: reload the last
                    const unsigned long long ij = i0 + j <= i_hi ? i0 + j : i_hi;
                    xa[j] = ld4(ij, 0);
                    xb[j] = ld4(ij, 1);
                }
#pragma unroll
                for (int j = 0; j < kFinishBatch; ++j) {
                    if (i0 + j <= i_hi) {
                        sa.x += xa[j].x; sa.y += xa[j].y; sa.z += xa[j].z; sa.w += xa[j].w;
                        sb.x += xb[j].x; sb.y += xb[j].y; sb.z += xb[j].z; sb.w += xb[j].w;
                    }
                }
            }
            const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
            // keys of the slice's first and second 16 rows
            unsigned long long kb0 = 0ull, kb1 = 0ull;
            if (tok < count) {
                const int dr = dest_of(tok);
                float* orow = p.out != nullptr && check(dr >= 0 && dr < p.out_rows, p.status)
                                  ? p.out + static_cast<size_t>(dr) * p.ldo
                                  : nullptr;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int n = n0 + rr + (j & 3) + ((j & 4) ? 16 : 0);
                    if (n < p.N) {
                        if (orow != nullptr) orow[n] = sv[j];
                        const unsigned long long k = am_key(sv[j], static_cast<uint32_t>(n));
                        if (j & 4) kb1 = umax64(kb1, k);
                        else kb0 = umax64(kb0, k);
                    }
                }
            }
            if (p.argmax_M > 0 || p.bmax != nullptr) {
                kb0 = umax64(kb0, __shfl_xor_sync(0xffffffffu, kb0, 1));
                kb0 = umax64(kb0, __shfl_xor_sync(0xffffffffu, kb0, 2));
                kb1 = umax64(kb1, __shfl_xor_sync(0xffffffffu, kb1, 1));
                kb1 = umax64(kb1, __shfl_xor_sync(0xffffffffu, kb1, 2));
                // lanes 4t .. 4t+3 hold row 8nt + t
                am_run[nt] = umax64(am_run[nt], umax64(kb0, kb1));
                if (p.bmax != nullptr && (lane & 3) == 0 && tok < count) {
                    float* bm = p.bmax + static_cast<size_t>(tok) * p.ldb;
                    if (n0 + wrow < p.N) bm[(n0 + wrow) / kBlockMaxRows] = key_value(kb0);
                    if (n0 + wrow + 16 < p.N) bm[(n0 + wrow + 16) / kBlockMaxRows] = key_value(kb1);
                }
            }
        }
    }
    if (p.argmax_M > 0) {
        // one 64-bit max per verify row and warp, then a ticket: the last of
        // the grid's consumer warps reads the maxima out
        const int t = lane >> 2;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = 8 * nt + t;
            if ((lane & 3) == 0 && row < p.argmax_M && am_run[nt])
                atomicMax(&p.am_key[row], am_run[nt]);
        }
        __syncwarp();
        uint32_t o2 = 0;
        if (lane == 0) o2 = atom_add_acq_rel_gpu(p.am_cnt, 1u);
        o2 = __shfl_sync(0xffffffffu, o2, 0);
        if (o2 + 1 == static_cast<uint32_t>(kConsumerWarps * G)) argmax_finish(p, lane);
    }
    }
    if (!cluster_mode) return;
combine:
    {
        // Fused split-K: the parts' partial tiles (rank order = k order) are
        // summed by the consumers of all the parts, each part taking its
        // share of the tile's elements (every partial of an element loaded
        // before the first add); the second barrier keeps every part's
        // shared memory alive until all have read it.
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        const int S = static_cast<int>(cl.num_blocks());
        if (warp < kConsumerWarps) {
            int aborted = 0;
            const float* parts[kMaxClusterSplit];
#pragma unroll
            for (int r = 0; r < kMaxClusterSplit; ++r) {
                parts[r] = nullptr;
                if (r < S) {
                    aborted |= *cl.map_shared_rank(const_cast<int*>(abort_flag), r);
                    parts[r] = cl.map_shared_rank(reinterpret_cast<float*>(smem + Sh::kSmemPart), r);
                }
            }
            const int n0 = static_cast<int>(blockIdx.x / S) * kTileRows;
            constexpr int kPairs = NR * kTileRows / 2;  // the tile as float2
            for (int e = static_cast<int>(cl.block_rank()) * kGemmConsumers + threadIdx.x;
                 e < kPairs; e += S * kGemmConsumers) {
                const int tok = e / (kTileRows / 2), r0 = (e % (kTileRows / 2)) * 2;
                float2 v[kMaxClusterSplit];
#pragma unroll
                for (int r = 0; r < kMaxClusterSplit; ++r)
                    if (r < S) v[r] = *reinterpret_cast<const float2*>(parts[r] + tok * kTileRows + r0);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int r = 0; r < kMaxClusterSplit; ++r)
                    if (r < S) {
                        acc.x += v[r].x;
                        acc.y += v[r].y;
                    }
                if (!aborted && tok < p.dense_M) {
                    float* orow = p.out + static_cast<size_t>(tok) * p.ldo;
                    if (n0 + r0 < p.N) orow[n0 + r0] = acc.x;
                    if (n0 + r0 + 1 < p.N) orow[n0 + r0 + 1] = acc.y;
                }
            }
        }
        cl.sync();
    }
}

// ------------------------------------------------------------ MoE combine
__global__ void combine_kernel(const float* __restrict__ pair_out, const float* __restrict__ gates,
                               const int32_t* __restrict__ ids, int E, int M, int topk, int N,
                               float* __restrict__ out, int ldo) {
    // launched early behind the GEMM; reads nothing before that grid is done
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
                            int n_counters, cudaStream_t s, int nr, const int32_t* ids, int E,
                            uint32_t* status, float* out_zero, int ldo, int N, int K_true) {
    if ((nr != 8 && nr != 16) || (nr == 16 && dense_M <= 0)) return cudaErrorInvalidValue;
    const int T = K / kStageK;
    const int vec_ok = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0 && lda % 8 == 0) ? 1 : 0;
    // a programmatic dependent of whatever kernel precedes it on the stream
    cudaLaunchConfig_t cfg{};
    // MoE: a few CTAs per segment, each computing the routing for several
    // stages, about 256 CTAs in all (the routing is redundant per CTA)
    int stage_ctas = T;
    if (dense_M <= 0) {
        stage_ctas = 256 / (n_seg_grid > 0 ? n_seg_grid : 1);
        stage_ctas = stage_ctas < 1 ? 1 : (stage_ctas > T ? T : stage_ctas);
    }
    cfg.gridDim = dim3(n_seg_grid * stage_ctas);
    cfg.blockDim = dim3(32 * nr);  // one warp per verify row
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prep_act_kernel, A, lda, vec_ok, K, K_true > 0 ? K_true : K,
                              fmt, nr, dense_M,
                              rows_are_pairs, topk, ws.seg, ws.act, ws.tile_cnt, n_counters,
                              ws.am_key, ws.am_cnt, ids, dense_M > 0 ? 0 : n_seg_grid, E, status,
                              out_zero, ldo, N, stage_ctas);
}

template <int FMT, int NR>
static cudaError_t launch_gemm_t(const CUtensorMap& tmW, const CUtensorMap& tmS,
                                 const GemmParams& p, int grid, int cluster, cudaStream_t s) {
    constexpr int kSmem = GemmShape<NR>::kSmem;
    static std::atomic<unsigned long long> attr_once{0};
    cudaError_t ea = set_attribute_per_device(attr_once, [] {
        return cudaFuncSetAttribute(gemm_w4_kernel<FMT, NR>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {  // the split parts of a tile: one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, gemm_w4_kernel<FMT, NR>, tmW, tmS, p);
}

cudaError_t launch_gemm(int fmt, int nr, const CUtensorMap& tmW, const CUtensorMap& tmS,
                        const GemmParams& p, int grid, int cluster, cudaStream_t s) {
    if (nr == 16) {
        if (p.dense_M <= 0) return cudaErrorInvalidValue;  // 16-row blocks are dense-only
        return fmt == 1 ? launch_gemm_t<1, 16>(tmW, tmS, p, grid, cluster, s)
                        : launch_gemm_t<2, 16>(tmW, tmS, p, grid, cluster, s);
    }
    return fmt == 1 ? launch_gemm_t<1, 8>(tmW, tmS, p, grid, cluster, s)
                    : launch_gemm_t<2, 8>(tmW, tmS, p, grid, cluster, s);
}

template <int FMT, int NR>
static int blocks_per_sm_t() {
    constexpr int kSmem = GemmShape<NR>::kSmem;
    int n = 0;
    cudaFuncSetAttribute(gemm_w4_kernel<FMT, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemm_w4_kernel<FMT, NR>, kGemmThreads, kSmem);
    return n > 0 ? n : 1;
}

int gemm_blocks_per_sm(int fmt, int nr) {
    if (nr == 16) return fmt == 1 ? blocks_per_sm_t<1, 16>() : blocks_per_sm_t<2, 16>();
    return fmt == 1 ? blocks_per_sm_t<1, 8>() : blocks_per_sm_t<2, 8>();
}

cudaError_t launch_combine(const float* pair_out, const float* gates, const int32_t* ids,
                               int E, int M, int topk, int N, float* out, int ldo, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((N + 255) / 256, M);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, pair_out, gates, ids, E, M, topk, N, out, ldo);
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
