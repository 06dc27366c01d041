// vw4_internal.cuh -- shapes, workspace layout and kernel parameter blocks
// shared by the kernels and the C-ABI layer.  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>

namespace vw4 {

// Kernel attributes set with cudaFuncSetAttribute apply to the current device
// only: `once` keeps one bit per device (devices past 63 set it every time).
inline cudaError_t set_attribute_per_device(std::atomic<unsigned long long>& once,
                                            cudaError_t (*set)()) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (bit && (once.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit) once.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// In-kernel bounds checks, compiled in by -DVW4_CHECKS (the checks build):
// check(ok, status) records a failed check in the device status word
// (VW4_DEV_BOUNDS) and returns false, so that the caller skips the access.
// In other builds it returns true and the test compiles away.
constexpr uint32_t kStatusBounds = 0x20u;
#ifdef VW4_CHECKS
constexpr bool kChecks = true;
#else
constexpr bool kChecks = false;
#endif
__device__ __forceinline__ bool check(bool ok, uint32_t* status) {
    if (kChecks && !ok) {
        atomicOr(status, kStatusBounds);
        return false;
    }
    return true;
}

constexpr int kMaxRows = 8;        // rows of one mma n-tile; verify rows per MoE segment
constexpr int kMaxVerifyRows = 16; // dense verify rows per call: two n-tiles
constexpr int kMaxSeg = 128;       // routed (token, expert) pairs per call: 16 tokens x top-8
constexpr int kTileRows = 128;     // weight rows per tile
constexpr int kStageK = 256;       // k elements per pipeline stage
constexpr int kMinUnitsPerCta = 4; // tile-aligned split-K: at least this many stages per part
constexpr int kMaxSplit = 6;       // tile-aligned split-K: at most this many parts
constexpr int kMaxClusterSplit = 6; // parts combined as one cluster (larger ones place poorly)
constexpr int kConsumerWarps = 4;  // each owns 32 rows of the tile
constexpr int kWarpRows = kTileRows / kConsumerWarps;  // 32
constexpr int kRowBlocks = kWarpRows / 16;             // 16-row MMA blocks per warp
constexpr int kGemmThreads = (kConsumerWarps + 1) * 32;
constexpr int kGemmConsumers = kConsumerWarps * 32;
constexpr int kBlockMaxRows = 16;  // the fused block maxima: one per 16 outputs
static_assert(kRowBlocks == 2, "the split-tile finish assumes two row blocks per warp");
constexpr int kWBytes = kTileRows * (kStageK / 2);     // 16384: packed nibbles
// Scales travel in boxes of 128 rows x (16 * g) bytes that cover g = min(4, T)
// consecutive stages (16 bytes per row per stage), into a ring of 2 slots: one
// request of two full sectors per row instead of four half-sector requests.
// Every box lies inside the row: the last one of a row is moved back to end
// at the row's end.
constexpr int kScaleGroup = 4;
static_assert((kScaleGroup & (kScaleGroup - 1)) == 0, "scale group must be a power of two");
constexpr int kSBoxBytes = 16 * kScaleGroup;           // 64 (slot row pitch)
constexpr int kSSlotBytes = kTileRows * kSBoxBytes;    // 8192
constexpr int kSSlots = 2;

// Activation block of one (segment, stage) for NR verify rows: fp16 [NR][256]
// (scaled, bank-swizzled), then float 2^-s [NR].
__host__ __device__ constexpr int act_bytes(int nr) { return nr * kStageK * 2; }
__host__ __device__ constexpr int act_stride(int nr) { return act_bytes(nr) + nr * 4; }

// The GEMM's shapes for NR verify rows (8: one mma n-tile; 16: two n-tiles
// sharing every unpacked weight fragment).  Shared memory:
// [W x kStages][S x kSSlots][A x kStages][barriers][partial tile]; every W slot
// is 1024-byte aligned (128-byte swizzle).  Sixteen rows double the
// activation slots and the partial tile, so that ring is one stage shorter
// to keep two CTAs per SM.
template <int NR>
struct GemmShape {
    static_assert(NR == 8 || NR == 16, "8 or 16 verify rows");
    static constexpr int kNT = NR / 8;
    static constexpr int kStages = NR == 8 ? 4 : 3;
    static constexpr int kABytes = act_bytes(NR);     // 4096 / 8192
    static constexpr int kAStride = act_stride(NR);   // 4128 / 8256
    static constexpr int kSmemS = kStages * kWBytes;
    static constexpr int kSmemA = kSmemS + kSSlots * kSSlotBytes;
    static constexpr int kSmemBar = kSmemA + kStages * kAStride;
    static constexpr int kSmemPart = kSmemBar + 256;  // cluster mode: this CTA's partial tile
    static constexpr int kPartialFloats = NR * kTileRows;
    static constexpr int kSmem = kSmemPart + kPartialFloats * 4 + 1024 /*align*/;
    static_assert(kAStride % 16 == 0 && kSmemA % 16 == 0, "bulk copies need 16-byte alignment");
    static_assert(kSmemBar % 8 == 0 && kSmemPart % 16 == 0, "barrier / partial alignment");
    static_assert(kSmem <= 113 * 1024, "two CTAs per SM");
};
inline int gemm_rows_for(int M) { return M <= kMaxRows ? 8 : 16; }

// A "segment" is the set of verify rows that share one weight matrix: the
// whole batch for a dense layer, or the pairs routed to one expert.
struct SegTable {
    int n_seg;
    int pad[3];
    int expert[kMaxSeg];
    int count[kMaxSeg];
    int dest[kMaxSeg][kMaxRows];  // output row of each segment row
};

struct GemmWorkspace {
    SegTable* seg;
    uint8_t* act;                // [seg][T] blocks of act_stride(nr) bytes
    float* partials;             // [2 * grid][nr][128] stream-K partial tiles
    uint32_t* tile_cnt;          // [seg * n_tiles * kConsumerWarps] slice arrival tickets
    unsigned long long* am_key;  // [16] packed (value, ~index) running maxima
    uint32_t* am_cnt;            // [1] quarter-tile tickets of the argmax
    float* pair_out;             // [pairs][N] MoE pair rows before the combine
    uint8_t* wpad;               // [N][Kp/2] nibbles padded to whole stages (K % 256 != 0)
    uint8_t* spad;               // [N][Kp/16] their scales
    size_t bytes;
};

struct GemmParams {
    int N, K, T, n_tiles;
    int sgroup;                   // stages per scale box, min(kScaleGroup, T)
    int split;                    // > 0: tile-aligned split-K into this many parts; 0: stream-K
    float tensor_scale;
    const SegTable* seg;
    const uint8_t* act;
    float* out;
    int ldo;
    int out_rows;                 // rows of out: the verify rows, or the routed pairs
    int dense_M;                  // > 0: one dense segment of dense_M rows (no table reads)
    int argmax_M;                 // 0 = no fused argmax
    float* partials;
    uint32_t* tile_cnt;
    unsigned long long* am_key;
    uint32_t* am_cnt;
    int32_t* row_argmax;
    float* bmax;                  // optional [M][ldb]: the largest output of every 16
    int ldb;
    uint32_t* status;
    unsigned long long wait_ns;
    // cluster != 0 (tile-aligned split-K without a fused reduction): the split
    // parts of a tile are launched as one cluster and combine their partial
    // tiles over distributed shared memory instead of tickets in L2.
    int cluster;
    // greedy accept in the same launch (greedy_B > 0, with the fused argmax
    // over M = greedy_B * (greedy_Kd + 1) rows): sequence b's target rows are
    // b (Kd + 1) .. b (Kd + 1) + Kd; out may then be null (no logits written)
    int greedy_B, greedy_Kd;
    const int32_t* drafts;
    int32_t* tokens;
    int32_t* len;
    // test hook: the consumers first wait on a barrier nothing completes, so
    // that the bounded wait runs out (the timeout path, without a fault)
    int stall_test;
};

// Lays the GEMM/MoE workspace out from `base` (nullptr: size only) for
// blocks of nr (8 or 16) verify rows.
// K: the stages' K (a multiple of 256); pad_rows > 0: room for a copy of
// that many weight rows padded to K.
GemmWorkspace gemm_workspace_layout(void* base, int n_seg_max, int N, int K, int grid,
                                    int pair_rows, int nr, int pad_rows = 0);

// Kernel launchers (gemm_w4.cu).  All asynchronous on `s`.
// nr: rows per activation block (8, or 16 for a dense call of 9..16 rows)
cudaError_t launch_prep_act(const uint16_t* A, int lda, int K, int fmt, int dense_M,
                            int rows_are_pairs, int topk, int n_seg_grid, const GemmWorkspace& ws,
                            int n_counters, cudaStream_t s, int nr, const int32_t* ids = nullptr,
                            int E = 0, uint32_t* status = nullptr, float* out_zero = nullptr,
                            int ldo = 0, int N = 0, int K_true = 0);
cudaError_t launch_pad_weights(const void* q, const void* sc, int N, int K, int Kp, uint8_t* qo,
                               uint8_t* so, cudaStream_t s);
cudaError_t launch_gemm(int fmt, int nr, const CUtensorMap& tmW, const CUtensorMap& tmS,
                        const GemmParams& p, int grid, int cluster, cudaStream_t s);
cudaError_t launch_combine(const float* pair_out, const float* gates, const int32_t* ids,
                           int E, int M, int topk, int N, float* out, int ldo, cudaStream_t s);
cudaError_t launch_q4_0_split(const uint8_t* blocks, int N, int K, uint8_t* q, __half* d,
                              cudaStream_t s);
int gemm_blocks_per_sm(int fmt, int nr);

// Accept launchers (accept.cu).
cudaError_t launch_accept_greedy(const float* logits, const int32_t* drafts,
                                 const int32_t* argmax_in, int B, int Kd, int V, int32_t* tokens,
                                 int32_t* len, uint32_t* status, cudaStream_t s);
size_t rejection_workspace_bytes(int B, int Kd, int V);
cudaError_t launch_own_exp(const float* x, float* y, long long n, cudaStream_t s);
cudaError_t launch_own_mass_pairs(const float* x, unsigned long long* W, long long n,
                                  cudaStream_t s);
cudaError_t launch_accept_rejection(const float* target, const float* draft,
                                    const int32_t* drafts, int B, int Kd, int V, float invT,
                                    uint64_t P, int top_k, uint64_t MP, uint64_t seed,
                                    uint64_t offset, int32_t* tokens,
                                    int32_t* len, void* ws, size_t ws_bytes, uint32_t* status,
                                    unsigned long long wait_ns, cudaStream_t s,
                                    const float* target_bmax = nullptr,
                                    const float* draft_bmax = nullptr);

// Copies the first `rows` row records of a rejection workspace (test hook).
cudaError_t copy_rejection_row_records(const void* ws, long long rows, void* out,
                                       cudaStream_t s);
size_t rejection_topk_workspace_bytes(int B, int Kd, int Kt);
cudaError_t launch_accept_rejection_topk(const int32_t* t_ids, const float* t_vals,
                                         const int32_t* d_ids, const float* d_vals,
                                         const int32_t* drafts, int B, int Kd, int Kt, int V,
                                         float invT, uint64_t P, int top_k, uint64_t MP,
                                         uint64_t seed, uint64_t offset, int32_t* tokens,
                                         int32_t* len, void* ws, size_t ws_bytes,
                                         uint32_t* status, cudaStream_t s);

}  // namespace vw4
