// api.cu -- the C ABI declared in include/vw4.h: host-side argument checks,
// workspace carving, TMA tensor-map encoding and kernel launches.  No call
// allocates device memory and none synchronizes (except the status read).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "vw4.h"
#include "vw4_internal.cuh"

namespace vw4 {

// One status word per device.  Kernels OR bits into it; vw4_get_device_status
// reads and clears it.
__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGrid = 608;  // upper bound of the persistent GEMM grid (workspace sizing)

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int occ[3][2] = {};  // GEMM CTAs per SM by fmt and row block (8, 16 rows)
    uint32_t* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
unsigned long long g_wait_ns = 2000000000ull;
std::atomic<int> g_stall_calls{0};  // test hook: GEMM launches left to stall

int take_stall() {
    int n = g_stall_calls.load();
    while (n > 0 && !g_stall_calls.compare_exchange_weak(n, n - 1)) {
    }
    return n > 0 ? 1 : 0;
}
thread_local std::string g_last_error;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

vw4_status cuda_fail(cudaError_t e, const char* where) {
    g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
    return VW4_ERR_CUDA;
}

vw4_status device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return VW4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        for (int f = 1; f <= 2; ++f) {
            d.occ[f][0] = gemm_blocks_per_sm(f, 8);
            d.occ[f][1] = gemm_blocks_per_sm(f, 16);
        }
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        d.status = static_cast<uint32_t*>(p);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || fn == nullptr || q != cudaDriverEntryPointSuccess)
                return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e,
                                 "cuTensorMapEncodeTiled entry point");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return VW4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D uint8 tensor map over a row-major [rows][inner_bytes] array.  Maps
// depend only on (address, shape, box, swizzle), so recent ones are cached
// to keep the per-call host cost small.
struct MapKey {
    const void* base;
    uint64_t inner, rows;
    uint32_t box_inner, box_rows, sw;
    bool operator==(const MapKey& o) const {
        return base == o.base && inner == o.inner && rows == o.rows &&
               box_inner == o.box_inner && box_rows == o.box_rows && sw == o.sw;
    }
};
constexpr int kMapCache = 64;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_next = 0;
std::mutex g_map_mu;

vw4_status make_map(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    const MapKey key{base, inner_bytes, rows, box_inner, box_rows, static_cast<uint32_t>(sw)};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        for (int i = 0; i < kMapCache; ++i)
            if (g_map_keys[i] == key) {
                *map = g_maps[i];
                return VW4_OK;
            }
    }
    cuuint64_t dims[2] = {inner_bytes, rows};
    cuuint64_t strides[1] = {inner_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[128];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
        g_last_error = buf;
        return VW4_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_map_keys[g_map_next] = key;
    g_maps[g_map_next] = *map;
    g_map_next = (g_map_next + 1) % kMapCache;
    return VW4_OK;
}

vw4_status check_weight(const vw4_weight* W) {
    if (!W || !W->q_dev || !W->scales_dev) return VW4_ERR_INVALID_ARG;
    if (W->fmt != VW4_FMT_NVFP4 && W->fmt != VW4_FMT_Q4_0) return VW4_ERR_INVALID_ARG;
    if (W->reserved != 0 || W->reserved_f != 0.0f) return VW4_ERR_INVALID_ARG;
    if (W->N < 1 || W->K < 1) return VW4_ERR_INVALID_ARG;
    const int blk = W->fmt == VW4_FMT_NVFP4 ? 16 : 32;
    if (W->K % blk != 0) return VW4_ERR_INVALID_ARG;
    if (W->fmt == VW4_FMT_Q4_0 && W->tensor_scale != 1.0f) return VW4_ERR_INVALID_ARG;
    if (!std::isfinite(W->tensor_scale)) return VW4_ERR_INVALID_ARG;
    if (!aligned16(W->q_dev) || !aligned16(W->scales_dev)) return VW4_ERR_ALIGN;
    return VW4_OK;
}

// K rounded up to whole 256-wide stages (the TMA path's row pitches).
int padded_k(int K) { return (K + kStageK - 1) / kStageK * kStageK; }

}  // namespace
}  // namespace vw4

using namespace vw4;

extern "C" {

VW4_API int vw4_version(void) { return 100; }

VW4_API int vw4_build_flags(void) { return kChecks ? VW4_BUILD_CHECKS : 0; }

VW4_API const char* vw4_status_str(vw4_status s) {
    switch (s) {
        case VW4_OK: return "ok";
        case VW4_ERR_INVALID_ARG: return "invalid argument";
        case VW4_ERR_UNSUPPORTED: return "unsupported";
        case VW4_ERR_ALIGN: return "misaligned pointer or leading dimension";
        case VW4_ERR_CUDA: return "CUDA error";
        case VW4_ERR_TIMEOUT: return "device wait timed out";
        case VW4_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

VW4_API const char* vw4_last_error_string(void) { return g_last_error.c_str(); }

VW4_API void vw4_set_wait_limit_ns(uint64_t ns) {
    g_wait_ns = ns == 0 ? 2000000000ull : static_cast<unsigned long long>(ns);
}

VW4_API void vw4_test_inject_stall(int calls) { g_stall_calls.store(calls > 0 ? calls : 0); }

VW4_API size_t vw4_workspace_bytes(int op, int a, int b, int c) {
    if (op == VW4_OP_GEMM) {
        const int M = a, N = b, K = c;
        if (M < 1 || M > kMaxVerifyRows || N < 1 || K < 16 || K % 16) return 0;
        // K not a multiple of 256: room for the weights padded to whole stages
        const int Kp = padded_k(K);
        return gemm_workspace_layout(nullptr, 1, N, Kp, kMaxGrid, 0, gemm_rows_for(M),
                                     Kp != K ? N : 0).bytes;
    }
    if (op == VW4_OP_MOE) {
        const int P = a, N = b, K = c;
        if (P < 1 || P > kMaxSeg || N < 1 || K < kStageK || K % kStageK) return 0;
        return gemm_workspace_layout(nullptr, P, N, K, kMaxGrid, P, 8).bytes;
    }
    if (op == VW4_OP_REJECTION) {
        if (a < 1 || b < 0 || b > 8 || c < 1) return 0;
        return rejection_workspace_bytes(a, b, c);
    }
    if (op == VW4_OP_REJECTION_TOPK) {
        if (a < 1 || b < 0 || b > 8 || c < 1 || c > 1024) return 0;
        return rejection_topk_workspace_bytes(a, b, c);
    }
    return 0;
}

// The verify GEMM launch behind verify_gemm_w4 and verify_greedy_w4 (greedy
// non-null: the fused argmax feeds the greedy accept in the same launch, and
// out_dev may be null).
struct GreedyArgs {
    const int32_t* drafts;
    int B, Kd;
    int32_t* tokens;
    int32_t* len;
};

static vw4_status gemm_entry(const vw4_weight* W, const void* A_dev, int M, int lda,
                             float* out_dev, int ldo, int32_t* row_argmax_dev, float* bmax_dev,
                             int ldb, const GreedyArgs* greedy, void* workspace_dev,
                             size_t ws_bytes, void* stream) {
    vw4_status st = check_weight(W);
    if (st != VW4_OK) return st;
    if (!A_dev || (!out_dev && !greedy)) return VW4_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxVerifyRows || lda < W->K || (out_dev && ldo < W->N))
        return VW4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A_dev) & 1u) || (reinterpret_cast<uintptr_t>(out_dev) & 3u) ||
        (reinterpret_cast<uintptr_t>(bmax_dev) & 3u))
        return VW4_ERR_ALIGN;
    if (!workspace_dev) return VW4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return VW4_ERR_ALIGN;
    const int N = W->N, K_true = W->K;
    // K not a multiple of 256: the weights are first copied, zero-padded, into
    // the workspace, and the stages run over the padded K
    const int K = padded_k(K_true);
    const bool pad = K != K_true;
    // 1..8 rows: one mma n-tile; 9..16: two n-tiles over the same weights
    const int nr = gemm_rows_for(M);
    GemmWorkspace ws = gemm_workspace_layout(workspace_dev, 1, N, K, kMaxGrid, 0, nr, pad ? N : 0);
    if (ws.bytes > ws_bytes) return VW4_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != VW4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const void* q_src = W->q_dev;
    const void* s_src = W->scales_dev;
    if (pad) {
        cudaError_t e = launch_pad_weights(W->q_dev, W->scales_dev, N, K_true, K, ws.wpad, ws.spad, s);
        if (e != cudaSuccess) return cuda_fail(e, "pad_weights launch");
        q_src = ws.wpad;
        s_src = ws.spad;
    }
    CUtensorMap tmW, tmS;
    const int sgroup = K / kStageK < kScaleGroup ? K / kStageK : kScaleGroup;
    st = make_map(&tmW, q_src, static_cast<uint64_t>(K) / 2, N, kStageK / 2, kTileRows,
                  CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != VW4_OK) return st;
    st = make_map(&tmS, s_src, static_cast<uint64_t>(K) / 16, N, 16 * sgroup, kTileRows,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != VW4_OK) return st;

    const int T = K / kStageK;
    const int n_tiles = (N + kTileRows - 1) / kTileRows;
    const long long U = static_cast<long long>(n_tiles) * T;
    long long G = static_cast<long long>(d->sms) * d->occ[W->fmt][nr == 16 ? 1 : 0];
    if (G > kMaxGrid) G = kMaxGrid;
    // When every tile fits in one wave, split each tile's stages into S
    // nearly equal parts, one CTA each (no CTA spans two tiles, and a part has
    // at least kMinUnitsPerCta stages so that few partials are combined).
    // Otherwise stream-K over all units balances the work exactly.
    int split = 0;
    if (n_tiles <= G) {
        long long S = G / n_tiles;
        long long S_cap = T / kMinUnitsPerCta;
        if (S_cap < 1) S_cap = 1;
        if (S > S_cap) S = S_cap;
        if (S > kMaxSplit) S = kMaxSplit;
        split = static_cast<int>(S);
        G = n_tiles * S;
    }
    if (G > U) G = U;
    // Up to kMaxClusterSplit parts (and no fused reduction): the parts of a
    // tile form one cluster and combine over distributed shared memory.
    const bool fused_argmax = row_argmax_dev != nullptr || greedy != nullptr;
    const bool clustered =
        split > 1 && split <= kMaxClusterSplit && !fused_argmax && bmax_dev == nullptr;

    cudaError_t e = launch_prep_act(static_cast<const uint16_t*>(A_dev), lda, K, W->fmt, M, 0, 1,
                                    1, ws, n_tiles * kConsumerWarps, s, nr, nullptr, 0, nullptr,
                                    nullptr, 0, 0, K_true);
    if (e != cudaSuccess) return cuda_fail(e, "prep_act launch");
    GemmParams p{};
    p.N = N;
    p.K = K;
    p.T = T;
    p.n_tiles = n_tiles;
    p.sgroup = sgroup;
    p.split = split;
    p.tensor_scale = W->tensor_scale;
    p.seg = ws.seg;
    p.act = ws.act;
    p.out = out_dev;
    p.out_rows = M;
    p.ldo = ldo;
    p.dense_M = M;
    p.argmax_M = fused_argmax ? M : 0;
    p.partials = ws.partials;
    p.tile_cnt = ws.tile_cnt;
    p.am_key = ws.am_key;
    p.am_cnt = ws.am_cnt;
    p.row_argmax = row_argmax_dev;
    p.bmax = bmax_dev;
    p.ldb = ldb;
    p.status = d->status;
    p.wait_ns = g_wait_ns;
    p.cluster = clustered ? 1 : 0;
    p.stall_test = take_stall();
    if (greedy) {
        p.greedy_B = greedy->B;
        p.greedy_Kd = greedy->Kd;
        p.drafts = greedy->drafts;
        p.tokens = greedy->tokens;
        p.len = greedy->len;
    }
    e = launch_gemm(W->fmt, nr, tmW, tmS, p, static_cast<int>(G), clustered ? split : 1, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return VW4_OK;
}

VW4_API vw4_status verify_gemm_w4(const vw4_weight* W, const void* A_dev, int M, int lda,
                                  float* out_dev, int ldo, int32_t* row_argmax_dev,
                                  void* workspace_dev, size_t ws_bytes, void* stream) {
    return gemm_entry(W, A_dev, M, lda, out_dev, ldo, row_argmax_dev, nullptr, 0, nullptr,
                      workspace_dev, ws_bytes, stream);
}

VW4_API vw4_status verify_gemm_w4_blockmax(const vw4_weight* W, const void* A_dev, int M,
                                           int lda, float* out_dev, int ldo, float* block_max_dev,
                                           void* workspace_dev, size_t ws_bytes, void* stream) {
    if (!block_max_dev || !out_dev || !W || W->N < 1) return VW4_ERR_INVALID_ARG;
    return gemm_entry(W, A_dev, M, lda, out_dev, ldo, nullptr, block_max_dev,
                      (W->N + kBlockMaxRows - 1) / kBlockMaxRows, nullptr, workspace_dev,
                      ws_bytes, stream);
}

VW4_API vw4_status verify_greedy_w4(const vw4_weight* W, const void* A_dev, int lda,
                                    const int32_t* drafts_dev, int B, int Kd, int32_t* tokens_dev,
                                    int32_t* len_dev, float* out_dev, int ldo,
                                    void* workspace_dev, size_t ws_bytes, void* stream) {
    if (B < 1 || Kd < 0 || B * (Kd + 1) > kMaxVerifyRows) return VW4_ERR_INVALID_ARG;
    if (!tokens_dev || !len_dev || (Kd > 0 && !drafts_dev)) return VW4_ERR_INVALID_ARG;
    const GreedyArgs g{drafts_dev, B, Kd, tokens_dev, len_dev};
    return gemm_entry(W, A_dev, B * (Kd + 1), lda, out_dev, ldo, nullptr, nullptr, 0, &g,
                      workspace_dev, ws_bytes, stream);
}

VW4_API vw4_status verify_moe_w4(const vw4_weight* experts, int E, const void* A_dev, int lda,
                                 int rows_are_pairs, const int32_t* expert_ids_dev,
                                 const float* gates_dev, int M, int topk, int combine,
                                 float* out_dev, int ldo, void* workspace_dev, size_t ws_bytes,
                                 void* stream) {
    vw4_status st = check_weight(experts);
    if (st != VW4_OK) return st;
    // the experts are streamed in place: their rows need whole 256-wide stages
    if (experts->K % kStageK != 0) return VW4_ERR_UNSUPPORTED;
    if (E < 1 || !A_dev || !expert_ids_dev || !out_dev) return VW4_ERR_INVALID_ARG;
    if (combine && !gates_dev) return VW4_ERR_INVALID_ARG;
    if (M < 1 || M > kMaxVerifyRows || topk < 1 || topk > kMaxRows || M * topk > kMaxSeg)
        return VW4_ERR_INVALID_ARG;
    if ((rows_are_pairs != 0 && rows_are_pairs != 1) || (combine != 0 && combine != 1))
        return VW4_ERR_INVALID_ARG;
    const int N = experts->N, K = experts->K;
    if (static_cast<long long>(E) * N > 0x7fffffffLL) return VW4_ERR_INVALID_ARG;
    if (lda < K || ldo < N) return VW4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A_dev) & 1u) || (reinterpret_cast<uintptr_t>(out_dev) & 3u))
        return VW4_ERR_ALIGN;
    if (!workspace_dev) return VW4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return VW4_ERR_ALIGN;
    const int P = M * topk;
    GemmWorkspace ws = gemm_workspace_layout(workspace_dev, P, N, K, kMaxGrid, P, 8);
    if (ws.bytes > ws_bytes) return VW4_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != VW4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    CUtensorMap tmW, tmS;
    const uint64_t rows = static_cast<uint64_t>(E) * N;
    const int sgroup = K / kStageK < kScaleGroup ? K / kStageK : kScaleGroup;
    st = make_map(&tmW, experts->q_dev, static_cast<uint64_t>(K) / 2, rows, kStageK / 2,
                  kTileRows, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != VW4_OK) return st;
    st = make_map(&tmS, experts->scales_dev, static_cast<uint64_t>(K) / 16, rows, 16 * sgroup, kTileRows,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != VW4_OK) return st;

    const int T = K / kStageK;
    const int n_tiles = (N + kTileRows - 1) / kTileRows;
    long long G = static_cast<long long>(d->sms) * d->occ[experts->fmt][0];
    if (G > kMaxGrid) G = kMaxGrid;
    const long long U_max = static_cast<long long>(P) * n_tiles * T;
    if (G > U_max) G = U_max;

    // the prep launch routes the pairs as well
    cudaError_t e = launch_prep_act(static_cast<const uint16_t*>(A_dev), lda, K, experts->fmt, 0,
                                    rows_are_pairs, topk, P, ws, P * n_tiles * kConsumerWarps, s,
                                    8, expert_ids_dev, E, d->status, combine ? nullptr : out_dev, ldo,
                                    N);
    if (e != cudaSuccess) return cuda_fail(e, "prep_act launch");
    GemmParams p{};
    p.N = N;
    p.K = K;
    p.T = T;
    p.n_tiles = n_tiles;
    p.sgroup = sgroup;
    p.tensor_scale = experts->tensor_scale;
    p.seg = ws.seg;
    p.act = ws.act;
    p.out = combine ? ws.pair_out : out_dev;
    p.out_rows = P;
    p.ldo = combine ? N : ldo;
    p.dense_M = 0;
    p.argmax_M = 0;
    // whole tiles per CTA: a segment's tiles are short (an expert's rows),
    // and splitting them across CTAs costs more than the imbalance
    p.split = -1;
    p.partials = ws.partials;
    p.tile_cnt = ws.tile_cnt;
    p.am_key = ws.am_key;
    p.am_cnt = ws.am_cnt;
    p.row_argmax = nullptr;
    p.status = d->status;
    p.wait_ns = g_wait_ns;
    p.stall_test = take_stall();
    e = launch_gemm(experts->fmt, 8, tmW, tmS, p, static_cast<int>(G), 1, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    if (combine) {
        e = launch_combine(ws.pair_out, gates_dev, expert_ids_dev, E, M, topk, N, out_dev, ldo, s);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    }
    return VW4_OK;
}

VW4_API vw4_status accept_greedy(const float* target_logits_dev, const int32_t* drafts_dev,
                                 const int32_t* target_argmax_dev, int B, int Kd, int V,
                                 int32_t* tokens_dev, int32_t* len_dev, void* stream) {
    if (B < 1 || Kd < 0 || Kd > kMaxRows || V < 1) return VW4_ERR_INVALID_ARG;
    if (!tokens_dev || !len_dev) return VW4_ERR_INVALID_ARG;
    if (Kd > 0 && !drafts_dev) return VW4_ERR_INVALID_ARG;
    if (!target_argmax_dev && !target_logits_dev) return VW4_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * (Kd + 1) * 8 > 0x7fffffffLL) return VW4_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    vw4_status st = device_info(&d);
    if (st != VW4_OK) return st;
    cudaError_t e = launch_accept_greedy(target_logits_dev, drafts_dev, target_argmax_dev, B, Kd,
                                         V, tokens_dev, len_dev, d->status,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "accept_greedy launch");
    return VW4_OK;
}

static vw4_status rejection_entry(const float* target_logits_dev, const float* target_bmax_dev,
                                  const float* draft_logits_dev, const float* draft_bmax_dev,
                                  const int32_t* drafts_dev, int B, int Kd, int V,
                                  const vw4_sampling* params, uint64_t seed, uint64_t offset,
                                  int32_t* tokens_dev, int32_t* len_dev, void* workspace_dev,
                                  size_t ws_bytes, void* stream) {
    if (!params || !target_logits_dev || !tokens_dev || !len_dev) return VW4_ERR_INVALID_ARG;
    if (B < 1 || Kd < 0 || Kd > kMaxRows || V < 1 || V > (1 << 24)) return VW4_ERR_INVALID_ARG;
    if (Kd > 0 && (!drafts_dev || !draft_logits_dev)) return VW4_ERR_INVALID_ARG;
    const float T = params->temperature;
    if (!(T >= 0.0f) || !std::isfinite(T)) return VW4_ERR_INVALID_ARG;
    if (!(params->top_p > 0.0f) || !std::isfinite(params->top_p)) return VW4_ERR_INVALID_ARG;
    if (params->top_k < 0) return VW4_ERR_INVALID_ARG;
    if (!(params->min_p >= 0.0f && params->min_p <= 1.0f)) return VW4_ERR_INVALID_ARG;
    if (T == 0.0f)  // temperature 0 is the greedy rule: no random numbers drawn
        return accept_greedy(target_logits_dev, drafts_dev, nullptr, B, Kd, V, tokens_dev,
                             len_dev, stream);
    const size_t need = rejection_workspace_bytes(B, Kd, V);
    if (!workspace_dev || ws_bytes < need) return VW4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return VW4_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    vw4_status st = device_info(&d);
    if (st != VW4_OK) return st;
    const float invT = static_cast<float>(1.0 / static_cast<double>(T));
    const double pd = static_cast<double>(params->top_p) * 4294967296.0;
    uint64_t P = pd >= 4294967296.0 ? (1ull << 32) : static_cast<uint64_t>(std::llround(pd));
    if (P == 0) P = 1;  // keeps the top entry alone, exactly as P = 0 does
    // min-p in the same fixed point, 0 = off
    const double md = static_cast<double>(params->min_p) * 4294967296.0;
    const uint64_t MP = params->min_p > 0.0f
                            ? (md >= 4294967296.0 ? (1ull << 32)
                                                  : static_cast<uint64_t>(std::llround(md)))
                            : 0ull;
    cudaError_t e = launch_accept_rejection(target_logits_dev, draft_logits_dev, drafts_dev, B, Kd,
                                            V, invT, P, params->top_k, MP, seed, offset,
                                            tokens_dev, len_dev,
                                            workspace_dev, ws_bytes, d->status, g_wait_ns,
                                            static_cast<cudaStream_t>(stream), target_bmax_dev,
                                            Kd > 0 ? draft_bmax_dev : nullptr);
    if (e == cudaErrorNotSupported) return VW4_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e, "accept_rejection launch");
    return VW4_OK;
}

VW4_API vw4_status accept_rejection(const float* target_logits_dev, const float* draft_logits_dev,
                                    const int32_t* drafts_dev, int B, int Kd, int V,
                                    const vw4_sampling* params, uint64_t seed, uint64_t offset,
                                    int32_t* tokens_dev, int32_t* len_dev, void* workspace_dev,
                                    size_t ws_bytes, void* stream) {
    return rejection_entry(target_logits_dev, nullptr, draft_logits_dev, nullptr, drafts_dev, B,
                           Kd, V, params, seed, offset, tokens_dev, len_dev, workspace_dev,
                           ws_bytes, stream);
}

VW4_API vw4_status accept_rejection_blockmax(const float* target_logits_dev,
                                             const float* target_bmax_dev,
                                             const float* draft_logits_dev,
                                             const float* draft_bmax_dev,
                                             const int32_t* drafts_dev, int B, int Kd, int V,
                                             const vw4_sampling* params, uint64_t seed,
                                             uint64_t offset, int32_t* tokens_dev,
                                             int32_t* len_dev, void* workspace_dev,
                                             size_t ws_bytes, void* stream) {
    if (!target_bmax_dev || (Kd > 0 && !draft_bmax_dev)) return VW4_ERR_INVALID_ARG;
    return rejection_entry(target_logits_dev, target_bmax_dev, draft_logits_dev, draft_bmax_dev,
                           drafts_dev, B, Kd, V, params, seed, offset, tokens_dev, len_dev,
                           workspace_dev, ws_bytes, stream);
}

VW4_API vw4_status accept_rejection_topk(const int32_t* target_ids_dev,
                                         const float* target_vals_dev,
                                         const int32_t* draft_ids_dev, const float* draft_vals_dev,
                                         const int32_t* drafts_dev, int B, int Kd, int Kt, int V,
                                         const vw4_sampling* params, uint64_t seed,
                                         uint64_t offset, int32_t* tokens_dev, int32_t* len_dev,
                                         void* workspace_dev, size_t ws_bytes, void* stream) {
    if (!params || !target_ids_dev || !target_vals_dev || !tokens_dev || !len_dev)
        return VW4_ERR_INVALID_ARG;
    if (B < 1 || Kd < 0 || Kd > kMaxRows || V < 1 || V > (1 << 24) || Kt < 1)
        return VW4_ERR_INVALID_ARG;
    if (Kd > 0 && (!drafts_dev || !draft_ids_dev || !draft_vals_dev)) return VW4_ERR_INVALID_ARG;
    const float T = params->temperature;
    if (!(T >= 0.0f) || !std::isfinite(T)) return VW4_ERR_INVALID_ARG;
    if (!(params->top_p > 0.0f) || !std::isfinite(params->top_p)) return VW4_ERR_INVALID_ARG;
    if (params->top_k < 0) return VW4_ERR_INVALID_ARG;
    if (!(params->min_p >= 0.0f && params->min_p <= 1.0f)) return VW4_ERR_INVALID_ARG;
    if (T == 0.0f || Kt > 1024) return VW4_ERR_UNSUPPORTED;
    const size_t need = rejection_topk_workspace_bytes(B, Kd, Kt);
    if (!workspace_dev || ws_bytes < need) return VW4_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace_dev) & 255u) != 0) return VW4_ERR_ALIGN;
    DeviceInfo* d = nullptr;
    vw4_status st = device_info(&d);
    if (st != VW4_OK) return st;
    const float invT = static_cast<float>(1.0 / static_cast<double>(T));
    const double pd = static_cast<double>(params->top_p) * 4294967296.0;
    uint64_t P = pd >= 4294967296.0 ? (1ull << 32) : static_cast<uint64_t>(std::llround(pd));
    if (P == 0) P = 1;
    const double md = static_cast<double>(params->min_p) * 4294967296.0;
    const uint64_t MP = params->min_p > 0.0f
                            ? (md >= 4294967296.0 ? (1ull << 32)
                                                  : static_cast<uint64_t>(std::llround(md)))
                            : 0ull;
    cudaError_t e = launch_accept_rejection_topk(
        target_ids_dev, target_vals_dev, draft_ids_dev, draft_vals_dev, drafts_dev, B, Kd, Kt, V,
        invT, P, params->top_k, MP, seed, offset, tokens_dev, len_dev, workspace_dev, ws_bytes,
        d->status, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return VW4_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e, "accept_rejection_topk launch");
    return VW4_OK;
}

VW4_API vw4_status vw4_rejection_row_records(const void* workspace_dev, size_t ws_bytes, int B,
                                             int Kd, int V, vw4_row_record* records_dev,
                                             void* stream) {
    if (!workspace_dev || !records_dev) return VW4_ERR_INVALID_ARG;
    if (B < 1 || Kd < 0 || Kd > kMaxRows || V < 1 || V > (1 << 24)) return VW4_ERR_INVALID_ARG;
    if (ws_bytes < rejection_workspace_bytes(B, Kd, V)) return VW4_ERR_WORKSPACE;
    const long long rows = static_cast<long long>(B) * (2 * Kd + 1);
    cudaError_t e = copy_rejection_row_records(workspace_dev, rows, records_dev,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "row record copy");
    return VW4_OK;
}

VW4_API vw4_status vw4_get_device_status(uint32_t* bits, void* stream) {
    if (!bits) return VW4_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    vw4_status st = device_info(&d);
    if (st != VW4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpyFromSymbolAsync(&h, g_status_word, sizeof(h), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "read status");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    *bits |= h;
    return VW4_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free variant of verify_gemm_w4.
//
// Some callers cannot allocate device memory at the point where they need
// the verify GEMM: code running inside another framework's memory pool that
// forbids foreign allocations, a plugin handed only input and output
// pointers, or a path that must not call cudaMalloc because it would
// synchronize the device or fail under a capture.  For them this file keeps
// one fixed scratch array in device memory, reserved on every GPU that loads
// the library until the process exits.  The host only ever passes the
// array's device address, obtained once per device with
// cudaGetSymbolAddress while that device is current (the symbol itself is a
// host-side stand-in, not a device address).
// Every GPU has its own copy of the array.  Its size bounds the shapes this
// entry point accepts (the workspace of verify_gemm_w4 for that shape).
static constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kMaxDevices] = {};

extern "C" {

VW4_API vw4_status verify_gemm_w4_noalloc(const vw4_weight* W, const void* A_dev, int M, int lda,
                                          float* out_dev, int ldo, int32_t* row_argmax_dev,
                                          void* stream) {
    if (W && W->N >= 1 && W->K >= 16 && W->K % 16 == 0 && M >= 1 && M <= kMaxVerifyRows) {
        const int Kp = padded_k(W->K);
        const size_t need = gemm_workspace_layout(nullptr, 1, W->N, Kp, kMaxGrid, 0,
                                                  gemm_rows_for(M), Kp != W->K ? W->N : 0)
                                .bytes;
        if (need > kNoAllocScratchBytes) {
            char buf[160];
            snprintf(buf, sizeof buf,
                     "verify_gemm_w4_noalloc: M=%d N=%d K=%d needs %zu scratch bytes, above the "
                     "fixed %zu",
                     M, W->N, W->K, need, kNoAllocScratchBytes);
            g_last_error = buf;
            return VW4_ERR_WORKSPACE;
        }
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return VW4_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (g_noalloc_ptr[dev] == nullptr) {  // first call on this device
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr)
                return cuda_fail(e == cudaSuccess ? cudaErrorInvalidSymbol : e,
                                 "cudaGetSymbolAddress(noalloc scratch)");
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return verify_gemm_w4(W, A_dev, M, lda, out_dev, ldo, row_argmax_dev, scratch,
                          kNoAllocScratchBytes, stream);
}

VW4_API vw4_status vw4_own_exp(const float* x_dev, float* y_dev, int64_t n, void* stream) {
    if (!x_dev || !y_dev || n < 0) return VW4_ERR_INVALID_ARG;
    if (n == 0) return VW4_OK;
    cudaError_t e = launch_own_exp(x_dev, y_dev, n, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "own_exp launch");
    return VW4_OK;
}

VW4_API vw4_status vw4_own_mass_pairs(const float* x_dev, uint64_t* W_dev, int64_t n,
                                      void* stream) {
    if (!x_dev || !W_dev || n < 0) return VW4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W_dev) & 7u) != 0) return VW4_ERR_ALIGN;
    if (n == 0) return VW4_OK;
    cudaError_t e = launch_own_mass_pairs(x_dev, reinterpret_cast<unsigned long long*>(W_dev), n,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "own_mass_pairs launch");
    return VW4_OK;
}

VW4_API vw4_status vw4_q4_0_from_blocks(const void* blocks_dev, int N, int K, void* q_dev,
                                        void* d_dev, void* stream) {
    if (!blocks_dev || !q_dev || !d_dev || N < 1 || K < 32 || K % 32) return VW4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_dev) & 1u) != 0) return VW4_ERR_ALIGN;
    cudaError_t e = launch_q4_0_split(static_cast<const uint8_t*>(blocks_dev), N, K,
                                      static_cast<uint8_t*>(q_dev), static_cast<__half*>(d_dev),
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "q4_0 split launch");
    return VW4_OK;
}

}  // extern "C"
