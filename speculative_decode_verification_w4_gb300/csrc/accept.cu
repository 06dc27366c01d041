// accept.cu -- the on-GPU accept step.
//
// Greedy ("Accelerating Gemini Nano models on Pixel with frozen Multi-Token
// Prediction", section 3; Qiita roofline article on MTP, PART 2 section 2-4;
// Ollama mtp.go commit log, "Greedy is a special case of sampled decoding"):
// the longest draft prefix equal to the target's own argmax is accepted and
// the target's token at the first mismatch (or the bonus token) is always
// committed.  Argmax ties go to the lowest index; NaN never wins.
//
// Row argmax: one thread-block cluster of 16 CTAs per logits row, each CTA
// scanning one sixteenth of the vocabulary; the partial maxima are combined
// through distributed shared memory, so no global scratch is needed.
#include <cooperative_groups.h>

#include "vw4_internal.cuh"

namespace cg = cooperative_groups;

namespace vw4 {

constexpr uint32_t kStatusBadDraft = 0x1u;
constexpr int kArgCluster = 16;  // a non-portable cluster size, opted into at launch
constexpr int kArgThreads = 512;

// (ordered value, ~index): larger key = larger value, then smaller index.
__device__ __forceinline__ unsigned long long greedy_key(float v, uint32_t idx) {
    if (v != v) v = -INFINITY;
    if (v == 0.0f) v = 0.0f;
    const uint32_t b = __float_as_uint(v);
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - idx);
}

__device__ __forceinline__ unsigned long long kmax(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

__global__ void __cluster_dims__(kArgCluster, 1, 1) __launch_bounds__(kArgThreads)
    row_argmax_kernel(const float* __restrict__ logits, long long V, int vec,
                      int32_t* __restrict__ out) {
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ unsigned long long s_warp[kArgThreads / 32];
    __shared__ unsigned long long s_key;
    const int rank = static_cast<int>(cluster.block_rank());
    const long long row = blockIdx.x / kArgCluster;
    const float* x = logits + row * V;
    unsigned long long best = 0ull;
    if (vec) {
        // 16-byte rows: float4 groups, eight loads in flight per thread; the
        // CTA's slice is a whole number of groups
        const long long V4 = V >> 2;
        const long long chunk = (V4 + kArgCluster - 1) / kArgCluster;
        const long long lo = rank * chunk;
        const long long hi = (lo + chunk < V4) ? lo + chunk : V4;
        const float4* x4 = reinterpret_cast<const float4*>(x);
        for (long long g0 = lo + threadIdx.x; g0 < hi; g0 += 8 * kArgThreads) {
            float4 a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const long long g = g0 + static_cast<long long>(j) * kArgThreads;
                a[j] = g < hi ? __ldg(x4 + g) : make_float4(NAN, NAN, NAN, NAN);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t v = static_cast<uint32_t>(4 * (g0 + static_cast<long long>(j) * kArgThreads));
                best = kmax(best, greedy_key(a[j].x, v));
                best = kmax(best, greedy_key(a[j].y, v + 1));
                best = kmax(best, greedy_key(a[j].z, v + 2));
                best = kmax(best, greedy_key(a[j].w, v + 3));
            }
        }
    } else {
        const long long chunk = (V + kArgCluster - 1) / kArgCluster;
        const long long lo = rank * chunk;
        const long long hi = (lo + chunk < V) ? lo + chunk : V;
        long long v = lo + threadIdx.x;
        for (; v + 3 * kArgThreads < hi; v += 4 * kArgThreads) {
            const float a0 = __ldg(x + v), a1 = __ldg(x + v + kArgThreads);
            const float a2 = __ldg(x + v + 2 * kArgThreads), a3 = __ldg(x + v + 3 * kArgThreads);
            best = kmax(best, greedy_key(a0, static_cast<uint32_t>(v)));
            best = kmax(best, greedy_key(a1, static_cast<uint32_t>(v + kArgThreads)));
            best = kmax(best, greedy_key(a2, static_cast<uint32_t>(v + 2 * kArgThreads)));
            best = kmax(best, greedy_key(a3, static_cast<uint32_t>(v + 3 * kArgThreads)));
        }
        for (; v < hi; v += kArgThreads)
            best = kmax(best, greedy_key(__ldg(x + v), static_cast<uint32_t>(v)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = kmax(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long k = 0ull;
        for (int w = 0; w < kArgThreads / 32; ++w) k = kmax(k, s_warp[w]);
        s_key = k;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        unsigned long long k = 0ull;
        for (int r = 0; r < kArgCluster; ++r) k = kmax(k, *cluster.map_shared_rank(&s_key, r));
        // an empty row slice contributes 0, which every real key exceeds
        out[row] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k));
    }
    cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

// One thread per sequence: longest agreeing prefix, then commit.
__global__ void greedy_finish_kernel(const int32_t* __restrict__ drafts,
                                     const int32_t* argmax /* [B][Kd+1], may alias tokens */,
                                     int B, int Kd, int V, int32_t* tokens, int32_t* len,
                                     uint32_t* status) {
    // launched early behind the argmax (or whatever precedes it); reads
    // nothing before that grid is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int32_t g[9];
    for (int i = 0; i <= Kd; ++i) g[i] = argmax[static_cast<long long>(b) * (Kd + 1) + i];
    int n = 0;
    bool bad = false;
    for (int i = 0; i < Kd; ++i) {
        const int32_t x = drafts[static_cast<long long>(b) * Kd + i];
        if (x < 0 || x >= V) {
            bad = true;
            break;
        }
        if (x != g[i]) break;
        ++n;
    }
    check(g[n] >= 0 && g[n] < V, status);  // the row argmax was found
    for (int i = 0; i <= Kd; ++i) {
        int32_t t = -1;
        if (i < n) t = drafts[static_cast<long long>(b) * Kd + i];
        else if (i == n) t = g[n];
        tokens[static_cast<long long>(b) * (Kd + 1) + i] = t;
    }
    len[b] = n + 1;
    if (bad) atomicOr(status, kStatusBadDraft);
}

cudaError_t launch_accept_greedy(const float* logits, const int32_t* drafts,
                                 const int32_t* argmax_in, int B, int Kd, int V, int32_t* tokens,
                                 int32_t* len, uint32_t* status, cudaStream_t s) {
    const int32_t* am = argmax_in;
    if (am == nullptr) {
        const long long rows = static_cast<long long>(B) * (Kd + 1);
        const int vec = (V % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0) ? 1 : 0;
        static std::atomic<unsigned long long> attr_once{0};
        cudaError_t ea = set_attribute_per_device(attr_once, [] {
            return cudaFuncSetAttribute(row_argmax_kernel,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        });
        if (ea != cudaSuccess) return ea;
        row_argmax_kernel<<<static_cast<unsigned>(rows * kArgCluster), kArgThreads, 0, s>>>(
            logits, V, vec, tokens);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        am = tokens;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((B + 127) / 128);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, greedy_finish_kernel, drafts, am, B, Kd, V, tokens, len, status);
}

}  // namespace vw4
