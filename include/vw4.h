/*
 * vw4.h -- C ABI of the GB300 (sm_103a) library for the hot path of
 * multi-token-prediction speculative decoding verification with 4-bit
 * weights: the skinny verify GEMM, its MoE expert-gather variant, and the
 * on-GPU accept step (greedy longest-prefix match; rejection sampling with
 * residual correction).
 *
 * Conventions for every entry point
 *  - Pointers named *_dev are device pointers owned by the caller; nothing is
 *    copied and nothing is freed.  The library never allocates device memory
 *    in a call: scratch comes from the caller's workspace (sized by
 *    vw4_workspace_bytes) or is not needed.
 *  - A workspace needs no initialization: every call sets up what it reads
 *    (the verify GEMM clears its own counters at the start of each launch),
 *    so one workspace, sized for the largest use, may serve every entry
 *    point, one call after another on the same stream.
 *  - `stream` is a cudaStream_t (0 = the legacy default stream).  Every call
 *    is asynchronous on it; no call synchronizes except vw4_get_device_status.
 *  - Argument errors are detected on the host, before anything is launched,
 *    and returned as a vw4_status; nothing is written in that case.  A launch
 *    failure returns VW4_ERR_CUDA (the CUDA error string is available from
 *    vw4_last_error_string).  Conditions that only the device can see (an
 *    out-of-range draft id, an expert id out of range, a pipeline wait that
 *    ran out) set bits of a device status word that vw4_get_device_status
 *    reads and clears; kernels never trap.
 *  - Alignment: weight and scale base pointers must be 16-byte aligned (they
 *    are read by TMA); activations and outputs need only their natural
 *    alignment; lda and ldo are counted in elements.
 *
 * Formats (the pages name nvfp4 and Q4 without defining the bits; these are
 * the standard definitions):
 *  - nvfp4: q = u8 [N][K/2], element k of a row in byte k/2, the even element
 *    in the LOW nibble; each nibble is FP4 E2M1 (OCP MX v1.0: s e1 e0 m).
 *    scales = E4M3 (OCP fp8 "fn") [N][K/16], one per 16 consecutive k of a
 *    row; tensor_scale = one fp32 factor for the whole matrix.
 *    w[n][k] = e2m1(nibble) * e4m3(scale[n][k/16]) * tensor_scale.
 *  - Q4_0: q = u8 [N][K/2] and scales = fp16 [N][K/32] (one per 32-element
 *    block); in block b of a row, byte j (0..15) of the block holds element
 *    32b+j in its low nibble and element 32b+j+16 in its high nibble.
 *    w[n][k] = (nibble - 8) * scale[n][k/32].  tensor_scale must be 1.
 *  - Activations are bf16 [M][lda] row-major; outputs fp32 [rows][ldo].
 */
#ifndef VW4_H
#define VW4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define VW4_API __declspec(dllexport)
#else
#define VW4_API __attribute__((visibility("default")))
#endif

typedef enum { VW4_FMT_NVFP4 = 1, VW4_FMT_Q4_0 = 2 } vw4_fmt;

typedef enum {
    VW4_OK = 0,
    VW4_ERR_INVALID_ARG = 1,   /* null pointer, size or enum out of range       */
    VW4_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement  */
    VW4_ERR_ALIGN = 3,         /* a pointer or leading dimension is misaligned  */
    VW4_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed             */
    VW4_ERR_TIMEOUT = 5,       /* reported by vw4_get_device_status bits only   */
    VW4_ERR_WORKSPACE = 6      /* workspace missing or smaller than required    */
} vw4_status;

/* Bits of the device status word (vw4_get_device_status). */
#define VW4_DEV_BAD_DRAFT_ID   0x1u  /* a draft id outside [0, V): treated as a rejection */
#define VW4_DEV_BAD_EXPERT_ID  0x2u  /* an expert id outside [0, E): that pair is skipped  */
#define VW4_DEV_WAIT_TIMEOUT   0x4u  /* a pipeline wait gave up; outputs are incomplete    */
#define VW4_DEV_ZERO_RESIDUAL  0x8u  /* a forced rejection met p == q: drew from p instead */
#define VW4_DEV_BAD_LIST_ID    0x10u /* a top-k list id outside [0, V): entry dropped      */
#define VW4_DEV_BOUNDS         0x20u /* checks build only: an index that came from data was
                                        out of range (a library bug): a memory access it
                                        addressed was skipped; a token id is still written */

/* A block-quantized weight matrix [N][K] (see the format notes above). */
typedef struct vw4_weight {
    int32_t fmt;            /* vw4_fmt                                         */
    int32_t N;              /* output features (rows of the stored matrix)     */
    int32_t K;              /* reduction length (K % 16 == 0 nvfp4, % 32 Q4_0) */
    int32_t reserved;       /* must be 0                                       */
    const void* q_dev;      /* packed nibbles, u8 [N][K/2]                     */
    const void* scales_dev; /* nvfp4: e4m3 [N][K/16]; Q4_0: fp16 [N][K/32]     */
    float tensor_scale;     /* nvfp4 global factor; exactly 1.0f for Q4_0      */
    float reserved_f;       /* must be 0                                       */
} vw4_weight;

/* Sampling parameters of the accept step. */
typedef struct vw4_sampling {
    float temperature;      /* 0 routes to the greedy rule (no random numbers)  */
    float top_p;            /* (0, 1]; >= 1 keeps the whole vocabulary         */
    int32_t top_k;          /* 0 = off; >= V keeps everything; < 0 invalid      */
    float min_p;            /* 0 = off; in [0, 1]                               */
} vw4_sampling;

/* Operation ids for vw4_workspace_bytes. */
#define VW4_OP_GEMM       1
#define VW4_OP_MOE        2
#define VW4_OP_REJECTION  3
#define VW4_OP_REJECTION_TOPK 4

/*
 * verify_gemm_w4 -- the verification pass's skinny matmul.
 *
 * Defined by: "Faster Gemma 4 on MLX with multi-token prediction", the
 * paragraph on where verification time goes: a verify batch of usually 2 to 8
 * token rows multiplied by block-quantized (nvfp4) weights, each weight block
 * read and unpacked once and reused across the batch, with computation
 * identical to the per-row product; and the Qiita roofline article on MTP in
 * llama.cpp, PART 2 section 2-3 (verify turns the matrix-vector product into a
 * thin matrix product over the same weight bytes).
 *
 *   out[m][n] = sum_k A[m][k] * w[n][k]       m < M, n < N        (fp32 result)
 *
 * W           weight descriptor (host pointer to the struct; device data).
 * A_dev       bf16 [M][lda], lda >= K.
 * M           1..16 verify rows.  Up to 8 rows take one mma n-tile; 9..16
 *             take two that share every unpacked weight fragment (wider
 *             batches, as in the batched head forward of Ollama's mtp.go
 *             commit log, where per-token cost falls as the batch grows):
 *             each weight block is still read and unpacked once per call.
 * out_dev     fp32 [M][ldo], ldo >= N.
 * row_argmax_dev  optional (NULL = skip): int32 [M]; row m receives the index
 *             of its largest output (ties to the lowest index; NaN never
 *             wins), computed in the same launch from the fp32 results.
 * workspace_dev / ws_bytes  scratch of at least
 *             vw4_workspace_bytes(VW4_OP_GEMM, M, N, K) bytes, 256-byte
 *             aligned, reused freely between calls on the same stream.
 * Error behaviour: VW4_ERR_INVALID_ARG for null pointers, M outside 1..16,
 * N < 1, K not a positive multiple of the block, lda < K, ldo < N;
 * K a multiple of the block but not of 256 is accepted on a slower path: the
 * weights are streamed by TMA tensor copies in 256-wide k stages, whose row
 * pitches (K/2 and K/16 bytes) must be multiples of 16, so such a call first
 * copies the weights and scales, zero-padded to whole stages, into the
 * workspace (vw4_workspace_bytes counts the room) and reads them twice;
 * every K of the dense-layer, LM-head and MoE configurations is a multiple
 * of 256;
 * VW4_ERR_ALIGN for misaligned pointers or leading dimensions;
 * VW4_ERR_WORKSPACE when the workspace is too small.
 *
 * Precision.  Products of the unpacked weights (exact in fp16) with the
 * activations are accumulated in fp32 on the tensor cores.  The activations
 * enter as fp16 after an exact power-of-two scaling per verify row and
 * 256-wide k stage, chosen so that the stage's largest magnitude amax lies in
 * [2^14, 2^15).  An activation is carried exactly when it is zero or at least
 * 2^-31 * amax in magnitude (every bf16 value down to that ratio fits fp16's
 * range and 11-bit significand); a smaller one is rounded to a multiple of at
 * most 2^-39 * amax.  So every output satisfies
 *   |out - exact| <= 1e-3 * sum_k |a_k w_k| + 2^-39 * sum_k amax(k) * |w_k|,
 * amax(k) the largest |a| of the row in the stage of k; the second term is
 * zero unless a stage mixes activations more than 2^31 apart.
 */
VW4_API vw4_status verify_gemm_w4(const vw4_weight* W, const void* A_dev, int M, int lda,
                                  float* out_dev, int ldo, int32_t* row_argmax_dev,
                                  void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * verify_gemm_w4_blockmax -- verify_gemm_w4 that also hands the logits' block
 * maxima to the sampled accept.
 *
 * Defined by: "Faster Gemma 4 on MLX with multi-token prediction" (drafting,
 * sampling and verification run on the GPU as one pass, with no return to
 * the CPU) and Ollama's mtp.go commit log paragraph "rework the MLX sampler"
 * (the acceptance, residual and bonus draws reuse the target distribution):
 * the verify GEMM already holds every logit of a row in registers, so it
 * writes the row's maximum over every 16 consecutive outputs next to the
 * logits, and accept_rejection_blockmax takes the row max and its segment
 * maxima from them instead of reading the full rows for them.
 *
 * W, A_dev, M, lda, out_dev, ldo, workspace  as verify_gemm_w4 (out_dev is
 *             required).
 * block_max_dev  fp32 [M][ceil(N / 16)]: element (m, j) = the largest of
 *             out[m][16 j .. min(16 j + 16, N)), NaN read as -infinity, +0
 *             over -0.  4-byte aligned.
 * Errors as verify_gemm_w4; VW4_ERR_INVALID_ARG when block_max_dev or out_dev
 * is NULL.
 */
VW4_API vw4_status verify_gemm_w4_blockmax(const vw4_weight* W, const void* A_dev, int M,
                                           int lda, float* out_dev, int ldo, float* block_max_dev,
                                           void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * verify_greedy_w4 -- the verify GEMM, its row argmax and the greedy accept
 * in one launch.
 *
 * Defined by: "Accelerating Gemini Nano models on Pixel with frozen
 * Multi-Token Prediction", section 3 (verify the drafted tokens in one pass,
 * keep the longest prefix the target agrees with, plus the target's own token
 * at the first disagreement) with the argmax taken over the verify GEMM's
 * fp32 outputs as verify_gemm_w4's row_argmax does, and Ollama's mtp.go
 * commit log paragraph "Greedy is a special case of sampled decoding".
 *
 * The GEMM runs over M = B * (Kd + 1) rows: row b (Kd + 1) + i of A is
 * sequence b's hidden state at verify position i.  The last warp of the
 * launch turns the row argmaxes into the committed run, exactly as
 * accept_greedy does with them: tokens[b][i] = drafts[b][i] for i < n, the
 * argmax of position n at i == n, -1 after; len[b] = n + 1, n the length of
 * the agreeing prefix.
 *
 * W, A_dev, lda   as verify_gemm_w4; B * (Kd + 1) must be 1..16.
 * drafts_dev      int32 [B][Kd] (may be NULL when Kd == 0).
 * tokens_dev      int32 [B][Kd + 1]; len_dev int32 [B].
 * out_dev, ldo    optional fp32 [M][ldo] logits; NULL = not written.
 * workspace_dev / ws_bytes  as verify_gemm_w4 for M rows.
 * Errors: as verify_gemm_w4, and VW4_ERR_INVALID_ARG for B < 1, Kd < 0,
 * B * (Kd + 1) > 16 or null outputs.  A draft id outside [0, N) ends the
 * prefix and sets VW4_DEV_BAD_DRAFT_ID in the device status word.
 */
VW4_API vw4_status verify_greedy_w4(const vw4_weight* W, const void* A_dev, int lda,
                                    const int32_t* drafts_dev, int B, int Kd, int32_t* tokens_dev,
                                    int32_t* len_dev, float* out_dev, int ldo,
                                    void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * verify_moe_w4 -- segmented expert-gather verify GEMM for MoE heads.
 *
 * Defined by: Ollama commit log for x/mlxrunner/mtp.go, paragraph on the
 * batched head forward (the segmented gather path for MoE heads), and the
 * Qiita article PART 3 section on expert scattering (verify rows route to
 * different experts, so each touched expert's weights are read once for the
 * rows that chose it).
 *
 * experts     weight descriptor of ALL experts stacked: N = rows per expert,
 *             q_dev = u8 [E][N][K/2], scales_dev = [E][N][K/16] (or /32).
 * E           number of experts.
 * A_dev, lda  bf16 activation rows: M token rows (rows_are_pairs == 0) or
 *             M*topk pair rows, pair p = m*topk + j (rows_are_pairs == 1).
 * expert_ids_dev  int32 [M][topk] routed experts, distinct within a token.
 * gates_dev   fp32 [M][topk] (read only when combine == 1).
 * M           1..16 tokens; topk 1..8 (at most 128 routed pairs).  The pairs
 *             of an expert are gathered into segments of up to 8 rows, each
 *             streaming the expert's weights once.
 * combine     0: out[p][n] for every pair p (out has M*topk rows);
 *             1: out[m][n] = sum_j gates[m][j] * pair(m, j)[n], j ascending.
 * Each touched expert streams its weights once for all its pair rows.
 * Error behaviour as verify_gemm_w4, except that K must be a multiple of 256
 * (VW4_ERR_UNSUPPORTED otherwise: the experts are streamed in place); an
 * expert id outside [0, E) sets
 * VW4_DEV_BAD_EXPERT_ID and that pair contributes zeros.
 */
VW4_API vw4_status verify_moe_w4(const vw4_weight* experts, int E, const void* A_dev, int lda,
                                 int rows_are_pairs, const int32_t* expert_ids_dev,
                                 const float* gates_dev, int M, int topk, int combine,
                                 float* out_dev, int ldo, void* workspace_dev, size_t ws_bytes,
                                 void* stream);

/*
 * accept_greedy -- longest-prefix argmax match.
 *
 * Defined by: "Accelerating Gemini Nano models on Pixel with frozen
 * Multi-Token Prediction", section 3 (the longest prefix matching what the
 * backbone itself would produce is accepted); the Qiita article PART 2
 * section 2-4 (the target's token at the first mismatch is always committed);
 * the mtp.go commit log paragraph "Greedy is a special case of sampled
 * decoding" (temperature 0 is a point mass, acceptance is argmax match).
 *
 * target_logits_dev  fp32 [B][Kd+1][V].  May be NULL when target_argmax_dev
 *             is given.
 * drafts_dev  int32 [B][Kd] drafted ids.
 * target_argmax_dev  optional int32 [B][Kd+1] precomputed argmaxes (e.g. the
 *             row_argmax of verify_gemm_w4); NULL = computed here from the
 *             logits (ties to the lowest index, NaN never wins).
 * B >= 1, 0 <= Kd <= 8, V >= 1.
 * tokens_dev  int32 [B][Kd+1]: drafts[0..n-1], then the target's token at
 *             position n, then -1; len_dev int32 [B] = n + 1 in [1, Kd+1].
 *             tokens_dev is also used as scratch inside the call.
 * An out-of-range draft id never matches and sets VW4_DEV_BAD_DRAFT_ID.
 */
VW4_API vw4_status accept_greedy(const float* target_logits_dev, const int32_t* drafts_dev,
                                 const int32_t* target_argmax_dev, int B, int Kd, int V,
                                 int32_t* tokens_dev, int32_t* len_dev, void* stream);

/*
 * accept_rejection -- rejection sampling with residual correction.
 *
 * Defined by: "Your model may already ship a speculative decoder", section
 * "Why it is interesting on a Mac specifically" (Leviathan and Chen rejection
 * sampling with residual correction reproduces plain decoding at temperature
 * 0.6, top_p 0.95); the mtp.go commit log paragraphs "Greedy is a special case
 * of sampled decoding" and "rework the MLX sampler" (pipeline
 * top-k -> temperature / softmax -> top-p -> min-p -> normalize -> categorical;
 * acceptance, residual and bonus draws reuse the same draft and target
 * distributions; seeded, reproducible).
 *
 * Exact integer form (identical on the oracle, so ids are bit-exact): each
 * row's weights W_v = floor(exp_own((l_v - max l) * (1/T)) * 2^40).  Top-k
 * keeps the first top_k entries in (logit desc, index asc) order (NaN reads
 * as -inf, -0 as +0); top-p then keeps the shortest prefix of the kept
 * entries in (W desc, index asc) order whose mass satisfies
 * cum * 2^32 >= round(top_p * 2^32) * sum W; min-p then keeps the entries with
 * W >= round(min_p * 2^32) * 2^8 (the top entry's W is 2^40).  Philox4x32-10
 * block for draft position i of sequence b: counter (i, b, offset lo,
 * offset hi), key = seed; U = r0 >> 8 decides acceptance
 * (U * q(x) * Sp < 2^24 * p(x) * Sq), and the 64-bit r2:r1 draws the residual
 * max(0, p*Sq - q*Sp) at the first rejection or the bonus from p_Kd
 * (block (Kd, b)) when all drafts are accepted.
 *
 * target_logits_dev  fp32 [B][Kd+1][V]; draft_logits_dev fp32 [B][Kd][V]
 *             (may be NULL when Kd == 0); drafts_dev int32 [B][Kd].
 * B >= 1, 0 <= Kd <= 8, 1 <= V <= 2^24 (rows are streamed from memory).
 * params      temperature >= 0 (0 = greedy rule, no random numbers drawn),
 *             top_p in (0, 1] (finite, values above 1 act as 1), top_k >= 0,
 *             min_p in [0, 1]; anything else is VW4_ERR_INVALID_ARG.
 * seed, offset  Philox key and counter offset.
 * tokens_dev, len_dev  as accept_greedy.
 * workspace_dev / ws_bytes  at least vw4_workspace_bytes(VW4_OP_REJECTION, B, Kd, V).
 */
VW4_API vw4_status accept_rejection(const float* target_logits_dev, const float* draft_logits_dev,
                                    const int32_t* drafts_dev, int B, int Kd, int V,
                                    const vw4_sampling* params, uint64_t seed, uint64_t offset,
                                    int32_t* tokens_dev, int32_t* len_dev, void* workspace_dev,
                                    size_t ws_bytes, void* stream);

/*
 * accept_rejection_blockmax -- accept_rejection fed by the verify GEMM's
 * block maxima.
 *
 * Defined by: the passages of accept_rejection, with the fusion of
 * verify_gemm_w4_blockmax ("Faster Gemma 4 on MLX with multi-token
 * prediction": sampling and verification in one pass on the GPU).
 *
 * The arguments of accept_rejection, plus the block maxima of every logits
 * row as verify_gemm_w4_blockmax writes them:
 * target_bmax_dev  fp32 [B][Kd+1][ceil(V / 16)];
 * draft_bmax_dev   fp32 [B][Kd][ceil(V / 16)] (NULL when Kd == 0).
 * The first pass of the accept, which reads every logit for the row max and
 * the maxima of its 128-entry segments, takes them from these arrays instead.
 * The committed ids and lengths are those of accept_rejection on the same
 * logits, for every row whose NaN entries (if any) lie elsewhere than at
 * index 0.  Errors as accept_rejection; VW4_ERR_INVALID_ARG for a NULL
 * block-max array that is needed.
 */
VW4_API vw4_status accept_rejection_blockmax(const float* target_logits_dev,
                                             const float* target_bmax_dev,
                                             const float* draft_logits_dev,
                                             const float* draft_bmax_dev,
                                             const int32_t* drafts_dev, int B, int Kd, int V,
                                             const vw4_sampling* params, uint64_t seed,
                                             uint64_t offset, int32_t* tokens_dev,
                                             int32_t* len_dev, void* workspace_dev,
                                             size_t ws_bytes, void* stream);

/*
 * accept_rejection_topk -- accept_rejection over rows kept as top-k lists.
 *
 * Defined by: Ollama's mtp.go commit log, paragraph "rework the MLX sampler"
 * (the top-k stage keeps [B, K] ids and probabilities on the device, and the
 * acceptance, bonus and residual draws reuse them), with the rule of
 * accept_rejection above.
 *
 * Each row is given as Kt (id, logit) pairs, in any order; every id not
 * listed reads as a logit of -infinity.  The committed ids and lengths are
 * exactly those of accept_rejection on dense rows holding the listed logits
 * and -infinity elsewhere, with the same params (params->top_k may cut the
 * lists further).  The accept reads Kt * 8 bytes per row instead of V * 4.
 *
 * target_ids_dev / target_vals_dev  int32 / fp32 [B][Kd+1][Kt].
 * draft_ids_dev / draft_vals_dev    int32 / fp32 [B][Kd][Kt] (NULL when Kd == 0).
 * drafts_dev  int32 [B][Kd].
 * B >= 1, 0 <= Kd <= 8, 1 <= V <= 2^24, 1 <= Kt <= 1024 (larger Kt:
 *             VW4_ERR_UNSUPPORTED).  The ids of a row must be distinct; an id
 *             outside [0, V) is dropped (read as -infinity) and sets
 *             VW4_DEV_BAD_LIST_ID.
 * params      as accept_rejection, except that temperature 0 returns
 *             VW4_ERR_UNSUPPORTED (the greedy rule needs no distribution:
 *             accept_greedy takes the argmax of each row, its first entry).
 * seed, offset, tokens_dev, len_dev  as accept_rejection.
 * workspace_dev / ws_bytes  at least
 *             vw4_workspace_bytes(VW4_OP_REJECTION_TOPK, B, Kd, Kt).
 */
VW4_API vw4_status accept_rejection_topk(const int32_t* target_ids_dev,
                                         const float* target_vals_dev,
                                         const int32_t* draft_ids_dev, const float* draft_vals_dev,
                                         const int32_t* drafts_dev, int B, int Kd, int Kt, int V,
                                         const vw4_sampling* params, uint64_t seed,
                                         uint64_t offset, int32_t* tokens_dev, int32_t* len_dev,
                                         void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * verify_gemm_w4_noalloc -- verify_gemm_w4 for callers that cannot allocate.
 *
 * No counterpart in the source material: this is a deployment convenience.
 * Some callers have no way to provide a workspace: a plugin that is handed
 * only its input and output pointers, code living in another framework's
 * memory pool that must not allocate outside it, or a path where calling
 * cudaMalloc would synchronize the device.  This entry point takes no
 * workspace and allocates nothing; it uses one fixed 16 MiB scratch array in
 * device memory that the library reserves on every GPU it is loaded on, for
 * as long as the process lives.
 *
 * Arguments, result and errors are those of verify_gemm_w4, plus:
 * VW4_ERR_WORKSPACE (with a message from vw4_last_error_string) when the
 * shape needs more scratch than the fixed array holds -- every verify shape of
 * the dense layer and LM-head configurations fits.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress); make that
 * first call before any stream capture.  Each GPU has its own array, and each
 * call resets the parts of it that must start at zero, but all calls on one
 * GPU share it: calls that can overlap there (on different streams, from
 * different threads) race on it, so serialize them.
 */
VW4_API vw4_status verify_gemm_w4_noalloc(const vw4_weight* W, const void* A_dev, int M, int lda,
                                          float* out_dev, int ldo, int32_t* row_argmax_dev,
                                          void* stream);

/*
 * One row record of accept_rejection, as its first kernel leaves it in the
 * workspace.  It describes the row's distribution after top-k, temperature /
 * softmax, top-p and min-p in the exact integer form above: with
 * W_v = floor(exp_own((l_v - max) * (1/T)) * 2^40) the mass of entry v before
 * any cut, entry v is kept iff it passes top-k (its logit key is above
 * topk_key, or equal and v <= topk_idx) and W_v > tau, or W_v == tau and
 * v <= cut; kept_sum is the sum of the kept masses.
 */
typedef struct vw4_row_record {
    float max;              /* the row max (scanned from index 0 with ">")     */
    int32_t cut;            /* largest kept index among the entries W == tau   */
    uint64_t tau;           /* the smallest kept mass                           */
    uint64_t kept_sum;      /* sum of the kept masses (S)                       */
    uint32_t topk_key;      /* top-k cut key (0 when top-k is off)              */
    int32_t topk_idx;       /* top-k cut index (INT32_MAX when top-k is off)    */
} vw4_row_record;

/*
 * vw4_rejection_row_records -- test hook: the row records of an
 * accept_rejection call.
 *
 * No counterpart in the source material: it exposes the per-row state of the
 * accept step so that every row can be compared with an independent
 * implementation, not only the ids the draws commit.
 *
 * workspace_dev / ws_bytes  the workspace of an accept_rejection call with
 *             the same B, Kd and V, after that call (stream order).
 * records_dev vw4_row_record [B * (2 Kd + 1)], device memory: the target rows
 *             (b, i) for i = 0..Kd in order, then the draft rows (b, i) for
 *             i < Kd.  Asynchronous on `stream` (a device-to-device copy).
 * Errors: VW4_ERR_INVALID_ARG for null pointers or sizes out of range,
 * VW4_ERR_WORKSPACE when ws_bytes is below what that call needed.
 */
VW4_API vw4_status vw4_rejection_row_records(const void* workspace_dev, size_t ws_bytes, int B,
                                             int Kd, int V, vw4_row_record* records_dev,
                                             void* stream);

/* Workspace bytes needed by an operation:
 *   VW4_OP_GEMM:      (M, N, K)
 *   VW4_OP_MOE:       (M*topk, N, K)   -- pass the number of routed pairs first
 *   VW4_OP_REJECTION: (B, Kd, V)
 *   VW4_OP_REJECTION_TOPK: (B, Kd, Kt)
 * Returns 0 for an unknown op or invalid sizes. */
VW4_API size_t vw4_workspace_bytes(int op, int a, int b, int c);

/* Reads the device status word of the current device, ORs it into *bits and
 * clears it.  Synchronizes `stream` first. */
VW4_API vw4_status vw4_get_device_status(uint32_t* bits, void* stream);

/* Converts Q4_0 blocks stored as 18-byte records (fp16 d, then 16 bytes of
 * nibbles) [N][K/32] into the split layout used here (q [N][K/2], d [N][K/32]).
 * Device pointers; asynchronous on `stream`. */
VW4_API vw4_status vw4_q4_0_from_blocks(const void* blocks_dev, int N, int K, void* q_dev,
                                        void* d_dev, void* stream);

/* The sampler's own fp32 exp, applied elementwise: y[i] = exp(x[i]) for x in
 * [-32, 0], 0 below -32 or for NaN.  This is the exact function the
 * accept_rejection masses use (a Cody-Waite reduction and a degree-7 Taylor
 * polynomial with explicit fmas), exposed so that it can be checked bit for
 * bit against an independent implementation.  Device pointers. */
VW4_API vw4_status vw4_own_exp(const float* x_dev, float* y_dev, int64_t n, void* stream);

/* The integer masses W[i] = floor(own_exp(x[i]) * 2^40) of scaled logits x,
 * computed by the packed fp32-pair arithmetic the row statistics use (two
 * entries per operation), exposed so that it can be checked against
 * vw4_own_exp and an independent implementation.  x: float [n]; W: uint64 [n]
 * (8-byte aligned).  Device pointers; asynchronous on `stream`.
 * VW4_ERR_INVALID_ARG for null pointers or n < 0; VW4_ERR_ALIGN for W. */
VW4_API vw4_status vw4_own_mass_pairs(const float* x_dev, uint64_t* W_dev, int64_t n,
                                      void* stream);

/*
 * Draft-depth controller (host only, no GPU work).
 *
 * Defined by: the Ollama commit log for x/mlxrunner/mtp.go, the paragraph that
 * replaces the heuristic draft schedule by an engine-level controller drafting
 * the depth that maximizes committed tokens per wall-clock time from live
 * per-position acceptance and the persisted forward cost of each verify width;
 * and "Faster Gemma 4 on MLX with multi-token prediction" (draft length tuned
 * at runtime from acceptance rates and verification pass times, falling back
 * when drafting does not pay).
 *
 * State (caller-owned; call vw4_depth_ctl_init before any other use: a
 * zero-filled state is invalid -- decay 0 and verify costs of 0 are rejected,
 * choose returns -1 and the others VW4_ERR_INVALID_ARG):
 *   att[i], acc[i]  decayed counts of drafts attempted / accepted at position
 *                   i, given drafts 0..i-1 were accepted (i < 16);
 *   verify_us[w]    the cost of a verify pass over w = K + 1 rows (1..16);
 *   draft_us_fixed, draft_us_per_token   the cost of drafting K > 0 tokens,
 *                   fixed + K * per_token;
 *   k_max           the deepest draft considered (0..15: the verify GEMM
 *                   takes M = K + 1 <= 16 rows);
 *   decay           weight kept by old observations at each new one (0..1].
 * The acceptance estimate of position i is (acc[i] + 1) / (att[i] + 2).  The
 * expected committed run of depth K is sum_{j=0..K} prod_{i<j} alpha_i (the
 * target's own token always commits), its cost verify_us[K + 1] plus the
 * drafting cost (none at K = 0, plain decoding).
 */
typedef struct vw4_depth_ctl {
    double att[16], acc[16];
    float verify_us[17];
    float draft_us_fixed, draft_us_per_token;
    int k_max;
    float decay;
} vw4_depth_ctl;

/* Resets the counts and sets the limits; verify costs default to 1 us each. */
VW4_API vw4_status vw4_depth_ctl_init(vw4_depth_ctl* c, int k_max, float decay);

/* Records one verify step: `depth` drafts were verified and the first
 * `accepted` of them were accepted (0 <= accepted <= depth <= k_max). */
VW4_API vw4_status vw4_depth_ctl_observe(vw4_depth_ctl* c, int depth, int accepted);

/* Expected committed tokens of a run at `depth` and its cost in us. */
VW4_API vw4_status vw4_depth_ctl_expected(const vw4_depth_ctl* c, int depth, double* tokens,
                                          double* us);

/* The depth in 0..k_max with the most expected committed tokens per us (ties
 * to the shallower depth); -1 for an invalid state. */
VW4_API int vw4_depth_ctl_choose(const vw4_depth_ctl* c);

/* Human-readable name of a status code (static string). */
VW4_API const char* vw4_status_str(vw4_status s);

/* Text of the last CUDA error seen by this thread in a library call. */
VW4_API const char* vw4_last_error_string(void);

/* Library version (major * 10000 + minor * 100 + patch). */
VW4_API int vw4_version(void);

/* How this copy of the library was built: VW4_BUILD_CHECKS is set in the
 * checks build (compiled with -DVW4_CHECKS, libvw4_checks.so), whose kernels
 * test the indexes that come from data -- the output row a MoE routing table
 * names, the activation row a segment reads, the token ids an accept commits
 * -- and report a failed test as VW4_DEV_BOUNDS: an out-of-range row is not
 * touched, an out-of-range token id is flagged.  Results are otherwise
 * identical to the plain build. */
#define VW4_BUILD_CHECKS 0x1
VW4_API int vw4_build_flags(void);

/* Test hook: upper bound, in nanoseconds, of every pipeline wait inside the
 * kernels (default 2e9).  A wait that runs out sets VW4_DEV_WAIT_TIMEOUT and
 * the kernel returns early with its copies drained.  0 restores the default. */
VW4_API void vw4_set_wait_limit_ns(uint64_t ns);

/* Test hook: the next `calls` verify GEMM launches of this process (through
 * verify_gemm_w4, verify_greedy_w4, verify_moe_w4 or the no-alloc variant)
 * make their consumer warps wait, before their first stage, on a pipeline
 * barrier that nothing ever completes, so that the bounded wait runs out: the
 * launch sets VW4_DEV_WAIT_TIMEOUT, lets its copies in flight land and returns
 * without writing its results.  0 cancels.  With vw4_set_wait_limit_ns it
 * exercises the timeout path without faulting or hanging the GPU. */
VW4_API void vw4_test_inject_stall(int calls);

#ifdef __cplusplus
}
#endif

#endif /* VW4_H */
