// controller.cpp -- the draft-depth controller (host code).
//
// Ollama's mtp.go commit log (the paragraph replacing the heuristic draft
// schedule) drafts the depth that maximizes committed tokens per wall-clock
// time, from live per-position acceptance and the persisted forward cost of
// each verify width.  "Faster Gemma 4 on MLX with multi-token prediction"
// adds that drafting falls back when it does not pay.  Depth 0 is plain
// decoding here: one verify row, nothing drafted.
//
// Acceptance at position i is the probability that draft i is accepted given
// drafts 0..i-1 were.  It is estimated from decayed counts with one
// pseudo-acceptance and one pseudo-rejection (a uniform prior), so that
// positions not tried yet read as 1/2.
#include <cmath>

#include "vw4.h"

namespace {

constexpr int kMaxDepth = 15;  // verify rows K + 1 <= 16, the verify GEMM's widest call
constexpr int kPositions = kMaxDepth + 1;

bool valid(const vw4_depth_ctl* c) {
    if (c == nullptr || c->k_max < 0 || c->k_max > kMaxDepth) return false;
    if (!(c->decay > 0.0f && c->decay <= 1.0f)) return false;
    for (int w = 1; w <= c->k_max + 1; ++w)
        if (!(c->verify_us[w] > 0.0f) || !std::isfinite(c->verify_us[w])) return false;
    return c->draft_us_fixed >= 0.0f && c->draft_us_per_token >= 0.0f &&
           std::isfinite(c->draft_us_fixed) && std::isfinite(c->draft_us_per_token);
}

double alpha(const vw4_depth_ctl* c, int i) { return (c->acc[i] + 1.0) / (c->att[i] + 2.0); }

}  // namespace

extern "C" {

VW4_API vw4_status vw4_depth_ctl_init(vw4_depth_ctl* c, int k_max, float decay) {
    if (c == nullptr || k_max < 0 || k_max > kMaxDepth || !(decay > 0.0f && decay <= 1.0f))
        return VW4_ERR_INVALID_ARG;
    for (int i = 0; i < kPositions; ++i) c->att[i] = c->acc[i] = 0.0;
    for (int w = 0; w <= kPositions; ++w) c->verify_us[w] = 1.0f;
    c->draft_us_fixed = 0.0f;
    c->draft_us_per_token = 0.0f;
    c->k_max = k_max;
    c->decay = decay;
    return VW4_OK;
}

VW4_API vw4_status vw4_depth_ctl_observe(vw4_depth_ctl* c, int depth, int accepted) {
    if (!valid(c) || depth < 0 || depth > c->k_max || accepted < 0 || accepted > depth)
        return VW4_ERR_INVALID_ARG;
    for (int i = 0; i < kPositions; ++i) {
        c->att[i] *= c->decay;
        c->acc[i] *= c->decay;
    }
    // positions 0..accepted-1 were accepted; position `accepted` (if drafted)
    // was tried and rejected; nothing is known past it
    for (int i = 0; i < accepted; ++i) {
        c->att[i] += 1.0;
        c->acc[i] += 1.0;
    }
    if (accepted < depth) c->att[accepted] += 1.0;
    return VW4_OK;
}

VW4_API vw4_status vw4_depth_ctl_expected(const vw4_depth_ctl* c, int depth, double* tokens,
                                          double* us) {
    if (!valid(c) || depth < 0 || depth > c->k_max || tokens == nullptr || us == nullptr)
        return VW4_ERR_INVALID_ARG;
    double run = 0.0, reach = 1.0;  // reach: probability that position j is reached
    for (int j = 0; j <= depth; ++j) {
        run += reach;
        if (j < depth) reach *= alpha(c, j);
    }
    *tokens = run;
    *us = static_cast<double>(c->verify_us[depth + 1]) +
          (depth > 0 ? static_cast<double>(c->draft_us_fixed) +
                           depth * static_cast<double>(c->draft_us_per_token)
                     : 0.0);
    return VW4_OK;
}

VW4_API int vw4_depth_ctl_choose(const vw4_depth_ctl* c) {
    if (!valid(c)) return -1;
    int best = 0;
    double best_rate = -1.0;
    for (int k = 0; k <= c->k_max; ++k) {
        double t = 0.0, us = 0.0;
        vw4_depth_ctl_expected(c, k, &t, &us);
        const double rate = t / us;
        if (rate > best_rate) {  // strict: ties keep the shallower depth
            best_rate = rate;
            best = k;
        }
    }
    return best;
}

}  // extern "C"
