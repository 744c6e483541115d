// Internal declarations of the float MoE layer (com.microsoft.MoE README):
// the validated problem, the workspace plan and the kernel launchers.
#pragma once

#include "moe.h"
#include "qmoe_internal.h"

namespace qmoe {

struct FProblem {
    int64_t T = 0, H = 0, I = 0, E = 0, k = 0;
    int act = MOE_ACT_RELU;
    int swiglu_fusion = 0;   // README Attributes.swiglu_fusion
    int64_t rows1 = 0;       // FC1 rows per expert: 2I for fused SwiGLU, else I
    int paired = 0;          // the activation reads two projections (SwiGLU, or SiLU x FC3)
    float alpha = 1.f, beta = 0.f;
    int has_limit = 0;
    float limit = 0.f;
    int normalize = 0;
    int path = MOE_PATH_GENERIC;
    const float* x = nullptr;
    const float* logits = nullptr;
    const float *w1 = nullptr, *b1 = nullptr, *w2 = nullptr, *b2 = nullptr;
    const float *w3 = nullptr, *b3 = nullptr;
    float* y = nullptr;
};

struct FPlan {
    int64_t slots = 0, route_chunks = 0, max_tiles = 0, srows = 0;
    int tile_tokens = 0;     // grouped path: rows per token tile (256)
    int bmax = 0;            // grouped path: token rows one stage holds (<= 256)
    int fc2_splits = 1;      // grouped path: split-K factor of FC2
    size_t bytes = 0;
    size_t off_ctrl, off_sel, off_pw, off_counts, off_offsets, off_hist, off_rank, off_perm,
        off_inv, off_tiles, off_active, off_xs, off_act, off_slot_out;
};

struct FWork {
    int32_t *ctrl, *sel, *counts, *offsets, *hist, *rank, *perm, *inv, *tiles, *active;
    float* pw;
    float* xs;         // grouped: tf32 activations, expert-sorted, K-blocked [H/32][srows][32]
    float* act;        // generic: [slots, I] sorted order; grouped: K-blocked [I/32][srows][32]
    float* slot_out;   // [splits][slots][H] FC2 rows by original slot (bias included)
};

constexpr int kFTileTokens = 256;

bool moe_grouped_shape_ok(const FProblem& p);
int moe_cta_group(const FPlan& pl);
int moe_fc2_splits(const FProblem& p, int64_t slots, int cta);
cudaError_t launch_moe_generic_fc1(const FProblem& p, const FPlan& pl, const FWork& w,
                                   cudaStream_t s);
cudaError_t launch_moe_generic_fc2(const FProblem& p, const FPlan& pl, const FWork& w,
                                   cudaStream_t s);
cudaError_t launch_moe_gather(const FProblem& p, const FPlan& pl, const FWork& w, cudaStream_t s);
cudaError_t launch_moe_grouped_fc(const FProblem& p, const FPlan& pl, const FWork& w, bool fc1,
                                  cudaStream_t s);

}  // namespace qmoe
