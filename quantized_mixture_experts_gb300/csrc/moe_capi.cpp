// Host side of the float MoE C ABI (com.microsoft.MoE README: Inputs,
// Outputs, Attributes, Type constraints): validation, workspace planning,
// path choice and kernel dispatch.  No device memory is allocated here.
#include <algorithm>
#include <cstring>

#include "moe_internal.h"

namespace qmoe {
namespace {

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Attribute checks and shape derivation from the input and FC1 weight shapes.
qmoe_status fderive(const int64_t* input_shape, int32_t input_rank, const int64_t* fc1_w_shape,
                    const moe_attrs* a, FProblem* p) {
    if (!input_shape || !fc1_w_shape || !a || !p) return QMOE_ERR_INVALID_ARGUMENT;
    if (a->use_sparse_mixer == 1) return QMOE_ERR_NOT_SUPPORTED;
    if (a->use_sparse_mixer != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (a->normalize_routing_weights != 0 && a->normalize_routing_weights != 1)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (a->activation_type < MOE_ACT_RELU || a->activation_type > MOE_ACT_IDENTITY)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (a->swiglu_fusion < 0 || a->swiglu_fusion > 2) return QMOE_ERR_INVALID_ARGUMENT;
    // a fused FC1 (interleaved or concatenated) exists only for SwiGLU
    if (a->swiglu_fusion != 0 && a->activation_type != MOE_ACT_SWIGLU)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (a->path != MOE_PATH_AUTO && a->path != MOE_PATH_GROUPED && a->path != MOE_PATH_GENERIC)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (input_rank != 2 && input_rank != 3) return QMOE_ERR_INVALID_ARGUMENT;
    int64_t T = 1;
    for (int d = 0; d < input_rank; ++d) {
        if (input_shape[d] < 0) return QMOE_ERR_INVALID_ARGUMENT;
        if (d < input_rank - 1) T *= input_shape[d];
    }
    const int64_t H = input_shape[input_rank - 1];
    if (H <= 0) return QMOE_ERR_INVALID_ARGUMENT;
    for (int d = 0; d < 3; ++d)
        if (fc1_w_shape[d] < 0) return QMOE_ERR_INVALID_ARGUMENT;
    p->T = T;
    p->H = H;
    p->E = fc1_w_shape[0];
    p->k = a->k;
    p->act = a->activation_type;
    p->swiglu_fusion = a->swiglu_fusion;
    const int fusion = (p->act == MOE_ACT_SWIGLU && p->swiglu_fusion != 0) ? 2 : 1;
    if (fc1_w_shape[1] % fusion != 0) return QMOE_ERR_INVALID_ARGUMENT;
    p->I = fc1_w_shape[1] / fusion;
    p->rows1 = fc1_w_shape[1];
    if (fc1_w_shape[2] != H) return QMOE_ERR_INVALID_ARGUMENT;
    if (p->E < 1 || p->k < 1 || p->k > p->E) return QMOE_ERR_INVALID_ARGUMENT;
    p->alpha = a->activation_alpha;
    p->beta = a->activation_beta;
    p->has_limit = a->has_swiglu_limit ? 1 : 0;
    p->limit = a->swiglu_limit;
    p->normalize = a->normalize_routing_weights;
    return QMOE_OK;
}

bool fpath_ok(const FProblem& p, int path) {
    if (path == MOE_PATH_GENERIC) return true;
    if (path == MOE_PATH_GROUPED) return moe_grouped_shape_ok(p);
    return false;
}

qmoe_status make_fplan(const FProblem& p, FPlan* out) {
    FPlan q;
    q.slots = p.T * p.k;
    q.route_chunks = (p.T + kRouteTokensPerChunk - 1) / kRouteTokensPerChunk;
    const bool grouped = p.path == MOE_PATH_GROUPED;
    q.tile_tokens = grouped ? kFTileTokens : 0;
    q.max_tiles = grouped ? (q.slots + kFTileTokens - 1) / kFTileTokens + p.E : 0;
    q.srows = grouped ? round_up(q.slots, 16) + 16 : 0;
    q.bmax = int(std::min<int64_t>(kFTileTokens, round_up(std::max<int64_t>(q.slots, 1), 16)));
    q.fc2_splits = grouped ? moe_fc2_splits(p, q.slots, moe_cta_group(q)) : 1;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + std::max<size_t>(bytes, 1), 256);
        return o;
    };
    const size_t slots = size_t(q.slots), E = size_t(p.E);
    q.off_ctrl = take(256);
    q.off_sel = take(4 * slots);
    q.off_pw = take(4 * slots);
    q.off_counts = take(4 * E);
    q.off_offsets = take(4 * (E + 1));
    q.off_hist = take(4 * size_t(q.route_chunks) * E);
    q.off_rank = take(4 * slots);
    q.off_perm = take(4 * slots);
    q.off_inv = take(4 * slots);
    q.off_tiles = take(4 * size_t(kTileHeader + 4 * q.max_tiles));
    q.off_active = take(4 * E);
    q.off_xs = take(grouped ? 4 * size_t(q.srows) * size_t(p.H) : 0);
    q.off_act = take(4 * (grouped ? size_t(q.srows) : slots) * size_t(p.I));
    q.off_slot_out = take(4 * size_t(q.fc2_splits) * slots * size_t(p.H));
    q.bytes = off;
    *out = q;
    return QMOE_OK;
}

qmoe_status fplan_for(const int64_t* input_shape, int32_t input_rank, const int64_t* fc1_w_shape,
                      const moe_attrs* attrs, FProblem* p, FPlan* pl) {
    qmoe_status st = fderive(input_shape, input_rank, fc1_w_shape, attrs, p);
    if (st != QMOE_OK) return st;
    if (attrs->path == MOE_PATH_AUTO)
        p->path = fpath_ok(*p, MOE_PATH_GROUPED) ? MOE_PATH_GROUPED : MOE_PATH_GENERIC;
    else
        p->path = attrs->path;
    if (!fpath_ok(*p, p->path)) return QMOE_ERR_NOT_SUPPORTED;
    return make_fplan(*p, pl);
}

// Remaining shape and presence checks of the README Inputs table.
qmoe_status fcheck(FProblem& p, const int64_t* router_shape, const int64_t* fc2_w_shape,
                   const int64_t* fc3_w_shape, const float* fc3_w) {
    if (!router_shape || !fc2_w_shape) return QMOE_ERR_INVALID_ARGUMENT;
    if (router_shape[0] != p.T || router_shape[1] != p.E) return QMOE_ERR_INVALID_ARGUMENT;
    if (fc2_w_shape[0] != p.E || fc2_w_shape[1] != p.H || fc2_w_shape[2] != p.I)
        return QMOE_ERR_INVALID_ARGUMENT;
    const bool has_fc3 = fc3_w != nullptr || fc3_w_shape != nullptr;
    if (has_fc3) {
        if (!fc3_w_shape) return QMOE_ERR_INVALID_ARGUMENT;
        if (fc3_w_shape[0] != p.E || fc3_w_shape[1] != p.I || fc3_w_shape[2] != p.H)
            return QMOE_ERR_INVALID_ARGUMENT;
    }
    // README Inputs.fc3_experts_weights: the separate linear operand of SwiGLU
    // with swiglu_fusion 0, or the multiplicative projection of SiLU.
    if (p.act == MOE_ACT_SWIGLU && p.swiglu_fusion == 0 && !has_fc3)
        return QMOE_ERR_INVALID_ARGUMENT;
    p.paired = (p.act == MOE_ACT_SWIGLU || (p.act == MOE_ACT_SILU && has_fc3)) ? 1 : 0;
    return QMOE_OK;
}

FWork fcarve(const FPlan& pl, void* ws) {
    char* b = static_cast<char*>(ws);
    FWork w;
    w.ctrl = reinterpret_cast<int32_t*>(b + pl.off_ctrl);
    w.sel = reinterpret_cast<int32_t*>(b + pl.off_sel);
    w.pw = reinterpret_cast<float*>(b + pl.off_pw);
    w.counts = reinterpret_cast<int32_t*>(b + pl.off_counts);
    w.offsets = reinterpret_cast<int32_t*>(b + pl.off_offsets);
    w.hist = reinterpret_cast<int32_t*>(b + pl.off_hist);
    w.rank = reinterpret_cast<int32_t*>(b + pl.off_rank);
    w.perm = reinterpret_cast<int32_t*>(b + pl.off_perm);
    w.inv = reinterpret_cast<int32_t*>(b + pl.off_inv);
    w.tiles = reinterpret_cast<int32_t*>(b + pl.off_tiles);
    w.active = reinterpret_cast<int32_t*>(b + pl.off_active);
    w.xs = reinterpret_cast<float*>(b + pl.off_xs);
    w.act = reinterpret_cast<float*>(b + pl.off_act);
    w.slot_out = reinterpret_cast<float*>(b + pl.off_slot_out);
    return w;
}

// Whether the grouped path may read these buffers through TMA and 16-byte loads.
bool grouped_pointers_ok(const FProblem& p) {
    return aligned16(p.x) && aligned16(p.w1) && aligned16(p.w2) && (!p.paired || aligned16(p.w3));
}

qmoe_status frun(FProblem& p, FPlan pl, void* workspace, int32_t* topk_idx_out,
                 float* topk_w_out, cudaStream_t s) {
    FWork w = fcarve(pl, workspace);
    if (topk_idx_out) w.sel = topk_idx_out;
    if (topk_w_out) w.pw = topk_w_out;
    if (p.T == 0) return QMOE_OK;
    if (p.path == MOE_PATH_GROUPED && !grouped_pointers_ok(p)) {
        // the generic layout fits in the grouped plan's workspace
        p.path = MOE_PATH_GENERIC;
        pl.tile_tokens = 0;
        pl.fc2_splits = 1;
    }
    // routing and grouping through the layer's shared kernels
    Problem rp;
    rp.T = p.T;
    rp.H = p.H;
    rp.E = p.E;
    rp.k = p.k;
    rp.x = p.x;
    rp.logits = p.logits;
    rp.y = p.y;
    rp.full_softmax = p.normalize ? 0 : 1;
    Plan rpl;
    rpl.slots = pl.slots;
    rpl.route_chunks = pl.route_chunks;
    rpl.tile_tokens = pl.tile_tokens;
    rpl.max_tiles = pl.max_tiles;
    rpl.Hp = 0;
    Work rw;
    std::memset(&rw, 0, sizeof(rw));
    rw.ctrl = w.ctrl;
    rw.sel = w.sel;
    rw.pw = w.pw;
    rw.counts = w.counts;
    rw.offsets = w.offsets;
    rw.hist = w.hist;
    rw.rank = w.rank;
    rw.perm = w.perm;
    rw.inv = w.inv;
    rw.tiles = w.tiles;
    rw.active = w.active;
    rw.x16 = nullptr;
    rw.slot_out = w.slot_out;
    cudaError_t e;
    if (small_route_ok(rp, rpl)) {
        if ((e = launch_route_group_small(rp, rpl, rw, 0, s)) != cudaSuccess) return QMOE_ERR_CUDA;
    } else {
        if ((e = launch_route(rp, rpl, rw, 0, s)) != cudaSuccess) return QMOE_ERR_CUDA;
        if ((e = launch_group(rp, rpl, rw, s)) != cudaSuccess) return QMOE_ERR_CUDA;
    }
    if (p.path == MOE_PATH_GROUPED) {
        if ((e = launch_moe_gather(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
        if ((e = launch_moe_grouped_fc(p, pl, w, true, s)) != cudaSuccess) return QMOE_ERR_CUDA;
        if ((e = launch_moe_grouped_fc(p, pl, w, false, s)) != cudaSuccess) return QMOE_ERR_CUDA;
    } else {
        if ((e = launch_moe_generic_fc1(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
        if ((e = launch_moe_generic_fc2(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
    }
    if ((e = launch_combine(rp, rpl, rw, pl.fc2_splits, s)) != cudaSuccess) return QMOE_ERR_CUDA;
    return QMOE_OK;
}

qmoe_status fprepare(const float* input, const int64_t* input_shape, int32_t input_rank,
                     const int64_t* router_shape, const float* fc1_w, const int64_t* fc1_w_shape,
                     const float* fc1_bias, const float* fc2_w, const int64_t* fc2_w_shape,
                     const float* fc2_bias, const float* fc3_w, const int64_t* fc3_w_shape,
                     const float* fc3_bias, const moe_attrs* attrs, FProblem* p, FPlan* pl) {
    qmoe_status st = fplan_for(input_shape, input_rank, fc1_w_shape, attrs, p, pl);
    if (st != QMOE_OK) return st;
    st = fcheck(*p, router_shape, fc2_w_shape, fc3_w_shape, fc3_w);
    if (st != QMOE_OK) return st;
    const bool uses_fc3 = (p->act == MOE_ACT_SWIGLU && p->swiglu_fusion == 0) ||
                          (p->act == MOE_ACT_SILU && p->paired);
    if (p->T > 0 && p->I > 0) {
        if (!fc1_w || !fc2_w) return QMOE_ERR_INVALID_ARGUMENT;
        if (uses_fc3 && !fc3_w) return QMOE_ERR_INVALID_ARGUMENT;
    }
    (void)input;
    p->w1 = fc1_w;
    p->b1 = fc1_bias;
    p->w2 = fc2_w;
    p->b2 = fc2_bias;
    p->w3 = uses_fc3 ? fc3_w : nullptr;
    p->b3 = uses_fc3 ? fc3_bias : nullptr;
    return QMOE_OK;
}

}  // namespace
}  // namespace qmoe

using namespace qmoe;

extern "C" {

void moe_attrs_default(moe_attrs* a) {
    if (!a) return;
    std::memset(a, 0, sizeof(*a));
    a->k = 1;
    a->activation_type = MOE_ACT_RELU;
    a->swiglu_fusion = 0;
    a->activation_alpha = 1.0f;
    a->activation_beta = 0.0f;
    a->has_swiglu_limit = 0;
    a->swiglu_limit = 0.0f;
    a->normalize_routing_weights = 0;
    a->use_sparse_mixer = 0;
    a->path = MOE_PATH_AUTO;
}

qmoe_status moe_workspace_size(const int64_t* input_shape, int32_t input_rank,
                               const int64_t* fc1_w_shape, const moe_attrs* attrs, size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    FProblem p;
    FPlan pl;
    qmoe_status st = fplan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    *bytes = pl.bytes;
    return QMOE_OK;
}

qmoe_status moe_choose_path(const int64_t* input_shape, int32_t input_rank,
                            const int64_t* fc1_w_shape, const moe_attrs* attrs, int32_t* path) {
    if (!path) return QMOE_ERR_INVALID_ARGUMENT;
    FProblem p;
    FPlan pl;
    qmoe_status st = fplan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    *path = p.path;
    return QMOE_OK;
}

qmoe_status moe_forward(const float* input, const int64_t* input_shape, int32_t input_rank,
                        const float* router_probs, const int64_t* router_shape,
                        const float* fc1_w, const int64_t* fc1_w_shape, const float* fc1_bias,
                        const float* fc2_w, const int64_t* fc2_w_shape, const float* fc2_bias,
                        const float* fc3_w, const int64_t* fc3_w_shape, const float* fc3_bias,
                        float* output, const moe_attrs* attrs, void* workspace,
                        size_t workspace_bytes, int32_t* topk_idx_out, float* topk_w_out,
                        void* cuda_stream) {
    FProblem p;
    FPlan pl;
    qmoe_status st = fprepare(input, input_shape, input_rank, router_shape, fc1_w, fc1_w_shape,
                              fc1_bias, fc2_w, fc2_w_shape, fc2_bias, fc3_w, fc3_w_shape,
                              fc3_bias, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    if (p.T > 0) {
        if (!input || !router_probs || !output || !workspace) return QMOE_ERR_INVALID_ARGUMENT;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return QMOE_ERR_INVALID_ARGUMENT;
        if (workspace_bytes < pl.bytes) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    }
    p.x = input;
    p.logits = router_probs;
    p.y = output;
    if (attrs->path == MOE_PATH_GROUPED && p.T > 0 && !grouped_pointers_ok(p))
        return QMOE_ERR_NOT_SUPPORTED;
    return frun(p, pl, workspace, topk_idx_out, topk_w_out, static_cast<cudaStream_t>(cuda_stream));
}

qmoe_status moe_hostio_workspace_size(const int64_t* input_shape, int32_t input_rank,
                                      const int64_t* fc1_w_shape, const moe_attrs* attrs,
                                      size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    FProblem p;
    FPlan pl;
    qmoe_status st = fplan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    const size_t xb = align_up(sizeof(float) * size_t(p.T) * size_t(p.H), 256);
    const size_t lb = align_up(sizeof(float) * size_t(p.T) * size_t(p.E), 256);
    *bytes = pl.bytes + 2 * xb + lb;
    return QMOE_OK;
}

qmoe_status moe_forward_hostio(const float* host_input, const int64_t* input_shape,
                               int32_t input_rank, const float* host_router_probs,
                               const int64_t* router_shape, const float* fc1_w,
                               const int64_t* fc1_w_shape, const float* fc1_bias,
                               const float* fc2_w, const int64_t* fc2_w_shape,
                               const float* fc2_bias, const float* fc3_w,
                               const int64_t* fc3_w_shape, const float* fc3_bias,
                               float* host_output, const moe_attrs* attrs, void* workspace,
                               size_t workspace_bytes, void* cuda_stream) {
    FProblem p;
    FPlan pl;
    qmoe_status st = fprepare(host_input, input_shape, input_rank, router_shape, fc1_w,
                              fc1_w_shape, fc1_bias, fc2_w, fc2_w_shape, fc2_bias, fc3_w,
                              fc3_w_shape, fc3_bias, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    if (p.T == 0) return QMOE_OK;
    const size_t xbytes = sizeof(float) * size_t(p.T) * size_t(p.H);
    const size_t lbytes = sizeof(float) * size_t(p.T) * size_t(p.E);
    const size_t xb = align_up(xbytes, 256), lb = align_up(lbytes, 256);
    if (!host_input || !host_router_probs || !host_output || !workspace)
        return QMOE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < pl.bytes + 2 * xb + lb) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    char* base = static_cast<char*>(workspace);
    float* d_x = reinterpret_cast<float*>(base + pl.bytes);
    float* d_l = reinterpret_cast<float*>(base + pl.bytes + xb);
    float* d_y = reinterpret_cast<float*>(base + pl.bytes + xb + lb);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemcpyAsync(d_x, host_input, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    if (cudaMemcpyAsync(d_l, host_router_probs, lbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    p.x = d_x;
    p.logits = d_l;
    p.y = d_y;
    if (attrs->path == MOE_PATH_GROUPED && !grouped_pointers_ok(p)) return QMOE_ERR_NOT_SUPPORTED;
    st = frun(p, pl, workspace, nullptr, nullptr, s);
    if (st != QMOE_OK) return st;
    if (cudaMemcpyAsync(host_output, d_y, xbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    return QMOE_OK;
}

qmoe_status moe_get_device_error(const void* workspace, void* cuda_stream, int32_t* code) {
    return qmoe_get_device_error(const_cast<void*>(workspace), cuda_stream, code);
}

}  // extern "C"
