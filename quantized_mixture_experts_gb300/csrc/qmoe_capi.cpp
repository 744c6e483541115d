// Host side of the C ABI: contract validation (QMoE manifest
// derive.quantContract and its parts), workspace planning, path choice and
// kernel dispatch.  No device memory is allocated here.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "qmoe_internal.h"

namespace qmoe {

// ---------------------------------------------------------------------------
// Launch bookkeeping and profiling hooks
// ---------------------------------------------------------------------------
namespace {
std::atomic<uint64_t> g_launches{0};
// The wait limit and the dropped-stage test hook belong to the host thread that
// sets them: they apply to the launches that thread makes, so a hook one thread
// sets cannot make another thread's layer time out.
thread_local uint64_t t_wait_limit_ns = 2000000000ull;
thread_local int64_t t_drop_stage = -1;

struct ProfPair {
    cudaEvent_t a = nullptr, b = nullptr;
};
std::mutex g_prof_mu;
int g_prof_kernel = -1000;
std::vector<ProfPair> g_prof_pool;
size_t g_prof_used = 0;
bool g_prof_open = false;
}  // namespace

uint64_t wait_limit_ns() { return t_wait_limit_ns; }
int64_t drop_stage() { return t_drop_stage; }

void note_launch(int kernel_id, cudaStream_t stream, bool begin, int nkernels) {
    if (!begin) g_launches.fetch_add(uint64_t(nkernels), std::memory_order_relaxed);
    if (kernel_id != g_prof_kernel) return;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (kernel_id != g_prof_kernel) return;
    if (begin) {
        if (g_prof_used == g_prof_pool.size()) {
            ProfPair pp;
            if (cudaEventCreate(&pp.a) != cudaSuccess || cudaEventCreate(&pp.b) != cudaSuccess)
                return;
            g_prof_pool.push_back(pp);
        }
        cudaEventRecord(g_prof_pool[g_prof_used].a, stream);
        g_prof_open = true;
    } else if (g_prof_open) {
        cudaEventRecord(g_prof_pool[g_prof_used].b, stream);
        ++g_prof_used;
        g_prof_open = false;
    }
}

// ---------------------------------------------------------------------------
// Validation (QMoE manifest: attributeConstraints, typeConstraints, derive.*)
// ---------------------------------------------------------------------------
namespace {

inline bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Attribute checks and shape derivation from input + fc1 weight shapes.
qmoe_status derive(const int64_t* input_shape, int32_t input_rank, const int64_t* fc1_w_shape,
                   const qmoe_attrs* a, Problem* p) {
    if (!input_shape || !fc1_w_shape || !a || !p) return QMOE_ERR_INVALID_ARGUMENT;
    // attributeConstraints
    if (a->quant_type_is_int != 1) return QMOE_ERR_NOT_SUPPORTED;
    if (a->expert_weight_bits != 4 && a->expert_weight_bits != 8) return QMOE_ERR_NOT_SUPPORTED;
    if (a->use_sparse_mixer == 1) return QMOE_ERR_NOT_SUPPORTED;
    if (a->use_sparse_mixer != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (a->weights_prepacked == 1) return QMOE_ERR_NOT_SUPPORTED;
    if (a->weights_prepacked != -1 && a->weights_prepacked != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (a->normalize_routing_weights != 0 && a->normalize_routing_weights != 1)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (a->activation_type != QMOE_ACT_RELU && a->activation_type != QMOE_ACT_SWIGLU)
        return QMOE_ERR_NOT_SUPPORTED;
    if (a->swiglu_fusion == 2) return QMOE_ERR_NOT_SUPPORTED;
    // derive.activationSupported
    const bool act_ok = (a->activation_type == QMOE_ACT_RELU && a->swiglu_fusion == 0) ||
                        (a->activation_type == QMOE_ACT_SWIGLU && a->swiglu_fusion == 1);
    if (!act_ok) return QMOE_ERR_INVALID_ARGUMENT;
    if (a->path < QMOE_PATH_AUTO || a->path > QMOE_PATH_GENERIC) return QMOE_ERR_INVALID_ARGUMENT;
    // input ranks and hidden size (derive.inputOutputShapeOk)
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
    p->bits = a->expert_weight_bits;
    p->pack = p->bits == 4 ? 2 : 1;          // derive.packSize
    p->mid = p->bits == 4 ? 8 : 128;         // derive.quantMidpoint
    p->act = a->activation_type;
    p->fusion = p->act == QMOE_ACT_SWIGLU ? 2 : 1;   // derive.fusionSize
    if (fc1_w_shape[1] % p->fusion != 0) return QMOE_ERR_INVALID_ARGUMENT;
    p->I = fc1_w_shape[1] / p->fusion;       // derive.interSize
    if (fc1_w_shape[2] * p->pack != H) return QMOE_ERR_INVALID_ARGUMENT;
    if (p->k < 1 || p->k > p->E) return QMOE_ERR_INVALID_ARGUMENT;
    // derive.quantBlockSizeOk
    p->bs = a->block_size;
    if (p->bs < 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (p->bs != 0) {
        if (p->bs < 16 || !is_pow2(p->bs) || H % p->bs != 0 || p->I % p->bs != 0)
            return QMOE_ERR_INVALID_ARGUMENT;
        p->nb1 = H / p->bs;
        p->nb2 = p->I / p->bs;
    } else {
        p->nb1 = p->nb2 = 1;
    }
    p->alpha = a->activation_alpha;
    p->beta = a->activation_beta;
    p->has_limit = a->has_swiglu_limit ? 1 : 0;
    p->limit = a->swiglu_limit;
    return QMOE_OK;
}

// Remaining tensor shape checks (derive.quantShapeOk, quantScalesOk).
qmoe_status check_shapes(const Problem& p, const int64_t* router_shape,
                         const int64_t* fc1_s_shape, int32_t fc1_s_rank,
                         const int64_t* fc2_w_shape, const int64_t* fc2_s_shape,
                         int32_t fc2_s_rank) {
    if (!router_shape || !fc1_s_shape || !fc2_w_shape || !fc2_s_shape)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (router_shape[0] != p.T || router_shape[1] != p.E) return QMOE_ERR_INVALID_ARGUMENT;
    if (fc2_w_shape[0] != p.E || fc2_w_shape[1] != p.H || fc2_w_shape[2] * p.pack != p.I)
        return QMOE_ERR_INVALID_ARGUMENT;
    const int want_rank = p.bs == 0 ? 2 : 3;
    if (fc1_s_rank != want_rank || fc2_s_rank != want_rank) return QMOE_ERR_INVALID_ARGUMENT;
    if (fc1_s_shape[0] != p.E || fc1_s_shape[1] != p.fusion * p.I) return QMOE_ERR_INVALID_ARGUMENT;
    if (fc2_s_shape[0] != p.E || fc2_s_shape[1] != p.H) return QMOE_ERR_INVALID_ARGUMENT;
    if (want_rank == 3 && (fc1_s_shape[2] != p.nb1 || fc2_s_shape[2] != p.nb2))
        return QMOE_ERR_INVALID_ARGUMENT;
    return QMOE_OK;
}

// Whether a kernel path can take this shape.
bool path_ok(const Problem& p, int path) {
    switch (path) {
        case QMOE_PATH_GENERIC: return true;
        case QMOE_PATH_DECODE: return decode_shape_ok(p);
        case QMOE_PATH_GROUPED: return grouped_shape_ok(p);
        default: return false;
    }
}

int choose_path(const Problem& p, int requested) {
    if (requested != QMOE_PATH_AUTO) return requested;
    if (p.T <= kDecodeMaxTokens && path_ok(p, QMOE_PATH_DECODE)) return QMOE_PATH_DECODE;
    if (path_ok(p, QMOE_PATH_GROUPED)) return QMOE_PATH_GROUPED;
    return QMOE_PATH_GENERIC;
}

qmoe_status make_plan(const Problem& p, Plan* pl) {
    Plan q;
    q.slots = p.T * p.k;
    q.route_chunks = (p.T + kRouteTokensPerChunk - 1) / kRouteTokensPerChunk;
    q.Hp = round_up(p.H, 64);
    q.Ip = round_up(std::max<int64_t>(p.I, 1), 64);
    q.tile_tokens = p.path == QMOE_PATH_GROUPED ? grouped_tile_tokens() : 0;
    q.max_tiles = q.tile_tokens ? (q.slots + q.tile_tokens - 1) / q.tile_tokens + p.E : 0;
    q.fc2_splits = p.path == QMOE_PATH_DECODE ? decode_fc2_splits(p) : 1;
    // grouped path: a token tile may read up to 15 rows past the last slot (its MMA
    // width is rounded up to 16), so the K-blocked layouts carry 16 spare rows
    q.srows = p.path == QMOE_PATH_GROUPED ? round_up(q.slots, 16) + 16 : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + std::max<size_t>(bytes, 1), 256);
        return o;
    };
    const size_t slots = size_t(q.slots);
    const size_t E = size_t(p.E);
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
    const bool generic = p.path == QMOE_PATH_GENERIC;
    // fp16 copy of x: the decode path's operand (the grouped path converts into
    // its sorted rows directly)
    q.off_x16 = take(p.path == QMOE_PATH_DECODE ? 2 * size_t(p.T) * size_t(q.Hp) : 0);
    const bool grouped = p.path == QMOE_PATH_GROUPED;
    q.off_xs16 = take(grouped ? 2 * size_t(q.srows) * size_t(q.Hp) : 0);
    q.off_act = take(generic ? 4 * slots * size_t(p.I)
                             : 2 * (grouped ? size_t(q.srows) : slots) * size_t(q.Ip));
    q.off_slot_out = take(4 * size_t(q.fc2_splits) * slots * size_t(p.H));
    q.bytes = off;
    *pl = q;
    return QMOE_OK;
}

Work carve(const Plan& pl, void* ws) {
    char* b = static_cast<char*>(ws);
    Work w;
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
    w.x16 = reinterpret_cast<__half*>(b + pl.off_x16);
    w.xs16 = reinterpret_cast<__half*>(b + pl.off_xs16);
    w.act = b + pl.off_act;
    w.slot_out = reinterpret_cast<float*>(b + pl.off_slot_out);
    return w;
}

qmoe_status plan_for(const int64_t* input_shape, int32_t input_rank, const int64_t* fc1_w_shape,
                     const qmoe_attrs* attrs, Problem* p, Plan* pl) {
    qmoe_status st = derive(input_shape, input_rank, fc1_w_shape, attrs, p);
    if (st != QMOE_OK) return st;
    p->path = choose_path(*p, attrs->path);
    if (!path_ok(*p, p->path)) return QMOE_ERR_NOT_SUPPORTED;
    return make_plan(*p, pl);
}

inline qmoe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA; }

qmoe_status run_forward(Problem& p, const Plan& pl, void* workspace, int32_t* topk_idx_out,
                        float* topk_w_out, cudaStream_t s) {
    Work w = carve(pl, workspace);
    if (topk_idx_out) w.sel = topk_idx_out;
    if (topk_w_out) w.pw = topk_w_out;
    if (p.T == 0) return QMOE_OK;
    cudaError_t e;
    if (p.I == 0) {
        // variant quant_zero_inter: the output is all zeros.
        e = cudaMemsetAsync(p.y, 0, sizeof(float) * size_t(p.T) * size_t(p.H), s);
        note_launch(-1, s, false, 1);
        if (e != cudaSuccess) return QMOE_ERR_CUDA;
        if (topk_idx_out || topk_w_out) {
            Work wr = w;
            wr.x16 = nullptr;
            e = launch_route(p, pl, wr, 0, s);
        } else {
            e = cudaMemsetAsync(w.ctrl, 0, sizeof(int32_t), s);
            note_launch(-1, s, false, 1);
        }
        return cuda_status(e);
    }
    switch (p.path) {
        case QMOE_PATH_GENERIC: {
            Work wr = w;
            wr.x16 = nullptr;
            if ((e = launch_route(p, pl, wr, 0, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_group(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_generic_fc1(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_generic_fc2(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_combine(p, pl, w, 1, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            return QMOE_OK;
        }
        case QMOE_PATH_DECODE: {
            const int mode = p.bits == 4 ? 2 : 0;   // layout the decode kernel reads
            if (small_route_ok(p, pl)) {
                if ((e = launch_route_group_small(p, pl, w, mode, s)) != cudaSuccess)
                    return QMOE_ERR_CUDA;
            } else {
                if ((e = launch_route(p, pl, w, mode, s)) != cudaSuccess) return QMOE_ERR_CUDA;
                if ((e = launch_group(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            }
            if ((e = launch_decode_fc(p, pl, w, true, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_decode_fc(p, pl, w, false, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_combine(p, pl, w, pl.fc2_splits, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            return QMOE_OK;
        }
        case QMOE_PATH_GROUPED: {
            // routing and grouping only: the sorted fp16 rows are converted from x directly
            // (in the operand order of the nibble conversion for 4-bit weights)
            Work wr = w;
            wr.x16 = nullptr;
            if (small_route_ok(p, pl)) {
                if ((e = launch_route_group_small(p, pl, wr, 0, s)) != cudaSuccess)
                    return QMOE_ERR_CUDA;
            } else {
                if ((e = launch_route(p, pl, wr, 0, s)) != cudaSuccess) return QMOE_ERR_CUDA;
                if ((e = launch_group(p, pl, wr, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            }
            if ((e = launch_sort_convert(p, pl, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_grouped_fc(p, pl, w, true, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_grouped_fc(p, pl, w, false, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            if ((e = launch_combine16(p, w, s)) != cudaSuccess) return QMOE_ERR_CUDA;
            return QMOE_OK;
        }
        default:
            return QMOE_ERR_NOT_SUPPORTED;
    }
}

}  // namespace
}  // namespace qmoe

namespace qmoe {
namespace {
// Device address of page-locked host memory mapped into the current device's
// address space, or null (pageable memory, or memory the device cannot map).
void* mapped_host(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();   // clear the (non-sticky) error of an unknown pointer
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return at.devicePointer;
}
}  // namespace
}  // namespace qmoe

using namespace qmoe;

extern "C" {

void qmoe_attrs_default(qmoe_attrs* a) {
    if (!a) return;
    std::memset(a, 0, sizeof(*a));
    a->k = 1;
    a->expert_weight_bits = 4;
    a->activation_type = QMOE_ACT_RELU;
    a->block_size = 0;
    a->swiglu_fusion = 0;
    a->activation_alpha = 1.0f;
    a->activation_beta = 0.0f;
    a->has_swiglu_limit = 0;
    a->swiglu_limit = 0.0f;
    a->normalize_routing_weights = 0;
    a->use_sparse_mixer = 0;
    a->weights_prepacked = -1;
    a->quant_type_is_int = 1;
    a->path = QMOE_PATH_AUTO;
}

const char* qmoe_status_string(qmoe_status s) {
    switch (s) {
        case QMOE_OK: return "ok";
        case QMOE_ERR_INVALID_ARGUMENT: return "invalid argument";
        case QMOE_ERR_NOT_SUPPORTED: return "not supported";
        case QMOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case QMOE_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

qmoe_status qmoe_workspace_size(const int64_t* input_shape, int32_t input_rank,
                                const int64_t* fc1_w_shape, const qmoe_attrs* attrs,
                                size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    Problem p;
    Plan pl;
    qmoe_status st = plan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    *bytes = pl.bytes;
    return QMOE_OK;
}

qmoe_status qmoe_choose_path(const int64_t* input_shape, int32_t input_rank,
                             const int64_t* fc1_w_shape, const qmoe_attrs* attrs, int32_t* path) {
    if (!path) return QMOE_ERR_INVALID_ARGUMENT;
    Problem p;
    Plan pl;
    qmoe_status st = plan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    *path = p.path;
    return QMOE_OK;
}

qmoe_status qmoe_forward(const float* input, const int64_t* input_shape, int32_t input_rank,
                         const float* router_probs, const int64_t* router_shape,
                         const uint8_t* fc1_w, const int64_t* fc1_w_shape,
                         const float* fc1_scales, const int64_t* fc1_scales_shape,
                         int32_t fc1_scales_rank, const uint8_t* fc2_w,
                         const int64_t* fc2_w_shape, const float* fc2_scales,
                         const int64_t* fc2_scales_shape, int32_t fc2_scales_rank,
                         float* output, const qmoe_attrs* attrs, void* workspace,
                         size_t workspace_bytes, int32_t* topk_idx_out, float* topk_w_out,
                         void* cuda_stream) {
    Problem p;
    Plan pl;
    qmoe_status st = plan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    st = check_shapes(p, router_shape, fc1_scales_shape, fc1_scales_rank, fc2_w_shape,
                      fc2_scales_shape, fc2_scales_rank);
    if (st != QMOE_OK) return st;
    if (p.T > 0) {
        if (!input || !router_probs || !output || !workspace) return QMOE_ERR_INVALID_ARGUMENT;
        if (p.I > 0 && (!fc1_w || !fc2_w || !fc1_scales || !fc2_scales))
            return QMOE_ERR_INVALID_ARGUMENT;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return QMOE_ERR_INVALID_ARGUMENT;
        if (workspace_bytes < pl.bytes) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    }
    p.x = input;
    p.logits = router_probs;
    p.w1 = fc1_w;
    p.s1 = fc1_scales;
    p.w2 = fc2_w;
    p.s2 = fc2_scales;
    p.y = output;
    return run_forward(p, pl, workspace, topk_idx_out, topk_w_out,
                       static_cast<cudaStream_t>(cuda_stream));
}

qmoe_status qmoe_hostio_workspace_size(const int64_t* input_shape, int32_t input_rank,
                                       const int64_t* fc1_w_shape, const qmoe_attrs* attrs,
                                       size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    Problem p;
    Plan pl;
    qmoe_status st = plan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    const size_t xb = align_up(sizeof(float) * size_t(p.T) * size_t(p.H), 256);
    const size_t lb = align_up(sizeof(float) * size_t(p.T) * size_t(p.E), 256);
    *bytes = pl.bytes + 2 * xb + lb;
    return QMOE_OK;
}

qmoe_status qmoe_forward_hostio(const float* host_input, const int64_t* input_shape,
                                int32_t input_rank, const float* host_router_probs,
                                const int64_t* router_shape, const uint8_t* fc1_w,
                                const int64_t* fc1_w_shape, const float* fc1_scales,
                                const int64_t* fc1_scales_shape, int32_t fc1_scales_rank,
                                const uint8_t* fc2_w, const int64_t* fc2_w_shape,
                                const float* fc2_scales, const int64_t* fc2_scales_shape,
                                int32_t fc2_scales_rank, float* host_output,
                                const qmoe_attrs* attrs, void* workspace, size_t workspace_bytes,
                                void* cuda_stream) {
    Problem p;
    Plan pl;
    qmoe_status st = plan_for(input_shape, input_rank, fc1_w_shape, attrs, &p, &pl);
    if (st != QMOE_OK) return st;
    st = check_shapes(p, router_shape, fc1_scales_shape, fc1_scales_rank, fc2_w_shape,
                      fc2_scales_shape, fc2_scales_rank);
    if (st != QMOE_OK) return st;
    if (p.T == 0) return QMOE_OK;
    const size_t xbytes = sizeof(float) * size_t(p.T) * size_t(p.H);
    const size_t lbytes = sizeof(float) * size_t(p.T) * size_t(p.E);
    const size_t xb = align_up(xbytes, 256), lb = align_up(lbytes, 256);
    if (!host_input || !host_router_probs || !host_output || !workspace)
        return QMOE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < pl.bytes + 2 * xb + lb) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    if (p.I > 0 && (!fc1_w || !fc2_w || !fc1_scales || !fc2_scales))
        return QMOE_ERR_INVALID_ARGUMENT;
    char* base = static_cast<char*>(workspace);
    float* d_x = reinterpret_cast<float*>(base + pl.bytes);
    float* d_l = reinterpret_cast<float*>(base + pl.bytes + xb);
    float* d_y = reinterpret_cast<float*>(base + pl.bytes + xb + lb);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    p.w1 = fc1_w;
    p.s1 = fc1_scales;
    p.w2 = fc2_w;
    p.s2 = fc2_scales;
    // small activations in mapped page-locked memory: the kernels read and write them in
    // place over the host link, without the copies' fixed costs
    if (xbytes <= QMOE_HOSTIO_DIRECT_BYTES) {
        void* mx = mapped_host(host_input);
        void* ml = mapped_host(host_router_probs);
        void* my = mapped_host(host_output);
        if (mx && ml && my) {
            p.x = static_cast<const float*>(mx);
            p.logits = static_cast<const float*>(ml);
            p.y = static_cast<float*>(my);
            return run_forward(p, pl, workspace, nullptr, nullptr, s);
        }
    }
    if (cudaMemcpyAsync(d_x, host_input, xbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    if (cudaMemcpyAsync(d_l, host_router_probs, lbytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    p.x = d_x;
    p.logits = d_l;
    p.y = d_y;
    st = run_forward(p, pl, workspace, nullptr, nullptr, s);
    if (st != QMOE_OK) return st;
    if (cudaMemcpyAsync(host_output, d_y, xbytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return QMOE_ERR_CUDA;
    return QMOE_OK;
}

qmoe_status grouped_matmul_workspace_size(size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    *bytes = 256;
    return QMOE_OK;
}

qmoe_status grouped_matmul_workspace_size_for(int64_t M, int64_t K, int64_t G, int64_t N,
                                              int64_t S, int32_t dtype, size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    if (M < 0 || K < 0 || G < 0 || N < 0 || S < 0) return QMOE_ERR_INVALID_ARGUMENT;
    const size_t tc = grouped_matmul_tc_workspace(M, K, G, N, S, dtype);
    *bytes = std::max<size_t>(256, tc);
    return QMOE_OK;
}

qmoe_status grouped_matmul(const void* input, int64_t M, int64_t K, const void* weights,
                           int64_t G, int64_t N, const void* group_indices, int64_t S,
                           int32_t index_dtype, const void* bias, void* output, int32_t dtype,
                           void* workspace, size_t workspace_bytes, void* cuda_stream) {
    if (M < 0 || K < 0 || G < 0 || N < 0 || S < 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (dtype < QMOE_DT_F32 || dtype > QMOE_DT_F64) return QMOE_ERR_INVALID_ARGUMENT;
    if (index_dtype != QMOE_IDX_I32 && index_dtype != QMOE_IDX_I64)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (!workspace) return QMOE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < 256) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int32_t* err = static_cast<int32_t*>(workspace);
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return QMOE_ERR_CUDA;
    note_launch(-1, s, false, 1);
    if (M * S == 0 || N == 0) return QMOE_OK;
    if (!input && K > 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (!group_indices || !output) return QMOE_ERR_INVALID_ARGUMENT;
    if (!weights && K > 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (G == 0) {
        // every index is out of range
    }
    // tensor cores when the shape, type, alignment and workspace allow it
    const size_t tc = grouped_matmul_tc_workspace(M, K, G, N, S, dtype);
    const auto aligned16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (tc > 0 && workspace_bytes >= tc && aligned16(input) && aligned16(weights) &&
        aligned16(output) && (reinterpret_cast<uintptr_t>(bias) & 1) == 0) {
        cudaError_t e = launch_grouped_matmul_tc(input, M, K, weights, G, N, group_indices, S,
                                                 index_dtype == QMOE_IDX_I64, bias, output, dtype,
                                                 workspace, s);
        return e == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
    }
    cudaError_t e = launch_grouped_matmul(input, M, K, weights, G, N, group_indices, S,
                                          index_dtype == QMOE_IDX_I64, bias, output, dtype, err,
                                          s);
    return e == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

qmoe_status qmoe_get_device_error(void* workspace, void* cuda_stream, int32_t* code) {
    if (!workspace || !code) return QMOE_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return QMOE_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
        return QMOE_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof(int32_t)) != cudaSuccess) return QMOE_ERR_CUDA;
    *code = v;
    return QMOE_OK;
}

void qmoe_set_wait_limit_ns(uint64_t ns) { t_wait_limit_ns = ns ? ns : 1; }

void qmoe_debug_drop_stage(int64_t stage) { t_drop_stage = stage < 0 ? -1 : stage; }

qmoe_status qmoe_profile_begin(int32_t kernel_id) {
    if (kernel_id < QMOE_KERNEL_ROUTE || kernel_id > QMOE_KERNEL_GMM)
        return QMOE_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_kernel = kernel_id;
    g_prof_used = 0;
    g_prof_open = false;
    return QMOE_OK;
}

qmoe_status qmoe_profile_end(int64_t* launches, double* total_ms) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    double total = 0.0;
    for (size_t i = 0; i < g_prof_used; ++i) {
        if (cudaEventSynchronize(g_prof_pool[i].b) != cudaSuccess) return QMOE_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_prof_pool[i].a, g_prof_pool[i].b) != cudaSuccess)
            return QMOE_ERR_CUDA;
        total += ms;
    }
    if (launches) *launches = int64_t(g_prof_used);
    if (total_ms) *total_ms = total;
    g_prof_kernel = -1000;
    g_prof_used = 0;
    g_prof_open = false;
    return QMOE_OK;
}

uint64_t qmoe_launch_count(void) { return g_launches.load(); }

}  // extern "C"
