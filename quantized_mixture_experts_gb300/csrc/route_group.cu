// Routing (top-k + softmax over the selected logits) and expert grouping
// (histogram, exclusive scan, stable permutation, tile table, and the
// expert-sorted fp16 token rows the grouped GEMMs read).
//
// QMoE manifest: `description` (the routing weights are a softmax over the k
// selected logits only), attributeDescriptions.normalize_routing_weights (same
// routing for 0 and 1), passes QMoE.RouteStage and QMoE.GroupStage
// (intermediates routeExpert, routeMix, slotList, tileMeta;
// derive.groupSlots, derive.groupMaxTiles).
// The float MoE (com.microsoft.MoE README, Description and Attributes) takes
// the softmax over all experts before top-k; with normalize_routing_weights = 1
// its weights are renormalised over the selection, which is the softmax over
// the selected logits again.  `full` selects the all-expert denominator.
#include <cuda_fp16.h>

#include <algorithm>

#include "ptx.cuh"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr int kRouteThreads = 1024;   // 32 routing warps: two tokens each per chunk
constexpr unsigned kFull = 0xffffffffu;

// Total order of the selection: larger logit first, equal logits by lower index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

// One warp selects the k best logits of row `row` (length E) in selection
// order and writes experts, logits (temporarily) and routing weights.
// General form: any E and k; every selection round re-reads the row.
__device__ void route_one_token_any(const float* __restrict__ row, int E, int k, int32_t* sel,
                                    float* pw, int32_t* s_exp, int lane, int full) {
    float prev_v = 0.f;
    int prev_i = -1;
    float vmax = 0.f;
    for (int i = 0; i < k; ++i) {
        float best_v = 0.f;
        int best_i = -1;
        for (int e = lane; e < E; e += 32) {
            float v = row[e];
            bool after_prev = (prev_i < 0) || better(prev_v, prev_i, v, e);
            if (after_prev && (best_i < 0 || better(v, e, best_v, best_i))) {
                best_v = v;
                best_i = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float ov = __shfl_xor_sync(kFull, best_v, off);
            int oi = __shfl_xor_sync(kFull, best_i, off);
            if (oi >= 0 && (best_i < 0 || better(ov, oi, best_v, best_i))) {
                best_v = ov;
                best_i = oi;
            }
        }
        prev_v = best_v;
        prev_i = best_i;
        if (i == 0) vmax = best_v;
        if (lane == 0) {
            sel[i] = best_i;
            pw[i] = best_v;
            s_exp[i] = best_i;
        }
    }
    __syncwarp();
    // softmax over the k selected logits (or every logit), max subtracted first
    float part = 0.f;
    if (full)
        for (int e = lane; e < E; e += 32) part += expf(row[e] - vmax);
    else
        for (int i = lane; i < k; i += 32) part += expf(pw[i] - vmax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    __syncwarp();
    for (int i = lane; i < k; i += 32) pw[i] = expf(pw[i] - vmax) / part;
}

// Order-preserving 32-bit key of a logit: key(a) > key(b) exactly when a > b
// (-0 is taken as +0 so that equal logits stay equal; NaN is out of contract).
// Every real key is above 0, which marks a removed entry.
__device__ __forceinline__ uint32_t logit_key(float v) {
    if (v == 0.f) v = 0.f;
    const uint32_t u = __float_as_uint(v);
    return u ^ ((u >> 31) ? 0xFFFFFFFFu : 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k >> 31) ? (k ^ 0x80000000u) : ~k);
}

// Same selection for E <= 32 * RR and k <= 32: the key of expert lane + 32 j
// sits in slot j of the lane's registers, read once.  Round i takes the
// largest remaining key over the warp (one max reduction), then the lowest
// expert index holding it (one min reduction), so ties go to the lower index
// as in the general form; the winner's lane marks it taken, and lane i keeps
// round i's winner, so the rounds and the softmax touch no memory.  The
// softmax sums in the same shuffle tree as the general form.
template <int RR>
__device__ __forceinline__ void route_one_token_regs(const float* __restrict__ row, int E, int k,
                                                     int32_t* sel, float* pw, int32_t* s_exp,
                                                     int lane, int full) {
    uint32_t key[RR];
#pragma unroll
    for (int j = 0; j < RR; ++j) key[j] = lane + 32 * j < E ? logit_key(row[lane + 32 * j]) : 0u;
    uint32_t taken = 0;   // bit j: slot j already selected
    float vmax = 0.f;
    float mine_v = 0.f;   // lane i: the logit selected in round i
    int mine_i = -1;
    for (int i = 0; i < k; ++i) {
        uint32_t bk = 0;
        int bj = 0;
#pragma unroll
        for (int j = 0; j < RR; ++j)
            if (!((taken >> j) & 1u) && key[j] > bk) {   // strict: the lower slot wins a tie
                bk = key[j];
                bj = j;
            }
        const uint32_t m = __reduce_max_sync(kFull, bk);
        const int win = __reduce_min_sync(kFull, bk == m ? lane + 32 * bj : 0x7FFFFFFF);
        if (lane == (win & 31)) taken |= 1u << (win >> 5);
        const float wv = key_logit(m);
        if (i == 0) vmax = wv;
        if (lane == i) {
            mine_v = wv;
            mine_i = win;
        }
    }
    // softmax over the k selected logits (or every logit), max subtracted first
    float part = lane < k ? expf(mine_v - vmax) : 0.f;
    const float mine_e = part;
    if (full) {
        part = 0.f;
#pragma unroll
        for (int j = 0; j < RR; ++j)
            if (lane + 32 * j < E) part += expf(key_logit(key[j]) - vmax);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    if (lane < k) {
        sel[lane] = mine_i;
        s_exp[lane] = mine_i;
        pw[lane] = mine_e / part;
    }
    __syncwarp();
}

// Routing of one token by one warp: the register form for E <= 256 and k <= 32
// (as few register slots per lane as E needs), the general form otherwise.
__device__ __forceinline__ void route_one_token(const float* __restrict__ row, int E, int k,
                                                int32_t* sel, float* pw, int32_t* s_exp, int lane,
                                                int full) {
    if (k > 32 || E > 256) route_one_token_any(row, E, k, sel, pw, s_exp, lane, full);
    else if (E <= 32) route_one_token_regs<1>(row, E, k, sel, pw, s_exp, lane, full);
    else if (E <= 64) route_one_token_regs<2>(row, E, k, sel, pw, s_exp, lane, full);
    else if (E <= 128) route_one_token_regs<4>(row, E, k, sel, pw, s_exp, lane, full);
    else route_one_token_regs<8>(row, E, k, sel, pw, s_exp, lane, full);
}

// Eight activations of row t (columns 8g..8g+7) stored as fp16 in layout mode
// `mode` (see convert_group).
__device__ __forceinline__ void store_group(const float* v, int64_t t, int64_t g,
                                            __half* __restrict__ x16, int64_t Hp, int mode) {
    __half2 h[4];
    if (mode == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) h[q] = __floats2half2_rn(v[q], v[q + 4]);
    } else if (mode == 2) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int src = (q >> 1) + 2 * (q & 1);     // pairs (0,4),(2,6),(1,5),(3,7)
            const float f = (src & 1) ? 0.0625f : 1.f;
            h[q] = __floats2half2_rn(v[src] * f, v[src + 4] * f);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) h[q] = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
    }
    uint4 o;
    o.x = ptx::h2_as_u32(h[0]); o.y = ptx::h2_as_u32(h[1]);
    o.z = ptx::h2_as_u32(h[2]); o.w = ptx::h2_as_u32(h[3]);
    reinterpret_cast<uint4*>(x16 + t * Hp)[g] = o;
}

// One group of eight activations of row t (columns 8g..8g+7), converted to fp16
// in layout mode:
//   0  natural order;
//   1  each group of eight stored in the order 0,4,1,5,2,6,3,7 (the pair order
//      of the 4-bit conversion);
//   2  each group of eight stored in the order 0,4,2,6,1,5,3,7 with the odd
//      elements divided by 16 (exact): the 4-bit decode kernel pairs
//      (0,4),(2,6) with low nibbles and (1,5),(3,7) with high nibbles, which
//      it feeds with 16x the code.
// Columns past H are zero.
__device__ __forceinline__ void convert_group(const float* __restrict__ x, int64_t t, int64_t g,
                                              int64_t H, bool vec, __half* __restrict__ x16,
                                              int64_t Hp, int mode) {
    const float* __restrict__ xr = x + t * H;
    float v[8];
    if (vec) {
        if (g * 8 < H) {
            const float4 a = reinterpret_cast<const float4*>(xr)[2 * g];
            const float4 b = reinterpret_cast<const float4*>(xr)[2 * g + 1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = 0.f;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = (g * 8 + q < H) ? xr[g * 8 + q] : 0.f;
    }
    __half2 h[4];
    if (mode == 1) {
#pragma unroll
        for (int q = 0; q < 4; ++q) h[q] = __floats2half2_rn(v[q], v[q + 4]);
    } else if (mode == 2) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int src = (q >> 1) + 2 * (q & 1);     // pairs (0,4),(2,6),(1,5),(3,7)
            const float f = (src & 1) ? 0.0625f : 1.f;
            h[q] = __floats2half2_rn(v[src] * f, v[src + 4] * f);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) h[q] = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
    }
    reinterpret_cast<uint4*>(x16 + t * Hp)[g] = *reinterpret_cast<uint4*>(h);
}

// fp16 copy of all T rows of the activations, zero padded to Hp (layout modes
// as in convert_group): the groups of eight columns of every row, flattened
// row-major, are taken in a grid-stride loop by `ncta` CTAs, two per thread
// per pass with both loads issued before the conversions.
__device__ void convert_all(const float* __restrict__ x, int64_t T, int64_t H,
                            __half* __restrict__ x16, int64_t Hp, int mode, int cta, int ncta) {
    const int64_t G8 = Hp / 8;
    const int64_t total = T * G8;
    const bool vec = (H & 7) == 0 && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
    const int64_t stride = int64_t(ncta) * blockDim.x;
    for (int64_t f0 = int64_t(cta) * blockDim.x + threadIdx.x; f0 < total; f0 += 2 * stride) {
        float v[2][8];
        int64_t t[2], g[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int64_t f = f0 + q * stride;
            t[q] = f / G8;
            g[q] = f - t[q] * G8;
            const float* __restrict__ xr = x + t[q] * H;
            if (f < total && vec && g[q] * 8 < H) {
                const float4 lo = reinterpret_cast<const float4*>(xr)[2 * g[q]];
                const float4 hi = reinterpret_cast<const float4*>(xr)[2 * g[q] + 1];
                v[q][0] = lo.x; v[q][1] = lo.y; v[q][2] = lo.z; v[q][3] = lo.w;
                v[q][4] = hi.x; v[q][5] = hi.y; v[q][6] = hi.z; v[q][7] = hi.w;
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    v[q][c] = (f < total && !vec && g[q] * 8 + c < H) ? xr[g[q] * 8 + c] : 0.f;
            }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (f0 + q * stride < total) store_group(v[q], t[q], g[q], x16, Hp, mode);
    }
}

// Blocks of 32 slots of a routing chunk, and the largest per-block count table
// (blocks x experts) the parallel ranking keeps in shared memory.
constexpr int kRankCap = 8192;
__host__ __device__ inline int rank_blocks(int k) { return (kRouteTokensPerChunk * k + 31) / 32; }
__host__ __device__ inline bool rank_parallel(int E, int k) {
    return int64_t(rank_blocks(k)) * E <= kRankCap && rank_blocks(k) <= kRouteThreads / 32;
}

// Grid chunks + conv CTAs.  CTA c < chunks routes chunk c's tokens (one warp
// per token), then ranks the chunk's slots per expert (stable, in slot order)
// and writes the chunk histogram: block b of 32 slots is ranked by warp b
// (in-block ranks and counts), an exclusive scan over blocks per expert gives
// each block's bases.  The other `conv` CTAs convert the activations to fp16
// (convert_all) while the routing CTAs run.
__global__ void __launch_bounds__(kRouteThreads) route_kernel(
    const float* __restrict__ logits, int64_t T, int E, int k, int32_t* __restrict__ sel,
    float* __restrict__ pw, int32_t* __restrict__ hist, int32_t* __restrict__ rank,
    const float* __restrict__ x, int64_t H, __half* __restrict__ x16, int64_t Hp,
    int x16_mode, int full, int32_t* __restrict__ ctrl, int chunks) {
    // the grouping kernels launched after this one may be scheduled now (they wait
    // for its completion before reading anything)
    ptx::griddep_launch_dependents();
    if (int(blockIdx.x) >= chunks) {
        convert_all(x, T, H, x16, Hp, x16_mode, int(blockIdx.x) - chunks, int(gridDim.x) - chunks);
        return;
    }
    extern __shared__ int32_t smem[];
    int32_t* s_cnt = smem;        // [E]
    int32_t* s_exp = smem + E;    // [chunk tokens * k]
    int32_t* s_blk = s_exp + kRouteTokensPerChunk * k;   // [rank_blocks(k)][E] (parallel ranking)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x) * kRouteTokensPerChunk;
    const int ntok = int(T - t0 < kRouteTokensPerChunk ? T - t0 : kRouteTokensPerChunk);
    if (blockIdx.x == 0 && threadIdx.x == 0 && ctrl) ctrl[0] = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    const bool par = rank_parallel(E, k);
    const int nslots = ntok * k;
    const int nblk = (nslots + 31) / 32;
    if (par)
        for (int j = threadIdx.x; j < nblk * E; j += blockDim.x) s_blk[j] = 0;
    for (int lt = warp; lt < ntok; lt += kRouteThreads / 32) {
        const int64_t t = t0 + lt;
        route_one_token(logits + t * E, E, k, sel + t * k, pw + t * k, s_exp + lt * k, lane, full);
    }
    __syncthreads();
    if (par) {
        int32_t* rank_out = rank + t0 * k;
        // in-block rank of each slot and the block's count per expert
        int e = -1, r = 0;
        if (warp < nblk) {
            const int j = warp * 32 + lane;
            e = j < nslots ? s_exp[j] : -1 - lane;   // distinct dummies
            const unsigned mask = __match_any_sync(kFull, e);
            r = __popc(mask & ((1u << lane) - 1u));
            if (e >= 0 && lane == __ffs(mask) - 1) s_blk[warp * E + e] = __popc(mask);
        }
        __syncthreads();
        // exclusive scan over blocks, per expert; the totals are the chunk histogram
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int run = 0;
            for (int b = 0; b < nblk; ++b) {
                const int c = s_blk[b * E + x];
                s_blk[b * E + x] = run;
                run += c;
            }
            s_cnt[x] = run;
        }
        __syncthreads();
        if (warp < nblk && e >= 0) rank_out[warp * 32 + lane] = s_blk[warp * E + e] + r;
    } else if (warp == 0) {
        int32_t* rank_out = rank + t0 * k;
        for (int base = 0; base < nslots; base += 32) {
            const int j = base + lane;
            const int e = j < nslots ? s_exp[j] : -1 - lane;   // distinct dummies
            const unsigned mask = __match_any_sync(kFull, e);
            const int leader = __ffs(mask) - 1;
            const int r = __popc(mask & ((1u << lane) - 1u));
            int c = (lane == leader && e >= 0) ? s_cnt[e] : 0;
            c = __shfl_sync(kFull, c, leader);
            if (e >= 0) rank_out[j] = c + r;
            __syncwarp();
            if (lane == leader && e >= 0) s_cnt[e] = c + __popc(mask);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[int64_t(blockIdx.x) * E + e] = s_cnt[e];
}

// Whole routing + grouping for small batches in one launch.  CTA 0 (1024
// threads) routes every token, ranks the slots per expert, scans the counts
// and writes offsets, the active-expert list, the tile table and the
// permutation; CTAs 1.. convert the activations to fp16.
__global__ void __launch_bounds__(1024) route_group_small_kernel(
    const float* __restrict__ logits, int64_t T, int E, int k, int32_t* __restrict__ sel,
    float* __restrict__ pw, const float* __restrict__ x, int64_t H, __half* __restrict__ x16,
    int64_t Hp, int x16_mode, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ tiles, int32_t* __restrict__ active, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int tile_tokens, int full, int32_t* __restrict__ ctrl) {
    extern __shared__ int32_t smem[];
    if (blockIdx.x > 0) {
        if (x16) {
            const int64_t G8 = Hp / 8;
            const int64_t nconv = gridDim.x - 1;
            const int64_t total = T * G8;
            const int64_t per = (total + nconv - 1) / nconv;
            const int64_t lo = int64_t(blockIdx.x - 1) * per;
            const int64_t hi = lo + per < total ? lo + per : total;
            // walk the flat (token, group) range
            const bool vec = (H & 7) == 0 && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
            for (int64_t idx = lo + threadIdx.x; idx < hi; idx += blockDim.x) {
                const int64_t t = idx / G8;
                convert_group(x, t, idx - t * G8, H, vec, x16, Hp, x16_mode);
            }
        }
        return;
    }
    const int slots = int(T) * k;
    int32_t* s_cnt = smem;              // [E]
    int32_t* s_off = s_cnt + E;         // [E + 1]
    int32_t* s_tb = s_off + E + 1;      // [E]
    int32_t* s_exp = s_tb + E;          // [slots]
    int32_t* s_rank = s_exp + slots;    // [slots]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (threadIdx.x == 0 && ctrl) ctrl[0] = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    for (int t = warp; t < T; t += nw)
        route_one_token(logits + int64_t(t) * E, E, k, sel + int64_t(t) * k, pw + int64_t(t) * k,
                        s_exp + t * k, lane, full);
    __syncthreads();
    if (warp == 0) {
        for (int base = 0; base < slots; base += 32) {
            const int j = base + lane;
            const int e = j < slots ? s_exp[j] : -1 - lane;
            const unsigned mask = __match_any_sync(kFull, e);
            const int leader = __ffs(mask) - 1;
            const int r = __popc(mask & ((1u << lane) - 1u));
            int c = (lane == leader && e >= 0) ? s_cnt[e] : 0;
            c = __shfl_sync(kFull, c, leader);
            if (e >= 0) s_rank[j] = c + r;
            __syncwarp();
            if (lane == leader && e >= 0) s_cnt[e] = c + __popc(mask);
            __syncwarp();
        }
        int32_t off_run = 0, tile_run = 0, act_run = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int32_t cnt = e < E ? s_cnt[e] : 0;
            const int32_t nt = tile_tokens > 0 ? (cnt + tile_tokens - 1) / tile_tokens : 0;
            const int32_t is_act = cnt > 0 ? 1 : 0;
            int32_t a = cnt, b = nt, c = is_act;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t ya = __shfl_up_sync(kFull, a, off);
                const int32_t yb = __shfl_up_sync(kFull, b, off);
                const int32_t yc = __shfl_up_sync(kFull, c, off);
                if (lane >= off) { a += ya; b += yb; c += yc; }
            }
            if (e < E) {
                s_off[e] = off_run + a - cnt;
                s_tb[e] = tile_run + b - nt;
                counts[e] = cnt;
                offsets[e] = off_run + a - cnt;
                if (is_act) active[act_run + c - 1] = e;
            }
            off_run += __shfl_sync(kFull, a, 31);
            tile_run += __shfl_sync(kFull, b, 31);
            act_run += __shfl_sync(kFull, c, 31);
        }
        if (lane == 0) {
            s_off[E] = off_run;
            offsets[E] = off_run;
            tiles[0] = tile_run;
            tiles[1] = act_run;
            tiles[2] = tile_tokens;
            tiles[3] = 0;
        }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < slots; j += blockDim.x) {
        const int32_t pos = s_off[s_exp[j]] + s_rank[j];
        perm[pos] = j;
        inv[j] = pos;
    }
    if (tile_tokens > 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int32_t cnt = s_cnt[e];
            for (int32_t j = 0; j * tile_tokens < cnt; ++j) {
                int32_t* tt = tiles + kTileHeader + 4 * (s_tb[e] + j);
                tt[0] = e;
                tt[1] = s_off[e] + j * tile_tokens;
                tt[2] = min(tile_tokens, cnt - j * tile_tokens);
                tt[3] = s_tb[e];
            }
        }
    }
}

// Single CTA: per-expert totals, chunk bases (in place over `hist`), offsets,
// active-expert list and the expert tile table.
__global__ void __launch_bounds__(1024) group_scan_kernel(
    int32_t* __restrict__ hist, int64_t chunks, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ tiles, int32_t* __restrict__ active,
    int tile_tokens) {
    // launched as a programmatic dependent of the routing kernel
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    extern __shared__ int32_t sh[];
    const int tid = threadIdx.x, nthr = blockDim.x;
    // Phase 1: parts x experts partial sums.  P parts split the chunk range.
    const int P = E >= nthr ? 1 : nthr / E;
    int32_t* s_part = sh;                 // [P * E]
    for (int e0 = 0; e0 < E; e0 += nthr / P) {
        const int e = e0 + tid % (nthr / P);
        const int part = tid / (nthr / P);
        const bool on = (e < E) && (part < P) && (e - e0 < nthr / P);
        const int64_t c_lo = chunks * part / P, c_hi = chunks * (part + 1) / P;
        int32_t sum = 0;
        if (on) {
            // eight loads in flight per batch
            int64_t c = c_lo;
            for (; c + 8 <= c_hi; c += 8) {
                int32_t v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = hist[(c + q) * E + e];
#pragma unroll
                for (int q = 0; q < 8; ++q) sum += v[q];
            }
            for (; c < c_hi; ++c) sum += hist[c * E + e];
            s_part[part * E + e] = sum;
        }
    }
    __syncthreads();
    // Phase 2: exclusive scan over parts for each expert; totals.
    for (int e = tid; e < E; e += nthr) {
        int32_t run = 0;
        for (int part = 0; part < P; ++part) {
            int32_t v = s_part[part * E + e];
            s_part[part * E + e] = run;
            run += v;
        }
        counts[e] = run;
    }
    __syncthreads();
    // Phase 3: chunk bases within each part.
    for (int e0 = 0; e0 < E; e0 += nthr / P) {
        const int e = e0 + tid % (nthr / P);
        const int part = tid / (nthr / P);
        const bool on = (e < E) && (part < P) && (e - e0 < nthr / P);
        if (on) {
            const int64_t c_lo = chunks * part / P, c_hi = chunks * (part + 1) / P;
            int32_t run = s_part[part * E + e];
            int64_t c = c_lo;
            for (; c + 8 <= c_hi; c += 8) {   // batches of eight: loads first, then stores
                int32_t v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = hist[(c + q) * E + e];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    hist[(c + q) * E + e] = run;
                    run += v[q];
                }
            }
            for (; c < c_hi; ++c) {
                const int32_t v = hist[c * E + e];
                hist[c * E + e] = run;
                run += v;
            }
        }
    }
    __syncthreads();
    // Phase 4: one warp scans counts -> offsets, tile bases, active list.
    int32_t* s_tile_base = sh;            // reuse: [E]
    if (tid < 32) {
        const int lane = tid;
        int32_t off_run = 0, tile_run = 0, act_run = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int32_t cnt = e < E ? counts[e] : 0;
            const int32_t nt = tile_tokens > 0 ? (cnt + tile_tokens - 1) / tile_tokens : 0;
            const int32_t is_act = cnt > 0 ? 1 : 0;
            int32_t a = cnt, b = nt, c = is_act;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int32_t ya = __shfl_up_sync(kFull, a, off);
                int32_t yb = __shfl_up_sync(kFull, b, off);
                int32_t yc = __shfl_up_sync(kFull, c, off);
                if (lane >= off) { a += ya; b += yb; c += yc; }
            }
            if (e < E) {
                offsets[e] = off_run + a - cnt;
                s_tile_base[e] = tile_run + b - nt;
                if (is_act) active[act_run + c - 1] = e;
            }
            off_run += __shfl_sync(kFull, a, 31);
            tile_run += __shfl_sync(kFull, b, 31);
            act_run += __shfl_sync(kFull, c, 31);
        }
        if (lane == 0) {
            offsets[E] = off_run;
            tiles[0] = tile_run;
            tiles[1] = act_run;
            tiles[2] = tile_tokens;
            tiles[3] = 0;
        }
    }
    __syncthreads();
    // Phase 5: tile table entries (expert, first sorted row, rows, the expert's first tile).
    if (tile_tokens > 0) {
        for (int e = tid; e < E; e += nthr) {
            const int32_t cnt = counts[e];
            const int32_t base = s_tile_base[e];
            const int32_t row0 = offsets[e];
            for (int32_t j = 0; j * tile_tokens < cnt; ++j) {
                int32_t* tt = tiles + kTileHeader + 4 * (base + j);
                tt[0] = e;
                tt[1] = row0 + j * tile_tokens;
                tt[2] = min(tile_tokens, cnt - j * tile_tokens);
                tt[3] = base;
            }
        }
    }
}

// perm[pos] = slot, inv[slot] = pos, pos = offsets[e] + chunk base + rank.
__global__ void group_scatter_kernel(const int32_t* __restrict__ sel,
                                     const int32_t* __restrict__ rank,
                                     const int32_t* __restrict__ hist,
                                     const int32_t* __restrict__ offsets, int64_t slots, int k,
                                     int E, int32_t* __restrict__ perm,
                                     int32_t* __restrict__ inv) {
    // launched as a programmatic dependent of the scan
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    const int64_t s = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (s >= slots) return;
    const int e = sel[s];
    const int64_t chunk = (s / k) / kRouteTokensPerChunk;
    const int32_t pos = offsets[e] + hist[chunk * E + e] + rank[s];
    perm[pos] = int32_t(s);
    inv[s] = pos;
}

// The fp16 activations in expert-sorted slot order (row pos = token
// perm[pos] / k), K-blocked [Hp/64][srows][64] with the 128-byte swizzle of the
// row's position in its token tile applied: 16-byte chunk c of a 64-column
// block is stored at c ^ ((pos - offsets[expert]) & 7).  Token tiles start at
// multiples of their expert's first row plus multiples of 8, so a tile's rows
// of one K block are one contiguous, already swizzled 128-byte-row block.
//
// Written straight from the fp32 input: `parts` warps per token (interleaved
// passes of 128 groups of eight columns, four per lane) read the row once,
// convert it to fp16 in the operand order `mode` (0 natural; 1 each group of
// eight as 0,4,1,5,2,6,3,7, the pair order of the 4-bit conversion), and store
// it at each of the token's k sorted positions.  Columns past H are zero.
__global__ void sort_convert_kernel(const float* __restrict__ x, int64_t T, int64_t H,
                                    int64_t Hp, int vec, int mode, int parts,
                                    const int32_t* __restrict__ inv,
                                    const int32_t* __restrict__ sel,
                                    const int32_t* __restrict__ offsets, int k, int64_t srows,
                                    uint4* __restrict__ xs16) {
    // launched as a programmatic dependent of the grouping kernels; the grouped GEMM
    // after it may start its prologue on SMs this grid leaves
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * wpb;
    const int G8 = int(Hp / 8);
    for (int64_t wi = int64_t(blockIdx.x) * wpb + (threadIdx.x >> 5); wi < T * parts; wi += nwarps) {
        const int64_t t = wi / parts;
        const int part = int(wi - t * parts);
        // lane i: sorted position of the token's slot i (i < 32) and its swizzle phase
        int my_pos = 0, my_ph = 0;
        if (lane < k) {
            my_pos = __ldg(inv + t * k + lane);
            my_ph = (my_pos - __ldg(offsets + __ldg(sel + t * k + lane))) & 7;
        }
        const float* __restrict__ xr = x + t * H;
        for (int g0 = part * 32 * U; g0 < G8; g0 += parts * 32 * U) {
            uint4 val[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int g = g0 + u * 32 + lane;
                float v[8];
                if (vec && int64_t(g) * 8 < H) {
                    const float4 lo = __ldg(reinterpret_cast<const float4*>(xr) + 2 * g);
                    const float4 hi = __ldg(reinterpret_cast<const float4*>(xr) + 2 * g + 1);
                    v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
                    v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = (!vec && g < G8 && int64_t(g) * 8 + c < H) ? xr[int64_t(g) * 8 + c] : 0.f;
                }
                __half2 h[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    h[q] = mode == 1 ? __floats2half2_rn(v[q], v[q + 4])
                                     : __floats2half2_rn(v[2 * q], v[2 * q + 1]);
                val[u] = make_uint4(ptx::h2_as_u32(h[0]), ptx::h2_as_u32(h[1]),
                                    ptx::h2_as_u32(h[2]), ptx::h2_as_u32(h[3]));
            }
            for (int i = 0; i < k; ++i) {
                int pos = __shfl_sync(kFull, my_pos, i & 31);
                int ph = __shfl_sync(kFull, my_ph, i & 31);
                if (i >= 32) {   // slots past the first 32 (k > 32): read directly
                    pos = __ldg(inv + t * k + i);
                    ph = (pos - __ldg(offsets + __ldg(sel + t * k + i))) & 7;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int g = g0 + u * 32 + lane;
                    if (g < G8) xs16[(int64_t(g >> 3) * srows + pos) * 8 + ((g & 7) ^ ph)] = val[u];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_route(const Problem& p, const Plan& pl, const Work& w, int x16_mode,
                         cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (size_t(p.E) + size_t(kRouteTokensPerChunk) * p.k +
                                           (rank_parallel(int(p.E), int(p.k))
                                                ? size_t(rank_blocks(int(p.k))) * p.E : 0));
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(route_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
    }
    // conversion CTAs: the SMs the routing CTAs leave (at least half of them), one
    // 1024-thread CTA per SM
    int conv = 0;
    if (w.x16) {
        const int sms = device_sm_count();
        conv = std::max(sms / 2, sms - int(std::min<int64_t>(pl.route_chunks, sms)));
    }
    note_launch(QMOE_KERNEL_ROUTE, s, true);
    route_kernel<<<unsigned(pl.route_chunks + conv), kRouteThreads, smem, s>>>(
        p.logits, p.T, int(p.E), int(p.k), w.sel, w.pw, w.hist, w.rank, p.x, p.H, w.x16, pl.Hp,
        x16_mode, p.full_softmax, w.ctrl, int(pl.route_chunks));
    note_launch(QMOE_KERNEL_ROUTE, s, false);
    return cudaGetLastError();
}

bool small_route_ok(const Problem& p, const Plan& pl) {
    return pl.slots <= kSmallRouteSlots && p.E <= 1024;
}

cudaError_t launch_route_group_small(const Problem& p, const Plan& pl, const Work& w,
                                     int x16_mode, cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (3 * size_t(p.E) + 1 + 2 * size_t(pl.slots));
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(route_group_small_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
    }
    int conv = 0;
    if (w.x16) conv = int(std::min<int64_t>(64, std::max<int64_t>(1, p.T * (pl.Hp / 8) / 2048)));
    note_launch(QMOE_KERNEL_ROUTE, s, true);
    route_group_small_kernel<<<unsigned(1 + conv), 1024, smem, s>>>(
        p.logits, p.T, int(p.E), int(p.k), w.sel, w.pw, p.x, p.H, w.x16, pl.Hp,
        x16_mode, w.counts, w.offsets, w.tiles, w.active, w.perm, w.inv,
        pl.tile_tokens, p.full_softmax, w.ctrl);
    note_launch(QMOE_KERNEL_ROUTE, s, false);
    return cudaGetLastError();
}

// Counts, offsets, tile table and stable permutation of `slots` items with
// group ids sel[0..slots) in [0, E), from per-chunk histograms (chunks of
// kRouteTokensPerChunk * k items) and in-chunk ranks.
cudaError_t launch_group_items(int32_t* hist, int64_t chunks, int E, int32_t* counts,
                               int32_t* offsets, int32_t* tiles, int32_t* active, int tile_tokens,
                               const int32_t* sel, const int32_t* rank, int64_t slots, int k,
                               int32_t* perm, int32_t* inv, cudaStream_t s) {
    const int nthr = 1024;
    const int P = E >= nthr ? 1 : nthr / E;
    const size_t smem = sizeof(int32_t) * std::max<size_t>(size_t(P) * E, size_t(E));
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(group_scan_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
    }
    group_scan_kernel<<<1, nthr, smem, s>>>(hist, chunks, E, counts, offsets, tiles, active,
                                            tile_tokens);
    group_scatter_kernel<<<unsigned((slots + 255) / 256), 256, 0, s>>>(sel, rank, hist, offsets,
                                                                       slots, k, E, perm, inv);
    return cudaGetLastError();
}

cudaError_t launch_group(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s) {
    const int E = int(p.E);
    const int nthr = 1024;
    const int P = E >= nthr ? 1 : nthr / E;
    const size_t smem = sizeof(int32_t) * std::max<size_t>(size_t(P) * E, size_t(E));
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(group_scan_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
    }
    note_launch(QMOE_KERNEL_GROUP, s, true);
    // each a programmatic dependent of the kernel before it
    cudaError_t e = launch_dependent(group_scan_kernel, dim3(1), dim3(nthr), smem, s, w.hist,
                                     int64_t(pl.route_chunks), E, w.counts, w.offsets, w.tiles,
                                     w.active, int(pl.tile_tokens));
    const int64_t slots = pl.slots;
    if (e == cudaSuccess)
        e = launch_dependent(group_scatter_kernel, dim3(unsigned((slots + 255) / 256)), dim3(256),
                             0, s, (const int32_t*)w.sel, (const int32_t*)w.rank,
                             (const int32_t*)w.hist, (const int32_t*)w.offsets, slots, int(p.k),
                             E, w.perm, w.inv);
    note_launch(QMOE_KERNEL_GROUP, s, false, 2);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_sort_convert(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s) {
    // warps per token: enough warps for 32 per SM, at most one per 128-group pass
    const int64_t passes = (pl.Hp / 8 + 127) / 128;
    const int64_t want = (int64_t(32) * device_sm_count() + p.T - 1) / std::max<int64_t>(1, p.T);
    const int parts = int(std::max<int64_t>(1, std::min<int64_t>(want, passes)));
    const int64_t warps = std::max<int64_t>(1, p.T * parts);
    const int blocks = int(std::min<int64_t>((warps + 7) / 8, int64_t(device_sm_count()) * 8));
    const int vec = (p.H % 8 == 0 && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0) ? 1 : 0;
    note_launch(QMOE_KERNEL_GROUP, s, true);
    const cudaError_t e = launch_dependent(
        sort_convert_kernel, dim3(unsigned(std::max(blocks, 1))), dim3(256), 0, s, p.x,
        int64_t(p.T), int64_t(p.H), int64_t(pl.Hp), vec, p.bits == 4 ? 1 : 0, parts,
        (const int32_t*)w.inv, (const int32_t*)w.sel, (const int32_t*)w.offsets, int(p.k),
        int64_t(pl.srows), reinterpret_cast<uint4*>(w.xs16));
    note_launch(QMOE_KERNEL_GROUP, s, false);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmoe
