// Kernels of the float (unquantized) MoE layer, com.microsoft.MoE README
// (Description, Inputs, Attributes):
//
//  * scalar fp32 FC1/FC3 and FC2 kernels for any shape (one warp per output
//    element, fixed summation order);
//  * the expert-grouped path: the routed token rows gathered in expert order
//    as TF32 values, K-blocked with the 128-byte swizzle pre-applied, and one
//    persistent tcgen05 kernel (kind::tf32, fp32 accumulators in TMEM) per
//    projection:
//
//      warp 0      TMA producer: per 32-wide K stage, two 128-row weight tiles
//                  straight from the fp32 weights (boxes of 32 x 128 with the
//                  128-byte swizzle: the K-major A operand as stored) and the
//                  token tile as one 1-D bulk copy of its gathered rows;
//      warp 1      TMEM allocator and MMA issuer (one lane);
//      warps 2-9   epilogue: tcgen05.ld, + bias, activation (FC1: written as
//                  TF32 in the K-blocked layout FC2 reads) or FC2 rows by
//                  routing slot (fp32, bias added by the first K split).
//
//    The two weight tiles of an item are the gate and linear projections of
//    the same 128 intermediate units when the activation pairs them (SwiGLU
//    in its three layouts, SiLU times FC3), else 256 consecutive rows.
#include <algorithm>
#include <cstring>

#include "moe_internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Activations (README Attributes.activation_type, swiglu_fusion)
// ---------------------------------------------------------------------------
// sigmoid(v) = 1 / (1 + exp(-v)); the Fast form uses the identity
// sigmoid(v) = (1 + tanh(v/2)) / 2 with the hardware tanh approximation (relative
// error near 2^-11, the size of the TF32 rounding its result then takes).
template <bool Fast>
__device__ __forceinline__ float sigm(float v) {
    if constexpr (Fast) {
        float t;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * v));
        return fmaf(0.5f, t, 0.5f);
    } else {
        return __fdividef(1.f, 1.f + __expf(-v));
    }
}

template <bool Fast>
__device__ __forceinline__ float act_single(int act, float h) {
    switch (act) {
        case MOE_ACT_RELU: return fmaxf(h, 0.f);
        case MOE_ACT_GELU: return 0.5f * h * erfcf(-h * 0.70710678118654752f);   // h * Phi(h)
        case MOE_ACT_SILU: return h * sigm<Fast>(h);
        default: return h;                                                       // identity
    }
}

// Activations of two projections: SiLU(g) * u, or SwiGLU g*sigmoid(alpha*g)*(u+beta)
// after the optional clamp (gate from above, linear branch on both sides).
template <bool Fast>
__device__ __forceinline__ float act_pair(int act, float g, float u, float alpha, float beta,
                                          int has_limit, float limit) {
    if (act == MOE_ACT_SILU) return g * sigm<Fast>(g) * u;
    if (has_limit) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    return g * sigm<Fast>(alpha * g) * (u + beta);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

// fp32 -> TF32 (10-bit mantissa), round to nearest, ties away from zero.
__device__ __forceinline__ float to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// ---------------------------------------------------------------------------
// Scalar path
// ---------------------------------------------------------------------------

// One warp per (intermediate unit j, sorted row pos): the FC1 (and FC3) dot
// products, biases and activation; act is [slots, I] in sorted order.
__global__ void moe_generic_fc1_kernel(FProblem p, const int32_t* __restrict__ perm,
                                       const int32_t* __restrict__ sel, float* __restrict__ act,
                                       int64_t slots) {
    const int64_t widx = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (widx >= slots * p.I) return;
    const int64_t j = widx / slots, pos = widx % slots;   // unit-major: weight rows stay in cache
    const int32_t s = perm[pos];
    const int64_t t = s / p.k, e = sel[s];
    const float* __restrict__ xt = p.x + t * p.H;
    const float* __restrict__ r0;
    const float* __restrict__ r1 = nullptr;
    float b0 = 0.f, b1 = 0.f;
    if (p.act == MOE_ACT_SWIGLU && p.swiglu_fusion == 1) {          // rows 2j (gate), 2j+1
        r0 = p.w1 + (e * p.rows1 + 2 * j) * p.H;
        r1 = r0 + p.H;
        if (p.b1) { b0 = p.b1[e * p.rows1 + 2 * j]; b1 = p.b1[e * p.rows1 + 2 * j + 1]; }
    } else if (p.act == MOE_ACT_SWIGLU && p.swiglu_fusion == 2) {   // rows j (gate), I + j
        r0 = p.w1 + (e * p.rows1 + j) * p.H;
        r1 = p.w1 + (e * p.rows1 + p.I + j) * p.H;
        if (p.b1) { b0 = p.b1[e * p.rows1 + j]; b1 = p.b1[e * p.rows1 + p.I + j]; }
    } else {
        r0 = p.w1 + (e * p.I + j) * p.H;
        if (p.b1) b0 = p.b1[e * p.I + j];
        if (p.paired) {                                             // FC3 row j
            r1 = p.w3 + (e * p.I + j) * p.H;
            if (p.b3) b1 = p.b3[e * p.I + j];
        }
    }
    float g = 0.f, u = 0.f;
    if (r1) {
        for (int64_t kk = lane; kk < p.H; kk += 32) {
            const float xv = xt[kk];
            g += xv * r0[kk];
            u += xv * r1[kk];
        }
        g = warp_sum(g) + b0;
        u = warp_sum(u) + b1;
        g = act_pair<false>(p.act, g, u, p.alpha, p.beta, p.has_limit, p.limit);
    } else {
        for (int64_t kk = lane; kk < p.H; kk += 32) g += xt[kk] * r0[kk];
        g = act_single<false>(p.act, warp_sum(g) + b0);
    }
    if (lane == 0) act[pos * p.I + j] = g;
}

// One warp per (output column d, sorted row pos): FC2 + bias, written to the
// row of the original slot.
__global__ void moe_generic_fc2_kernel(FProblem p, const int32_t* __restrict__ perm,
                                       const int32_t* __restrict__ sel,
                                       const float* __restrict__ act, float* __restrict__ slot_out,
                                       int64_t slots) {
    const int64_t widx = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (widx >= slots * p.H) return;
    const int64_t d = widx / slots, pos = widx % slots;
    const int32_t s = perm[pos];
    const int64_t e = sel[s];
    const float* __restrict__ wr = p.w2 + (e * p.H + d) * p.I;
    const float* __restrict__ ar = act + pos * p.I;
    float o = 0.f;
    for (int64_t kk = lane; kk < p.I; kk += 32) o += ar[kk] * wr[kk];
    o = warp_sum(o);
    if (p.b2) o += p.b2[e * p.H + d];
    if (lane == 0) slot_out[int64_t(s) * p.H + d] = o;
}

unsigned blocks_for(int64_t n, int per) { return unsigned((n + per - 1) / per); }

// ---------------------------------------------------------------------------
// Grouped path
// ---------------------------------------------------------------------------

// Expert-sorted TF32 rows of x, K-blocked [H/32][srows][32]: the 16-byte chunk c
// of sorted row pos is stored at c ^ ((pos - offsets[e]) & 7), the 128-byte
// swizzle of the row's position in its token tile (tiles start at multiples of
// 256 rows of their expert).  One warp per sorted row.
__global__ void moe_gather_kernel(const float4* __restrict__ x, int64_t H4,
                                  const int32_t* __restrict__ perm,
                                  const int32_t* __restrict__ sel,
                                  const int32_t* __restrict__ offsets, int k, int64_t slots,
                                  int64_t srows, float4* __restrict__ xs) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * wpb;
    for (int64_t pos = int64_t(blockIdx.x) * wpb + (threadIdx.x >> 5); pos < slots; pos += nwarps) {
        const int32_t r = __ldg(perm + pos);
        const int e = __ldg(sel + r);
        const int phase = int(pos - __ldg(offsets + e)) & 7;
        const float4* __restrict__ src = x + int64_t(r / k) * H4;
        for (int64_t q = lane; q < H4; q += 32) {
            float4 v = __ldg(src + q);
            v.x = to_tf32(v.x);
            v.y = to_tf32(v.y);
            v.z = to_tf32(v.z);
            v.w = to_tf32(v.w);
            xs[((q >> 3) * srows + pos) * 8 + ((q & 7) ^ phase)] = v;
        }
    }
}

constexpr int kFM = 128;                       // weight rows per CTA per MMA tile
constexpr int kFMaxN = 256;                    // token rows per tile (MMA N upper bound)
constexpr int kFK = 32;                        // K per stage: 32 fp32 = one 128-byte row
constexpr uint32_t kFATile = kFM * 128;        // one CTA's weight tile per stage
constexpr uint32_t kFABytes = 2 * kFATile;
constexpr int kFBBox = 32;                     // token rows per TMA box (CTA pairs)
constexpr int kFMaxStages = 8;
constexpr int kFEpiWarps = 16;                 // 4 per TMEM lane quadrant
constexpr int kFChunk = 16;                    // accumulator columns per TMEM load
constexpr int kFThreads = 32 * (2 + kFEpiWarps);
constexpr uint64_t kFDrainWaitNs = 200000000ull;

struct FtcArgs {
    CUtensorMap tm0;         // weight rows {K, rows, E}, boxes {32, 128, 1}, 128-byte swizzle
    CUtensorMap tm1;         // second projection of a pair (same layout)
    CUtensorMap tm_b;        // CTA pairs: token rows {32, srows, K/32}, boxes {32, 32, 1}
    const float* xs;         // token rows, K-blocked [K/32][srows][32], pre-swizzled TF32
    int64_t srows;
    const int32_t* tiles;    // header + (expert, first sorted row, rows, 0)
    const int32_t* perm;     // sorted position -> slot
    int64_t N, K, slots;
    int n_pairs, gm, splits, kb_per_split;
    int paired, fc1;
    int stages;
    uint32_t stage_bytes;
    const float* bias0;      // bias of tile 0 rows (and tile 1 when unpaired): [e*es + j*js]
    int64_t b0_es, b0_js;
    const float* bias1;      // bias of the paired projection
    int64_t b1_es, b1_js;
    int act;
    float alpha, beta;
    int has_limit;
    float limit;
    float* act_out;          // FC1: K-blocked [N/32][srows][32] TF32
    float* slot_out;         // FC2: [splits][slots][N]
    int32_t* err;
    uint64_t wait_ns;
};

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory descriptor of a K-major operand with the 128-byte swizzle:
// 128-byte rows, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t saddr) {
    uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t(1) << 16;                 // leading byte offset (unused with this swizzle)
    d |= uint64_t(1024 >> 4) << 32;         // stride byte offset
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor: TF32 A and B, fp32 accumulator, both K-major, M x N.
__device__ __forceinline__ uint32_t tf32_idesc(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(n >> 3) << 17) |
           (uint32_t(m >> 4) << 24);
}

// One MMA.  With CTA pairs (issued by CTA 0) A is M = 256 rows, 128 from each
// CTA's shared memory at the same offset, B is N rows, N/2 from each CTA, and
// each CTA's tensor memory receives its 128 rows of D.
template <int kCta>
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    if constexpr (kCta == 2)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
            ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive on `bar` when the issuing thread's MMAs complete: in this CTA, or (CTA
// pairs, both = true) at the same offset in both CTAs.
template <int kCta>
__device__ __forceinline__ void mma_commit(uint64_t* bar, bool both) {
    if constexpr (kCta == 2) {
        if (both)
            asm volatile(
                "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
                " [%0], %1;" ::"r"(ptx::smem_u32(bar)), "h"(uint16_t(3))
                : "memory");
        else
            asm volatile(
                "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                ::"r"(ptx::smem_u32(bar))
                : "memory");
    } else {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            ::"r"(ptx::smem_u32(bar))
            : "memory");
    }
}

// Tiled 3-D load into this CTA's shared memory, completion counted on the
// barrier at shared::cluster address `bar` (CTA pairs: CTA 0's barrier).
template <int kCta>
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint32_t bar) {
    if constexpr (kCta == 2)
        asm volatile(
            "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];"
            ::"r"(ptx::smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
            : "memory");
    else
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];"
            ::"r"(ptx::smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
            : "memory");
}

// 16 consecutive accumulator columns of this thread's TMEM lane; `wait` = false
// leaves the wait to a later tmem_wait() so that two loads overlap.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct FItem {
    int e, row0, rows, n0, nt, kb0, kb1, sp;
};

// Work item i: batches of gm row groups; inside a batch token tile by token
// tile, then row group, then K split.  A row group is 128 * kCta units of a
// paired activation (gate and linear tiles) or 256 * kCta rows otherwise.
template <int kCta>
__device__ __forceinline__ FItem ft_item(const FtcArgs& a, int64_t i, int ntiles, int nkb) {
    const int64_t per_batch = int64_t(ntiles) * a.gm * a.splits;
    const int pg = int(i / per_batch);
    const int64_t rem = i % per_batch;
    const int tau = int(rem / (a.gm * a.splits));
    const int r2 = int(rem % (a.gm * a.splits));
    const int pm = r2 / a.splits;
    FItem it;
    it.sp = r2 % a.splits;
    const int32_t* t = a.tiles + kTileHeader + 4 * tau;
    it.e = t[0];
    it.row0 = t[1];
    it.rows = t[2];
    it.n0 = (pg * a.gm + pm) * (a.paired ? kFM * kCta : 2 * kFM * kCta);
    it.nt = kCta == 2 ? (it.rows + 31) & ~31 : (it.rows + 15) & ~15;
    it.kb0 = it.sp * a.kb_per_split;
    it.kb1 = min(nkb, it.kb0 + a.kb_per_split);
    return it;
}

// kCta = 1: one CTA per item.  kCta = 2: a cluster of two CTAs per item; CTA 0
// issues the MMAs (cta_group::2), both CTAs load their halves of A and B with
// completion on CTA 0's barriers, and MMA completions are multicast to both.
template <int kCta>
__global__ void __launch_bounds__(kFThreads, 1) moe_tf32_kernel(const __grid_constant__ FtcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t load_full[kFMaxStages];
    __shared__ __align__(8) uint64_t load_empty[kFMaxStages];
    __shared__ __align__(8) uint64_t acc_full;
    __shared__ __align__(8) uint64_t acc_empty;
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = a.stages;
    const uint32_t rank = kCta == 2 ? ptx::cluster_rank() : 0u;
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            ptx::mbar_init(&load_full[s], 1);
            ptx::mbar_init(&load_empty[s], 1);
        }
        ptx::mbar_init(&acc_full, 1);
        ptx::mbar_init(&acc_empty, kFEpiWarps * kCta);
        ptx::mbar_init(&drain_bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        if constexpr (kCta == 2) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(ptx::smem_u32(&tmem_base_s)), "r"(512)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(ptx::smem_u32(&tmem_base_s)), "r"(512)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    if constexpr (kCta == 2) ptx::cluster_sync(); else __syncthreads();
    tc_fence_after();
    // the next kernel in the stream may start its prologue
    ptx::griddep_launch_dependents();
    const uint32_t tmem_base = tmem_base_s;
    const int ntiles = a.tiles[0];
    const int64_t items = int64_t(ntiles) * a.n_pairs * a.splits;
    const int nkb = int(a.K / kFK);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int64_t first = blockIdx.x / kCta, step = gridDim.x / kCta;
    // this CTA's first weight row of tile t of an item starting at n0
    const int tile_stride = a.paired ? 0 : kFM * kCta;
    const int row_off = kFM * int(rank);

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            ptx::prefetch_tmap(&a.tm0);
            if (a.paired) ptx::prefetch_tmap(&a.tm1);
            if (kCta == 2) ptx::prefetch_tmap(&a.tm_b);
        }
        uint32_t it = 0, sl = 0, ph = 0;
        bool ok = true;
        for (int64_t i = first; i < items && ok; i += step) {
            const FItem w = ft_item<kCta>(a, i, ntiles, nkb);
            const int nbox = (w.nt / 2 + kFBBox - 1) / kFBBox;   // CTA pairs: B boxes per CTA
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                if (!ptx::mbar_wait(&load_empty[sl], ph ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint8_t* sp = smem + size_t(sl) * a.stage_bytes;
                    const uint32_t fb = kCta == 2 ? ptx::leader_addr(&load_full[sl])
                                                  : ptx::smem_u32(&load_full[sl]);
                    if (leader)
                        ptx::mbar_arrive_expect_tx(
                            &load_full[sl],
                            kCta == 2 ? 2u * (kFABytes + uint32_t(nbox) * kFBBox * 128u)
                                      : kFABytes + uint32_t(w.nt) * 128u);
                    tma_load_3d<kCta>(sp, &a.tm0, kb * kFK, w.n0 + row_off, w.e, fb);
                    tma_load_3d<kCta>(sp + kFATile, a.paired ? &a.tm1 : &a.tm0, kb * kFK,
                                      w.n0 + tile_stride + row_off, w.e, fb);
                    if constexpr (kCta == 2) {
                        const int r0 = w.row0 + int(rank) * (w.nt / 2);
                        for (int b = 0; b < nbox; ++b)
                            tma_load_3d<2>(sp + kFABytes + b * (kFBBox * 128), &a.tm_b, 0,
                                           r0 + b * kFBBox, kb, fb);
                    } else {
                        ptx::bulk_g2s(sp + kFABytes, a.xs + (int64_t(kb) * a.srows + w.row0) * kFK,
                                      uint32_t(w.nt) * 128u, &load_full[sl]);
                    }
                }
                __syncwarp();
                if (++sl == uint32_t(stages)) { sl = 0; ph ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
            abort_flag = 1;
            // wait (bounded) for the copies still in flight before leaving; with CTA
            // pairs they complete on CTA 0's barriers, and the final cluster barrier
            // keeps CTA 1 resident until CTA 0 has drained
            if (leader)
                for (uint32_t j = it > uint32_t(stages) ? it - stages : 0; j < it; ++j) {
                    volatile int never = 0;
                    ptx::mbar_wait(&load_full[j % stages], (j / stages) & 1u, kFDrainWaitNs, &never);
                }
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer -------------------------------
        if (leader) {
            uint32_t sl = 0, ph = 0, item_it = 0;
            bool ok = true, issued = false;
            for (int64_t i = first; i < items && ok; i += step) {
                const FItem w = ft_item<kCta>(a, i, ntiles, nkb);
                // both CTAs' epilogues arrive here: acquire at cluster scope
                if (!ptx::mbar_wait_cluster(&acc_empty, (item_it & 1u) ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                ++item_it;
                tc_fence_after();
                const uint32_t idesc = tf32_idesc(kFM * kCta, w.nt);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!ptx::mbar_wait(&load_full[sl], ph, a.wait_ns, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t sa = sbase + sl * a.stage_bytes;
                        const uint32_t sb = sa + kFABytes;
#pragma unroll
                        for (int kk = 0; kk < kFK / 8; ++kk) {   // K = 8 per MMA (32 bytes)
                            const uint64_t bd = kmajor_sw128_desc(sb + 32u * kk);
#pragma unroll
                            for (int t = 0; t < 2; ++t)
                                mma_tf32<kCta>(tmem_base + uint32_t(t * kFMaxN),
                                               kmajor_sw128_desc(sa + uint32_t(t) * kFATile + 32u * kk),
                                               bd, idesc, (kb > w.kb0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit<kCta>(&load_empty[sl], true);
                        issued = true;
                    }
                    __syncwarp();
                    if (++sl == uint32_t(stages)) { sl = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (lane == 0) mma_commit<kCta>(&acc_full, true);
                __syncwarp();
            }
            if (!ok && lane == 0) {
                atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
                abort_flag = 1;
            }
            if (lane == 0 && issued) {
                mma_commit<kCta>(&drain_bar, false);
                volatile int never = 0;
                ptx::mbar_wait(&drain_bar, 0, kFDrainWaitNs, &never);
            }
            __syncwarp();
        }
    } else {
        // -------------------------------- epilogue --------------------------------
        const int ew = warp - 2;                   // 0..15
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int cg = ew >> 2;                    // column chunks cg, cg + 4, ... of 16
        const uint32_t empty_addr = kCta == 2 ? ptx::leader_addr(&acc_empty) : ptx::smem_u32(&acc_empty);
        constexpr int kChunks = kFMaxN / (4 * kFChunk);   // chunks per warp
        uint32_t item_it = 0;
        for (int64_t i = first; i < items; i += step) {
            const FItem w = ft_item<kCta>(a, i, ntiles, nkb);
            const uint32_t aph = item_it & 1u;
            ++item_it;
            // FC2: lane l < 16 holds the slot of token row c0 + l of each of the warp's chunks
            int slot_c[kChunks];
#pragma unroll
            for (int m = 0; m < kChunks; ++m) {
                const int col = (cg + 4 * m) * kFChunk + lane;
                slot_c[m] = (!a.fc1 && lane < kFChunk && col < w.rows) ? __ldg(a.perm + w.row0 + col) : 0;
            }
            // this lane's output rows and their biases
            const int64_t j0 = int64_t(w.n0) + row_off + quad * 32 + lane;      // tile 0
            const int64_t j1 = j0 + tile_stride;                                 // tile 1
            const bool use_bias = a.fc1 || w.sp == 0;
            float bias0 = 0.f, bias1 = 0.f;
            if (use_bias && a.bias0 && j0 < a.N) bias0 = __ldg(a.bias0 + w.e * a.b0_es + j0 * a.b0_js);
            if (a.paired) {
                if (a.bias1 && j1 < a.N) bias1 = __ldg(a.bias1 + w.e * a.b1_es + j1 * a.b1_js);
            } else if (use_bias && a.bias0 && j1 < a.N) {
                bias1 = __ldg(a.bias0 + w.e * a.b0_es + j1 * a.b0_js);
            }
            // FC1: element (token row c0 + q, unit j) of the K-blocked output sits at
            // rowbase(j) + q * 32 + ((chunk(j) ^ (q & 7)) << 2) for 16-aligned c0
            float* const ob0 = a.act_out + ((j0 >> 5) * a.srows + w.row0) * 32 + (j0 & 3);
            float* const ob1 = a.act_out + ((j1 >> 5) * a.srows + w.row0) * 32 + (j1 & 3);
            const int ch0 = int((j0 & 31) >> 2), ch1 = int((j1 & 31) >> 2);
            if (!ptx::mbar_wait(&acc_full, aph, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
                    abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const uint32_t tq = tmem_base + (uint32_t(quad * 32) << 16);
#pragma unroll
            for (int m = 0; m < kChunks; ++m) {
                const int c0 = (cg + 4 * m) * kFChunk;
                if (c0 >= w.nt) break;
                float v0[kFChunk], v1[kFChunk];
                tmem_ld16(tq + uint32_t(c0), v0);
                tmem_ld16(tq + uint32_t(kFMaxN + c0), v1);
                tmem_wait();
                if (a.fc1) {
                    float* const p0 = ob0 + int64_t(c0) * 32;
                    float* const p1 = ob1 + int64_t(c0) * 32;
                    if (a.paired) {
                        if (j0 < a.N) {
#pragma unroll
                            for (int q = 0; q < kFChunk; ++q)
                                if (c0 + q < w.rows)
                                    p0[q * 32 + ((ch0 ^ (q & 7)) << 2)] =
                                        to_tf32(act_pair<true>(a.act, v0[q] + bias0, v1[q] + bias1,
                                                               a.alpha, a.beta, a.has_limit, a.limit));
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < kFChunk; ++q) {
                            if (c0 + q >= w.rows) break;
                            if (j0 < a.N)
                                p0[q * 32 + ((ch0 ^ (q & 7)) << 2)] =
                                    to_tf32(act_single<true>(a.act, v0[q] + bias0));
                            if (j1 < a.N)
                                p1[q * 32 + ((ch1 ^ (q & 7)) << 2)] =
                                    to_tf32(act_single<true>(a.act, v1[q] + bias1));
                        }
                    }
                } else {
                    float* outp = a.slot_out + int64_t(w.sp) * a.slots * a.N;
#pragma unroll
                    for (int q = 0; q < kFChunk; ++q) {
                        const int slot = __shfl_sync(kFull, slot_c[m], q);
                        if (c0 + q < w.rows) {
                            if (j0 < a.N) outp[int64_t(slot) * a.N + j0] = v0[q] + bias0;
                            if (j1 < a.N) outp[int64_t(slot) * a.N + j1] = v1[q] + bias1;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (kCta == 2)   // CTA 0's barrier counts both CTAs' epilogues
                    ptx::mbar_arrive_cluster(empty_addr);
                else
                    ptx::mbar_arrive(&acc_empty);
            }
        }
    }

    tc_fence_before();
    if constexpr (kCta == 2) ptx::cluster_sync(); else __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if constexpr (kCta == 2)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(512)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(512)
                         : "memory");
    }
}

// Weight rows as a 3-D tensor {K, rows, E} of fp32 with the given row and
// expert strides (elements); boxes of 32 (K) x 128 rows.
bool encode_rows(CUtensorMap* map, const float* base, int64_t K, int64_t rows, int64_t E,
                 int64_t row_stride, int64_t expert_stride) {
    const uint64_t dims[3] = {uint64_t(K), uint64_t(rows), uint64_t(E)};
    const uint64_t strides[2] = {uint64_t(row_stride) * 4, uint64_t(expert_stride) * 4};
    const uint32_t box[3] = {uint32_t(kFK), uint32_t(kFM), 1};
    return encode_tmap_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

// Stages of the load ring that fit in shared memory.
int ring_stages(uint32_t stage_bytes) {
    const int n = int((225u * 1024u) / stage_bytes);
    return std::max(2, std::min(kFMaxStages, n));
}

// Token rows one CTA holds per stage: the whole tile, or half of it in boxes of
// kFBBox rows for CTA pairs.
uint32_t b_rows_per_cta(int bmax, int cta) {
    if (cta == 1) return uint32_t(bmax);
    return uint32_t((bmax / 2 + kFBBox - 1) / kFBBox * kFBBox);
}

}  // namespace

bool moe_grouped_shape_ok(const FProblem& p) {
    return p.H % kFK == 0 && p.I % kFK == 0 && p.I > 0 && p.H > 0 && p.E <= 65535 &&
           p.T * p.k <= (int64_t(1) << 30);
}

// CTAs per work item: pairs (cta_group::2) once token tiles are large enough
// that the shared-memory traffic per MMA matters; single CTAs for few tokens.
int moe_cta_group(const FPlan& pl) { return pl.bmax >= 128 ? 2 : 1; }

// Split-K factor of the grouped FC2: the count s that minimises the estimated
// time, rounds of work units per SM times the K blocks of a unit (about 0.7 us
// each, tensor- or HBM-bound alike) plus the partial rows every split writes
// and the combine reads back (ties to the smaller s).  The token tiles are
// estimated from the slot count.
int moe_fc2_splits(const FProblem& p, int64_t slots, int cta) {
    const int64_t sms = device_sm_count() / cta;
    const int64_t tiles = std::max<int64_t>((slots + kFTileTokens - 1) / kFTileTokens,
                                            std::min<int64_t>(p.E, slots));
    const int64_t items = tiles * ((p.H + 2 * kFM * cta - 1) / (2 * kFM * cta));
    const int64_t nkb = p.I / kFK;
    const double stage_us = 0.7, bytes_per_us = 6.5e6;
    int best = 1;
    double best_cost = -1.0;
    for (int s = 1; s <= 16 && s <= nkb; ++s) {
        const int64_t per = (nkb + s - 1) / s;
        if ((nkb + per - 1) / per != s) continue;   // every split non-empty
        const double cost = double((items * s + sms - 1) / sms) * double(per) * stage_us +
                            double(s) * double(slots) * double(p.H) * 8.0 / bytes_per_us;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

cudaError_t launch_moe_generic_fc1(const FProblem& p, const FPlan& pl, const FWork& w,
                                   cudaStream_t s) {
    const int64_t total = pl.slots * p.I;
    if (total == 0) return cudaSuccess;
    note_launch(QMOE_KERNEL_FC1, s, true);
    moe_generic_fc1_kernel<<<blocks_for(total, 8), 256, 0, s>>>(p, w.perm, w.sel, w.act, pl.slots);
    note_launch(QMOE_KERNEL_FC1, s, false);
    return cudaGetLastError();
}

cudaError_t launch_moe_generic_fc2(const FProblem& p, const FPlan& pl, const FWork& w,
                                   cudaStream_t s) {
    const int64_t total = pl.slots * p.H;
    note_launch(QMOE_KERNEL_FC2, s, true);
    moe_generic_fc2_kernel<<<blocks_for(total, 8), 256, 0, s>>>(p, w.perm, w.sel, w.act,
                                                                w.slot_out, pl.slots);
    note_launch(QMOE_KERNEL_FC2, s, false);
    return cudaGetLastError();
}

cudaError_t launch_moe_gather(const FProblem& p, const FPlan& pl, const FWork& w, cudaStream_t s) {
    const int blocks = int(std::min<int64_t>((pl.slots + 7) / 8, int64_t(device_sm_count()) * 8));
    note_launch(QMOE_KERNEL_GROUP, s, true);
    moe_gather_kernel<<<std::max(blocks, 1), 256, 0, s>>>(
        reinterpret_cast<const float4*>(p.x), p.H / 4, w.perm, w.sel, w.offsets, int(p.k),
        pl.slots, pl.srows, reinterpret_cast<float4*>(w.xs));
    note_launch(QMOE_KERNEL_GROUP, s, false);
    return cudaGetLastError();
}

cudaError_t launch_moe_grouped_fc(const FProblem& p, const FPlan& pl, const FWork& w, bool fc1,
                                  cudaStream_t s) {
    FtcArgs a;
    std::memset(&a, 0, sizeof(a));
    const int64_t H = p.H, I = p.I, E = p.E;
    bool ok;
    if (fc1) {
        a.K = H;
        a.N = I;
        a.paired = p.paired;
        a.xs = w.xs;
        if (p.act == MOE_ACT_SWIGLU && p.swiglu_fusion == 1) {
            // interleaved: gate rows 2j, linear rows 2j + 1
            ok = encode_rows(&a.tm0, p.w1, H, I, E, 2 * H, 2 * I * H) &&
                 encode_rows(&a.tm1, p.w1 + H, H, I, E, 2 * H, 2 * I * H);
            a.bias0 = p.b1; a.b0_es = 2 * I; a.b0_js = 2;
            a.bias1 = p.b1 ? p.b1 + 1 : nullptr; a.b1_es = 2 * I; a.b1_js = 2;
        } else if (p.act == MOE_ACT_SWIGLU && p.swiglu_fusion == 2) {
            // concatenated: gate rows [0, I), linear rows [I, 2I)
            ok = encode_rows(&a.tm0, p.w1, H, I, E, H, 2 * I * H) &&
                 encode_rows(&a.tm1, p.w1 + I * H, H, I, E, H, 2 * I * H);
            a.bias0 = p.b1; a.b0_es = 2 * I; a.b0_js = 1;
            a.bias1 = p.b1 ? p.b1 + I : nullptr; a.b1_es = 2 * I; a.b1_js = 1;
        } else {
            ok = encode_rows(&a.tm0, p.w1, H, I, E, H, I * H);
            a.bias0 = p.b1; a.b0_es = I; a.b0_js = 1;
            if (p.paired) {   // FC3 supplies the linear projection
                ok = ok && encode_rows(&a.tm1, p.w3, H, I, E, H, I * H);
                a.bias1 = p.b3; a.b1_es = I; a.b1_js = 1;
            }
        }
        a.splits = 1;
        a.act_out = w.act;
    } else {
        a.K = I;
        a.N = H;
        a.paired = 0;
        a.xs = w.act;
        ok = encode_rows(&a.tm0, p.w2, I, H, E, I, H * I);
        a.bias0 = p.b2; a.b0_es = H; a.b0_js = 1;
        a.splits = pl.fc2_splits;
        a.slot_out = w.slot_out;
    }
    if (!ok) return cudaErrorInvalidValue;
    const int cta = moe_cta_group(pl);
    const int nkb = int(a.K / kFK);
    a.kb_per_split = (nkb + a.splits - 1) / a.splits;
    a.fc1 = fc1 ? 1 : 0;
    a.srows = pl.srows;
    a.tiles = w.tiles;
    a.perm = w.perm;
    a.slots = pl.slots;
    const int64_t rows_per_item = (a.paired ? kFM : 2 * kFM) * cta;
    a.n_pairs = int((a.N + rows_per_item - 1) / rows_per_item);
    a.gm = 1;
    for (int g = 8; g > 1; --g)
        if (a.n_pairs % g == 0) { a.gm = g; break; }
    a.stage_bytes = kFABytes + b_rows_per_cta(pl.bmax, cta) * 128u;
    a.stages = ring_stages(a.stage_bytes);
    a.act = p.act;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.has_limit = p.has_limit;
    a.limit = p.limit;
    a.err = w.ctrl;
    a.wait_ns = wait_limit_ns();
    const size_t smem = 1024 + size_t(a.stages) * a.stage_bytes;
    const int64_t items_max = pl.max_tiles * a.n_pairs * a.splits;
    cudaError_t e;
    note_launch(fc1 ? QMOE_KERNEL_FC1 : QMOE_KERNEL_FC2, s, true);
    if (cta == 2) {
        // token rows through TMA: {32 floats, srows, K/32}, boxes of kFBBox rows, copied as
        // stored (the rows carry their swizzle already)
        const uint64_t dims[3] = {32, uint64_t(pl.srows), uint64_t(a.K / kFK)};
        const uint64_t strides[2] = {128, uint64_t(pl.srows) * 128};
        const uint32_t box[3] = {32, uint32_t(kFBBox), 1};
        if (!encode_tmap_3d(&a.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.xs, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        if ((e = cudaFuncSetAttribute(moe_tf32_kernel<2>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) !=
            cudaSuccess)
            return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(kFThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * unsigned(device_sm_count() / 2));
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, moe_tf32_kernel<2>, &cfg) != cudaSuccess ||
            clusters <= 0) {
            cudaGetLastError();
            clusters = device_sm_count() / 2;
        }
        clusters = int(std::max<int64_t>(1, std::min<int64_t>(items_max, clusters)));
        cfg.gridDim = dim3(2 * unsigned(clusters));
        e = cudaLaunchKernelEx(&cfg, moe_tf32_kernel<2>, a);
    } else {
        if ((e = cudaFuncSetAttribute(moe_tf32_kernel<1>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))) !=
            cudaSuccess)
            return e;
        const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items_max, device_sm_count())));
        moe_tf32_kernel<1><<<grid, kFThreads, smem, s>>>(a);
        e = cudaSuccess;
    }
    note_launch(fc1 ? QMOE_KERNEL_FC1 : QMOE_KERNEL_FC2, s, false);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmoe
