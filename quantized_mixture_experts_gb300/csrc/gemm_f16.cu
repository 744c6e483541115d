// GroupedMatMul on the 5th-generation tensor cores, for f16 and bf16, and for
// f32 as three TF32 products per step (see gmm_f32_kernel below).
//
// GroupedMatMul-29 (Summary): output[m, i, :] = input[m, :] @ weights[g] (+ bias[g]),
// g = group_indices[m, i].  The (m, i) rows are grouped by g (stable, as the
// layer groups its slots by expert), each group's rows are gathered into token
// tiles of up to 256 rows, and one work item computes D[128 output columns x 2,
// tile rows] = W[g]^T * X^T with tcgen05.mma (fp32 accumulators in TMEM):
//
//   warp 0      TMA producer: per 64-wide K stage, the two 128-column weight
//               tiles as four 64 x 64 boxes of weights[g] (N-contiguous rows of
//               K, 128-byte swizzle: the MN-major A operand, read by the MMA as
//               is) and the token tile as one 1-D bulk copy of the gathered rows
//               (K-blocked, 128-byte swizzle pre-applied);
//   warp 1      TMEM allocator and MMA issuer (one lane);
//   warps 2-9   epilogue: tcgen05.ld, + bias, conversion to T, rows staged in
//               shared memory and stored as whole 16-byte pieces.
// Rows whose index is outside [0, G) form an extra group G: the grouping pass
// writes their output rows as zeros and records QMOE_DEVERR_INDEX, and no item
// covers them.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "ptx.cuh"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr int kGM = 128;                 // output columns per MMA (M)
constexpr int kGPair = 2;                // column tiles per item (share the token tile)
constexpr int kGMaxN = 256;              // token rows per tile (MMA N upper bound)
constexpr int kGK = 64;                  // K per stage
constexpr int kGStages = 3;              // load ring
constexpr int kGEpiWarps = 8;
constexpr int kGThreads = 32 * (2 + kGEpiWarps);
constexpr uint32_t kGBox = 64 * 128;     // one 64 (N) x 64 (K) box of 16-bit values
constexpr uint32_t kGABytes = kGPair * 2 * kGBox;   // weights per stage
constexpr uint32_t kGBBytes = kGMaxN * 128;         // token tile per stage
constexpr uint32_t kGStageBytes = kGABytes + kGBBytes;
constexpr uint32_t kGEpiBytes = 32 * 32 * 2;        // per epilogue warp: 32 tokens x 32 columns
constexpr int kGMaxGroups = 8191;        // G + 1 counters in shared memory while ranking
constexpr unsigned kFull = 0xffffffffu;
constexpr uint64_t kDrainWaitNs = 200000000ull;

struct GmmArgs {
    CUtensorMap tm_w;          // weights [G][K][N], boxes {64, 64, 1}, 128-byte swizzle
    const uint16_t* xs;        // gathered rows, K-blocked [K/64][srows][64], pre-swizzled
    int64_t srows;
    const int32_t* tiles;      // header + (group, first sorted row, rows, 0)
    const int32_t* perm;       // sorted position -> flattened row m * S + i
    const uint16_t* bias;      // [G, N] or null
    uint16_t* out;             // [M * S, N]
    int64_t N, K, G;
    int n_pairs, gm, bf16;
    int32_t* err;
    uint64_t wait_ns;
};

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor with the 128-byte swizzle.  K-major (the token
// tile): 8-row atoms 1024 bytes apart.  MN-major (the weight tile): 64-element
// rows of N along K, atoms of 8 K rows 1024 bytes apart (stride byte offset),
// the next 64 columns of N `lbo` bytes further (leading byte offset).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo) {
    uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t(1024 >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor: 16-bit A and B (f16 or bf16), fp32 accumulator,
// A MN-major (transposed), B K-major, M x N.
__device__ __forceinline__ uint32_t gmm_idesc(int m, int n, int bf16) {
    const uint32_t fmt = bf16 ? 1u : 0u;
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 15) | (uint32_t(n >> 3) << 17) |
           (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(ptx::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            int32_t z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(ptx::smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(ptx::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float load16(uint16_t v, int bf16) {
    return bf16 ? __bfloat162float(__ushort_as_bfloat16(v)) : __half2float(__ushort_as_half(v));
}
__device__ __forceinline__ uint16_t store16(float v, int bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

struct GItem {
    int g, row0, rows, n0, nt;   // group, first sorted row, rows, first output column, MMA N
};

__device__ __forceinline__ GItem gmm_item(const GmmArgs& a, int64_t i, int ntiles) {
    // batches of gm column pairs; inside a batch, token tile by token tile
    const int64_t per_group = int64_t(ntiles) * a.gm;
    const int pg = int(i / per_group);
    const int64_t rem = i % per_group;
    const int tau = int(rem / a.gm);
    const int pm = int(rem % a.gm);
    const int32_t* t = a.tiles + kTileHeader + 4 * tau;
    GItem it;
    it.g = t[0];
    it.row0 = t[1];
    it.rows = t[2];
    it.n0 = (pg * a.gm + pm) * kGPair * kGM;
    it.nt = (it.rows + 15) & ~15;
    return it;
}

__global__ void __launch_bounds__(kGThreads, 1) gmm_tc_kernel(const __grid_constant__ GmmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t load_full[kGStages];
    __shared__ __align__(8) uint64_t load_empty[kGStages];
    __shared__ __align__(8) uint64_t acc_full;
    __shared__ __align__(8) uint64_t acc_empty;
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            ptx::mbar_init(&load_full[s], 1);
            ptx::mbar_init(&load_empty[s], 1);
        }
        ptx::mbar_init(&acc_full, 1);
        ptx::mbar_init(&acc_empty, kGEpiWarps);
        ptx::mbar_init(&drain_bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(ptx::smem_u32(&tmem_base_s)), "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    const int ntiles = a.tiles[0];
    const int64_t items = int64_t(ntiles) * a.n_pairs;
    const int nkb = int(a.K / kGK);
    const uint32_t sbase = ptx::smem_u32(smem);

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) ptx::prefetch_tmap(&a.tm_w);
        uint32_t it = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const GItem w = gmm_item(a, i, ntiles);
            if (w.g >= a.G) continue;   // rows with an invalid index (already zeroed)
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % kGStages);
                if (!ptx::mbar_wait(&load_empty[sl], ((it / kGStages) & 1u) ^ 1u, a.wait_ns,
                                    &abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint8_t* sp = smem + size_t(sl) * kGStageBytes;
                    ptx::mbar_arrive_expect_tx(&load_full[sl], kGABytes + uint32_t(w.nt) * 128u);
#pragma unroll
                    for (int b = 0; b < kGPair * 2; ++b)   // tile b / 2, columns half b % 2
                        tma_load_3d(sp + b * kGBox, &a.tm_w, w.n0 + b * 64, kb * kGK, w.g,
                                    &load_full[sl]);
                    ptx::bulk_g2s(sp + kGABytes, a.xs + (int64_t(kb) * a.srows + w.row0) * kGK,
                                  uint32_t(w.nt) * 128u, &load_full[sl]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
            abort_flag = 1;
            for (uint32_t j = it > kGStages ? it - kGStages : 0; j < it; ++j) {
                volatile int never = 0;
                ptx::mbar_wait(&load_full[j % kGStages], (j / kGStages) & 1u, kDrainWaitNs, &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer -------------------------------
        uint32_t it = 0, item_it = 0;
        bool ok = true, issued = false;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const GItem w = gmm_item(a, i, ntiles);
            if (w.g >= a.G) continue;
            if (!ptx::mbar_wait(&acc_empty, (item_it & 1u) ^ 1u, a.wait_ns, &abort_flag)) {
                ok = false;
                break;
            }
            ++item_it;
            tc_fence_after();
            const uint32_t idesc = gmm_idesc(kGM, w.nt, a.bf16);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % kGStages);
                if (!ptx::mbar_wait(&load_full[sl], (it / kGStages) & 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = sbase + uint32_t(sl) * kGStageBytes;
                    const uint32_t sb = sa + kGABytes;
#pragma unroll
                    for (int kk = 0; kk < kGK / 16; ++kk) {
                        const uint64_t bd = sw128_desc(sb + 32u * kk, 16u);
#pragma unroll
                        for (int t = 0; t < kGPair; ++t)
                            mma_ss(tmem_base + uint32_t(t * kGMaxN),
                                   sw128_desc(sa + uint32_t(t) * 2u * kGBox + 2048u * kk, kGBox), bd,
                                   idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&load_empty[sl]);
                    issued = true;
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(&acc_full);
            __syncwarp();
        }
        if (!ok && lane == 0) {
            atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
            abort_flag = 1;
        }
        if (lane == 0 && issued) {
            mma_commit(&drain_bar);
            volatile int never = 0;
            ptx::mbar_wait(&drain_bar, 0, kDrainWaitNs, &never);
        }
        __syncwarp();
    } else {
        // -------------------------------- epilogue --------------------------------
        const int ew = warp - 2;                   // 0..7
        const int tile = ew / 4;                   // column tile of the item
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        uint16_t* stile = reinterpret_cast<uint16_t*>(smem + kGStages * kGStageBytes +
                                                      uint32_t(ew) * kGEpiBytes);
        uint32_t item_it = 0;
        for (int64_t i = blockIdx.x; i < items; i += gridDim.x) {
            const GItem w = gmm_item(a, i, ntiles);
            if (w.g >= a.G) continue;
            const uint32_t aph = item_it & 1u;
            ++item_it;
            // each lane's row of every 32-row chunk, fetched before the accumulator
            int row_c[kGMaxN / 32];
#pragma unroll
            for (int ch = 0; ch < kGMaxN / 32; ++ch) {
                const int col = ch * 32 + lane;
                row_c[ch] = col < w.rows ? __ldg(a.perm + w.row0 + col) : 0;
            }
            const int64_t nbase = int64_t(w.n0) + tile * kGM + quad * 32;   // this warp's columns
            const int64_t n = nbase + lane;                                  // this lane's column
            const float bv = (a.bias && n < a.N) ? load16(a.bias[int64_t(w.g) * a.N + n], a.bf16) : 0.f;
            if (!ptx::mbar_wait(&acc_full, aph, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
                    abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(tile * kGMaxN);
            for (int c0 = 0; c0 < w.nt; c0 += 32) {
                float v[32];
                tmem_ld32(tbase + uint32_t(c0), v);
#pragma unroll
                for (int q = 0; q < 32; ++q) stile[q * 32 + lane] = store16(v[q] + bv, a.bf16);
                __syncwarp();
                int my_row = 0;
#pragma unroll
                for (int ch = 0; ch < kGMaxN / 32; ++ch)   // registers: select, not index
                    if (ch * 32 == c0) my_row = row_c[ch];
                if (c0 + lane < w.rows && nbase < a.N) {
                    uint16_t* dst = a.out + int64_t(my_row) * a.N + nbase;
                    const uint16_t* src = stile + lane * 32;
                    if (nbase + 32 <= a.N) {
#pragma unroll
                        for (int h = 0; h < 4; ++h)
                            reinterpret_cast<uint4*>(dst)[h] = reinterpret_cast<const uint4*>(src)[h];
                    } else {
                        for (int j = 0; j < int(a.N - nbase); ++j) dst[j] = src[j];
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(512)
                     : "memory");
}

// Validates the indices of one chunk of kRouteTokensPerChunk input rows (S
// indices each), ranks its rows stably by group and writes the chunk's
// histogram.  An index outside [0, G) joins group G: its output row is zeroed
// here and the device error word records QMOE_DEVERR_INDEX.
template <typename TI>
__global__ void __launch_bounds__(256) gmm_rank_kernel(const TI* __restrict__ idx, int64_t M,
                                                       int64_t S, int64_t G, int64_t N,
                                                       int32_t* __restrict__ sel,
                                                       int32_t* __restrict__ rank,
                                                       int32_t* __restrict__ hist,
                                                       uint16_t* __restrict__ out,
                                                       int32_t* __restrict__ err) {
    // N counts 16-bit units of an output row (2 per element for f32)
    extern __shared__ int32_t s_cnt[];   // [G + 1]
    const int E = int(G) + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = int64_t(blockIdx.x) * kRouteTokensPerChunk * S;
    const int64_t r_end = r0 + kRouteTokensPerChunk * S;
    const int64_t r1 = r_end < M * S ? r_end : M * S;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        const int64_t g = int64_t(idx[r]);
        const bool bad = g < 0 || g >= G;
        sel[r] = bad ? int32_t(G) : int32_t(g);
        if (bad) {
            atomicCAS(err, 0, int32_t(QMOE_DEVERR_INDEX));
            for (int64_t n = 0; n < N; ++n) out[r * N + n] = 0;
        }
    }
    __syncthreads();
    if (warp == 0) {
        for (int64_t base = r0; base < r1; base += 32) {
            const int64_t r = base + lane;
            const int e = r < r1 ? sel[r] : -1 - lane;   // distinct dummies
            const unsigned mask = __match_any_sync(kFull, e);
            const int leader = __ffs(mask) - 1;
            const int rk = __popc(mask & ((1u << lane) - 1u));
            int c = (lane == leader && e >= 0) ? s_cnt[e] : 0;
            c = __shfl_sync(kFull, c, leader);
            if (e >= 0) rank[r] = c + rk;
            __syncwarp();
            if (lane == leader && e >= 0) s_cnt[e] = c + __popc(mask);
            __syncwarp();
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[int64_t(blockIdx.x) * E + e] = s_cnt[e];
}

// The input rows in group-sorted order, K-blocked [K/64][srows][64] with the
// 128-byte swizzle of each row's position in its token tile applied (tiles
// start at multiples of 256 rows of their group).  One warp per sorted row.
__global__ void gmm_gather_kernel(const uint4* __restrict__ x, int row_vec,
                                  const int32_t* __restrict__ perm, const int32_t* __restrict__ sel,
                                  const int32_t* __restrict__ offsets, int64_t S, int64_t R,
                                  int G, int64_t srows, uint4* __restrict__ xs) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * wpb;
    for (int64_t pos = int64_t(blockIdx.x) * wpb + (threadIdx.x >> 5); pos < R; pos += nwarps) {
        const int32_t r = __ldg(perm + pos);
        const int g = __ldg(sel + r);
        if (g >= G) continue;
        const int phase = int(pos - __ldg(offsets + g)) & 7;
        const uint4* __restrict__ src = x + int64_t(r / S) * row_vec;
        for (int q = lane; q < row_vec; q += 32)
            xs[(int64_t(q >> 3) * srows + pos) * 8 + ((q & 7) ^ phase)] = __ldg(src + q);
    }
}

// ---------------------------------------------------------------------------
// f32: three TF32 products per K step.  With x = x_hi + x_lo and w = w_hi + w_lo
// split at the TF32 precision (hi = x rounded to TF32, lo = x - hi rounded to
// TF32), x * w is x_hi w_hi + x_lo w_hi + x_hi w_lo up to about 2^-21 |x w|;
// the three products accumulate in fp32 in tensor memory.  TF32 operands are
// K-major, so the weight tile ([K][N] rows, N contiguous) is transposed in shared
// memory on the way.  One work item = (token tile of up to 128 rows of one
// group, 128 output columns); per CTA:
//   warp 0      TMA producer: per 32-wide K stage, the weight tile as four
//               32 (N) x 32 (K) boxes (128-byte swizzle) and the two planes of
//               the token tile (x_hi, x_lo) as 1-D bulk copies;
//   warp 1      TMEM allocator and MMA issuer (one lane): tcgen05.mma kind::tf32;
//   warps 2-5   split: one thread per output column reads its 32 weights of
//               the stage and writes w_hi and w_lo as K-major 128-byte rows
//               (128-byte swizzle), the layout of the token planes;
//   warps 6-9   epilogue: tcgen05.ld, + bias, fp32 rows stored whole.
// ---------------------------------------------------------------------------
constexpr int kFM = 128;                 // output columns per item (M)
constexpr int kFMaxN = 128;              // token rows per tile (MMA N upper bound)
constexpr int kFK = 32;                  // K per stage: one 128-byte row of fp32
constexpr int kFStages = 2;
constexpr int kFSplitWarps = 4;
constexpr int kFEpiWarps = 4;
constexpr int kFThreads = 32 * (2 + kFSplitWarps + kFEpiWarps);
constexpr uint32_t kFBox = 32 * 128;               // one 32 (N) x 32 (K) fp32 box
constexpr uint32_t kFATile = 4 * kFBox;            // 128 x 32 fp32 (16 KB)
constexpr uint32_t kFBPlane = kFMaxN * 128;        // one plane of the token tile per stage
// stage: weights as loaded | w_hi | w_lo (K-major) | x_hi | x_lo
constexpr uint32_t kFOffHi = kFATile, kFOffLo = 2 * kFATile, kFOffB = 3 * kFATile;
constexpr uint32_t kFStageBytes = 3 * kFATile + 2 * kFBPlane;
constexpr uint32_t kFEpiBytes = 32 * 32 * 4;       // per epilogue warp: 32 rows x 32 columns

struct GmmF32Args {
    CUtensorMap tm_w;          // weights [G][K][N] fp32, boxes {32, 32, 1}, 128-byte swizzle
    const float* xs;           // two planes, each K-blocked [K/32][srows][32], pre-swizzled
    int64_t plane;             // floats per plane
    int64_t srows;
    const int32_t* tiles;
    const int32_t* perm;
    const float* bias;         // [G, N] or null
    float* out;                // [M * S, N]
    int64_t N, K, G;
    int n_mt, gm;
    int32_t* err;
    uint64_t wait_ns;
};

// Nearest TF32 value of v (ties away from zero), as an fp32 bit pattern.
__device__ __forceinline__ float tf32_round(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// Instruction descriptor: TF32 A and B (both K-major), fp32 accumulator, M x N.
__device__ __forceinline__ uint32_t f32_idesc(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct FItem {
    int g, row0, rows, n0, nt;
};

__device__ __forceinline__ FItem gmm_f32_item(const GmmF32Args& a, int64_t i, int ntiles) {
    // batches of gm column tiles; inside a batch, token tile by token tile
    const int64_t per_group = int64_t(ntiles) * a.gm;
    const int pg = int(i / per_group);
    const int64_t rem = i % per_group;
    const int tau = int(rem / a.gm);
    const int pm = int(rem % a.gm);
    const int32_t* t = a.tiles + kTileHeader + 4 * tau;
    FItem it;
    it.g = t[0];
    it.row0 = t[1];
    it.rows = t[2];
    it.n0 = (pg * a.gm + pm) * kFM;
    it.nt = (it.rows + 15) & ~15;
    return it;
}

__global__ void __launch_bounds__(kFThreads, 1) gmm_f32_kernel(const __grid_constant__ GmmF32Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t load_full[kFStages];
    __shared__ __align__(8) uint64_t lo_full[kFStages];
    __shared__ __align__(8) uint64_t load_empty[kFStages];
    __shared__ __align__(8) uint64_t acc_full;
    __shared__ __align__(8) uint64_t acc_empty;
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kFStages; ++s) {
            ptx::mbar_init(&load_full[s], 1);
            ptx::mbar_init(&lo_full[s], kFSplitWarps);
            ptx::mbar_init(&load_empty[s], 1);
        }
        ptx::mbar_init(&acc_full, 1);
        ptx::mbar_init(&acc_empty, kFEpiWarps);
        ptx::mbar_init(&drain_bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(ptx::smem_u32(&tmem_base_s)), "r"(128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;
    const int ntiles = a.tiles[0];
    const int64_t items = int64_t(ntiles) * a.n_mt;
    const int nkb = int(a.K / kFK);
    const uint32_t sbase = ptx::smem_u32(smem);

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) ptx::prefetch_tmap(&a.tm_w);
        uint32_t it = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const FItem w = gmm_f32_item(a, i, ntiles);
            if (w.g >= a.G) continue;   // rows with an invalid index (already zeroed)
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % kFStages);
                if (!ptx::mbar_wait(&load_empty[sl], ((it / kFStages) & 1u) ^ 1u, a.wait_ns,
                                    &abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    uint8_t* sp = smem + size_t(sl) * kFStageBytes;
                    ptx::mbar_arrive_expect_tx(&load_full[sl], kFATile + 2u * uint32_t(w.nt) * 128u);
#pragma unroll
                    for (int b = 0; b < 4; ++b)   // columns n0 + 32 b .. n0 + 32 b + 31
                        tma_load_3d(sp + b * kFBox, &a.tm_w, w.n0 + b * 32, kb * kFK, w.g,
                                    &load_full[sl]);
                    const float* xb = a.xs + (int64_t(kb) * a.srows + w.row0) * kFK;
                    ptx::bulk_g2s(sp + kFOffB, xb, uint32_t(w.nt) * 128u, &load_full[sl]);
                    ptx::bulk_g2s(sp + kFOffB + kFBPlane, xb + a.plane, uint32_t(w.nt) * 128u,
                                  &load_full[sl]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
            abort_flag = 1;
            for (uint32_t j = it > kFStages ? it - kFStages : 0; j < it; ++j) {
                volatile int never = 0;
                ptx::mbar_wait(&load_full[j % kFStages], (j / kFStages) & 1u, kDrainWaitNs, &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer -------------------------------
        uint32_t it = 0, item_it = 0;
        bool ok = true, issued = false;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const FItem w = gmm_f32_item(a, i, ntiles);
            if (w.g >= a.G) continue;
            if (!ptx::mbar_wait(&acc_empty, (item_it & 1u) ^ 1u, a.wait_ns, &abort_flag)) {
                ok = false;
                break;
            }
            ++item_it;
            tc_fence_after();
            const uint32_t idesc = f32_idesc(kFM, w.nt);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % kFStages);
                // the split warps arrive after the stage's copies landed
                if (!ptx::mbar_wait(&lo_full[sl], (it / kFStages) & 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sp = sbase + uint32_t(sl) * kFStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kFK / 8; ++kk) {   // K = 8 per MMA: 32 bytes of a row
                        const uint64_t ah = sw128_desc(sp + kFOffHi + 32u * kk, 16u);
                        const uint64_t al = sw128_desc(sp + kFOffLo + 32u * kk, 16u);
                        const uint64_t bh = sw128_desc(sp + kFOffB + 32u * kk, 16u);
                        const uint64_t bl = sw128_desc(sp + kFOffB + kFBPlane + 32u * kk, 16u);
                        mma_tf32(tmem_base, ah, bh, idesc, (kb | kk) != 0 ? 1u : 0u);
                        mma_tf32(tmem_base, ah, bl, idesc, 1u);
                        mma_tf32(tmem_base, al, bh, idesc, 1u);
                    }
                    mma_commit(&load_empty[sl]);
                    issued = true;
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(&acc_full);
            __syncwarp();
        }
        if (!ok && lane == 0) {
            atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
            abort_flag = 1;
        }
        if (lane == 0 && issued) {
            mma_commit(&drain_bar);
            volatile int never = 0;
            ptx::mbar_wait(&drain_bar, 0, kDrainWaitNs, &never);
        }
        __syncwarp();
    } else if (warp < 2 + kFSplitWarps) {
        // --------------------------------- split ----------------------------------
        const int n = threadIdx.x - 64;            // output column of the tile (0..127)
        uint32_t it = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const FItem w = gmm_f32_item(a, i, ntiles);
            if (w.g >= a.G) continue;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % kFStages);
                if (!ptx::mbar_wait(&load_full[sl], (it / kFStages) & 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sp = ptx::launder(sbase + uint32_t(sl) * kFStageBytes);
                // element (k, n) of the loaded tile: box n / 32, row k, 16-byte piece
                // (n % 32) / 4 stored at piece ^ (k % 8), word n % 4
                const uint32_t src = sp + uint32_t(n >> 5) * kFBox + uint32_t(n & 3) * 4u;
                const uint32_t piece = uint32_t((n & 31) >> 2);
                const uint32_t dhi = sp + kFOffHi + uint32_t(n) * 128u;
                const uint32_t dlo = sp + kFOffLo + uint32_t(n) * 128u;
#pragma unroll
                for (int c = 0; c < kFK / 4; ++c) {   // K 4c .. 4c + 3 -> piece c of row n
                    float hv[4], lv[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t k = uint32_t(4 * c + j);
                        const float v = ptx::ld_f32(src + k * 128u + ((piece ^ (k & 7u)) << 4));
                        hv[j] = tf32_round(v);
                        lv[j] = tf32_round(v - hv[j]);
                    }
                    const uint32_t o = (uint32_t(c) ^ uint32_t(n & 7)) << 4;
                    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(dhi + o), "f"(hv[0]),
                                 "f"(hv[1]), "f"(hv[2]), "f"(hv[3])
                                 : "memory");
                    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(dlo + o), "f"(lv[0]),
                                 "f"(lv[1]), "f"(lv[2]), "f"(lv[3])
                                 : "memory");
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&lo_full[sl]);
            }
        }
        if (!ok && lane == 0) {
            atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
            abort_flag = 1;
        }
    } else {
        // -------------------------------- epilogue --------------------------------
        const int quad = warp & 3;                 // TMEM lane quadrant = 32 output columns
        const int ew = warp - 2 - kFSplitWarps;    // 0..3
        float* stile = reinterpret_cast<float*>(smem + kFStages * kFStageBytes + uint32_t(ew) * kFEpiBytes);
        uint32_t item_it = 0;
        for (int64_t i = blockIdx.x; i < items; i += gridDim.x) {
            const FItem w = gmm_f32_item(a, i, ntiles);
            if (w.g >= a.G) continue;
            const uint32_t aph = item_it & 1u;
            ++item_it;
            int row_c[kFMaxN / 32];
#pragma unroll
            for (int ch = 0; ch < kFMaxN / 32; ++ch) {
                const int col = ch * 32 + lane;
                row_c[ch] = col < w.rows ? __ldg(a.perm + w.row0 + col) : 0;
            }
            const int64_t nbase = int64_t(w.n0) + quad * 32;   // this warp's columns
            const int64_t n = nbase + lane;
            const float bv = (a.bias && n < a.N) ? __ldg(a.bias + int64_t(w.g) * a.N + n) : 0.f;
            if (!ptx::mbar_wait(&acc_full, aph, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    atomicCAS(a.err, 0, int32_t(QMOE_DEVERR_TIMEOUT));
                    abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (uint32_t(quad * 32) << 16);
            for (int c0 = 0; c0 < w.nt; c0 += 32) {
                float v[32];
                tmem_ld32(tbase + uint32_t(c0), v);
                // lane = output column n; v[q] = token row c0 + q: transpose through the
                // staging tile (row-major 32 x 32, column index rotated by the row)
#pragma unroll
                for (int q = 0; q < 32; ++q) stile[q * 32 + ((lane + q) & 31)] = v[q] + bv;
                __syncwarp();
                int my_row = 0;
#pragma unroll
                for (int ch = 0; ch < kFMaxN / 32; ++ch)
                    if (ch * 32 == c0) my_row = row_c[ch];
                if (c0 + lane < w.rows && nbase < a.N) {
                    float* dst = a.out + int64_t(my_row) * a.N + nbase;
                    const float* src = stile + lane * 32;
                    if (nbase + 32 <= a.N) {
#pragma unroll
                        for (int h = 0; h < 8; ++h) {
                            float4 o;
                            o.x = src[(4 * h + 0 + lane) & 31];
                            o.y = src[(4 * h + 1 + lane) & 31];
                            o.z = src[(4 * h + 2 + lane) & 31];
                            o.w = src[(4 * h + 3 + lane) & 31];
                            reinterpret_cast<float4*>(dst)[h] = o;
                        }
                    } else {
                        for (int j = 0; j < int(a.N - nbase); ++j) dst[j] = src[(j + lane) & 31];
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(128)
                     : "memory");
}

// The input rows in group-sorted order as two TF32 planes (x_hi, x_lo), each
// K-blocked [K/32][srows][32] with the 128-byte swizzle of each row's position in
// its token tile applied.  One warp per sorted row.
__global__ void gmm_gather_f32_kernel(const float4* __restrict__ x, int row_vec,
                                      const int32_t* __restrict__ perm,
                                      const int32_t* __restrict__ sel,
                                      const int32_t* __restrict__ offsets, int64_t S, int64_t R,
                                      int G, int64_t srows, int64_t plane4,
                                      float4* __restrict__ xs) {
    const int lane = threadIdx.x & 31;
    const int64_t wpb = blockDim.x >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * wpb;
    for (int64_t pos = int64_t(blockIdx.x) * wpb + (threadIdx.x >> 5); pos < R; pos += nwarps) {
        const int32_t r = __ldg(perm + pos);
        const int g = __ldg(sel + r);
        if (g >= G) continue;
        const int phase = int(pos - __ldg(offsets + g)) & 7;
        const float4* __restrict__ src = x + int64_t(r / S) * row_vec;
        for (int q = lane; q < row_vec; q += 32) {
            const float4 v = __ldg(src + q);
            float4 hi, lo;
            hi.x = tf32_round(v.x); lo.x = tf32_round(v.x - hi.x);
            hi.y = tf32_round(v.y); lo.y = tf32_round(v.y - hi.y);
            hi.z = tf32_round(v.z); lo.z = tf32_round(v.z - hi.z);
            hi.w = tf32_round(v.w); lo.w = tf32_round(v.w - hi.w);
            const int64_t o = (int64_t(q >> 3) * srows + pos) * 8 + ((q & 7) ^ phase);
            xs[o] = hi;
            xs[o + plane4] = lo;
        }
    }
}

struct GmmPlan {
    int64_t R, chunks, srows, max_tiles;
    size_t off_sel, off_rank, off_perm, off_inv, off_hist, off_counts, off_offsets, off_tiles,
        off_active, off_xs, bytes;
};

GmmPlan gmm_plan(int64_t M, int64_t K, int64_t G, int64_t S, int xs_bytes_per_elem = 2,
                 int tile_rows = kGMaxN) {
    GmmPlan q;
    q.R = M * S;
    q.chunks = (M + kRouteTokensPerChunk - 1) / kRouteTokensPerChunk;
    q.srows = (q.R + 15) / 16 * 16 + 16;
    q.max_tiles = (q.R + tile_rows - 1) / tile_rows + G + 1;
    size_t off = 256;   // device error word
    auto take = [&](size_t b) {
        const size_t o = off;
        off = (off + std::max<size_t>(b, 1) + 255) / 256 * 256;
        return o;
    };
    const size_t E = size_t(G) + 1;
    q.off_sel = take(4 * size_t(q.R));
    q.off_rank = take(4 * size_t(q.R));
    q.off_perm = take(4 * size_t(q.R));
    q.off_inv = take(4 * size_t(q.R));
    q.off_hist = take(4 * size_t(q.chunks) * E);
    q.off_counts = take(4 * E);
    q.off_offsets = take(4 * (E + 1));
    q.off_tiles = take(4 * size_t(kTileHeader + 4 * q.max_tiles));
    q.off_active = take(4 * E);
    q.off_xs = take(size_t(xs_bytes_per_elem) * size_t(K) * size_t(q.srows));
    q.bytes = off;
    return q;
}

// f32: the gather into TF32 planes and the three-product GEMM (after the grouping).
cudaError_t launch_gmm_f32(const void* input, int64_t M, int64_t K, const void* weights, int64_t G,
                           int64_t N, int64_t S, const void* bias, void* out, int32_t* err,
                           const int32_t* perm, const int32_t* sel, const int32_t* offsets,
                           const int32_t* tiles, int64_t R, int64_t srows, int64_t max_tiles,
                           float* xs, int blocks, cudaStream_t s) {
    (void)M;
    const int64_t plane = K * srows;   // floats per plane
    gmm_gather_f32_kernel<<<std::max(blocks, 1), 256, 0, s>>>(
        static_cast<const float4*>(input), int(K / 4), perm, sel, offsets, S, R, int(G), srows,
        plane / 4, reinterpret_cast<float4*>(xs));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    GmmF32Args a;
    std::memset(&a, 0, sizeof(a));
    const uint64_t dims[3] = {uint64_t(N), uint64_t(K), uint64_t(G)};
    const uint64_t strides[2] = {uint64_t(N) * 4, uint64_t(K) * uint64_t(N) * 4};
    const uint32_t box[3] = {32, kFK, 1};
    if (!encode_tmap_3d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, weights, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    a.xs = xs;
    a.plane = plane;
    a.srows = srows;
    a.tiles = tiles;
    a.perm = perm;
    a.bias = static_cast<const float*>(bias);
    a.out = static_cast<float*>(out);
    a.N = N;
    a.K = K;
    a.G = G;
    a.n_mt = int((N + kFM - 1) / kFM);
    a.gm = 1;
    for (int g = 8; g > 1; --g)
        if (a.n_mt % g == 0) { a.gm = g; break; }
    a.err = err;
    a.wait_ns = wait_limit_ns();
    const size_t smem = 1024 + size_t(kFStages) * kFStageBytes + size_t(kFEpiWarps) * kFEpiBytes;
    if ((e = cudaFuncSetAttribute(gmm_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem))) != cudaSuccess)
        return e;
    const int64_t items_max = max_tiles * a.n_mt;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items_max, device_sm_count())));
    note_launch(-1, s, false, 4);   // ranking, the two grouping launches, the gather
    note_launch(QMOE_KERNEL_GMM, s, true);
    gmm_f32_kernel<<<grid, kFThreads, smem, s>>>(a);
    note_launch(QMOE_KERNEL_GMM, s, false, 1);
    return cudaGetLastError();
}

}  // namespace

size_t grouped_matmul_tc_workspace(int64_t M, int64_t K, int64_t G, int64_t N, int64_t S,
                                   int dtype) {
    if (M <= 0 || S <= 0 || N <= 0 || G <= 0 || K <= 0) return 0;
    if (M * S > (int64_t(1) << 30) || G * K * N >= (int64_t(1) << 46) || G > kGMaxGroups) return 0;
    if (dtype == QMOE_DT_F32) {
        if (K % kFK != 0 || N % 4 != 0) return 0;
        return gmm_plan(M, K, G, S, 8, kFMaxN).bytes;   // x_hi and x_lo planes, 128-row tiles
    }
    if (dtype != QMOE_DT_F16 && dtype != QMOE_DT_BF16) return 0;
    if (K % kGK != 0 || N % 8 != 0) return 0;
    return gmm_plan(M, K, G, S).bytes;
}

cudaError_t launch_grouped_matmul_tc(const void* input, int64_t M, int64_t K, const void* weights,
                                     int64_t G, int64_t N, const void* idx, int64_t S, int idx64,
                                     const void* bias, void* out, int dtype, void* workspace,
                                     cudaStream_t s) {
    const bool f32 = dtype == QMOE_DT_F32;
    const GmmPlan pl = gmm_plan(M, K, G, S, f32 ? 8 : 2, f32 ? kFMaxN : kGMaxN);
    char* b = static_cast<char*>(workspace);
    int32_t* err = reinterpret_cast<int32_t*>(b);
    int32_t* sel = reinterpret_cast<int32_t*>(b + pl.off_sel);
    int32_t* rank = reinterpret_cast<int32_t*>(b + pl.off_rank);
    int32_t* perm = reinterpret_cast<int32_t*>(b + pl.off_perm);
    int32_t* inv = reinterpret_cast<int32_t*>(b + pl.off_inv);
    int32_t* hist = reinterpret_cast<int32_t*>(b + pl.off_hist);
    int32_t* counts = reinterpret_cast<int32_t*>(b + pl.off_counts);
    int32_t* offsets = reinterpret_cast<int32_t*>(b + pl.off_offsets);
    int32_t* tiles = reinterpret_cast<int32_t*>(b + pl.off_tiles);
    int32_t* active = reinterpret_cast<int32_t*>(b + pl.off_active);
    uint16_t* xs = reinterpret_cast<uint16_t*>(b + pl.off_xs);
    const int E = int(G) + 1;
    cudaError_t e;
    // 1. group the (m, i) rows
    const size_t rank_smem = sizeof(int32_t) * size_t(E);
    if (rank_smem > 48 * 1024) {
        e = idx64 ? cudaFuncSetAttribute(gmm_rank_kernel<int64_t>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(rank_smem))
                  : cudaFuncSetAttribute(gmm_rank_kernel<int32_t>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(rank_smem));
        if (e != cudaSuccess) return e;
    }
    note_launch(-1, s, true);
    if (idx64)
        gmm_rank_kernel<int64_t><<<unsigned(pl.chunks), 256, rank_smem, s>>>(
            static_cast<const int64_t*>(idx), M, S, G, f32 ? 2 * N : N, sel, rank, hist,
            static_cast<uint16_t*>(out), err);
    else
        gmm_rank_kernel<int32_t><<<unsigned(pl.chunks), 256, rank_smem, s>>>(
            static_cast<const int32_t*>(idx), M, S, G, f32 ? 2 * N : N, sel, rank, hist,
            static_cast<uint16_t*>(out), err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_group_items(hist, pl.chunks, E, counts, offsets, tiles, active,
                                f32 ? kFMaxN : kGMaxN, sel, rank,
                                pl.R, int(S), perm, inv, s)) != cudaSuccess)
        return e;
    const int blocks = int(std::min<int64_t>((pl.R + 7) / 8, int64_t(device_sm_count()) * 8));
    if (f32) return launch_gmm_f32(input, M, K, weights, G, N, S, bias, out, err, perm, sel, offsets,
                                   tiles, pl.R, pl.srows, pl.max_tiles,
                                   reinterpret_cast<float*>(b + pl.off_xs), blocks, s);
    // 2. gather the input rows in group order
    const int row_vec = int(K / 8);
    gmm_gather_kernel<<<std::max(blocks, 1), 256, 0, s>>>(
        static_cast<const uint4*>(input), row_vec, perm, sel, offsets, S, pl.R, int(G), pl.srows,
        reinterpret_cast<uint4*>(xs));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. the grouped GEMM
    GmmArgs a;
    std::memset(&a, 0, sizeof(a));
    const uint64_t dims[3] = {uint64_t(N), uint64_t(K), uint64_t(G)};
    const uint64_t strides[2] = {uint64_t(N) * 2, uint64_t(K) * uint64_t(N) * 2};
    const uint32_t box[3] = {64, kGK, 1};
    if (!encode_tmap_3d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT16, weights, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    a.xs = xs;
    a.srows = pl.srows;
    a.tiles = tiles;
    a.perm = perm;
    a.bias = static_cast<const uint16_t*>(bias);
    a.out = static_cast<uint16_t*>(out);
    a.N = N;
    a.K = K;
    a.G = G;
    const int64_t n_mtiles = (N + kGM - 1) / kGM;
    a.n_pairs = int((n_mtiles + kGPair - 1) / kGPair);
    a.gm = 1;
    for (int g = 8; g > 1; --g)
        if (a.n_pairs % g == 0) { a.gm = g; break; }
    a.bf16 = dtype == QMOE_DT_BF16 ? 1 : 0;
    a.err = err;
    a.wait_ns = wait_limit_ns();
    const size_t smem = 1024 + size_t(kGStages) * kGStageBytes + size_t(kGEpiWarps) * kGEpiBytes;
    if ((e = cudaFuncSetAttribute(gmm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem))) != cudaSuccess)
        return e;
    const int64_t items_max = pl.max_tiles * a.n_pairs;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items_max, device_sm_count())));
    note_launch(-1, s, false, 4);   // ranking, the two grouping launches, the gather
    note_launch(QMOE_KERNEL_GMM, s, true);
    gmm_tc_kernel<<<grid, kGThreads, smem, s>>>(a);
    note_launch(QMOE_KERNEL_GMM, s, false, 1);
    return cudaGetLastError();
}

}  // namespace qmoe
