// Grouped path of the QMoE layer: expert-grouped GEMMs on the 5th-generation
// tensor cores (tcgen05) with TMEM accumulators.
//
// QMoE manifest passes QMoE.FC1ActivationStageGrouped / QMoE.OutputStageGrouped
// (tiles of one expert's routed tokens against that expert's weights,
// derive.groupMaxTiles) and GroupedMatMul-29 Summary (a runtime should fuse
// DequantizeLinear + GroupedMatMul so the dequantized [G, K, N] weights are
// never materialised).
//
// One work item = (token tile of one expert: up to 256 expert-sorted rows,
// 128-row weight tile).  The MMA computes D[128 weight rows, N tokens] =
// deq(W)[128, K] * X[N, K]^T with the weights as the A operand (M = 128) and
// the tokens as the B operand (N = tile rows rounded up to 16), so a sparsely
// routed expert costs a narrow MMA instead of a padded one.
//
// Per CTA (one per SM, persistent), warp-specialised:
//   warp 0      TMA producer: the weight tile's packed bytes for a 64-wide K
//               block and its block scales (2-D boxes; scales only when a new
//               group of four blocks starts) and the tile's token rows into a
//               3-stage ring.  The token rows are stored K-blocked with the
//               128-byte swizzle already applied, so one 1-D bulk copy of up to
//               32 KB lands the whole swizzled tile;
//   warp 1      TMEM allocator and MMA issuer (one lane): per stage four K = 16
//               steps of one tcgen05.mma per weight tile, into the item's two
//               256-column accumulators (one per weight tile; all 512 columns,
//               so the epilogue of an item precedes the next item's MMAs);
//   warps 2-9   dequantisers: packed codes -> (q - mid) * scale in fp16,
//               written to shared memory in the 128-byte-swizzled K-major
//               layout the MMA descriptor expects;
//   warps 10-17 epilogue: tcgen05.ld of the accumulator, FC1 ReLU / SwiGLU to
//               fp16 activations, FC2 rows per routing slot already multiplied
//               by the slot's routing weight (fp16; the combine adds a token's k
//               rows in fixed order).
// Every wait is a bounded mbarrier wait; on expiry the CTA records
// QMOE_DEVERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cstring>

#include "ptx.cuh"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr int kTcM = 128;            // weight rows per MMA (M)
constexpr int kPair = 2;             // weight tiles per work item (share one token tile)
constexpr int kItemRows = kPair * kTcM;
constexpr int kTcMaxN = 256;         // tokens per tile (MMA N upper bound)
constexpr int kTcK = 64;             // K per stage: one 128-byte row of fp16
constexpr int kLoadStages = 4;       // TMA ring depth upper bound (the launch picks what fits)
constexpr int kAStages = 2;          // ring of dequantised weight tiles
constexpr int kDeqWarps = 8;         // one thread per weight row of the item
constexpr int kEpiWarps = 8;         // two per TMEM lane quadrant (one per weight tile)
constexpr int kTcWarps = 2 + kDeqWarps + kEpiWarps;
constexpr int kTcThreads = 32 * kTcWarps;
constexpr int kAccCols = 256;        // TMEM columns per accumulator (one per weight tile)
constexpr uint32_t kTmemCols = kPair * kAccCols;
constexpr uint32_t kBBytes = kTcMaxN * 128;   // token tile, fp16, swizzled
constexpr uint32_t kABytes = kTcM * 128;      // one dequantised weight tile, fp16, swizzled
constexpr uint32_t kAStageBytes = kPair * kABytes;
constexpr unsigned kFull = 0xffffffffu;
// Bound on the waits that drain a CTA's own copies / MMAs before it exits after
// a timeout: independent of the (possibly tiny) configured wait limit.
constexpr uint64_t kDrainWaitNs = 200000000ull;

struct TcArgs {
    CUtensorMap tm_w;           // packed weights [E*N rows, K/pack bytes], box {64/pack, 256}
    CUtensorMap tm_s;           // block scales [E*N rows, nb] fp32, box {4, 256}
    const float* scales;        // [E*N, nb] (nb = 1 for column-wise)
    const int32_t* tiles;       // header + (expert, first sorted row, rows, 0)
    const int32_t* perm;        // sorted position -> slot
    const float* pw;            // routing weight of each slot
    const __half* bsrc;         // token rows, K-blocked [K/64][srows][64], pre-swizzled
    int64_t srows;
    int64_t N, K;
    int nb, lbs;                // scale blocks per row; log2(block size) (-1: column-wise)
    int topk, n_pairs, gm;
    __half* act_out;            // FC1 output, K-blocked like bsrc
    int act, has_limit;
    float alpha, beta, limit;
    __half* slot16;             // FC2 output: [slots, N] fp16, weighted by the slot's routing weight
    int32_t* err;
    uint64_t wait_ns;
    int scale_tma;              // block scales staged by TMA (nb % 4 == 0)
    int scale_every;            // stages per TMA-staged group of four scale blocks
    int64_t drop_it;            // test hook: stage whose copies the producer skips
    uint32_t off_s, off_b, load_bytes, nload;
    uint32_t off_epi;           // epilogue staging tiles (one per epilogue warp, FC1)
    uint32_t epi_stage;         // bytes of one staging tile
};

__device__ __forceinline__ void record_error(int32_t* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
    d |= uint64_t(1) << 16;                 // leading byte offset (unused for this layout)
    d |= uint64_t(1024 >> 4) << 32;         // stride byte offset between 8-row atoms
    d |= uint64_t(1) << 46;                 // descriptor version
    d |= uint64_t(2) << 61;                 // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp16 A and B (K-major), fp32 accumulator, M x N.
__device__ __forceinline__ uint32_t f16_idesc(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
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

__device__ __forceinline__ float swiglu(float g, float u, float alpha, float beta, int has_limit,
                                        float limit) {
    if (has_limit) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    return __fdividef(g, 1.f + __expf(-alpha * g)) * (u + beta);
}

__device__ __forceinline__ float pick4(float4 v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

struct Item {
    int e, row0, rows, m, nt;   // expert, first sorted row, token rows, weight tile, MMA N
};

// Work item i: batches of gm weight-tile pairs; inside a batch token tile by
// token tile, then pair, so that the items of a wave share token tiles and
// weight tiles in L2.
__device__ __forceinline__ Item decode_item(const TcArgs& a, int64_t i, int ntiles) {
    const int64_t per_group = int64_t(ntiles) * a.gm;
    const int pg = int(i / per_group);
    const int64_t rem = i % per_group;
    const int tau = int(rem / a.gm);           // token tile
    const int pm = int(rem % a.gm);
    const int32_t* t = a.tiles + kTileHeader + 4 * tau;
    Item it;
    it.e = t[0];
    it.row0 = t[1];
    it.rows = t[2];
    it.m = (pg * a.gm + pm) * kPair;           // first weight tile of the pair
    it.nt = (it.rows + 15) & ~15;
    return it;
}

// The conversion is the exponent-bias method of turning small integers into
// floating point: with the exponent of a power-of-two constant fixed, the
// integer written into the low mantissa bits gives constant + integer exactly,
// and subtracting the constant leaves the integer.  Its use for int4/int8
// weight dequantisation is described by Kim et al., "Who Says Elephants Can't
// Run: Bringing Large Scale MoE Models into Cloud Scale Production" (2022).
//
// Eight packed 4-bit codes (low nibble first) -> four fp16 pairs
// ((q0,q4),(q1,q5),(q2,q6),(q3,q7)) of (q - 8) [* s].  The activations of the
// 4-bit path are stored with the same order inside every group of eight, so
// A and B agree on the K order without a shuffle.  A low nibble OR-ed into the
// mantissa of fp16 1024 gives 1024 + q; a high nibble left in place gives
// 1024 + 16 q, whose pairs are scaled by s / 16 (1/16 when unscaled), which is
// exact.
template <bool SCALE>
__device__ __forceinline__ void deq4(uint32_t w, __half2 s, __half2 s16, uint32_t* out) {
    const __half2 lo_bias = ptx::u32_as_h2(0x64086408u);   // 1032
    const __half2 hi_bias = ptx::u32_as_h2(0x64806480u);   // 1152 = 1024 + 16 * 8
    const uint32_t w8 = w >> 8;
    const __half2 d0 = __hsub2(ptx::u32_as_h2(ptx::and_or(w, 0x000F000Fu, 0x64006400u)), lo_bias);
    const __half2 d1 = __hsub2(ptx::u32_as_h2(ptx::and_or(w, 0x00F000F0u, 0x64006400u)), hi_bias);
    const __half2 d2 = __hsub2(ptx::u32_as_h2(ptx::and_or(w8, 0x000F000Fu, 0x64006400u)), lo_bias);
    const __half2 d3 = __hsub2(ptx::u32_as_h2(ptx::and_or(w8, 0x00F000F0u, 0x64006400u)), hi_bias);
    out[0] = ptx::h2_as_u32(SCALE ? __hmul2(d0, s) : d0);
    out[1] = ptx::h2_as_u32(__hmul2(d1, s16));
    out[2] = ptx::h2_as_u32(SCALE ? __hmul2(d2, s) : d2);
    out[3] = ptx::h2_as_u32(__hmul2(d3, s16));
}

// Four 8-bit codes -> natural-order fp16 pairs ((q0,q1),(q2,q3)) of (q - 128) [* s].
template <bool SCALE>
__device__ __forceinline__ void deq8(uint32_t w, __half2 s, uint32_t* out) {
    const __half2 bias = ptx::u32_as_h2(0x64806480u);
    const __half2 d0 = __hsub2(ptx::u32_as_h2(ptx::prmt(w, 0x64646464u, 0x4140u)), bias);
    const __half2 d1 = __hsub2(ptx::u32_as_h2(ptx::prmt(w, 0x64646464u, 0x4342u)), bias);
    out[0] = ptx::h2_as_u32(SCALE ? __hmul2(d0, s) : d0);
    out[1] = ptx::h2_as_u32(SCALE ? __hmul2(d1, s) : d1);
}

// Position of column j in a row stored with groups of eight in the order
// 0,4,1,5,2,6,3,7 (the 4-bit operand order).
__device__ __forceinline__ int perm8(int j) {
    const int q = j & 7;
    return (j & ~7) + (q < 4 ? 2 * q : 2 * (q - 4) + 1);
}

template <int BITS, bool FC1, bool SCOL>
__global__ void __launch_bounds__(kTcThreads, 1) grouped_gemm_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t load_full[kLoadStages];   // TMA bytes landed
    __shared__ __align__(8) uint64_t load_empty[kLoadStages];  // MMAs reading the stage done
    __shared__ __align__(8) uint64_t a_full[kAStages];         // dequantised weights written
    __shared__ __align__(8) uint64_t a_empty[kAStages];        // MMAs reading them done
    __shared__ __align__(8) uint64_t acc_full;    // the item's MMAs done
    __shared__ __align__(8) uint64_t acc_empty;   // its epilogue done
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    constexpr int PACK = BITS == 4 ? 2 : 1;
    constexpr uint32_t kRawRow = kTcK / PACK;                   // packed bytes per row per stage

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < a.nload; ++s) {
            ptx::mbar_init(&load_full[s], 1);
            ptx::mbar_init(&load_empty[s], 1);
        }
        for (int s = 0; s < kAStages; ++s) {
            ptx::mbar_init(&a_full[s], kDeqWarps);
            ptx::mbar_init(&a_empty[s], 1);
        }
        ptx::mbar_init(&acc_full, 1);
        ptx::mbar_init(&acc_empty, kEpiWarps);
        ptx::mbar_init(&drain_bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(ptx::smem_u32(&tmem_base_s)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;

    // the combine after FC2 may start its prologue on SMs this grid leaves
    ptx::griddep_launch_dependents();
    const int ntiles = a.tiles[0];
    const int64_t items = int64_t(ntiles) * a.n_pairs;
    const int nkb = int(a.K / kTcK);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t abase = sbase + a.nload * a.load_bytes;   // dequantised-weight ring

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            ptx::prefetch_tmap(&a.tm_w);
            if (a.scale_tma) ptx::prefetch_tmap(&a.tm_s);
        }
        uint32_t it = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const Item w = decode_item(a, i, ntiles);
            if (w.rows <= 0) continue;
            const int32_t wrow0 = int32_t(int64_t(w.e) * a.N + int64_t(w.m) * kTcM);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % a.nload);
                const uint32_t ph = (it / a.nload) & 1u;
                if (!ptx::mbar_wait(&load_empty[sl], ph ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (int64_t(it) == a.drop_it) continue;   // test hook: this stage never fills
                uint8_t* sp = smem + size_t(sl) * a.load_bytes;
                if (lane == 0) {
                    // a staged group of four scale blocks covers scale_every stages
                    const bool scales = a.scale_tma && kb % a.scale_every == 0;
                    ptx::mbar_arrive_expect_tx(&load_full[sl], kItemRows * kRawRow +
                                               (scales ? kItemRows * 16u : 0u) +
                                               uint32_t(w.nt) * 128u);
                    ptx::tma_load_2d(sp, &a.tm_w, kb * int(kRawRow), wrow0, &load_full[sl]);
                    if (scales)
                        ptx::tma_load_2d(sp + a.off_s, &a.tm_s, ((kb * kTcK) >> a.lbs) & ~3,
                                         wrow0, &load_full[sl]);
                    // the token tile of this K block: nt contiguous 128-byte rows
                    ptx::bulk_g2s(sp + a.off_b, a.bsrc + (int64_t(kb) * a.srows + w.row0) * kTcK,
                                  uint32_t(w.nt) * 128u, &load_full[sl]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
            for (uint32_t j = it > a.nload ? it - a.nload : 0; j < it; ++j) {
                volatile int never = 0;
                ptx::mbar_wait(&load_full[j % a.nload], (j / a.nload) & 1u, kDrainWaitNs,
                               &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------- MMA issuer -------------------------------
        uint32_t it = 0, item_it = 0;
        bool ok = true;
        bool issued = false;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const Item w = decode_item(a, i, ntiles);
            if (w.rows <= 0) continue;
            const uint32_t aph = item_it & 1u;
            ++item_it;
            if (!ptx::mbar_wait(&acc_empty, aph ^ 1u, a.wait_ns, &abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dbase = tmem_base;
            const uint32_t idesc = f16_idesc(kTcM, w.nt);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % a.nload);
                const int sa = int(it % kAStages);
                if (!ptx::mbar_wait(&a_full[sa], (it / kAStages) & 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sb = sbase + uint32_t(sl) * a.load_bytes + a.off_b;
                    const uint32_t sa0 = abase + uint32_t(sa) * kAStageBytes;
#pragma unroll
                    for (int kk = 0; kk < kTcK / 16; ++kk) {
                        const uint64_t bd = sw128_desc(sb + 32u * kk);
#pragma unroll
                        for (int t = 0; t < kPair; ++t)
                            mma_f16(dbase + uint32_t(t * kAccCols),
                                    sw128_desc(sa0 + uint32_t(t) * kABytes + 32u * kk), bd, idesc,
                                    (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_commit(&load_empty[sl]);
                    mma_commit(&a_empty[sa]);
                    issued = true;
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(&acc_full);
            __syncwarp();
        }
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
        if (lane == 0 && issued) {
            // every MMA this thread issued completes before TMEM is released
            mma_commit(&drain_bar);
            volatile int never = 0;
            ptx::mbar_wait(&drain_bar, 0, kDrainWaitNs, &never);
        }
        __syncwarp();
    } else if (warp < 2 + kDeqWarps) {
        // ------------------------------ dequantisers ------------------------------
        const int r = threadIdx.x - 64;            // row of the 256-row item (two weight tiles)
        const int tile = r >> 7, rr = r & (kTcM - 1);
        uint32_t it = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; i < items && ok; i += gridDim.x) {
            const Item w = decode_item(a, i, ntiles);
            if (w.rows <= 0) continue;
            const int64_t row = int64_t(w.m) * kTcM + r;   // weight row within the expert
            const bool valid = row < a.N;
            const float* srow = a.scales + (int64_t(w.e) * a.N + (valid ? row : 0)) * a.nb;
            float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);   // staged group of four scale blocks
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int sl = int(it % a.nload);
                const int sa = int(it % kAStages);
                if (!ptx::mbar_wait(&load_full[sl], (it / a.nload) & 1u, a.wait_ns, &abort_flag) ||
                    !ptx::mbar_wait(&a_empty[sa], ((it / kAStages) & 1u) ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sp = ptx::launder(sbase + uint32_t(sl) * a.load_bytes);
                const uint32_t arow = abase + uint32_t(sa) * kAStageBytes + uint32_t(tile) * kABytes +
                                      uint32_t(rr) * 128u;
                // Block scales of this K block: the staged group of four covers it.
                // Column-wise scales are applied to the accumulator instead.
                __half2 sc[4] = {};
                if (!SCOL) {
                    // the four staged blocks start at ((kb * 64) >> lbs) & ~3; rows whose scale
                    // row is not 16-byte aligned (nb % 4 != 0) read them from global memory
                    if (a.scale_tma) {
                        if (kb % a.scale_every == 0) s4 = ptx::ld_f32x4(sp + a.off_s + uint32_t(r) * 16u);
                    } else {
                        const int g0 = ((kb * kTcK) >> a.lbs) & ~3;
                        s4.x = valid && g0 < a.nb ? __ldg(srow + g0) : 0.f;
                        s4.y = valid && g0 + 1 < a.nb ? __ldg(srow + g0 + 1) : 0.f;
                        s4.z = valid && g0 + 2 < a.nb ? __ldg(srow + g0 + 2) : 0.f;
                        s4.w = valid && g0 + 3 < a.nb ? __ldg(srow + g0 + 3) : 0.f;
                    }
                    if (a.lbs >= 6) {            // one block per K block
                        const int sx0 = ((kb * kTcK) >> a.lbs) & ~3;
                        sc[0] = sc[1] = sc[2] = sc[3] =
                            __float2half2_rn(pick4(s4, ((kb * kTcK) >> a.lbs) - sx0));
                    } else if (a.lbs == 5) {     // two blocks of 32
                        const int o = (2 * kb) & 3;
                        sc[0] = sc[1] = __float2half2_rn(pick4(s4, o));
                        sc[2] = sc[3] = __float2half2_rn(pick4(s4, o + 1));
                    } else {                     // four blocks of 16
                        sc[0] = __float2half2_rn(s4.x);
                        sc[1] = __float2half2_rn(s4.y);
                        sc[2] = __float2half2_rn(s4.z);
                        sc[3] = __float2half2_rn(s4.w);
                    }
                }
                uint32_t outv[32];
                if (BITS == 4) {
                    // 32 packed bytes; the two 16-byte halves are read in an order that
                    // keeps each quarter warp on distinct banks
                    const bool swp = ((r >> 2) & 1) != 0;
                    const uint4 p0 = ptx::lds128(sp + uint32_t(r) * 32u + (swp ? 16u : 0u));
                    const uint4 p1 = ptx::lds128(sp + uint32_t(r) * 32u + (swp ? 0u : 16u));
                    const uint4 lo = swp ? p1 : p0, hi = swp ? p0 : p1;
                    const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    const __half2 inv16 = __float2half2_rn(0.0625f);
                    __half2 sc16[4];
#pragma unroll
                    for (int b = 0; b < 4; ++b) sc16[b] = SCOL ? inv16 : __hmul2(sc[b], inv16);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (SCOL) deq4<false>(wv[q], sc[0], inv16, outv + 4 * q);
                        else deq4<true>(wv[q], sc[q >> 1], sc16[q >> 1], outv + 4 * q);   // word q: K 8q..8q+7
                    }
                } else {
                    uint32_t wv[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 pj = ptx::lds128(sp + uint32_t(r) * 64u + uint32_t(j) * 16u);
                        wv[4 * j] = pj.x; wv[4 * j + 1] = pj.y; wv[4 * j + 2] = pj.z; wv[4 * j + 3] = pj.w;
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        if (SCOL) deq8<false>(wv[q], sc[0], outv + 2 * q);
                        else deq8<true>(wv[q], sc[q >> 2], outv + 2 * q);   // word q: K 4q..4q+3
                    }
                }
                // 64 fp16 = eight 16-byte chunks of the 128-byte row, swizzled
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t addr = arow + uint32_t((c ^ (rr & 7)) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr),
                                 "r"(outv[4 * c]), "r"(outv[4 * c + 1]), "r"(outv[4 * c + 2]),
                                 "r"(outv[4 * c + 3])
                                 : "memory");
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&a_full[sa]);
            }
        }
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
    } else {
        // -------------------------------- epilogue --------------------------------
        const int ew = warp - 2 - kDeqWarps;       // 0..7
        const int tile = ew / 4;                   // weight tile of the item
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int r = quad * 32 + lane;            // row in the weight tile
        __half* stile = reinterpret_cast<__half*>(smem + a.off_epi + uint32_t(ew) * a.epi_stage);
        // outputs outside the fp16 range: the largest magnitude and a NaN-propagating
        // sum of every output this lane computes, checked once at the end
        float omax = 0.f, osum = 0.f;
        uint32_t item_it = 0;
        for (int64_t i = blockIdx.x; i < items; i += gridDim.x) {
            const Item w = decode_item(a, i, ntiles);
            if (w.rows <= 0) continue;
            const uint32_t aph = item_it & 1u;
            ++item_it;
            // FC2: each lane's token of every 32-token chunk, its slot and routing
            // weight, loaded before the accumulator is ready (the loads are a
            // dependent chain and would otherwise stall every chunk)
            int slot_c[kTcMaxN / 32];
            float p_c[kTcMaxN / 32];
            if (!FC1) {
#pragma unroll
                for (int ch = 0; ch < kTcMaxN / 32; ++ch) {
                    const int col = ch * 32 + lane;
                    slot_c[ch] = col < w.rows ? __ldg(a.perm + w.row0 + col) : 0;
                }
#pragma unroll
                for (int ch = 0; ch < kTcMaxN / 32; ++ch)
                    p_c[ch] = ch * 32 + lane < w.rows ? __ldg(a.pw + slot_c[ch]) : 0.f;
            }
            // column-wise scale of this output row (applied here, not in the operand), also
            // loaded before the accumulator is ready
            const int64_t row = int64_t(w.m + tile) * kTcM + r;
            const float srow = SCOL && row < a.N ? __ldg(a.scales + int64_t(w.e) * a.N + row) : 1.f;
            if (!ptx::mbar_wait(&acc_full, aph, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    record_error(a.err, QMOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + (uint32_t(quad * 32) << 16) +
                                   uint32_t(tile * kAccCols);
            for (int c0 = 0; c0 < w.nt; c0 += 32) {
                float v[32];
                tmem_ld32(tbase + uint32_t(c0), v);
                if (SCOL) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] *= srow;
                }
                // a tile's last chunk: columns past its rows hold stale sums; zero them so
                // that their (unstored) outputs stay finite
                if (c0 + 32 > w.rows) {
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (c0 + q >= w.rows) v[q] = 0.f;
                }
                if (FC1) {
                    // The warp's outputs for these 32 tokens (16 SwiGLU or 32 ReLU
                    // activation columns, already in the stored column order) go
                    // through a shared-memory tile so that each token row leaves as
                    // contiguous 16-byte stores.
                    const int ncol = a.act == QMOE_ACT_SWIGLU ? 16 : 32;   // columns per warp
                    if (a.act == QMOE_ACT_SWIGLU) {
                        // even lane: gate row, tokens c0..c0+15; odd lane: tokens c0+16..c0+31
                        const bool even = (lane & 1) == 0;
                        const int jl = lane >> 1;                       // column within the warp
                        const int pos = BITS == 4 ? perm8(jl) : jl;
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float send = even ? v[16 + q] : v[q];
                            const float recv = __shfl_xor_sync(kFull, send, 1);
                            const float gate = even ? v[q] : recv;
                            const float lin = even ? recv : v[16 + q];
                            const float o = swiglu(gate, lin, a.alpha, a.beta, a.has_limit, a.limit);
                            omax = fmaxf(omax, fabsf(o));
                            osum += o;
                            stile[(even ? q : 16 + q) * 16 + pos] = __float2half_rn(o);
                        }
                    } else {
                        const int pos = BITS == 4 ? perm8(lane) : lane;
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const float o = fmaxf(v[q], 0.f);
                            omax = fmaxf(omax, o);
                            stile[q * 32 + pos] = __float2half_rn(o);
                        }
                    }
                    __syncwarp();
                    // lane = token of the chunk; its ncol outputs are 2 or 4 16-byte chunks
                    // of one 64-column K block of the K-blocked FC2 input, stored at
                    // chunk ^ (token & 7): the 128-byte swizzle of the token's row in a
                    // tile (tiles start on multiples of 8 rows of their expert)
                    const int64_t jbase = (int64_t(w.m + tile) * kTcM + quad * 32) / (ncol == 16 ? 2 : 1);
                    // rows past N (a partial last weight tile) produce no outputs
                    const int col = c0 + lane;
                    if (col < w.rows && jbase < a.N / (ncol == 16 ? 2 : 1)) {
                        const uint4* src = reinterpret_cast<const uint4*>(stile + lane * ncol);
                        uint4* dst = reinterpret_cast<uint4*>(
                            a.act_out + ((jbase / kTcK) * a.srows + w.row0 + col) * kTcK);
                        const int ch0 = int(jbase % kTcK) / 8;
                        for (int h = 0; h < ncol / 8; ++h) dst[(ch0 + h) ^ (col & 7)] = src[h];
                    }
                    __syncwarp();
                } else {
                    // FC2: lane = token c0 + lane, with its slot and routing weight.  The
                    // warp's 32 output rows of each token are staged in shared memory and
                    // leave as one 64-byte piece of the slot's row.
                    const int col = c0 + lane;
                    const bool valid_col = col < w.rows;
                    int my_slot = 0;
                    float my_p = 0.f;
#pragma unroll
                    for (int ch = 0; ch < kTcMaxN / 32; ++ch)   // registers: select, not index
                        if (ch * 32 == c0) { my_slot = slot_c[ch]; my_p = p_c[ch]; }
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const float o = v[q] * __shfl_sync(kFull, my_p, q);
                        omax = fmaxf(omax, fabsf(o));
                        osum += o;
                        stile[q * 32 + lane] = __float2half_rn(o);
                    }
                    __syncwarp();
                    const int64_t hbase = int64_t(w.m + tile) * kTcM + quad * 32;
                    if (valid_col && hbase < a.N) {
                        const uint4* src = reinterpret_cast<const uint4*>(stile + lane * 32);
                        uint4* dst = reinterpret_cast<uint4*>(a.slot16 + int64_t(my_slot) * a.N + hbase);
#pragma unroll
                        for (int h = 0; h < 4; ++h) dst[h] = src[h];
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&acc_empty);
        }
        const bool bad = !(omax <= 65504.f) || osum != osum;
        if (__any_sync(kFull, bad) && lane == 0) record_error(a.err, QMOE_DEVERR_NONFINITE);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
}

template <int BITS, bool FC1, bool SCOL>
cudaError_t launch_tc(const TcArgs& args, int grid, size_t smem, cudaStream_t s) {
    auto kern = grouped_gemm_kernel<BITS, FC1, SCOL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, kTcThreads, smem, s>>>(args);
    return cudaGetLastError();
}

int ilog2(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return l;
}

int pick_group(int n_mtiles) {
    for (int g = 8; g > 1; --g)
        if (n_mtiles % g == 0) return g;
    return 1;
}

}  // namespace

int grouped_tile_tokens() { return kTcMaxN; }

bool grouped_shape_ok(const Problem& p) {
    if (p.H % kTcK != 0 || p.I % kTcK != 0) return false;
    return true;
}

cudaError_t launch_grouped_fc(const Problem& p, const Plan& pl, const Work& w, bool fc1,
                              cudaStream_t s) {
    TcArgs a;
    std::memset(&a, 0, sizeof(a));
    const uint8_t* wt = fc1 ? p.w1 : p.w2;
    a.N = fc1 ? p.fusion * p.I : p.H;
    a.K = fc1 ? p.H : p.I;
    a.nb = int(fc1 ? p.nb1 : p.nb2);
    a.lbs = p.bs ? ilog2(p.bs) : -1;
    a.scales = fc1 ? p.s1 : p.s2;
    const int pack = p.pack;
    if (!encode_tmap_2d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt, uint64_t(a.K / pack),
                        uint64_t(p.E * a.N), uint64_t(a.K / pack), uint32_t(kTcK / pack), kItemRows,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    a.bsrc = fc1 ? w.xs16 : static_cast<const __half*>(w.act);
    a.srows = pl.srows;
    a.scale_tma = (p.bs != 0 && a.nb % 4 == 0) ? 1 : 0;
    // four staged scale blocks of bs columns cover 4 * bs / 64 stages (bs >= 16)
    a.scale_every = p.bs >= 16 ? int(4 * p.bs / kTcK) : 1;
    if (a.scale_tma &&
        !encode_tmap_2d(&a.tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.scales, uint64_t(a.nb),
                        uint64_t(p.E * a.N), uint64_t(a.nb) * 4, 4, kItemRows,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    a.tiles = w.tiles;
    a.perm = w.perm;
    a.topk = int(p.k);
    const int n_mtiles = int((a.N + kTcM - 1) / kTcM);
    a.n_pairs = (n_mtiles + kPair - 1) / kPair;
    a.gm = pick_group(a.n_pairs);
    a.act_out = static_cast<__half*>(w.act);
    a.act = p.act;
    a.has_limit = p.has_limit;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.limit = p.limit;
    a.slot16 = reinterpret_cast<__half*>(w.slot_out);
    a.pw = w.pw;
    a.err = w.ctrl;
    a.wait_ns = wait_limit_ns();
    a.drop_it = drop_stage();
    const uint32_t raw_bytes = uint32_t(kItemRows * (kTcK / pack));
    a.off_s = raw_bytes;                          // 256 rows x 4 scales (TMA-staged scales only)
    a.off_b = (raw_bytes + (a.scale_tma ? kItemRows * 16u : 0u) + 1023u) & ~1023u;
    // per epilogue warp: 32 tokens x 16 (SwiGLU) or 32 (ReLU, FC2) fp16 outputs
    a.epi_stage = 32u * (fc1 && p.act == QMOE_ACT_SWIGLU ? 16u : 32u) * 2u;
    a.load_bytes = a.off_b + kBBytes;
    const size_t smem_cap = 232448 - 1024;   // 227 KB per CTA, minus static shared memory
    const size_t fixed = size_t(kAStages) * kAStageBytes + size_t(kEpiWarps) * a.epi_stage;
    a.nload = uint32_t(std::min<size_t>(kLoadStages, (smem_cap - 1024 - fixed) / a.load_bytes));
    if (a.nload < 2) return cudaErrorInvalidValue;
    a.off_epi = a.nload * a.load_bytes + uint32_t(kAStages) * kAStageBytes;
    const size_t smem = 1024 + size_t(a.nload) * a.load_bytes + fixed;
    const int64_t items_max = pl.max_tiles * a.n_pairs;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(items_max, device_sm_count())));
    const int kid = fc1 ? QMOE_KERNEL_FC1 : QMOE_KERNEL_FC2;
    note_launch(kid, s, true);
    cudaError_t e;
    const bool scol = p.bs == 0;
#define QMOE_TC_LAUNCH(B, C) \
    (fc1 ? launch_tc<B, true, C>(a, grid, smem, s) : launch_tc<B, false, C>(a, grid, smem, s))
    if (p.bits == 4) e = scol ? QMOE_TC_LAUNCH(4, true) : QMOE_TC_LAUNCH(4, false);
    else e = scol ? QMOE_TC_LAUNCH(8, true) : QMOE_TC_LAUNCH(8, false);
#undef QMOE_TC_LAUNCH
    note_launch(kid, s, false);
    return e;
}

}  // namespace qmoe
