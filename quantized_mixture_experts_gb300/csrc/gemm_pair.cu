// Grouped path of the QMoE layer: expert-grouped GEMMs on CTA pairs of the
// 5th-generation tensor cores (tcgen05.mma.cta_group::2), dequantising the
// packed expert weights on the way into shared memory.
//
// QMoE manifest passes QMoE.FC1ActivationStageGrouped / QMoE.OutputStageGrouped
// (tiles of one expert's routed tokens against that expert's weights,
// derive.groupMaxTiles) and GroupedMatMul-29 Summary (a runtime should fuse
// DequantizeLinear + GroupedMatMul so the dequantized [G, K, N] weights are
// never materialised).
//
// One work item = (token tile: up to 256 expert-sorted rows of one expert,
// 256-row weight tile of that expert), computed by a cluster of two CTAs:
//   D[256 weight rows, n] = deq(W)[256, K] * X[n, K]^T,  n = rows rounded up to 32
// The dequantised weights are the MMA's A operand (M = 256: each CTA converts
// and holds its own 128 rows), the tokens its B operand (N = n: rows
// [rank * n/2, rank * n/2 + n/2) of the tile in each CTA), and each CTA's
// tensor memory receives its 128 weight rows x n token columns, so the tensor
// cores work in proportion to the routed tokens.  Two 256-column accumulators
// alternate between items: the epilogue of one item runs while the next
// item's MMAs run, transposing its 32 x 32 blocks through a per-warp shared
// tile into token rows.
//
// Operand exchange within the pair.  Each CTA's tensor core reads the other
// CTA's token rows, and only its own dequantised rows.  The token rows are
// therefore copied by the tensor-copy engine with completion counted on CTA 0's
// barrier (.cta_group::2), which orders them for both tensor cores, while the
// rows the dequantisers write in the generic proxy stay CTA-local (fenced to
// the async proxy at CTA scope).  The earlier arrangement (tokens as A, the
// dequantised weights as B, whose halves each tensor core reads from both
// CTAs, with the token copies completing on each CTA's own barrier) let about
// one call in a few hundred compute an item from stale operands.
//
// Per CTA (persistent, one per SM), warp-specialised, a ring of stages each
// holding the K = 64 slice of the CTA's n/2 token rows, its 128 packed weight
// rows with their block scales, and the dequantised fp16 weight rows:
//   warp 0      TMA producer: packed weights and staged block scales (2-D
//               tensor boxes, on this CTA's barrier), the token rows (one 3-D
//               box of 128 rows: the rows are stored K-blocked with the
//               128-byte swizzle already applied; on CTA 0's barrier);
//   warp 1      tensor-memory allocation; in CTA 0 of the pair, one lane
//               issues the MMAs of both CTAs and commits their completion to
//               both CTAs' barriers;
//   warps 2-4, 6-8, 10-11
//               dequantisers: (q - mid) * scale in fp16, written in the
//               128-byte-swizzled K-major layout; two groups of four warps take
//               alternate stages (one thread per weight row), so two stages are
//               converted at once; they arrive on CTA 0's operand barrier
//               (warps 5 and 9 stay idle: see kEpiWarp0);
//   warps 12-19 epilogue: FC1 ReLU / SwiGLU to fp16 activations in the
//               K-blocked layout FC2 reads; FC2 rows per routing slot, already
//               multiplied by the slot's routing weight (fp16; the combine adds
//               a token's k rows in fixed order).
// Every wait is bounded; on expiry the CTA records QMOE_DEVERR_TIMEOUT, stops,
// and both CTAs meet at the final cluster barrier before freeing tensor memory.
// The producer, the dequantisers and the epilogue wait inside mbarrier.try_wait
// with a suspend-time hint (they are woken when the phase completes), so that
// waiting warps leave their schedulers' issue slots to the working ones.
#include <algorithm>
#include <cstring>

#include "ptx.cuh"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr int kRowsCta = 128;         // token rows and weight rows per CTA of a pair
constexpr int kTileRows = 2 * kRowsCta;
constexpr int kK = 64;                // K per stage: one 128-byte row of fp16
constexpr int kMaxStages = 6;        // ring depth upper bound (the launch picks what fits)
constexpr int kDeqGroupWarps = 4;     // warps of a group (the group takes every other stage)
constexpr int kEpiWarps = 8;          // two per TMEM lane quadrant (one per column half)
// Warp roles.  A warp runs on scheduler (warp % 4); the MMA-issuing warp 1
// shares scheduler 1 only with epilogue warps and two idle warps (5, 9), so
// the dequantisers' arithmetic does not delay the issue of the next stage.
constexpr int kEpiWarp0 = 12;         // warps 12-19: epilogue
constexpr int kWarps = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = 32 * kWarps;
constexpr uint32_t kAccCols = 256;    // accumulator columns (N) of one item
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr uint32_t kABytes = kRowsCta * 128;   // token rows of one stage
constexpr uint32_t kBBytes = kRowsCta * 128;   // dequantised weight rows of one stage
constexpr uint32_t kSBytes = kRowsCta * 16;    // four staged scale blocks per row
constexpr unsigned kFull = 0xffffffffu;
constexpr uint64_t kDrainWaitNs = 200000000ull;
// Token tiles of at most this many rows run with the tokens as the MMA's N.
constexpr int kTokBox = kRowsCta;     // token rows per tensor-copy box (one box per CTA and stage)

struct PairArgs {
    CUtensorMap tm_w;           // packed weights [E*N rows, K/pack bytes], box {64/pack, 128}
    CUtensorMap tm_b;           // token rows [K/64][srows][64] fp16 (pre-swizzled), box {64, 128, 1}
    CUtensorMap tm_s;           // block scales [E*N rows, nb] fp32, box {4, 128}
    const float* scales;        // [E*N, nb] (nb = 1 for column-wise)
    const int32_t* tiles;       // header + (expert, first sorted row, rows, expert's first tile)
    const int32_t* counts;      // slots per expert
    const int32_t* perm;        // sorted position -> slot
    const float* pw;            // routing weight of each slot
    const __half* bsrc;         // token rows, K-blocked [K/64][srows][64], pre-swizzled
    int64_t srows;
    int64_t N, K;               // weight rows per expert, reduction length
    int64_t n_out;              // valid output columns: I (FC1 activations) or H (FC2)
    int nb, lbs;                // scale blocks per row; log2(block size) (-1: column-wise)
    int n_mt, gm;               // weight tiles per expert; weight tiles per item group
    __half* act_out;            // FC1 output, K-blocked like bsrc
    int act, has_limit;
    float alpha, beta, limit;
    __half* slot16;             // FC2 output: [slots, n_out] fp16, weighted by routing weight
    int32_t* err;
    uint64_t wait_ns;
    int scale_tma;              // block scales staged by TMA (nb % 4 == 0)
    int64_t drop_it;            // test hook: stage whose copies the producer skips
    uint32_t stage_bytes, off_b, off_raw, off_s, raw_bytes, nstages;
    uint32_t off_epi;           // epilogue staging: 2 KB per epilogue warp, after the ring
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

// One MMA of the pair (issued by CTA 0): A = 256 token rows, 128 from each
// CTA's shared memory at the same offset; B = 256 weight rows, 128 from each.
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` (same offset in both CTAs) when the issuing thread's MMAs complete.
__device__ __forceinline__ void commit_both(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(ptx::smem_u32(bar)), "h"(uint16_t(3))
        : "memory");
}

__device__ __forceinline__ void commit_local(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(ptx::smem_u32(bar))
        : "memory");
}

// Arrive with the default (release, CTA scope) semantics on the barrier at
// shared::cluster address `addr` (CTA 0's copy).  The dequantisers publish
// their shared-memory writes to the tensor core with fence.proxy.async before
// arriving.
__device__ __forceinline__ void arrive_remote(uint32_t addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// Token rows box (64 fp16 x kTokBox rows of K block kb) into this CTA's shared
// memory, completion counted on CTA 0's barrier at shared::cluster address `bar`.
__device__ __forceinline__ void tma_tokens(void* dst, const CUtensorMap* map, int32_t row, int32_t kb,
                                           uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(ptx::smem_u32(dst)), "l"(map), "r"(0), "r"(row), "r"(kb), "r"(bar)
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

// The integer-to-half conversions below use the exponent-bias method: with the
// exponent of a power-of-two constant fixed, an integer written into the low
// mantissa bits gives constant + integer exactly, and subtracting the
// constant leaves the integer.  Its use for int4/int8 weight dequantisation is
// described by Kim et al., "Who Says Elephants Can't Run: Bringing Large Scale
// MoE Models into Cloud Scale Production" (2022).
//
// Eight packed 4-bit codes (low nibble first) -> four fp16 pairs
// ((q0,q4),(q1,q5),(q2,q6),(q3,q7)) of (q - 8) [* s]: one 16-byte piece of a
// row in the order the 4-bit path stores its activations in every group of
// eight.  A low nibble in the mantissa of fp16 1024 gives 1024 + q; a high
// nibble left in place gives 1024 + 16 q, whose pairs are scaled by s / 16
// (1/16 when unscaled), which is exact.
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

// Two fp32 values -> one fp16 pair (round to nearest even).
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    return ptx::h2_as_u32(__floats2half2_rn(a, b));
}

struct Item {
    int e, row0, rows, m;       // expert, first sorted row of the tile, its rows, weight tile
};

// Token columns of a tokens-as-N item (a multiple of 32: N / 2 rows per CTA, a
// multiple of the 16 rows the instruction takes with M = 256 on a pair), or 0
// for an item that runs with the tokens as M.
__device__ __forceinline__ int item_ncols(const Item& w) {
    return (w.rows + 31) & ~31;
}

// Byte offset of output column c (of a warp's 32) of token row t in the
// epilogue's 2 KB staging tile: 64 bytes per token row, 16-byte piece g of
// row t at piece g ^ ((t >> 1) & 3) (conflict-free for a warp writing one row
// and for a warp reading 16-byte pieces of eight rows).  PERM4 places the
// eight values of a piece in the 4-bit operand order 0,4,1,5,2,6,3,7.
template <bool PERM4>
__device__ __forceinline__ uint32_t stage_off(int t, int c) {
    const int q = c & 7;
    const int pos = PERM4 ? (q < 4 ? 2 * q : 2 * (q - 4) + 1) : q;
    return uint32_t(t) * 64u + ((uint32_t(c >> 3) ^ ((uint32_t(t) >> 1) & 3u)) << 4) +
           uint32_t(pos) * 2u;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, float v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(__half_as_ushort(__float2half_rn(v)))
                 : "memory");
}

// Epilogue of a tokens-as-N item.  The warp's tensor-memory lane quadrant
// holds 32 weight rows (lane = weight row) x nc token columns; the two warps
// of a quadrant take alternate blocks of 32 tokens (at most four each).  A
// block is scaled (column-wise scales: one per lane), activated (FC1) or
// multiplied by each slot's routing weight (FC2), written transposed into the
// warp's staging tile, and stored from there as whole 16-byte pieces of each
// token's output row, in the layouts the tokens-as-M epilogue writes.  The
// lanes of a pair (weight rows 2i, 2i + 1) trade values so that every lane
// works: for SwiGLU a lane computes activation i for every other token, for
// FC2 it stores columns (2i, 2i + 1) of every other token as one 32-bit word.
// slot[m], p[m]: FC2 routing slot and weight of token chalf*32 + 64m + lane,
// loaded by the caller before the accumulator is ready.
template <int BITS, bool FC1, bool SCOL>
__device__ __forceinline__ void epilogue_tokens_as_n(const PairArgs& a, const Item& w, int nc,
                                                     uint32_t tq, uint32_t stg, int rank,
                                                     int quad, int chalf, int lane,
                                                     const int* slot, const float* p, float& omax,
                                                     float& osum) {
    const int64_t wcol = int64_t(w.m) * kTileRows + rank * kRowsCta + quad * 32;   // lane 0's row
    const int64_t wrow = wcol + lane;
    const bool glu = FC1 && a.act == QMOE_ACT_SWIGLU;
    const int odd = lane & 1;
    // the warp's run of output columns: 16 activations (SwiGLU: weight rows 2j, 2j + 1 are
    // gate and linear of activation j) or 32 columns; n_out is a multiple of 64, so the
    // run is wholly valid or wholly past the end
    const int64_t c_first = glu ? (wcol >> 1) : wcol;
    const bool cols_ok = c_first < a.n_out;
    float cs = 1.f;
    if (SCOL) cs = wrow < a.N ? __ldg(a.scales + int64_t(w.e) * a.N + wrow) : 0.f;
#pragma unroll
    for (int m = 0; m < kTileRows / 64; ++m) {
        const int tb = chalf * 32 + 64 * m;
        if (tb >= nc) break;
        float v[32];
        tmem_ld32(tq + uint32_t(tb), v);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            float x0 = v[j], x1 = v[j + 1];
            if (SCOL) {
                x0 *= cs;
                x1 *= cs;
            }
            // even lane: token j; odd lane: token j + 1
            const int t = j + odd;
            const bool tv = tb + t < w.rows;
            const float recv = __shfl_xor_sync(kFull, odd ? x0 : x1, 1);
            if (glu) {
                // even: gate x0 with the odd lane's linear of token j; odd: the even
                // lane's gate of token j + 1 with linear x1
                const float o = tv ? swiglu(odd ? recv : x0, odd ? x1 : recv, a.alpha, a.beta,
                                            a.has_limit, a.limit)
                                   : 0.f;
                if (cols_ok) {
                    omax = fmaxf(omax, fabsf(o));
                    osum += o;
                }
                st_shared_u16(stg + stage_off<BITS == 4>(t, lane >> 1), o);
            } else if (FC1) {
                // values of columns (lane & ~1, lane | 1) for token t
                const float o0 = tv ? fmaxf(odd ? recv : x0, 0.f) : 0.f;
                const float o1 = tv ? fmaxf(odd ? x1 : recv, 0.f) : 0.f;
                if (cols_ok) omax = fmaxf(omax, fmaxf(o0, o1));
                st_shared_u16(stg + stage_off<BITS == 4>(t, lane & ~1), o0);
                st_shared_u16(stg + stage_off<BITS == 4>(t, lane | 1), o1);
            } else {
                const float pt = __shfl_sync(kFull, p[m], t);
                const float o0 = tv ? (odd ? recv : x0) * pt : 0.f;
                const float o1 = tv ? (odd ? x1 : recv) * pt : 0.f;
                if (cols_ok) {
                    omax = fmaxf(omax, fmaxf(fabsf(o0), fabsf(o1)));
                    osum += o0 + o1;
                }
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(stg + stage_off<false>(t, lane & ~1)),
                             "r"(pack_h2(o0, o1))
                             : "memory");
            }
        }
        __syncwarp();
        if (FC1) {
            const int tok = tb + lane;             // the token row this lane stores
            if (tok < w.rows && cols_ok) {
                const int npc = glu ? 2 : 4;
                for (int g = 0; g < npc; ++g) {
                    const uint4 val = ptx::lds128(
                        stg + uint32_t(lane) * 64u + ((uint32_t(g) ^ ((uint32_t(lane) >> 1) & 3u)) << 4));
                    uint4* dst = reinterpret_cast<uint4*>(
                        a.act_out + ((c_first / kK) * a.srows + w.row0 + tok) * kK);
                    const int ch = int(c_first % kK) / 8 + g;
                    dst[ch ^ (tok & 7)] = val;
                }
            }
        } else if (cols_ok) {
            // each store instruction writes 8 token rows x 64 contiguous bytes: lane
            // (r, j) stores 16-byte piece j of token row r of the block
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 8 * i + (lane >> 2);
                const int j = lane & 3;
                const int rslot = __shfl_sync(kFull, slot[m], r);
                const uint4 val = ptx::lds128(
                    stg + uint32_t(r) * 64u + ((uint32_t(j) ^ ((uint32_t(r) >> 1) & 3u)) << 4));
                if (tb + r < w.rows)
                    reinterpret_cast<uint4*>(a.slot16 + int64_t(rslot) * a.n_out + c_first)[j] = val;
            }
        }
        __syncwarp();   // the tile is read before the next block overwrites it
    }
}

// Position in a ring of n stages: slot and the parity of its current phase,
// advanced without divisions (the issuing thread's per-stage work is on the
// tensor pipe's critical path).
struct Ring {
    uint32_t sl = 0, ph = 0;
    __device__ __forceinline__ void next(uint32_t n) {
        if (++sl == n) {
            sl = 0;
            ph ^= 1u;
        }
    }
};

// Work item i.  An expert's items are contiguous: with its token tiles
// tau0 .. tau0 + nt - 1, they are items tau0 * n_mt .. (tau0 + nt) * n_mt - 1,
// in groups of gm weight tiles, inside a group token tile by token tile, so
// that the items running at the same time share weight tiles and token tiles
// in L2 and each weight tile is read from DRAM about once.
__device__ __forceinline__ Item pair_item(const PairArgs& a, int64_t i) {
    const int tg = int(i / a.n_mt);                    // a token tile of the same expert
    const int e = __ldg(a.tiles + kTileHeader + 4 * tg);
    const int tau0 = __ldg(a.tiles + kTileHeader + 4 * tg + 3);
    const int nt = (__ldg(a.counts + e) + kTileRows - 1) / kTileRows;
    const int64_t idx = i - int64_t(tau0) * a.n_mt;
    const int per_group = nt * a.gm;
    const int g = int(idx / per_group), rem = int(idx - int64_t(g) * per_group);
    const int tau = tau0 + rem / a.gm;
    Item it;
    it.e = e;
    it.row0 = __ldg(a.tiles + kTileHeader + 4 * tau + 1);
    it.rows = __ldg(a.tiles + kTileHeader + 4 * tau + 2);
    it.m = g * a.gm + rem % a.gm;
    return it;
}

template <int BITS, bool FC1, bool SCOL>
__global__ void __launch_bounds__(kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ PairArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t ld_full[kMaxStages];    // this CTA's packed rows and scales landed
    __shared__ __align__(8) uint64_t tok_full[kMaxStages];   // CTA 0: both CTAs' token rows landed
    __shared__ __align__(8) uint64_t op_full[kMaxStages];    // CTA 0: both CTAs' operands ready
    __shared__ __align__(8) uint64_t st_free[kMaxStages];    // the stage's MMAs completed
    __shared__ __align__(8) uint64_t acc_full[2];            // an item's MMAs completed
    __shared__ __align__(8) uint64_t acc_empty[2];           // CTA 0: both epilogues done
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_flag;
    __shared__ int stage_nc[kMaxStages];                     // token columns of the stage's item
    constexpr int PACK = BITS == 4 ? 2 : 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_rank();
    const bool leader = rank == 0;
    const uint32_t S = a.nstages;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            ptx::mbar_init(&ld_full[s], 1);
            ptx::mbar_init(&tok_full[s], 1);
            ptx::mbar_init(&op_full[s], 2 * kDeqGroupWarps);
            ptx::mbar_init(&st_free[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&acc_full[b], 1);
            ptx::mbar_init(&acc_empty[b], 2 * kEpiWarps);
        }
        ptx::mbar_init(&drain_bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(ptx::smem_u32(&tmem_base_s)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    ptx::cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_s;

    // launched as a programmatic dependent of the kernel that writes its operands and
    // tile table: the prologue above overlaps that kernel's end
    ptx::griddep_wait();
    // the kernel after this one may start its prologue on SMs this grid leaves
    ptx::griddep_launch_dependents();
    const int64_t items = int64_t(__ldg(a.tiles)) * a.n_mt;
    const int nkb = int(a.K / kK);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int64_t first = blockIdx.x >> 1, step = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            ptx::prefetch_tmap(&a.tm_w);
            ptx::prefetch_tmap(&a.tm_b);
            if (a.scale_tma) ptx::prefetch_tmap(&a.tm_s);
        }
        // Item descriptions for 32 items at a time, one per lane (their table lookups
        // run in parallel); the current one is read by shuffle.
        Item lw = Item{0, 0, 0, 0};
        auto shfl_item = [&](int src) {
            Item w;
            w.e = __shfl_sync(kFull, lw.e, src);
            w.row0 = __shfl_sync(kFull, lw.row0, src);
            w.rows = __shfl_sync(kFull, lw.rows, src);
            w.m = __shfl_sync(kFull, lw.m, src);
            return w;
        };
        // where item w's packed rows, scales and this CTA's token rows are
        auto wrow_of = [&](const Item& w) {
            return int32_t(int64_t(w.e) * a.N + int64_t(w.m) * kTileRows + int(rank) * kRowsCta);
        };
        uint32_t it = 0;
        Ring r;
        bool ok = true;
        int64_t j = 0;   // this CTA's items so far
        const uint32_t tok_addr = ptx::leader_addr(&tok_full[0]);
        for (int64_t i = first; i < items && ok; i += step, ++j) {
            const int lj = int(j & 31);
            if (lj == 0) {
                const int64_t ii = i + int64_t(lane) * step;
                if (ii < items) lw = pair_item(a, ii);
            }
            const Item w = shfl_item(lj);
            // token rows of this CTA: its n/2 of the item's n token columns, copied in boxes
            // of kTokBox rows that complete on CTA 0's token barrier (the other CTA's tensor
            // core reads them: the copy engine's completion orders them for both)
            const int nc = item_ncols(w);
            const int half = nc >> 1;
            auto rows_of = [&](int rk) { return min(max(w.rows - rk * half, 0), half); };
            // one box of kTokBox rows per CTA that has rows (rows past the tile's are read
            // too and never stored; past the buffer the copy fills zeros)
            const int nbox = rows_of(int(rank)) > 0 ? 1 : 0;
            const uint32_t tok_bytes =
                uint32_t((rows_of(0) > 0 ? 1 : 0) + (rows_of(1) > 0 ? 1 : 0)) * kTokBox * 128u;
            const int32_t ty0 = w.row0 + int(rank) * half;
            const int32_t wrow = wrow_of(w);
            for (int kb = 0; kb < nkb; ++kb, ++it, r.next(S)) {
                const uint32_t sl = r.sl;
                if (!ptx::mbar_wait_sleep(&st_free[sl], r.ph ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (int64_t(it) == a.drop_it) continue;   // test hook: this stage never fills
                if (lane == 0) {
                    uint8_t* sp = smem + size_t(sl) * a.stage_bytes;
                    const bool scales = a.scale_tma != 0;   // the group of four blocks of this stage
                    // the item's form for the MMA issuer, released with the stage's
                    // barrier (and, through the dequantisers' arrival, its operand barrier)
                    stage_nc[sl] = nc;
                    ptx::mbar_arrive_expect_tx(&ld_full[sl], a.raw_bytes + (scales ? kSBytes : 0u));
                    ptx::tma_load_2d(sp + a.off_raw, &a.tm_w, kb * (kK / PACK), wrow, &ld_full[sl]);
                    if (scales)
                        ptx::tma_load_2d(sp + a.off_s, &a.tm_s, ((kb * kK) >> a.lbs) & ~3, wrow,
                                         &ld_full[sl]);
                    if (leader) ptx::mbar_arrive_expect_tx(&tok_full[sl], tok_bytes);
                    for (int bx = 0; bx < nbox; ++bx)
                        tma_tokens(sp + bx * (kTokBox * 128), &a.tm_b, ty0 + bx * kTokBox, kb,
                                   tok_addr + sl * 8u);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
            for (uint32_t j = it > S ? it - S : 0; j < it; ++j) {
                volatile int never = 0;
                ptx::mbar_wait(&ld_full[j % S], (j / S) & 1u, kDrainWaitNs, &never);
                if (leader) ptx::mbar_wait(&tok_full[j % S], (j / S) & 1u, kDrainWaitNs, &never);
            }
        }
    } else if (warp == 1) {
        // --------------------------- MMA issuer (CTA 0) ---------------------------
        if (leader) {
            uint32_t item_it = 0;
            Ring r;
            bool ok = true, issued = false;
            for (int64_t i = first; i < items && ok; i += step, ++item_it) {
                const uint32_t b = item_it & 1u;
                // tokens as M: A = token rows (stage offset 0), B = weight rows; tokens as
                // N: A = weight rows, B = the nc token rows (nc from the item's first stage)
                uint32_t idesc = 0, a_off = 0, b_off = 0;
                // both CTAs' epilogues released this accumulator: acquire at cluster scope
                if (!ptx::mbar_wait_cluster(&acc_empty[b], ((item_it >> 1) & 1u) ^ 1u,
                                                              a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + b * kAccCols;
                for (int kb = 0; kb < nkb; ++kb, r.next(S)) {
                    const uint32_t sl = r.sl;
                    // both CTAs' weight rows converted and (through CTA 0's dequantisers,
                    // which wait for them) both CTAs' token rows landed
                    if (!ptx::mbar_wait(&op_full[sl], r.ph, a.wait_ns, &abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (kb == 0) {
                        const int nc = *reinterpret_cast<volatile int*>(&stage_nc[sl]);
                        idesc = f16_idesc(2 * kRowsCta, nc);
                        a_off = a.off_b;   // A: the dequantised weight rows
                        b_off = 0u;        // B: the nc token columns
                    }
                    if (lane == 0) {
                        const uint32_t sp = sbase + sl * a.stage_bytes;
                        const uint32_t sa = sp + a_off;
                        const uint32_t sb = sp + b_off;
#pragma unroll
                        for (int kk = 0; kk < kK / 16; ++kk)
                            mma_pair(d, sw128_desc(sa + 32u * kk), sw128_desc(sb + 32u * kk), idesc,
                                     (kb | kk) != 0 ? 1u : 0u);
                        commit_both(&st_free[sl]);
                        issued = true;
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) commit_both(&acc_full[b]);
                __syncwarp();
            }
            if (!ok && lane == 0) {
                record_error(a.err, QMOE_DEVERR_TIMEOUT);
                abort_flag = 1;
            }
            if (lane == 0 && issued) {
                // every MMA this thread issued completes before tensor memory is released
                commit_local(&drain_bar);
                volatile int never = 0;
                ptx::mbar_wait(&drain_bar, 0, kDrainWaitNs, &never);
            }
            __syncwarp();
        }
    } else if (warp < kEpiWarp0 && warp != 5 && warp != 9) {
        // ------------------------------ dequantisers ------------------------------
        // two groups of four warps take alternate stages; a thread converts one whole
        // weight row (64 K values) of its group's stages
        const int d = warp - 2 - (warp > 5 ? 1 : 0) - (warp > 9 ? 1 : 0);   // 0..7
        const int grp = d / kDeqGroupWarps;                          // 0 or 1
        const int rr = (d % kDeqGroupWarps) * 32 + lane;             // weight row of this CTA's 128
        const uint32_t op_addr = ptx::leader_addr(&op_full[0]);
        uint32_t it = 0;
        Ring r;
        bool ok = true;
        for (int64_t i = first; i < items && ok; i += step) {
            const Item w = pair_item(a, i);
            const int64_t row = int64_t(w.m) * kTileRows + int(rank) * kRowsCta + rr;
            const bool valid = row < a.N;
            const float* srow = a.scales + (int64_t(w.e) * a.N + (valid ? row : 0)) * a.nb;
            for (int kb = 0; kb < nkb; ++kb, ++it, r.next(S)) {
                if (int(it & 1u) != grp) continue;
                const uint32_t sl = r.sl;
                if (!ptx::mbar_wait_sleep(&ld_full[sl], r.ph, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sp = ptx::launder(sbase + sl * a.stage_bytes);
                // block scales of the four 16-wide quarters of this stage's K range (the
                // group of four staged blocks starting at block ((kb * 64) >> lbs) & ~3);
                // column-wise scales are applied to the accumulator instead
                __half2 sq[4];
                if (SCOL) {
                    sq[0] = sq[1] = sq[2] = sq[3] = __float2half2_rn(1.f);
                } else {
                    float4 s4;
                    const int b0 = (kb * kK) >> a.lbs;                 // block of K value 0
                    if (a.scale_tma) {
                        s4 = ptx::ld_f32x4(sp + a.off_s + uint32_t(rr) * 16u);
                    } else {
                        const int g0 = b0 & ~3;
                        s4.x = valid && g0 < a.nb ? __ldg(srow + g0) : 0.f;
                        s4.y = valid && g0 + 1 < a.nb ? __ldg(srow + g0 + 1) : 0.f;
                        s4.z = valid && g0 + 2 < a.nb ? __ldg(srow + g0 + 2) : 0.f;
                        s4.w = valid && g0 + 3 < a.nb ? __ldg(srow + g0 + 3) : 0.f;
                    }
                    if (a.lbs >= 6) {              // one block for the whole stage
                        const __half2 v = __float2half2_rn(pick4(s4, b0 & 3));
                        sq[0] = sq[1] = sq[2] = sq[3] = v;
                    } else if (a.lbs == 5) {       // blocks of 32: two per stage
                        sq[0] = sq[1] = __float2half2_rn(pick4(s4, b0 & 3));
                        sq[2] = sq[3] = __float2half2_rn(pick4(s4, (b0 & 3) + 1));
                    } else {                       // blocks of 16: four per stage
                        sq[0] = __float2half2_rn(s4.x);
                        sq[1] = __float2half2_rn(s4.y);
                        sq[2] = __float2half2_rn(s4.z);
                        sq[3] = __float2half2_rn(s4.w);
                    }
                }
                const uint32_t brow = sp + a.off_b + uint32_t(rr) * 128u;
                const uint32_t rawb = sp + a.off_raw;
                if (BITS == 4) {
                    // 32 packed bytes (64 codes) staged with the 32-byte swizzle: 16-byte
                    // piece c of row r sits at piece c ^ ((r >> 2) & 1)
                    const uint32_t x = uint32_t(rr >> 2) & 1u;
                    const uint4 p0 = ptx::lds128(rawb + uint32_t(rr) * 32u + ((0u ^ x) << 4));
                    const uint4 p1 = ptx::lds128(rawb + uint32_t(rr) * 32u + ((1u ^ x) << 4));
                    const uint32_t wv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                    const __half2 inv16 = __float2half2_rn(0.0625f);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {   // word q: K 8q .. 8q + 7 -> 16-byte piece q
                        uint32_t o[4];
                        if (SCOL) deq4<false>(wv[q], sq[0], inv16, o);
                        else deq4<true>(wv[q], sq[q >> 1], __hmul2(sq[q >> 1], inv16), o);
                        const uint32_t addr = brow + ((uint32_t(q) ^ uint32_t(rr & 7)) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(o[0]),
                                     "r"(o[1]), "r"(o[2]), "r"(o[3])
                                     : "memory");
                    }
                } else {
                    // 64 packed bytes staged with the 64-byte swizzle: 16-byte piece c of
                    // row r sits at piece c ^ ((r >> 1) & 3)
                    const uint32_t x = uint32_t(rr >> 1) & 3u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {   // piece c: K 16c .. 16c + 15
                        const uint4 pc = ptx::lds128(rawb + uint32_t(rr) * 64u + ((uint32_t(c) ^ x) << 4));
                        const uint32_t wv[4] = {pc.x, pc.y, pc.z, pc.w};
                        uint32_t o[8];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (SCOL) deq8<false>(wv[q], sq[0], o + 2 * q);
                            else deq8<true>(wv[q], sq[c], o + 2 * q);
                        }
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint32_t addr =
                                brow + ((uint32_t(2 * c + hh) ^ uint32_t(rr & 7)) << 4);
                            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr),
                                         "r"(o[4 * hh]), "r"(o[4 * hh + 1]), "r"(o[4 * hh + 2]),
                                         "r"(o[4 * hh + 3])
                                         : "memory");
                        }
                    }
                }
                // the dequantised weight rows are the A operand: only this CTA's tensor core
                // reads them
                ptx::fence_proxy_async();
                __syncwarp();
                // CTA 0's arrival also stands for the token rows of both CTAs, whose copies
                // complete on CTA 0's token barrier
                if (leader && !ptx::mbar_wait(&tok_full[sl], r.ph, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) arrive_remote(op_addr + sl * 8u);
            }
        }
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
        }
    } else if (warp >= kEpiWarp0) {
        // -------------------------------- epilogue --------------------------------
        const int ew = warp - kEpiWarp0;           // 0..7
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int chalf = ew >> 2;                 // column half: weight rows 128 * chalf ..
        const uint32_t empty_addr = ptx::leader_addr(&acc_empty[0]);
        // outputs outside the fp16 range: the largest magnitude and a NaN-propagating
        // sum of every output this lane stores, checked once at the end
        float omax = 0.f, osum = 0.f;
        uint32_t item_it = 0;
        for (int64_t i = first; i < items; i += step, ++item_it) {
            const Item w = pair_item(a, i);
            const uint32_t b = item_it & 1u;
            const int nc = item_ncols(w);
            // the slots and routing weights of this lane's tokens in the warp's blocks (FC2)
            int tslot[kTileRows / 64];
            float tp[kTileRows / 64];
#pragma unroll
            for (int m = 0; m < kTileRows / 64; ++m) {
                const int tok = chalf * 32 + 64 * m + lane;
                tslot[m] = 0;
                tp[m] = 0.f;
                if (!FC1 && tok < w.rows) tslot[m] = __ldg(a.perm + w.row0 + tok);
            }
#pragma unroll
            for (int m = 0; m < kTileRows / 64; ++m)
                if (!FC1 && chalf * 32 + 64 * m + lane < w.rows) tp[m] = __ldg(a.pw + tslot[m]);
            if (!ptx::mbar_wait_sleep(&acc_full[b], (item_it >> 1) & 1u, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    record_error(a.err, QMOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            epilogue_tokens_as_n<BITS, FC1, SCOL>(
                a, w, nc, tmem_base + (uint32_t(quad * 32) << 16) + b * kAccCols,
                sbase + a.off_epi + uint32_t(ew) * 2048u, int(rank), quad, chalf, lane, tslot, tp,
                omax, osum);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(empty_addr + b * 8u);
        }
        const bool bad = !(omax <= 65504.f) || osum != osum;
        if (__any_sync(kFull, bad) && lane == 0) record_error(a.err, QMOE_DEVERR_NONFINITE);
    }

    tc_fence_before();
    ptx::cluster_sync();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kTmemCols)
                     : "memory");
}

template <int BITS, bool FC1, bool SCOL>
cudaError_t launch_pair(const PairArgs& args, int pairs, size_t smem, cudaStream_t s) {
    auto kern = pair_gemm_kernel<BITS, FC1, SCOL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * unsigned(pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BITS, bool FC1, bool SCOL>
int max_pairs(size_t smem) {
    auto kern = pair_gemm_kernel<BITS, FC1, SCOL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) return 0;
    return clusters;
}

int ilog2(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return l;
}

// Weight tiles per item group: a divisor of the expert's weight-tile count, at
// most 16 (a group's weight tiles and the expert's token tiles stay in L2).
int pick_group(int n_mt) {
    for (int g = 16; g > 1; --g)
        if (n_mt % g == 0) return g;
    return 1;
}

}  // namespace

int grouped_tile_tokens() { return kTileRows; }

bool grouped_shape_ok(const Problem& p) {
    if (p.H % kK != 0 || p.I % kK != 0) return false;
    return true;
}

cudaError_t launch_grouped_fc(const Problem& p, const Plan& pl, const Work& w, bool fc1,
                              cudaStream_t s) {
    PairArgs a;
    std::memset(&a, 0, sizeof(a));
    const uint8_t* wt = fc1 ? p.w1 : p.w2;
    a.N = fc1 ? p.fusion * p.I : p.H;
    a.K = fc1 ? p.H : p.I;
    a.n_out = fc1 ? p.I : p.H;
    a.nb = int(fc1 ? p.nb1 : p.nb2);
    a.lbs = p.bs ? ilog2(p.bs) : -1;
    a.scales = fc1 ? p.s1 : p.s2;
    const int pack = p.pack;
    // packed rows: 32 bytes per stage (4-bit) or 64 (8-bit), staged with the 32- or
    // 64-byte swizzle so that the dequantisers' reads of a row's pieces spread over
    // all banks
    if (!encode_tmap_2d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt, uint64_t(a.K / pack),
                        uint64_t(p.E * a.N), uint64_t(a.K / pack), uint32_t(kK / pack), kRowsCta,
                        pack == 1 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorInvalidValue;
    a.bsrc = fc1 ? w.xs16 : static_cast<const __half*>(w.act);
    a.srows = pl.srows;
    {
        const uint64_t dims[3] = {uint64_t(kK), uint64_t(pl.srows), uint64_t(a.K / kK)};
        const uint64_t strides[2] = {uint64_t(kK) * 2, uint64_t(pl.srows) * kK * 2};
        const uint32_t box[3] = {uint32_t(kK), uint32_t(kTokBox), 1u};
        if (!encode_tmap_3d(&a.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.bsrc, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    a.scale_tma = (p.bs != 0 && a.nb % 4 == 0) ? 1 : 0;
    if (a.scale_tma &&
        !encode_tmap_2d(&a.tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.scales, uint64_t(a.nb),
                        uint64_t(p.E * a.N), uint64_t(a.nb) * 4, 4, kRowsCta,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    a.tiles = w.tiles;
    a.counts = w.counts;
    a.perm = w.perm;
    a.pw = w.pw;
    a.n_mt = int((a.N + kTileRows - 1) / kTileRows);
    a.gm = pick_group(a.n_mt);
    a.act_out = static_cast<__half*>(w.act);
    a.act = p.act;
    a.has_limit = p.has_limit;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.limit = p.limit;
    a.slot16 = reinterpret_cast<__half*>(w.slot_out);
    a.err = w.ctrl;
    a.wait_ns = wait_limit_ns();
    a.drop_it = drop_stage();
    // stage: token rows | dequantised weight rows | packed rows | staged scales (block-wise
    // only); after the ring, the epilogue's staging tiles
    a.raw_bytes = uint32_t(kRowsCta * (kK / pack));
    a.off_b = kABytes;
    a.off_raw = kABytes + kBBytes;
    a.off_s = a.off_raw + a.raw_bytes;
    a.stage_bytes = (a.off_s + (p.bs != 0 ? kSBytes : 0u) + 1023u) & ~1023u;
    const size_t smem_cap = 232448 - 1024;   // 227 KB per CTA, minus static shared memory
    const size_t epi = size_t(kEpiWarps) * 2048;
    a.nstages = uint32_t(std::min<size_t>(kMaxStages, (smem_cap - 1024 - epi) / a.stage_bytes));
    if (a.nstages < 2) return cudaErrorInvalidValue;
    a.off_epi = a.nstages * a.stage_bytes;
    const size_t smem = 1024 + size_t(a.nstages) * a.stage_bytes + epi;
    const bool scol = p.bs == 0;
    int cap = 0;
#define QMOE_PAIR_CAP(B, C) (fc1 ? max_pairs<B, true, C>(smem) : max_pairs<B, false, C>(smem))
    if (p.bits == 4) cap = scol ? QMOE_PAIR_CAP(4, true) : QMOE_PAIR_CAP(4, false);
    else cap = scol ? QMOE_PAIR_CAP(8, true) : QMOE_PAIR_CAP(8, false);
#undef QMOE_PAIR_CAP
    if (cap <= 0) cap = device_sm_count() / 2;
    const int64_t items_max = pl.max_tiles * a.n_mt;
    const int pairs = int(std::max<int64_t>(1, std::min<int64_t>(items_max, cap)));
    const int kid = fc1 ? QMOE_KERNEL_FC1 : QMOE_KERNEL_FC2;
    note_launch(kid, s, true);
    cudaError_t e;
#define QMOE_PAIR_LAUNCH(B, C) \
    (fc1 ? launch_pair<B, true, C>(a, pairs, smem, s) : launch_pair<B, false, C>(a, pairs, smem, s))
    if (p.bits == 4) e = scol ? QMOE_PAIR_LAUNCH(4, true) : QMOE_PAIR_LAUNCH(4, false);
    else e = scol ? QMOE_PAIR_LAUNCH(8, true) : QMOE_PAIR_LAUNCH(8, false);
#undef QMOE_PAIR_LAUNCH
    note_launch(kid, s, false);
    return e;
}

}  // namespace qmoe
