// Decode path of the QMoE layer: split-K weight-streaming GEMV for few tokens.
//
// QMoE manifest: passes QMoE.FC1ActivationStageGemv / QMoE.OutputStageGemv
// (derive.decodeContract, splitFc1Blocks) give the idea: when few tokens are
// routed, the layer is bound by the bytes of the touched experts' weights.
// Here each weight byte is read from HBM exactly once per call: a work unit
// is (touched expert, 128-row block, K split) and covers every token routed
// to that expert (at most 16).
//
// Per CTA (one per SM, persistent): warp 0 is a TMA producer that fills a
// 3-stage ring in shared memory with
//   - the unit's 128 weight rows x 256 packed bytes (two 128-byte-swizzled
//     2-D tensor boxes),
//   - the matching block scales (one 2-D box),
//   - the routed tokens' fp16 activation rows for this K chunk (1-D bulk
//     copies gathered by the expert permutation);
// warps 1..8 each own 16 weight rows: they dequantize w = (q - mid) * scale
// into fp16 registers (LOP3/PRMT magic-number conversion, exact for the
// integer part) and run mma.sync m16n8k16 with the tokens as the N side,
// accumulating in fp32.  FC1 applies ReLU / interleaved SwiGLU in the
// epilogue and writes fp16 activations; FC2 writes fp32 per-slot partial
// sums per K split, reduced in fixed order by the combine kernel.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "ptx.cuh"
#include "qkv_internal.h"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr int kDecRowGroups = 8;               // 16-row MMA groups per unit
constexpr int kDecKParts = 2;                  // consumer warps per row group (K split among them)
constexpr int kDecConsumers = kDecKParts * kDecRowGroups;
constexpr int kDecThreads = 32 * (1 + kDecConsumers);
constexpr int kDecStages = 4;                  // upper bound; the launch picks what fits
constexpr int kDecRows = 16 * kDecRowGroups;   // 128 weight rows per unit
constexpr int kDecRedBytes = kDecKParts > 1 ? 2 * kDecRowGroups * 32 * 8 * 4 : 0;
constexpr int kChunkBytes = 256;               // packed bytes per row per stage
constexpr int kBoxBytes = 128;                 // one 128-byte swizzle span
constexpr int kBoxTile = kBoxBytes * kDecRows; // 16 KB per weight box
constexpr int kDecMaxTokens = 16;
constexpr unsigned kFull = 0xffffffffu;
// Bound on the waits that drain a CTA's own copies / MMAs before it exits after
// a timeout: independent of the (possibly tiny) configured wait limit.
constexpr uint64_t kDrainWaitNs = 200000000ull;

// Where the dequantization scale is applied.
constexpr int kScaleCol = 0;    // column-wise: once per output, after the K loop
constexpr int kScalePost = 1;   // block-wise, each 32-K MMA pair inside one block: fp32 per pair
constexpr int kScalePre = 2;    // block size 16 with 4-bit codes: fp16 weights pre-scaled

struct DecodeArgs {
    CUtensorMap tm_w;           // packed weights [E*N rows, K/pack bytes], 128B swizzle
    CUtensorMap tm_s;           // block scales [E*N rows, nb] fp32
    const float* scales_col;    // column-wise scales [E*N] (null when block-wise)
    const __half* b_src;        // FC1: x16 [T, b_pitch]; FC2: act16 [slots, b_pitch]
    int64_t b_pitch;
    const int32_t* perm;
    const int32_t* counts;
    const int32_t* offsets;
    const int32_t* active;
    const int32_t* tiles;       // tiles[1] = number of touched experts
    int64_t N, K;
    int topk, n_rb, nkc, splits, cps, lbs, nsc;
    uint32_t stage_bytes, off_s, off_b, pitch_b, nstages;
    __half* act_out;
    int64_t act_pitch;
    int act, act_mode, has_limit;   // act_mode: 2 = 4-bit operand layout, 0 = natural
    float alpha, beta, limit;
    float* slot_out;
    int64_t slots;
    int32_t* err;
    uint64_t wait_ns;
    int64_t drop_it;            // test hook: stage whose copies the producer skips
};

// Position in the stage ring: slot and the parity of its current phase.
struct Ring {
    uint32_t st = 0, ph = 0;
    __device__ __forceinline__ void advance(uint32_t n) {
        if (++st == n) {
            st = 0;
            ph ^= 1u;
        }
    }
};

__device__ __forceinline__ void record_error(int32_t* err, int code) {
    atomicCAS(err, 0, code);
}

// Eight 4-bit codes of `w` (low nibble first, element e in bits 4e..4e+3) ->
// four fp16 pairs, each exact and each 1160 above its weight:
//   h[0] = 1152 + (q0, q4)         h[1] = 1152 + (q2, q6)        (low nibbles of each byte)
//   h[2] = 1032 + 16 * (q1, q5)    h[3] = 1032 + 16 * (q3, q7)   (high nibbles, kept in place)
// A nibble OR-ed into the mantissa of fp16 1152 gives 1152 + q; a high nibble
// left at bits 4..7 of fp16 1032 gives 1032 + 16 q.  The activations feeding
// the high pairs are stored divided by 16, so every pair is (q - 8) + 1160 in
// units of its activation: (1152 + q) - 1160 = q - 8 and
// (1032 + 16 q) - 1160 = 16 (q - 8).
__device__ __forceinline__ void biased4(uint32_t w, uint32_t* h) {
    const uint32_t w8 = w >> 8;
    h[0] = ptx::and_or(w, 0x000F000Fu, 0x64806480u);
    h[1] = ptx::and_or(w8, 0x000F000Fu, 0x64806480u);
    h[2] = ptx::and_or(w, 0x00F000F0u, 0x64086408u);
    h[3] = ptx::and_or(w8, 0x00F000F0u, 0x64086408u);
}

// As biased4 with the offset removed: h[0], h[1] = q - 8; h[2], h[3] = 16 (q - 8).
__device__ __forceinline__ void dequant4(uint32_t w, uint32_t* h) {
    const __half2 bias = ptx::u32_as_h2(0x64886488u);   // (1160, 1160)
    biased4(w, h);
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(h[q]), bias));
}

// As dequant4, every pair multiplied by the fp16 scale (block size 16).
__device__ __forceinline__ void dequant4_scaled(uint32_t w, __half2 s, uint32_t* h) {
    dequant4(w, h);
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = ptx::h2_as_u32(__hmul2(ptx::u32_as_h2(h[q]), s));
}

// Four 8-bit codes -> two fp16 pairs ((q0,q1),(q2,q3)) holding q - 128 exactly.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t* h) {
    const __half2 bias = ptx::u32_as_h2(0x64806480u);   // (1152, 1152)
    const uint32_t lo = ptx::prmt(w, 0x64646464u, 0x4140u);
    const uint32_t hi = ptx::prmt(w, 0x64646464u, 0x4342u);
    h[0] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(lo), bias));
    h[1] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(hi), bias));
}

__device__ __forceinline__ float swiglu(float g, float u, float alpha, float beta, int has_limit,
                                        float limit) {
    if (has_limit) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    return __fdividef(g, 1.f + __expf(-alpha * g)) * (u + beta);
}

// Position of activation column j in a row stored with 8-groups in the
// order 0,4,2,6,1,5,3,7 (pairs (0,4),(2,6) meet low nibbles, (1,5),(3,7) high).
__device__ __forceinline__ int64_t perm8(int64_t j) {
    const int q = int(j & 3);
    const int slot = (q & 1) ? 2 + (q >> 1) : (q >> 1);
    return (j & ~int64_t(7)) + 2 * slot + ((j >> 2) & 1);
}

// Stores activation v of column j in the layout the 4-bit FC2 reads (mode 2:
// pair order above, odd columns divided by 16) or in natural order (mode 0).
__device__ __forceinline__ void store_act(__half* row, int64_t j, float v, int mode) {
    if (mode == 2) row[perm8(j)] = __float2half_rn((j & 1) ? v * 0.0625f : v);
    else row[j] = __float2half_rn(v);
}

// Expert of work unit u (units are ordered expert-major: touched expert, then
// 128-row block, then K split), or -1 past the last unit.
__device__ __forceinline__ int unit_expert(const DecodeArgs& a, int64_t u, int64_t units) {
    return u < units ? __ldg(a.active + u / (int64_t(a.splits) * a.n_rb)) : -1;
}

// Shared-memory byte offsets of one consumer thread relative to a stage's base.
// Consumer warp (row group rgi, K part kh) owns rows r_g = 16 rgi + g and
// r_g + 8 of the unit and the 64-byte segments s = kh, kh + kDecKParts, ... of each
// row's 256 packed bytes; lane (g, c) reads word c of every 16-byte chunk.
struct ThreadOffsets {
    uint32_t a[2][4];   // A word of row r_g in step i of an even / odd segment
                        // (128-byte swizzle applied; first box)
    uint32_t b;         // B fragment of token row g at step 0 of the warp's first segment
    uint32_t b8;        // the same for token row g + 8
    uint32_t s;         // block scales of row r_g for the warp's first segment (post-scaled)
                        // or the scale of its step 0 (pre-scaled)
    uint32_t s8;        // distance from row r_g's scales to row r_g + 8's
};

// The NBS block scales of one row that one 64-byte segment spans (fp32, or
// fp16 when SH).
template <int NBS, bool SH = false>
__device__ __forceinline__ void load_seg_scales(uint32_t addr, float* v) {
    if constexpr (SH) {
        if (NBS == 4) {
            const uint2 t = ptx::ld_u32x2(addr);
            const float2 a = __half22float2(ptx::u32_as_h2(t.x)), b = __half22float2(ptx::u32_as_h2(t.y));
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else if (NBS == 2) {
            const float2 a = __half22float2(ptx::u32_as_h2(ptx::ld_u32(addr)));
            v[0] = a.x; v[1] = a.y;
        } else {
            v[0] = __half2float(__ushort_as_half(uint16_t(ptx::ld_u32(addr & ~3u) >> ((addr & 2u) * 8u))));
        }
        return;
    }
    if (NBS == 4) {
        const float4 t = ptx::ld_f32x4(addr);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else if (NBS == 2) {
        const float2 t = ptx::ld_f32x2(addr);
        v[0] = t.x; v[1] = t.y;
    } else {
        v[0] = ptx::ld_f32(addr);
    }
}

// All MMAs of one pipeline stage for one consumer warp.  nsp = how many of the
// warp's two segments the stage holds (fewer on a ragged last chunk).  NT =
// token tiles of 8 (2 when more than 8 tokens are routed to the expert).
// Block-scaled codes accumulate one scale block in a scratch accumulator
// (exact integer weights times fp16 activations) and fold it into acc with
// the block's fp32 scale; column-wise codes accumulate directly and are scaled
// after the K loop; 4-bit codes with 16-element blocks are pre-scaled in fp16.
template <int BITS, int SMODE, int NBS, int NT, bool SH = false>
__device__ __forceinline__ void consume_stage(uint32_t sA, const ThreadOffsets& o, int nsp, bool ld0,
                                              bool ld1, uint4 (&bq)[NT], float (&acc)[NT][4],
                                              float (&accB)[NT][4]) {
    constexpr int SPW = 4 / kDecKParts;                    // segments per warp per stage
    constexpr uint32_t kSegB = (BITS == 4 ? 256u : 128u) * kDecKParts;   // B bytes between them
    constexpr uint32_t kStepB = BITS == 4 ? 64u : 32u;    // B bytes per step
    constexpr int IPB = NBS > 0 ? 4 / NBS : 1;            // steps per scale block
#pragma unroll
    for (int sp = 0; sp < SPW; ++sp) {
        if (sp >= nsp) break;
        // segment s = kh + kDecKParts * sp: box s / 2, parity s % 2 (kh is folded into o)
        const int par = kDecKParts == 1 ? (sp & 1) : 0;
        const uint32_t box = uint32_t(kDecKParts == 1 ? (sp >> 1) : (kDecKParts * sp) >> 1) * kBoxTile;
        float sg[4], s8[4];
        if constexpr (SMODE == kScalePost) {
            const uint32_t sa = sA + o.s + uint32_t(kDecKParts * sp * NBS) * (SH ? 2u : 4u);
            load_seg_scales<NBS, SH>(sa, sg);
            load_seg_scales<NBS, SH>(sa + o.s8, s8);
        }
        float tmp[NT][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t aw = sA + o.a[par][i] + box;
            const uint32_t wa = ptx::ld_u32(aw);
            const uint32_t wb = ptx::ld_u32(aw + 8u * kBoxBytes);
            // B fragment: 8 fp16 (16 bytes) per step for 4-bit codes, 4 (8 bytes) for
            // 8-bit.  Lanes of token rows >= ne skip the load (no shared-memory
            // traffic) and keep stale registers, which only reach output columns
            // that are never stored.
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t ba = sA + (nt ? o.b8 : o.b) + uint32_t(sp) * kSegB + uint32_t(i) * kStepB;
                if constexpr (BITS == 4)
                    ptx::ld128_pred(bq[nt], ba, nt ? ld1 : ld0);
                else
                    ptx::ld64_pred(bq[nt].x, bq[nt].y, ba, nt ? ld1 : ld0);
            }
            const bool first = i % IPB == 0, last = i % IPB == IPB - 1;
            if constexpr (BITS == 4 && SMODE == kScalePost) {
                uint32_t ha[4], hb[4];
                dequant4(wa, ha);
                dequant4(wb, hb);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    // low pairs (K 0,4 | 2,6) with b.x|b.y; high pairs (K 1,5 | 3,7) with b.z|b.w
                    if (first)
                        ptx::mma_16816_z(tmp[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                    else
                        ptx::mma_16816(tmp[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                    ptx::mma_16816(tmp[nt], ha[2], hb[2], ha[3], hb[3], bq[nt].z, bq[nt].w);
                    if (last) {
                        acc[nt][0] = fmaf(sg[i / IPB], tmp[nt][0], acc[nt][0]);
                        acc[nt][1] = fmaf(sg[i / IPB], tmp[nt][1], acc[nt][1]);
                        acc[nt][2] = fmaf(s8[i / IPB], tmp[nt][2], acc[nt][2]);
                        acc[nt][3] = fmaf(s8[i / IPB], tmp[nt][3], acc[nt][3]);
                    }
                }
            } else if constexpr (BITS == 4) {
                uint32_t ha[4], hb[4];
                if constexpr (SMODE == kScalePre) {
                    const uint32_t sa = sA + o.s + uint32_t(32 * kDecKParts * sp + 8 * i);
                    dequant4_scaled(wa, __float2half2_rn(ptx::ld_f32(sa)), ha);
                    dequant4_scaled(wb, __float2half2_rn(ptx::ld_f32(sa + o.s8)), hb);
                } else {
                    dequant4(wa, ha);
                    dequant4(wb, hb);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    ptx::mma_16816(acc[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                    ptx::mma_16816(accB[nt], ha[2], hb[2], ha[3], hb[3], bq[nt].z, bq[nt].w);
                }
            } else {
                uint32_t ha[2], hb[2];
                dequant8(wa, ha);
                dequant8(wb, hb);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (SMODE == kScalePost) {
                        if (first)
                            ptx::mma_16816_z(tmp[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                        else
                            ptx::mma_16816(tmp[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                        if (last) {
                            acc[nt][0] = fmaf(sg[i / IPB], tmp[nt][0], acc[nt][0]);
                            acc[nt][1] = fmaf(sg[i / IPB], tmp[nt][1], acc[nt][1]);
                            acc[nt][2] = fmaf(s8[i / IPB], tmp[nt][2], acc[nt][2]);
                            acc[nt][3] = fmaf(s8[i / IPB], tmp[nt][3], acc[nt][3]);
                        }
                    } else if (i & 1) {
                        ptx::mma_16816(accB[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                    } else {
                        ptx::mma_16816(acc[nt], ha[0], hb[0], ha[1], hb[1], bq[nt].x, bq[nt].y);
                    }
                }
            }
        }
    }
}

// The K loop of one unit for one consumer warp: waits for each stage, runs its
// MMAs and releases it.  Returns false when a wait gave up.  On return, out
// holds the warp's partial sums (column-wise scales applied).
template <int BITS, int SMODE, int NBS, int NT, bool SH = false, typename Args = DecodeArgs>
__device__ __forceinline__ bool consume_unit(const Args& a, uint64_t* full_bar,
                                             uint64_t* empty_bar, volatile int* abort_flag,
                                             uint32_t sbase0, const ThreadOffsets& o, Ring& ring,
                                             int c0, int c1, int tail_nsp, int ne, int g, int lane,
                                             float scol_g, float scol_g8, float (&out)[2][4]) {
    constexpr bool POST = SMODE == kScalePost;
    float acc[NT][4], accB[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = accB[nt][q] = 0.f;
    uint4 bq[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) bq[nt] = make_uint4(0u, 0u, 0u, 0u);
    const bool ld0 = g < ne, ld1 = g + 8 < ne;
    for (int kc = c0; kc < c1; ++kc, ring.advance(a.nstages)) {
        if (!ptx::mbar_wait(&full_bar[ring.st], ring.ph, a.wait_ns, abort_flag)) {
            if (lane == 0) {
                record_error(a.err, QMOE_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            return false;
        }
        const uint32_t sA = ptx::launder(sbase0 + ring.st * a.stage_bytes);
        // the warp's segments in this chunk: both, except on a ragged last chunk
        const int nsp = kc == a.nkc - 1 ? tail_nsp : 4 / kDecKParts;
        consume_stage<BITS, SMODE, NBS, NT, SH>(sA, o, nsp, ld0, ld1, bq, acc, accB);
        // every shared load of this stage feeds the accumulators: finish them first
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ptx::depend(acc[nt][q]);
                if (!POST) ptx::depend(accB[nt][q]);
            }
        __syncwarp();
        ptx::mbar_arrive_if(&empty_bar[ring.st], lane == 0);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int src = nt < NT ? nt : 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float v = 0.f;
            if (nt < NT) v = POST ? acc[src][q] : acc[src][q] + accB[src][q];
            if (SMODE == kScaleCol) v *= q < 2 ? scol_g : scol_g8;
            out[nt][q] = v;
        }
    }
    return true;
}

template <int BITS, int SMODE, int NBS, bool FC1>
__global__ void __launch_bounds__(kDecThreads, 1) decode_gemv_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kDecStages];
    __shared__ __align__(8) uint64_t empty_bar[kDecStages];
    __shared__ __align__(8) uint64_t red_full[2];    // K-half 1 -> K-half 0 partial sums
    __shared__ __align__(8) uint64_t red_empty[2];
    __shared__ int abort_flag;
    // FC2: token-row copies held back until FC1 has completed (see the producer)
    __shared__ const __half* held_src[kDecStages][32];
    __shared__ uint32_t held_meta[kDecStages][3];   // stage slot, bytes, token rows
    constexpr int KC = kChunkBytes * (BITS == 4 ? 2 : 1);   // K values per chunk
    constexpr int SEGK = BITS == 4 ? 128 : 64;              // K values per 64-byte segment
    constexpr bool SCOL = SMODE == kScaleCol;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < a.nstages; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], kDecConsumers);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&red_full[s], kDecRowGroups);
            ptx::mbar_init(&red_empty[s], kDecRowGroups);
        }
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    // the next kernel (FC2 after FC1, the combine after FC2) may start its
    // prologue on SMs this grid leaves
    ptx::griddep_launch_dependents();
    const int n_active = a.tiles[1];
    const int64_t units = int64_t(n_active) * a.n_rb * a.splits;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            ptx::prefetch_tmap(&a.tm_w);
            if (!SCOL) ptx::prefetch_tmap(&a.tm_s);
        }
        uint32_t it = 0;   // stages issued (for the drain after a timeout)
        Ring ring;
        bool ok = true;
        // FC2 is launched as a dependent of FC1: the weight and scale boxes of the
        // first stages are issued at once, the copies of FC1's output (the token
        // rows) only after griddepcontrol.wait.  Up to nstages stages are held back.
        bool dep_done = FC1;
        uint32_t held = 0;
        auto release_held = [&]() {
            ptx::griddep_wait();
            __syncwarp();
            for (uint32_t h = 0; h < held; ++h) {
                const uint32_t hs = held_meta[h][0];
                if (lane < int(held_meta[h][2]))
                    ptx::bulk_g2s(smem + size_t(hs) * a.stage_bytes + a.off_b + lane * a.pitch_b,
                                  held_src[h][lane], held_meta[h][1], &full_bar[hs]);
            }
            held = 0;
            dep_done = true;
        };
        // Unit metadata is a chain of dependent loads (expert -> its token count
        // and offset -> its token rows); it is loaded ahead of use (experts three
        // units ahead, counts two, token rows one) so that the producer never waits
        // on it between units.
        const int64_t G = gridDim.x;
        int64_t u = blockIdx.x;
        int e0 = unit_expert(a, u, units), e1 = unit_expert(a, u + G, units);
        int e2 = unit_expert(a, u + 2 * G, units);
        int ne0 = e0 >= 0 ? __ldg(a.counts + e0) : 0, off0 = e0 >= 0 ? __ldg(a.offsets + e0) : 0;
        int ne1 = e1 >= 0 ? __ldg(a.counts + e1) : 0, off1 = e1 >= 0 ? __ldg(a.offsets + e1) : 0;
        auto token_row = [&](int ne_, int off_) -> int64_t {
            if (lane >= ne_) return 0;
            return FC1 ? int64_t(__ldg(a.perm + off_ + lane) / a.topk) : int64_t(off_ + lane);
        };
        int64_t brow0 = token_row(ne0, off0);
        for (; u < units && ok; u += G) {
            const int e3 = unit_expert(a, u + 3 * G, units);
            const int ne2 = e2 >= 0 ? __ldg(a.counts + e2) : 0;
            const int off2 = e2 >= 0 ? __ldg(a.offsets + e2) : 0;
            const int64_t brow1 = token_row(ne1, off1);
            const int e = e0, ne = ne0;
            const int64_t brow = brow0;
            const int ks = int(u % a.splits);
            const int rb = int((u / a.splits) % a.n_rb);
            const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
            const int32_t row0 = int32_t(int64_t(e) * a.N + int64_t(rb) * kDecRows);
            for (int kc = c0; kc < c1; ++kc, ++it, ring.advance(a.nstages)) {
                const uint32_t st = ring.st;
                // a stage about to be reused needs the held copies of the first round
                if (!dep_done && it >= a.nstages) release_held();
                if (!ptx::mbar_wait_sleep(&empty_bar[st], ring.ph ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                if (int64_t(it) == a.drop_it) continue;   // test hook: this stage never fills
                const int64_t krem = a.K - int64_t(kc) * KC;
                const int kvalid = int(krem < KC ? krem : KC);
                uint8_t* sbase = smem + size_t(st) * a.stage_bytes;
                const uint32_t bbytes = uint32_t(kvalid) * 2u;
                if (lane == 0) {
                    const uint32_t tx = 2u * kBoxTile + (SCOL ? 0u : uint32_t(kDecRows) * a.nsc * 4u) +
                                        uint32_t(ne) * bbytes;
                    ptx::mbar_arrive_expect_tx(&full_bar[st], tx);
                    ptx::tma_load_2d(sbase, &a.tm_w, kc * kChunkBytes, row0, &full_bar[st]);
                    ptx::tma_load_2d(sbase + kBoxTile, &a.tm_w, kc * kChunkBytes + kBoxBytes, row0,
                                     &full_bar[st]);
                    if (!SCOL)
                        ptx::tma_load_2d(sbase + a.off_s, &a.tm_s, kc * a.nsc, row0, &full_bar[st]);
                }
                __syncwarp();
                if (dep_done) {
                    if (lane < ne)
                        ptx::bulk_g2s(sbase + a.off_b + lane * a.pitch_b,
                                      a.b_src + brow * a.b_pitch + int64_t(kc) * KC, bbytes,
                                      &full_bar[st]);
                } else {
                    held_src[held][lane] = a.b_src + brow * a.b_pitch + int64_t(kc) * KC;
                    if (lane == 0) {
                        held_meta[held][0] = st;
                        held_meta[held][1] = bbytes;
                        held_meta[held][2] = uint32_t(ne);
                    }
                    __syncwarp();
                    ++held;
                }
            }
            e0 = e1; ne0 = ne1; off0 = off1; brow0 = brow1;
            e1 = e2; ne1 = ne2; off1 = off2;
            e2 = e3;
        }
        if (!dep_done && held > 0) release_held();
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
            // drain copies still in flight (bounded) before the CTA exits
            for (uint32_t j = it > a.nstages ? it - a.nstages : 0; j < it; ++j) {
                volatile int never = 0;
                ptx::mbar_wait(&full_bar[j % a.nstages], (j / a.nstages) & 1u, kDrainWaitNs, &never);
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    // Warps 1..16: row group rgi (16 rows) x K half kh (alternate 64-byte segments).
    const int cw = warp - 1;
    const int rgi = cw % kDecRowGroups, kh = cw / kDecRowGroups;
    const int g = lane >> 2, c = lane & 3;
    const int r_g = 16 * rgi + g;   // row of this thread inside the 128-row box (and r_g + 8)
    float* red = reinterpret_cast<float*>(smem + size_t(a.nstages) * a.stage_bytes);
    const uint32_t sbase0 = ptx::smem_u32(smem);
    ThreadOffsets o;
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // the warp's segments of parity p (one parity only with two K parts)
            const int par = kDecKParts == 1 ? p : (kh & 1);
            o.a[p][i] = uint32_t(r_g) * kBoxBytes + (uint32_t(((par << 2) + i) ^ g) << 4) +
                        uint32_t(c) * 4u;
        }
    o.b = a.off_b + uint32_t(g) * a.pitch_b +
          (BITS == 4 ? uint32_t(256 * kh + 16 * c) : uint32_t(128 * kh + 8 * c));
    o.b8 = o.b + 8u * a.pitch_b;
    o.s8 = 8u * uint32_t(a.nsc) * 4u;
    if (SMODE == kScalePost) {
        // segment s spans scale blocks s * NBS .. s * NBS + NBS - 1 (block size <= segment)
        o.s = a.off_s + uint32_t(r_g * a.nsc + kh * NBS) * 4u;
    } else {
        // pre-scaled (block size 16): the scale of K index 128 s + 32 i + 8 c
        o.s = a.off_s + uint32_t(r_g * a.nsc) * 4u + uint32_t(32 * kh + 4 * (c >> 1));
    }
    // segments of this warp in the last K chunk (ragged when K is not a multiple of KC)
    const int tail_seg = int((a.K - int64_t(a.nkc - 1) * KC) / SEGK);
    const int tail_nsp = tail_seg > kh ? (tail_seg - kh + kDecKParts - 1) / kDecKParts : 0;
    Ring ring;
    uint32_t un = 0;   // units processed by this CTA (reduction buffer parity)
    // unit metadata loaded ahead of use (experts two units ahead, counts one)
    const int64_t G = gridDim.x;
    int e_cur = unit_expert(a, blockIdx.x, units);
    int ne_cur = e_cur >= 0 ? __ldg(a.counts + e_cur) : 0;
    int off_cur = e_cur >= 0 ? __ldg(a.offsets + e_cur) : 0;
    int e_nxt = unit_expert(a, blockIdx.x + G, units);
    for (int64_t u = blockIdx.x; u < units; u += G, ++un) {
        const int ne_nxt = e_nxt >= 0 ? __ldg(a.counts + e_nxt) : 0;
        const int off_nxt = e_nxt >= 0 ? __ldg(a.offsets + e_nxt) : 0;
        const int e_nn = unit_expert(a, u + 2 * G, units);
        const int e = e_cur, ne = ne_cur, off = off_cur;
        e_cur = e_nxt; ne_cur = ne_nxt; off_cur = off_nxt; e_nxt = e_nn;
        const int ks = int(u % a.splits);
        const int rb = int((u / a.splits) % a.n_rb);
        const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
        // FC2 stores by original slot: fetch the slot ids now, use them after the K loop
        int32_t slot_of[2][2] = {{0, 0}, {0, 0}};
        if (!FC1) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = nt * 8 + 2 * c + q;
                    if (n < ne) slot_of[nt][q] = __ldg(a.perm + off + n);
                }
        }
        const int64_t rg = int64_t(rb) * kDecRows + r_g;   // row within the expert
        const int64_t rg8 = rg + 8;
        float scol_g = 1.f, scol_g8 = 1.f;
        if (SCOL) {
            const float* sc = a.scales_col + int64_t(e) * a.N;
            scol_g = rg < a.N ? sc[rg] : 0.f;
            scol_g8 = rg8 < a.N ? sc[rg8] : 0.f;
        }
        float acc[2][4];
        const bool ok = ne > 8
            ? consume_unit<BITS, SMODE, NBS, 2>(a, full_bar, empty_bar, &abort_flag, sbase0, o, ring,
                                                c0, c1, tail_nsp, ne, g, lane, scol_g, scol_g8, acc)
            : consume_unit<BITS, SMODE, NBS, 1>(a, full_bar, empty_bar, &abort_flag, sbase0, o, ring,
                                                c0, c1, tail_nsp, ne, g, lane, scol_g, scol_g8, acc);
        if (!ok) return;

        // ---- with K parts, part 1 hands its partial sums to part 0 through shared memory ----
        if (kDecKParts > 1) {
        const int rb_buf = int(un & 1u);
        const uint32_t rph = (un >> 1) & 1u;
        float* slot = red + ((rb_buf * kDecRowGroups + rgi) * 32 + lane) * 8;
        if (kh == 1) {
            if (!ptx::mbar_wait(&red_empty[rb_buf], rph ^ 1u, a.wait_ns, &abort_flag)) {
                if (lane == 0) { record_error(a.err, QMOE_DEVERR_TIMEOUT); abort_flag = 1; }
                return;
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) slot[nt * 4 + q] = acc[nt][q];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&red_full[rb_buf]);
            continue;
        }
        if (!ptx::mbar_wait(&red_full[rb_buf], rph, a.wait_ns, &abort_flag)) {
            if (lane == 0) { record_error(a.err, QMOE_DEVERR_TIMEOUT); abort_flag = 1; }
            return;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[nt][q] += slot[nt * 4 + q];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&red_empty[rb_buf]);
        }

        // -------------------------------- epilogue --------------------------------
        if (FC1) {
            if (a.act == QMOE_ACT_SWIGLU) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float pv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) pv[q] = __shfl_down_sync(kFull, acc[nt][q], 4);
                    if ((g & 1) == 0) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int n = nt * 8 + 2 * c + q;
                            if (n >= ne) continue;
                            __half* dst = a.act_out + int64_t(off + n) * a.act_pitch;
                            if (rg < a.N) {
                                const float v = swiglu(acc[nt][q], pv[q], a.alpha, a.beta,
                                                       a.has_limit, a.limit);
                                if (!(fabsf(v) <= 65504.f)) record_error(a.err, QMOE_DEVERR_NONFINITE);
                                store_act(dst, rg >> 1, v, a.act_mode);
                            }
                            if (rg8 < a.N) {
                                const float v = swiglu(acc[nt][2 + q], pv[2 + q], a.alpha, a.beta,
                                                       a.has_limit, a.limit);
                                if (!(fabsf(v) <= 65504.f)) record_error(a.err, QMOE_DEVERR_NONFINITE);
                                store_act(dst, rg8 >> 1, v, a.act_mode);
                            }
                        }
                    }
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int n = nt * 8 + 2 * c + q;
                        if (n >= ne) continue;
                        __half* dst = a.act_out + int64_t(off + n) * a.act_pitch;
                        if (rg < a.N) {
                            const float v = fmaxf(acc[nt][q], 0.f);
                            if (!(v <= 65504.f)) record_error(a.err, QMOE_DEVERR_NONFINITE);
                            store_act(dst, rg, v, a.act_mode);
                        }
                        if (rg8 < a.N) {
                            const float v = fmaxf(acc[nt][2 + q], 0.f);
                            if (!(v <= 65504.f)) record_error(a.err, QMOE_DEVERR_NONFINITE);
                            store_act(dst, rg8, v, a.act_mode);
                        }
                    }
                }
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = nt * 8 + 2 * c + q;
                    if (n >= ne) continue;
                    float* dst = a.slot_out + (int64_t(ks) * a.slots + slot_of[nt][q]) * a.N;
                    if (rg < a.N) dst[rg] = acc[nt][q];
                    if (rg8 < a.N) dst[rg8] = acc[nt][2 + q];
                }
            }
        }
    }
}

template <int BITS, int SMODE, int NBS, bool FC1>
cudaError_t launch_variant(const DecodeArgs& args, int grid, size_t smem, cudaStream_t s) {
    auto kern = decode_gemv_kernel<BITS, SMODE, NBS, FC1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (FC1) {
        kern<<<grid, kDecThreads, smem, s>>>(args);
        return cudaGetLastError();
    }
    // FC2 overlaps FC1's last wave: it waits for FC1 only before reading its output
    return launch_dependent(kern, dim3(grid), dim3(kDecThreads), smem, s, args);
}


// ---------------------------------------------------------------------------
// The same GEMV over the three weight tensors of a Q/K/V projection
// (com.microsoft.MatMulNBitsQkv manifest, pass MatMulNBitsQkv.Projection):
// every row of the input is "routed" to each projection.  A work unit is
// (projection, 128-row block, K split); units of projection 0 come first.
// ---------------------------------------------------------------------------
struct QkvArgs {
    CUtensorMap tm_w[3];        // packed weights [N_p rows, K/2 bytes], 128-byte swizzle
    CUtensorMap tm_s[3];        // block scales [N_p rows, K/32], fp32 or fp16
    const __half* b_src;        // normalised rows [rows, b_pitch], 4-bit operand order
    int64_t b_pitch;
    int64_t N[3];
    int n_rb[3];
    int64_t ubound[2];          // first unit of projection 1 and of projection 2
    int64_t units;
    int64_t K;
    int rows, nkc, splits, cps, nsc;
    uint32_t stage_bytes, off_s, off_b, pitch_b, nstages, ssize;
    float* part[3];             // [splits][rows][N_p] partial sums (splits > 1)
    void* out[3];               // [rows][N_p] results, fp32 or fp16 (out_f16), splits == 1
    int out_f16;
    int32_t* err;
    uint64_t wait_ns;
};

// Result element idx of projection p (K not split).
__device__ __forceinline__ void qkv_store(const QkvArgs& a, int p, int64_t idx, float v) {
    if (a.out_f16) static_cast<__half*>(a.out[p])[idx] = __float2half_rn(v);
    else static_cast<float*>(a.out[p])[idx] = v;
}

template <bool SH>
__global__ void __launch_bounds__(kDecThreads, 1) qkv_gemv_kernel(const __grid_constant__ QkvArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kDecStages];
    __shared__ __align__(8) uint64_t empty_bar[kDecStages];
    __shared__ __align__(8) uint64_t red_full[2];
    __shared__ __align__(8) uint64_t red_empty[2];
    __shared__ int abort_flag;
    __shared__ uint32_t held_meta[kDecStages][3];   // stage slot, bytes, K chunk
    constexpr int KC = kChunkBytes * 2;             // K values per chunk (4-bit codes)
    constexpr int SEGK = 128;
    constexpr int NBS = 4;                          // block size 32: four scales per segment

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < a.nstages; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], kDecConsumers);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&red_full[s], kDecRowGroups);
            ptx::mbar_init(&red_empty[s], kDecRowGroups);
        }
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    ptx::griddep_launch_dependents();
    const int64_t units = a.units;
    auto unit_proj = [&](int64_t u, int64_t* v) {
        const int p = u < a.ubound[0] ? 0 : (u < a.ubound[1] ? 1 : 2);
        *v = u - (p == 0 ? 0 : a.ubound[p - 1]);
        return p;
    };

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0)
            for (int p = 0; p < 3; ++p) {
                ptx::prefetch_tmap(&a.tm_w[p]);
                ptx::prefetch_tmap(&a.tm_s[p]);
            }
        uint32_t it = 0;
        Ring ring;
        bool ok = true;
        // the normalised rows come from the previous kernel: weight and scale boxes
        // of the first stages go out at once, the row copies after griddepcontrol.wait
        bool dep_done = false;
        uint32_t held = 0;
        const int ne = a.rows;
        auto release_held = [&]() {
            ptx::griddep_wait();
            __syncwarp();
            for (uint32_t h = 0; h < held; ++h) {
                const uint32_t hs = held_meta[h][0];
                if (lane < ne)
                    ptx::bulk_g2s(smem + size_t(hs) * a.stage_bytes + a.off_b + lane * a.pitch_b,
                                  a.b_src + int64_t(lane) * a.b_pitch + int64_t(held_meta[h][2]) * KC,
                                  held_meta[h][1], &full_bar[hs]);
            }
            held = 0;
            dep_done = true;
        };
        for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
            int64_t v;
            const int p = unit_proj(u, &v);
            const int ks = int(v % a.splits);
            const int rb = int(v / a.splits);
            const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
            const int32_t row0 = rb * kDecRows;
            for (int kc = c0; kc < c1; ++kc, ++it, ring.advance(a.nstages)) {
                const uint32_t st = ring.st;
                if (!dep_done && it >= a.nstages) release_held();
                if (!ptx::mbar_wait_sleep(&empty_bar[st], ring.ph ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                const int64_t krem = a.K - int64_t(kc) * KC;
                const int kvalid = int(krem < KC ? krem : KC);
                uint8_t* sbase = smem + size_t(st) * a.stage_bytes;
                const uint32_t bbytes = uint32_t(kvalid) * 2u;
                if (lane == 0) {
                    const uint32_t tx = 2u * kBoxTile + uint32_t(kDecRows) * a.nsc * a.ssize +
                                        uint32_t(ne) * bbytes;
                    ptx::mbar_arrive_expect_tx(&full_bar[st], tx);
                    ptx::tma_load_2d(sbase, &a.tm_w[p], kc * kChunkBytes, row0, &full_bar[st]);
                    ptx::tma_load_2d(sbase + kBoxTile, &a.tm_w[p], kc * kChunkBytes + kBoxBytes, row0,
                                     &full_bar[st]);
                    ptx::tma_load_2d(sbase + a.off_s, &a.tm_s[p], kc * a.nsc, row0, &full_bar[st]);
                }
                __syncwarp();
                if (dep_done) {
                    if (lane < ne)
                        ptx::bulk_g2s(sbase + a.off_b + lane * a.pitch_b,
                                      a.b_src + int64_t(lane) * a.b_pitch + int64_t(kc) * KC, bbytes,
                                      &full_bar[st]);
                } else {
                    if (lane == 0) {
                        held_meta[held][0] = st;
                        held_meta[held][1] = bbytes;
                        held_meta[held][2] = uint32_t(kc);
                    }
                    __syncwarp();
                    ++held;
                }
            }
        }
        if (!dep_done && held > 0) release_held();
        if (!ok && lane == 0) {
            record_error(a.err, QMOE_DEVERR_TIMEOUT);
            abort_flag = 1;
            for (uint32_t j = it > a.nstages ? it - a.nstages : 0; j < it; ++j) {
                volatile int never = 0;
                ptx::mbar_wait(&full_bar[j % a.nstages], (j / a.nstages) & 1u, kDrainWaitNs, &never);
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int cw = warp - 1;
    const int rgi = cw % kDecRowGroups, kh = cw / kDecRowGroups;
    const int g = lane >> 2, c = lane & 3;
    const int r_g = 16 * rgi + g;
    float* red = reinterpret_cast<float*>(smem + size_t(a.nstages) * a.stage_bytes);
    const uint32_t sbase0 = ptx::smem_u32(smem);
    ThreadOffsets o;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int par = kDecKParts == 1 ? pp : (kh & 1);
            o.a[pp][i] = uint32_t(r_g) * kBoxBytes + (uint32_t(((par << 2) + i) ^ g) << 4) +
                         uint32_t(c) * 4u;
        }
    o.b = a.off_b + uint32_t(g) * a.pitch_b + uint32_t(256 * kh + 16 * c);
    o.b8 = o.b + 8u * a.pitch_b;
    o.s8 = 8u * uint32_t(a.nsc) * a.ssize;
    o.s = a.off_s + uint32_t(r_g * a.nsc + kh * NBS) * a.ssize;
    const int tail_seg = int((a.K - int64_t(a.nkc - 1) * KC) / SEGK);
    const int tail_nsp = tail_seg > kh ? (tail_seg - kh + kDecKParts - 1) / kDecKParts : 0;
    const int ne = a.rows;
    Ring ring;
    uint32_t un = 0;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++un) {
        int64_t v;
        const int p = unit_proj(u, &v);
        const int ks = int(v % a.splits);
        const int rb = int(v / a.splits);
        const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
        const int64_t rg = int64_t(rb) * kDecRows + r_g;
        const int64_t rg8 = rg + 8;
        float acc[2][4];
        const bool ok = ne > 8
            ? consume_unit<4, kScalePost, NBS, 2, SH>(a, full_bar, empty_bar, &abort_flag,
                                                       sbase0, o, ring, c0, c1, tail_nsp, ne, g, lane,
                                                       1.f, 1.f, acc)
            : consume_unit<4, kScalePost, NBS, 1, SH>(a, full_bar, empty_bar, &abort_flag,
                                                       sbase0, o, ring, c0, c1, tail_nsp, ne, g, lane,
                                                       1.f, 1.f, acc);
        if (!ok) return;
        if (kDecKParts > 1) {
            const int rb_buf = int(un & 1u);
            const uint32_t rph = (un >> 1) & 1u;
            float* slot = red + ((rb_buf * kDecRowGroups + rgi) * 32 + lane) * 8;
            if (kh == 1) {
                if (!ptx::mbar_wait(&red_empty[rb_buf], rph ^ 1u, a.wait_ns, &abort_flag)) {
                    if (lane == 0) { record_error(a.err, QMOE_DEVERR_TIMEOUT); abort_flag = 1; }
                    return;
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int q = 0; q < 4; ++q) slot[nt * 4 + q] = acc[nt][q];
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&red_full[rb_buf]);
                continue;
            }
            if (!ptx::mbar_wait(&red_full[rb_buf], rph, a.wait_ns, &abort_flag)) {
                if (lane == 0) { record_error(a.err, QMOE_DEVERR_TIMEOUT); abort_flag = 1; }
                return;
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[nt][q] += slot[nt * 4 + q];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&red_empty[rb_buf]);
        }
        const int64_t Np = a.N[p];
        if (a.splits == 1) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = nt * 8 + 2 * c + q;
                    if (n >= ne) continue;
                    if (rg < Np) qkv_store(a, p, int64_t(n) * Np + rg, acc[nt][q]);
                    if (rg8 < Np) qkv_store(a, p, int64_t(n) * Np + rg8, acc[nt][2 + q]);
                }
            continue;
        }
        float* part = a.part[p] + int64_t(ks) * a.rows * Np;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int n = nt * 8 + 2 * c + q;
                if (n >= ne) continue;
                if (rg < Np) part[int64_t(n) * Np + rg] = acc[nt][q];
                if (rg8 < Np) part[int64_t(n) * Np + rg8] = acc[nt][2 + q];
            }
    }
}

int ilog2(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return l;
}

}  // namespace

bool qkv_gemv_shape_ok(int64_t K, bool scales_f16) {
    if (K <= 0 || K % 128 != 0) return false;            // whole 64-byte segments per row
    if (scales_f16 && (K / 32) % 8 != 0) return false;    // 16-byte strided fp16 scale rows
    return true;
}

// Split K so that the units (projection x 128-row block x K split) spread evenly
// over the SMs: minimise the K chunks of the most loaded SM, counting 1.5 chunks
// of fixed cost per unit (pipeline ramp, K-half hand-off, stores) and 2 chunks
// for the partial-sum reduction that any split needs.
int qkv_gemv_splits(const int64_t N[3], int64_t K) {
    const int64_t KC = int64_t(kChunkBytes) * 2;
    const int64_t nkc = (K + KC - 1) / KC;
    int64_t n_rb = 0;
    for (int p = 0; p < 3; ++p) n_rb += (N[p] + kDecRows - 1) / kDecRows;
    const int64_t sms = device_sm_count();
    int64_t best = 1;
    double best_cost = 0.0;
    for (int64_t cps = nkc; cps >= 1; --cps) {
        const int64_t splits = (nkc + cps - 1) / cps;
        if ((nkc + splits - 1) / splits != cps) continue;   // same cps as the launch derives
        const int64_t units = n_rb * splits;
        const double cost = double((units + sms - 1) / sms) * (double(cps) + 1.5) +
                            (splits > 1 ? 2.0 : 0.0);
        if (best_cost == 0.0 || cost < best_cost) {
            best_cost = cost;
            best = splits;
        }
    }
    return int(best);
}

cudaError_t launch_qkv_gemv(const QkvGemvParams& q, cudaStream_t s) {
    QkvArgs a;
    std::memset(&a, 0, sizeof(a));
    const int64_t KC = int64_t(kChunkBytes) * 2;
    const int64_t nb = q.K / 32;
    a.nsc = int(KC / 32);
    a.ssize = q.scales_f16 ? 2u : 4u;
    for (int p = 0; p < 3; ++p) {
        if (!encode_tmap_2d(&a.tm_w[p], CU_TENSOR_MAP_DATA_TYPE_UINT8, q.w[p], uint64_t(q.K / 2),
                            uint64_t(q.N[p]), uint64_t(q.K / 2), kBoxBytes, kDecRows,
                            CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        if (!encode_tmap_2d(&a.tm_s[p],
                            q.scales_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                            q.s[p], uint64_t(nb), uint64_t(q.N[p]), uint64_t(nb) * a.ssize,
                            uint32_t(a.nsc), kDecRows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        a.N[p] = q.N[p];
        a.n_rb[p] = int((q.N[p] + kDecRows - 1) / kDecRows);
        a.part[p] = q.part[p];
        a.out[p] = q.out[p];
    }
    a.out_f16 = q.scales_f16 ? 1 : 0;
    a.b_src = q.b_src;
    a.b_pitch = q.b_pitch;
    a.K = q.K;
    a.rows = q.rows;
    a.nkc = int((q.K + KC - 1) / KC);
    a.cps = (a.nkc + q.splits - 1) / q.splits;
    a.splits = (a.nkc + a.cps - 1) / a.cps;
    if (a.splits != q.splits) return cudaErrorInvalidValue;   // every split must own K chunks
    a.ubound[0] = int64_t(a.n_rb[0]) * a.splits;
    a.ubound[1] = a.ubound[0] + int64_t(a.n_rb[1]) * a.splits;
    a.units = a.ubound[1] + int64_t(a.n_rb[2]) * a.splits;
    const uint32_t bytes_a = 2 * kBoxTile;
    const uint32_t bytes_s = uint32_t(kDecRows) * a.nsc * a.ssize;
    a.pitch_b = uint32_t(KC * 2 + 64);
    a.off_s = bytes_a;
    a.off_b = bytes_a + ((bytes_s + 127u) & ~127u);
    const int b_rows = q.rows > 8 ? kDecMaxTokens : 8;
    a.stage_bytes = (a.off_b + uint32_t(b_rows) * a.pitch_b + 1023u) & ~1023u;
    a.err = q.err;
    a.wait_ns = wait_limit_ns();
    const size_t smem_cap = 232448 - 1024;
    a.nstages = uint32_t(std::min<size_t>(kDecStages, (smem_cap - 1024 - kDecRedBytes) / a.stage_bytes));
    if (a.nstages < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + size_t(a.nstages) * a.stage_bytes + kDecRedBytes;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(a.units, device_sm_count())));
    auto kern = q.scales_f16 ? qkv_gemv_kernel<true> : qkv_gemv_kernel<false>;
    // the shared-memory limit is raised once per kernel (not inside a stream capture)
    static std::atomic<size_t> smem_set[2] = {{0}, {0}};
    std::atomic<size_t>& cur = smem_set[q.scales_f16 ? 1 : 0];
    cudaError_t e = cudaSuccess;
    if (cur.load() < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        cur.store(smem);
    }
    note_launch(QMOE_KERNEL_FC1, s, true);
    e = launch_dependent(kern, dim3(grid), dim3(kDecThreads), smem, s, a);
    note_launch(QMOE_KERNEL_FC1, s, false);
    return e != cudaSuccess ? e : cudaGetLastError();
}

bool decode_shape_ok(const Problem& p) {
    if (p.T > kDecMaxTokens) return false;
    if (p.H % 128 != 0 || p.I % 128 != 0) return false;
    const int64_t KC = int64_t(kChunkBytes) * p.pack;
    if (p.bs != 0) {
        if (KC / p.bs < 4) return false;           // at least 16 bytes of scales per box row
        if (p.nb1 % 4 != 0 || p.nb2 % 4 != 0) return false;
    }
    return true;
}

int decode_fc2_splits(const Problem& p) {
    // Split K so that the units (touched expert x 128-row block x K split) spread
    // evenly over the SMs: minimise the chunks of the most loaded SM, counting
    // half a chunk of fixed cost per unit (hand-off of the K halves, epilogue).
    // The touched-expert count is bounded by min(E, T * k) here (routing has not
    // run yet); the kernel iterates over the experts actually touched.
    const int64_t KC = int64_t(kChunkBytes) * p.pack;
    const int64_t nkc = (p.I + KC - 1) / KC;
    const int64_t n_rb = (p.H + kDecRows - 1) / kDecRows;
    const int64_t experts = std::min<int64_t>(p.E, p.T * p.k);
    const int64_t sms = device_sm_count();
    int64_t best = 1;
    double best_cost = 0.0;
    for (int64_t cps = nkc; cps >= 1; --cps) {
        const int64_t splits = (nkc + cps - 1) / cps;
        const int64_t units = experts * n_rb * splits;
        const double cost = double((units + sms - 1) / sms) * (double(cps) + 0.5);
        if (best_cost == 0.0 || cost < best_cost) {
            best_cost = cost;
            best = splits;
        }
    }
    return int(best);
}

cudaError_t launch_decode_fc(const Problem& p, const Plan& pl, const Work& w, bool fc1,
                             cudaStream_t s) {
    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    const int64_t KC = int64_t(kChunkBytes) * p.pack;
    const uint8_t* wt = fc1 ? p.w1 : p.w2;
    const float* sc = fc1 ? p.s1 : p.s2;
    a.N = fc1 ? p.fusion * p.I : p.H;
    a.K = fc1 ? p.H : p.I;
    const int64_t nb = fc1 ? p.nb1 : p.nb2;
    if (!encode_tmap_2d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt, uint64_t(a.K / p.pack),
                        uint64_t(p.E * a.N), uint64_t(a.K / p.pack), kBoxBytes, kDecRows,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const bool scol = p.bs == 0;
    if (!scol) {
        a.nsc = int(KC / p.bs);
        a.lbs = ilog2(p.bs);
        if (!encode_tmap_2d(&a.tm_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, sc, uint64_t(nb),
                            uint64_t(p.E * a.N), uint64_t(nb) * 4, uint32_t(a.nsc), kDecRows,
                            CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        a.scales_col = sc;
    }
    a.b_src = fc1 ? w.x16 : static_cast<const __half*>(w.act);
    a.b_pitch = fc1 ? pl.Hp : pl.Ip;
    a.perm = w.perm;
    a.counts = w.counts;
    a.offsets = w.offsets;
    a.active = w.active;
    a.tiles = w.tiles;
    a.topk = int(p.k);
    a.n_rb = int((a.N + kDecRows - 1) / kDecRows);
    a.nkc = int((a.K + KC - 1) / KC);
    a.splits = fc1 ? 1 : pl.fc2_splits;
    a.cps = (a.nkc + a.splits - 1) / a.splits;
    const uint32_t bytes_a = 2 * kBoxTile;
    const uint32_t bytes_s = scol ? 0u : uint32_t(kDecRows) * a.nsc * 4u;
    // token-row pitch chosen so that one quarter/half warp reads distinct banks
    a.pitch_b = uint32_t(KC * 2 + (p.bits == 4 ? 64 : 32));
    a.off_s = bytes_a;
    a.off_b = bytes_a + ((bytes_s + 127u) & ~127u);
    // token rows per stage: every consumer lane reads row g < 8 (and g + 8 when
    // more than 8 tokens can be routed), so those rows exist even when unused
    const int b_rows = p.T > 8 ? kDecMaxTokens : 8;
    a.stage_bytes = (a.off_b + uint32_t(b_rows) * a.pitch_b + 1023u) & ~1023u;
    a.act_out = static_cast<__half*>(w.act);
    a.act_pitch = pl.Ip;
    a.act = p.act;
    a.act_mode = p.bits == 4 ? 2 : 0;
    a.has_limit = p.has_limit;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.limit = p.limit;
    a.slot_out = w.slot_out;
    a.slots = pl.slots;
    a.err = w.ctrl;
    a.wait_ns = wait_limit_ns();
    a.drop_it = drop_stage();
    const size_t smem_cap = 232448 - 1024;   // 227 KB per CTA, minus static shared memory
    a.nstages = uint32_t(std::min<size_t>(kDecStages, (smem_cap - 1024 - kDecRedBytes) / a.stage_bytes));
    if (a.nstages < 2) return cudaErrorInvalidValue;
    const size_t smem = 1024 + size_t(a.nstages) * a.stage_bytes + kDecRedBytes;
    const int64_t experts = std::min<int64_t>(p.E, pl.slots);
    const int64_t units_max = experts * a.n_rb * a.splits;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(units_max, device_sm_count())));
    const int kid = fc1 ? QMOE_KERNEL_FC1 : QMOE_KERNEL_FC2;
    note_launch(kid, s, true);
    cudaError_t e;
    const int smode = scol ? kScaleCol : (p.bits == 4 && p.bs < 32 ? kScalePre : kScalePost);
    // block scales per 64-byte segment (128 K for 4-bit, 64 K for 8-bit codes), at most 4
    const int64_t segk = p.bits == 4 ? 128 : 64;
    const int nbs = scol ? 0 : (segk / p.bs >= 4 ? 4 : segk / p.bs >= 2 ? 2 : 1);
#define QMOE_DEC_LAUNCH(B, M, NB) \
    (fc1 ? launch_variant<B, M, NB, true>(a, grid, smem, s) : launch_variant<B, M, NB, false>(a, grid, smem, s))
    if (p.bits == 4) {
        if (smode == kScaleCol) e = QMOE_DEC_LAUNCH(4, kScaleCol, 0);
        else if (smode == kScalePre) e = QMOE_DEC_LAUNCH(4, kScalePre, 0);
        else if (nbs == 4) e = QMOE_DEC_LAUNCH(4, kScalePost, 4);
        else if (nbs == 2) e = QMOE_DEC_LAUNCH(4, kScalePost, 2);
        else e = QMOE_DEC_LAUNCH(4, kScalePost, 1);
    } else {
        if (smode == kScaleCol) e = QMOE_DEC_LAUNCH(8, kScaleCol, 0);
        else if (nbs == 4) e = QMOE_DEC_LAUNCH(8, kScalePost, 4);
        else if (nbs == 2) e = QMOE_DEC_LAUNCH(8, kScalePost, 2);
        else e = QMOE_DEC_LAUNCH(8, kScalePost, 1);
    }
#undef QMOE_DEC_LAUNCH
    note_launch(kid, s, false);
    return e;
}

}  // namespace qmoe
