// Weight-streaming decode GEMV core shared by the QMoE layer's decode path
// (gemv_decode.cu) and the Q/K/V projection (qkv_gemv.cu): tile constants,
// the stage ring, the 4/8-bit magic-number dequantisation, and one consumer
// warp's MMAs over a stage and over a work unit's K chunks (mma.sync m16n8k16,
// weights on M, the few routed rows on N).
#pragma once

#include "ptx.cuh"
#include "qmoe_internal.h"

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

// The conversion is the exponent-bias method of turning small integers into
// floating point: with the exponent of a power-of-two constant fixed, the
// integer written into the low mantissa bits gives constant + integer exactly,
// and subtracting the constant leaves the integer.  Its use for int4/int8
// weight dequantisation is described by Kim et al., "Who Says Elephants Can't
// Run: Bringing Large Scale MoE Models into Cloud Scale Production" (2022).
//
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
template <int BITS, int SMODE, int NBS, int NT, bool SH = false, typename Args = void>
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

}  // namespace
}  // namespace qmoe
