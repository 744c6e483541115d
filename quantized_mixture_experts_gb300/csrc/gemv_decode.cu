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
#include <cstring>

#include "ptx.cuh"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr int kDecRowGroups = 8;               // 16-row MMA groups per unit
constexpr int kDecConsumers = 2 * kDecRowGroups; // two K halves per row group
constexpr int kDecThreads = 32 * (1 + kDecConsumers);
constexpr int kDecStages = 4;                  // upper bound; the launch picks what fits
constexpr int kDecRows = 16 * kDecRowGroups;   // 128 weight rows per unit
constexpr int kDecRedBytes = 2 * kDecRowGroups * 32 * 8 * 4;
constexpr int kChunkBytes = 256;               // packed bytes per row per stage
constexpr int kBoxBytes = 128;                 // one 128-byte swizzle span
constexpr int kBoxTile = kBoxBytes * kDecRows; // 16 KB per weight box
constexpr int kDecMaxTokens = 16;
constexpr int kTargetUnitsPerSm = 10;
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

__device__ __forceinline__ void record_error(int32_t* err, int code) {
    atomicCAS(err, 0, code);
}

// Eight 4-bit codes of `w` (low nibble first, element e in bits 4e..4e+3) ->
// four fp16 pairs, each exact:
//   h[0] = (q0, q4) - 8          h[2] = (q2, q6) - 8         (low nibbles of each byte)
//   h[1] = 16 * ((q1, q5) - 8)   h[3] = 16 * ((q3, q7) - 8)  (high nibbles, kept in place)
// A nibble OR-ed into the mantissa of fp16 1024 gives 1024 + q; a high nibble
// left at bits 4..7 gives 1024 + 16 q.  The activations feeding the high
// pairs are stored divided by 16, so each product is unchanged.
__device__ __forceinline__ void dequant4(uint32_t w, uint32_t* h) {
    const __half2 lo_bias = ptx::u32_as_h2(0x64086408u);   // (1032, 1032)
    const __half2 hi_bias = ptx::u32_as_h2(0x64806480u);   // (1152, 1152)
    const uint32_t w8 = w >> 8;
    h[0] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(ptx::and_or(w, 0x000F000Fu, 0x64006400u)), lo_bias));
    h[1] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(ptx::and_or(w, 0x00F000F0u, 0x64006400u)), hi_bias));
    h[2] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(ptx::and_or(w8, 0x000F000Fu, 0x64006400u)), lo_bias));
    h[3] = ptx::h2_as_u32(__hsub2(ptx::u32_as_h2(ptx::and_or(w8, 0x00F000F0u, 0x64006400u)), hi_bias));
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
// order 0,4,1,5,2,6,3,7.
__device__ __forceinline__ int64_t perm8(int64_t j) {
    const int q = int(j & 7);
    return (j & ~int64_t(7)) + (q < 4 ? 2 * q : 2 * (q - 4) + 1);
}

// Stores activation v of column j in the layout the 4-bit FC2 reads (mode 2:
// pair order, odd columns divided by 16) or in natural order (mode 0).
__device__ __forceinline__ void store_act(__half* row, int64_t j, float v, int mode) {
    if (mode == 2) row[perm8(j)] = __float2half_rn((j & 1) ? v * 0.0625f : v);
    else row[j] = __float2half_rn(v);
}

template <int BITS, int SMODE, bool FC1>
__global__ void __launch_bounds__(kDecThreads, 1) decode_gemv_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kDecStages];
    __shared__ __align__(8) uint64_t empty_bar[kDecStages];
    __shared__ __align__(8) uint64_t red_full[2];    // K-half 1 -> K-half 0 partial sums
    __shared__ __align__(8) uint64_t red_empty[2];
    __shared__ int abort_flag;
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

    const int n_active = a.tiles[1];
    const int64_t units = int64_t(n_active) * a.n_rb * a.splits;

    if (warp == 0) {
        // ------------------------------ producer ------------------------------
        if (lane == 0) {
            ptx::prefetch_tmap(&a.tm_w);
            if (!SCOL) ptx::prefetch_tmap(&a.tm_s);
        }
        uint32_t it = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; u < units && ok; u += gridDim.x) {
            const int ks = int(u % a.splits);
            const int rb = int((u / a.splits) % a.n_rb);
            const int ai = int(u / (int64_t(a.splits) * a.n_rb));
            const int e = a.active[ai];
            const int ne = a.counts[e];
            const int off = a.offsets[e];
            const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
            const int32_t row0 = int32_t(int64_t(e) * a.N + int64_t(rb) * kDecRows);
            int64_t brow = 0;
            if (lane < ne) brow = FC1 ? int64_t(a.perm[off + lane] / a.topk) : int64_t(off + lane);
            for (int kc = c0; kc < c1; ++kc, ++it) {
                const int st = int(it % a.nstages);
                const uint32_t ph = (it / a.nstages) & 1u;
                if (!ptx::mbar_wait(&empty_bar[st], ph ^ 1u, a.wait_ns, &abort_flag)) {
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
                if (lane < ne)
                    ptx::bulk_g2s(sbase + a.off_b + lane * a.pitch_b,
                                  a.b_src + brow * a.b_pitch + int64_t(kc) * KC, bbytes,
                                  &full_bar[st]);
            }
        }
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
    uint32_t it = 0;
    uint32_t un = 0;   // units processed by this CTA (reduction buffer parity)
    // B fragments keep stale values for token columns >= ne; those columns of
    // the MMA result are never stored.
    uint4 bq[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++un) {
        const int ks = int(u % a.splits);
        const int rb = int((u / a.splits) % a.n_rb);
        const int ai = int(u / (int64_t(a.splits) * a.n_rb));
        const int e = a.active[ai];
        const int ne = a.counts[e];
        const int off = a.offsets[e];
        const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
        const int64_t rg = int64_t(rb) * kDecRows + r_g;   // row within the expert
        const int64_t rg8 = rg + 8;
        float scol_g = 1.f, scol_g8 = 1.f;
        if (SCOL) {
            const float* sc = a.scales_col + int64_t(e) * a.N;
            scol_g = rg < a.N ? sc[rg] : 0.f;
            scol_g8 = rg8 < a.N ? sc[rg8] : 0.f;
        }
        float acc[2][4], accB[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[nt][q] = accB[nt][q] = 0.f;
        const bool two = ne > 8;
        const bool ld0 = g < ne, ld1 = g + 8 < ne;

        for (int kc = c0; kc < c1; ++kc, ++it) {
            const int st = int(it % a.nstages);
            const uint32_t ph = (it / a.nstages) & 1u;
            if (!ptx::mbar_wait(&full_bar[st], ph, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    record_error(a.err, QMOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                return;
            }
            const uint32_t sA = ptx::launder(sbase0 + uint32_t(st) * a.stage_bytes);
            const uint32_t sS = sA + a.off_s;
            const uint32_t sB = sA + a.off_b;
            const uint32_t rowA = sA + uint32_t(r_g) * kBoxBytes;
            const uint32_t rowA8 = rowA + 8u * kBoxBytes;
            const int64_t krem = a.K - int64_t(kc) * KC;
            const int nseg = int(krem < KC ? krem : KC) / SEGK;
            for (int s = kh; s < nseg; s += 2) {
                const uint32_t half = uint32_t(s >> 1) * kBoxTile;
                float sgv[4], sg8v[4];
                if (SMODE == kScalePost) {
                    // word i of every lane lies in scale block (SEGK*s + SEGK/4*i) >> lbs;
                    // the seg spans 4, 2 or 1 blocks (block sizes SEGK/4, SEGK/2, >= SEGK)
                    const int nbs = SEGK >> a.lbs;   // blocks per segment (0 when bs > SEGK)
                    const int si0 = (SEGK * s) >> a.lbs;
                    const uint32_t a0 = sS + uint32_t(r_g * a.nsc + si0) * 4u;
                    const uint32_t a8 = a0 + uint32_t(8 * a.nsc) * 4u;
                    if (nbs >= 4) {
                        const float4 v0 = ptx::ld_f32x4(a0), v8 = ptx::ld_f32x4(a8);
                        sgv[0] = v0.x; sgv[1] = v0.y; sgv[2] = v0.z; sgv[3] = v0.w;
                        sg8v[0] = v8.x; sg8v[1] = v8.y; sg8v[2] = v8.z; sg8v[3] = v8.w;
                    } else if (nbs == 2) {
                        const float2 v0 = ptx::ld_f32x2(a0), v8 = ptx::ld_f32x2(a8);
                        sgv[0] = sgv[1] = v0.x; sgv[2] = sgv[3] = v0.y;
                        sg8v[0] = sg8v[1] = v8.x; sg8v[2] = sg8v[3] = v8.y;
                    } else {
                        const float v0 = ptx::ld_f32(a0), v8 = ptx::ld_f32(a8);
                        sgv[0] = sgv[1] = sgv[2] = sgv[3] = v0;
                        sg8v[0] = sg8v[1] = sg8v[2] = sg8v[3] = v8;
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // word i of lane c: packed bytes 16i + 4c of this 64-byte segment
                    const int jchunk = ((s & 1) << 2) + i;
                    const uint32_t offw = half + uint32_t((jchunk ^ g) << 4) + uint32_t(c) * 4u;
                    const uint32_t wa = ptx::ld_u32(rowA + offw);
                    const uint32_t wb = ptx::ld_u32(rowA8 + offw);
                    const int kin = BITS == 4 ? (SEGK * s + 32 * i + 8 * c) : (SEGK * s + 16 * i + 4 * c);
                    const uint32_t boff = uint32_t(kin) * 2u;
                    if (BITS == 4) {
                        uint32_t hg[4], hg8[4];
                        if (SMODE == kScalePre) {
                            const int si = kin >> a.lbs;
                            const __half2 s0 = __float2half2_rn(ptx::ld_f32(sS + uint32_t(r_g * a.nsc + si) * 4u));
                            const __half2 s8 = __float2half2_rn(ptx::ld_f32(sS + uint32_t((r_g + 8) * a.nsc + si) * 4u));
                            dequant4_scaled(wa, s0, hg);
                            dequant4_scaled(wb, s8, hg8);
                        } else {
                            dequant4(wa, hg);
                            dequant4(wb, hg8);
                        }
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            if (nt == 1 && !two) break;
                            ptx::ld128_pred(bq[nt], sB + uint32_t(g + 8 * nt) * a.pitch_b + boff,
                                            nt == 0 ? ld0 : ld1);
                            // low pairs (K 0,4 | 2,6) with b.x|b.z; high pairs (K 1,5 | 3,7),
                            // 16x larger, with b.y|b.w stored divided by 16
                            if (SMODE == kScalePost) {
                                float tmp[4];
                                ptx::mma_16816_z(tmp, hg[0], hg8[0], hg[2], hg8[2], bq[nt].x, bq[nt].z);
                                ptx::mma_16816(tmp, hg[1], hg8[1], hg[3], hg8[3], bq[nt].y, bq[nt].w);
                                acc[nt][0] = fmaf(sgv[i], tmp[0], acc[nt][0]);
                                acc[nt][1] = fmaf(sgv[i], tmp[1], acc[nt][1]);
                                acc[nt][2] = fmaf(sg8v[i], tmp[2], acc[nt][2]);
                                acc[nt][3] = fmaf(sg8v[i], tmp[3], acc[nt][3]);
                            } else {
                                ptx::mma_16816(acc[nt], hg[0], hg8[0], hg[2], hg8[2], bq[nt].x, bq[nt].z);
                                ptx::mma_16816(accB[nt], hg[1], hg8[1], hg[3], hg8[3], bq[nt].y, bq[nt].w);
                            }
                        }
                    } else {
                        uint32_t hg[2], hg8[2];
                        dequant8(wa, hg);
                        dequant8(wb, hg8);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            if (nt == 1 && !two) break;
                            ptx::ld64_pred(bq[nt].x, bq[nt].y,
                                           sB + uint32_t(g + 8 * nt) * a.pitch_b + boff,
                                           nt == 0 ? ld0 : ld1);
                            if (SMODE == kScalePost) {
                                float tmp[4];
                                ptx::mma_16816_z(tmp, hg[0], hg8[0], hg[1], hg8[1], bq[nt].x, bq[nt].y);
                                acc[nt][0] = fmaf(sgv[i], tmp[0], acc[nt][0]);
                                acc[nt][1] = fmaf(sgv[i], tmp[1], acc[nt][1]);
                                acc[nt][2] = fmaf(sg8v[i], tmp[2], acc[nt][2]);
                                acc[nt][3] = fmaf(sg8v[i], tmp[3], acc[nt][3]);
                            } else if (i & 1) {
                                ptx::mma_16816(accB[nt], hg[0], hg8[0], hg[1], hg8[1], bq[nt].x, bq[nt].y);
                            } else {
                                ptx::mma_16816(acc[nt], hg[0], hg8[0], hg[1], hg8[1], bq[nt].x, bq[nt].y);
                            }
                        }
                    }
                }
            }
            // every shared load of this stage feeds the accumulators: finish them first
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ptx::depend(acc[nt][q]);
                    ptx::depend(accB[nt][q]);
                }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty_bar[st]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[nt][q] += accB[nt][q];
            if (SCOL) {
                acc[nt][0] *= scol_g; acc[nt][1] *= scol_g;
                acc[nt][2] *= scol_g8; acc[nt][3] *= scol_g8;
            }
        }

        // ---- K-half 1 hands its partial sums to K-half 0 through shared memory ----
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
                    const int64_t slot_id = a.perm[off + n];
                    float* dst = a.slot_out + (int64_t(ks) * a.slots + slot_id) * a.N;
                    if (rg < a.N) dst[rg] = acc[nt][q];
                    if (rg8 < a.N) dst[rg8] = acc[nt][2 + q];
                }
            }
        }
    }
}

template <int BITS, int SMODE, bool FC1>
cudaError_t launch_variant(const DecodeArgs& args, int grid, size_t smem, cudaStream_t s) {
    auto kern = decode_gemv_kernel<BITS, SMODE, FC1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid, kDecThreads, smem, s>>>(args);
    return cudaGetLastError();
}

int ilog2(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return l;
}

}  // namespace

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
    const int64_t KC = int64_t(kChunkBytes) * p.pack;
    const int64_t nkc = (p.I + KC - 1) / KC;
    const int64_t n_rb = (p.H + kDecRows - 1) / kDecRows;
    const int64_t experts = std::min<int64_t>(p.E, p.T * p.k);
    const int64_t want = int64_t(kTargetUnitsPerSm) * 152;
    int64_t splits = (want + experts * n_rb - 1) / (experts * n_rb);
    splits = std::max<int64_t>(1, std::min<int64_t>(splits, nkc));
    const int64_t cps = (nkc + splits - 1) / splits;
    return int((nkc + cps - 1) / cps);
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
    const int max_tok = int(std::min<int64_t>(p.T, kDecMaxTokens));
    a.stage_bytes = (a.off_b + uint32_t(max_tok) * a.pitch_b + 1023u) & ~1023u;
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
#define QMOE_DEC_LAUNCH(B, M) \
    (fc1 ? launch_variant<B, M, true>(a, grid, smem, s) : launch_variant<B, M, false>(a, grid, smem, s))
    if (p.bits == 4) {
        e = smode == kScaleCol ? QMOE_DEC_LAUNCH(4, kScaleCol)
            : smode == kScalePost ? QMOE_DEC_LAUNCH(4, kScalePost) : QMOE_DEC_LAUNCH(4, kScalePre);
    } else {
        e = smode == kScaleCol ? QMOE_DEC_LAUNCH(8, kScaleCol) : QMOE_DEC_LAUNCH(8, kScalePost);
    }
#undef QMOE_DEC_LAUNCH
    note_launch(kid, s, false);
    return e;
}

}  // namespace qmoe
