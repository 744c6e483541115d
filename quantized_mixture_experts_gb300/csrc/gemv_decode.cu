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

constexpr int kDecConsumers = 8;
constexpr int kDecThreads = 32 * (1 + kDecConsumers);
constexpr int kDecStages = 3;
constexpr int kDecRows = 16 * kDecConsumers;   // 128 weight rows per unit
constexpr int kChunkBytes = 256;               // packed bytes per row per stage
constexpr int kBoxBytes = 128;                 // one 128-byte swizzle span
constexpr int kBoxTile = kBoxBytes * kDecRows; // 16 KB per weight box
constexpr int kDecMaxTokens = 16;
constexpr int kTargetUnitsPerSm = 10;
constexpr unsigned kFull = 0xffffffffu;

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
    uint32_t stage_bytes, off_s, off_b, pitch_b;
    __half* act_out;
    int64_t act_pitch;
    int act, interleave8, has_limit;
    float alpha, beta, limit;
    float* slot_out;
    int64_t slots;
    int32_t* err;
    uint64_t wait_ns;
};

__device__ __forceinline__ void record_error(int32_t* err, int code) {
    atomicCAS(err, 0, code);
}

// Eight 4-bit codes of `w` (low nibble first) -> four fp16 pairs
// ((q0,q4),(q1,q5),(q2,q6),(q3,q7)) of (q - 8) * scale.  1024 + q is built
// exactly by OR-ing the nibble into the fp16 mantissa of 1024.
__device__ __forceinline__ void dequant4(uint32_t w, __half2 s, uint32_t* h) {
    const __half2 bias = ptx::u32_as_h2(0x64086408u);   // (1032, 1032)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t v = ptx::and_or(w >> (4 * q), 0x000F000Fu, 0x64006400u);
        h[q] = ptx::h2_as_u32(__hmul2(__hsub2(ptx::u32_as_h2(v), bias), s));
    }
}

// Four 8-bit codes -> two fp16 pairs ((q0,q1),(q2,q3)) of (q - 128) * scale.
__device__ __forceinline__ void dequant8(uint32_t w, __half2 s, uint32_t* h) {
    const __half2 bias = ptx::u32_as_h2(0x64806480u);   // (1152, 1152)
    const uint32_t lo = ptx::prmt(w, 0x64646464u, 0x4140u);
    const uint32_t hi = ptx::prmt(w, 0x64646464u, 0x4342u);
    h[0] = ptx::h2_as_u32(__hmul2(__hsub2(ptx::u32_as_h2(lo), bias), s));
    h[1] = ptx::h2_as_u32(__hmul2(__hsub2(ptx::u32_as_h2(hi), bias), s));
}

__device__ __forceinline__ float swiglu(float g, float u, float alpha, float beta, int has_limit,
                                        float limit) {
    if (has_limit) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    return g * (1.f / (1.f + expf(-alpha * g))) * (u + beta);
}

// Position of activation column j in a row stored with 8-groups in the
// order 0,4,1,5,2,6,3,7.
__device__ __forceinline__ int64_t perm8(int64_t j) {
    const int q = int(j & 7);
    return (j & ~int64_t(7)) + (q < 4 ? 2 * q : 2 * (q - 4) + 1);
}

template <int BITS, bool SCOL, bool FC1>
__global__ void __launch_bounds__(kDecThreads, 1) decode_gemv_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kDecStages];
    __shared__ __align__(8) uint64_t empty_bar[kDecStages];
    __shared__ int abort_flag;
    constexpr int KC = kChunkBytes * (BITS == 4 ? 2 : 1);   // K values per chunk
    constexpr int SEGK = BITS == 4 ? 128 : 64;              // K values per 64-byte segment

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            ptx::mbar_init(&full_bar[s], 1);
            ptx::mbar_init(&empty_bar[s], kDecConsumers);
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
                const int st = int(it % kDecStages);
                const uint32_t ph = (it / kDecStages) & 1u;
                if (!ptx::mbar_wait(&empty_bar[st], ph ^ 1u, a.wait_ns, &abort_flag)) {
                    ok = false;
                    break;
                }
                const int kvalid = int(a.K - int64_t(kc) * KC < KC ? a.K - int64_t(kc) * KC : KC);
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
        if (!ok) {
            if (lane == 0) {
                record_error(a.err, QMOE_DEVERR_TIMEOUT);
                abort_flag = 1;
                // drain copies still in flight (bounded) before the CTA exits
                for (uint32_t j = it > kDecStages ? it - kDecStages : 0; j < it; ++j) {
                    volatile int never = 0;
                    ptx::mbar_wait(&full_bar[j % kDecStages], (j / kDecStages) & 1u, a.wait_ns,
                                   &never);
                }
            }
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    const int cw = warp - 1;
    const int g = lane >> 2, c = lane & 3;
    const int r_g = 16 * cw + g;   // row of this thread inside the 128-row box (and r_g + 8)
    uint32_t it = 0;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int ks = int(u % a.splits);
        const int rb = int((u / a.splits) % a.n_rb);
        const int ai = int(u / (int64_t(a.splits) * a.n_rb));
        const int e = a.active[ai];
        const int ne = a.counts[e];
        const int off = a.offsets[e];
        const int c0 = ks * a.cps, c1 = min(a.nkc, c0 + a.cps);
        const int64_t rg = int64_t(rb) * kDecRows + r_g;   // row within the expert
        const int64_t rg8 = rg + 8;
        __half2 scol_g = __float2half2_rn(0.f), scol_g8 = scol_g;
        if (SCOL) {
            const float* sc = a.scales_col + int64_t(e) * a.N;
            scol_g = __float2half2_rn(rg < a.N ? sc[rg] : 0.f);
            scol_g8 = __float2half2_rn(rg8 < a.N ? sc[rg8] : 0.f);
        }
        float acc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
        const bool two = ne > 8;

        for (int kc = c0; kc < c1; ++kc, ++it) {
            const int st = int(it % kDecStages);
            const uint32_t ph = (it / kDecStages) & 1u;
            if (!ptx::mbar_wait(&full_bar[st], ph, a.wait_ns, &abort_flag)) {
                if (lane == 0) {
                    record_error(a.err, QMOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                return;
            }
            const uint8_t* sA = smem + size_t(st) * a.stage_bytes;
            const float* sS = reinterpret_cast<const float*>(sA + a.off_s);
            const uint8_t* sB = sA + a.off_b;
            const int kvalid = int(a.K - int64_t(kc) * KC < KC ? a.K - int64_t(kc) * KC : KC);
            const int nseg = kvalid / SEGK;
            for (int s = 0; s < nseg; ++s) {
                const int jchunk = ((s & 1) << 2) + c;
                const uint32_t offA = uint32_t(s >> 1) * kBoxTile + uint32_t((jchunk ^ g) << 4);
                const uint4 wg = *reinterpret_cast<const uint4*>(sA + offA + r_g * kBoxBytes);
                const uint4 wg8 = *reinterpret_cast<const uint4*>(sA + offA + (r_g + 8) * kBoxBytes);
                const uint32_t wv[4] = {wg.x, wg.y, wg.z, wg.w};
                const uint32_t wv8[4] = {wg8.x, wg8.y, wg8.z, wg8.w};
                __half2 sc_g = scol_g, sc_g8 = scol_g8;
                int si_prev = -1;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kin = BITS == 4 ? (SEGK * s + 32 * c + 8 * i) : (SEGK * s + 16 * c + 4 * i);
                    if (!SCOL) {
                        // the block index changes with i in the same way for every lane
                        const int si = kin >> a.lbs;
                        if (si != si_prev) {
                            sc_g = __float2half2_rn(sS[r_g * a.nsc + si]);
                            sc_g8 = __float2half2_rn(sS[(r_g + 8) * a.nsc + si]);
                            si_prev = si;
                        }
                    }
                    if (BITS == 4) {
                        uint32_t hg[4], hg8[4];
                        dequant4(wv[i], sc_g, hg);
                        dequant4(wv8[i], sc_g8, hg8);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            if (nt == 1 && !two) break;
                            const int tok = nt * 8 + g;
                            uint4 bv = make_uint4(0u, 0u, 0u, 0u);
                            if (tok < ne)
                                bv = *reinterpret_cast<const uint4*>(sB + tok * a.pitch_b + kin * 2);
                            ptx::mma_16816(acc[nt], hg[0], hg8[0], hg[1], hg8[1], bv.x, bv.y);
                            ptx::mma_16816(acc[nt], hg[2], hg8[2], hg[3], hg8[3], bv.z, bv.w);
                        }
                    } else {
                        uint32_t hg[2], hg8[2];
                        dequant8(wv[i], sc_g, hg);
                        dequant8(wv8[i], sc_g8, hg8);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            if (nt == 1 && !two) break;
                            const int tok = nt * 8 + g;
                            uint2 bv = make_uint2(0u, 0u);
                            if (tok < ne)
                                bv = *reinterpret_cast<const uint2*>(sB + tok * a.pitch_b + kin * 2);
                            ptx::mma_16816(acc[nt], hg[0], hg8[0], hg[1], hg8[1], bv.x, bv.y);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty_bar[st]);
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
                                const int64_t j = rg >> 1;
                                dst[a.interleave8 ? perm8(j) : j] = __float2half_rn(v);
                            }
                            if (rg8 < a.N) {
                                const float v = swiglu(acc[nt][2 + q], pv[2 + q], a.alpha, a.beta,
                                                       a.has_limit, a.limit);
                                if (!(fabsf(v) <= 65504.f)) record_error(a.err, QMOE_DEVERR_NONFINITE);
                                const int64_t j = rg8 >> 1;
                                dst[a.interleave8 ? perm8(j) : j] = __float2half_rn(v);
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
                            dst[a.interleave8 ? perm8(rg) : rg] = __float2half_rn(v);
                        }
                        if (rg8 < a.N) {
                            const float v = fmaxf(acc[nt][2 + q], 0.f);
                            if (!(v <= 65504.f)) record_error(a.err, QMOE_DEVERR_NONFINITE);
                            dst[a.interleave8 ? perm8(rg8) : rg8] = __float2half_rn(v);
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
                    const int64_t slot = a.perm[off + n];
                    float* dst = a.slot_out + (int64_t(ks) * a.slots + slot) * a.N;
                    if (rg < a.N) dst[rg] = acc[nt][q];
                    if (rg8 < a.N) dst[rg8] = acc[nt][2 + q];
                }
            }
        }
    }
}

template <int BITS, bool SCOL, bool FC1>
cudaError_t launch_variant(const DecodeArgs& args, int grid, size_t smem, cudaStream_t s) {
    auto kern = decode_gemv_kernel<BITS, SCOL, FC1>;
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
    a.pitch_b = uint32_t(KC * 2 + 16);
    a.off_s = bytes_a;
    a.off_b = bytes_a + ((bytes_s + 127u) & ~127u);
    a.stage_bytes = (a.off_b + kDecMaxTokens * a.pitch_b + 1023u) & ~1023u;
    a.act_out = static_cast<__half*>(w.act);
    a.act_pitch = pl.Ip;
    a.act = p.act;
    a.interleave8 = p.bits == 4 ? 1 : 0;
    a.has_limit = p.has_limit;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.limit = p.limit;
    a.slot_out = w.slot_out;
    a.slots = pl.slots;
    a.err = w.ctrl;
    a.wait_ns = wait_limit_ns();
    const size_t smem = 1024 + size_t(kDecStages) * a.stage_bytes;
    const int64_t experts = std::min<int64_t>(p.E, pl.slots);
    const int64_t units_max = experts * a.n_rb * a.splits;
    const int grid = int(std::max<int64_t>(1, std::min<int64_t>(units_max, device_sm_count())));
    const int kid = fc1 ? QMOE_KERNEL_FC1 : QMOE_KERNEL_FC2;
    note_launch(kid, s, true);
    cudaError_t e;
    if (p.bits == 4) {
        if (scol) e = fc1 ? launch_variant<4, true, true>(a, grid, smem, s) : launch_variant<4, true, false>(a, grid, smem, s);
        else e = fc1 ? launch_variant<4, false, true>(a, grid, smem, s) : launch_variant<4, false, false>(a, grid, smem, s);
    } else {
        if (scol) e = fc1 ? launch_variant<8, true, true>(a, grid, smem, s) : launch_variant<8, true, false>(a, grid, smem, s);
        else e = fc1 ? launch_variant<8, false, true>(a, grid, smem, s) : launch_variant<8, false, false>(a, grid, smem, s);
    }
    note_launch(kid, s, false);
    return e;
}

}  // namespace qmoe
