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
// ring of up to 4 stages in shared memory (as many as fit) with
//   - the unit's 128 weight rows x 256 packed bytes (two 128-byte-swizzled
//     2-D tensor boxes),
//   - the matching block scales (one 2-D box),
//   - the routed tokens' fp16 activation rows for this K chunk (1-D bulk
//     copies gathered by the expert permutation);
// 16 consumer warps, 8 row groups of 16 weight rows x 2 halves of each
// stage's K, dequantize w = (q - mid) * scale into fp16 registers (the
// integer-to-half conversion by placing the code in the mantissa of a
// power-of-two constant and subtracting it, done with LOP3/PRMT; exact for the
// integer part) and run mma.sync m16n8k16 with the tokens as the N side,
// accumulating in fp32; the two K halves of a row group add their partial
// sums through shared memory.  FC1 applies ReLU / interleaved SwiGLU in the
// epilogue and writes fp16 activations; FC2 writes fp32 per-slot partial
// sums per K split, reduced in fixed order by the combine kernel.
#include <algorithm>
#include <cstring>

#include "decode_core.cuh"
#include "ptx.cuh"
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

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
