// Few-row GEMV of the RMSNorm + 4-bit Q/K/V projection (com.microsoft.
// MatMulNBitsQkv manifest, pass MatMulNBitsQkv.Projection): the decode GEMV core
// of the QMoE layer (decode_core.cuh) over the three weight tensors in one launch.
#include <algorithm>
#include <atomic>
#include <cstring>

#include "decode_core.cuh"
#include "ptx.cuh"
#include "qkv_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

// ---------------------------------------------------------------------------
// The same GEMV over the three weight tensors of a Q/K/V projection
// (com.microsoft.MatMulNBitsQkv manifest, pass MatMulNBitsQkv.Projection):
// every row of the input is "routed" to each projection.
//
// Work split (stream-K): the (128-row block, K chunk) pairs of the three
// projections, row block by row block, form one flat range that the CTAs cut
// into equal contiguous pieces, so every SM streams the same number of K chunks
// with one pipeline ramp.  A row block inside one CTA's range is stored
// directly; one that two or three CTAs share leaves a partial sum per CTA (slot
// = the CTA's position among them), added in slot order by the reduction.
// ---------------------------------------------------------------------------
struct QkvArgs {
    CUtensorMap tm_w[3];        // packed weights [N_p rows, K/2 bytes], 128-byte swizzle
    CUtensorMap tm_s[3];        // block scales [N_p rows, K/32], fp32 or fp16
    const __half* b_src;        // normalised rows [rows, b_pitch], 4-bit operand order
    int64_t b_pitch;
    int64_t N[3];
    int n_rb[3];
    int64_t total;              // flat (row block, K chunk) pairs of the three projections
    int64_t K;
    int rows, nkc, nsc;
    uint32_t stage_bytes, off_s, off_b, pitch_b, nstages, ssize;
    float* part[3];             // [slots][rows][N_p] partial sums of shared row blocks
    void* out[3];               // [rows][N_p] results, fp32 or fp16 (out_f16)
    int out_f16;
    int32_t* err;
    uint64_t wait_ns;
};

// CTA (of G) whose range holds flat chunk f: the last c with floor(c * total / G) <= f.
__device__ __forceinline__ int cta_of(int64_t f, int64_t total, int64_t G) {
    return int(((f + 1) * G - 1) / total);
}

// The part of flat range [f, fend) inside the row block of chunk f.
struct Piece {
    int p, rb;        // projection, row block within it
    int c0, c1;       // K chunks
    int slot, n;      // this CTA's position among the CTAs sharing the row block; their count
};

__device__ __forceinline__ Piece piece_at(const QkvArgs& a, int64_t f, int64_t fend) {
    const int64_t rbg = f / a.nkc;
    Piece pc;
    pc.p = rbg < a.n_rb[0] ? 0 : (rbg < a.n_rb[0] + a.n_rb[1] ? 1 : 2);
    pc.rb = int(rbg - (pc.p > 0 ? a.n_rb[0] : 0) - (pc.p > 1 ? a.n_rb[1] : 0));
    const int64_t f0 = rbg * a.nkc;
    pc.c0 = int(f - f0);
    pc.c1 = int(min(int64_t(a.nkc), fend - f0));
    const int clo = cta_of(f0, a.total, gridDim.x);
    pc.slot = int(blockIdx.x) - clo;
    pc.n = cta_of(f0 + a.nkc - 1, a.total, gridDim.x) - clo + 1;
    return pc;
}

// Result element idx of projection p (row block not shared).
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
    // this CTA's flat chunk range
    const int64_t fbeg = int64_t(blockIdx.x) * a.total / gridDim.x;
    const int64_t fend = (int64_t(blockIdx.x) + 1) * a.total / gridDim.x;

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
        for (int64_t f = fbeg; f < fend && ok;) {
            const Piece pc = piece_at(a, f, fend);
            f += pc.c1 - pc.c0;
            const int p = pc.p;
            const int c0 = pc.c0, c1 = pc.c1;
            const int32_t row0 = pc.rb * kDecRows;
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
    for (int64_t f = fbeg; f < fend; ++un) {
        const Piece pc = piece_at(a, f, fend);
        f += pc.c1 - pc.c0;
        const int p = pc.p;
        const int c0 = pc.c0, c1 = pc.c1;
        const int64_t rg = int64_t(pc.rb) * kDecRows + r_g;
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
        if (pc.n == 1) {
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
        float* part = a.part[p] + int64_t(pc.slot) * a.rows * Np;
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

}  // namespace

bool qkv_gemv_shape_ok(int64_t K, bool scales_f16) {
    if (K <= 0 || K % 128 != 0) return false;            // whole 64-byte segments per row
    if (scales_f16 && (K / 32) % 8 != 0) return false;    // 16-byte strided fp16 scale rows
    return true;
}

static_assert(kDecRows == kQkvRowBlock, "row block of the GEMV and of its reduction");

// (row block, K chunk) pairs of the three projections and the GEMV's grid.
void qkv_gemv_geometry(const int64_t N[3], int64_t K, int64_t* nkc, int64_t* n_rb,
                       int64_t* total, int64_t* grid) {
    const int64_t KC = int64_t(kChunkBytes) * 2;
    *nkc = (K + KC - 1) / KC;
    *n_rb = 0;
    for (int p = 0; p < 3; ++p) *n_rb += (N[p] + kDecRows - 1) / kDecRows;
    *total = *n_rb * *nkc;
    *grid = std::max<int64_t>(1, std::min<int64_t>(*total, device_sm_count()));
}

namespace {
int host_cta_of(int64_t f, int64_t total, int64_t G) { return int(((f + 1) * G - 1) / total); }
}  // namespace

// Partial-sum slots the GEMV needs: the most CTAs that share one row block
// (1 when every row block lies inside one CTA's range).
int qkv_gemv_splits(const int64_t N[3], int64_t K) {
    int64_t nkc, n_rb, total, G;
    qkv_gemv_geometry(N, K, &nkc, &n_rb, &total, &G);
    int most = 1;
    for (int64_t rb = 0; rb < n_rb; ++rb)
        most = std::max(most, host_cta_of(rb * nkc + nkc - 1, total, G) -
                                  host_cta_of(rb * nkc, total, G) + 1);
    return most;
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
    int64_t nkc, n_rb, total, grid;
    qkv_gemv_geometry(q.N, q.K, &nkc, &n_rb, &total, &grid);
    if (qkv_gemv_splits(q.N, q.K) > q.splits) return cudaErrorInvalidValue;   // slots planned
    a.nkc = int(nkc);
    a.total = total;
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
    e = launch_dependent(kern, dim3(unsigned(grid)), dim3(kDecThreads), smem, s, a);
    note_launch(QMOE_KERNEL_FC1, s, false);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmoe
