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
// directly.  A row block that several CTAs share is finished by the CTA that
// holds its first chunks (slot 0): for that CTA it is the last piece of its
// range, while for every other sharer (slots 1, 2, ...) it is the first.  The
// others store their partial sums and then a flag holding the launch's grid
// identifier (%gridid, distinct for every launch in the context, so a flag
// left by an earlier launch, or never set, does not count); slot 0 waits for
// the flags (bounded), adds the partial sums to its own in slot order and
// stores the result.  A CTA waits only for CTAs of higher index that finish
// their part before any wait of their own.
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
    unsigned long long* flags;  // [row blocks of the three][slots]: the grid identifier
    int slots;
    uint32_t pre_stages;        // stages whose weights go out before griddepcontrol.wait
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
    int p, rb, rbg;   // projection, row block within it, row block of the three
    int c0, c1;       // K chunks
    int slot, n;      // this CTA's position among the CTAs sharing the row block; their count
};

__device__ __forceinline__ Piece piece_at(const QkvArgs& a, int64_t f, int64_t fend) {
    const int64_t rbg = f / a.nkc;
    Piece pc;
    pc.rbg = int(rbg);
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

// Lane 0 of a slot-0 CTA: wait until sharers 1 .. n - 1 have set their flags to
// this launch's grid identifier (bounded; false on expiry or abort).
__device__ __forceinline__ bool flags_seen(const unsigned long long* flag, int n, unsigned long long gid,
                                           uint64_t limit_ns, volatile int* abort) {
    const uint64_t t0 = ptx::globaltimer();
    for (int s = 1; s < n; ++s) {
        for (;;) {
            unsigned long long v;
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(flag + s) : "memory");
            if (v == gid) break;
            if (*abort || ptx::globaltimer() - t0 > limit_ns) return false;
            __nanosleep(64);
        }
    }
    return true;
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
    __shared__ __align__(8) uint64_t part_bar;      // the 8 summing warps stored a shared piece
    __shared__ __align__(8) uint64_t last_bar;      // the other sharers' flags were seen
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
        ptx::mbar_init(&part_bar, kDecRowGroups);
        ptx::mbar_init(&last_bar, 1);
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
                // a few stages' weights before the wait: more would hold up the previous
                // kernel's completion behind this grid's copies
                if (!dep_done && it >= a.pre_stages) release_held();
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
        // a shared row block (see the work split above)
        const int64_t pstride = int64_t(a.rows) * Np;
        const float* part = a.part[p];
        unsigned long long* flag = a.flags + int64_t(pc.rbg) * a.slots;
        unsigned long long gid;
        asm volatile("mov.u64 %0, %%gridid;" : "=l"(gid));
        if (pc.slot > 0) {
            float* mine = a.part[p] + int64_t(pc.slot) * pstride;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int n = nt * 8 + 2 * c + q;
                    if (n >= ne) continue;
                    if (rg < Np) mine[int64_t(n) * Np + rg] = acc[nt][q];
                    if (rg8 < Np) mine[int64_t(n) * Np + rg8] = acc[nt][2 + q];
                }
            __threadfence();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&part_bar);
            if (cw == 0) {
                if (!ptx::mbar_wait(&part_bar, 0, a.wait_ns, &abort_flag)) {
                    if (lane == 0) { record_error(a.err, QMOE_DEVERR_TIMEOUT); abort_flag = 1; }
                    return;
                }
                if (lane == 0)
                    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(flag + pc.slot), "l"(gid)
                                 : "memory");
                __syncwarp();
            }
            continue;
        }
        if (cw == 0) {
            if (lane == 0) {
                if (!flags_seen(flag, pc.n, gid, a.wait_ns, &abort_flag)) {
                    record_error(a.err, QMOE_DEVERR_TIMEOUT);
                    abort_flag = 1;
                }
                ptx::mbar_arrive(&last_bar);
            }
            __syncwarp();
        }
        if (!ptx::mbar_wait(&last_bar, 0, a.wait_ns, &abort_flag) || abort_flag) {
            if (lane == 0) { record_error(a.err, QMOE_DEVERR_TIMEOUT); abort_flag = 1; }
            return;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int n = nt * 8 + 2 * c + q;
                if (n >= ne) continue;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t row = h ? rg8 : rg;
                    if (row >= Np) continue;
                    const int64_t idx = int64_t(n) * Np + row;
                    float sum = acc[nt][2 * h + q];   // slot 0: this CTA
                    for (int s0 = 1; s0 < pc.n; s0 += 4) {
                        float v[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            v[u] = s0 + u < pc.n ? __ldcg(part + (s0 + u) * pstride + idx) : 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (s0 + u < pc.n) sum += v[u];
                    }
                    qkv_store(a, p, idx, sum);
                }
            }
    }
}

}  // namespace

bool qkv_gemv_shape_ok(int64_t K, bool scales_f16) {
    if (K <= 0 || K % 128 != 0) return false;            // whole 64-byte segments per row
    if (scales_f16 && (K / 32) % 8 != 0) return false;    // 16-byte strided fp16 scale rows
    return true;
}

static_assert(kDecRows == kQkvRowBlock, "row block of the GEMV and of its partial sums");

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
// (1 when every row block lies inside one CTA's range).  Slot 0 keeps its sums in
// registers; the space for it stays unused.
int qkv_gemv_splits(const int64_t N[3], int64_t K) {
    int64_t nkc, n_rb, total, G;
    qkv_gemv_geometry(N, K, &nkc, &n_rb, &total, &G);
    int most = 1;
    for (int64_t rb = 0; rb < n_rb; ++rb)
        most = std::max(most, host_cta_of(rb * nkc + nkc - 1, total, G) -
                                  host_cta_of(rb * nkc, total, G) + 1);
    return most;
}

int64_t qkv_gemv_row_blocks(const int64_t N[3], int64_t K) {
    int64_t nkc, n_rb, total, G;
    qkv_gemv_geometry(N, K, &nkc, &n_rb, &total, &G);
    return n_rb;
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
    a.flags = q.flags;
    a.slots = q.splits;
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
    a.pre_stages = std::min<uint32_t>(a.nstages, kQkvPreStages);
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
