// RMSNorm + 4-bit Q/K/V projection (com.microsoft.MatMulNBitsQkv manifest):
// the normalisation kernels, the scalar path and the
// host side of the C ABI (validation per attributeConstraints and
// derive.weightShapeOk / scaleShapeOk / ioShapeOk / normContractOk, workspace
// planning, dispatch).  The few-row projection runs in the weight-streaming
// GEMV of qkv_gemv.cu (over the QMoE decode path's consumer core).
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "ptx.cuh"
#include "qkv_internal.h"

namespace qmoe {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kNormThreads = 256;

__device__ __forceinline__ float ld(const float* p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld(const __half* p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ void st(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__half* p, int64_t i, float v) { p[i] = __float2half_rn(v); }

// Eight consecutive elements (16-byte aligned) to / from fp32 registers.
__device__ __forceinline__ void load8(const float* p, float* v) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __half* p, float* v) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(ptx::u32_as_h2(w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void store8(float* p, const float* v) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__half* p, const float* v) {
    uint4 u;
    u.x = ptx::h2_as_u32(__floats2half2_rn(v[0], v[1]));
    u.y = ptx::h2_as_u32(__floats2half2_rn(v[2], v[3]));
    u.z = ptx::h2_as_u32(__floats2half2_rn(v[4], v[5]));
    u.w = ptx::h2_as_u32(__floats2half2_rn(v[6], v[7]));
    *reinterpret_cast<uint4*>(p) = u;
}

// Position of element j in a row whose groups of eight are stored in the order
// 0,4,2,6,1,5,3,7: the operand layout of the 4-bit decode GEMV, which pairs
// (0,4),(2,6) with low nibbles and (1,5),(3,7) with high nibbles in place.
__device__ __forceinline__ int64_t operand_pos(int64_t j) {
    const int q = int(j & 3);
    const int slot = (q & 1) ? 2 + (q >> 1) : (q >> 1);
    return (j & ~int64_t(7)) + 2 * slot + ((j >> 2) & 1);
}

// MatMulNBitsQkv.RmsNorm, one CTA per row: x = A (+ skip), residual = x,
// normed = x / sqrt(mean(x^2) + eps) * norm_scale, in fp32.  The normalised row
// goes out as fp32 (n32) and/or as fp16 in the GEMV operand layout (n16, odd
// elements divided by 16: the GEMV keeps high nibbles in place, at 16 x).
template <typename T>
__global__ void __launch_bounds__(kNormThreads) qkv_norm_kernel(
    const T* __restrict__ A, const T* __restrict__ skip, const T* __restrict__ gamma, int64_t K,
    float eps, T* __restrict__ residual, __half* __restrict__ n16, int64_t pitch16,
    float* __restrict__ n32, int32_t* __restrict__ err) {
    // the projection may start streaming weights while this kernel runs
    ptx::griddep_launch_dependents();
    __shared__ float s_part[kNormThreads / 32];
    const int64_t r = blockIdx.x;
    if (r == 0 && threadIdx.x == 0 && err) err[0] = 0;
    const T* a = A + r * K;
    const T* sk = skip ? skip + r * K : nullptr;
    float ss = 0.f;
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
        const float x = ld(a, k) + (sk ? ld(sk, k) : 0.f);
        ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];   // fixed order
    const float inv = rsqrtf(tot / float(K) + eps);
    for (int64_t k = threadIdx.x; k < K; k += blockDim.x) {
        const float x = ld(a, k) + (sk ? ld(sk, k) : 0.f);
        if (residual) st(residual, r * K + k, x);
        const float v = x * inv * ld(gamma, k);
        if (n16) n16[r * pitch16 + operand_pos(k)] = __float2half_rn((k & 1) ? v * 0.0625f : v);
        if (n32) n32[r * K + k] = v;
    }
}

// The same normalisation for rows that fit in registers: 512 threads, each owning
// up to G groups of eight consecutive elements (16-byte loads for fp16, two for
// fp32), one pass over global memory.  K % 8 == 0, K <= 512 * 8 * G, 16-byte
// aligned rows.
template <typename T, int G>
__global__ void __launch_bounds__(512) qkv_norm_regs_kernel(
    const T* __restrict__ A, const T* __restrict__ skip, const T* __restrict__ gamma, int64_t K,
    float eps, T* __restrict__ residual, __half* __restrict__ n16, int64_t pitch16,
    float* __restrict__ n32, int32_t* __restrict__ err) {
    ptx::griddep_launch_dependents();
    __shared__ float s_part[16];
    const int64_t r = blockIdx.x;
    if (r == 0 && threadIdx.x == 0 && err) err[0] = 0;
    const int64_t ngroups = K / 8;
    float x[G][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < G; ++i) {
        const int64_t grp = threadIdx.x + int64_t(i) * blockDim.x;
#pragma unroll
        for (int e = 0; e < 8; ++e) x[i][e] = 0.f;
        if (grp < ngroups) {
            load8(A + r * K + grp * 8, x[i]);
            if (skip) {
                float y[8];
                load8(skip + r * K + grp * 8, y);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[i][e] += y[e];
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[i][e], x[i][e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) tot += s_part[w];   // fixed order
    const float inv = rsqrtf(tot / float(K) + eps);
#pragma unroll
    for (int i = 0; i < G; ++i) {
        const int64_t grp = threadIdx.x + int64_t(i) * blockDim.x;
        if (grp >= ngroups) continue;
        if (residual) store8(residual + r * K + grp * 8, x[i]);
        float g[8], v[8];
        load8(gamma + grp * 8, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = x[i][e] * inv * g[e];
        if (n16) {
            // operand order 0,4,2,6,1,5,3,7 with the odd elements divided by 16
            const __half2 h0 = __floats2half2_rn(v[0], v[4]);
            const __half2 h1 = __floats2half2_rn(v[2], v[6]);
            const __half2 h2 = __floats2half2_rn(v[1] * 0.0625f, v[5] * 0.0625f);
            const __half2 h3 = __floats2half2_rn(v[3] * 0.0625f, v[7] * 0.0625f);
            uint4 u;
            u.x = ptx::h2_as_u32(h0);
            u.y = ptx::h2_as_u32(h1);
            u.z = ptx::h2_as_u32(h2);
            u.w = ptx::h2_as_u32(h3);
            *reinterpret_cast<uint4*>(n16 + r * pitch16 + grp * 8) = u;
        }
        if (n32) store8(n32 + r * K + grp * 8, v);
    }
}

struct Proj3 {
    const uint8_t* B[3];
    const void* S[3];
    int64_t N[3];
    void* out[3];
};

// Scalar path: one warp per (projection, output n, row); the codes are
// dequantised on the fly (zero point 8, block-32 scales).
template <typename T>
__global__ void qkv_generic_kernel(Proj3 pj, const float* __restrict__ normed, int64_t rows,
                                   int64_t K) {
    int64_t widx = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    int p = 0;
    while (p < 3 && widx >= rows * pj.N[p]) widx -= rows * pj.N[p++];
    if (p >= 3) return;
    const int64_t n = widx / rows, r = widx % rows;   // output-major: weight rows stay in cache
    const int64_t kb = (K + 31) / 32;
    const uint8_t* brow = pj.B[p] + n * kb * 16;
    const T* srow = static_cast<const T*>(pj.S[p]) + n * kb;
    const float* x = normed + r * K;
    float acc = 0.f;
    for (int64_t k = lane; k < K; k += 32) {
        const uint8_t byte = brow[(k >> 5) * 16 + ((k & 31) >> 1)];
        const int q = (k & 1) ? (byte >> 4) : (byte & 15);
        acc = fmaf(x[k], float(q - 8) * ld(srow, k >> 5), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (lane == 0) st(static_cast<T*>(pj.out[p]), r * pj.N[p] + n, acc);
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct QkvProblem {
    int64_t rows = 0, K = 0, N[3] = {0, 0, 0}, kblocks = 0;
    bool f16 = false;
    float eps = 0.f;
    int path = QKV_PATH_GENERIC;
};

struct QkvPlan {
    int splits = 1;
    int64_t pitch16 = 0;
    size_t off_n16 = 0, off_n32 = 0, off_part = 0, off_flags = 0, bytes = 0;
};

qmoe_status qderive(const int64_t* a_shape, int32_t a_rank, const qkv_attrs* at, int32_t dtype,
                    QkvProblem* p) {
    if (!a_shape || !at || !p) return QMOE_ERR_INVALID_ARGUMENT;
    if (at->K <= 0 || at->Nq <= 0 || at->Nkv <= 0 || at->block_size <= 0)
        return QMOE_ERR_INVALID_ARGUMENT;                         // required attributes
    if (at->bits != 4 || at->block_size != 32 || at->accuracy_level != 0)
        return QMOE_ERR_NOT_SUPPORTED;                            // attributeConstraints
    if (dtype != QMOE_DT_F32 && dtype != QMOE_DT_F16) return QMOE_ERR_NOT_SUPPORTED;
    if (at->path != QKV_PATH_AUTO && at->path != QKV_PATH_DECODE && at->path != QKV_PATH_GENERIC)
        return QMOE_ERR_INVALID_ARGUMENT;
    if (!(at->epsilon >= 0.f)) return QMOE_ERR_INVALID_ARGUMENT;
    if (a_rank != 2 && a_rank != 3) return QMOE_ERR_INVALID_ARGUMENT;
    int64_t rows = 1;
    for (int d = 0; d < a_rank; ++d) {
        if (a_shape[d] < 0) return QMOE_ERR_INVALID_ARGUMENT;
        if (d < a_rank - 1) rows *= a_shape[d];
    }
    if (a_shape[a_rank - 1] != at->K) return QMOE_ERR_INVALID_ARGUMENT;   // ioShapeOk
    p->rows = rows;
    p->K = at->K;
    p->N[0] = at->Nq;
    p->N[1] = p->N[2] = at->Nkv;
    p->kblocks = (at->K + 31) / 32;
    p->f16 = dtype == QMOE_DT_F16;
    p->eps = at->epsilon;
    const bool decode_ok = rows <= kQkvDecodeRows && qkv_gemv_shape_ok(p->K, p->f16);
    if (at->path == QKV_PATH_AUTO) p->path = decode_ok ? QKV_PATH_DECODE : QKV_PATH_GENERIC;
    else p->path = at->path;
    if (p->path == QKV_PATH_DECODE && !decode_ok) return QMOE_ERR_NOT_SUPPORTED;
    return QMOE_OK;
}

// The plan covers the generic layout as well, so that a call whose tensors
// are not aligned for the GEMV can fall back within the same workspace.
QkvPlan qplan(const QkvProblem& p) {
    QkvPlan q;
    size_t off = 256;   // device error word
    auto take = [&](size_t b) {
        const size_t o = off;
        off = align_up(off + std::max<size_t>(b, 1), 256);
        return o;
    };
    q.off_n32 = take(4 * size_t(p.rows) * size_t(p.K));
    if (p.path == QKV_PATH_DECODE) {
        q.splits = qkv_gemv_splits(p.N, p.K);
        q.pitch16 = p.K;
        q.off_n16 = take(2 * size_t(p.rows) * size_t(q.pitch16));
        q.off_part = take(4 * size_t(q.splits) * size_t(p.rows) * size_t(p.N[0] + p.N[1] + p.N[2]));
        q.off_flags = take(8 * size_t(q.splits) * size_t(qkv_gemv_row_blocks(p.N, p.K)));
    }
    q.bytes = off;
    return q;
}

bool shape3(const int64_t* s, int64_t a, int64_t b, int64_t c) {
    return s && s[0] == a && s[1] == b && s[2] == c;
}
bool shape2(const int64_t* s, int64_t a, int64_t b) { return s && s[0] == a && s[1] == b; }

// The normalisation launch: the register form when the row fits (K % 8 == 0,
// K <= 16384, 16-byte aligned tensors), else one strided CTA per row.
template <typename T>
cudaError_t launch_norm(const QkvProblem& p, const void* A, const void* skip, const void* gamma,
                        void* residual, __half* n16, int64_t pitch16, float* n32, int32_t* err,
                        cudaStream_t s) {
    const unsigned rows = unsigned(p.rows);
    const bool regs = p.K % 8 == 0 && p.K <= 512 * 8 * 4 && aligned16(A) && aligned16(skip) &&
                      aligned16(gamma) && aligned16(residual);
    note_launch(QMOE_KERNEL_ROUTE, s, true);
    if (regs)
        qkv_norm_regs_kernel<T, 4><<<rows, 512, 0, s>>>(
            static_cast<const T*>(A), static_cast<const T*>(skip), static_cast<const T*>(gamma), p.K,
            p.eps, static_cast<T*>(residual), n16, pitch16, n32, err);
    else
        qkv_norm_kernel<T><<<rows, kNormThreads, 0, s>>>(
            static_cast<const T*>(A), static_cast<const T*>(skip), static_cast<const T*>(gamma), p.K,
            p.eps, static_cast<T*>(residual), n16, pitch16, n32, err);
    note_launch(QMOE_KERNEL_ROUTE, s, false);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_typed(const QkvProblem& p, const QkvPlan& q, const void* A, const void* skip,
                      const void* gamma, const Proj3& pj, void* residual, void* ws, cudaStream_t s) {
    char* base = static_cast<char*>(ws);
    int32_t* err = reinterpret_cast<int32_t*>(base);
    float* n32 = reinterpret_cast<float*>(base + q.off_n32);
    cudaError_t e;
    if (p.path == QKV_PATH_DECODE) {
        __half* n16 = reinterpret_cast<__half*>(base + q.off_n16);
        if ((e = launch_norm<T>(p, A, skip, gamma, residual, n16, q.pitch16, nullptr, err, s)) !=
            cudaSuccess)
            return e;
        float* part = reinterpret_cast<float*>(base + q.off_part);
        QkvGemvParams g;
        for (int i = 0; i < 3; ++i) {
            g.w[i] = pj.B[i];
            g.s[i] = pj.S[i];
            g.N[i] = p.N[i];
            g.out[i] = pj.out[i];
        }
        g.part[0] = part;
        g.part[1] = part + int64_t(q.splits) * p.rows * p.N[0];
        g.part[2] = g.part[1] + int64_t(q.splits) * p.rows * p.N[1];
        g.K = p.K;
        g.rows = int(p.rows);
        g.scales_f16 = p.f16;
        g.b_src = n16;
        g.b_pitch = q.pitch16;
        g.splits = q.splits;
        g.flags = reinterpret_cast<unsigned long long*>(base + q.off_flags);
        g.err = err;
        return launch_qkv_gemv(g, s);
    }
    if ((e = launch_norm<T>(p, A, skip, gamma, residual, nullptr, 0, n32, err, s)) != cudaSuccess)
        return e;
    const int64_t warps = p.rows * (p.N[0] + p.N[1] + p.N[2]);
    note_launch(QMOE_KERNEL_FC1, s, true);
    qkv_generic_kernel<T><<<unsigned((warps + 7) / 8), 256, 0, s>>>(pj, n32, p.rows, p.K);
    note_launch(QMOE_KERNEL_FC1, s, false);
    return cudaGetLastError();
}

}  // namespace
}  // namespace qmoe

using namespace qmoe;

extern "C" {

void qkv_attrs_default(qkv_attrs* a) {
    if (!a) return;
    std::memset(a, 0, sizeof(*a));
    a->bits = 4;
    a->accuracy_level = 0;
    a->epsilon = 9.999999974752427e-7f;
    a->path = QKV_PATH_AUTO;
}

qmoe_status qkv_workspace_size(const int64_t* a_shape, int32_t a_rank, const qkv_attrs* attrs,
                               int32_t dtype, size_t* bytes) {
    if (!bytes) return QMOE_ERR_INVALID_ARGUMENT;
    QkvProblem p;
    qmoe_status st = qderive(a_shape, a_rank, attrs, dtype, &p);
    if (st != QMOE_OK) return st;
    *bytes = qplan(p).bytes;
    return QMOE_OK;
}

qmoe_status qkv_choose_path(const int64_t* a_shape, int32_t a_rank, const qkv_attrs* attrs,
                            int32_t dtype, int32_t* path) {
    if (!path) return QMOE_ERR_INVALID_ARGUMENT;
    QkvProblem p;
    qmoe_status st = qderive(a_shape, a_rank, attrs, dtype, &p);
    if (st != QMOE_OK) return st;
    *path = p.path;
    return QMOE_OK;
}

qmoe_status matmul_nbits_qkv(const void* A, const int64_t* a_shape, int32_t a_rank,
                             const void* skip, const void* norm_scale, const uint8_t* q_B,
                             const int64_t* q_B_shape, const void* q_scales,
                             const int64_t* q_scales_shape, const uint8_t* k_B,
                             const int64_t* k_B_shape, const void* k_scales,
                             const int64_t* k_scales_shape, const uint8_t* v_B,
                             const int64_t* v_B_shape, const void* v_scales,
                             const int64_t* v_scales_shape, void* Q, void* Kout, void* V,
                             void* residual, int32_t dtype, const qkv_attrs* attrs,
                             void* workspace, size_t workspace_bytes, void* cuda_stream) {
    QkvProblem p;
    qmoe_status st = qderive(a_shape, a_rank, attrs, dtype, &p);
    if (st != QMOE_OK) return st;
    // derive.weightShapeOk and scaleShapeOk: [N, kBlocks, blobSize] with blobSize * 8 == 32 * 4
    if (!shape3(q_B_shape, p.N[0], p.kblocks, 16) || !shape3(k_B_shape, p.N[1], p.kblocks, 16) ||
        !shape3(v_B_shape, p.N[2], p.kblocks, 16))
        return QMOE_ERR_INVALID_ARGUMENT;
    if (!shape2(q_scales_shape, p.N[0], p.kblocks) || !shape2(k_scales_shape, p.N[1], p.kblocks) ||
        !shape2(v_scales_shape, p.N[2], p.kblocks))
        return QMOE_ERR_INVALID_ARGUMENT;
    if (residual && !skip) return QMOE_ERR_INVALID_ARGUMENT;      // normContractOk
    QkvPlan q = qplan(p);
    if (p.rows == 0) return QMOE_OK;
    if (!A || !norm_scale || !q_B || !k_B || !v_B || !q_scales || !k_scales || !v_scales || !Q ||
        !Kout || !V || !workspace)
        return QMOE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return QMOE_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < q.bytes) return QMOE_ERR_WORKSPACE_TOO_SMALL;
    if (p.path == QKV_PATH_DECODE) {
        const bool ok = aligned16(q_B) && aligned16(k_B) && aligned16(v_B) && aligned16(q_scales) &&
                        aligned16(k_scales) && aligned16(v_scales);
        if (!ok) {
            if (attrs->path == QKV_PATH_DECODE) return QMOE_ERR_NOT_SUPPORTED;
            p.path = QKV_PATH_GENERIC;   // the plan's n32 region serves the scalar path
        }
    }
    Proj3 pj;
    pj.B[0] = q_B; pj.B[1] = k_B; pj.B[2] = v_B;
    pj.S[0] = q_scales; pj.S[1] = k_scales; pj.S[2] = v_scales;
    pj.out[0] = Q; pj.out[1] = Kout; pj.out[2] = V;
    for (int i = 0; i < 3; ++i) pj.N[i] = p.N[i];
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e = p.f16 ? run_typed<__half>(p, q, A, skip, norm_scale, pj, residual, workspace, s)
                          : run_typed<float>(p, q, A, skip, norm_scale, pj, residual, workspace, s);
    return e == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

}  // extern "C"
