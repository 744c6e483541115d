// GroupedMatMul (ONNX "GroupedMatMul - 29", Summary):
//   output[m, i, :] = input[m, :] @ weights[g] (+ bias[g]),  g = group_indices[m, i].
//
// Tiled kernel: one CTA computes a 64-column strip of the output for a block
// of (m, i) rows that share nothing but the layout; each thread owns one
// column and 4 rows, the input rows are staged in shared memory in K-chunks.
// Accumulation is fp32 for f32/f16/bf16 and fp64 for f64.  An index outside
// [0, G) is invalid input on the page; the row is written as zeros and the
// device error word records QMOE_DEVERR_INDEX.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qmoe_internal.h"

namespace qmoe {
namespace {

template <typename T> struct Acc { using type = float; };
template <> struct Acc<double> { using type = double; };

template <typename T> __device__ __forceinline__ typename Acc<T>::type to_acc(T v) {
    return static_cast<typename Acc<T>::type>(v);
}
template <> __device__ __forceinline__ float to_acc<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_acc<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_acc(typename Acc<T>::type v) {
    return static_cast<T>(v);
}
template <> __device__ __forceinline__ __half from_acc<__half>(float v) {
    return __float2half_rn(v);
}
template <> __device__ __forceinline__ __nv_bfloat16 from_acc<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

constexpr int kCols = 64;     // output columns per CTA (one per thread in x)
constexpr int kRowsY = 4;     // thread rows
constexpr int kRowsPer = 4;   // (m,i) rows per thread
constexpr int kRows = kRowsY * kRowsPer;   // 16 (m,i) rows per CTA
constexpr int kKChunk = 64;

template <typename T, typename TI>
__global__ void __launch_bounds__(kCols * kRowsY) gmm_kernel(
    const T* __restrict__ input, int64_t M, int64_t K, const T* __restrict__ weights, int64_t G,
    int64_t N, const TI* __restrict__ idx, int64_t S, const T* __restrict__ bias,
    T* __restrict__ out, int32_t* __restrict__ err) {
    using A = typename Acc<T>::type;
    __shared__ A s_x[kRows][kKChunk];
    __shared__ int64_t s_g[kRows];
    const int tx = threadIdx.x % kCols, ty = threadIdx.x / kCols;
    const int64_t n = int64_t(blockIdx.y) * kCols + tx;
    const int64_t r0 = int64_t(blockIdx.x) * kRows;   // first flattened (m,i) row
    const int64_t R = M * S;
    if (threadIdx.x < kRows) {
        const int64_t r = r0 + threadIdx.x;
        int64_t g = -1;
        if (r < R) {
            g = int64_t(idx[r]);
            if (g < 0 || g >= G) {
                atomicCAS(err, 0, int32_t(QMOE_DEVERR_INDEX));
                g = -1;
            }
        }
        s_g[threadIdx.x] = g;
    }
    __syncthreads();
    A acc[kRowsPer];
#pragma unroll
    for (int q = 0; q < kRowsPer; ++q) acc[q] = A(0);
    for (int64_t k0 = 0; k0 < K; k0 += kKChunk) {
        __syncthreads();
        for (int e = threadIdx.x; e < kRows * kKChunk; e += blockDim.x) {
            const int rr = e / kKChunk, kk = e % kKChunk;
            const int64_t r = r0 + rr;
            A v = A(0);
            if (r < R && k0 + kk < K) v = to_acc<T>(input[(r / S) * K + k0 + kk]);
            s_x[rr][kk] = v;
        }
        __syncthreads();
        if (n < N) {
            const int kmax = int(K - k0 < kKChunk ? K - k0 : kKChunk);
#pragma unroll
            for (int q = 0; q < kRowsPer; ++q) {
                const int rr = ty * kRowsPer + q;
                const int64_t g = s_g[rr];
                if (g < 0) continue;
                const T* __restrict__ wcol = weights + (g * K + k0) * N + n;
                A a = acc[q];
                for (int kk = 0; kk < kmax; ++kk) a += s_x[rr][kk] * to_acc<T>(wcol[int64_t(kk) * N]);
                acc[q] = a;
            }
        }
    }
    if (n >= N) return;
#pragma unroll
    for (int q = 0; q < kRowsPer; ++q) {
        const int rr = ty * kRowsPer + q;
        const int64_t r = r0 + rr;
        if (r >= R) continue;
        const int64_t g = s_g[rr];
        A v = A(0);
        if (g >= 0) {
            v = acc[q];
            if (bias) v += to_acc<T>(bias[g * N + n]);
        }
        out[r * N + n] = from_acc<T>(v);
    }
}

template <typename T, typename TI>
cudaError_t run(const void* input, int64_t M, int64_t K, const void* weights, int64_t G,
                int64_t N, const void* idx, int64_t S, const void* bias, void* out, int32_t* err,
                cudaStream_t s) {
    const int64_t R = M * S;
    dim3 grid(unsigned((R + kRows - 1) / kRows), unsigned((N + kCols - 1) / kCols));
    gmm_kernel<T, TI><<<grid, kCols * kRowsY, 0, s>>>(
        static_cast<const T*>(input), M, K, static_cast<const T*>(weights), G, N,
        static_cast<const TI*>(idx), S, static_cast<const T*>(bias), static_cast<T*>(out), err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_t(const void* input, int64_t M, int64_t K, const void* weights, int64_t G,
                  int64_t N, const void* idx, int64_t S, int idx64, const void* bias, void* out,
                  int32_t* err, cudaStream_t s) {
    if (idx64) return run<T, int64_t>(input, M, K, weights, G, N, idx, S, bias, out, err, s);
    return run<T, int32_t>(input, M, K, weights, G, N, idx, S, bias, out, err, s);
}

}  // namespace

cudaError_t launch_grouped_matmul(const void* input, int64_t M, int64_t K, const void* weights,
                                  int64_t G, int64_t N, const void* idx, int64_t S, int idx64,
                                  const void* bias, void* out, int dtype, int32_t* err,
                                  cudaStream_t s) {
    note_launch(QMOE_KERNEL_GMM, s, true);
    cudaError_t e;
    switch (dtype) {
        case QMOE_DT_F32: e = run_t<float>(input, M, K, weights, G, N, idx, S, idx64, bias, out, err, s); break;
        case QMOE_DT_F16: e = run_t<__half>(input, M, K, weights, G, N, idx, S, idx64, bias, out, err, s); break;
        case QMOE_DT_BF16: e = run_t<__nv_bfloat16>(input, M, K, weights, G, N, idx, S, idx64, bias, out, err, s); break;
        default: e = run_t<double>(input, M, K, weights, G, N, idx, S, idx64, bias, out, err, s); break;
    }
    note_launch(QMOE_KERNEL_GMM, s, false);
    return e;
}

}  // namespace qmoe
