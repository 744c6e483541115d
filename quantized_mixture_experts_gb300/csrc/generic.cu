// Scalar fp32 kernels of the QMoE layer for shapes the tensor-core paths do
// not take (no alignment requirements), plus the weighted combine shared by
// every path.
//
// QMoE manifest: inputs[2..5] (packed layouts), derive.quantMidpoint /
// packSize (w = (q - mid) * scale, low nibble first), attributeDescriptions
// (ReLU, interleaved SwiGLU, alpha, beta, swiglu_limit), pass QMoE.MixStage.
#include "qmoe_internal.h"
#include "tma_host.h"

namespace qmoe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float deq(const uint8_t* __restrict__ row,
                                     const float* __restrict__ srow, int64_t j, int bits, int mid,
                                     int64_t bs) {
    int q;
    if (bits == 8) {
        q = row[j];
    } else {
        const uint8_t b = row[j >> 1];
        q = (j & 1) ? (b >> 4) : (b & 15);
    }
    const float sc = bs ? srow[j / bs] : srow[0];
    return float(q - mid) * sc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

__device__ __forceinline__ float swiglu(float g, float u, float alpha, float beta, int has_limit,
                                        float limit) {
    if (has_limit) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    const float sig = 1.f / (1.f + expf(-alpha * g));
    return g * sig * (u + beta);
}

// One warp per (sorted row, output column j): FC1 dot product(s) + activation.
__global__ void generic_fc1_kernel(Problem p, const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ sel, float* __restrict__ act,
                                   int64_t total) {
    const int64_t widx = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (widx >= total) return;
    const int64_t slots = total / p.I;
    const int64_t j = widx / slots, pos = widx % slots;   // weight-row major: rows stay in cache
    const int32_t s = perm[pos];
    const int64_t t = s / p.k;
    const int64_t e = sel[s];
    const int64_t rows1 = p.fusion * p.I;
    const int64_t pc = p.H / p.pack;
    const float* __restrict__ xt = p.x + t * p.H;
    const uint8_t* __restrict__ we = p.w1 + e * rows1 * pc;
    const float* __restrict__ se = p.s1 + e * rows1 * p.nb1;
    float out;
    if (p.act == QMOE_ACT_SWIGLU) {
        const int64_t rg = 2 * j, ru = 2 * j + 1;
        float g = 0.f, u = 0.f;
        for (int64_t kk = lane; kk < p.H; kk += 32) {
            const float xv = xt[kk];
            g += xv * deq(we + rg * pc, se + rg * p.nb1, kk, p.bits, p.mid, p.bs);
            u += xv * deq(we + ru * pc, se + ru * p.nb1, kk, p.bits, p.mid, p.bs);
        }
        g = warp_sum(g);
        u = warp_sum(u);
        out = swiglu(g, u, p.alpha, p.beta, p.has_limit, p.limit);
    } else {
        float h = 0.f;
        for (int64_t kk = lane; kk < p.H; kk += 32)
            h += xt[kk] * deq(we + j * pc, se + j * p.nb1, kk, p.bits, p.mid, p.bs);
        h = warp_sum(h);
        out = fmaxf(h, 0.f);
    }
    if (lane == 0) act[pos * p.I + j] = out;
}

// One warp per (sorted row, output column d): FC2 dot product, written to the
// row of the original slot.
__global__ void generic_fc2_kernel(Problem p, const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ sel,
                                   const float* __restrict__ act, float* __restrict__ slot_out,
                                   int64_t total) {
    const int64_t widx = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (widx >= total) return;
    const int64_t slots = total / p.H;
    const int64_t d = widx / slots, pos = widx % slots;
    const int32_t s = perm[pos];
    const int64_t e = sel[s];
    const int64_t pc = p.I / p.pack;
    const uint8_t* __restrict__ wr = p.w2 + (e * p.H + d) * pc;
    const float* __restrict__ sr = p.s2 + (e * p.H + d) * p.nb2;
    const float* __restrict__ ar = act + pos * p.I;
    float o = 0.f;
    for (int64_t kk = lane; kk < p.I; kk += 32) o += ar[kk] * deq(wr, sr, kk, p.bits, p.mid, p.bs);
    o = warp_sum(o);
    if (lane == 0) slot_out[int64_t(s) * p.H + d] = o;
}

// y[t, d] = sum_i pw[t,i] * sum_split slot_out[split][t*k+i][d], in ascending
// i and split order (deterministic, no atomics).
__global__ void combine_kernel(const float* __restrict__ slot_out, const float* __restrict__ pw,
                               float* __restrict__ y, int64_t T, int64_t H, int k, int splits,
                               int64_t slots, int vec) {
    // launched as a dependent of the kernel that writes slot_out
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec) {
        const int64_t H4 = H / 4;
        if (idx >= T * H4) return;
        const int64_t t = idx / H4, d4 = idx % H4;
        const float4* base = reinterpret_cast<const float4*>(slot_out + t * k * H) + d4;
        const int64_t sstride = slots * H / 4;   // between K splits
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (splits == 1 && k <= 16) {
            // issue every slot's load first; the sum keeps ascending slot order
            float4 v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i < k) v[i] = __ldg(base + int64_t(i) * (H / 4));
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i < k) {
                    const float w = pw[t * k + i];
                    acc.x += w * v[i].x; acc.y += w * v[i].y; acc.z += w * v[i].z; acc.w += w * v[i].w;
                }
        } else {
            for (int i = 0; i < k; ++i) {
                float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
                if (splits <= 8) {
                    float4 v[8];
#pragma unroll
                    for (int sp = 0; sp < 8; ++sp)
                        if (sp < splits) v[sp] = __ldg(base + int64_t(i) * (H / 4) + sp * sstride);
#pragma unroll
                    for (int sp = 0; sp < 8; ++sp)
                        if (sp < splits) {
                            part.x += v[sp].x; part.y += v[sp].y; part.z += v[sp].z; part.w += v[sp].w;
                        }
                } else {
                    for (int sp = 0; sp < splits; ++sp) {
                        const float4 v = __ldg(base + int64_t(i) * (H / 4) + sp * sstride);
                        part.x += v.x; part.y += v.y; part.z += v.z; part.w += v.w;
                    }
                }
                const float w = pw[t * k + i];
                acc.x += w * part.x; acc.y += w * part.y; acc.z += w * part.z; acc.w += w * part.w;
            }
        }
        reinterpret_cast<float4*>(y + t * H)[d4] = acc;
    } else {
        if (idx >= T * H) return;
        const int64_t t = idx / H, d = idx % H;
        float acc = 0.f;
        for (int i = 0; i < k; ++i) {
            float part = 0.f;
            for (int sp = 0; sp < splits; ++sp)
                part += slot_out[(int64_t(sp) * slots + t * k + i) * H + d];
            acc += pw[t * k + i] * part;
        }
        y[t * H + d] = acc;
    }
}

// Same sums for large batches: CTA (t, column block); each thread owns eight
// adjacent outputs of token t (two float4), so the index math is per CTA and a
// thread keeps 2 * k * splits loads in flight.  H % 8 == 0, 16-byte aligned rows.
__global__ void combine_rows_kernel(const float* __restrict__ slot_out,
                                    const float* __restrict__ pw, float* __restrict__ y, int H4,
                                    int k, int splits, int64_t slots) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t t = blockIdx.x;
    const int d4 = 2 * (blockIdx.y * blockDim.x + threadIdx.x);
    if (d4 >= H4) return;
    const float4* __restrict__ base =
        reinterpret_cast<const float4*>(slot_out) + (t * k) * H4 + d4;
    const int64_t sstride = slots * H4;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    for (int i = 0; i < k; ++i) {
        const float w = __ldg(pw + t * k + i);
        float4 p0 = __ldg(base + int64_t(i) * H4), p1 = __ldg(base + int64_t(i) * H4 + 1);
        for (int sp = 1; sp < splits; ++sp) {
            const float4 q0 = __ldg(base + int64_t(i) * H4 + sp * sstride);
            const float4 q1 = __ldg(base + int64_t(i) * H4 + sp * sstride + 1);
            p0.x += q0.x; p0.y += q0.y; p0.z += q0.z; p0.w += q0.w;
            p1.x += q1.x; p1.y += q1.y; p1.z += q1.z; p1.w += q1.w;
        }
        a0.x += w * p0.x; a0.y += w * p0.y; a0.z += w * p0.z; a0.w += w * p0.w;
        a1.x += w * p1.x; a1.y += w * p1.y; a1.z += w * p1.z; a1.w += w * p1.w;
    }
    float4* o = reinterpret_cast<float4*>(y + t * H4 * 4) + d4;
    o[0] = a0;
    o[1] = a1;
}

unsigned blocks_for(int64_t n, int per) { return unsigned((n + per - 1) / per); }

}  // namespace

cudaError_t launch_generic_fc1(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s) {
    const int64_t total = pl.slots * p.I;
    note_launch(QMOE_KERNEL_FC1, s, true);
    generic_fc1_kernel<<<blocks_for(total, 8), 256, 0, s>>>(p, w.perm, w.sel,
                                                            static_cast<float*>(w.act), total);
    note_launch(QMOE_KERNEL_FC1, s, false);
    return cudaGetLastError();
}

cudaError_t launch_generic_fc2(const Problem& p, const Plan& pl, const Work& w, cudaStream_t s) {
    const int64_t total = pl.slots * p.H;
    note_launch(QMOE_KERNEL_FC2, s, true);
    generic_fc2_kernel<<<blocks_for(total, 8), 256, 0, s>>>(
        p, w.perm, w.sel, static_cast<const float*>(w.act), w.slot_out, total);
    note_launch(QMOE_KERNEL_FC2, s, false);
    return cudaGetLastError();
}

// y[t] = sum over i < k of s16[t * k + i]: the grouped path's FC2 rows, already
// weighted by their routing weight, added in fp32 in ascending slot order.
// One thread per 8 output columns (H % 8 == 0 on the grouped path).
__global__ void combine16_kernel(const uint4* __restrict__ s16, float* __restrict__ y, int64_t T,
                                 int64_t H, int k, int aligned) {
    // launched as a dependent of the kernel that writes the slot rows
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t H8 = H / 8;
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= T * H8) return;
    const int64_t t = idx / H8, d8 = idx % H8;
    const uint4* base = s16 + t * k * H8 + d8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i0 = 0; i0 < k; i0 += 8) {
        // issue up to eight slots' loads first; the sum keeps ascending slot order
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (i0 + j < k) v[j] = __ldg(base + int64_t(i0 + j) * H8);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (i0 + j < k) {
                const __half2* h = reinterpret_cast<const __half2*>(&v[j]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __half22float2(h[q]);
                    acc[2 * q] += f.x;
                    acc[2 * q + 1] += f.y;
                }
            }
    }
    float* out = y + t * H + 8 * d8;
    if (aligned) {
        reinterpret_cast<float4*>(out)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(out)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) out[q] = acc[q];
    }
}

cudaError_t launch_combine16(const Problem& p, const Work& w, cudaStream_t s) {
    const int64_t n = p.T * (p.H / 8);
    note_launch(QMOE_KERNEL_COMBINE, s, true);
    const int threads = n < 152 * 256 ? 64 : 256;
    cudaError_t e = launch_dependent(
        combine16_kernel, dim3(unsigned(blocks_for(n, threads))), dim3(threads), 0, s,
        reinterpret_cast<const uint4*>(w.slot_out), p.y, p.T, p.H, int(p.k),
        (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 ? 1 : 0);
    note_launch(QMOE_KERNEL_COMBINE, s, false);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_combine(const Problem& p, const Plan& pl, const Work& w, int splits,
                           cudaStream_t s) {
    const int vec = (p.H & 3) == 0 && (reinterpret_cast<uintptr_t>(p.y) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(w.slot_out) & 15) == 0;
    const int64_t n = vec ? p.T * (p.H / 4) : p.T * p.H;
    note_launch(QMOE_KERNEL_COMBINE, s, true);
    if (vec && (p.H & 7) == 0 && p.T * (p.H / 8) >= int64_t(device_sm_count()) * 256 &&
        p.T < (int64_t(1) << 31)) {
        const int H4 = int(p.H / 4);
        const int threads = H4 / 2 >= 256 ? 256 : 128;
        const dim3 grid(unsigned(p.T), unsigned((H4 / 2 + threads - 1) / threads));
        cudaError_t e = launch_dependent(combine_rows_kernel, grid, dim3(threads), 0, s,
                                         static_cast<const float*>(w.slot_out),
                                         static_cast<const float*>(w.pw), p.y, H4, int(p.k),
                                         splits, pl.slots);
        note_launch(QMOE_KERNEL_COMBINE, s, false);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int threads = n < 152 * 256 ? 64 : 256;   // spread small batches over more SMs
    cudaError_t e = launch_dependent(combine_kernel, dim3(unsigned(blocks_for(n, threads))),
                                     dim3(threads), 0, s, static_cast<const float*>(w.slot_out),
                                     static_cast<const float*>(w.pw), p.y, p.T, p.H, int(p.k),
                                     splits, pl.slots, vec);
    note_launch(QMOE_KERNEL_COMBINE, s, false);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qmoe
