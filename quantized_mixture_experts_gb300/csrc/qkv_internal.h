// Internal declarations of the RMSNorm + 4-bit Q/K/V projection
// (com.microsoft.MatMulNBitsQkv manifest): the weight-streaming GEMV shared
// with the decode path of the QMoE layer, and the validated problem.
#pragma once

#include <cuda_fp16.h>

#include "qkv.h"
#include "qmoe_internal.h"

namespace qmoe {

// Few-row GEMV over the three projections in one launch.  Weights [N_p, K/2]
// bytes (the [N, kBlocks, 16] blobs read as rows), block-32 scales [N_p, K/32]
// (fp32, or fp16 when scales_f16).  Activations: the normalised rows in fp16,
// in the 4-bit operand order of the decode path (groups of eight stored as
// 0,4,2,6,1,5,3,7 with the odd elements divided by 16), b_pitch halves apart.
// Writes the results out[p][row][N_p] in T1 (fp16 when scales_f16, as T1 is the
// scales' type).  Row blocks that several CTAs share pass fp32 partial sums
// through part[p][slot][row][N_p] and completion flags flags[row block][slot]
// (any initial content) to the CTA that finishes them.  Launched as a
// programmatic dependent of the kernel that writes b_src.
struct QkvGemvParams {
    const uint8_t* w[3] = {nullptr, nullptr, nullptr};
    const void* s[3] = {nullptr, nullptr, nullptr};
    int64_t N[3] = {0, 0, 0};
    int64_t K = 0;
    int rows = 0;
    bool scales_f16 = false;
    const __half* b_src = nullptr;
    int64_t b_pitch = 0;
    float* part[3] = {nullptr, nullptr, nullptr};
    unsigned long long* flags = nullptr;
    void* out[3] = {nullptr, nullptr, nullptr};
    int splits = 1;
    int32_t* err = nullptr;
};

constexpr int kQkvDecodeRows = 16;   // rows the GEMV path takes
constexpr int kQkvRowBlock = 128;    // weight rows per GEMV work piece
constexpr uint32_t kQkvPreStages = 2; // stages whose weights the GEMV loads before its inputs are ready

// The GEMV's flat work range: K chunks per row, (row block, K chunk) pairs of the
// three projections, and its grid (each CTA takes an equal contiguous piece).
void qkv_gemv_geometry(const int64_t N[3], int64_t K, int64_t* nkc, int64_t* n_rb,
                       int64_t* total, int64_t* grid);

bool qkv_gemv_shape_ok(int64_t K, bool scales_f16);
// Partial-sum slots of the GEMV: the most CTAs that share one row block.
int qkv_gemv_splits(const int64_t N[3], int64_t K);
// Row blocks of the three projections (flags per slot each).
int64_t qkv_gemv_row_blocks(const int64_t N[3], int64_t K);
cudaError_t launch_qkv_gemv(const QkvGemvParams& p, cudaStream_t s);

}  // namespace qmoe
