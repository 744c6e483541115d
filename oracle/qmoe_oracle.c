/*
 * Reference oracle for the QMoE layer and for GroupedMatMul.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, scalar CPU
 * restatement of the operator definitions in double precision.  Only the
 * test-suite, the package smoke check and the CPU-baseline leg of the bench
 * may load it.  It shares no code, header, table or helper with the CUDA
 * library; neither side includes or links the other.
 *
 * Sources (web pages, cited by title and section):
 *   [GMM]  ONNX operator page "GroupedMatMul - 29", sections Summary, Inputs,
 *          Outputs, Type Constraints.
 *   [QMOE] com.microsoft.QMoE WebGPU kernel manifest (v1): keys description,
 *          inputs[], attributes, attributeDescriptions, attributeConstraints,
 *          derive.*.
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes of the repository):
 *   - nibble order: the low nibble of byte b holds element 2b, the high
 *     nibble element 2b+1 (plain shift-and-mask from bit 0);
 *   - interleaved SwiGLU: FC1 row 2j is the gate, row 2j+1 the linear branch;
 *   - SwiGLU: a = g * sigmoid(alpha*g) * (u + beta);
 *   - swiglu_limit clamps the gate from above and the linear branch on both
 *     sides (parity unpinned: no page value fixes it);
 *   - top-k: descending logit, ties to the lower expert index.
 *
 * All arithmetic is IEEE double.  Inputs given as float are widened exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_INDEX (-1)
#define ORACLE_BAD_ARG (-2)
#define ORACLE_NO_MEMORY (-3)

/* ------------------------------------------------------------------------ */
/* GroupedMatMul                                                             */
/* ------------------------------------------------------------------------ */

/*
 * [GMM] Summary: output[m, i] = input[m] @ weights[group_indices[m, i]],
 * plus bias[group_indices[m, i]] when the optional bias is present.
 * input [M,K], weights [G,K,N], group_indices [M,S], bias [G,N] or NULL,
 * output [M,S,N].  An index outside [0,G) is invalid input [GMM] Summary;
 * the oracle reports it and leaves that output row untouched.
 */
int oracle_grouped_matmul(const double *input, int64_t M, int64_t K,
                          const double *weights, int64_t G, int64_t N,
                          const int64_t *group_indices, int64_t S,
                          const double *bias, double *output)
{
    int status = ORACLE_OK;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t i = 0; i < S; ++i) {
            int64_t g = group_indices[m * S + i];
            if (g < 0 || g >= G) {
                status = ORACLE_BAD_INDEX;
                continue;
            }
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += input[m * K + k] * weights[(g * K + k) * N + n];
                if (bias)
                    acc += bias[g * N + n];
                output[(m * S + i) * N + n] = acc;
            }
        }
    }
    return status;
}

/*
 * [GMM] Summary, second paragraph: the function body defines the result by
 * Gather, Expand and MatMul.  This routine follows that decomposition
 * literally: it gathers the selected weights into W_sel[M*S, K, N], expands
 * each input row to its S selections, and runs one MatMul per selection.  It
 * exists to cross-check oracle_grouped_matmul; it does not share its loops.
 */
int oracle_grouped_matmul_decomposed(const double *input, int64_t M, int64_t K,
                                     const double *weights, int64_t G, int64_t N,
                                     const int64_t *group_indices, int64_t S,
                                     const double *bias, double *output)
{
    int64_t P = M * S;
    if (P == 0 || N == 0)
        return ORACLE_OK;
    for (int64_t p = 0; p < P; ++p)
        if (group_indices[p] < 0 || group_indices[p] >= G)
            return ORACLE_BAD_INDEX;
    /* Gather: W_sel[p] = weights[group_indices[p]]  ([M*S, K, N]). */
    double *w_sel = (double *)malloc((size_t)(P * (K > 0 ? K : 1) * N) * sizeof(double));
    /* Expand: x_exp[p] = input[p / S]  ([M*S, K]). */
    double *x_exp = (double *)malloc((size_t)(P * (K > 0 ? K : 1)) * sizeof(double));
    if (!w_sel || !x_exp) {
        free(w_sel);
        free(x_exp);
        return ORACLE_NO_MEMORY;
    }
    for (int64_t p = 0; p < P; ++p) {
        memcpy(w_sel + p * K * N, weights + group_indices[p] * K * N,
               (size_t)(K * N) * sizeof(double));
        memcpy(x_exp + p * K, input + (p / S) * K, (size_t)K * sizeof(double));
    }
    /* MatMul per selection: [1,K] x [K,N] -> [1,N], accumulated k-outer. */
    for (int64_t p = 0; p < P; ++p) {
        double *out = output + p * N;
        for (int64_t n = 0; n < N; ++n)
            out[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double xv = x_exp[p * K + k];
            const double *wrow = w_sel + (p * K + k) * N;
            for (int64_t n = 0; n < N; ++n)
                out[n] += xv * wrow[n];
        }
        if (bias) {
            const double *b = bias + group_indices[p] * N;
            for (int64_t n = 0; n < N; ++n)
                out[n] += b[n];
        }
    }
    free(w_sel);
    free(x_exp);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* QMoE pieces                                                               */
/* ------------------------------------------------------------------------ */

/*
 * [QMOE] derive.quantMidpoint / derive.packSize and inputs[2], inputs[4]:
 * symmetric integer code of element j of a packed row.  8-bit: one code per
 * byte.  4-bit: two codes per byte, element j in byte j/2, low nibble first.
 */
int oracle_weight_code(const uint8_t *packed_row, int64_t j, int bits)
{
    if (bits == 8)
        return (int)packed_row[j];
    uint8_t byte = packed_row[j / 2];
    return (j % 2 == 0) ? (int)(byte & 0x0F) : (int)(byte >> 4);
}

/*
 * [QMOE] description ("4- and 8-bit symmetric dequantization") with
 * derive.quantMidpoint (8 for 4-bit, 128 for 8-bit) and
 * attributeDescriptions.block_size (omitted => one scale per stored row,
 * else one scale per block_size run of the reduction axis):
 *   w = (q - midpoint) * scale.
 * `scale_row` points at the scales of this stored row: one value when
 * block_size == 0, else K / block_size values.
 */
double oracle_dequant(const uint8_t *packed_row, const float *scale_row,
                      int64_t j, int bits, int64_t block_size)
{
    int midpoint = (bits == 4) ? 8 : 128;
    int q = oracle_weight_code(packed_row, j, bits);
    double scale = (block_size == 0) ? (double)scale_row[0]
                                     : (double)scale_row[j / block_size];
    return (double)(q - midpoint) * scale;
}

/* Dequantize `rows` full rows of length K (test helper over oracle_dequant). */
void oracle_dequant_rows(const uint8_t *packed, const float *scales, int64_t rows,
                         int64_t K, int bits, int64_t block_size, double *out)
{
    int64_t packed_cols = (bits == 4) ? K / 2 : K;
    int64_t scale_cols = (block_size == 0) ? 1 : K / block_size;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < K; ++j)
            out[r * K + j] = oracle_dequant(packed + r * packed_cols,
                                            scales + r * scale_cols, j, bits,
                                            block_size);
}

/*
 * [QMOE] description (the routing weights are a softmax taken over the k
 * selected logits only) and attributeDescriptions.normalize_routing_weights
 * (the same softmax for either value of the attribute).  Selection i is the i-th
 * largest logit; equal logits go to the lower expert index.  Then
 *   p_i = exp(l_i - l_max) / sum_j exp(l_j - l_max)  over the k selected.
 */
int oracle_route(const float *logits_row, int64_t E, int64_t k,
                 int32_t *sel, double *p)
{
    if (k < 1 || k > E)
        return ORACLE_BAD_ARG;
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    if (!taken)
        return ORACLE_NO_MEMORY;
    for (int64_t i = 0; i < k; ++i) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || (double)logits_row[e] > (double)logits_row[best])
                best = e;
        }
        taken[best] = 1;
        sel[i] = (int32_t)best;
    }
    free(taken);
    double lmax = (double)logits_row[sel[0]];
    double denom = 0.0;
    for (int64_t i = 0; i < k; ++i)
        denom += exp((double)logits_row[sel[i]] - lmax);
    for (int64_t i = 0; i < k; ++i)
        p[i] = exp((double)logits_row[sel[i]] - lmax) / denom;
    return ORACLE_OK;
}

/*
 * [QMOE] attributeDescriptions.activation_type / swiglu_fusion /
 * activation_alpha / activation_beta / swiglu_limit.
 * ReLU: a[n] = max(0, h[n]) for n < inter.
 * Interleaved SwiGLU: g = h[2j] (gate), u = h[2j+1] (linear),
 *   optional clamp, a[j] = g * sigmoid(alpha*g) * (u + beta).
 */
void oracle_activation(const double *h, int64_t inter, int activation,
                       double alpha, double beta, int has_limit, double limit,
                       double *a)
{
    if (activation == 0) {
        for (int64_t n = 0; n < inter; ++n)
            a[n] = h[n] > 0.0 ? h[n] : 0.0;
        return;
    }
    for (int64_t j = 0; j < inter; ++j) {
        double g = h[2 * j];
        double u = h[2 * j + 1];
        if (has_limit) {
            if (g > limit)
                g = limit;
            if (u > limit)
                u = limit;
            if (u < -limit)
                u = -limit;
        }
        double sig = 1.0 / (1.0 + exp(-alpha * g));
        a[j] = g * sig * (u + beta);
    }
}

typedef struct {
    const float *x;
    int64_t H;
    const float *logits;
    int64_t E;
    const uint8_t *w1;
    const float *s1;
    const uint8_t *w2;
    const float *s2;
    int64_t I;
    int bits;
    int64_t block_size;
    int activation;
    double alpha, beta;
    int has_limit;
    double limit;
    int64_t k;
    int dense;               /* 1 => brute-force evaluation over all experts */
    const int64_t *tokens;   /* token ids to evaluate                        */
    int64_t first, last;     /* [first,last) range of `tokens` for a thread  */
    double *y;               /* [ntok, H]                                     */
    int32_t *sel_out;        /* [ntok, k] or NULL                             */
    double *p_out;           /* [ntok, k] or NULL                             */
    int status;
} oracle_job;

/*
 * One expert's feed-forward for one token, [QMOE] inputs[2..5]:
 *   FC1  h[n] = sum_{j<H} x[j] * deq(W1[e, n, j]),  n < fusion*inter
 *   act  a    = activation(h)
 *   FC2  o[d] = sum_{j<inter} a[j] * deq(W2[e, d, j]),  d < H
 */
static void oracle_expert_ffn(const oracle_job *job, const float *xt, int64_t e,
                              double *h, double *a, double *o)
{
    const int64_t H = job->H, I = job->I;
    const int fusion = (job->activation == 1) ? 2 : 1;
    const int64_t rows1 = fusion * I;
    const int64_t pc1 = (job->bits == 4) ? H / 2 : H;
    const int64_t pc2 = (job->bits == 4) ? I / 2 : I;
    const int64_t sc1 = (job->block_size == 0) ? 1 : H / job->block_size;
    const int64_t sc2 = (job->block_size == 0) ? 1 : I / job->block_size;
    const uint8_t *w1e = job->w1 + e * rows1 * pc1;
    const float *s1e = job->s1 + e * rows1 * sc1;
    const uint8_t *w2e = job->w2 + e * H * pc2;
    const float *s2e = job->s2 + e * H * sc2;

    for (int64_t n = 0; n < rows1; ++n) {
        double acc = 0.0;
        for (int64_t j = 0; j < H; ++j)
            acc += (double)xt[j] * oracle_dequant(w1e + n * pc1, s1e + n * sc1, j,
                                                  job->bits, job->block_size);
        h[n] = acc;
    }
    oracle_activation(h, I, job->activation, job->alpha, job->beta,
                      job->has_limit, job->limit, a);
    for (int64_t d = 0; d < H; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < I; ++j)
            acc += a[j] * oracle_dequant(w2e + d * pc2, s2e + d * sc2, j,
                                         job->bits, job->block_size);
        o[d] = acc;
    }
}

static void *oracle_qmoe_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    const int64_t H = job->H, I = job->I, E = job->E, k = job->k;
    const int fusion = (job->activation == 1) ? 2 : 1;
    double *h = (double *)malloc((size_t)(fusion * I + 1) * sizeof(double));
    double *a = (double *)malloc((size_t)(I + 1) * sizeof(double));
    double *o = (double *)malloc((size_t)(H + 1) * sizeof(double));
    int32_t *sel = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    double *p = (double *)malloc((size_t)k * sizeof(double));
    if (!h || !a || !o || !sel || !p) {
        job->status = ORACLE_NO_MEMORY;
        goto done;
    }
    for (int64_t r = job->first; r < job->last; ++r) {
        int64_t t = job->tokens[r];
        const float *xt = job->x + t * H;
        double *yt = job->y + r * H;
        int st = oracle_route(job->logits + t * E, E, k, sel, p);
        if (st != ORACLE_OK) {
            job->status = st;
            goto done;
        }
        if (job->sel_out)
            for (int64_t i = 0; i < k; ++i)
                job->sel_out[r * k + i] = sel[i];
        if (job->p_out)
            for (int64_t i = 0; i < k; ++i)
                job->p_out[r * k + i] = p[i];
        for (int64_t d = 0; d < H; ++d)
            yt[d] = 0.0;
        /* [QMOE] variants[quant_zero_inter]: inter_size == 0 gives zeros. */
        if (I == 0)
            continue;
        if (!job->dense) {
            /* Weighted sum over the k selections, [QMOE] pass QMoE.MixStage. */
            for (int64_t i = 0; i < k; ++i) {
                oracle_expert_ffn(job, xt, sel[i], h, a, o);
                for (int64_t d = 0; d < H; ++d)
                    yt[d] += p[i] * o[d];
            }
        } else {
            /* Brute force: every expert, weight 0 unless selected. */
            for (int64_t e = 0; e < E; ++e) {
                double r_e = 0.0;
                for (int64_t i = 0; i < k; ++i)
                    if (sel[i] == e)
                        r_e = p[i];
                oracle_expert_ffn(job, xt, e, h, a, o);
                for (int64_t d = 0; d < H; ++d)
                    yt[d] += r_e * o[d];
            }
        }
    }
done:
    free(h);
    free(a);
    free(o);
    free(sel);
    free(p);
    return NULL;
}

/*
 * The QMoE layer for the listed tokens ([QMOE] description, inputs,
 * attributes).  x [T,H] (any leading shape flattened by the caller),
 * logits [T,E], w1 [E, fusion*I, H/pack], s1 [E, fusion*I] or
 * [E, fusion*I, H/bs], w2 [E, H, I/pack], s2 [E, H] or [E, H, I/bs].
 * tokens: the ntok token ids to evaluate; y [ntok, H] receives their
 * outputs; sel_out / p_out (nullable) [ntok, k] receive the routing.
 * dense = 1 selects the brute-force evaluation over all experts.
 * nthreads splits the token list into contiguous ranges, one per thread;
 * every token is computed the same way whatever the split.
 */
int oracle_qmoe(const float *x, int64_t H, const float *logits, int64_t E,
                const uint8_t *w1, const float *s1, const uint8_t *w2,
                const float *s2, int64_t I, int bits, int64_t block_size,
                int activation, double alpha, double beta, int has_limit,
                double limit, int64_t k, const int64_t *tokens, int64_t ntok,
                int dense, double *y, int32_t *sel_out, double *p_out,
                int nthreads)
{
    if (bits != 4 && bits != 8)
        return ORACLE_BAD_ARG;
    if (activation != 0 && activation != 1)
        return ORACLE_BAD_ARG;
    if (k < 1 || k > E)
        return ORACLE_BAD_ARG;
    if (ntok <= 0)
        return ORACLE_OK;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > ntok)
        nthreads = (int)ntok;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_NO_MEMORY;
    }
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->x = x; j->H = H; j->logits = logits; j->E = E;
        j->w1 = w1; j->s1 = s1; j->w2 = w2; j->s2 = s2; j->I = I;
        j->bits = bits; j->block_size = block_size; j->activation = activation;
        j->alpha = alpha; j->beta = beta; j->has_limit = has_limit; j->limit = limit;
        j->k = k; j->dense = dense; j->tokens = tokens;
        j->first = ntok * t / nthreads;
        j->last = ntok * (t + 1) / nthreads;
        j->y = y; j->sel_out = sel_out; j->p_out = p_out;
        j->status = ORACLE_OK;
    }
    int status = ORACLE_OK;
    if (nthreads == 1) {
        oracle_qmoe_worker(&jobs[0]);
    } else {
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&tids[t], NULL, oracle_qmoe_worker, &jobs[t]) != 0)
                break;
            ++started;
        }
        for (int t = started; t < nthreads; ++t)
            oracle_qmoe_worker(&jobs[t]);
        for (int t = 0; t < started; ++t)
            pthread_join(tids[t], NULL);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != ORACLE_OK)
            status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}
