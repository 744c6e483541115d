/*
 * Reference oracle for the float (unquantized) mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  A plain, slow, scalar CPU restatement of the
 * operator in double precision.  Only the test-suite, the package smoke check
 * and the CPU-baseline leg of the bench may load it.  It shares no code,
 * header, table or helper with the CUDA library (nor with the QMoE oracle in
 * qmoe_oracle.c, whose routing is different).
 *
 * Source (web page, cited by title and section):
 *   [MOE]  com.microsoft.MoE kernel README (v1): sections Description,
 *          Inputs, Outputs, Attributes, Type constraints.
 *   [QMOE] com.microsoft.QMoE WebGPU kernel manifest (v1),
 *          attributeDescriptions.activation_alpha / activation_beta /
 *          swiglu_limit (the SwiGLU parameters the MoE README leaves open).
 *
 * What the page fixes ([MOE] Description, Inputs, Attributes):
 *   p      = softmax over ALL E router logits of the token;
 *   sel    = the k experts of largest p;
 *   w_i    = p[sel_i], divided by sum_i p[sel_i] when
 *            normalize_routing_weights = 1;
 *   FC1    h1 = x . W1[e]^T + b1[e]     (W1 [E, fusion*I, H], b1 optional)
 *   FC3    h3 = x . W3[e]^T + b3[e]     (W3 [E, I, H], only when consumed)
 *   act    relu | gelu | silu | swiglu | identity on h1 (SwiGLU operands
 *          from FC3 with swiglu_fusion 0, interleaved FC1 rows with 1,
 *          concatenated FC1 halves with 2; SiLU times h3 when FC3 is given)
 *   FC2    o = a . W2[e]^T + b2[e]      (W2 [E, H, I]; bias added before
 *          the routing weight)
 *   y      = sum_i w_i * o_i.
 *
 * Readings taken where the page leaves a step open (each is listed in the
 * design notes of the repository):
 *   - top-k order: descending probability, equal probabilities to the lower
 *     expert index;
 *   - gelu is the exact form h*Phi(h) = 0.5*h*(1 + erf(h/sqrt(2)));
 *   - silu is h*sigmoid(h); alpha and beta belong to SwiGLU only ([QMOE]
 *     attributeDescriptions.activation_alpha / activation_beta describe them
 *     as SwiGLU parameters);
 *   - SwiGLU: a = g*sigmoid(alpha*g)*(u + beta); interleaved: row 2j gate,
 *     row 2j+1 linear; concatenated: rows [0, I) gate, rows [I, 2I) linear;
 *     swiglu_limit clamps the gate from above and the linear branch on both
 *     sides (parity unpinned: no page value fixes the clamp).
 *
 * All arithmetic is IEEE double.  Inputs given as float are widened exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define MOE_ORACLE_OK 0
#define MOE_ORACLE_BAD_ARG (-2)
#define MOE_ORACLE_NO_MEMORY (-3)

/* Activation codes ([MOE] Attributes, activation_type). */
#define MOE_ACT_RELU 0
#define MOE_ACT_GELU 1
#define MOE_ACT_SILU 2
#define MOE_ACT_SWIGLU 3
#define MOE_ACT_IDENTITY 4

/*
 * [MOE] Description and Attributes.normalize_routing_weights:
 * softmax over all E logits, then the k largest probabilities.
 */
int oracle_moe_route(const float *logits_row, int64_t E, int64_t k, int normalize,
                     int32_t *sel, double *w)
{
    if (k < 1 || k > E)
        return MOE_ORACLE_BAD_ARG;
    double *prob = (double *)malloc((size_t)E * sizeof(double));
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    if (!prob || !taken) {
        free(prob);
        free(taken);
        return MOE_ORACLE_NO_MEMORY;
    }
    double lmax = (double)logits_row[0];
    for (int64_t e = 1; e < E; ++e)
        if ((double)logits_row[e] > lmax)
            lmax = (double)logits_row[e];
    double z = 0.0;
    for (int64_t e = 0; e < E; ++e) {
        prob[e] = exp((double)logits_row[e] - lmax);
        z += prob[e];
    }
    for (int64_t e = 0; e < E; ++e)
        prob[e] /= z;
    for (int64_t i = 0; i < k; ++i) {
        int64_t best = -1;
        for (int64_t e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || prob[e] > prob[best])
                best = e;
        }
        taken[best] = 1;
        sel[i] = (int32_t)best;
        w[i] = prob[best];
    }
    if (normalize) {
        double s = 0.0;
        for (int64_t i = 0; i < k; ++i)
            s += w[i];
        for (int64_t i = 0; i < k; ++i)
            w[i] /= s;
    }
    free(prob);
    free(taken);
    return MOE_ORACLE_OK;
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/*
 * [MOE] Attributes.activation_type / swiglu_fusion, Inputs.fc3_experts_weights.
 * h1: FC1 output (fusion*I values); h3: FC3 output (I values) or NULL.
 * a: I values.
 */
void oracle_moe_activation(const double *h1, const double *h3, int64_t I, int act,
                           int fusion, double alpha, double beta, int has_limit,
                           double limit, double *a)
{
    for (int64_t j = 0; j < I; ++j) {
        double v = h1[j];
        switch (act) {
        case MOE_ACT_RELU:
            a[j] = v > 0.0 ? v : 0.0;
            break;
        case MOE_ACT_GELU:
            /* h * Phi(h) with Phi(h) = erfc(-h/sqrt 2) / 2, which keeps the
             * relative accuracy of 1 + erf(h/sqrt 2) where erf is near -1. */
            a[j] = 0.5 * v * erfc(-v / sqrt(2.0));
            break;
        case MOE_ACT_SILU:
            a[j] = v * sigmoid(v) * (h3 ? h3[j] : 1.0);
            break;
        case MOE_ACT_IDENTITY:
            a[j] = v;
            break;
        default: { /* SwiGLU */
            double g, u;
            if (fusion == 1) {
                g = h1[2 * j];
                u = h1[2 * j + 1];
            } else if (fusion == 2) {
                g = h1[j];
                u = h1[I + j];
            } else {
                g = h1[j];
                u = h3[j];
            }
            if (has_limit) {
                if (g > limit)
                    g = limit;
                if (u > limit)
                    u = limit;
                if (u < -limit)
                    u = -limit;
            }
            a[j] = g * sigmoid(alpha * g) * (u + beta);
        }
        }
    }
}

typedef struct {
    const float *x;
    int64_t H;
    const float *logits;
    int64_t E;
    const float *w1, *b1, *w2, *b2, *w3, *b3;
    int64_t I;
    int act, fusion;
    double alpha, beta;
    int has_limit;
    double limit;
    int64_t k;
    int normalize;
    int dense;
    const int64_t *tokens;
    int64_t first, last;
    double *y;
    int32_t *sel_out;
    double *w_out;
    int status;
} moe_job;

/* One expert's feed-forward for one token ([MOE] Inputs fc1..fc3, bias rows). */
static void moe_expert(const moe_job *job, const float *xt, int64_t e, double *h1,
                       double *h3, double *a, double *o)
{
    const int64_t H = job->H, I = job->I;
    const int fused = job->act == MOE_ACT_SWIGLU && job->fusion != 0;
    const int64_t rows1 = fused ? 2 * I : I;
    const int uses_fc3 = job->w3 != NULL &&
                         ((job->act == MOE_ACT_SWIGLU && job->fusion == 0) ||
                          job->act == MOE_ACT_SILU);
    for (int64_t n = 0; n < rows1; ++n) {
        const float *row = job->w1 + (e * rows1 + n) * H;
        double acc = 0.0;
        for (int64_t j = 0; j < H; ++j)
            acc += (double)xt[j] * (double)row[j];
        if (job->b1)
            acc += (double)job->b1[e * rows1 + n];
        h1[n] = acc;
    }
    if (uses_fc3) {
        for (int64_t n = 0; n < I; ++n) {
            const float *row = job->w3 + (e * I + n) * H;
            double acc = 0.0;
            for (int64_t j = 0; j < H; ++j)
                acc += (double)xt[j] * (double)row[j];
            if (job->b3)
                acc += (double)job->b3[e * I + n];
            h3[n] = acc;
        }
    }
    oracle_moe_activation(h1, uses_fc3 ? h3 : NULL, I, job->act, job->fusion, job->alpha,
                          job->beta, job->has_limit, job->limit, a);
    for (int64_t d = 0; d < H; ++d) {
        const float *row = job->w2 + (e * H + d) * I;
        double acc = 0.0;
        for (int64_t j = 0; j < I; ++j)
            acc += a[j] * (double)row[j];
        if (job->b2)
            acc += (double)job->b2[e * H + d];
        o[d] = acc;
    }
}

static void *moe_worker(void *arg)
{
    moe_job *job = (moe_job *)arg;
    const int64_t H = job->H, I = job->I, E = job->E, k = job->k;
    double *h1 = (double *)malloc((size_t)(2 * I + 1) * sizeof(double));
    double *h3 = (double *)malloc((size_t)(I + 1) * sizeof(double));
    double *a = (double *)malloc((size_t)(I + 1) * sizeof(double));
    double *o = (double *)malloc((size_t)(H + 1) * sizeof(double));
    int32_t *sel = (int32_t *)malloc((size_t)k * sizeof(int32_t));
    double *w = (double *)malloc((size_t)k * sizeof(double));
    if (!h1 || !h3 || !a || !o || !sel || !w) {
        job->status = MOE_ORACLE_NO_MEMORY;
        goto done;
    }
    for (int64_t r = job->first; r < job->last; ++r) {
        const int64_t t = job->tokens[r];
        const float *xt = job->x + t * H;
        double *yt = job->y + r * H;
        int st = oracle_moe_route(job->logits + t * E, E, k, job->normalize, sel, w);
        if (st != MOE_ORACLE_OK) {
            job->status = st;
            goto done;
        }
        for (int64_t i = 0; i < k; ++i) {
            if (job->sel_out)
                job->sel_out[r * k + i] = sel[i];
            if (job->w_out)
                job->w_out[r * k + i] = w[i];
        }
        for (int64_t d = 0; d < H; ++d)
            yt[d] = 0.0;
        if (!job->dense) {
            for (int64_t i = 0; i < k; ++i) {
                moe_expert(job, xt, sel[i], h1, h3, a, o);
                for (int64_t d = 0; d < H; ++d)
                    yt[d] += w[i] * o[d];
            }
        } else {
            /* Brute force: every expert, weight 0 unless selected. */
            for (int64_t e = 0; e < E; ++e) {
                double we = 0.0;
                for (int64_t i = 0; i < k; ++i)
                    if (sel[i] == e)
                        we = w[i];
                moe_expert(job, xt, e, h1, h3, a, o);
                for (int64_t d = 0; d < H; ++d)
                    yt[d] += we * o[d];
            }
        }
    }
done:
    free(h1);
    free(h3);
    free(a);
    free(o);
    free(sel);
    free(w);
    return NULL;
}

/*
 * The float MoE layer for the listed tokens ([MOE] Description, Inputs,
 * Attributes).  x [T,H]; logits [T,E]; w1 [E, fusion*I, H]; b1 [E, fusion*I]
 * or NULL; w2 [E, H, I]; b2 [E, H] or NULL; w3 [E, I, H] or NULL; b3 [E, I] or
 * NULL.  fusion is 2 rows per intermediate unit for SwiGLU with
 * swiglu_fusion 1 or 2, else 1.  SwiGLU with swiglu_fusion 0 needs w3.
 * tokens: ntok token ids; y [ntok,H]; sel_out / w_out (nullable) [ntok,k].
 */
int oracle_moe(const float *x, int64_t H, const float *logits, int64_t E,
               const float *w1, const float *b1, const float *w2, const float *b2,
               const float *w3, const float *b3, int64_t I, int act, int fusion,
               double alpha, double beta, int has_limit, double limit, int64_t k,
               int normalize, const int64_t *tokens, int64_t ntok, int dense, double *y,
               int32_t *sel_out, double *w_out, int nthreads)
{
    if (act < MOE_ACT_RELU || act > MOE_ACT_IDENTITY || fusion < 0 || fusion > 2)
        return MOE_ORACLE_BAD_ARG;
    if (act == MOE_ACT_SWIGLU && fusion == 0 && w3 == NULL)
        return MOE_ORACLE_BAD_ARG;
    if (k < 1 || k > E)
        return MOE_ORACLE_BAD_ARG;
    if (ntok <= 0)
        return MOE_ORACLE_OK;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > ntok)
        nthreads = (int)ntok;
    moe_job *jobs = (moe_job *)calloc((size_t)nthreads, sizeof(moe_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return MOE_ORACLE_NO_MEMORY;
    }
    for (int t = 0; t < nthreads; ++t) {
        moe_job *j = &jobs[t];
        j->x = x; j->H = H; j->logits = logits; j->E = E;
        j->w1 = w1; j->b1 = b1; j->w2 = w2; j->b2 = b2; j->w3 = w3; j->b3 = b3;
        j->I = I; j->act = act; j->fusion = fusion; j->alpha = alpha; j->beta = beta;
        j->has_limit = has_limit; j->limit = limit; j->k = k; j->normalize = normalize;
        j->dense = dense; j->tokens = tokens;
        j->first = ntok * t / nthreads;
        j->last = ntok * (t + 1) / nthreads;
        j->y = y; j->sel_out = sel_out; j->w_out = w_out;
        j->status = MOE_ORACLE_OK;
    }
    int started = 0;
    if (nthreads > 1)
        for (int t = 0; t < nthreads; ++t) {
            if (pthread_create(&tids[t], NULL, moe_worker, &jobs[t]) != 0)
                break;
            ++started;
        }
    for (int t = started; t < nthreads; ++t)
        moe_worker(&jobs[t]);
    for (int t = 0; t < started; ++t)
        pthread_join(tids[t], NULL);
    int status = MOE_ORACLE_OK;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status != MOE_ORACLE_OK)
            status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}
