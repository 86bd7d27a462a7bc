/*
 * tw_oracle.c -- fp64 CPU oracle for TokenWeave's reduce + residual add +
 * RMSNorm, in both the traditional and the reordered order.
 *
 * TEST INFRASTRUCTURE ONLY: the product library never calls, links or loads
 * this file.  It is plain, slow and written to be checked by eye against the
 * pages it follows:
 *
 *   "TokenWeave 策略详解：以大模型推理为例" (nanhubrain.csdn.net)
 *     §1 背景        output = RMSNorm(residual + allreduce_output) * weight;
 *                    RMSNorm is per token, over all hidden features.
 *     §2 核心思想    traditional order AllReduce -> residual add -> RMSNorm;
 *                    reordered ReduceScatter -> residual add -> RMSNorm ->
 *                    AllGather, with the scatter split on token boundaries.
 *     §3.2-3.4      tokens split evenly over the GPUs; each GPU reads only its
 *                    token slice of the replicated residual; the gather makes
 *                    every GPU hold the full normalised tensor, equal to the
 *                    traditional output.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *   - eps sits inside the square root: rms = sqrt(mean(x^2) + eps), mean over
 *     all H features.
 *   - the weight multiplies the normalised value, y = (x / rms) * w, with no
 *     bias and no (1 + w) offset.
 *   - the AllReduce / ReduceScatter sum adds the ranks in rank order starting
 *     from 0.0, and the residual is added after the sum.
 *   - an uneven token split uses floor bounds floor(r*n/N), so a rank may own
 *     no token.
 *   - residual_out receives x = sum + residual for the rows in [t0, t1).
 *
 * Arithmetic is IEEE fp64 as written: build with -ffp-contract=off so no
 * multiply-add is fused, which keeps x86 and Arm results identical.
 */
#include "tw_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads of the token loops: 0 = the OpenMP runtime's default.  Passed to
   every loop explicitly, so it holds whichever OpenMP runtime the process
   resolved the loops against. */
static int g_threads = 0;

static int bad_args(const double* const* partials, int n_parts,
                    const double* residual, const double* weight,
                    double* const* out, int n_out, double* residual_out,
                    int64_t T, int64_t H, double eps, int64_t t0, int64_t t1)
{
    if (!partials || !residual || !weight || !out || !residual_out) return 1;
    if (n_parts < 1 || n_out < 1) return 1;
    if (T < 0 || H < 1 || t0 < 0 || t0 > t1 || t1 > T) return 1;
    if (!(eps >= 0.0) || isinf(eps)) return 1;
    for (int r = 0; r < n_parts; ++r)
        if (!partials[r]) return 1;
    for (int k = 0; k < n_out; ++k)
        if (!out[k]) return 1;
    return 0;
}

/* RMSNorm of one token (§1 背景): y[h] = x[h] / sqrt(mean_h(x^2) + eps) * w[h]. */
static void rmsnorm_token(const double* x, const double* w, int64_t H,
                          double eps, double* y)
{
    double sum_sq = 0.0;
    for (int64_t h = 0; h < H; ++h)
        sum_sq += x[h] * x[h];
    const double rms = sqrt(sum_sq / (double)H + eps);
    for (int64_t h = 0; h < H; ++h)
        y[h] = (x[h] / rms) * w[h];
}

int tw_oracle_token_slice(int64_t n_tokens, int n_ranks, int r,
                          int64_t* first, int64_t* last)
{
    if (n_tokens < 0 || n_ranks < 1 || r < 0 || r >= n_ranks || !first || !last)
        return -1;
    /* §3.2: tokens are handed out evenly; floor bounds for the uneven case. */
    *first = (n_tokens * (int64_t)r) / n_ranks;
    *last = (n_tokens * (int64_t)(r + 1)) / n_ranks;
    return 0;
}

int tw_oracle_traditional(const double* const* partials, int n_parts,
                          const double* residual, const double* weight,
                          double* const* out, int n_out, double* residual_out,
                          int64_t T, int64_t H, double eps,
                          int64_t t0, int64_t t1)
{
    if (bad_args(partials, n_parts, residual, weight, out, n_out, residual_out,
                 T, H, eps, t0, t1))
        return -1;
    const int64_t n_rows = t1 - t0;
    if (n_rows == 0) return 0;

    /* Step 1, AllReduce(sum): every rank receives sum_r partials[r] for all
     * tokens of the range (§1: the reduced tensor is [T, H] on every GPU). */
    double* reduced = (double*)malloc((size_t)(n_rows * H) * sizeof(double));
    if (!reduced) return -1;
#pragma omp parallel for schedule(static) num_threads(tw_oracle_threads())
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t t = t0 + i;
        for (int64_t h = 0; h < H; ++h) {
            double s = 0.0;
            for (int r = 0; r < n_parts; ++r)
                s += partials[r][t * H + h];
            reduced[i * H + h] = s;
        }
    }

    /* Step 2, on each rank k (the redundant N-fold work of §1): residual add,
     * then RMSNorm of every token, into that rank's own destination. */
    for (int k = 0; k < n_out; ++k) {
#pragma omp parallel for schedule(static) num_threads(tw_oracle_threads())
        for (int64_t i = 0; i < n_rows; ++i) {
            const int64_t t = t0 + i;
            double* x = (double*)malloc((size_t)H * sizeof(double));
            for (int64_t h = 0; h < H; ++h)
                x[h] = reduced[i * H + h] + residual[t * H + h];
            rmsnorm_token(x, weight, H, eps, out[k] + t * H);
            if (k == 0)
                memcpy(residual_out + t * H, x, (size_t)H * sizeof(double));
            free(x);
        }
    }
    free(reduced);
    return 0;
}

int tw_oracle_reordered(const double* const* partials, int n_parts,
                        const double* residual, const double* weight,
                        double* const* out, int n_out, double* residual_out,
                        int64_t T, int64_t H, double eps,
                        int64_t t0, int64_t t1)
{
    if (bad_args(partials, n_parts, residual, weight, out, n_out, residual_out,
                 T, H, eps, t0, t1))
        return -1;
    const int64_t n_rows = t1 - t0;
    if (n_rows == 0) return 0;

    /* One simulated rank per partial (the tensor-parallel degree N). */
    for (int r = 0; r < n_parts; ++r) {
        int64_t first, last;
        tw_oracle_token_slice(n_rows, n_parts, r, &first, &last);
        const int64_t n_mine = last - first;
        if (n_mine == 0) continue;
        double* mine = (double*)malloc((size_t)(n_mine * H) * sizeof(double));
        if (!mine) return -1;

        /* ReduceScatter on token boundaries (§3.2): rank r receives the
         * sum over all ranks of its own token slice, full feature width. */
#pragma omp parallel for schedule(static) num_threads(tw_oracle_threads())
        for (int64_t i = 0; i < n_mine; ++i) {
            const int64_t t = t0 + first + i;
            for (int64_t h = 0; h < H; ++h) {
                double s = 0.0;
                for (int q = 0; q < n_parts; ++q)
                    s += partials[q][t * H + h];
                mine[i * H + h] = s;
            }
        }

        /* Residual add on the slice only, then RMSNorm (§3.3).  The
         * normalised slice overwrites the reduced one in place per token. */
#pragma omp parallel for schedule(static) num_threads(tw_oracle_threads())
        for (int64_t i = 0; i < n_mine; ++i) {
            const int64_t t = t0 + first + i;
            double* row = mine + i * H;
            for (int64_t h = 0; h < H; ++h)
                row[h] = row[h] + residual[t * H + h];
            memcpy(residual_out + t * H, row, (size_t)H * sizeof(double));
            double* y = (double*)malloc((size_t)H * sizeof(double));
            rmsnorm_token(row, weight, H, eps, y);
            memcpy(row, y, (size_t)H * sizeof(double));
            free(y);
        }

        /* AllGather (§3.4): every destination receives rank r's slice at the
         * same absolute rows. */
        for (int k = 0; k < n_out; ++k)
            memcpy(out[k] + (t0 + first) * H, mine,
                   (size_t)(n_mine * H) * sizeof(double));
        free(mine);
    }
    return 0;
}

int tw_oracle_threads(void)
{
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

void tw_oracle_set_threads(int n)
{
    if (n >= 1)
        g_threads = n;
}
