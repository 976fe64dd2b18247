/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the selected-token logprob.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The
 * product (the CUDA library under invariant_token_logprob_gb300/) never calls
 * it and shares no code, header, table or helper with it.
 *
 * What it follows (pages cited by title and section):
 *   [RLK]  "大模型强化学习后训练：如何通过 RL-Kernel 彻底消除训推 LogP 偏差"
 *          (RL-Kernel blog), §一 (importance ratio, worked example),
 *          §四 (five reduction classes; "Linear LogP" normalises over the whole
 *          vocabulary; LogSumExp and its max-shifted stable form; blockwise
 *          merge of per-block max m_j and exp-sum s_j).
 *   [VLC]  "Finish RL Training Faster: Bitwise-Consistent, High-Performance,
 *          Agent-Driven" (vLLM consistency blog summary), section
 *          "训练-推理一致性的多维判定标准", paragraph "diff = 0 的数学定义"
 *          (max / mean / std of |p_rollout - p_train| and the k3 KL r-1-log r).
 *
 * Readings where the pages are silent or garbled (each also listed in the
 * design notes):
 *   - The LSE formula itself is lost in the extraction of [RLK] §四; the
 *     surviving sentence gives the stable form m + log sum exp(x_i - m), which
 *     is what logprob_row() computes (two passes: max, then exp-sum).
 *   - Temperature is not on the pages: z = (h . W_v) * inv_temp, one multiply by
 *     the fp32 value of inv_temp, after the full dot product.
 *   - Argmax ties go to the lowest vocabulary index.
 *   - A target outside [0, V) is an ignored row: logp = 0.
 *   - k3 uses r = exp(p_train - p_rollout) (probability ratio from the two
 *     log-probabilities), computed as expm1(d) - d with d = a - b, a = train.
 *   - std is the population standard deviation (divide by n_valid).
 *
 * Arithmetic: every floating-point step is in IEEE double.  bf16 -> double is
 * exact, each bf16 x bf16 product is exact in double, the dot product is summed
 * sequentially over k = 0..H-1.  Build without -ffast-math and with
 * -ffp-contract=off so both host architectures give the same bits.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake; the
 * test suite builds each mutant to show that some pin fails for it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* z[v] = (sum_k h[k] * W[v,k]) * inv_temp for v = 0..V-1 ([RLK] §四: the
 * Linear LogP class scores the whole vocabulary).  hd holds h as doubles. */
static void logits_row(const double *hd, const uint16_t *W, int64_t H,
                       int64_t V, double inv_temp, double *z)
{
    for (int64_t v = 0; v < V; ++v) {
        const uint16_t *w = W + v * H;
        double acc = 0.0;
#if ORACLE_MUTANT == 1
        for (int64_t k = 0; k + 1 < H; ++k)      /* mutant: drops the last term */
#else
        for (int64_t k = 0; k < H; ++k)
#endif
            acc += hd[k] * bf16_to_double(w[k]);
#if ORACLE_MUTANT == 2
        z[v] = acc / inv_temp;                   /* mutant: divides by inv_temp */
#else
        z[v] = acc * inv_temp;
#endif
    }
}

typedef struct {
    double logp, lse, zmax, ztgt, top2gap;
    int64_t argmax;
} row_result;

/* One row: max, lowest-index argmax, two-pass LSE, selected-token logp. */
static row_result logprob_row(const double *z, int64_t V, int32_t target)
{
    row_result r;
    double m = z[0];
    int64_t a = 0;
    for (int64_t v = 1; v < V; ++v) {
#if ORACLE_MUTANT == 3
        if (z[v] >= m) { m = z[v]; a = v; }      /* mutant: highest index wins ties */
#else
        if (z[v] > m) { m = z[v]; a = v; }
#endif
    }
    /* second pass: sum of exp(z - m); the stable form of [RLK] §四 */
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v)
        s += exp(z[v] - m);
#if ORACLE_MUTANT == 4
    double lse = log(s);                         /* mutant: forgets to add m back */
#else
    double lse = m + log(s);
#endif
    double second = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if (v != a && z[v] > second) second = z[v];
    r.zmax = m;
    r.argmax = a;
    r.lse = lse;
    r.top2gap = m - second;                      /* +inf when V == 1 */
    if (target >= 0 && (int64_t)target < V) {
        r.ztgt = z[target];
#if ORACLE_MUTANT == 5
        r.logp = lse - z[target];                /* mutant: sign flipped */
#else
        r.logp = z[target] - lse;
#endif
    } else {
        r.ztgt = 0.0;
        r.logp = 0.0;                            /* ignored row */
    }
    return r;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Selected-token logprob for the rows listed in `rows` (or all T rows when
 * rows == NULL; then n_rows must equal T).  h is [T,H] bf16 bits, W is [V,H]
 * bf16 bits, both row-major.  Outputs are indexed by position in `rows`.
 * Any output pointer may be NULL.  Returns 0, or -1 on bad arguments / memory.
 */
int oracle_logprob(const uint16_t *h, const uint16_t *W, const int32_t *targets,
                   int64_t T, int64_t H, int64_t V, float inv_temp,
                   const int64_t *rows, int64_t n_rows,
                   double *out_logp, double *out_lse, int64_t *out_argmax,
                   double *out_top2gap, double *out_ztgt, double *out_zmax)
{
    if (!h || !W || !targets || T < 0 || H <= 0 || V <= 0 || n_rows < 0)
        return -1;
    if (!rows && n_rows != T)
        return -1;
    int bad = 0;
    const double it = (double)inv_temp;
#pragma omp parallel
    {
        double *z = (double *)malloc((size_t)V * sizeof(double));
        double *hd = (double *)malloc((size_t)H * sizeof(double));
        if (!z || !hd) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (!z || !hd) continue;
            int64_t t = rows ? rows[i] : i;
            if (t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int64_t k = 0; k < H; ++k)
                hd[k] = bf16_to_double(h[t * H + k]);
            logits_row(hd, W, H, V, it, z);
            row_result r = logprob_row(z, V, targets[t]);
            if (out_logp) out_logp[i] = r.logp;
            if (out_lse) out_lse[i] = r.lse;
            if (out_argmax) out_argmax[i] = r.argmax;
            if (out_top2gap) out_top2gap[i] = r.top2gap;
            if (out_ztgt) out_ztgt[i] = r.ztgt;
            if (out_zmax) out_zmax[i] = r.zmax;
        }
        free(z);
        free(hd);
    }
    return bad ? -1 : 0;
}

/*
 * Per-block statistics of [RLK] §四 ("each block keeps a local max m_j and a
 * local exp-sum s_j"): the vocabulary is cut into consecutive blocks of `bn`
 * columns; block j covers columns [j*bn, min((j+1)*bn, V)).  For each listed
 * row and block: m = max z, a = lowest index attaining m, s = sum exp(z - m)
 * in ascending column order, zt = z[target] if the target lies in the block
 * else 0.  Outputs are [n_rows][n_blocks] with n_blocks = ceil(V / bn).
 */
int oracle_block_stats(const uint16_t *h, const uint16_t *W, const int32_t *targets,
                       int64_t T, int64_t H, int64_t V, float inv_temp, int64_t bn,
                       const int64_t *rows, int64_t n_rows,
                       double *out_m, double *out_s, int64_t *out_a, double *out_zt)
{
    if (!h || !W || !targets || T < 0 || H <= 0 || V <= 0 || bn <= 0 || n_rows < 0)
        return -1;
    if (!rows && n_rows != T)
        return -1;
    const int64_t nb = (V + bn - 1) / bn;
    const double it = (double)inv_temp;
    int bad = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc((size_t)V * sizeof(double));
        double *hd = (double *)malloc((size_t)H * sizeof(double));
        if (!z || !hd) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (!z || !hd) continue;
            int64_t t = rows ? rows[i] : i;
            if (t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int64_t k = 0; k < H; ++k)
                hd[k] = bf16_to_double(h[t * H + k]);
            logits_row(hd, W, H, V, it, z);
            for (int64_t j = 0; j < nb; ++j) {
                int64_t lo = j * bn, hi = lo + bn < V ? lo + bn : V;
                double m = z[lo];
                int64_t a = lo;
                for (int64_t v = lo + 1; v < hi; ++v)
                    if (z[v] > m) { m = z[v]; a = v; }
                double s = 0.0;
                for (int64_t v = lo; v < hi; ++v)
                    s += exp(z[v] - m);
                int32_t tg = targets[t];
                double zt = (tg >= lo && tg < hi) ? z[tg] : 0.0;
                if (out_m) out_m[i * nb + j] = m;
                if (out_s) out_s[i * nb + j] = s;
                if (out_a) out_a[i * nb + j] = a;
                if (out_zt) out_zt[i * nb + j] = zt;
            }
        }
        free(z);
        free(hd);
    }
    return bad ? -1 : 0;
}

/*
 * Merge of per-block statistics ([RLK] §四 blockwise merge; §七 LogP: local
 * statistics merged over vocabulary tiles).  The exact-arithmetic definition:
 * M = max_j m_j, A = lowest a_j among blocks with m_j == M,
 * S = sum_j s_j * exp(m_j - M), LSE = M + log S; logp = zt - LSE where zt is
 * the target entry of the block holding the target.  Inputs are fp32 (the
 * precision the partials are stored in), promoted to double; the sum runs over
 * blocks in ascending order.  Blocks with m_j = -inf contribute nothing.
 * Layout [n_rows][n_blocks]; targets are per row; bn is the block width used
 * to find the target's block.  Returns 0 or -1.
 */
int oracle_merge_blocks(const float *m, const float *s, const int32_t *a,
                        const float *zt, const int32_t *targets,
                        int64_t n_rows, int64_t n_blocks, int64_t V, int64_t bn,
                        double *out_lse, double *out_logp, int64_t *out_argmax)
{
    if (!m || !s || !a || n_rows < 0 || n_blocks <= 0 || V <= 0 || bn <= 0)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        const float *mr = m + r * n_blocks, *sr = s + r * n_blocks;
        const int32_t *ar = a + r * n_blocks;
        double M = -INFINITY;
        int64_t A = INT64_MAX;
        for (int64_t j = 0; j < n_blocks; ++j) {
            double mj = (double)mr[j];
            if (mj > M) { M = mj; A = ar[j]; }
            else if (mj == M && ar[j] < A) A = ar[j];
        }
        double S = 0.0;
        for (int64_t j = 0; j < n_blocks; ++j) {
            double mj = (double)mr[j];
            if (mj == -INFINITY) continue;
            S += (double)sr[j] * exp(mj - M);
        }
        double lse = M + log(S);
        if (out_lse) out_lse[r] = lse;
        if (out_argmax) out_argmax[r] = A;
        if (out_logp) {
            double lp = 0.0;
            if (targets && zt) {
                int32_t tg = targets[r];
                if (tg >= 0 && (int64_t)tg < V)
                    lp = (double)zt[r * n_blocks + tg / bn] - lse;
            }
            out_logp[r] = lp;
        }
    }
    return 0;
}

/*
 * Acceptance statistics of [VLC] "diff = 0 的数学定义" over valid tokens
 * (mask == NULL: all valid; else mask[i] != 0 is valid).  a = train logp,
 * b = rollout logp, d = a - b in double.
 *   out[0] max |d|          out[1] mean |d|        out[2] population std of |d|
 *   out[3] mean k3 = expm1(d) - d                  out[4] sum d
 *   out[5] n_valid          out[6] number of valid i whose fp32 bit patterns differ
 *   out[7] lowest valid index with differing bits, or -1
 * With n_valid == 0 every statistic is 0 and out[7] = -1.  Returns 0 or -1.
 */
int oracle_consistency_stats(const float *a, const float *b, const int8_t *mask,
                             int64_t n, double *out)
{
    if (!out || n < 0 || (n > 0 && (!a || !b)))
        return -1;
    double nv = 0.0, mx = 0.0, sabs = 0.0, sd = 0.0, sk3 = 0.0, nmis = 0.0;
    int64_t first = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (mask && mask[i] == 0) continue;
#if ORACLE_MUTANT == 6
        double d = (double)b[i] - (double)a[i];  /* mutant: direction swapped */
#else
        double d = (double)a[i] - (double)b[i];
#endif
        double ad = fabs(d);
        nv += 1.0;
        if (ad > mx) mx = ad;
        sabs += ad;
        sd += d;
        sk3 += expm1(d) - d;
        uint32_t ua, ub;
        memcpy(&ua, &a[i], 4);
        memcpy(&ub, &b[i], 4);
        if (ua != ub) {
            nmis += 1.0;
            if (first < 0) first = i;
        }
    }
    double mean = nv > 0 ? sabs / nv : 0.0;
    double ss = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (mask && mask[i] == 0) continue;
        double ad = fabs((double)a[i] - (double)b[i]);
        ss += (ad - mean) * (ad - mean);
    }
#if ORACLE_MUTANT == 7
    double var = nv > 1 ? ss / (nv - 1.0) : 0.0; /* mutant: sample variance */
#else
    double var = nv > 0 ? ss / nv : 0.0;
#endif
    out[0] = mx;
    out[1] = mean;
    out[2] = sqrt(var);
    out[3] = nv > 0 ? sk3 / nv : 0.0;
    out[4] = sd;
    out[5] = nv;
    out[6] = nmis;
    out[7] = (double)first;
    return 0;
}


/* ------------------------------------------------------------------------
 * Backward of the selected-token logprob (the training half of the method:
 * "Finish RL Training Faster ...", section "核心设计范式：推理算子定义数值基准，
 * 训练仅挂接反向求导" -- the forward values come from the inference kernel, the
 * training side supplies the derivative through a custom autograd function).
 * With p = softmax(z) and upstream gradient g[t] of logp[t]:
 *   dz[t,v] = g[t] * ([v == target[t]] - p[t,v])      (0 for an ignored row)
 *   dh[t,k] = inv_temp * sum_v dz[t,v] W[v,k]
 *   dW[v,k] = inv_temp * sum_t dz[t,v] h[t,k]
 * (z = inv_temp * h.W^T, so dlogp/dh and dlogp/dW carry one inv_temp factor.)
 * Computed by definition in fp64: logits and LSE as in oracle_logprob, p by
 * exp(z - LSE), sums in index order.  Small problems only (T*V*H work).
 * Outputs: dz [T][V], dh [T][H], dW [V][H] (any may be NULL).
 */
static void logits_all(const double *hd, const double *Wd, int64_t H, int64_t V,
                       double it, double *z)
{
    for (int64_t v = 0; v < V; ++v) {
        double acc = 0.0;
        for (int64_t k = 0; k < H; ++k)
            acc += hd[k] * Wd[v * H + k];
        z[v] = acc * it;
    }
}

static int backward_core(const double *hd, const double *Wd, const int32_t *targets,
                         const double *grad, int64_t T, int64_t H, int64_t V, double it,
                         double *out_dz, double *out_dh, double *out_dW)
{
    double *z = (double *)malloc((size_t)V * sizeof(double));
    double *dz = (double *)malloc((size_t)T * (size_t)V * sizeof(double));
    if (!z || !dz) { free(z); free(dz); return -1; }
    for (int64_t t = 0; t < T; ++t) {
        logits_all(hd + t * H, Wd, H, V, it, z);
        row_result r = logprob_row(z, V, targets[t]);
        int32_t tg = targets[t];
        int valid = tg >= 0 && (int64_t)tg < V;
        for (int64_t v = 0; v < V; ++v) {
#if ORACLE_MUTANT == 9
            double p = exp(z[v] - r.zmax);       /* mutant: unnormalised softmax */
#else
            double p = exp(z[v] - r.lse);
#endif
            dz[t * V + v] = valid ? grad[t] * ((v == tg ? 1.0 : 0.0) - p) : 0.0;
        }
    }
    if (out_dz) memcpy(out_dz, dz, (size_t)T * (size_t)V * sizeof(double));
    if (out_dh)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t k = 0; k < H; ++k) {
                double acc = 0.0;
                for (int64_t v = 0; v < V; ++v)
                    acc += dz[t * V + v] * Wd[v * H + k];
#if ORACLE_MUTANT == 8
                out_dh[t * H + k] = acc;         /* mutant: drops the inv_temp factor */
#else
                out_dh[t * H + k] = it * acc;
#endif
            }
    if (out_dW)
        for (int64_t v = 0; v < V; ++v)
            for (int64_t k = 0; k < H; ++k) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t)
                    acc += dz[t * V + v] * hd[t * H + k];
                out_dW[v * H + k] = it * acc;
            }
    free(z);
    free(dz);
    return 0;
}

int oracle_logprob_backward(const uint16_t *h, const uint16_t *W, const int32_t *targets,
                            const double *grad, int64_t T, int64_t H, int64_t V, float inv_temp,
                            double *out_dz, double *out_dh, double *out_dW)
{
    if (!h || !W || !targets || !grad || T < 1 || H < 1 || V < 1)
        return -1;
    double *hd = (double *)malloc((size_t)T * (size_t)H * sizeof(double));
    double *Wd = (double *)malloc((size_t)V * (size_t)H * sizeof(double));
    if (!hd || !Wd) { free(hd); free(Wd); return -1; }
    for (int64_t i = 0; i < T * H; ++i) hd[i] = bf16_to_double(h[i]);
    for (int64_t i = 0; i < V * H; ++i) Wd[i] = bf16_to_double(W[i]);
    int rc = backward_core(hd, Wd, targets, grad, T, H, V, (double)inv_temp, out_dz, out_dh,
                           out_dW);
    free(hd);
    free(Wd);
    return rc;
}

/* Forward on fp64 inputs (used to pin the backward by finite differences:
 * the oracle's own logp, perturbed input by input). */
int oracle_logprob_f64(const double *h, const double *W, const int32_t *targets, int64_t T,
                       int64_t H, int64_t V, double inv_temp, double *out_logp, double *out_lse)
{
    if (!h || !W || !targets || T < 1 || H < 1 || V < 1)
        return -1;
    double *z = (double *)malloc((size_t)V * sizeof(double));
    if (!z) return -1;
    for (int64_t t = 0; t < T; ++t) {
        logits_all(h + t * H, W, H, V, inv_temp, z);
        row_result r = logprob_row(z, V, targets[t]);
        if (out_logp) out_logp[t] = r.logp;
        if (out_lse) out_lse[t] = r.lse;
    }
    free(z);
    return 0;
}


/*
 * Per-token entropy of the softmax over the whole vocabulary, -sum_v p_v log p_v
 * with p = softmax(z) -- the actor-entropy signal the consistency blog reports
 * beside the rewards ("Finish RL Training Faster ...", Nemotron results: actor
 * entropy 0.05 vs 2.6).  By definition in fp64: logits and two-pass LSE as in
 * oracle_logprob, then -sum_v exp(z_v - LSE) * (z_v - LSE) in index order.
 */
int oracle_entropy(const uint16_t *h, const uint16_t *W, int64_t T, int64_t H, int64_t V,
                   float inv_temp, const int64_t *rows, int64_t n_rows, double *out_entropy)
{
    if (!h || !W || !out_entropy || T < 0 || H <= 0 || V <= 0 || n_rows < 0)
        return -1;
    if (!rows && n_rows != T)
        return -1;
    int bad = 0;
    const double it = (double)inv_temp;
#pragma omp parallel
    {
        double *z = (double *)malloc((size_t)V * sizeof(double));
        double *hd = (double *)malloc((size_t)H * sizeof(double));
        if (!z || !hd) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (!z || !hd) continue;
            int64_t t = rows ? rows[i] : i;
            if (t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int64_t k = 0; k < H; ++k)
                hd[k] = bf16_to_double(h[t * H + k]);
            logits_row(hd, W, H, V, it, z);
            row_result r = logprob_row(z, V, -1);
            double e = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                double lp = z[v] - r.lse;
#if ORACLE_MUTANT == 10
                e -= exp(lp) * z[v];                 /* mutant: forgets the LSE shift */
#else
                e -= exp(lp) * lp;
#endif
            }
            out_entropy[i] = e;
        }
        free(z);
        free(hd);
    }
    return bad ? -1 : 0;
}


/* ------------------------------------------------------------------------
 * FP8 (W8A8) variant.  The consistency blog runs its dense layers as
 * block-FP8 W8A8 GEMMs with round-to-nearest-even quantisation and one fixed
 * accumulation order per output ("Finish RL Training Faster ...", sections on
 * the dense GEMM and the expert GEMM: RNE quantisation, fixed accumulation
 * tree).  Reading taken here for the LM head: one fp32 scale per row of h
 * (per token) and per row of W (per vocabulary entry), s = amax / 448 (s = 1
 * for an all-zero row), code = RNE-to-e4m3(x / s) with the division in fp32,
 * saturating at +-448.  z = (sum_k qh[k] qW[k]) * s_h * s_W * inv_temp.
 */

/* Value of an e4m3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * no infinities; exponent 15 with mantissa 7 is NaN). */
static double e4m3_value(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m/8 * 2^-6 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round a float to the nearest e4m3 value, ties to an even mantissa,
 * saturating at +-448: by scanning the 127 non-negative finite codes. */
static uint8_t e4m3_rne(float x)
{
    double ax = fabs((double)x);
    uint8_t best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 126; ++c) {
        double d = fabs(e4m3_value((uint8_t)c) - ax);
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) { bd = d; best = (uint8_t)c; }
    }
#if ORACLE_MUTANT == 11
    best = (uint8_t)(ax > e4m3_value(best) && best < 126 ? best + 1 : best); /* mutant: rounds up */
#endif
    if (ax > 448.0) best = 126;                      /* saturate to 448 */
    /* rounding keeps the operand's sign, also when the magnitude rounds to 0 */
    return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/* Quantise rows of a bf16 matrix [rows][H]: codes [rows][H], scales [rows]. */
int oracle_quantize_fp8_rows(const uint16_t *x, int64_t rows, int64_t H, uint8_t *codes,
                             float *scales)
{
    if (!x || !codes || !scales || rows < 0 || H <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < H; ++k) {
            float v = (float)bf16_to_double(x[r * H + k]);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = sc;
        for (int64_t k = 0; k < H; ++k) {
            float v = (float)bf16_to_double(x[r * H + k]);
            codes[r * H + k] = e4m3_rne(v / sc);
        }
    }
    return 0;
}

/* Selected-token logprob from quantised operands, by definition in fp64. */
int oracle_logprob_fp8(const uint8_t *qh, const float *sh, const uint8_t *qw, const float *sw,
                       const int32_t *targets, int64_t T, int64_t H, int64_t V, float inv_temp,
                       const int64_t *rows, int64_t n_rows, double *out_logp, double *out_lse,
                       int64_t *out_argmax, double *out_top2gap)
{
    if (!qh || !sh || !qw || !sw || !targets || T < 0 || H <= 0 || V <= 0 || n_rows < 0)
        return -1;
    if (!rows && n_rows != T) return -1;
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = e4m3_value((uint8_t)c);
    int bad = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc((size_t)V * sizeof(double));
        if (!z) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (!z) continue;
            int64_t t = rows ? rows[i] : i;
            if (t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int64_t v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int64_t k = 0; k < H; ++k)
                    acc += lut[qh[t * H + k]] * lut[qw[v * H + k]];
                z[v] = acc * (double)sh[t] * (double)sw[v] * (double)inv_temp;
            }
            row_result r = logprob_row(z, V, targets[t]);
            if (out_logp) out_logp[i] = r.logp;
            if (out_lse) out_lse[i] = r.lse;
            if (out_argmax) out_argmax[i] = r.argmax;
            if (out_top2gap) out_top2gap[i] = r.top2gap;
        }
        free(z);
    }
    return bad ? -1 : 0;
}


/* ------------------------------------------------------------------------
 * Block-scaled FP8 (W8A8) variant.  The consistency blog's dense layers use
 * block-FP8 weights in DeepGEMM's W8A8 batch-invariant mode ("Finish RL
 * Training Faster ...", section on the dense GEMM: FP8 computation with one
 * fixed reduction order; RNE quantisation).  The page gives no block shape
 * for an LM head; the reading taken is DeepGEMM's: activations in 1 x 128
 * blocks (one token, 128 consecutive k) and weights in 128 x 128 blocks (128
 * vocabulary rows, 128 consecutive k).  Per block s = amax / 448 in fp32
 * (1 for an all-zero block) and code = RNE-to-e4m3(x / s), fp32 division.
 * The logit is the sum over k blocks b of each block's code dot product
 * times both blocks' scales:
 *   z[t][v] = inv_temp * sum_b s_h[t][b] s_W[v / 128][b] sum_{k in b} qh[t][k] qW[v][k]
 */

/* Quantise a bf16 matrix [rows][H] in blocks of block_rows x 128: codes
 * [rows][H], scales [ceil(rows / block_rows)][ceil(H / 128)]. */
int oracle_quantize_fp8_blocks(const uint16_t *x, int64_t rows, int64_t H, int64_t block_rows,
                               uint8_t *codes, float *scales)
{
    if (!x || !codes || !scales || rows < 0 || H <= 0 || block_rows <= 0) return -1;
    const int64_t nkb = (H + 127) / 128, nrb = (rows + block_rows - 1) / block_rows;
#pragma omp parallel for schedule(static)
    for (int64_t rb = 0; rb < nrb; ++rb) {
        const int64_t r0 = rb * block_rows, r1 = r0 + block_rows < rows ? r0 + block_rows : rows;
        for (int64_t b = 0; b < nkb; ++b) {
            const int64_t k0 = b * 128, k1 = k0 + 128 < H ? k0 + 128 : H;
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t k = k0; k < k1; ++k) {
                    float v = (float)bf16_to_double(x[r * H + k]);
                    if (fabsf(v) > amax) amax = fabsf(v);
                }
            float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[rb * nkb + b] = sc;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t k = k0; k < k1; ++k) {
                    float v = (float)bf16_to_double(x[r * H + k]);
                    codes[r * H + k] = e4m3_rne(v / sc);
                }
        }
    }
    return 0;
}

/* Selected-token logprob from block-quantised operands, by definition in fp64:
 * sh [T][ceil(H/128)], sw [ceil(V/128)][ceil(H/128)]. */
int oracle_logprob_fp8_block(const uint8_t *qh, const float *sh, const uint8_t *qw,
                             const float *sw, const int32_t *targets, int64_t T, int64_t H,
                             int64_t V, float inv_temp, const int64_t *rows, int64_t n_rows,
                             double *out_logp, double *out_lse, int64_t *out_argmax,
                             double *out_top2gap)
{
    if (!qh || !sh || !qw || !sw || !targets || T < 0 || H <= 0 || V <= 0 || n_rows < 0)
        return -1;
    if (!rows && n_rows != T) return -1;
    const int64_t nkb = (H + 127) / 128;
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = e4m3_value((uint8_t)c);
    int bad = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc((size_t)V * sizeof(double));
        if (!z) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; ++i) {
            if (!z) continue;
            int64_t t = rows ? rows[i] : i;
            if (t < 0 || t >= T) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int64_t v = 0; v < V; ++v) {
                double acc = 0.0;
                for (int64_t b = 0; b < nkb; ++b) {
                    const int64_t k0 = b * 128, k1 = k0 + 128 < H ? k0 + 128 : H;
                    double part = 0.0;
                    for (int64_t k = k0; k < k1; ++k) part += lut[qh[t * H + k]] * lut[qw[v * H + k]];
#if ORACLE_MUTANT == 12
                    /* mutant: the next W block row's scale (wrapping) */
                    const double swb = (double)sw[((v / 128 + 1) % ((V + 127) / 128)) * nkb + b];
#else
                    const double swb = (double)sw[(v / 128) * nkb + b];
#endif
#if ORACLE_MUTANT == 13
                    const double shb = (double)sh[t * nkb]; /* mutant: block 0's scale for every block */
#else
                    const double shb = (double)sh[t * nkb + b];
#endif
                    acc += shb * swb * part;
                }
                z[v] = acc * (double)inv_temp;
            }
            row_result r = logprob_row(z, V, targets[t]);
            if (out_logp) out_logp[i] = r.logp;
            if (out_lse) out_lse[i] = r.lse;
            if (out_argmax) out_argmax[i] = r.argmax;
            if (out_top2gap) out_top2gap[i] = r.top2gap;
        }
        free(z);
    }
    return bad ? -1 : 0;
}
