/*
 * oracle.c -- plain CPU statement of the bitwise-reproducible int8 QAT linear
 * layer (forward, backward) and of the fixed-order gradient reduction.
 *
 * TEST INFRASTRUCTURE ONLY: see oracle.h for who may load it, for the
 * arithmetic model and for the canonical reduction order.  Nothing here is
 * blocked, fused or reordered beyond what those definitions state; loops over
 * independent output elements may run on several threads, which changes no
 * bit because every element's own sequence of operations is fixed.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math
 *           -fexcess-precision=standard [-fopenmp] -fPIC -shared oracle.c -lm
 */
#include "oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Elementary operations.  [P4] "How it works": subnormals are flushed on     */
/* every backend; a*b+c is never contracted.  Operands are flushed first      */
/* (denormals-are-zero), the IEEE result is formed by the host's binary32     */
/* unit in its default round-to-nearest-even mode, then a subnormal result is */
/* flushed.                                                                   */
/* ------------------------------------------------------------------------ */

float oracle_flush(float x)
{
    if (x != 0.0f && fabsf(x) < FLT_MIN)
        return copysignf(0.0f, x);
    return x;
}

float oracle_add(float a, float b)
{
    float r = oracle_flush(a) + oracle_flush(b);
    return oracle_flush(r);
}

float oracle_mul(float a, float b)
{
    float r = oracle_flush(a) * oracle_flush(b);
    return oracle_flush(r);
}

float oracle_div(float a, float b)
{
    float r = oracle_flush(a) / oracle_flush(b);
    return oracle_flush(r);
}

float oracle_sqrt(float a)
{
    float r = sqrtf(oracle_flush(a)); /* IEEE 754 requires correct rounding */
    return oracle_flush(r);
}

float oracle_i2f(int64_t v)
{
    return (float)v; /* round to nearest even in the default mode */
}

/* [P4] "How to use": int8 weights and activations.  The quantiser is
 * q = clamp(round_half_even(x (/) s), -qmax, qmax) with q_max = 127, so -128
 * is never produced.  Special cases: a zero (or flushed) scale maps every
 * element to 0; a NaN quotient maps to 0; +-Inf clamps to +-qmax. */
int oracle_quant_one(float x, float s, int qmax)
{
    float sf = oracle_flush(s);
    if (sf == 0.0f)
        return 0;
    float v = oracle_div(x, sf);
    if (v != v)
        return 0;
    float r = rintf(v); /* integral value, ties to even (default mode) */
    if (r > (float)qmax)
        return qmax;
    if (r < -(float)qmax)
        return -qmax;
    return (int)r;
}

/* ------------------------------------------------------------------------ */
/* Canonical sum: chunks of 64 summed left to right (seeded with the chunk's  */
/* first term), chunk partials combined by the stride-doubling pairwise tree. */
/* ------------------------------------------------------------------------ */

float oracle_canon_sum(const float* p, int64_t L)
{
    if (L <= 0)
        return 0.0f;
    int64_t C = (L + ORACLE_CHUNK - 1) / ORACLE_CHUNK;
    float* t = (float*)malloc((size_t)C * sizeof(float));
    for (int64_t c = 0; c < C; ++c) {
        int64_t lo = c * ORACLE_CHUNK;
        int64_t hi = lo + ORACLE_CHUNK;
        if (hi > L)
            hi = L;
        float a = p[lo];
        for (int64_t i = lo + 1; i < hi; ++i)
            a = oracle_add(a, p[i]);
        t[c] = a;
    }
    for (int64_t s = 1; s < C; s *= 2)
        for (int64_t j = 0; j + s < C; j += 2 * s)
            t[j] = oracle_add(t[j], t[j + s]);
    float r = t[0];
    free(t);
    return r;
}

/* ------------------------------------------------------------------------ */
/* A1 / A2: scales.                                                           */
/* mode 0 (weights, [P4] "How to use" and "Premises and limits": the step    */
/*   size is re-pinned from the weights every optimiser step as              */
/*   2*mean(|w|)/sqrt(q_max)):                                               */
/*     S = canon(|w_0|, ..., |w_{n-1}|); mean = S (/) i2f(n);                 */
/*     s_w = (2 (x) mean) (/) sqrt(i2f(q_max)).                               */
/* mode 1 (activations): s_x = max_i |x_i| (/) i2f(q_max); max is exact.      */
/* ------------------------------------------------------------------------ */

float oracle_wscale(const float* x, int64_t n, int mode, int qmax)
{
    if (mode == 0) {
        float* a = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
        for (int64_t i = 0; i < n; ++i)
            a[i] = fabsf(x[i]); /* clears the sign bit: exact */
        float S = oracle_canon_sum(a, n);
        free(a);
        float mean = oracle_div(S, oracle_i2f(n));
        return oracle_div(oracle_mul(2.0f, mean), oracle_sqrt(oracle_i2f(qmax)));
    }
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float v = fabsf(oracle_flush(x[i]));
        if (v > m)
            m = v;
    }
    return oracle_div(m, oracle_i2f(qmax));
}

void oracle_quant_i8(const float* x, int64_t n, float s, int qmax, int8_t* q)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        q[i] = (int8_t)oracle_quant_one(x[i], s, qmax);
}

/* ------------------------------------------------------------------------ */
/* A5: forward.  The int8 x int8 products and their sum are exact integers,  */
/* so the accumulation order cannot matter; the dequantisation is two        */
/* unfused multiplies, left to right: (i2f(acc) (x) s_x) (x) s_w.            */
/* ------------------------------------------------------------------------ */

int64_t oracle_int_dot(const int8_t* xq, const int8_t* wq, int64_t m, int64_t n,
                       int64_t K)
{
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k)
        acc += (int64_t)xq[m * K + k] * (int64_t)wq[n * K + k];
    return acc;
}

static float fwd_one(const int8_t* xq, const int8_t* wq, float s_x, float s_w,
                     int64_t m, int64_t n, int64_t K)
{
    int64_t acc = oracle_int_dot(xq, wq, m, n, K);
    return oracle_mul(oracle_mul(oracle_i2f(acc), s_x), s_w);
}

void oracle_linear_fwd(const int8_t* xq, const int8_t* wq, float s_x, float s_w,
                       float* y, int64_t M, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            y[m * N + n] = fwd_one(xq, wq, s_x, s_w, m, n, K);
}

void oracle_linear_fwd_at(const int8_t* xq, const int8_t* wq, float s_x, float s_w,
                          int64_t M, int64_t N, int64_t K,
                          const int64_t* idx_m, const int64_t* idx_n, int64_t cnt,
                          float* out)
{
    (void)M;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; ++i)
        out[i] = fwd_one(xq, wq, s_x, s_w, idx_m[i], idx_n[i], K);
}

/* ------------------------------------------------------------------------ */
/* A6-A8: backward in fp32.  The dequantised operands are recomputed from    */
/* int8 (W^ = i2f(Wq) (x) s_w, X^ = i2f(Xq) (x) s_x); each output is the      */
/* canonical sum of its rounded products in increasing reduction index.      */
/* ------------------------------------------------------------------------ */

static float dx_one(const float* dy, const int8_t* wq, float s_w, int64_t m, int64_t k,
                    int64_t N, int64_t K, float* terms)
{
    for (int64_t n = 0; n < N; ++n) {
        float w_hat = oracle_mul(oracle_i2f(wq[n * K + k]), s_w);
        terms[n] = oracle_mul(dy[m * N + n], w_hat);
    }
    return oracle_canon_sum(terms, N);
}

static float dw_one(const float* dy, const int8_t* xq, float s_x, int64_t n, int64_t k,
                    int64_t M, int64_t N, int64_t K, float* terms)
{
    for (int64_t m = 0; m < M; ++m) {
        float x_hat = oracle_mul(oracle_i2f(xq[m * K + k]), s_x);
        terms[m] = oracle_mul(dy[m * N + n], x_hat);
    }
    return oracle_canon_sum(terms, M);
}

void oracle_linear_bwd_dx(const float* dy, const int8_t* wq, float s_w, float* dx,
                          int64_t M, int64_t N, int64_t K)
{
#pragma omp parallel
    {
        float* terms = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
#pragma omp for schedule(static)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t k = 0; k < K; ++k)
                dx[m * K + k] = dx_one(dy, wq, s_w, m, k, N, K, terms);
        free(terms);
    }
}

void oracle_linear_bwd_dw(const float* dy, const int8_t* xq, float s_x, float* dw,
                          int64_t M, int64_t N, int64_t K)
{
#pragma omp parallel
    {
        float* terms = (float*)malloc((size_t)(M > 0 ? M : 1) * sizeof(float));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t k = 0; k < K; ++k)
                dw[n * K + k] = dw_one(dy, xq, s_x, n, k, M, N, K, terms);
        free(terms);
    }
}

void oracle_linear_bwd_dx_at(const float* dy, const int8_t* wq, float s_w,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t* idx_m, const int64_t* idx_k, int64_t cnt,
                             float* out)
{
    (void)M;
#pragma omp parallel
    {
        float* terms = (float*)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
#pragma omp for schedule(static)
        for (int64_t i = 0; i < cnt; ++i)
            out[i] = dx_one(dy, wq, s_w, idx_m[i], idx_k[i], N, K, terms);
        free(terms);
    }
}

void oracle_linear_bwd_dw_at(const float* dy, const int8_t* xq, float s_x,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t* idx_n, const int64_t* idx_k, int64_t cnt,
                             float* out)
{
#pragma omp parallel
    {
        float* terms = (float*)malloc((size_t)(M > 0 ? M : 1) * sizeof(float));
#pragma omp for schedule(static)
        for (int64_t i = 0; i < cnt; ++i)
            out[i] = dw_one(dy, xq, s_x, idx_n[i], idx_k[i], M, N, K, terms);
        free(terms);
    }
}

/* ------------------------------------------------------------------------ */
/* A9: micro-batch accumulation, level 1 of the audit's three-level          */
/* reduction ([P4] "Premises and limits"): one elementwise add per           */
/* micro-batch, in micro-batch order.                                        */
/* ------------------------------------------------------------------------ */

void oracle_grad_accum(float* acc, const float* g, int64_t n)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        acc[i] = oracle_add(acc[i], g[i]);
}

/* ------------------------------------------------------------------------ */
/* Level 2: the intra-node reduce-scatter is replayed as a running sum in one */
/* loop over virtual ranks in mesh order, so only one partial is resident     */
/* ([P4] "Premises and limits"): a left fold in shard order, first partial    */
/* taken as it is.                                                            */
/* ------------------------------------------------------------------------ */

void oracle_running_sum(const float* const* parts, int S, int64_t n, float* out)
{
    if (S < 1)
        return;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float a = parts[0][i];
        for (int s = 1; s < S; ++s)
            a = oracle_add(a, parts[s][i]);
        out[i] = a;
    }
}

/* ------------------------------------------------------------------------ */
/* A10: TreeFold ([P4] "Premises and limits": the replica all-reduce is      */
/* replayed by folding partials in the pairing order of the cluster's        */
/* recursive-doubling all-reduce).  For R not a power of two the pre-step of */
/* the recursive-doubling all-reduce of Thakur, Rabenseifner and Gropp       */
/* (IJHPCA 2005) is used: with p' the largest power of two <= R and          */
/* r = R - p', ranks 2i and 2i+1 (i < r) combine first; then p' survivors    */
/* exchange with partner (rank XOR d) for d = 1, 2, ..., p'/2.  The lower    */
/* rank's operand is written first (bits do not depend on it: IEEE addition  */
/* commutes).                                                                */
/* ------------------------------------------------------------------------ */

static int pow2_floor(int R)
{
    int p = 1;
    while (p * 2 <= R)
        p *= 2;
    return p;
}

/* runs the exchange; v must hold room for p' values; returns p' */
static int rd_allreduce(const float* vals, int R, float* v)
{
    int p2 = pow2_floor(R);
    int r = R - p2;
    for (int i = 0; i < r; ++i)
        v[i] = oracle_add(vals[2 * i], vals[2 * i + 1]);
    for (int i = r; i < p2; ++i)
        v[i] = vals[r + i];
    float nv[64];
    for (int d = 1; d < p2; d *= 2) {
        for (int j = 0; j < p2; ++j) {
            int q = j ^ d;
            nv[j] = (j < q) ? oracle_add(v[j], v[q]) : oracle_add(v[q], v[j]);
        }
        memcpy(v, nv, (size_t)p2 * sizeof(float));
    }
    return p2;
}

float oracle_treefold_one(const float* vals, int R)
{
    float v[64];
    if (R < 1 || R > 64)
        return NAN;
    rd_allreduce(vals, R, v);
    return v[0];
}

void oracle_treefold_all_ranks(const float* vals, int R, float* rank_out)
{
    float v[64];
    if (R < 1 || R > 64)
        return;
    int p2 = rd_allreduce(vals, R, v);
    int r = R - p2;
    for (int q = 0; q < R; ++q) {
        int newrank = (q < 2 * r) ? q / 2 : q - r;
        rank_out[q] = v[newrank];
    }
}

void oracle_treefold(const float* const* parts, int R, int64_t n, float* out)
{
    if (R < 1 || R > 64)
        return;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float vals[64];
        for (int r = 0; r < R; ++r)
            vals[r] = parts[r][i];
        out[i] = oracle_treefold_one(vals, R);
    }
}

/* ------------------------------------------------------------------------ */
/* Optimiser step (see oracle.h for the fixed operation order).               */
/* ------------------------------------------------------------------------ */

float oracle_sumsq(const float* g, int64_t n)
{
    float* t = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    for (int64_t i = 0; i < n; ++i)
        t[i] = oracle_mul(g[i], g[i]);
    float S = oracle_canon_sum(t, n);
    free(t);
    return oracle_flush(S);
}

float oracle_pow_t(float b, int64_t t)
{
    float r = 1.0f, base = b;
    while (t > 0) {
        if (t & 1)
            r = oracle_mul(r, base);
        base = oracle_mul(base, base);
        t >>= 1;
    }
    return r;
}

float oracle_clip_coef(float sumsq, float max_norm)
{
    float norm = oracle_sqrt(sumsq);
    float coef = oracle_div(max_norm, oracle_add(norm, 1e-6f));
    return coef < 1.0f ? coef : 1.0f;
}

void oracle_adamw_step(float* p, float* m, float* v, const float* g, int64_t n, float sumsq,
                       const oracle_adamw_hparams* hp, int64_t t)
{
    const float coef = oracle_clip_coef(sumsq, hp->max_norm);
    const float one_b1 = oracle_add(1.0f, -hp->beta1);
    const float one_b2 = oracle_add(1.0f, -hp->beta2);
    const float bc1 = oracle_add(1.0f, -oracle_pow_t(hp->beta1, t));
    const float bc2 = oracle_add(1.0f, -oracle_pow_t(hp->beta2, t));
    const float decay = oracle_add(1.0f, -oracle_mul(hp->lr, hp->weight_decay));
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const float gc = oracle_mul(g[i], coef);
        const float mi = oracle_add(oracle_mul(hp->beta1, m[i]), oracle_mul(one_b1, gc));
        const float vi = oracle_add(oracle_mul(hp->beta2, v[i]),
                                    oracle_mul(one_b2, oracle_mul(gc, gc)));
        const float mh = oracle_div(mi, bc1);
        const float vh = oracle_div(vi, bc2);
        const float den = oracle_add(oracle_sqrt(vh), hp->eps);
        const float upd = oracle_mul(hp->lr, oracle_div(mh, den));
        p[i] = oracle_add(oracle_mul(p[i], decay), -upd);
        m[i] = mi;
        v[i] = vi;
    }
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
