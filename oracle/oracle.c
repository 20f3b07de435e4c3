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

/* ------------------------------------------------------------------------ */
/* Attention with int8 P.V ([P4] "How to use": inside flash attention the    */
/* P.V product runs on int8 while the QK^T logits and the softmax stay in    */
/* high precision; the attention backward accumulates dQ in 64-bit fixed     */
/* point).  The pages fix no operation order; the readings taken here:       */
/*   logits  s_ij = canon_d(q_id (x) k_jd) (x) c, c = 1 (/) sqrt(D);         */
/*   keys    j in [lo_i, i], lo_i = max(0, i - W + 1) for a sliding window  */
/*           of W tokens, 0 for W = 0 (full causal); GQA: query head h      */
/*           reads kv head h / (Hq / Hkv);                                   */
/*   m_i     = max_j s_ij (exact, so the softmax is taken in two passes);    */
/*   p_ij    = exp_r(s_ij (-) m_i), l_i = canon_j(p_ij) over j ascending;    */
/*   int8 P  P_ij = clamp(rint(p_ij (x) 127), 0, 127); V = V_q with scale s_v;*/
/*   o_id    = (i2f(sum_j P_ij V_q,jd) (x) s_v) (/) (l_i (x) 127), the       */
/*           integer sum exact.                                              */
/* Layout: q, o [B][T][Hq][D]; k, v [B][T][Hkv][D]; m, l [B][T][Hq].         */
/* ------------------------------------------------------------------------ */

/* e^x: range reduction of Cody and Waite ("Software Manual for the          */
/* Elementary Functions", 1980) with ln 2 split as C1 + C2, C1 = 355/512     */
/* (exact in 9 bits, so k (x) C1 is exact), then the degree-7 Taylor         */
/* polynomial of e^r in Horner form with binary32 coefficients RN(1/n!),     */
/* then the exact scaling by 2^k; every operation rounded and flushed.       */
#define EXP_LOG2E 0x1.715476p+0f   /* RN(1/ln 2) */
#define EXP_C1 0x1.63p-1f            /* 355/512 */
#define EXP_C2 -0x1.bd0106p-13f      /* RN(ln 2 - 355/512) */

float oracle_exp(float x)
{
    const float kf = nearbyintf(oracle_mul(x, EXP_LOG2E)); /* ties to even */
    const float r = oracle_add(oracle_add(x, -oracle_mul(kf, EXP_C1)), -oracle_mul(kf, EXP_C2));
    /* RN(1/n!), n = 0..7 */
    static const float c[8] = {1.0f, 1.0f, 0.5f, 0x1.555556p-3f, 0x1.555556p-5f, 0x1.111112p-7f,
                               0x1.6c16c2p-10f, 0x1.a01a02p-13f};
    float p = c[7];
    for (int n = 6; n >= 0; --n)
        p = oracle_add(oracle_mul(p, r), c[n]);
    if (kf < -126.0f)
        return 0.0f;
    if (kf > 254.0f)
        return INFINITY; /* 2^k alone overflows, whatever p is (so e^+inf = +inf) */
    if (kf != kf)
        return kf; /* NaN */
    return oracle_flush(ldexpf(p, (int)kf));
}

static float attn_c(int64_t D)
{
    return oracle_div(1.0f, oracle_sqrt((float)D));
}

static int64_t attn_lo(int64_t i, int64_t W)
{
    return (W > 0 && i - W + 1 > 0) ? i - W + 1 : 0;
}

static float attn_logit(const float* q, const float* k, int64_t b, int64_t i, int64_t j,
                        int64_t h, int64_t g, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                        float c, float* tmp)
{
    const float* qi = q + ((b * T + i) * Hq + h) * D;
    const float* kj = k + ((b * T + j) * Hkv + g) * D;
    for (int64_t d = 0; d < D; ++d)
        tmp[d] = oracle_mul(qi[d], kj[d]);
    return oracle_mul(oracle_canon_sum(tmp, D), c);
}

int oracle_attn_quant_p(float p)
{
    float r = nearbyintf(oracle_mul(p, 127.0f));
    if (r != r)
        return 0; /* NaN: the clamp's lower bound */
    if (r > 127.0f)
        r = 127.0f;
    if (r < 0.0f)
        r = 0.0f;
    return (int)r;
}

/* one query row: o[D], m, l */
static void attn_fwd_row(const float* q, const float* k, const int8_t* vq, float s_v,
                         int64_t b, int64_t i, int64_t h, int64_t T, int64_t Hq, int64_t Hkv,
                         int64_t D, int64_t W, float* o, float* m_out, float* l_out)
{
    const int64_t g = h / (Hq / Hkv), lo = attn_lo(i, W), n = i - lo + 1;
    const float c = attn_c(D);
    float* s = (float*)malloc((size_t)n * sizeof(float));
    float* tmp = (float*)malloc((size_t)(D > n ? D : n) * sizeof(float));
    int64_t* acc = (int64_t*)calloc((size_t)D, sizeof(int64_t));
    float m = -INFINITY; /* the maximum of no logit */
    for (int64_t t = 0; t < n; ++t) {
        s[t] = attn_logit(q, k, b, i, lo + t, h, g, T, Hq, Hkv, D, c, tmp);
        if (s[t] > m) /* a NaN logit never compares greater: it is passed over */
            m = s[t];
    }
    if (m == 0.0f)
        m = 0.0f; /* a zero maximum is stored as +0 */
    for (int64_t t = 0; t < n; ++t) {
        const float p = oracle_exp(oracle_add(s[t], -m));
        tmp[t] = p;
        const int pq = oracle_attn_quant_p(p);
        const int8_t* vj = vq + ((b * T + lo + t) * Hkv + g) * D;
        for (int64_t d = 0; d < D; ++d)
            acc[d] += (int64_t)pq * vj[d];
    }
    const float l = oracle_canon_sum(tmp, n);
    const float den = oracle_mul(l, 127.0f);
    for (int64_t d = 0; d < D; ++d)
        o[d] = oracle_div(oracle_mul(oracle_i2f(acc[d]), s_v), den);
    *m_out = m;
    *l_out = l;
    free(s);
    free(tmp);
    free(acc);
}

void oracle_attn_fwd(const float* q, const float* k, const int8_t* vq, float s_v, float* o,
                     float* mrow, float* lrow, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                     int64_t D, int64_t W)
{
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < B * T * Hq; ++r) {
        const int64_t h = r % Hq, bi = r / Hq, i = bi % T, b = bi / T;
        attn_fwd_row(q, k, vq, s_v, b, i, h, T, Hq, Hkv, D, W, o + r * D, mrow + r, lrow + r);
    }
}

void oracle_attn_fwd_rows(const float* q, const float* k, const int8_t* vq, float s_v,
                          const int64_t* rows, int64_t nrows, float* o, float* mrow,
                          float* lrow, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                          int64_t D, int64_t W)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nrows; ++t) {
        const int64_t r = rows[t];
        const int64_t h = r % Hq, bi = r / Hq, i = bi % T, b = bi / T;
        attn_fwd_row(q, k, vq, s_v, b, i, h, T, Hq, Hkv, D, W, o + t * D, mrow + t, lrow + t);
    }
}

/* Backward (straight-through for both quantisations):                        */
/*   a_ij  = p_ij (/) l_i, p_ij recomputed as in the forward from m_i;        */
/*   V^_jd = i2f(V_q,jd) (x) s_v;  Dr_i = canon_d(dO_id (x) O_id);            */
/*   dA_ij = canon_d(dO_id (x) V^_jd);  dS_ij = a_ij (x) (dA_ij (-) Dr_i);    */
/*   dQ_id = (fix2f(sum over key tiles t of fx(T_t))) (x) c, where T_t is the */
/*     left-to-right sum over the valid keys j of the 64-aligned key tile t   */
/*     of dS_ij (x) k_jd (seeded with the first such term), fx(x) = the       */
/*     nearest int64 to x * 2^48 (ties to even, saturating, NaN to 0) and     */
/*     fix2f(A) = flush(i2f(A) * 2^-48): the tile partials are accumulated in */
/*     64-bit fixed point, exactly and in any order (the int64 sum wraps      */
/*     modulo 2^64 where saturated partials overflow it);                     */
/*   dK_jd = (fold) (x) c and dV_jd = (fold), where the terms dS_ij (x) q_id  */
/*     (dK) and a_ij (x) dO_id (dV) run over the query heads h of kv head g   */
/*     in ascending order and, within a head, over the valid queries i;       */
/*     they are grouped by 64-aligned query tile, each group summed left to   */
/*     right from its first term, and the group partials folded left in      */
/*     (head, tile) order.                                                    */
#define ATTN_FIX_BITS 48
#define ATTN_TILE 64

int64_t oracle_attn_fx(float x)
{
    const double v = nearbyint((double)oracle_flush(x) * 281474976710656.0); /* exact */
    if (v != v)
        return 0; /* NaN */
    if (v >= 9223372036854775807.0)
        return INT64_MAX;
    if (v <= -9223372036854775808.0)
        return INT64_MIN;
    return (int64_t)v;
}

float oracle_attn_fix2f(int64_t a)
{
    return oracle_flush(oracle_i2f(a) * (1.0f / 281474976710656.0f)); /* exact but for the flush */
}

static float attn_drow(const float* o, const float* dout, int64_t r, int64_t D, float* tmp)
{
    for (int64_t d = 0; d < D; ++d)
        tmp[d] = oracle_mul(dout[r * D + d], o[r * D + d]);
    return oracle_canon_sum(tmp, D);
}

/* a_ij and dS_ij for one (query row, key) pair */
static void attn_pair(const float* q, const float* k, const int8_t* vq, float s_v,
                      const float* dout, const float* mrow, const float* lrow, float drow,
                      int64_t b, int64_t i, int64_t j, int64_t h, int64_t g, int64_t T,
                      int64_t Hq, int64_t Hkv, int64_t D, float c, float* tmp, float* a_out,
                      float* ds_out)
{
    const int64_t r = (b * T + i) * Hq + h;
    const float s = attn_logit(q, k, b, i, j, h, g, T, Hq, Hkv, D, c, tmp);
    const float a = oracle_div(oracle_exp(oracle_add(s, -mrow[r])), lrow[r]);
    const int8_t* vj = vq + ((b * T + j) * Hkv + g) * D;
    for (int64_t d = 0; d < D; ++d)
        tmp[d] = oracle_mul(dout[r * D + d], oracle_mul(oracle_i2f(vj[d]), s_v));
    const float dA = oracle_canon_sum(tmp, D);
    *a_out = a;
    *ds_out = oracle_mul(a, oracle_add(dA, -drow));
}

static void attn_dq_row(const float* q, const float* k, const int8_t* vq, float s_v,
                        const float* o, const float* dout, const float* mrow, const float* lrow,
                        int64_t b, int64_t i, int64_t h, int64_t T, int64_t Hq, int64_t Hkv,
                        int64_t D, int64_t W, float* dq)
{
    const int64_t g = h / (Hq / Hkv), lo = attn_lo(i, W), r = (b * T + i) * Hq + h;
    const float c = attn_c(D);
    float* tmp = (float*)malloc((size_t)D * sizeof(float));
    float* part = (float*)malloc((size_t)D * sizeof(float));
    uint64_t* acc = (uint64_t*)calloc((size_t)D, sizeof(uint64_t)); /* wraps modulo 2^64 */
    const float drow = attn_drow(o, dout, r, D, tmp);
    for (int64_t t0 = (lo / ATTN_TILE) * ATTN_TILE; t0 <= i; t0 += ATTN_TILE) {
        const int64_t jb = t0 > lo ? t0 : lo, je = t0 + ATTN_TILE - 1 < i ? t0 + ATTN_TILE - 1 : i;
        for (int64_t j = jb; j <= je; ++j) {
            float a, ds;
            attn_pair(q, k, vq, s_v, dout, mrow, lrow, drow, b, i, j, h, g, T, Hq, Hkv, D, c,
                      tmp, &a, &ds);
            const float* kj = k + ((b * T + j) * Hkv + g) * D;
            for (int64_t d = 0; d < D; ++d) {
                const float t = oracle_mul(ds, kj[d]);
                part[d] = j == jb ? t : oracle_add(part[d], t);
            }
        }
        for (int64_t d = 0; d < D; ++d)
            acc[d] += (uint64_t)oracle_attn_fx(part[d]);
    }
    for (int64_t d = 0; d < D; ++d) {
        int64_t a;
        memcpy(&a, &acc[d], sizeof a); /* the two's-complement value */
        dq[d] = oracle_mul(oracle_attn_fix2f(a), c);
    }
    free(tmp);
    free(part);
    free(acc);
}

static void attn_dkdv_row(const float* q, const float* k, const int8_t* vq, float s_v,
                          const float* o, const float* dout, const float* mrow,
                          const float* lrow, int64_t b, int64_t j, int64_t g, int64_t T,
                          int64_t Hq, int64_t Hkv, int64_t D, int64_t W, float* dk, float* dv)
{
    const int64_t G = Hq / Hkv;
    const float c = attn_c(D);
    const int64_t ihi = (W > 0 && j + W - 1 < T - 1) ? j + W - 1 : T - 1;
    float* tmp = (float*)malloc((size_t)D * sizeof(float));
    float* pk = (float*)malloc((size_t)D * sizeof(float));
    float* pv = (float*)malloc((size_t)D * sizeof(float));
    float* fk = (float*)malloc((size_t)D * sizeof(float));
    float* fv = (float*)malloc((size_t)D * sizeof(float));
    int first_group = 1;
    for (int64_t hh = 0; hh < G; ++hh) {
        const int64_t h = g * G + hh;
        for (int64_t t0 = (j / ATTN_TILE) * ATTN_TILE; t0 <= ihi; t0 += ATTN_TILE) {
            const int64_t ib = t0 > j ? t0 : j;
            const int64_t ie = t0 + ATTN_TILE - 1 < ihi ? t0 + ATTN_TILE - 1 : ihi;
            for (int64_t i = ib; i <= ie; ++i) {
                const int64_t r = (b * T + i) * Hq + h;
                const float drow = attn_drow(o, dout, r, D, tmp);
                float a, ds;
                attn_pair(q, k, vq, s_v, dout, mrow, lrow, drow, b, i, j, h, g, T, Hq, Hkv, D,
                          c, tmp, &a, &ds);
                const float* qi = q + r * D;
                const float* di = dout + r * D;
                for (int64_t d = 0; d < D; ++d) {
                    const float tk = oracle_mul(ds, qi[d]);
                    const float tv = oracle_mul(a, di[d]);
                    pk[d] = i == ib ? tk : oracle_add(pk[d], tk);
                    pv[d] = i == ib ? tv : oracle_add(pv[d], tv);
                }
            }
            for (int64_t d = 0; d < D; ++d) {
                fk[d] = first_group ? pk[d] : oracle_add(fk[d], pk[d]);
                fv[d] = first_group ? pv[d] : oracle_add(fv[d], pv[d]);
            }
            first_group = 0;
        }
    }
    for (int64_t d = 0; d < D; ++d) {
        dk[d] = oracle_mul(fk[d], c);
        dv[d] = fv[d];
    }
    free(tmp);
    free(pk);
    free(pv);
    free(fk);
    free(fv);
}

void oracle_attn_bwd(const float* q, const float* k, const int8_t* vq, float s_v, const float* o,
                     const float* dout, const float* mrow, const float* lrow, float* dq, float* dk,
                     float* dv, int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                     int64_t W)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < B * T * Hq; ++r) {
        const int64_t h = r % Hq, bi = r / Hq, i = bi % T, b = bi / T;
        attn_dq_row(q, k, vq, s_v, o, dout, mrow, lrow, b, i, h, T, Hq, Hkv, D, W, dq + r * D);
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < B * T * Hkv; ++r) {
        const int64_t g = r % Hkv, bj = r / Hkv, j = bj % T, b = bj / T;
        attn_dkdv_row(q, k, vq, s_v, o, dout, mrow, lrow, b, j, g, T, Hq, Hkv, D, W, dk + r * D,
                      dv + r * D);
    }
}

/* sampled rows: dq for query rows qrows[] (flat (b, i, h) indices), dk/dv for
 * key rows krows[] (flat (b, j, g) indices) */
void oracle_attn_bwd_rows(const float* q, const float* k, const int8_t* vq, float s_v,
                          const float* o, const float* dout, const float* mrow,
                          const float* lrow, const int64_t* qrows, int64_t nq, float* dq,
                          const int64_t* krows, int64_t nk, float* dk, float* dv, int64_t B,
                          int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t W)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nq; ++t) {
        const int64_t r = qrows[t];
        const int64_t h = r % Hq, bi = r / Hq, i = bi % T, b = bi / T;
        attn_dq_row(q, k, vq, s_v, o, dout, mrow, lrow, b, i, h, T, Hq, Hkv, D, W, dq + t * D);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nk; ++t) {
        const int64_t r = krows[t];
        const int64_t g = r % Hkv, bj = r / Hkv, j = bj % T, b = bj / T;
        attn_dkdv_row(q, k, vq, s_v, o, dout, mrow, lrow, b, j, g, T, Hq, Hkv, D, W, dk + t * D,
                      dv + t * D);
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

/* threads for the parallel loops over output elements from now on (n >= 1);
 * no element's sequence of operations depends on it */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
