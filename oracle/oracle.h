/*
 * oracle.h -- plain, slow, obviously-correct CPU statement of the
 * bitwise-reproducible int8 QAT linear layer and its fixed-order gradient
 * reduction.
 *
 * THIS IS TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  The CUDA library never calls it,
 * shares no source with it, and must fail loudly rather than fall back to it.
 *
 * Sources (web pages about the preprint "OPEN-1B: A Fully Auditable Training
 * Run", Gensyn):
 *   [P1] arxivdaily.com/papers/2609.17380, English abstract.
 *   [P3] rit.work blog "open-1b-auditable-training", paragraphs 2-4.
 *   [P4] onedev.kr/papers/92 ("Open-1B" review), sections
 *        "How it works" (어떻게 동작하나), "How to use" (어떻게 쓰나),
 *        "Premises and limits" (전제와 한계).
 *
 * Arithmetic model (every float operation below, no exceptions):
 *   - binary32, round-to-nearest-even;
 *   - no fused multiply-add: a*b+c is a rounded multiply then a rounded add
 *     ([P4] "How it works": contraction disabled on CPU builds);
 *   - subnormals flushed: each operand that is subnormal is replaced by a zero
 *     of the same sign before the operation, and a result that is subnormal
 *     after IEEE rounding (gradual underflow) is replaced by a zero of the same
 *     sign ([P4] "How it works", [P3] paragraph 2: every backend flushes, to
 *     match the least permissive one).
 *   The file must be compiled with -ffp-contract=off and without fast-math;
 *   the floating-point environment is never modified.
 *
 * Canonical reduction order ("a fixed reduction order on all hardware",
 * [P4] "How it works"; [P1]): a sum of L terms p_0..p_{L-1} is
 *   1. cut into chunks of 64 consecutive terms (the last chunk may be short);
 *   2. each chunk summed left to right, seeded with its first term;
 *   3. the chunk partials t_0..t_{C-1} combined by a stride-doubling pairwise
 *      tree: for s = 1, 2, 4, ...: t_j <- t_j + t_{j+s} for every j that is a
 *      multiple of 2s with j+s < C; the result is t_0.  L = 0 gives +0.
 *
 * Parity status: every function here is pinned by the tests against exact
 * rational arithmetic, hand-worked cases, closed forms or invariants; none is
 * "parity unpinned".
 */
#ifndef REPRO_ORACLE_H
#define REPRO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_CHUNK 64

/* ---- elementary operations (the arithmetic model above) ---- */
float oracle_flush(float x);               /* subnormal -> signed zero      */
float oracle_add(float a, float b);        /* a (+) b                        */
float oracle_mul(float a, float b);        /* a (x) b                        */
float oracle_div(float a, float b);        /* a (/) b                        */
float oracle_sqrt(float a);                /* correctly rounded sqrt, flushed */
float oracle_i2f(int64_t v);               /* integer -> binary32, RNE        */
int   oracle_quant_one(float x, float s, int qmax); /* clamp(rint(x (/) s))  */

/* ---- canonical sum (order above) ---- */
float oracle_canon_sum(const float* p, int64_t L);

/* ---- A1/A2: scales.  mode 0: 2*mean|w|/sqrt(qmax); mode 1: max|x|/qmax ---- */
float oracle_wscale(const float* x, int64_t n, int mode, int qmax);

/* ---- A3/A4: q = clamp(rint_half_even(x (/) s), -qmax, qmax) ---- */
void oracle_quant_i8(const float* x, int64_t n, float s, int qmax, int8_t* q);

/* ---- A5: Y[m,n] = (i2f(sum_k Xq[m,k] Wq[n,k]) (x) s_x) (x) s_w ---- */
void oracle_linear_fwd(const int8_t* xq, const int8_t* wq, float s_x, float s_w,
                       float* y, int64_t M, int64_t N, int64_t K);
/* the same, at `cnt` sampled outputs (row idx_a[i], column idx_b[i]) */
void oracle_linear_fwd_at(const int8_t* xq, const int8_t* wq, float s_x, float s_w,
                          int64_t M, int64_t N, int64_t K,
                          const int64_t* idx_m, const int64_t* idx_n, int64_t cnt,
                          float* out);
/* exact integer accumulator (for pinning only) */
int64_t oracle_int_dot(const int8_t* xq, const int8_t* wq, int64_t m, int64_t n,
                       int64_t K);

/* ---- A6-A8: backward.  W^[n,k] = i2f(Wq[n,k]) (x) s_w, X^[m,k] likewise.
 *   dX[m,k] = canon_{n}( dY[m,n] (x) W^[n,k] )
 *   dW[n,k] = canon_{m}( dY[m,n] (x) X^[m,k] )                              */
void oracle_linear_bwd_dx(const float* dy, const int8_t* wq, float s_w, float* dx,
                          int64_t M, int64_t N, int64_t K);
void oracle_linear_bwd_dw(const float* dy, const int8_t* xq, float s_x, float* dw,
                          int64_t M, int64_t N, int64_t K);
void oracle_linear_bwd_dx_at(const float* dy, const int8_t* wq, float s_w,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t* idx_m, const int64_t* idx_k, int64_t cnt,
                             float* out);
void oracle_linear_bwd_dw_at(const float* dy, const int8_t* xq, float s_x,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t* idx_n, const int64_t* idx_k, int64_t cnt,
                             float* out);

/* ---- A9: acc[i] <- acc[i] (+) g[i] ---- */
void oracle_grad_accum(float* acc, const float* g, int64_t n);

/* ---- level 2 of the replayed reduction: running sum over S shard partials in
 * mesh order, out = (...((P0 (+) P1) (+) P2) ...) (+) P_{S-1} ---- */
void oracle_running_sum(const float* const* parts, int S, int64_t n, float* out);

/* ---- A10: TreeFold over R replica partials, recursive-doubling pairing ---- */
float oracle_treefold_one(const float* vals, int R);
void  oracle_treefold(const float* const* parts, int R, int64_t n, float* out);
/* every rank's final value of the simulated recursive-doubling all-reduce
 * (for the invariant that all ranks agree); `rank_out` has R entries */
void  oracle_treefold_all_ranks(const float* vals, int R, float* rank_out);

/* ---- optimiser step after TreeFold: global-norm clip + AdamW ----
 * Recipe ([P4] "Premises and limits"): AdamW(beta1 0.9, beta2 0.95, eps 1e-8),
 * decoupled weight decay 0.1, gradient clipping at global L2 norm 1.0.  The
 * pages give no operation order; this one is fixed (binary32, flushed):
 *   sumsq = canon_sum(g_i (x) g_i) over the flat gradient; norm = sqrt(sumsq)
 *   coef  = min(max_norm (/) (norm (+) 1e-6), 1);  g' = g (x) coef
 *   b^t by right-to-left binary exponentiation: r = 1, base = b; for each bit
 *   of t from the lowest: if set r = r (x) base; then base = base (x) base
 *   m = (b1 (x) m) (+) ((1 (-) b1) (x) g');  v = (b2 (x) v) (+) ((1 (-) b2) (x) (g' (x) g'))
 *   mh = m (/) (1 (-) b1^t);  vh = v (/) (1 (-) b2^t)
 *   p = (p (x) (1 (-) (lr (x) wd))) (-) (lr (x) (mh (/) (sqrt(vh) (+) eps)))   */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay, max_norm;
} oracle_adamw_hparams;
float oracle_sumsq(const float* g, int64_t n);
float oracle_pow_t(float b, int64_t t);
float oracle_clip_coef(float sumsq, float max_norm);
void oracle_adamw_step(float* p, float* m, float* v, const float* g, int64_t n, float sumsq,
                       const oracle_adamw_hparams* hp, int64_t t);

/* threads the parallel loops use (1 when built without OpenMP) */
/* Attention with int8 P.V (see oracle.c for the readings and the order). */
float oracle_exp(float x);
int oracle_attn_quant_p(float p);
int64_t oracle_attn_fx(float x);
float oracle_attn_fix2f(int64_t a);
void oracle_attn_fwd(const float* q, const float* k, const int8_t* vq, float s_v, float* o,
                     float* mrow, float* lrow, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                     int64_t D, int64_t W);
void oracle_attn_fwd_rows(const float* q, const float* k, const int8_t* vq, float s_v,
                          const int64_t* rows, int64_t nrows, float* o, float* mrow,
                          float* lrow, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                          int64_t D, int64_t W);
void oracle_attn_bwd(const float* q, const float* k, const int8_t* vq, float s_v, const float* o,
                     const float* dout, const float* mrow, const float* lrow, float* dq, float* dk,
                     float* dv, int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                     int64_t W);
void oracle_attn_bwd_rows(const float* q, const float* k, const int8_t* vq, float s_v,
                          const float* o, const float* dout, const float* mrow,
                          const float* lrow, const int64_t* qrows, int64_t nq, float* dq,
                          const int64_t* krows, int64_t nk, float* dk, float* dv, int64_t B,
                          int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t W);

int oracle_threads(void);
void oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
