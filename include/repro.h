/*
 * repro.h -- C ABI of the bitwise-reproducible int8 quantisation-aware linear
 * layer (forward and backward) and of the fixed-order gradient reduction that
 * follows it, for one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages about the preprint "OPEN-1B: A Fully Auditable Training
 * Run", Gensyn):
 *   [abstract]  arxivdaily.com/papers/2609.17380, English abstract: a definite
 *               order is imposed on GPU kernel reductions, batch ordering and
 *               collectives so any step replays bit for bit on one device.
 *   [works]     Open-1B review, onedev.kr/papers/92, section "How it works"
 *               (어떻게 동작하나): fixed reduction order on every backend,
 *               explicit unfused multiply-add, subnormals flushed to zero.
 *   [use]       same page, section "How to use" (어떻게 쓰나): every attention
 *               and feed-forward linear is int8 QAT (LSQ-based) with 8-bit
 *               weights and activations; the weight scale is re-pinned every
 *               optimiser step to 2*mean(|w|)/sqrt(q_max).
 *   [limits]    same page, section "Premises and limits" (전제와 한계): the
 *               audit replays a three-level reduction on one device --
 *               micro-batch accumulation, intra-node reduce-scatter, and the
 *               replica all-reduce as a TreeFold in recursive-doubling pairing
 *               order; stochastic rounding is rejected.
 *
 * Numerics, for every call (the library's fixing of what the pages leave open):
 *   - binary32, round-to-nearest-even, never a fused multiply-add;
 *   - subnormal operands are read as signed zero, subnormal results (after
 *     IEEE rounding) are written as signed zero;
 *   - "canonical sum" of L terms: chunks of 64 consecutive terms summed left
 *     to right seeded with the chunk's first term, then the chunk partials
 *     combined by the stride-doubling pairwise tree (t_j += t_{j+s}, j a
 *     multiple of 2s, j+s < C, s = 1, 2, 4, ...).  L = 0 gives +0.
 *   - q_max = 127; int8 codes lie in [-127, 127].
 * Results are bit-identical across runs, streams and launch configurations.
 *
 * Conventions:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; tensors are
 *     dense row-major.  Scales are single floats in DEVICE memory, so a whole
 *     step can run without host synchronisation.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call only enqueues work on it and returns; nothing is synchronous
 *     except repro_device_check().
 *   - Errors are returned as negative repro_status codes; nothing is launched
 *     when the arguments are invalid.  Device pointers must be 16-byte aligned.
 *   - The library allocates no device memory: calls that need scratch space
 *     take a caller-provided workspace and report its size through *_ws_bytes.
 *     A workspace belongs to one call at a time: calls that may run at the
 *     same time (on different streams) need different workspaces.  Calls on
 *     different streams that touch different buffers may overlap freely; the
 *     results do not depend on how they overlap.
 *   - The library keeps no state between calls except a per-device
 *     architecture check, the launch-configuration override and the device
 *     error word read by repro_device_check().
 */
#ifndef REPRO_H
#define REPRO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define REPRO_VERSION 1
#define REPRO_QMAX 127
#define REPRO_CHUNK 64
#define REPRO_MAX_REPLICAS 64

typedef enum {
    REPRO_OK = 0,
    REPRO_ERR_ARG = -1,       /* NULL pointer, unknown mode/flag, q_max != 127, R out of range */
    REPRO_ERR_SHAPE = -2,     /* negative size, empty tensor where a value is required, K too large */
    REPRO_ERR_ALIGN = -3,     /* a device pointer is not 16-byte aligned */
    REPRO_ERR_ARCH = -4,      /* the current device is not compute capability 10.3 (GB300) */
    REPRO_ERR_LAUNCH = -5,    /* the CUDA runtime reported an error while enqueueing */
    REPRO_ERR_TIMEOUT = -6,   /* a bounded device-side wait gave up (repro_device_check) */
    REPRO_ERR_WORKSPACE = -7, /* workspace NULL or smaller than *_ws_bytes() */
    REPRO_ERR_ALIAS = -8,     /* two buffers that must not overlap do */
    REPRO_ERR_SELFTEST = -9,  /* repro_selftest found the tensor-core forward inexact */
    REPRO_ERR_NONFINITE = -10 /* debug mode: a float input held a NaN or an infinity
                                 (repro_device_check; see repro_set_debug) */
} repro_status;

typedef enum {
    REPRO_SCALE_WEIGHT_MEANABS = 0, /* s = (2 (x) (canon_sum|x| (/) n)) (/) sqrt(q_max) */
    REPRO_SCALE_ACT_AMAX = 1        /* s = max|x| (/) q_max                             */
} repro_scale_mode;

/* ------------------------------------------------------------------------
 * Scale ([use]; [limits]: the learned LSQ step size diverged in int8
 * pre-training and is instead recomputed from the weights every step).
 *   mode WEIGHT_MEANABS: S = canonical sum of |x_i| over the flat tensor,
 *     mean = S (/) float(n), s = (2 (x) mean) (/) sqrt(float(q_max)).
 *   mode ACT_AMAX: s = (max_i |x_i|) (/) float(q_max) (max is exact, so its
 *     evaluation order is free).
 * x: n floats; scale_out: 1 float (device).  ws: workspace of at least
 * repro_wscale_ws_bytes(n) bytes (contents on entry are ignored).
 * Errors: n <= 0 -> REPRO_ERR_SHAPE; unknown mode or q_max != 127 ->
 * REPRO_ERR_ARG; small ws -> REPRO_ERR_WORKSPACE.
 * ------------------------------------------------------------------------ */
int repro_wscale(const float* x, int64_t n, int mode, int qmax, float* scale_out,
                 void* ws, size_t ws_bytes, void* stream);
size_t repro_wscale_ws_bytes(int64_t n);

/* ------------------------------------------------------------------------
 * Quantise ([use]: 8-bit weights and activations; [limits]: deterministic
 * rounding).  q_i = clamp(round_half_even(x_i (/) s), -127, 127), where the
 * quotient is the correctly rounded binary32 division (rounding the quotient
 * and then the integer is the defined double rounding).  s <= subnormal gives
 * q = 0 everywhere; a NaN quotient gives 0; +-Inf clamps.
 * x: n floats; scale: 1 float (device); q_out: n int8.  n == 0 is a no-op.
 * ------------------------------------------------------------------------ */
int repro_quant_i8(const float* x, int64_t n, const float* scale, int qmax,
                   int8_t* q_out, void* stream);

/* ------------------------------------------------------------------------
 * Several tensors at once ([use], [limits]: the weight scale is re-pinned
 * from the weights every optimiser step, and every linear's weights are then
 * quantised): the same results, bit for bit, as repro_wscale on each xs[t]
 * (into scales_out[t]) and repro_quant_i8 of each xs[t] with scales[t] (into
 * q_outs[t]), in one pass over all of them -- one launch for the quantiser,
 * two for the scales -- so a step's weights do not pay one short launch
 * chain per tensor.
 * xs, ns, q_outs: HOST arrays of `count` (1 .. REPRO_MAX_TENSORS) device
 * pointers and element counts; scales_out / scales: `count` floats (DEVICE).
 * repro_wscale_multi: every ns[t] >= 1; ws of repro_wscale_multi_ws_bytes
 * bytes (0 returned for invalid sizes); scales_out must not overlap the xs.
 * repro_quant_i8_multi: ns[t] == 0 skips tensor t; no q_out may overlap an x,
 * the scales or another q_out.  Errors as the single-tensor calls.
 * ------------------------------------------------------------------------ */
#define REPRO_MAX_TENSORS 64
int repro_wscale_multi(const float* const* xs, const int64_t* ns, int count, int mode, int qmax,
                       float* scales_out, void* ws, size_t ws_bytes, void* stream);
size_t repro_wscale_multi_ws_bytes(const int64_t* ns, int count);
int repro_quant_i8_multi(const float* const* xs, const int64_t* ns, int count,
                         const float* scales, int qmax, int8_t* const* q_outs, void* stream);

/* ------------------------------------------------------------------------
 * Forward ([use]; [abstract]).  acc[m,n] = sum_k Xq[m,k]*Wq[n,k] computed
 * exactly as an integer (so its order cannot matter), then
 * Y[m,n] = (float(acc) (x) s_x) (x) s_w -- two unfused multiplies, left to
 * right.  xq: M x K int8, wq: N x K int8 (nn.Linear layout), y: M x N float.
 * Requires K <= 133144 so that |acc| <= 127*127*K fits in int32, and
 * M, N <= 4194240 (REPRO_ERR_SHAPE otherwise).  M, N or K may be 0 (K == 0
 * writes +0 times the scales).
 * When K is a multiple of 8 the product runs on the tensor cores from bf16
 * copies of the codes, which the call writes into `ws` (at least
 * repro_linear_fwd_ws_bytes(M, N, K) bytes; 0 for shapes that use the exact
 * CUDA-core path).  Too small a workspace -> REPRO_ERR_WORKSPACE.
 * The tensor-core path is exact only if the tensor core adds integer products
 * exactly inside each 512-term slice, which the hardware documentation does
 * not state; so the first such call on a device first runs the check of
 * repro_selftest in `ws` and synchronises `stream` (once per device and
 * process).  If the check fails, that call and every later one on the device
 * take the exact CUDA-core path, and the next repro_device_check returns
 * REPRO_ERR_SELFTEST.  A call made while `stream` is being captured into a
 * CUDA graph cannot synchronise: before the check has run on the device it
 * takes the CUDA-core path (so make one call before capturing).
 * ------------------------------------------------------------------------ */
int repro_linear_fwd(const int8_t* xq, const int8_t* wq, const float* s_x,
                     const float* s_w, float* y, int64_t M, int64_t N, int64_t K,
                     void* ws, size_t ws_bytes, void* stream);
size_t repro_linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K);

/* ------------------------------------------------------------------------
 * Backward ([works]: fixed order, unfused multiply then add).  Operands are
 * dequantised from int8 on the fly, identically every time:
 *   W^[n,k] = float(Wq[n,k]) (x) s_w,   X^[m,k] = float(Xq[m,k]) (x) s_x
 *   dX[m,k] = canonical sum over n = 0..N-1 of ( dY[m,n] (x) W^[n,k] )
 *   dW[n,k] = canonical sum over m = 0..M-1 of ( dY[m,n] (x) X^[m,k] )
 * (straight-through estimator; no clipping mask.)
 * dy: M x N float; xq: M x K int8; wq: N x K int8; dx: M x K float or NULL
 * (skip); dw: N x K float or NULL (skip).  xq/s_x may be NULL when dw is NULL;
 * wq/s_w may be NULL when dx is NULL.
 * flags: REPRO_BWD_DW_ACCUMULATE -- instead of storing dW, update
 *   dw[n,k] <- dw[n,k] (+) dW[n,k] (one add of the fully formed dW; the same
 *   bits as repro_grad_accum on a stored dW).
 * ws: at least repro_linear_bwd_ws_bytes(M, N, K) bytes for the current
 * launch configuration.  Long reductions, and grids too small to fill whole
 * waves of SMs, are split into aligned segments whose partials live there.
 * With the default kernel (16-byte-aligned rows: N % 4 == 0, K % 16 == 0) the
 * call first writes its prepared operands there too -- flushed dY (transposed
 * for dX) and the dequantised int8 operand, max(N*pad4(M) + N*K, M*N + M*K)
 * floats after the segment partials -- and the main kernel reads them with
 * tensor copies; the values, and so the bits, are those defined above.
 * M, N <= 4194240 (REPRO_ERR_SHAPE otherwise).
 * dx and dw must not overlap dy, xq or wq, and ws must overlap none of the
 * other buffers (REPRO_ERR_ALIAS).
 * ------------------------------------------------------------------------ */
#define REPRO_BWD_DW_ACCUMULATE 1
int repro_linear_bwd(const float* dy, const int8_t* xq, const int8_t* wq,
                     const float* s_x, const float* s_w, float* dx, float* dw,
                     int64_t M, int64_t N, int64_t K, int flags,
                     void* ws, size_t ws_bytes, void* stream);
size_t repro_linear_bwd_ws_bytes(int64_t M, int64_t N, int64_t K);

/* ------------------------------------------------------------------------
 * Micro-batch accumulation ([limits], level 1 of the replayed reduction):
 * acc[i] <- acc[i] (+) g[i].  Called once per micro-batch after the first, in
 * micro-batch order (the first micro-batch's gradient is the accumulator's
 * initial value).  acc and g must not overlap (REPRO_ERR_ALIAS).
 * ------------------------------------------------------------------------ */
int repro_grad_accum(float* acc, const float* g, int64_t n, void* stream);

/* ------------------------------------------------------------------------
 * Reduce-scatter replay ([limits], level 2: the intra-node reduce-scatter is
 * replayed as a running sum in one loop over virtual ranks in mesh order,
 * replica-major and shard-minor, with one partial resident at a time):
 * out = (...((P0 (+) P1) (+) P2) ...) (+) P_{S-1}, shard index increasing.
 * The same bits as starting an accumulator from P0 and calling
 * repro_grad_accum with P1 .. P_{S-1} in order, which is the streaming form
 * that keeps one partial resident; this call folds resident partials in one
 * pass.  parts: HOST array of S device pointers (1 <= S <= 64); out may alias
 * parts[0] exactly (no other overlap).
 * ------------------------------------------------------------------------ */
int repro_running_sum(const float* const* parts, int S, int64_t n, float* out,
                      void* stream);

/* ------------------------------------------------------------------------
 * TreeFold ([limits], level 3: the replica all-reduce replayed on one device,
 * pairing partials in the order of a recursive-doubling all-reduce).  With
 * p' = largest power of two <= R and r = R - p': survivors are
 * [P0(+)P1, ..., P_{2r-2}(+)P_{2r-1}, P_{2r}, ..., P_{R-1}]; then for
 * d = 1, 2, ..., p'/2 survivor j is combined with survivor j XOR d; the
 * result is survivor 0 (equal on every rank).  For R = 2^k this is the
 * adjacent-pair tree.
 * parts: HOST array of R device pointers, each to n floats (any memory
 * placement; only the logical order of the array matters); out: n floats and
 * may alias parts[0] exactly (no other overlap).  1 <= R <= 64.
 * ------------------------------------------------------------------------ */
int repro_treefold(const float* const* parts, int R, int64_t n, float* out,
                   void* stream);

/* ------------------------------------------------------------------------
 * Optimiser step after TreeFold ([limits]: AdamW, beta1 0.9, beta2 0.95,
 * eps 1e-8, decoupled weight decay 0.1, global L2-norm clipping at 1.0).
 * The pages fix no operation order; the library's is (binary32, rounded and
 * flushed, never fused):
 *   repro_sumsq: out = canonical sum of g_i (x) g_i over the flat gradient.
 *   repro_adamw_step, per element, with norm = sqrt(*sumsq):
 *     coef = min(max_norm (/) (norm (+) 1e-6), 1);  g' = g (x) coef
 *     m = (b1 (x) m) (+) ((1 (-) b1) (x) g')
 *     v = (b2 (x) v) (+) ((1 (-) b2) (x) (g' (x) g'))
 *     p = (p (x) (1 (-) lr (x) wd)) (-) lr (x) ((m (/) (1 (-) b1^t)) (/)
 *                                             (sqrt(v (/) (1 (-) b2^t)) (+) eps))
 *   where b^t is computed by right-to-left binary exponentiation with rounded
 *   multiplies and t >= 1 is the step number.  p, m, v are updated in place;
 *   all are n floats (device), sumsq 1 float (device), hp a HOST struct.
 *   The learning rate schedule belongs to the caller (lr per call).
 * ------------------------------------------------------------------------ */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay, max_norm;
} repro_adamw_hparams;
int repro_sumsq(const float* g, int64_t n, float* out, void* ws, size_t ws_bytes,
                void* stream);
size_t repro_sumsq_ws_bytes(int64_t n);
int repro_adamw_step(float* p, float* m, float* v, const float* g, int64_t n,
                     const float* sumsq, const repro_adamw_hparams* hp, int64_t t,
                     void* stream);

/* ------------------------------------------------------------------------
 * Attention with int8 P.V ([use]: inside flash attention the P.V product runs
 * on int8 while the QK^T logits and the softmax stay in high precision).  The
 * pages fix no order; the library's, per query row i of head h (every
 * operation binary32, rounded, subnormals flushed, never fused):
 *   keys j in [lo_i, i]: causal, lo_i = max(0, i - W + 1) for a sliding
 *     window of W tokens (W = 0: full causal); head h reads kv head
 *     h / (Hq / Hkv) (grouped-query attention);
 *   s_ij = canon_d(q_id (x) k_jd) (x) c, c = 1 (/) sqrt(128);
 *   m_i = max_j s_ij, exact (a zero maximum is +0);
 *   p_ij = exp_r(s_ij (-) m_i), where exp_r is Cody-Waite range reduction
 *     with ln 2 = 0x1.63p-1 + (-0x1.bd0106p-13), k = rint(x (x) 0x1.715476p+0),
 *     r = (x (-) k (x) C1) (-) k (x) C2, the degree-7 Taylor polynomial in
 *     Horner form with coefficients RN(1/n!), times 2^k (0 for k < -126);
 *   l_i = canon_j(p_ij), j ascending from lo_i;
 *   P_ij = clamp(rint(p_ij (x) 127), 0, 127) (int8), and with V as int8 codes
 *     V_q and per-tensor scale s_v (repro_wscale AMAX + repro_quant_i8):
 *   o_id = (i2f(sum_j P_ij V_q,jd) (x) s_v) (/) (l_i (x) 127), the integer
 *     sum exact.
 * q, o: [B][T][Hq][128] fp32; k: [B][T][Hkv][128] fp32; vq: [B][T][Hkv][128]
 * int8; s_v: 1 float (device); m, l: [B][T][Hq] fp32 outputs (row maxima and
 * sums, the backward's inputs).  All DEVICE pointers, 16-byte aligned (m, l
 * and s_v 4-byte).  D must be 128, Hq a multiple of Hkv, T <= 131072 (the
 * exact int32 P.V bound), B and Hq <= 65535 (REPRO_ERR_SHAPE otherwise).
 * o, m, l must not overlap the inputs or each other (REPRO_ERR_ALIAS).
 * The exact maximum needs the logits twice.  ws (optional, DEVICE): with at
 * least repro_attn_fwd_ws_bytes(B, T, Hq, W) bytes the first pass stores its
 * logits there and the second reads them back and replaces each by
 * p_ij = e^(s_ij - m_i) (0 for masked pairs), which repro_attn_bwd can reuse;
 * with ws == NULL the second pass recomputes the logits.  Same bits either way.
 * With the cache, P.V runs on the tensor cores (the int8 codes as bf16 into
 * tcgen05 kind::f16, fp32 accumulation over exact slices of 512 keys, each
 * converted to int32) on a device whose forward exactness check has passed
 * (repro_linear_fwd: run here in `ws` if it has not run yet, when ws holds at
 * least repro_selftest_ws_bytes()); otherwise, and without the cache, with
 * dp4a on CUDA cores.  The integer sum, and so every bit, is the same.  The cache holds every visited
 * 64 x 64 logit tile: about 4 * 64 * (W + 64) bytes per query row and head for a
 * window W, 2 * T bytes per query row and head for full causal.
 * ------------------------------------------------------------------------ */
#define REPRO_ATTN_HEAD_DIM 128
#define REPRO_ATTN_MAX_T 131072
int repro_attn_fwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                   float* o, float* m, float* l, int64_t B, int64_t T, int64_t Hq,
                   int64_t Hkv, int64_t D, int64_t W, void* ws, size_t ws_bytes,
                   void* stream);
size_t repro_attn_fwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W);

/* ------------------------------------------------------------------------
 * Attention backward ([use]: the attention backward accumulates dQ in 64-bit
 * fixed point for reproducibility).  Straight-through for the quantisation
 * of P and V; the library's order, with p recomputed from the forward's m:
 *   a_ij = p_ij (/) l_i;  V^_jd = i2f(V_q,jd) (x) s_v;
 *   Dr_i = canon_d(dO_id (x) O_id);  dA_ij = canon_d(dO_id (x) V^_jd);
 *   dS_ij = a_ij (x) (dA_ij (-) Dr_i);
 *   dQ_id = fix2f(sum over 64-aligned key tiles t of fx(S_t)) (x) c, where
 *     S_t is the left-to-right sum over the valid keys of tile t of
 *     dS_ij (x) k_jd (seeded with the first term), fx(x) = the nearest int64
 *     to x * 2^48 (ties to even, saturating, NaN to 0) and
 *     fix2f(A) = i2f(A) * 2^-48, flushed: the key tiles' partials meet in
 *     64-bit fixed point, exactly and in any order (the int64 sum wraps
 *     modulo 2^64 if saturated partials overflow it);
 *   dK_jd = F_K (x) c and dV_jd = F_V, where the terms dS_ij (x) q_id (F_K)
 *     and a_ij (x) dO_id (F_V) run over the query heads of kv head g in
 *     ascending order and, within a head, over the valid queries i, grouped
 *     by 64-aligned query tile; each group is summed left to right from its
 *     first term and the group partials are folded left in (head, tile) order.
 * Inputs as repro_attn_fwd plus o (its output), dout [B][T][Hq][128] and its
 * m, l; outputs dq [B][T][Hq][128], dk, dv [B][T][Hkv][128] (DEVICE, 16-byte
 * aligned, no overlaps).  ws: repro_attn_bwd_ws_bytes(B, T, Hq, W) bytes, not
 * overlapping anything else: the Dr_i and, without fwd_ws, the int64 dQ
 * accumulator; with fwd_ws also the a_ij and dS_ij tiles of the window and
 * flushed copies of K, V^, Q and dO laid out for the three kernels of that
 * route.  A call without fwd_ws needs only the first
 * repro_attn_bwd_ws_bytes(B, T, Hq, -1) bytes.
 * fwd_ws (optional): the cache repro_attn_fwd filled for these same inputs,
 * unchanged since (read only); the backward then reads p_ij from it instead
 * of computing the logits and e^x again (same bits).  NULL recomputes.
 * ------------------------------------------------------------------------ */
int repro_attn_bwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                   const float* o, const float* dout, const float* m, const float* l,
                   float* dq, float* dk, float* dv, int64_t B, int64_t T, int64_t Hq,
                   int64_t Hkv, int64_t D, int64_t W, void* ws, size_t ws_bytes,
                   const void* fwd_ws, size_t fwd_ws_bytes, void* stream);
size_t repro_attn_bwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W);

/* ------------------------------------------------------------------------
 * Per-step state hash ([rit] paragraph 4, [limits]: a hash of the state is
 * recorded after every step and a replay must reproduce it; the pages hash on
 * the host and name on-device hashing as future work).  The pages fix no
 * construction; the library's is the Merkle Tree Hash of RFC 6962 section
 * 2.1 over SHA-256 (FIPS 180-4):
 *   leaves: each buffer cut into REPRO_HASH_LEAF_BYTES consecutive bytes (the
 *     last leaf of a buffer may be shorter; an empty buffer has none), the
 *     buffers' leaves in buffer order;
 *   MTH({}) = SHA-256(""), MTH({d}) = SHA-256(0x00 || d),
 *   MTH(D[0:n]) = SHA-256(0x01 || MTH(D[0:k]) || MTH(D[k:n])), k the largest
 *     power of two below n.
 * bufs, nbytes: HOST arrays of nbuf (0 .. REPRO_HASH_MAX_BUFFERS) device
 *   pointers (16-byte aligned; NULL allowed when the size is 0) and byte
 *   counts.  digest: 32 bytes of DEVICE memory (16-byte aligned), written in
 *   the standard SHA-256 byte order.  ws: repro_state_hash_ws_bytes bytes
 *   (0 for a single leaf), not overlapping the buffers or the digest.
 * Hashing is integer work: the bits never depend on the launch.
 * ------------------------------------------------------------------------ */
#define REPRO_HASH_LEAF_BYTES 4096
#define REPRO_HASH_MAX_BUFFERS 64
int repro_state_hash(const void* const* bufs, const int64_t* nbytes, int nbuf,
                     uint8_t* digest, void* ws, size_t ws_bytes, void* stream);
size_t repro_state_hash_ws_bytes(const int64_t* nbytes, int nbuf);

/* ------------------------------------------------------------------------
 * Housekeeping.
 * repro_status_str: static description of a status code.
 * repro_version: REPRO_VERSION.
 * repro_device_check: synchronises `stream`, then reads and clears the
 *   device error word set by bounded device-side waits; returns REPRO_OK,
 *   REPRO_ERR_TIMEOUT, or REPRO_ERR_SELFTEST once after the forward's
 *   exactness check failed on the current device (REPRO_ERR_LAUNCH if the
 *   stream reported an error).
 * repro_launch_count: number of kernels this library has enqueued in this
 *   process (all devices, all streams); a diagnostic for counting launches.
 * repro_set_launch_cfg: test hook that changes how work is split across
 *   thread blocks (never the arithmetic); NULL restores the defaults.  Used
 *   to show that results do not depend on the launch configuration.  Not
 *   thread-safe; affects subsequent calls in this process.
 * ------------------------------------------------------------------------ */
typedef struct {
    int bwd_segment_log2;   /* -1: chosen per shape (whole-wave CTA counts); else 2^k chunks
                               per backward reduction segment (0..8) */
    int reduce_block_log2;  /* -1: default; else 2^k chunk partials per block in repro_wscale (0..10) */
    int fwd_path;           /* -1: default (tensor cores, 128 x 256 output tiles, when K % 8 == 0);
                               0: CUDA cores; 1: tensor cores, 128 x 256 tiles; 2: tensor cores,
                               128 x 128 tiles */
    int elementwise_blocks; /* -1 or 0: default; else grid size of streaming kernels, of
                               the weight scale's first pass and of the activation-scale
                               pass (that one capped at the ceil(n / 64) + 64 partial
                               slots of its workspace) */
    int bwd_kernel;         /* -1: default (8); 8: operands prepared once per call, then fed
                               to the products by tensor copies (needs 16-byte-aligned rows:
                               N % 4 == 0 and K % 16 == 0, else 1 runs); 1: register-prefetch
                               kernel, any row alignment.  Other values: REPRO_ERR_ARG */
    int fwd_selftest;       /* -1: default (the tensor-core forward runs only on a device whose
                               exactness self-test has passed, see repro_linear_fwd); 1: test
                               hook that acts as if the self-test had failed on every device */
} repro_launch_cfg;

/* ------------------------------------------------------------------------
 * Allocation-free scale, for callers that cannot hand the library any device
 * memory: code whose device allocations all belong to another owner (a host
 * application's private pool, a plugin without allocator hooks), or a loop
 * that must never call cudaMalloc because that would synchronise the device.
 * The pages have no counterpart: this is an interface convenience only, with
 * the same arithmetic and the same bits as repro_wscale.
 * Same arguments and results as repro_wscale, minus the workspace: the
 * scratch is a fixed array of REPRO_NOALLOC_SCRATCH_FLOATS floats (256 KB)
 * inside the library, held by every GPU that loads the library until the
 * process exits.  n may be at most REPRO_NOALLOC_MAX_N (REPRO_ERR_SHAPE
 * otherwise); the block split is always the default one.  Each call outside
 * a stream capture looks up the array's device address on the current device
 * (so a cudaDeviceReset is picked up by the next such call); a call made
 * during a capture reuses the address the last lookup on that device found,
 * so the first call on a device must come before any stream capture (a first
 * call inside a capture returns REPRO_ERR_LAUNCH and launches nothing).
 * Calls share the array and race if their work overlaps on the GPU; nothing
 * in it needs clearing.  Allocates nothing.
 * ------------------------------------------------------------------------ */
#define REPRO_NOALLOC_SCRATCH_FLOATS 65536
#define REPRO_NOALLOC_MAX_N 535822336LL   /* 65408 blocks of 8192 elements */
int repro_wscale_noalloc(const float* x, int64_t n, int mode, int qmax, float* scale_out,
                         void* stream);

const char* repro_status_str(int status);

/* ------------------------------------------------------------------------
 * Exactness self-test of the tensor-core forward ([use]: the int8 forward
 * must be exact).  The forward's tensor-core path relies on fp32 accumulation
 * over 512-term K-slices of integer products staying exact, which the
 * hardware documentation does not state; this runs it and the CUDA-core
 * (dp4a) path on adversarial codes (all at the clamp, alternating signs, a
 * sign flip at the slice boundary, a slice whose running sum reaches
 * 511 * 127 * 127 just below 2^23 before a product of +-1, hashed codes;
 * 128 x 256 outputs, K = 1024,
 * unit scales) and compares every output bit, for both tensor-core tile
 * widths (128 x 256, the default, and 128 x 128).  Synchronises `stream`.  ws: device workspace of
 * repro_selftest_ws_bytes() bytes.  Returns REPRO_OK, REPRO_ERR_SELFTEST on a
 * mismatch, or an argument / launch error.  The result also decides, for the
 * current device, whether later default-path forwards use the tensor cores.
 * ------------------------------------------------------------------------ */
int repro_selftest(void* ws, size_t ws_bytes, void* stream);
size_t repro_selftest_ws_bytes(void);
/* ------------------------------------------------------------------------
 * Failure-detection hook.  Every pipeline wait in the library is bounded: a
 * wait that is not satisfied within about two seconds at the boost clock
 * sets the device error word, lets the kernel return, and is reported by
 * repro_device_check() as REPRO_ERR_TIMEOUT, leaving the CUDA context usable
 * (REPRO_ERR_NONFINITE is the debug mode's report, see repro_set_debug).
 * repro_wait_probe enqueues one thread that performs that same bounded wait
 * on a shared-memory barrier phase which completes only when `arrive` is 1.
 * With arrive = 0 nothing completes it, so the wait runs out (about two
 * seconds) and the next repro_device_check() returns REPRO_ERR_TIMEOUT (and
 * clears the word); with arrive = 1 it returns at once and sets nothing.
 * Enqueues only.  arrive outside {0, 1} -> REPRO_ERR_ARG.
 * ------------------------------------------------------------------------ */
int repro_wait_probe(int arrive, void* stream);

/* ------------------------------------------------------------------------
 * Debug checks, all off by default (flags = 0).  Non-finite inputs are
 * outside the method's contract (the calls still compute their documented
 * results for them: a NaN quotient quantises to 0, a NaN logit is passed over
 * by the row maximum, and so on); this mode finds where they enter.
 *   REPRO_DEBUG_CHECK_FINITE: every call that reads float tensors or scales
 *     first enqueues, on its own stream, one scan of each of them (an extra
 *     read of every such input); a NaN or an infinity sets the device error
 *     word, and the next repro_device_check() returns REPRO_ERR_NONFINITE (a
 *     bounded wait that gave up in the same interval reports
 *     REPRO_ERR_TIMEOUT instead).  The scan does not stop the call.
 * Process-wide, like the launch configuration.  Unknown flags ->
 * REPRO_ERR_ARG.
 * ------------------------------------------------------------------------ */
#define REPRO_DEBUG_CHECK_FINITE 1
int repro_set_debug(int flags);
int repro_version(void);
int repro_device_check(void* stream);
uint64_t repro_launch_count(void);
int repro_set_launch_cfg(const repro_launch_cfg* cfg);

#ifdef __cplusplus
}
#endif
#endif /* REPRO_H */
