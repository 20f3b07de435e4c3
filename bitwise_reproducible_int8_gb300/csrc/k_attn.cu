// k_attn.cu -- attention with int8 P.V: inside flash attention the P.V
// product runs on int8 while the QK^T logits and the softmax stay in high
// precision (Open-1B review, onedev.kr/papers/92, section "How to use").
// The pages fix no operation order; the library's (every operation binary32,
// rounded, subnormal operands and results flushed, no fused multiply-add):
//   s_ij = canon_d(q_id (x) k_jd) (x) c,  c = 1 (/) sqrt(128)
//   keys of row i: j in [lo_i, i], lo_i = max(0, i - W + 1) (W = 0: lo_i = 0);
//   query head h reads kv head h / (Hq / Hkv)
//   m_i  = max_j s_ij (exact; a zero maximum is +0)
//   p_ij = exp_r(s_ij (-) m_i),  l_i = canon_j(p_ij), j ascending from lo_i
//   P_ij = clamp(rint(p_ij (x) 127), 0, 127)
//   o_id = (i2f(sum_j P_ij V_q,jd) (x) s_v) (/) (l_i (x) 127), the sum exact
// exp_r: Cody-Waite range reduction (ln 2 = 355/512 + RN(ln 2 - 355/512)),
// degree-7 Taylor polynomial in Horner form with RN(1/n!) coefficients, exact
// scaling by 2^k.
//
// The row maximum must be exact before any p is quantised, so the forward
// visits the key tiles of the window twice: pass 1 computes the logits and the
// row maxima, pass 2 forms p and the int8 codes, streams the row sums through
// the canonical-order chunk/tree stack (one thread per row) and accumulates
// P.V exactly.  Two routes:
//   * with the logit cache and a device whose tensor-core exactness check has
//     passed (the default): k_attn_rows<false> (pass 1) and k_attn_pv (pass 2, P.V
//     on the tensor cores), described before them below;
//   * otherwise k_attn_fwd: one CTA per (64-row query tile, query head,
//     sequence) runs both passes; pass 2 reads the cached logits or recomputes
//     them, and P.V runs on dp4a (exact int32).  Logits: 256 threads own 4 x 4
//     outputs each, packed f32x2 products over d with the chunk-of-64 order.
#include <type_traits>

#include "bwd_tile.cuh"
#include "common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace repro {
namespace {

typedef unsigned long long u64;

constexpr int AT = 64;       // query and key tile
constexpr int HD = 128;      // head dimension
constexpr int PT = 68;       // pitch (floats) of the transposed q / k tiles
constexpr int PS = 65;       // pitch of the p tile
constexpr int PP = 17;       // pitch (words) of the packed int8 P tile
constexpr int MAXL = 24;     // stack levels of the row-sum tree
constexpr int NT = 256;

struct AttnFwdArgs {
    const float* q;
    const float* k;
    const int8_t* vq;
    const float* s_v;
    float* o;
    float* m;
    float* l;
    float* cache;      // optional: pass-1 logits, read back by pass 2 (NULL: recompute)
    int64_t T, Hq, Hkv, W;
    int64_t tiles_bh;  // cached logit tiles per (sequence, head)
    float c;
    int* err;          // device error word (bounded waits of the tensor-core P.V)
};

// key tiles visited by query tiles 0 .. qt-1 (tile u visits tiles
// max(0, 64u - W + 1) / 64 .. u): the offset of query tile qt's logits in the
// per-(sequence, head) cache, in 64 x 64 tiles
__host__ __device__ __forceinline__ int64_t tile_prefix(int64_t qt, int64_t W)
{
    if (W <= 0)
        return qt * (qt + 1) / 2;
    const int64_t D = W - 1;
    const int64_t c1 = (D + 63) / 64;   // every tile past the first ones visits c1 + 1 tiles
    const int64_t us = D / 64 + 1;      // first query tile whose window starts after key 0
    const int64_t mq = qt < us ? qt : us;
    return mq * (mq + 1) / 2 + (qt > us ? (qt - us) * (c1 + 1) : 0);
}

constexpr size_t FWD_SMEM = (size_t)(2 * HD * PT + AT * PS) * 4 + (size_t)(AT * PP) * 4 +
                            (size_t)(AT / 4 * HD) * 4 + (size_t)(AT * (MAXL + 1)) * 4 +
                            (size_t)(3 * AT) * 4;

// pass 1's second key tile lives in pass 2's scratch (Ps .. stk)
static_assert(HD * PT <= AT * PS + AT * PP + AT / 4 * HD + AT * (MAXL + 1),
              "second key tile does not fit in the pass-2 scratch");

// e^x: the reduction, polynomial and scaling stated above
__device__ __forceinline__ float exp_r(float x)
{
    x = flush(x);
    const float kf = rintf(fmul_flush(x, 0x1.715476p+0f));
    const float r = fadd_ftz(fadd_ftz(x, -fmul_flush(kf, 0x1.63p-1f)),
                             -fmul_flush(kf, -0x1.bd0106p-13f));
    float p = 0x1.a01a02p-13f;
    p = fadd_ftz(fmul_rn(p, r), 0x1.6c16c2p-10f);
    p = fadd_ftz(fmul_rn(p, r), 0x1.111112p-7f);
    p = fadd_ftz(fmul_rn(p, r), 0x1.555556p-5f);
    p = fadd_ftz(fmul_rn(p, r), 0x1.555556p-3f);
    p = fadd_ftz(fmul_rn(p, r), 0.5f);
    p = fadd_ftz(fmul_rn(p, r), 1.0f);
    p = fadd_ftz(fmul_rn(p, r), 1.0f);
    if (kf < -126.0f)
        return 0.0f;
    if (kf > 254.0f)
        return __int_as_float(0x7f800000);
    const int k = (int)kf;
    if (k > 127)
        return flush(fmul_rn(fmul_rn(p, 0x1p127f), __int_as_float((k - 127 + 127) << 23)));
    return flush(fmul_rn(p, __int_as_float((k + 127) << 23)));
}

// e^x of two lanes: the same operations as exp_r, lane by lane, with the
// reduction and the polynomial on packed pairs
__device__ __forceinline__ float exp_scale(float p, float kf)
{
    if (kf < -126.0f)
        return 0.0f;
    if (kf > 254.0f)
        return __int_as_float(0x7f800000);
    const int k = (int)kf;
    if (k > 127)
        return flush(fmul_rn(fmul_rn(p, 0x1p127f), __int_as_float((k - 127 + 127) << 23)));
    return flush(fmul_rn(p, __int_as_float((k + 127) << 23)));
}

__device__ __forceinline__ u64 exp_r2(u64 x)
{
    const u64 z = pack2(-0.0f, -0.0f);
    x = fadd2_ftz(x, z);
    float t0, t1;
    unpack2(fadd2_ftz(fmul2_rn(x, pack2(0x1.715476p+0f, 0x1.715476p+0f)), z), t0, t1);
    const float k0 = rintf(t0), k1 = rintf(t1);
    const u64 kf = pack2(k0, k1);
    // x (-) RN(kf c1), then (-) RN(kf c2); the negated products are RN(kf (-c))
    const u64 r = fadd2_ftz(fadd2_ftz(x, fadd2_ftz(fmul2_rn(kf, pack2(-0x1.63p-1f, -0x1.63p-1f)), z)),
                            fadd2_ftz(fmul2_rn(kf, pack2(0x1.bd0106p-13f, 0x1.bd0106p-13f)), z));
    u64 p = pack2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
    p = fadd2_ftz(fmul2_rn(p, r), pack2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = fadd2_ftz(fmul2_rn(p, r), pack2(0x1.111112p-7f, 0x1.111112p-7f));
    p = fadd2_ftz(fmul2_rn(p, r), pack2(0x1.555556p-5f, 0x1.555556p-5f));
    p = fadd2_ftz(fmul2_rn(p, r), pack2(0x1.555556p-3f, 0x1.555556p-3f));
    p = fadd2_ftz(fmul2_rn(p, r), pack2(0.5f, 0.5f));
    p = fadd2_ftz(fmul2_rn(p, r), pack2(1.0f, 1.0f));
    p = fadd2_ftz(fmul2_rn(p, r), pack2(1.0f, 1.0f));
    // 2^k exactly as a normal float for -126 <= k <= 127: both lanes scale in
    // one packed multiply; any other lane takes exp_scale's branches
    if (k0 >= -126.0f && k0 <= 127.0f && k1 >= -126.0f && k1 <= 127.0f) {
        const u64 sc = pack2(__int_as_float(((int)k0 + 127) << 23), __int_as_float(((int)k1 + 127) << 23));
        return fadd2_ftz(fmul2_rn(p, sc), z);
    }
    float p0, p1;
    unpack2(p, p0, p1);
    return pack2(exp_scale(p0, k0), exp_scale(p1, k1));
}

// the int8 code of p as a float: rint(p (x) 127) clamped to [0, 127] (quant_p)
__device__ __forceinline__ float quant_pf(float t)
{
    return fminf(fmaxf(rintf(t), 0.0f), 127.0f);
}

__device__ __forceinline__ int quant_p(float p)
{
    float r = rintf(fmul_flush(p, 127.0f));
    r = fminf(fmaxf(r, 0.0f), 127.0f);
    return (int)r;
}

// tile of 64 rows x 128 floats of a [.., H, 128] tensor, flushed and
// transposed into t[d][r] (pitch PT); rows outside [0, T) read as 0.
// Warp lanes cover 8 rows x 4 float4 columns per step; step it covers
// d = 16 it .. 16 it + 15, so steps 0-3 and 4-7 are the two halves of d.
// tile_fetch / tile_put split one half into its global loads and its shared
// stores, so the loads of the next tile can be in flight during a product
__device__ __forceinline__ void tile_fetch(float4 (&v)[4], const float* __restrict__ src,
                                           int64_t row0, int64_t T, int64_t row_stride, int tid,
                                           int half)
{
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int it = 4 * half + u;
        const int e = tid + it * NT;            // 2048 float4 pieces
        const int lane = e & 31, w = e >> 5;    // w: 64 groups of 8 rows x 4 columns
        const int r = (w & 7) * 8 + (lane & 7);
        const int c4 = (w >> 3) * 4 + (lane >> 3);
        const int64_t row = row0 + r;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row >= 0 && row < T)
            v[u] = *reinterpret_cast<const float4*>(src + row * row_stride + 4 * c4);
    }
}

__device__ __forceinline__ void tile_put(float* __restrict__ t, const float4 (&v)[4], int tid,
                                         int half)
{
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int it = 4 * half + u;
        const int e = tid + it * NT;
        const int lane = e & 31, w = e >> 5;
        const int r = (w & 7) * 8 + (lane & 7);
        const int c4 = (w >> 3) * 4 + (lane >> 3);
        const float4 f = flush4(v[u]);
        t[(4 * c4 + 0) * PT + r] = f.x;
        t[(4 * c4 + 1) * PT + r] = f.y;
        t[(4 * c4 + 2) * PT + r] = f.z;
        t[(4 * c4 + 3) * PT + r] = f.w;
    }
}

__device__ __forceinline__ void load_tile_t(float* __restrict__ t, const float* __restrict__ src,
                                            int64_t row0, int64_t T, int64_t row_stride, int tid)
{
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float4 v[4];
        tile_fetch(v, src, row0, T, row_stride, tid, half);
        tile_put(t, v, tid, half);
    }
}

// the thread's 4 x 4 logits: rows 4ty..4ty+3 (as 2 packed pairs), columns
// 4tx..4tx+3; canonical order over d: two chunks of 64, then one pairwise add.
// logit_chunk is one chunk's left-to-right sum (d0 = 0 or 64), logit_finish the
// pairwise add and the scaling
__device__ __forceinline__ void logit_chunk(u64 (&acc)[8], const float* __restrict__ Qt,
                                            const float* __restrict__ Kt, int ty, int tx, int d0)
{
    // operands are loaded one step ahead of their products
    const float* qp = Qt + 4 * ty;
    const float* kp = Kt + 4 * tx;
    ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(qp + d0 * PT);
    float4 kb = *reinterpret_cast<const float4*>(kp + d0 * PT);
    {
        const u64 P[2] = {qa.x, qa.y};
        const u64 D[4] = {pack2(kb.x, kb.x), pack2(kb.y, kb.y), pack2(kb.z, kb.z),
                          pack2(kb.w, kb.w)};
        qa = *reinterpret_cast<const ulonglong2*>(qp + (d0 + 1) * PT);
        kb = *reinterpret_cast<const float4*>(kp + (d0 + 1) * PT);
#pragma unroll
        for (int ip = 0; ip < 2; ++ip)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[ip * 4 + j] = fmul2_rn(P[ip], D[j]);
    }
#pragma unroll 9
    for (int dd = 1; dd < 64; ++dd) {
        const u64 P[2] = {qa.x, qa.y};
        const u64 D[4] = {pack2(kb.x, kb.x), pack2(kb.y, kb.y), pack2(kb.z, kb.z),
                          pack2(kb.w, kb.w)};
        const int dn = d0 + (dd + 1 < 64 ? dd + 1 : dd);
        qa = *reinterpret_cast<const ulonglong2*>(qp + dn * PT);
        kb = *reinterpret_cast<const float4*>(kp + dn * PT);
#pragma unroll
        for (int ip = 0; ip < 2; ++ip)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[ip * 4 + j] = fadd2_ftz(acc[ip * 4 + j], fmul2_rn(P[ip], D[j]));
    }
}

__device__ __forceinline__ void logit_finish(u64 (&s)[8], const u64 (&t0)[8], const u64 (&t1)[8],
                                             float c)
{
    const u64 cc = pack2(c, c);
#pragma unroll
    for (int e = 0; e < 8; ++e)   // (x) c, flushed
        s[e] = fadd2_ftz(fmul2_rn(fadd2_ftz(t0[e], t1[e]), cc), pack2(-0.0f, -0.0f));
}

__device__ __forceinline__ void logits4x4(u64 (&s)[8], const float* __restrict__ Qt,
                                          const float* __restrict__ Kt, int ty, int tx, float c)
{
    u64 t0[8], t1[8];
    logit_chunk(t0, Qt, Kt, ty, tx, 0);
    logit_chunk(t1, Qt, Kt, ty, tx, 64);
    logit_finish(s, t0, t1, c);
}

// logit (row 4ty + 2ip + h, column 4tx + j) is lane h of s[ip*4 + j]
__device__ __forceinline__ float lane_of(const u64 (&s)[8], int ip, int j, int h)
{
    float lo, hi;
    unpack2(s[ip * 4 + j], lo, hi);
    return h ? hi : lo;
}

// P.V on the tensor cores (the default forward route, k_attn_pv below): per
// 64-key tile the P codes go to shared memory as bf16 (exact for 0..127) in
// the 128-byte-swizzled K-major layout of umma.cuh, rows 0-63 and again as
// rows 64-127, beside V^T[d][key] likewise; one thread issues tcgen05.mma
// kind::f16, M = 128, N = 128, K = 64 (four K = 16 steps) into a 128-column
// fp32 accumulator in tensor memory.  Every product is an integer of magnitude
// at most 16129, and a row's sum over a slice is exact in fp32 while it stays
// below 2^23: a slice of at most 8 tiles holds at most 512 valid keys of a
// row, and so does any slice when W <= 520 (520 x 16129 < 2^23).  After each
// slice the threads convert the accumulator to int32 and add it to their
// registers.  The duplicated rows let all eight warps read the accumulator:
// warp w reads tensor-memory lanes 32 (w % 4) .. + 31, i.e. query row
// 32 (w % 2) + lane, columns 32 (2 ((w % 4) / 2) + w / 4) .. + 31.
constexpr int TC_SLICE_TILES = 8;          // 512 keys per exact slice (W > 520)
constexpr int TC_TILE_BYTES = 128 * 128;   // 128 rows of 64 bf16

// byte offset of element (row, col) in a 128-row x 64-column bf16 tile
__device__ __forceinline__ uint32_t sw128_off(int row, int col)
{
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((col >> 3) ^ (row & 7))) << 4) +
                      ((col & 7) << 1));
}

__device__ __forceinline__ uint32_t bf16_bits(int v)
{
    return __float_as_uint((float)v) >> 16;   // exact: |v| <= 127
}

__global__ void __launch_bounds__(NT, 2) k_attn_fwd(const AttnFwdArgs a)
{
    extern __shared__ __align__(16) float sma[];
    float* Qt = sma;                                       // [HD][PT]
    float* Kt = Qt + HD * PT;                              // [HD][PT]
    float* Ps = Kt + HD * PT;                              // [AT][PS]
    int* Pp = reinterpret_cast<int*>(Ps + AT * PS);        // [AT][PP]
    int* Vp = Pp + AT * PP;                                // [AT/4][HD]
    float* stk = reinterpret_cast<float*>(Vp + AT / 4 * HD);   // [AT][MAXL+1]
    float* mrow = stk + AT * (MAXL + 1);                   // [AT]
    float* lrow = mrow + AT;                               // [AT]

    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int64_t b = blockIdx.z, h = blockIdx.y, i0 = (int64_t)blockIdx.x * AT;
    const int64_t T = a.T, W = a.W;
    const int64_t g = h / (a.Hq / a.Hkv);
    const int64_t qstride = a.Hq * HD, kstride = a.Hkv * HD;
    const float* qbase = a.q + (b * T * a.Hq + h) * HD;
    const float* kbase = a.k + (b * T * a.Hkv + g) * HD;
    const int8_t* vbase = a.vq + (b * T * a.Hkv + g) * HD;

    const int64_t jlo = W > 0 ? max((int64_t)0, i0 - W + 1) : 0;
    const int64_t jhi = min(i0 + AT - 1, T - 1);
    const int64_t t_lo = jlo / AT, t_hi = jhi / AT;
    // this CTA's cached logits: tile t at (t - t_lo) * 4096 floats, thread tid's
    // 16 values (its 4 x 4 outputs as 8 packed pairs) at tid * 16
    float* cache = a.cache ? a.cache + ((b * a.Hq + h) * a.tiles_bh +
                                        tile_prefix((int64_t)blockIdx.x, W)) * (AT * AT)
                           : nullptr;

    load_tile_t(Qt, qbase, i0, T, qstride, tid);

    // ---------------------------------------------------------- pass 1: maxima
    // the key tiles alternate between Kt and K2 (pass 2's scratch, idle until
    // then); tile t + 1 is fetched while tile t's logits are formed, so each
    // tile needs one barrier
    float* K2 = Ps;
    {
        float4 v[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tile_fetch(v, kbase, t_lo * AT, T, kstride, tid, half);
            tile_put(Kt, v, tid, half);
        }
    }
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for (int64_t t = t_lo; t <= t_hi; ++t) {
        const int64_t j0 = t * AT;
        const bool odd = ((t - t_lo) & 1) != 0;
        const float* Kc = odd ? K2 : Kt;
        float* Kn = odd ? Kt : K2;
        const bool more = t < t_hi;
        __syncthreads();   // tile t is in Kc, and every reader of Kn (tile t - 1) is done
        u64 s[8];
        {
            u64 t0[8], t1[8];
            float4 v[4];
            if (more)
                tile_fetch(v, kbase, j0 + AT, T, kstride, tid, 0);
            logit_chunk(t0, Qt, Kc, ty, tx, 0);
            if (more) {
                tile_put(Kn, v, tid, 0);
                tile_fetch(v, kbase, j0 + AT, T, kstride, tid, 1);
            }
            logit_chunk(t1, Qt, Kc, ty, tx, 64);
            if (more)
                tile_put(Kn, v, tid, 1);
            logit_finish(s, t0, t1, a.c);
        }
        if (cache) {
            ulonglong2* dst = reinterpret_cast<ulonglong2*>(cache + (t - t_lo) * (AT * AT) + tid * 16);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_ulonglong2(s[2 * e], s[2 * e + 1]);
        }
#pragma unroll
        for (int ip = 0; ip < 2; ++ip)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int rr = 2 * ip + hh;
                const int64_t i = i0 + 4 * ty + rr;
                const int64_t lo = W > 0 ? max((int64_t)0, i - W + 1) : 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t jj = j0 + 4 * tx + j;
                    if (i < T && jj >= lo && jj <= i)
                        mx[rr] = fmaxf(mx[rr], lane_of(s, ip, j, hh));
                }
            }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], off));
        if (mx[rr] == 0.0f)
            mx[rr] = 0.0f;   // a zero maximum is +0
    }
    if (tx == 0)
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
            mrow[4 * ty + rr] = mx[rr];

    // ------------------------------------- pass 2: p, codes, row sums and P.V
    // row-sum state (threads 0..63, one query row each)
    const int64_t my_i = i0 + tid;
    const int64_t my_lo = W > 0 ? max((int64_t)0, my_i - W + 1) : 0;
    const int64_t my_n = my_i - my_lo + 1;
    int64_t pos = 0;
    float cs = 0.f, lsum = 0.f;

    // P.V outputs of this thread: rows 4ri..4ri+3, d 8di..8di+7, acc[r][u]
    const int ri = tid >> 4, di = tid & 15;
    int acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int u = 0; u < 8; ++u)
            acc[r][u] = 0;

    for (int64_t t = t_lo; t <= t_hi; ++t) {
        const int64_t j0 = t * AT;
        __syncthreads();   // Kt, Ps, Pp, Vp free
        if (!cache)
            load_tile_t(Kt, kbase, j0, T, kstride, tid);
        // V codes as packed words: Vp[jq][d] = bytes of keys 4jq .. 4jq+3 at column d
#pragma unroll
        for (int it = 0; it < (AT / 4 * HD / 4) / NT; ++it) {
            const int e = tid + it * NT;             // 512 items: jq (16) x d4 (32)
            const int jq = e >> 5, d4 = e & 31;
            int w[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int64_t jj = j0 + 4 * jq + kk;
                w[kk] = jj < T ? *reinterpret_cast<const int*>(vbase + jj * kstride + 4 * d4) : 0;
            }
            const int lo01 = __byte_perm(w[0], w[1], 0x5140), hi01 = __byte_perm(w[0], w[1], 0x7362);
            const int lo23 = __byte_perm(w[2], w[3], 0x5140), hi23 = __byte_perm(w[2], w[3], 0x7362);
            int4 out;
            out.x = __byte_perm(lo01, lo23, 0x5410);   // d = 4 d4 + 0
            out.y = __byte_perm(lo01, lo23, 0x7632);   // d = 4 d4 + 1
            out.z = __byte_perm(hi01, hi23, 0x5410);   // d = 4 d4 + 2
            out.w = __byte_perm(hi01, hi23, 0x7632);   // d = 4 d4 + 3
            *reinterpret_cast<int4*>(Vp + jq * HD + 4 * d4) = out;
        }
        __syncthreads();
        {
            u64 s[8];
            if (cache) {
                const ulonglong2* src =
                    reinterpret_cast<const ulonglong2*>(cache + (t - t_lo) * (AT * AT) + tid * 16);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const ulonglong2 v = src[e];
                    s[2 * e] = v.x;
                    s[2 * e + 1] = v.y;
                }
            } else {
                logits4x4(s, Qt, Kt, ty, tx, a.c);
            }
            float pv[16];   // this thread's p, in the cache's layout (pair e, lane h at 2e + h)
#pragma unroll
            for (int ip = 0; ip < 2; ++ip)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int rr = 2 * ip + hh;
                    const int r = 4 * ty + rr;
                    const int64_t i = i0 + r;
                    const int64_t lo = W > 0 ? max((int64_t)0, i - W + 1) : 0;
                    const float m = mrow[r];
                    uint32_t word = 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int64_t jj = j0 + 4 * tx + j;
                        float p = 0.f;
                        if (i < T && jj >= lo && jj <= i)
                            p = exp_r(fadd_ftz(lane_of(s, ip, j, hh), -m));
                        Ps[r * PS + 4 * tx + j] = p;
                        pv[2 * (ip * 4 + j) + hh] = p;
                        word |= (uint32_t)quant_p(p) << (8 * j);
                    }
                    Pp[r * PP + tx] = (int)word;
                }
            if (cache) {
                // the cache now holds p in place of each logit: the backward
                // reads p from it instead of evaluating e^x again
                float4* dst = reinterpret_cast<float4*>(cache + (t - t_lo) * (AT * AT) + tid * 16);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(pv[4 * e], pv[4 * e + 1], pv[4 * e + 2], pv[4 * e + 3]);
            }
        }
        __syncthreads();
        // row sums: the valid p of this tile, left to right, through the
        // chunk-of-64 / pairwise-tree stack
        if (tid < AT && my_i < T) {
            const int64_t cb = max(my_lo, j0), ce = min(my_i, j0 + AT - 1);
            const float* prow = Ps + tid * PS;   // column jj - j0
            int64_t jj = cb;
            while (jj <= ce) {
                // one run up to the next chunk boundary: left to right, seeded
                // with the chunk's first term
                const int room = 64 - (int)(pos & 63);
                const int len = (int)min((int64_t)room, ce - jj + 1);
                int k = 0;
                const float* pr = prow + (int)(jj - j0);
                if ((pos & 63) == 0) {
                    cs = pr[0];
                    k = 1;
                }
#pragma unroll 8
                for (; k < len; ++k)
                    cs = fadd_ftz(cs, pr[k]);
                jj += len;
                pos += len;
                if ((pos & 63) == 0 || pos == my_n) {
                    const int64_t c = (pos - 1) >> 6;
                    float acc_t = cs;
                    if (pos == my_n) {
                        for (int lvl = 0; lvl < MAXL; ++lvl)
                            if ((c >> lvl) & 1)
                                acc_t = fadd_ftz(stk[tid * (MAXL + 1) + lvl], acc_t);
                        lsum = acc_t;
                    } else {
                        const int tz = __ffsll(~c) - 1;
                        for (int lvl = 0; lvl < tz; ++lvl)
                            acc_t = fadd_ftz(stk[tid * (MAXL + 1) + lvl], acc_t);
                        stk[tid * (MAXL + 1) + tz] = acc_t;
                    }
                }
            }
        }
        // P.V, exact: 16 groups of 4 keys
#pragma unroll 4
        for (int jq = 0; jq < AT / 4; ++jq) {
            const int4 v0 = *reinterpret_cast<const int4*>(Vp + jq * HD + 8 * di);
            const int4 v1 = *reinterpret_cast<const int4*>(Vp + jq * HD + 8 * di + 4);
            const int vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int pw = Pp[(4 * ri + r) * PP + jq];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    acc[r][u] = __dp4a(pw, vv[u], acc[r][u]);
            }
        }
    }
    if (tid < AT)
        lrow[tid] = lsum;
    __syncthreads();

    // ---------------------------------------------------------------- epilogue
    const float sv = flush(*a.s_v);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int rr = 4 * ri + r;
        const int64_t i = i0 + rr;
        if (i >= T)
            continue;
        const float den = fmul_flush(lrow[rr], 127.0f);
        float ov[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            ov[u] = flush(__fdiv_rn(fmul_flush(__int2float_rn(acc[r][u]), sv), den));
        float* dst = a.o + ((b * T + i) * a.Hq + h) * HD + 8 * di;
        *reinterpret_cast<float4*>(dst) = make_float4(ov[0], ov[1], ov[2], ov[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(ov[4], ov[5], ov[6], ov[7]);
        if (di == 0) {
            a.m[(b * T + i) * a.Hq + h] = mrow[rr];
            a.l[(b * T + i) * a.Hq + h] = lrow[rr];
        }
    }
}

// ---------------------------------------------------------------------------
// Default forward route (logit cache and tensor-core P.V), two kernels.
//
// k_attn_rows<false>: pass 1 -- every logit of the window written to the cache and
// the exact row maxima written to m -- as a banded product in the canonical
// order over d.  (k_attn_rows<true> is the backward's dA / a / dS pass: the
// same product of dO and V^, described with the backward below.)  A CTA holds two groups of 128 threads; each group takes its
// own query tiles (64 rows, one head, one sequence) in turn.  A thread owns 8
// rows x 4 keys of a 64 x 64 tile (rows as packed pairs: the tile of the
// linear backward, bwd_tile.cuh), so it loads 12 floats per 32 outputs per d.
// The group's Q^T tile is staged once per query tile; the K^T tiles of all its
// query tiles stream through a two-stage ring filled by bulk copies from an
// image of K (k_attn_kimg: per (sequence, kv head, 64-key tile) the flushed
// K^T[d][key], 32 KB) and released per warp on an mbarrier, so no group-wide
// barrier is taken per key tile.  The logits land in the cache in the same
// layout as the other forward route's (4 x 4 blocks of 16 floats), which the
// second pass and the backward read.
//
// k_attn_pv: pass 2 -- p, the int8 codes, the row sums and P.V -- one CTA of
// 256 threads per query tile, two CTAs per SM.  The P and V^T tiles and the p
// tile are double-buffered, so tile t + 1 is written while the MMA of tile t
// runs and the row sums of tile t are read; V^T comes from the image of the V
// codes (k_attn_vimg) by one bulk copy per tile.
constexpr int LG_NT = 256;                       // threads per CTA: two groups
constexpr int LG_G = 128;                        // threads per group
constexpr uint32_t KIMG_TILE = HD * AT * 4;      // bytes of one K^T tile
constexpr int LG_Q_BYTES = HD * PT * 4;          // Q^T [d][64 rows], pitch PT
constexpr int LG_GROUP_BYTES = LG_Q_BYTES + 2 * (int)KIMG_TILE + 2 * AT * 4;   // + l, Dr rows (backward)
constexpr int BT_P = 68;                         // pitch (floats) of the backward's a / dS tiles
constexpr uint32_t BT_TILE = AT * BT_P * 4;      // bytes of one a or dS tile
constexpr size_t LG_SMEM = 2 * (size_t)LG_GROUP_BYTES;
constexpr uint32_t VIMG_TILE = 128 * 64 * 2;     // bytes of one V^T tile
static_assert(LG_GROUP_BYTES % 128 == 0, "group layout alignment");

// K^T image: tile (b, g, t) holds the flushed K[b, 64 t + key, g, d] at
// [d][key] (keys at or past T are 0).  One thread moves one float4 of d.
// Also zeroes the work counter of k_attn_rows<false>
__global__ void k_attn_kimg(const float* __restrict__ k, float* __restrict__ img, int64_t T,
                            int64_t Hkv, int64_t nkt, int64_t n, unsigned long long* counter)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *counter = 0;   // the logits kernel's work counter, for the launch after this one
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int key = (int)(e & (AT - 1));
        const int d4 = (int)((e >> 6) & (HD / 4 - 1));
        const int64_t tile = e >> 11;
        const int64_t t = tile % nkt, bg = tile / nkt;
        const int64_t bb = bg / Hkv, gg = bg % Hkv;
        const int64_t j = t * AT + key;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < T)
            v = flush4(*reinterpret_cast<const float4*>(k + ((bb * T + j) * Hkv + gg) * HD + 4 * d4));
        float* dst = img + tile * (HD * AT) + (4 * d4) * AT + key;
        dst[0] = v.x;
        dst[AT] = v.y;
        dst[2 * AT] = v.z;
        dst[3 * AT] = v.w;
    }
}

struct AttnLogitArgs {
    const float* q;                // forward: q; backward: dO
    const float* kimg;             // forward: the K^T image; backward: the V^T image
    float* cache;                  // forward: written (logits); backward: read (p)
    float* m;                      // forward: the row maxima
    unsigned long long* counter;   // query tiles handed out (zero at launch)
    int64_t T, Hq, Hkv, W, tiles_bh, nqt, nkt, items;
    float c;
    int* err;
    // backward: l_i and Dr_i in; the a_ij and dS_ij tiles out ([64][BT_P] per tile)
    const float* l;
    const float* drow;
    float* at;
    float* st;
};

// the k-th query tile handed out: the last query tiles of every (sequence,
// head) first, so the longest windows start first and the shortest fill the end
__device__ __forceinline__ int64_t item_of(const AttnLogitArgs& a, int64_t k)
{
    const int64_t bhs = a.items / a.nqt;
    const int64_t qt = a.nqt - 1 - k / bhs, bh = k % bhs;
    return bh * a.nqt + qt;
}

// one query tile's place: sequence, head, kv head, first row, key tiles
struct QTile {
    int64_t b, h, g;
    int i0, t_lo, t_hi;
};

__device__ __forceinline__ QTile qtile_of(const AttnLogitArgs& a, int64_t item)
{
    QTile r;
    const int qt = (int)(item % a.nqt);
    const int64_t bh = item / a.nqt;
    r.h = bh % a.Hq;
    r.b = bh / a.Hq;
    r.g = r.h / (a.Hq / a.Hkv);
    r.i0 = qt * AT;
    const int T = (int)a.T, W = (int)a.W;
    const int jlo = W > 0 ? max(0, r.i0 - W + 1) : 0;
    r.t_lo = jlo / AT;
    r.t_hi = min(r.i0 + AT - 1, T - 1) / AT;
    return r;
}

// one 64-term chunk of the thread's 8 x 4 sums, operands loaded one step ahead
__device__ __forceinline__ void logit_chunk84(u64 (&acc)[16], const float* __restrict__ Ar,
                                              const float* __restrict__ Br)
{
    ulonglong2 a03 = *reinterpret_cast<const ulonglong2*>(Ar);
    ulonglong2 a47 = *reinterpret_cast<const ulonglong2*>(Ar + 4);
    float4 b = *reinterpret_cast<const float4*>(Br);
    {
        const ulonglong2 c03 = a03, c47 = a47;
        const float4 cb = b;
        a03 = *reinterpret_cast<const ulonglong2*>(Ar + PT);
        a47 = *reinterpret_cast<const ulonglong2*>(Ar + PT + 4);
        b = *reinterpret_cast<const float4*>(Br + AT);
        step<true>(acc, c03, c47, cb);
    }
#pragma unroll 9
    for (int d = 1; d < 64; ++d) {
        const ulonglong2 c03 = a03, c47 = a47;
        const float4 cb = b;
        const int dn = d + 1 < 64 ? d + 1 : d;
        a03 = *reinterpret_cast<const ulonglong2*>(Ar + dn * PT);
        a47 = *reinterpret_cast<const ulonglong2*>(Ar + dn * PT + 4);
        b = *reinterpret_cast<const float4*>(Br + dn * AT);
        step<false>(acc, c03, c47, cb);
    }
}

template <bool BWD>
__global__ void __launch_bounds__(LG_NT, 1) k_attn_rows(const AttnLogitArgs a)
{
    extern __shared__ __align__(128) uint8_t sml[];
    __shared__ uint64_t full[2][2], empty[2][2];
    __shared__ int64_t queue[2][8];   // per group: the query tiles handed to it, in order (-1: none left)
    const int tid = threadIdx.x, gp = tid >> 7, lt = tid & (LG_G - 1);
    const int lane = tid & 31;
    const int ty = lt >> 4, tx = lt & 15;      // rows 8ty .. 8ty+7, keys 4tx .. 4tx+3
    const int gbar = 1 + gp;
    uint8_t* gbase = sml + (size_t)gp * LG_GROUP_BYTES;
    float* Qt = reinterpret_cast<float*>(gbase);                   // [HD][PT]
    float* Kr = reinterpret_cast<float*>(gbase + LG_Q_BYTES);      // [2][HD][AT]
    float* lrw = Kr + 2 * HD * AT;                                  // [AT] l_i (backward)
    float* drw = lrw + AT;                                          // [AT] Dr_i (backward)
    if (tid == 0) {
        for (int x = 0; x < 2; ++x)
            for (int s = 0; s < 2; ++s) {
                mbar_init(&full[x][s], 1);
                mbar_init(&empty[x][s], LG_G / 32);   // one arrival per warp
            }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int T = (int)a.T, W = (int)a.W;
    const int64_t qstride = a.Hq * HD;

    // issuer (group thread 0): takes the group's query tiles from the counter
    // one ahead of the one whose key tiles it walks, so the entry of query
    // tile k + 1 is written before the first key tile of query tile k is
    // issued -- and is visible to every thread that has waited on that copy.
    // It runs at most two key tiles ahead of the group: at most four entries
    // are live
    int iss_k = 0, iss_t = 0;
    bool have = false;
    uint32_t issued = 0;
    QTile iss_q;
    auto take = [&](int kslot) {
        const int64_t k = (int64_t)atomicAdd(a.counter, 1ull);
        queue[gp][kslot & 7] = k < a.items ? item_of(a, k) : -1;
    };
    auto start = [&](int kslot) {   // walk query tile kslot (already taken)
        const int64_t item = queue[gp][kslot & 7];
        have = item >= 0;
        if (have) {
            take(kslot + 1);
            iss_q = qtile_of(a, item);
            iss_t = iss_q.t_lo;
        }
    };
    auto issue_next = [&]() {
        if (!have)
            return;
        const int s = issued & 1;
        mbar_expect_tx(&full[gp][s], KIMG_TILE);
        bulk_load(Kr + s * (HD * AT), a.kimg + ((iss_q.b * a.Hkv + iss_q.g) * a.nkt + iss_t) * (HD * AT),
                  KIMG_TILE, &full[gp][s]);
        ++issued;
        if (++iss_t > iss_q.t_hi)
            start(++iss_k);
    };
    if (lt == 0) {
        take(0);
        start(0);
        issue_next();
        issue_next();
    }

    uint32_t used = 0;      // key tiles consumed by the group
    bool fail = false, dead = false;
    for (int kk = 0;; ++kk) {
        // a failed wait anywhere in the group stops it at the next query tile;
        // the barrier also frees Qt and publishes the issuer's queue entry
        {
            uint32_t r;
            asm volatile(
                "{\n\t.reg .pred q, o;\n\t"
                "setp.ne.u32 q, %1, 0;\n\t"
                "bar.red.or.pred o, %2, %3, q;\n\t"
                "selp.u32 %0, 1, 0, o;\n\t}"
                : "=r"(r)
                : "r"((uint32_t)(fail || dead)), "r"(gbar), "n"(LG_G)
                : "memory");
            dead = r != 0;
        }
        const int64_t item = queue[gp][kk & 7];
        if (dead || item < 0)
            break;
        const QTile qt = qtile_of(a, item);
        // Q^T of this query tile, flushed: 64 rows x 32 float4, 16 per thread
        {
            const float* qbase = a.q + (qt.b * a.T * a.Hq + qt.h) * HD;
#pragma unroll
            for (int it = 0; it < (AT * HD / 4) / LG_G; ++it) {
                const int e = lt + it * LG_G;
                const int l8 = e & 31, w = e >> 5;     // 8 rows x 4 float4 per warp step
                const int r = (w & 7) * 8 + (l8 & 7);
                const int c4 = (w >> 3) * 4 + (l8 >> 3);
                const int64_t row = qt.i0 + r;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row < T)
                    v = flush4(*reinterpret_cast<const float4*>(qbase + row * qstride + 4 * c4));
                Qt[(4 * c4 + 0) * PT + r] = v.x;
                Qt[(4 * c4 + 1) * PT + r] = v.y;
                Qt[(4 * c4 + 2) * PT + r] = v.z;
                Qt[(4 * c4 + 3) * PT + r] = v.w;
            }
        }
        if constexpr (BWD) {
            if (lt < AT) {
                const int64_t i = qt.i0 + lt;
                lrw[lt] = i < T ? a.l[(qt.b * a.T + i) * a.Hq + qt.h] : 1.0f;
            } else {
                const int64_t i = qt.i0 + lt - AT;
                drw[lt - AT] = i < T ? a.drow[(qt.b * a.T + i) * a.Hq + qt.h] : 0.0f;
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(gbar), "n"(LG_G) : "memory");
        const int64_t tile0 = (qt.b * a.Hq + qt.h) * a.tiles_bh + tile_prefix(qt.i0 / AT, W);
        float* cache = a.cache + tile0 * (AT * AT);
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            mx[e] = -INFINITY;
        for (int t = qt.t_lo; t <= qt.t_hi; ++t) {
            const int s = used & 1;
            // the stage of the previous tile takes the tile after this one,
            // once every warp has released it
            if (lt == 0 && used >= 1 && issued == used + 1 && have) {
                if (mbar_wait(&empty[gp][s ^ 1], ((used - 1) >> 1) & 1))
                    issue_next();
                else
                    fail = true;
            }
            if (!mbar_wait(&full[gp][s], (used >> 1) & 1))
                fail = true;
            if (t == qt.t_hi) {
                // the next query tile's Q rows into L2 while this tile is formed
                const int64_t nitem = queue[gp][(kk + 1) & 7];
                if (nitem >= 0) {
                    const QTile nq = qtile_of(a, nitem);
                    const int64_t row = nq.i0 + (lt >> 1);
                    if (row < T) {
                        const float* src = a.q + ((nq.b * a.T + row) * a.Hq + nq.h) * HD + (lt & 1) * 64;
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 32));
                    }
                }
            }
            const float* Kc = Kr + s * (HD * AT);
            u64 t0[16], t1[16];
            logit_chunk84(t0, Qt + 8 * ty, Kc + 4 * tx);
            logit_chunk84(t1, Qt + 64 * PT + 8 * ty, Kc + 64 * AT + 4 * tx);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[gp][s]);
            ++used;
            if constexpr (!BWD) {
                const u64 cc = pack2(a.c, a.c);
                u64 sv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)   // (t0 + t1) (x) c, flushed
                    sv[e] = fadd2_ftz(fmul2_rn(fadd2_ftz(t0[e], t1[e]), cc), pack2(-0.0f, -0.0f));
                {
                    // rows 8ty .. 8ty+3 are 4 x 4 block (2ty, tx) of the cached tile,
                    // rows 8ty+4 .. 8ty+7 block (2ty + 1, tx)
                    float* tile = cache + (int64_t)(t - qt.t_lo) * (AT * AT);
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        ulonglong2* dst = reinterpret_cast<ulonglong2*>(tile + ((2 * ty + blk) * 16 + tx) * 16);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_ulonglong2(sv[8 * blk + 2 * e], sv[8 * blk + 2 * e + 1]);
                    }
                }
                const int j0 = t * AT;
                const bool inner = qt.i0 + AT - 1 < T && j0 + AT - 1 <= qt.i0 && (W == 0 || j0 >= qt.i0 + AT - W);
#pragma unroll
                for (int ip = 0; ip < 4; ++ip)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float lo, hi;
                        unpack2(sv[ip * 4 + j], lo, hi);
                        if (inner) {
                            mx[2 * ip] = fmaxf(mx[2 * ip], lo);
                            mx[2 * ip + 1] = fmaxf(mx[2 * ip + 1], hi);
                        } else {
                            const int jj = j0 + 4 * tx + j;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int i = qt.i0 + 8 * ty + 2 * ip + h;
                                const int lo_i = W > 0 ? max(0, i - W + 1) : 0;
                                if (i < T && jj >= lo_i && jj <= i)
                                    mx[2 * ip + h] = fmaxf(mx[2 * ip + h], h ? hi : lo);
                            }
                        }
                    }
            } else {
                // dA = (t0 (+) t1); with p from the forward's cache (the pairs
                // sit where pass 1 wrote this thread's logits):
                //   a = p (/) l_i, dS = a (x) (dA (-) Dr_i), both flushed, +0 off the window
                const u64 z = pack2(-0.0f, -0.0f);
                const float* ptile = cache + (int64_t)(t - qt.t_lo) * (AT * AT);
                u64 pv[16];
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    const ulonglong2* src = reinterpret_cast<const ulonglong2*>(ptile + ((2 * ty + blk) * 16 + tx) * 16);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const ulonglong2 v = src[e];
                        pv[8 * blk + 2 * e] = v.x;
                        pv[8 * blk + 2 * e + 1] = v.y;
                    }
                }
                const int j0 = t * AT;
                const bool inner = qt.i0 + AT - 1 < T && j0 + AT - 1 <= qt.i0 && (W == 0 || j0 >= qt.i0 + AT - W);
                float av[8][4], dv[8][4];   // rows 8ty + rr, keys 4tx + j
#pragma unroll
                for (int ip = 0; ip < 4; ++ip)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int e = ip * 4 + j, r0 = 8 * ty + 2 * ip;
                        float p[2], aa[2];
                        unpack2(pv[e], p[0], p[1]);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            aa[h] = flush(__fdiv_rn(p[h], lrw[r0 + h]));
                        float d[2];
                        unpack2(fadd2_ftz(fmul2_rn(pack2(aa[0], aa[1]),
                                                   fadd2_ftz(fadd2_ftz(t0[e], t1[e]), pack2(-drw[r0], -drw[r0 + 1]))),
                                          z),
                                d[0], d[1]);
                        if (!inner) {
                            const int jj = j0 + 4 * tx + j;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int i = qt.i0 + r0 + h;
                                const int lo_i = W > 0 ? max(0, i - W + 1) : 0;
                                if (!(i < T && jj >= lo_i && jj <= i))
                                    aa[h] = d[h] = 0.f;
                            }
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            av[2 * ip + h][j] = aa[h];
                            dv[2 * ip + h][j] = d[h];
                        }
                    }
                const int64_t toff = (tile0 + (t - qt.t_lo)) * (int64_t)(AT * BT_P);
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int64_t off = toff + (8 * ty + rr) * BT_P + 4 * tx;
                    *reinterpret_cast<float4*>(a.at + off) = make_float4(av[rr][0], av[rr][1], av[rr][2], av[rr][3]);
                    *reinterpret_cast<float4*>(a.st + off) = make_float4(dv[rr][0], dv[rr][1], dv[rr][2], dv[rr][3]);
                }
            }
        }
        if constexpr (!BWD) {
            // the rows' maxima over the 16 threads of each row group
#pragma unroll
            for (int e = 0; e < 8; ++e) {
#pragma unroll
                for (int off = 1; off < 16; off <<= 1)
                    mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], off));
                if (mx[e] == 0.0f)
                    mx[e] = 0.0f;   // a zero maximum is +0
            }
            if (tx == 0)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t i = qt.i0 + 8 * ty + e;
                    if (i < T)
                        a.m[(qt.b * a.T + i) * a.Hq + qt.h] = mx[e];
                }
        }
    }
    // copies still in flight (only after a failed wait, or tiles issued ahead)
    if (lt == 0)
        while (used < issued && mbar_wait(&full[gp][used & 1], (used >> 1) & 1))
            ++used;
    if (fail)
        atomicExch(a.err, 1);
}

// the V codes as the P.V's B operand: tile (b, g, t) holds V^T[d][key] for
// the 64 keys of key tile t (keys at or past T are 0), bf16, in the 128-byte-
// swizzled K-major layout of umma.cuh.  One thread writes one 16-byte chunk
// (8 keys of one d)
__global__ void k_attn_vimg(const int8_t* __restrict__ vq, uint8_t* __restrict__ img, int64_t T,
                            int64_t Hkv, int64_t nkt, int64_t n_chunks)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_chunks;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int c8 = (int)(e & 7);
        const int d = (int)((e >> 3) & (HD - 1));
        const int64_t tile = e >> 10;
        const int64_t t = tile % nkt, bg = tile / nkt;
        const int64_t bb = bg / Hkv, gg = bg % Hkv;
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int v2[2];
#pragma unroll
            for (int z = 0; z < 2; ++z) {
                const int64_t j = t * AT + 8 * c8 + 2 * u + z;
                v2[z] = j < T ? (int)vq[((bb * T + j) * Hkv + gg) * HD + d] : 0;
            }
            w[u] = bf16_bits(v2[0]) | (bf16_bits(v2[1]) << 16);
        }
        *reinterpret_cast<uint4*>(img + tile * VIMG_TILE + sw128_off(d, 8 * c8)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

constexpr int PV_TC_BYTES = 2 * (2 * TC_TILE_BYTES) + 1024;   // two (P, V^T) buffers + alignment
constexpr int PV_PS_BYTES = 2 * AT * PS * 4;                  // two p tiles
constexpr int PV_STK_BYTES = AT * (MAXL + 1) * 4;
constexpr size_t PV_SMEM = (size_t)PV_TC_BYTES + PV_PS_BYTES + PV_STK_BYTES + 2 * AT * 4;
constexpr int PV_PROD = NT;             // producer threads: eight warps
constexpr int PV_NTH = NT + 96;         // two row-sum warps and the MMA warp

struct AttnPVArgs {
    AttnFwdArgs f;
    const uint8_t* vimg;
    int64_t nkt;
};

__global__ void __launch_bounds__(PV_NTH, 2) k_attn_pv(const AttnPVArgs pa)
{
    extern __shared__ __align__(16) uint8_t smv[];
    __shared__ uint64_t mma_bar[2], v_bar[2], ready[2], ps_free[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int dead_flag;
    const AttnFwdArgs& a = pa.f;

    const int lt = threadIdx.x;
    // buffer x: P at tcb0 + 2 x TC_TILE_BYTES, V^T TC_TILE_BYTES after it
    uint8_t* tcb0 = smv + ((1024u - (su32(smv) & 1023u)) & 1023u);
    auto tcbuf = [&](int x) { return tcb0 + x * (2 * TC_TILE_BYTES); };
    float* Psb = reinterpret_cast<float*>(smv + PV_TC_BYTES);   // [2][AT][PS]
    float* stk = Psb + 2 * AT * PS;                             // [AT][MAXL+1]
    float* mrow = stk + AT * (MAXL + 1);
    float* lrow = mrow + AT;

    const int T = (int)a.T, W = (int)a.W;
    const int64_t b = blockIdx.z, h = blockIdx.y;
    const int i0 = (int)blockIdx.x * AT;
    const int64_t g = h / (a.Hq / a.Hkv);
    const int jlo = W > 0 ? max(0, i0 - W + 1) : 0;
    const int jhi = min(i0 + AT - 1, T - 1);
    const int t_lo = jlo / AT, t_hi = jhi / AT;
    float* cache = a.cache + ((b * a.Hq + h) * a.tiles_bh + tile_prefix((int64_t)blockIdx.x, W)) * (AT * AT);
    const uint8_t* vsrc = pa.vimg + (b * a.Hkv + g) * pa.nkt * VIMG_TILE;
    // tiles per exact slice: a whole query tile when no row has more than 520
    // valid keys (W <= 520), else 8
    const int slice = (W > 0 && W <= 520) ? (1 << 30) : TC_SLICE_TILES;

    if (lt == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&mma_bar[x], 1);
            mbar_init(&v_bar[x], 1);
            mbar_init(&ready[x], PV_PROD / 32);   // one arrival per producer warp
            mbar_init(&ps_free[x], 2);            // one per consumer warp
        }
        dead_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (lt < 32) {
        // columns 0-127: the fp32 accumulator of the current slice; 128-255:
        // the int32 sums of the finished slices
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(
                         su32(&tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (lt < AT) {
        const int i = i0 + lt;
        mrow[lt] = i < T ? a.m[(b * a.T + i) * a.Hq + h] : 0.0f;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = tmem_slot;

    // bounded; returns false at once once any wait in the CTA has failed
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const long long t0 = clock64();
        while (!mbar_test(bar, parity)) {
            if (*reinterpret_cast<volatile int*>(&dead_flag))
                return false;
            if (clock64() - t0 > WAIT_CYCLES) {
                atomicExch(&dead_flag, 1);
                return false;
            }
        }
        return true;
    };

    if (lt < PV_PROD) {
        // ------------------------------------------------------------------
        // producers: p, the codes and the P tile of every key tile
        const int ty = lt >> 4, tx = lt & 15;
        // logits of the next two tiles in flight
        ulonglong2 sv4[4], sn4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            sv4[e] = reinterpret_cast<const ulonglong2*>(cache + lt * 16)[e];
            if (t_lo < t_hi)
                sn4[e] = reinterpret_cast<const ulonglong2*>(cache + AT * AT + lt * 16)[e];
        }
        for (int t = t_lo; t <= t_hi; ++t) {
            const int j0 = t * AT;
            const int it = t - t_lo;
            const int bf = it & 1;
            const bool more = t < t_hi;
            // the buffers of tile it - 2: read by its MMA and its row sums
            if (it >= 2) {
                wait(&mma_bar[bf], ((it - 2) >> 1) & 1);
                wait(&ps_free[bf], ((it - 2) >> 1) & 1);
            }
            u64 s[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[2 * e] = sv4[e].x;
                s[2 * e + 1] = sv4[e].y;
            }
            u64 pp[8];       // p as the cache's pairs: rows (r, r + 1) of key j in pp[ip*4 + j]
            uint32_t cw[8];  // bf16 codes: row 4ty + rr, keys 4tx + 2c, +1 in cw[2 rr + c]
            // every (query, key) pair of the tile valid: no per-pair test
            const bool inner = i0 + AT - 1 < T && j0 + AT - 1 <= i0 && (W == 0 || j0 >= i0 + AT - W);
            const u64 z = pack2(-0.0f, -0.0f), c127 = pack2(127.0f, 127.0f);
#pragma unroll
            for (int ip = 0; ip < 2; ++ip) {
                const int r = 4 * ty + 2 * ip;   // rows r, r + 1 are the lanes of s[ip*4 + j]
                const u64 nm = pack2(-mrow[r], -mrow[r + 1]);
                uint32_t qb[2][4];               // float bits of the codes, per lane and key
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    u64 e2 = exp_r2(fadd2_ftz(s[ip * 4 + j], nm));
                    if (!inner) {
                        float p[2];
                        unpack2(e2, p[0], p[1]);
                        const int jj = j0 + 4 * tx + j;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int i = i0 + r + hh;
                            const int lo = W > 0 ? max(0, i - W + 1) : 0;
                            if (!(i < T && jj >= lo && jj <= i))
                                p[hh] = 0.f;
                        }
                        e2 = pack2(p[0], p[1]);
                    }
                    pp[ip * 4 + j] = e2;
                    float t0, t1;
                    unpack2(fadd2_ftz(fmul2_rn(e2, c127), z), t0, t1);
                    qb[0][j] = __float_as_uint(quant_pf(t0));
                    qb[1][j] = __float_as_uint(quant_pf(t1));
                }
                // a code (0 .. 127) as bf16 is the high half of its float
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    cw[2 * (2 * ip + hh)] = __byte_perm(qb[hh][0], qb[hh][1], 0x7632);
                    cw[2 * (2 * ip + hh) + 1] = __byte_perm(qb[hh][2], qb[hh][3], 0x7632);
                }
            }
            if (more) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    sv4[e] = sn4[e];
                if (t + 1 < t_hi) {   // the logits two tiles ahead
                    const ulonglong2* src =
                        reinterpret_cast<const ulonglong2*>(cache + (int64_t)(it + 2) * (AT * AT) + lt * 16);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sn4[e] = src[e];
                }
            }
            float* Ps = Psb + bf * (AT * PS);
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int r = 4 * ty + rr;
                // the four codes at keys 4tx .. 4tx+3 of row r (rows 64-127 of
                // the MMA's A are never read back: only lanes 0-63 hold rows)
                *reinterpret_cast<uint2*>(tcbuf(bf) + sw128_off(r, 4 * tx)) = make_uint2(cw[2 * rr], cw[2 * rr + 1]);
                const int ip = rr >> 1, hh = rr & 1;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    Ps[r * PS + 4 * tx + j] = lane_of(pp, ip, j, hh);
            }
            {
                // the cache now holds p in place of each logit: the backward
                // reads p from it instead of evaluating e^x again
                ulonglong2* dst = reinterpret_cast<ulonglong2*>(cache + (int64_t)it * (AT * AT) + lt * 16);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_ulonglong2(pp[2 * e], pp[2 * e + 1]);
            }
            // the P tile's generic-proxy stores become visible to the tensor core
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if ((lt & 31) == 0)
                mbar_arrive(&ready[bf]);
        }
    } else if (lt < PV_PROD + 64) {
        // ------------------------------------------------------------------
        // row-sum warps: row cl's sums; warp cl / 32 reads tensor-memory lanes
        // 32 (cl / 32) .. + 31 (rows 0-63) at the end of every exact slice
        const int cl = lt - PV_PROD;
        const int lane = cl & 31;
        const uint32_t trow = tmem + ((uint32_t)(32 * (cl >> 5)) << 16);
        const int my_i = i0 + cl;
        const int my_lo = W > 0 ? max(0, my_i - W + 1) : 0;
        const int my_n = my_i - my_lo + 1;
        int pos = 0;
        float cs = 0.f, lsum = 0.f;
        bool first_slice = true;
        for (int t = t_lo; t <= t_hi; ++t) {
            const int j0 = t * AT;
            const int it = t - t_lo;
            const int bf = it & 1;
            const bool more = t < t_hi;
            wait(&ready[bf], (it >> 1) & 1);
            // the valid p of this tile, left to right, through the
            // chunk-of-64 / pairwise-tree stack
            if (my_i < T) {
                const int cb = max(my_lo, j0), ce = min(my_i, j0 + AT - 1);
                const float* prow = Psb + bf * (AT * PS) + cl * PS;   // column jj - j0
                int jj = cb;
                while (jj <= ce) {
                    // one run up to the next chunk boundary: left to right,
                    // seeded with the chunk's first term
                    const int room = 64 - (pos & 63);
                    const int len = min(room, ce - jj + 1);
                    int k = 0;
                    const float* pr = prow + (jj - j0);
                    if ((pos & 63) == 0) {
                        cs = pr[0];
                        k = 1;
                    }
#pragma unroll 8
                    for (; k < len; ++k)
                        cs = fadd_ftz(cs, pr[k]);
                    jj += len;
                    pos += len;
                    if ((pos & 63) == 0 || pos == my_n) {
                        const int c = (pos - 1) >> 6;
                        float acc_t = cs;
                        if (pos == my_n) {
                            for (int lvl = 0; lvl < MAXL; ++lvl)
                                if ((c >> lvl) & 1)
                                    acc_t = fadd_ftz(stk[cl * (MAXL + 1) + lvl], acc_t);
                            lsum = acc_t;
                        } else {
                            const int tz = __ffs(~c) - 1;
                            for (int lvl = 0; lvl < tz; ++lvl)
                                acc_t = fadd_ftz(stk[cl * (MAXL + 1) + lvl], acc_t);
                            stk[cl * (MAXL + 1) + tz] = acc_t;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ps_free[bf]);
            // end of an exact slice: its accumulator, as int32, into the sums
            if (it % slice == slice - 1 || !more) {
                const bool got = __all_sync(0xffffffffu, wait(&mma_bar[bf], (it >> 1) & 1));
                if (got) {
                    fence_after();
#pragma unroll
                    for (int c = 0; c < HD / 16; ++c) {
                        uint32_t v[16], u[16];
                        tmem_ld16(trow + 16 * c, v);
                        if (!first_slice)
                            tmem_ld16(trow + 128 + 16 * c, u);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            u[e] = (first_slice ? 0u : u[e]) + (uint32_t)__float2int_rn(__uint_as_float(v[e]));
                        tmem_st16(trow + 128 + 16 * c, u);
                    }
                    fence_before();
                }
                first_slice = false;
                // the accumulator has been read before the MMA warp starts
                // the next slice over it
                asm volatile("bar.sync 3, 96;" ::: "memory");
            }
        }

        lrow[cl] = lsum;
        if (my_i < T)
            a.l[(b * a.T + my_i) * a.Hq + h] = lsum;
    } else {
        // ------------------------------------------------------------------
        // the MMA warp: lane 0 copies V^T and issues the MMAs
        const bool issuer = lt == PV_PROD + 64;
        uint32_t vn[2] = {0, 0}, vw[2] = {0, 0};   // V^T copies issued / seen complete
        if (issuer) {   // V^T of the first tile
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(&v_bar[0], VIMG_TILE);
            bulk_load(tcbuf(0) + TC_TILE_BYTES, vsrc + (int64_t)t_lo * VIMG_TILE, VIMG_TILE, &v_bar[0]);
            vn[0] = 1;
        }
        for (int t = t_lo; t <= t_hi; ++t) {
            const int it = t - t_lo;
            const int bf = it & 1;
            const bool more = t < t_hi;
            if (issuer && wait(&ready[bf], (it >> 1) & 1) && wait(&v_bar[bf], (it >> 1) & 1)) {
                ++vw[bf];
                fence_after();
                const uint64_t ad = sdesc(su32(tcbuf(bf))), bd = sdesc(su32(tcbuf(bf) + TC_TILE_BYTES));
#pragma unroll
                for (int k = 0; k < AT / 16; ++k)
                    mma_bf16<HD>(tmem, ad + 2 * k, bd + 2 * k, (it % slice != 0 || k != 0) ? 1u : 0u);
                mma_commit(&mma_bar[bf]);
                // V^T of the next tile into the other buffer, once the MMA of
                // the previous tile has read it
                if (more && (it == 0 || wait(&mma_bar[bf ^ 1], ((it - 1) >> 1) & 1))) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(&v_bar[bf ^ 1], VIMG_TILE);
                    bulk_load(tcbuf(bf ^ 1) + TC_TILE_BYTES, vsrc + (int64_t)(t + 1) * VIMG_TILE, VIMG_TILE,
                              &v_bar[bf ^ 1]);
                    ++vn[bf ^ 1];
                }
            }
            __syncwarp();
            if (it % slice == slice - 1 || !more) {
                asm volatile("bar.sync 3, 96;" ::: "memory");   // the slice has been read
                fence_after();
            }
        }
        // copies still in flight (only after a failed wait) land before exit
        if (issuer)
            for (int x = 0; x < 2; ++x)
                while (vw[x] < vn[x] && mbar_wait(&v_bar[x], vw[x] & 1))
                    ++vw[x];
    }

    fence_before();
    __syncthreads();
    fence_after();
    // epilogue: o = (i2f(sum) (x) s_v) (/) (l (x) 127).  The six warps that can
    // read tensor-memory lanes 0-63 (warps 0, 4, 8: rows 0-31; 1, 5, 9: rows
    // 32-63) take 48, 48 and 32 of the 128 columns
    {
        const int w = lt >> 5;
        if (w < 10 && (w & 3) < 2) {
            const int q = w & 3, part = w >> 2;   // part 0, 1, 2 -> chunks 0-2, 3-5, 6-7
            const int row = 32 * q + (lt & 31);
            const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
            const int64_t i = i0 + row;
            const float sv = flush(*a.s_v);
            const float den = fmul_flush(lrow[row], 127.0f);
            float* dst = a.o + ((b * a.T + i) * a.Hq + h) * HD;
            const int c_end = part == 2 ? HD / 16 : 3 * part + 3;
#pragma unroll 1
            for (int c = 3 * part; c < c_end; ++c) {
                uint32_t u[16];
                tmem_ld16(trow + 128 + 16 * c, u);
                if (i < (int64_t)T) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        float ov[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            ov[e] = flush(__fdiv_rn(fmul_flush(__int2float_rn((int)u[4 * q4 + e]), sv), den));
                        *reinterpret_cast<float4*>(dst + 16 * c + 4 * q4) = make_float4(ov[0], ov[1], ov[2], ov[3]);
                    }
                }
            }
        }
    }
    fence_before();
    __syncthreads();
    if (lt < 32) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem) : "memory");
    }
    if (lt == 0 && dead_flag)
        atomicExch(a.err, 1);
}

// ---------------------------------------------------------------------------
// Backward (straight-through for both quantisations), per the readings:
//   a_ij  = p_ij (/) l_i (p recomputed from m_i as in the forward)
//   Dr_i  = canon_d(dO_id (x) O_id)
//   dA_ij = canon_d(dO_id (x) V^_jd),  V^ = i2f(V_q) (x) s_v
//   dS_ij = a_ij (x) (dA_ij (-) Dr_i)
//   dQ_id = fix2f(sum over 64-aligned key tiles of fx(T_tile)) (x) c, T_tile
//           the left-to-right sum over the tile's valid keys of dS_ij (x) k_jd;
//           fx(x) = nearest int64 to x * 2^48 (ties to even, saturating):
//           the tile partials meet in 64-bit fixed point through integer
//           atomics, exact in any order;
//   dK_jd = (fold) (x) c, dV_jd = (fold): terms dS_ij (x) q_id and
//           a_ij (x) dO_id over the query heads of kv head g (ascending) and
//           the 64-aligned query tiles (ascending), each tile summed left to
//           right from its first valid term, the tile partials folded left.
// k_attn_bwd (the route without the forward's cache): one CTA per (64-key
// tile, kv head, sequence) recomputes the logits and visits its query tiles
// in that order, so dK and dV stay in tensor memory; dQ tile partials go to
// an int64 accumulator with atomicAdd and are converted at the end.  With the
// cache the three kernels further below take its place.
// ---------------------------------------------------------------------------

constexpr int PR = 132;   // pitch (floats) of the row-major 64 x 128 tiles

struct AttnBwdArgs {
    const float* q;
    const float* k;
    const int8_t* vq;
    const float* s_v;
    const float* dout;
    const float* m;
    const float* l;
    const float* drow;
    unsigned long long* dq_acc;
    float* dk;
    float* dv;
    int64_t T, Hq, Hkv, W;
    int64_t tiles_bh;
    float c;
};

constexpr int PB = 68;    // pitch (floats) of the a, dS and transposed dS tiles

__device__ __forceinline__ void tm_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t w[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
          "=r"(w[7]), "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]),
          "=r"(w[14]), "=r"(w[15]), "=r"(w[16]), "=r"(w[17]), "=r"(w[18]), "=r"(w[19]),
          "=r"(w[20]), "=r"(w[21]), "=r"(w[22]), "=r"(w[23]), "=r"(w[24]), "=r"(w[25]),
          "=r"(w[26]), "=r"(w[27]), "=r"(w[28]), "=r"(w[29]), "=r"(w[30]), "=r"(w[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 32; ++e)
        v[e] = __uint_as_float(w[e]);
}

__device__ __forceinline__ void tm_st32(uint32_t taddr, const float (&v)[32])
{
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 32; ++e)
        w[e] = __float_as_uint(v[e]);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
        "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
        "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
constexpr size_t BWD_SMEM = (size_t)(4 * AT * PR + 3 * AT * PB + 3 * AT) * 4 + 16;

// 64 rows of a [.., H, 128] tensor into t[r][d] (pitch PR), flushed; rows
// outside [0, T) read as 0
__device__ __forceinline__ void load_tile_r(float* __restrict__ t, const float* __restrict__ src,
                                            int64_t row0, int64_t T, int64_t row_stride, int tid)
{
#pragma unroll
    for (int it = 0; it < (AT * HD / 4) / NT; ++it) {
        const int e = tid + it * NT;
        const int r = e >> 5, c4 = e & 31;
        const int64_t row = row0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row >= 0 && row < T)
            v = flush4(*reinterpret_cast<const float4*>(src + row * row_stride + 4 * c4));
        *reinterpret_cast<float4*>(t + r * PR + 4 * c4) = v;
    }
}

// out[r][c] = canon_d(X[ty+16r][d] (x) Y[tx+16c][d]), d = 0..127: two chunks
// of 64 summed left to right from their first product, then one pairwise add
__device__ __forceinline__ void tile_dot(float (&out)[4][4], const float* __restrict__ X,
                                         const float* __restrict__ Y, int ty, int tx)
{
    float t0[4][4];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float acc[4][4];
#pragma unroll 2
        for (int d4 = 0; d4 < 16; ++d4) {
            const int d = half * 64 + 4 * d4;
            float4 xv[4], yv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                xv[r] = *reinterpret_cast<const float4*>(X + (ty + 16 * r) * PR + d);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                yv[c] = *reinterpret_cast<const float4*>(Y + (tx + 16 * c) * PR + d);
#pragma unroll
            for (int e = 0; e < 4; ++e)
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float xe = e == 0 ? xv[r].x : (e == 1 ? xv[r].y : (e == 2 ? xv[r].z : xv[r].w));
                        const float ye = e == 0 ? yv[c].x : (e == 1 ? yv[c].y : (e == 2 ? yv[c].z : yv[c].w));
                        const float p = fmul_rn(xe, ye);
                        acc[r][c] = (d4 == 0 && e == 0) ? p : fadd_ftz(acc[r][c], p);
                    }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (half == 0)
                    t0[r][c] = acc[r][c];
                else
                    out[r][c] = fadd_ftz(t0[r][c], acc[r][c]);
            }
    }
}

// pp[q2][e] = sum over r = 0..63, left to right from the first (flushed)
// term, of W[r][2q2 .. 2q2+1] (x) X[r][e] for a thread's 8 x 4 block: W rows
// of pitch pw at Wp, X rows of pitch px at Xp; operands one step ahead
__device__ __forceinline__ void full_sum64(u64 (&pp)[4][4], const float* __restrict__ Wp, int pw,
                                           const float* __restrict__ Xp, int px)
{
    ulonglong2 w03 = *reinterpret_cast<const ulonglong2*>(Wp);
    ulonglong2 w47 = *reinterpret_cast<const ulonglong2*>(Wp + 4);
    float4 xv = *reinterpret_cast<const float4*>(Xp);
    {
        const u64 P[4] = {w03.x, w03.y, w47.x, w47.y};
        const u64 X2[4] = {pack2(xv.x, xv.x), pack2(xv.y, xv.y), pack2(xv.z, xv.z),
                           pack2(xv.w, xv.w)};
        w03 = *reinterpret_cast<const ulonglong2*>(Wp + pw);
        w47 = *reinterpret_cast<const ulonglong2*>(Wp + pw + 4);
        xv = *reinterpret_cast<const float4*>(Xp + px);
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pp[q2][e] = fadd2_ftz(fmul2_rn(P[q2], X2[e]), pack2(-0.0f, -0.0f));
    }
#pragma unroll 9
    for (int r = 1; r < AT; ++r) {
        const u64 P[4] = {w03.x, w03.y, w47.x, w47.y};
        const u64 X2[4] = {pack2(xv.x, xv.x), pack2(xv.y, xv.y), pack2(xv.z, xv.z),
                           pack2(xv.w, xv.w)};
        const int rn = r + 1 < AT ? r + 1 : r;
        w03 = *reinterpret_cast<const ulonglong2*>(Wp + rn * pw);
        w47 = *reinterpret_cast<const ulonglong2*>(Wp + rn * pw + 4);
        xv = *reinterpret_cast<const float4*>(Xp + rn * px);
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pp[q2][e] = fadd2_ftz(pp[q2][e], fmul2_rn(P[q2], X2[e]));
    }
}

// pp[q2][e] (+)= W[r][2q2 .. 2q2+1] (x) X[r][e] for r = lo .. hi, left to
// right, when every row pair of the thread's block is valid and already seeded
// over that range (the middle of a mask-edge tile); operands one step ahead
__device__ __forceinline__ void packed_range(u64 (&pp)[4][4], const float* __restrict__ Wp, int pw,
                                             const float* __restrict__ Xp, int px, int lo, int hi)
{
    ulonglong2 w03 = *reinterpret_cast<const ulonglong2*>(Wp + lo * pw);
    ulonglong2 w47 = *reinterpret_cast<const ulonglong2*>(Wp + lo * pw + 4);
    float4 xv = *reinterpret_cast<const float4*>(Xp + lo * px);
#pragma unroll 4
    for (int r = lo; r <= hi; ++r) {
        const u64 P[4] = {w03.x, w03.y, w47.x, w47.y};
        const u64 X2[4] = {pack2(xv.x, xv.x), pack2(xv.y, xv.y), pack2(xv.z, xv.z),
                           pack2(xv.w, xv.w)};
        const int rn = r < hi ? r + 1 : r;
        w03 = *reinterpret_cast<const ulonglong2*>(Wp + rn * pw);
        w47 = *reinterpret_cast<const ulonglong2*>(Wp + rn * pw + 4);
        xv = *reinterpret_cast<const float4*>(Xp + rn * px);
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pp[q2][e] = fadd2_ftz(pp[q2][e], fmul2_rn(P[q2], X2[e]));
    }
}

__global__ void __launch_bounds__(NT, 1) k_attn_bwd(const AttnBwdArgs a)
{
    extern __shared__ __align__(16) float smb[];
    float* Ks = smb;                     // [AT][PR] keys of this tile
    float* Vs = Ks + AT * PR;            // [AT][PR] dequantised values
    float* Qs = Vs + AT * PR;            // [AT][PR] queries of the current tile
    float* Gs = Qs + AT * PR;            // [AT][PR] dO of the current tile
    float* As = Gs + AT * PR;            // [AT][PB] a_ij, row i, column j
    float* Ss = As + AT * PB;            // [AT][PB] dS_ij
    float* St = Ss + AT * PB;            // [AT][PB] dS transposed: row j, column i
    float* rm = St + AT * PB;            // [AT] m_i
    float* rl = rm + AT;                 // [AT] l_i
    float* rd = rl + AT;                 // [AT] Dr_i
    uint32_t* tslot = reinterpret_cast<uint32_t*>(rd + AT);

    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;        // 4 x 4 tile: rows ty+16r, cols tx+16c
    const int grp = tid >> 5, dg = tid & 31;       // 8 rows grp*8.., 4 columns 4dg..
    const int64_t b = blockIdx.z, g = blockIdx.y, j0 = (int64_t)blockIdx.x * AT;
    const int64_t T = a.T, W = a.W, Hq = a.Hq, Hkv = a.Hkv, G = Hq / Hkv;
    const int64_t qstride = Hq * HD, kstride = Hkv * HD;
    const float c = a.c;

    load_tile_r(Ks, a.k + (b * T * Hkv + g) * HD, j0, T, kstride, tid);
    {
        const float sv = flush(*a.s_v);
        const int8_t* vb = a.vq + (b * T * Hkv + g) * HD;
#pragma unroll
        for (int it = 0; it < (AT * HD / 4) / NT; ++it) {
            const int e = tid + it * NT;
            const int r = e >> 5, c4 = e & 31;
            const int64_t row = j0 + r;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < T) {
                const int w = *reinterpret_cast<const int*>(vb + row * kstride + 4 * c4);
                v = make_float4(dequant((int)(int8_t)w, sv), dequant((int)(int8_t)(w >> 8), sv),
                                dequant((int)(int8_t)(w >> 16), sv), dequant((int)(int8_t)(w >> 24), sv));
            }
            *reinterpret_cast<float4*>(Vs + r * PR + 4 * c4) = v;
        }
    }

    // dK / dV fold state (keys grp*8 + r, columns 4dg + e) lives in tensor
    // memory: thread lane 32*(warp%4) + lane, columns (warp/4)*64 + [0, 32)
    // for dK and + [32, 64) for dV, element r*4 + e
    if (tid < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(tslot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int warp = tid >> 5;
    const uint32_t tfold =
        *tslot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 64);
    bool started[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        started[r] = false;

    const int64_t ilast = W > 0 ? min(T - 1, j0 + AT - 1 + W - 1) : T - 1;
    for (int64_t hh = 0; hh < G; ++hh) {
        const int64_t h = g * G + hh;
        for (int64_t i0 = j0; i0 <= ilast; i0 += AT) {
            __syncthreads();   // previous tile's readers are done
            load_tile_r(Qs, a.q + (b * T * Hq + h) * HD, i0, T, qstride, tid);
            load_tile_r(Gs, a.dout + (b * T * Hq + h) * HD, i0, T, qstride, tid);
            if (tid < AT) {
                const int64_t i = i0 + tid;
                const int64_t rr = (b * T + i) * Hq + h;
                rm[tid] = i < T ? a.m[rr] : 0.f;
                rl[tid] = i < T ? a.l[rr] : 1.f;
                rd[tid] = i < T ? a.drow[rr] : 0.f;
            }
            __syncthreads();

            // a and dS for the 64 x 64 pairs (query row ty+16r, key tx+16cc)
            {
                float sv[4][4], dav[4][4];
                tile_dot(sv, Qs, Ks, ty, tx);
                tile_dot(dav, Gs, Vs, ty, tx);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int ir = ty + 16 * r;
                    const int64_t i = i0 + ir;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int jc = tx + 16 * cc;
                        const int64_t j = j0 + jc;
                        float av = 0.f, dsv = 0.f;
                        if (i < T && j <= i && (W == 0 || i - j < W)) {
                            const float p = exp_r(fadd_ftz(fmul_flush(sv[r][cc], c), -rm[ir]));
                            av = flush(__fdiv_rn(p, rl[ir]));
                            dsv = fmul_flush(av, fadd_ftz(dav[r][cc], -rd[ir]));
                        }
                        As[ir * PB + jc] = av;
                        Ss[ir * PB + jc] = dsv;
                        St[jc * PB + ir] = dsv;
                    }
                }
            }
            __syncthreads();

            // dQ tile partials: rows grp*8 + r, columns 4dg + e, over the valid
            // keys of this tile left to right, then into 64-bit fixed point.
            // Key index outermost; a tile where every row sees all 64 keys takes
            // the packed path (pairs of rows), edge tiles the predicated one.
            {
                int jb[8], je[8];
                bool full = true;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int64_t i = i0 + grp * 8 + r;
                    const int64_t lo = W > 0 ? i - W + 1 : (int64_t)0;
                    jb[r] = (int)(max(j0, lo) - j0);
                    je[r] = (int)(min(i, j0 + AT - 1) - j0);
                    if (i >= T)
                        jb[r] = AT, je[r] = -1;
                    full = full && jb[r] == 0 && je[r] == AT - 1;
                }
                float part[8][4];
                if (full) {
                    u64 pp[4][4];   // [row pair][column]
                    full_sum64(pp, St + grp * 8, PB, Ks + 4 * dg, PR);
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            unpack2(pp[q2][e], part[2 * q2][e], part[2 * q2 + 1][e]);
                } else {
                    // mask-edge tile: a pair of rows takes the packed step where both
                    // rows are valid and already seeded, the scalar steps elsewhere
                    int pb[4], pe[4], lo_all = AT, hi_all = -1;
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        pb[q2] = max(jb[2 * q2], jb[2 * q2 + 1]) + 1;
                        pe[q2] = min(je[2 * q2], je[2 * q2 + 1]);
                        lo_all = min(lo_all, min(jb[2 * q2], jb[2 * q2 + 1]));
                        hi_all = max(hi_all, max(je[2 * q2], je[2 * q2 + 1]));
                    }
                    u64 pp[4][4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            pp[q2][e] = 0ull;
                    // keys [from, to] through the per-pair predicated steps
                    auto edge_steps = [&](int from, int to) {
                        ulonglong2 n03 = {0ull, 0ull}, n47 = {0ull, 0ull};
                        float4 nkv = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (from <= to) {
                            n03 = *reinterpret_cast<const ulonglong2*>(St + from * PB + grp * 8);
                            n47 = *reinterpret_cast<const ulonglong2*>(St + from * PB + grp * 8 + 4);
                            nkv = *reinterpret_cast<const float4*>(Ks + from * PR + 4 * dg);
                        }
                        for (int jc = from; jc <= to; ++jc) {
                            const ulonglong2 s03 = n03, s47 = n47;
                            const float4 kv = nkv;
                            const int jn = jc < to ? jc + 1 : jc;
                            n03 = *reinterpret_cast<const ulonglong2*>(St + jn * PB + grp * 8);
                            n47 = *reinterpret_cast<const ulonglong2*>(St + jn * PB + grp * 8 + 4);
                            nkv = *reinterpret_cast<const float4*>(Ks + jn * PR + 4 * dg);
                            const u64 P[4] = {s03.x, s03.y, s47.x, s47.y};
                            const float kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                            for (int q2 = 0; q2 < 4; ++q2) {
                                if (jc >= pb[q2] && jc <= pe[q2]) {
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        pp[q2][e] = fadd2_ftz(pp[q2][e], fmul2_rn(P[q2], pack2(kk[e], kk[e])));
                                } else {
                                    float sa, sb;
                                    unpack2(P[q2], sa, sb);
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        float la, lb;
                                        unpack2(pp[q2][e], la, lb);
                                        if (jc >= jb[2 * q2] && jc <= je[2 * q2]) {
                                            const float t = fmul_rn(sa, kk[e]);
                                            la = jc == jb[2 * q2] ? flush(t) : fadd_ftz(la, t);
                                        }
                                        if (jc >= jb[2 * q2 + 1] && jc <= je[2 * q2 + 1]) {
                                            const float t = fmul_rn(sb, kk[e]);
                                            lb = jc == jb[2 * q2 + 1] ? flush(t) : fadd_ftz(lb, t);
                                        }
                                        pp[q2][e] = pack2(la, lb);
                                    }
                                }
                            }
                        }
                    };
                    // keys where every pair takes the packed step run without the
                    // per-pair tests (same operations); the ragged ends keep them
                    int mid_lo = 0, mid_hi = AT - 1;
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        mid_lo = max(mid_lo, pb[q2]);
                        mid_hi = min(mid_hi, pe[q2]);
                    }
                    if (mid_lo <= mid_hi) {
                        edge_steps(lo_all, mid_lo - 1);
                        packed_range(pp, St + grp * 8, PB, Ks + 4 * dg, PR, mid_lo, mid_hi);
                        edge_steps(mid_hi + 1, hi_all);
                    } else {
                        edge_steps(lo_all, hi_all);
                    }
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            unpack2(pp[q2][e], part[2 * q2][e], part[2 * q2 + 1][e]);
                }
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    if (jb[r] > je[r])
                        continue;
                    const int64_t i = i0 + grp * 8 + r;
                    unsigned long long* dst = a.dq_acc + ((b * T + i) * Hq + h) * HD + 4 * dg;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // fx: the 64-bit rounding conversion saturates, and a
                        // NaN partial adds 0 (that conversion would give the
                        // minimum)
                        const float x = part[r][e];
                        const long long fx = x != x ? 0ll : __float2ll_rn(fmul_rn(x, 0x1p48f));
                        atomicAdd(dst + e, (unsigned long long)fx);
                    }
                }
            }

            // dK / dV tile partials: keys grp*8 + r, columns 4dg + e, over the
            // valid query rows of this tile left to right, then folded.  Query
            // index outermost; the packed path pairs keys.  dK first, then dV
            // (one partial set live at a time).
            {
                int ib[8], ie[8];
                bool full = true;
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int64_t j = j0 + grp * 8 + r;
                    ib[r] = (int)(max(i0, j) - i0);
                    ie[r] = (int)(min(min(i0 + AT - 1, T - 1), W > 0 ? j + W - 1 : T - 1) - i0);
                    if (j >= T)
                        ib[r] = AT, ie[r] = -1;
                    full = full && ib[r] == 0 && ie[r] == AT - 1;
                }
#pragma unroll 1
                for (int which = 0; which < 2; ++which) {
                    // which 0: dK terms dS_ij (x) q_id; which 1: dV terms a_ij (x) dO_id
                    const float* Wt = which == 0 ? Ss : As;
                    const float* Xr = which == 0 ? Qs : Gs;
                    float pt[8][4];
                    if (full) {
                        u64 pp[4][4];   // [key pair][column]
                        full_sum64(pp, Wt + grp * 8, PB, Xr + 4 * dg, PR);
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                unpack2(pp[q2][e], pt[2 * q2][e], pt[2 * q2 + 1][e]);
                    } else {
                        // mask-edge tile: a pair of keys takes the packed step where
                        // both keys are valid and already seeded, scalar steps elsewhere
                        int pb[4], pe[4], lo_all = AT, hi_all = -1;
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            pb[q2] = max(ib[2 * q2], ib[2 * q2 + 1]) + 1;
                            pe[q2] = min(ie[2 * q2], ie[2 * q2 + 1]);
                            lo_all = min(lo_all, min(ib[2 * q2], ib[2 * q2 + 1]));
                            hi_all = max(hi_all, max(ie[2 * q2], ie[2 * q2 + 1]));
                        }
                        u64 pp[4][4];
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                pp[q2][e] = 0ull;
                        // query rows [from, to] through the per-pair predicated steps
                        auto edge_steps = [&](int from, int to) {
                            ulonglong2 n03 = {0ull, 0ull}, n47 = {0ull, 0ull};
                            float4 nxv = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (from <= to) {
                                n03 = *reinterpret_cast<const ulonglong2*>(Wt + from * PB + grp * 8);
                                n47 = *reinterpret_cast<const ulonglong2*>(Wt + from * PB + grp * 8 + 4);
                                nxv = *reinterpret_cast<const float4*>(Xr + from * PR + 4 * dg);
                            }
                            for (int ir = from; ir <= to; ++ir) {
                                const ulonglong2 w03 = n03, w47 = n47;
                                const float4 xv = nxv;
                                const int rn = ir < to ? ir + 1 : ir;
                                n03 = *reinterpret_cast<const ulonglong2*>(Wt + rn * PB + grp * 8);
                                n47 = *reinterpret_cast<const ulonglong2*>(Wt + rn * PB + grp * 8 + 4);
                                nxv = *reinterpret_cast<const float4*>(Xr + rn * PR + 4 * dg);
                                const u64 P[4] = {w03.x, w03.y, w47.x, w47.y};
                                const float xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                                for (int q2 = 0; q2 < 4; ++q2) {
                                    if (ir >= pb[q2] && ir <= pe[q2]) {
#pragma unroll
                                        for (int e = 0; e < 4; ++e)
                                            pp[q2][e] = fadd2_ftz(pp[q2][e], fmul2_rn(P[q2], pack2(xx[e], xx[e])));
                                    } else {
                                        float wa, wb;
                                        unpack2(P[q2], wa, wb);
#pragma unroll
                                        for (int e = 0; e < 4; ++e) {
                                            float la, lb;
                                            unpack2(pp[q2][e], la, lb);
                                            if (ir >= ib[2 * q2] && ir <= ie[2 * q2]) {
                                                const float t = fmul_rn(wa, xx[e]);
                                                la = ir == ib[2 * q2] ? flush(t) : fadd_ftz(la, t);
                                            }
                                            if (ir >= ib[2 * q2 + 1] && ir <= ie[2 * q2 + 1]) {
                                                const float t = fmul_rn(wb, xx[e]);
                                                lb = ir == ib[2 * q2 + 1] ? flush(t) : fadd_ftz(lb, t);
                                            }
                                            pp[q2][e] = pack2(la, lb);
                                        }
                                    }
                                }
                            }
                        };
                        // rows where every pair takes the packed step run without the
                        // per-pair tests (same operations); the ragged ends keep them
                        int mid_lo = 0, mid_hi = AT - 1;
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) {
                            mid_lo = max(mid_lo, pb[q2]);
                            mid_hi = min(mid_hi, pe[q2]);
                        }
                        if (mid_lo <= mid_hi) {
                            edge_steps(lo_all, mid_lo - 1);
                            packed_range(pp, Wt + grp * 8, PB, Xr + 4 * dg, PR, mid_lo, mid_hi);
                            edge_steps(mid_hi + 1, hi_all);
                        } else {
                            edge_steps(lo_all, hi_all);
                        }
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                unpack2(pp[q2][e], pt[2 * q2][e], pt[2 * q2 + 1][e]);
                    }
                    // fold (keys and their ranges are the same for every lane of a warp)
                    float f[32];
                    const uint32_t ta = tfold + (uint32_t)(32 * which);
                    tm_ld32(ta, f);
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        if (ib[r] > ie[r])
                            continue;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            f[r * 4 + e] = started[r] ? fadd_ftz(f[r * 4 + e], pt[r][e]) : pt[r][e];
                    }
                    tm_st32(ta, f);
                }
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (ib[r] <= ie[r])
                        started[r] = true;
            }
        }
    }

    {
        float fk[32], fv[32];
        tm_ld32(tfold, fk);
        tm_ld32(tfold + 32, fv);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int64_t j = j0 + grp * 8 + r;
            if (j >= T)
                continue;
            const int64_t off = ((b * T + j) * Hkv + g) * HD + 4 * dg;
            *reinterpret_cast<float4*>(a.dk + off) =
                make_float4(fmul_flush(fk[4 * r], c), fmul_flush(fk[4 * r + 1], c),
                            fmul_flush(fk[4 * r + 2], c), fmul_flush(fk[4 * r + 3], c));
            *reinterpret_cast<float4*>(a.dv + off) =
                make_float4(fv[4 * r], fv[4 * r + 1], fv[4 * r + 2], fv[4 * r + 3]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid < 32) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(*tslot)
                     : "memory");
    }
}

// Dr_i = canon_d(dO_id (x) O_id) for 64 rows per CTA (rows contiguous, 128 floats)
__global__ void __launch_bounds__(NT) k_attn_drow(const float* __restrict__ o,
                                                 const float* __restrict__ dout,
                                                 float* __restrict__ drow, int64_t nrows)
{
    __shared__ float prod[AT * 129];
    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * AT;
#pragma unroll
    for (int it = 0; it < (AT * HD / 4) / NT; ++it) {
        const int e = tid + it * NT;
        const int r = e >> 5, c4 = e & 31;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f), y = x;
        if (r0 + r < nrows) {
            x = flush4(*reinterpret_cast<const float4*>(dout + (r0 + r) * HD + 4 * c4));
            y = flush4(*reinterpret_cast<const float4*>(o + (r0 + r) * HD + 4 * c4));
        }
        prod[r * 129 + 4 * c4 + 0] = fmul_rn(x.x, y.x);
        prod[r * 129 + 4 * c4 + 1] = fmul_rn(x.y, y.y);
        prod[r * 129 + 4 * c4 + 2] = fmul_rn(x.z, y.z);
        prod[r * 129 + 4 * c4 + 3] = fmul_rn(x.w, y.w);
    }
    __syncthreads();
    if (tid < AT && r0 + tid < nrows) {
        const float* p = prod + tid * 129;
        float t0 = flush(p[0]);
        for (int d = 1; d < 64; ++d)
            t0 = fadd_ftz(t0, p[d]);
        float t1 = flush(p[64]);
        for (int d = 65; d < 128; ++d)
            t1 = fadd_ftz(t1, p[d]);
        drow[r0 + tid] = fadd_ftz(t0, t1);
    }
}

// dQ = flush(i2f(acc) * 2^-48) (x) c
__global__ void __launch_bounds__(NT) k_attn_dq_final(const unsigned long long* __restrict__ acc,
                                                     float* __restrict__ dq, int64_t n, float c)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const float f = flush(fmul_rn(__ll2float_rn((long long)acc[e]), 0x1p-48f));
        dq[e] = fmul_flush(f, c);
    }
}

// ---------------------------------------------------------------------------
// Backward, default route (with the forward's cache).  Same arithmetic and
// orders as k_attn_bwd; the work is split by what each output needs:
//   k_attn_bimg        flushed copies of K, Q and dO by 64-row tile, the
//                      dequantised V^T by key tile, the work counters zeroed;
//   k_attn_rows<true>  per query tile (the forward logits kernel's
//                      structure): dA = canon_d(dO (x) V^), then a and dS from
//                      the cached p, written as [row][key] tiles (pitch BT_P);
//   k_attn_bdq         per query tile: each key tile's left-to-right dQ
//                      partial, into 64-bit fixed point in registers (no
//                      atomics), then dQ;
//   k_attn_bdkv        per key tile: the dK and dV group partials, folded
//                      left in (head, query tile) order in registers.
constexpr uint32_t ROW_TILE = AT * HD * 4;   // 64 rows x 128 floats

struct AttnBwdImg {
    const float* k;
    const int8_t* vq;
    const float* s_v;
    const float* q;
    const float* dout;
    float* vimg;   // [B][Hkv][nkt] x [d][key], dequantised and flushed
    float* krow;   // [B][Hkv][nkt] x [key][d], flushed
    float* qrow;   // [B][Hq][nkt] x [row][d], flushed
    float* grow;   // [B][Hq][nkt] x [row][d], flushed dO
    unsigned long long* counters;
    int64_t B, T, Hq, Hkv, nkt;
};

// blockIdx.y: 0 V^T, 1 K rows, 2 Q rows, 3 dO rows; rows at or past T are 0
__global__ void k_attn_bimg(const AttnBwdImg a)
{
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 4)
        a.counters[threadIdx.x] = 0;
    const int part = blockIdx.y;
    const int64_t H = part >= 2 ? a.Hq : a.Hkv;
    const int64_t n = a.B * H * a.nkt * (AT * HD / 4);
    const float sv = flush(*a.s_v);
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        if (part == 0) {   // key fastest: the transposed stores are contiguous
            const int key = (int)(e & (AT - 1));
            const int d4 = (int)((e >> 6) & (HD / 4 - 1));
            const int64_t tile = e >> 11;
            const int64_t t = tile % a.nkt, bh = tile / a.nkt;
            const int64_t j = t * AT + key;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < a.T) {
                const int w = *reinterpret_cast<const int*>(a.vq + ((bh / H * a.T + j) * H + bh % H) * HD + 4 * d4);
                v = make_float4(dequant((int)(int8_t)w, sv), dequant((int)(int8_t)(w >> 8), sv),
                                dequant((int)(int8_t)(w >> 16), sv), dequant((int)(int8_t)(w >> 24), sv));
            }
            float* dst = a.vimg + tile * (HD * AT) + (4 * d4) * AT + key;
            dst[0] = v.x;
            dst[AT] = v.y;
            dst[2 * AT] = v.z;
            dst[3 * AT] = v.w;
        } else {           // d fastest: rows copied whole
            const int d4 = (int)(e & (HD / 4 - 1));
            const int key = (int)((e >> 5) & (AT - 1));
            const int64_t tile = e >> 11;
            const int64_t t = tile % a.nkt, bh = tile / a.nkt;
            const int64_t j = t * AT + key;
            const float* src = part == 1 ? a.k : (part == 2 ? a.q : a.dout);
            float* img = part == 1 ? a.krow : (part == 2 ? a.qrow : a.grow);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < a.T)
                v = flush4(*reinterpret_cast<const float4*>(src + ((bh / H * a.T + j) * H + bh % H) * HD + 4 * d4));
            *reinterpret_cast<float4*>(img + tile * (AT * HD) + key * HD + 4 * d4) = v;
        }
    }
}


// fx(v) = the nearest int64 to v (x) 2^48, ties to even, saturating, for the
// two lanes of a pair -- the value of the 64-bit rounding conversion, which
// runs on the FP64 pipe, built from two 32-bit ones.  For a flushed v,
// |y| = |v| (x) 2^48 is exact unless it overflows.  |y| = h 2^32 + l with
// h = trunc(|y| 2^-32) and l = |y| (-) h 2^32, both exact (l is |y| when
// |y| < 2^32, else a multiple of |y|'s spacing below 2^32), so
// rn(|y|) = h 2^32 + rn(l) (h 2^32 is even) with h < 2^31 and rn(l) < 2^32;
// then the sign.  |y| >= 2^63 (or infinite) saturates; NaN converts to 0 in
// both halves.  No branches
__device__ __forceinline__ void fx48x2(u64 vv, unsigned long long& r0, unsigned long long& r1)
{
    float v[2];
    unpack2(vv, v[0], v[1]);
    float a[2] = {fabsf(v[0]), fabsf(v[1])};
    unpack2(fmul2_rn(pack2(a[0], a[1]), pack2(0x1p48f, 0x1p48f)), a[0], a[1]);
    float hs[2];
    unpack2(fmul2_rn(pack2(a[0], a[1]), pack2(0x1p-32f, 0x1p-32f)), hs[0], hs[1]);
    const float h0 = truncf(hs[0]), h1 = truncf(hs[1]);
    float l[2];
    unpack2(fadd2_ftz(pack2(a[0], a[1]), fmul2_rn(pack2(h0, h1), pack2(-0x1p32f, -0x1p32f))), l[0], l[1]);
    const float hf[2] = {h0, h1};
    unsigned long long out[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const unsigned long long mag =
            ((unsigned long long)__float2uint_rz(hf[x]) << 32) | (unsigned long long)__float2uint_rn(l[x]);
        const bool neg = __float_as_uint(v[x]) >> 31;
        unsigned long long r = neg ? 0ull - mag : mag;
        if (a[x] >= 0x1p63f)
            r = neg ? 0x8000000000000000ull : 0x7fffffffffffffffull;
        out[x] = r;
    }
    r0 = out[0];
    r1 = out[1];
}

struct AttnDqArgs {
    const float* st;     // dS tiles
    const float* krow;   // flushed K rows
    float* dq;
    unsigned long long* counter;
    int64_t T, Hq, Hkv, W, tiles_bh, nqt, nkt, items;
    float c;
    int* err;
};

constexpr int DQ_STAGE = (int)(BT_TILE + ROW_TILE);   // one dS tile and its K rows
constexpr size_t DQ_SMEM = 2 * (size_t)DQ_STAGE;

// dQ of one query tile at a time per CTA (256 threads, two CTAs per SM): a thread owns
// rows 4ty .. 4ty+3 and columns 4tx .. 4tx+3 and 64 + 4tx .. 64 + 4tx+3 (one
// 16-byte load each, contiguous across the warp: no bank conflicts) as four
// packed pairs along d, so a pair shares its row and its keys.  Per key tile: the left-to-right sum
// over the row's valid keys, from the first (flushed) product, then
// fx(x) = nearest int64 to x (x) 2^48 added in registers; at the end
// dQ = fix2f(sum) (x) c.  The dS tile and the key tile's K rows arrive by bulk
// copies into a two-stage ring released per warp; query tiles come from a
// counter, longest windows first
__global__ void __launch_bounds__(NT, 2) k_attn_bdq(const AttnDqArgs a)
{
    extern __shared__ __align__(128) uint8_t smq[];
    __shared__ uint64_t full[2], empty[2];
    __shared__ int64_t queue[8];
    __shared__ uint32_t tmem_slot;
    const int lt = threadIdx.x, lane = lt & 31;
    const int ty = lt >> 4, tx = lt & 15;
    if (lt == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NT / 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (lt < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(
                         su32(&tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    // this thread's 32 fixed-point sums live in its own tensor-memory lane:
    // lane 32 (warp % 4) + lane, columns 128 (warp / 4) .. + 63 (two 32-bit
    // columns per sum), keeping registers for two CTAs per SM; the next 32
    // columns park a key tile's 32 partials until the next key tile's loop
    // converts them (sum v at column 32 (v / 16) + 2 (v % 16), partial v at
    // 64 + v, v = 8 row + 2 pair + lane)
    const uint32_t tacc =
        tmem_slot + ((uint32_t)(32 * ((lt >> 5) & 3)) << 16) + (uint32_t)(128 * (lt >> 7));
    const int T = (int)a.T, W = (int)a.W;
    auto tile_of = [&](const QTile& q, int t) {   // the cache tile of (query tile q, key tile t)
        return ((q.b * a.Hq + q.h) * a.tiles_bh + tile_prefix(q.i0 / AT, W)) + (t - q.t_lo);
    };
    auto qtile = [&](int64_t item) {
        QTile r;
        const int qt = (int)(item % a.nqt);
        const int64_t bh = item / a.nqt;
        r.h = bh % a.Hq;
        r.b = bh / a.Hq;
        r.g = r.h / (a.Hq / a.Hkv);
        r.i0 = qt * AT;
        const int jlo = W > 0 ? max(0, r.i0 - W + 1) : 0;
        r.t_lo = jlo / AT;
        r.t_hi = min(r.i0 + AT - 1, T - 1) / AT;
        return r;
    };
    auto item_k = [&](int64_t k) {   // longest windows first
        const int64_t bhs = a.items / a.nqt;
        return (a.nqt - 1 - k / bhs) * 1 + (k % bhs) * a.nqt;
    };

    // issuer (thread 0): as the logits kernel's
    int iss_k = 0, iss_t = 0;
    bool have = false;
    uint32_t issued = 0;
    QTile iss_q;
    auto take = [&](int kslot) {
        const int64_t k = (int64_t)atomicAdd(a.counter, 1ull);
        queue[kslot & 7] = k < a.items ? item_k(k) : -1;
    };
    auto start = [&](int kslot) {
        const int64_t item = queue[kslot & 7];
        have = item >= 0;
        if (have) {
            take(kslot + 1);
            iss_q = qtile(item);
            iss_t = iss_q.t_lo;
        }
    };
    auto issue_next = [&]() {
        if (!have)
            return;
        const int s = issued & 1;
        uint8_t* stage = smq + s * DQ_STAGE;
        mbar_expect_tx(&full[s], BT_TILE + ROW_TILE);
        bulk_load(stage, a.st + tile_of(iss_q, iss_t) * (AT * BT_P), BT_TILE, &full[s]);
        bulk_load(stage + BT_TILE, a.krow + ((iss_q.b * a.Hkv + iss_q.g) * a.nkt + iss_t) * (AT * HD), ROW_TILE,
                  &full[s]);
        ++issued;
        if (++iss_t > iss_q.t_hi)
            start(++iss_k);
    };
    if (lt == 0) {
        take(0);
        start(0);
        issue_next();
        issue_next();
    }

    // partials v = 4c .. 4c + 3 of the previous key tile, parked in tensor
    // memory, into the fixed-point sums (the first key tile's start them); a
    // row without keys there parked +0, which adds nothing
    auto defer_chunk = [&](int c, bool first) {
        uint32_t rw[4], sw[8];
        const uint32_t scol = tacc + 32 * (c >> 2) + 8 * (c & 3);
        tmem_ld4_ld8(tacc + 64 + 4 * c, rw, scol, sw);
        u64 fx[4];
        fx48x2((u64)rw[0] | ((u64)rw[1] << 32), fx[0], fx[1]);
        fx48x2((u64)rw[2] | ((u64)rw[3] << 32), fx[2], fx[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            u64 f = fx[e];
            if (!first)
                f += (u64)sw[2 * e] | ((u64)sw[2 * e + 1] << 32);
            sw[2 * e] = (uint32_t)f;
            sw[2 * e + 1] = (uint32_t)(f >> 32);
        }
        tmem_st8(scol, sw);
    };
    uint32_t used = 0;
    bool fail = false, dead = false;
    const u64 z = pack2(-0.0f, -0.0f);
    for (int kk = 0;; ++kk) {
        dead = __syncthreads_or(fail || dead) != 0;   // also publishes the queue entry
        const int64_t item = queue[kk & 7];
        if (dead || item < 0)
            break;
        const QTile qt = qtile(item);
        for (int t = qt.t_lo; t <= qt.t_hi; ++t) {
            const int s = used & 1;
            if (lt == 0 && used >= 1 && issued == used + 1 && have) {
                if (mbar_wait(&empty[s ^ 1], ((used - 1) >> 1) & 1))
                    issue_next();
                else
                    fail = true;
            }
            if (!mbar_wait(&full[s], (used >> 1) & 1))
                fail = true;
            const float* S = reinterpret_cast<const float*>(smq + s * DQ_STAGE) + 4 * ty * BT_P;
            const float* Kr = reinterpret_cast<const float*>(smq + s * DQ_STAGE + BT_TILE) + 4 * tx;
            const int j0 = t * AT;
            int jb[4], je[4];
            bool whole = true;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = qt.i0 + 4 * ty + r;
                const int lo = W > 0 ? max(0, i - W + 1) : 0;
                jb[r] = max(lo, j0) - j0;
                je[r] = min(i, j0 + AT - 1) - j0;
                if (i >= T)
                    jb[r] = AT, je[r] = -1;
                whole = whole && jb[r] == 0 && je[r] == AT - 1;
            }
            // one path per warp (the edge path's warp reductions need every lane)
            whole = __all_sync(0xffffffffu, whole);
            u64 pp[4][4];   // [row][pair of columns]
            // operands of the next key, loaded one key ahead
            float sv[4];
            ulonglong2 k01, k23;
            auto load = [&](int j) {
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    sv[r] = S[r * BT_P + j];
                k01 = *reinterpret_cast<const ulonglong2*>(Kr + j * HD);
                k23 = *reinterpret_cast<const ulonglong2*>(Kr + j * HD + HD / 2);
            };
            // one key with every row valid: the products of row r + 1 formed
            // before the adds of row r, so no add waits on the multiply just
            // issued; FIRST seeds the sums with the flushed products; then key
            // `jn` is loaded
            auto key = [&](auto first_tag, int jn) {
                constexpr bool FIRST = decltype(first_tag)::value;
                const u64 D[4] = {k01.x, k01.y, k23.x, k23.y};
                const float c4[4] = {sv[0], sv[1], sv[2], sv[3]};
                load(jn);
                u64 cur[4];
                {
                    const u64 P = pack2(c4[0], c4[0]);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        cur[q] = fmul2_rn(P, D[q]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    u64 nxt[4];
                    if (r + 1 < 4) {
                        const u64 P = pack2(c4[r + 1], c4[r + 1]);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            nxt[q] = fmul2_rn(P, D[q]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        pp[r][q] = FIRST ? fadd2_ftz(cur[q], z) : fadd2_ftz(pp[r][q], cur[q]);
                    if (r + 1 < 4) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            cur[q] = nxt[q];
                    }
                }
            };
            // the previous key tile's partials, converted a chunk at a time
            // between groups of 8 keys (whole tiles) or before the keys (edge
            // tiles), so the integer work overlaps the products
            const bool defer = t > qt.t_lo, pfirst = t - 1 == qt.t_lo;
            if (whole) {
                load(0);
                key(std::true_type{}, 1);
#pragma unroll
                for (int j = 1; j < 8; ++j)
                    key(std::false_type{}, j + 1);
                if (defer)
                    defer_chunk(0, pfirst);
#pragma unroll 1
                for (int g = 1; g < AT / 8; ++g) {
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = 8 * g + jj;
                        key(std::false_type{}, j + 1 < AT ? j + 1 : j);
                    }
                    if (defer)
                        defer_chunk(g, pfirst);
                }
            } else {
                if (defer)
#pragma unroll 1
                    for (int c = 0; c < 8; ++c)
                        defer_chunk(c, pfirst);
                // mask-edge tile: each row over its own range of keys.  Keys
                // where all four rows of every thread of the warp are valid and
                // already seeded take the packed keys without tests (same
                // operations); the ragged ends keep them
                int lo_all = AT, hi_all = -1, mid_lo = 0, mid_hi = AT - 1;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    lo_all = min(lo_all, jb[r]);
                    hi_all = max(hi_all, je[r]);
                    mid_lo = max(mid_lo, jb[r] + 1);
                    mid_hi = min(mid_hi, je[r]);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        pp[r][q] = 0ull;
                }
                lo_all = __reduce_min_sync(0xffffffffu, lo_all);
                hi_all = __reduce_max_sync(0xffffffffu, hi_all);
                mid_lo = __reduce_max_sync(0xffffffffu, mid_lo);
                mid_hi = __reduce_min_sync(0xffffffffu, mid_hi);
                auto edge = [&](int from, int to) {
                    for (int j = from; j <= to; ++j) {
                        const ulonglong2 e01 = *reinterpret_cast<const ulonglong2*>(Kr + j * HD);
                        const ulonglong2 e23 = *reinterpret_cast<const ulonglong2*>(Kr + j * HD + HD / 2);
                        const u64 D[4] = {e01.x, e01.y, e23.x, e23.y};
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            if (j < jb[r] || j > je[r])
                                continue;
                            const float w = S[r * BT_P + j];
                            const u64 P = pack2(w, w);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const u64 pr = fmul2_rn(P, D[q]);
                                pp[r][q] = j == jb[r] ? fadd2_ftz(pr, z) : fadd2_ftz(pp[r][q], pr);
                            }
                        }
                    }
                };
                if (mid_lo <= mid_hi) {
                    edge(lo_all, mid_lo - 1);
                    load(mid_lo);
                    for (int j = mid_lo; j <= mid_hi; ++j)
                        key(std::false_type{}, j + 1 <= mid_hi ? j + 1 : j);
                    edge(mid_hi + 1, hi_all);
                } else {
                    edge(lo_all, hi_all);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
            ++used;
            if (t < qt.t_hi) {
                // parked for the next key tile's loop
                const u64 flat[16] = {pp[0][0], pp[0][1], pp[0][2], pp[0][3], pp[1][0], pp[1][1],
                                      pp[1][2], pp[1][3], pp[2][0], pp[2][1], pp[2][2], pp[2][3],
                                      pp[3][0], pp[3][1], pp[3][2], pp[3][3]};
                tmem_st32(tacc + 64, flat);
                continue;
            }
            // the query tile's last key tile: its partials into the fixed-point
            // sums now (wrapping like the int64 adds they replace); rows
            // without keys here add nothing
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {   // rows 2hf, 2hf + 1: 16 sums, 32 columns
                u64 f[16];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = 2 * hf + rr;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        u64 c0, c1;
                        fx48x2(pp[r][q], c0, c1);
                        const bool any = jb[r] <= je[r];
                        f[8 * rr + 2 * q] = any ? c0 : 0ull;
                        f[8 * rr + 2 * q + 1] = any ? c1 : 0ull;
                    }
                }
                if (t != qt.t_lo) {
                    uint32_t w[32];
                    tmem_ld32(tacc + 32 * hf, w);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        f[e] += (u64)w[2 * e] | ((u64)w[2 * e + 1] << 32);
                }
                tmem_st32(tacc + 32 * hf, f);
            }
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t w[32];
            tmem_ld32(tacc + 32 * hf, w);
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
            const int r = 2 * hf + rr;
            const int64_t i = qt.i0 + 4 * ty + r;
            if (i >= T)
                continue;
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const long long acc = (long long)((u64)w[2 * (8 * rr + e)] | ((u64)w[2 * (8 * rr + e) + 1] << 32));
                o[e] = fmul_flush(flush(fmul_rn(__ll2float_rn(acc), 0x1p-48f)), a.c);
            }
            float* dst = a.dq + ((qt.b * a.T + i) * a.Hq + qt.h) * HD + 4 * tx;
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(dst + HD / 2) = make_float4(o[4], o[5], o[6], o[7]);
            }
        }
    }
    if (lt == 0)
        while (used < issued && mbar_wait(&full[used & 1], (used >> 1) & 1))
            ++used;
    fence_before();
    __syncthreads();
    if (lt < 32) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem_slot) : "memory");
    }
    if (fail)
        atomicExch(a.err, 1);
}

struct AttnDkvArgs {
    const float* at;     // a tiles
    const float* st;     // dS tiles
    const float* qrow;   // flushed Q rows
    const float* grow;   // flushed dO rows
    float* dk;
    float* dv;
    unsigned long long* counter;
    int64_t B, T, Hq, Hkv, W, tiles_bh, nqt, items;
    float c;
    int* err;
};

constexpr int KV_STAGE = (int)(2 * BT_TILE + 2 * ROW_TILE);   // dS, a, Q rows, dO rows
constexpr size_t KV_SMEM = 2 * (size_t)KV_STAGE;

// dK and dV of one key tile at a time per CTA (256 threads, one CTA per SM).
// A thread owns keys 4ty .. 4ty+3 and columns 4tx .. 4tx+3 and 64 + 4tx ..
// 64 + 4tx+3 (conflict-free 16-byte loads) as four packed pairs along d, so a
// pair shares its key and its range of queries.  The
// groups (query head of the kv head, 64-aligned query tile) come in ascending
// order; per group each key's partial is the left-to-right sum over its valid
// queries from the first (flushed) product, and the partials are folded left
// in registers.  dK = F_K (x) c, dV = F_V.  A group's dS and a tiles and its
// flushed Q and dO rows arrive by bulk copies into a two-stage ring released
// per warp; key tiles come from a counter, longest first
__global__ void __launch_bounds__(NT, 1) k_attn_bdkv(const AttnDkvArgs a)
{
    extern __shared__ __align__(128) uint8_t smk[];
    __shared__ uint64_t full[2], empty[2];
    __shared__ int64_t queue[8];
    const int lt = threadIdx.x, lane = lt & 31;
    const int ty = lt >> 4, tx = lt & 15;
    if (lt == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NT / 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int T = (int)a.T, W = (int)a.W;
    const int64_t G = a.Hq / a.Hkv;
    // key tile: (sequence, kv head, tile) and its query tiles
    struct KTile {
        int64_t b, g;
        int t, u_lo, u_hi;   // query tiles u_lo .. u_hi of every head in the group
    };
    auto ktile = [&](int64_t item) {
        KTile r;
        const int64_t bgs = a.B * a.Hkv;
        r.t = (int)(item / bgs);
        const int64_t bg = item % bgs;
        r.b = bg / a.Hkv;
        r.g = bg % a.Hkv;
        r.u_lo = r.t;
        const int last = W > 0 ? min(T - 1, r.t * AT + AT - 1 + W - 1) : T - 1;
        r.u_hi = last / AT;
        return r;
    };
    // the cache tile of (query tile u of head h, key tile t)
    auto tile_of = [&](int64_t b, int64_t h, int u, int t) {
        const int t_lo = (W > 0 ? max(0, u * AT - W + 1) : 0) / AT;
        return (b * a.Hq + h) * a.tiles_bh + tile_prefix(u, W) + (t - t_lo);
    };

    // issuer (thread 0): the groups of each key tile in order
    int iss_k = 0, iss_h = 0, iss_u = 0;
    bool have = false;
    uint32_t issued = 0;
    KTile iss_q;
    auto take = [&](int kslot) {
        const int64_t k = (int64_t)atomicAdd(a.counter, 1ull);
        queue[kslot & 7] = k < a.items ? k : -1;   // hand-out order: key tile 0 (longest) first
    };
    auto start = [&](int kslot) {
        const int64_t item = queue[kslot & 7];
        have = item >= 0;
        if (have) {
            take(kslot + 1);
            iss_q = ktile(item);
            iss_h = 0;
            iss_u = iss_q.u_lo;
        }
    };
    auto issue_next = [&]() {
        if (!have)
            return;
        const int s = issued & 1;
        uint8_t* stage = smk + s * KV_STAGE;
        const int64_t h = iss_q.g * G + iss_h;
        const int64_t tl = tile_of(iss_q.b, h, iss_u, iss_q.t) * (AT * BT_P);
        const int64_t rl = ((iss_q.b * a.Hq + h) * a.nqt + iss_u) * (AT * HD);
        mbar_expect_tx(&full[s], 2 * BT_TILE + 2 * ROW_TILE);
        bulk_load(stage, a.st + tl, BT_TILE, &full[s]);
        bulk_load(stage + BT_TILE, a.at + tl, BT_TILE, &full[s]);
        bulk_load(stage + 2 * BT_TILE, a.qrow + rl, ROW_TILE, &full[s]);
        bulk_load(stage + 2 * BT_TILE + ROW_TILE, a.grow + rl, ROW_TILE, &full[s]);
        ++issued;
        if (++iss_u > iss_q.u_hi) {
            iss_u = iss_q.u_lo;
            if (++iss_h == G)
                start(++iss_k);
        }
    };
    if (lt == 0) {
        take(0);
        start(0);
        issue_next();
        issue_next();
    }

    uint32_t used = 0;
    bool fail = false, dead = false;
    const u64 z = pack2(-0.0f, -0.0f);
    for (int kk = 0;; ++kk) {
        dead = __syncthreads_or(fail || dead) != 0;   // also publishes the queue entry
        const int64_t item = queue[kk & 7];
        if (dead || item < 0)
            break;
        const KTile kt = ktile(item);
        const int j0 = kt.t * AT;
        u64 fk[4][4], fv[4][4];   // [key][pair of columns]
        bool started[4] = {false, false, false, false};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                fk[r][q] = fv[r][q] = 0ull;
        for (int hh = 0; hh < G; ++hh)
            for (int u = kt.u_lo; u <= kt.u_hi; ++u) {
                const int s = used & 1;
                if (lt == 0 && used >= 1 && issued == used + 1 && have) {
                    if (mbar_wait(&empty[s ^ 1], ((used - 1) >> 1) & 1))
                        issue_next();
                    else
                        fail = true;
                }
                if (!mbar_wait(&full[s], (used >> 1) & 1))
                    fail = true;
                const uint8_t* stage = smk + s * KV_STAGE;
                const float* S = reinterpret_cast<const float*>(stage) + 4 * ty;
                const float* A = reinterpret_cast<const float*>(stage + BT_TILE) + 4 * ty;
                const float* Qr = reinterpret_cast<const float*>(stage + 2 * BT_TILE) + 4 * tx;
                const float* Gr = reinterpret_cast<const float*>(stage + 2 * BT_TILE + ROW_TILE) + 4 * tx;
                const int i0 = u * AT;
                int ib[4], ie[4];
                bool whole = true;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int j = j0 + 4 * ty + r;
                    ib[r] = max(i0, j) - i0;
                    ie[r] = min(min(i0 + AT - 1, T - 1), W > 0 ? j + W - 1 : T - 1) - i0;
                    if (j >= T)
                        ib[r] = AT, ie[r] = -1;
                    whole = whole && ib[r] == 0 && ie[r] == AT - 1;
                }
                // one path per warp (the edge path's warp reductions need every lane)
                whole = __all_sync(0xffffffffu, whole);
                u64 pk[4][4], pv[4][4];
                // operands of the next query row, loaded one row ahead
                float4 sw, aw;
                ulonglong2 q01, q23, g01, g23;
                auto load = [&](int i) {
                    sw = *reinterpret_cast<const float4*>(S + i * BT_P);
                    aw = *reinterpret_cast<const float4*>(A + i * BT_P);
                    q01 = *reinterpret_cast<const ulonglong2*>(Qr + i * HD);
                    q23 = *reinterpret_cast<const ulonglong2*>(Qr + i * HD + HD / 2);
                    g01 = *reinterpret_cast<const ulonglong2*>(Gr + i * HD);
                    g23 = *reinterpret_cast<const ulonglong2*>(Gr + i * HD + HD / 2);
                };
                // one query row with every key valid: the 8 (key, tensor) rows of
                // products, those of row x + 1 formed before the adds of row x;
                // FIRST seeds the sums with the flushed products; then row `in`
                // is loaded
                auto row = [&](auto first_tag, int in) {
                    constexpr bool FIRST = decltype(first_tag)::value;
                    const float w8[8] = {sw.x, sw.y, sw.z, sw.w, aw.x, aw.y, aw.z, aw.w};
                    const u64 DQ[4] = {q01.x, q01.y, q23.x, q23.y}, DG[4] = {g01.x, g01.y, g23.x, g23.y};
                    load(in);
                    u64 cur[4];
                    {
                        const u64 P = pack2(w8[0], w8[0]);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            cur[q] = fmul2_rn(P, DQ[q]);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        u64 nxt[4];
                        if (x + 1 < 8) {
                            const u64 P = pack2(w8[x + 1], w8[x + 1]);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                nxt[q] = fmul2_rn(P, x + 1 < 4 ? DQ[q] : DG[q]);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            u64& acc = x < 4 ? pk[x][q] : pv[x - 4][q];
                            acc = FIRST ? fadd2_ftz(cur[q], z) : fadd2_ftz(acc, cur[q]);
                        }
                        if (x + 1 < 8) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                cur[q] = nxt[q];
                        }
                    }
                };
                if (whole) {
                    load(0);
                    row(std::true_type{}, 1);
#pragma unroll 3
                    for (int i = 1; i < AT; ++i)
                        row(std::false_type{}, i + 1 < AT ? i + 1 : i);
                } else {
                    // mask-edge group: each key over its own range of queries.
                    // Rows where all four keys of every thread of the warp are
                    // valid and already seeded take the packed rows without
                    // tests (same operations); the ragged ends keep them
                    int lo_all = AT, hi_all = -1, mid_lo = 0, mid_hi = AT - 1;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        lo_all = min(lo_all, ib[r]);
                        hi_all = max(hi_all, ie[r]);
                        mid_lo = max(mid_lo, ib[r] + 1);
                        mid_hi = min(mid_hi, ie[r]);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            pk[r][q] = pv[r][q] = 0ull;
                    }
                    lo_all = __reduce_min_sync(0xffffffffu, lo_all);
                    hi_all = __reduce_max_sync(0xffffffffu, hi_all);
                    mid_lo = __reduce_max_sync(0xffffffffu, mid_lo);
                    mid_hi = __reduce_min_sync(0xffffffffu, mid_hi);
                    auto edge = [&](int from, int to) {
                        for (int i = from; i <= to; ++i) {
                            load(i);
                            const float ws[4] = {sw.x, sw.y, sw.z, sw.w}, wa[4] = {aw.x, aw.y, aw.z, aw.w};
                            const u64 DQ[4] = {q01.x, q01.y, q23.x, q23.y}, DG[4] = {g01.x, g01.y, g23.x, g23.y};
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                if (i < ib[r] || i > ie[r])
                                    continue;
                                const u64 PS = pack2(ws[r], ws[r]), PA = pack2(wa[r], wa[r]);
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const u64 xk = fmul2_rn(PS, DQ[q]), xv = fmul2_rn(PA, DG[q]);
                                    pk[r][q] = i == ib[r] ? fadd2_ftz(xk, z) : fadd2_ftz(pk[r][q], xk);
                                    pv[r][q] = i == ib[r] ? fadd2_ftz(xv, z) : fadd2_ftz(pv[r][q], xv);
                                }
                            }
                        }
                    };
                    if (mid_lo <= mid_hi) {
                        edge(lo_all, mid_lo - 1);
                        load(mid_lo);
                        for (int i = mid_lo; i <= mid_hi; ++i)
                            row(std::false_type{}, i + 1 <= mid_hi ? i + 1 : i);
                        edge(mid_hi + 1, hi_all);
                    } else {
                        edge(lo_all, hi_all);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[s]);
                ++used;
                // fold the group partials, left to right over the groups
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if (ib[r] > ie[r])
                        continue;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        fk[r][q] = started[r] ? fadd2_ftz(fk[r][q], pk[r][q]) : pk[r][q];
                        fv[r][q] = started[r] ? fadd2_ftz(fv[r][q], pv[r][q]) : pv[r][q];
                    }
                    started[r] = true;
                }
            }
        const u64 cc = pack2(a.c, a.c);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int64_t j = j0 + 4 * ty + r;
            if (j >= T)
                continue;
            const int64_t off = ((kt.b * a.T + j) * a.Hkv + kt.g) * HD + 4 * tx;
            u64 k4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                k4[q] = fadd2_ftz(fmul2_rn(fk[r][q], cc), z);   // dK = F_K (x) c, flushed
            *reinterpret_cast<ulonglong2*>(a.dk + off) = make_ulonglong2(k4[0], k4[1]);
            *reinterpret_cast<ulonglong2*>(a.dk + off + HD / 2) = make_ulonglong2(k4[2], k4[3]);
            *reinterpret_cast<ulonglong2*>(a.dv + off) = make_ulonglong2(fv[r][0], fv[r][1]);
            *reinterpret_cast<ulonglong2*>(a.dv + off + HD / 2) = make_ulonglong2(fv[r][2], fv[r][3]);
        }
    }
    if (lt == 0)
        while (used < issued && mbar_wait(&full[used & 1], (used >> 1) & 1))
            ++used;
    if (fail)
        atomicExch(a.err, 1);
}

// the backward's workspace: Dr_i and the recomputing route's dQ accumulator,
// then (with the cache) the a / dS tiles, the images and the work counters
struct BwdWs {
    unsigned long long* acc;
    float* drow;
    float* at;
    float* st;
    float* vimg;
    float* krow;
    float* qrow;
    float* grow;
    unsigned long long* counters;
    size_t bytes;
};

static BwdWs bwd_ws_layout(void* ws, int64_t B, int64_t T, int64_t Hq, int64_t W)
{
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const uintptr_t base = reinterpret_cast<uintptr_t>(ws);   // 0: sizes only
    const int64_t rows = B * T * Hq, nqt = (T + AT - 1) / AT;
    BwdWs L = {};
    size_t off = 0;
    L.acc = reinterpret_cast<unsigned long long*>(base + off);
    off = al(off + (size_t)(rows * HD * 8));
    L.drow = reinterpret_cast<float*>(base + off);
    off += (size_t)(rows * 4);
    if (W < 0) {
        L.bytes = off;
        return L;
    }
    const size_t tiles = (size_t)(B * Hq * tile_prefix(nqt, W)), imgs = (size_t)(B * Hq * nqt);
    auto take = [&](size_t bytes) {
        off = al(off);
        const uintptr_t p = base + off;
        off += bytes;
        return p;
    };
    L.at = reinterpret_cast<float*>(take(tiles * BT_TILE));
    L.st = reinterpret_cast<float*>(take(tiles * BT_TILE));
    L.vimg = reinterpret_cast<float*>(take(imgs * KIMG_TILE));
    L.krow = reinterpret_cast<float*>(take(imgs * ROW_TILE));
    L.qrow = reinterpret_cast<float*>(take(imgs * ROW_TILE));
    L.grow = reinterpret_cast<float*>(take(imgs * ROW_TILE));
    L.counters = reinterpret_cast<unsigned long long*>(take(64));
    L.bytes = off;
    return L;
}

} // namespace

size_t attn_bwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W)
{
    return bwd_ws_layout(nullptr, B, T, Hq, W).bytes;
}

cudaError_t launch_attn_bwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                            const float* o, const float* dout, const float* m, const float* l,
                            float* dq, float* dk, float* dv, int64_t B, int64_t T, int64_t Hq,
                            int64_t Hkv, int64_t W, void* ws, const void* lcache,
                            cudaStream_t st)
{
    const int64_t rows = B * T * Hq;
    const BwdWs L = bwd_ws_layout(ws, B, T, Hq, lcache ? W : -1);
    const float c = 1.0f / sqrtf(128.0f);   // correctly rounded sqrt and division on the host
    int* err = device_error_word();
    if (!err)
        return cudaErrorInvalidValue;
    k_attn_drow<<<(unsigned)((rows + AT - 1) / AT), NT, 0, st>>>(o, dout, L.drow, rows);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    AttnBwdArgs a;
    a.q = q;
    a.k = k;
    a.vq = vq;
    a.s_v = s_v;
    a.dout = dout;
    a.m = m;
    a.l = l;
    a.drow = L.drow;
    a.dq_acc = L.acc;
    a.dk = dk;
    a.dv = dv;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.W = W;
    a.tiles_bh = tile_prefix((T + AT - 1) / AT, W);
    a.c = c;
    if (lcache) {
        const int64_t nqt = (T + AT - 1) / AT, items = B * Hq * nqt;
        const int64_t Wc = W > T ? T : W;   // the same windows and cache layout; W in 32 bits
        const int64_t cap = (int64_t)num_sms() * 8;
        AttnBwdImg im;
        im.k = k;
        im.vq = vq;
        im.s_v = s_v;
        im.q = q;
        im.dout = dout;
        im.vimg = L.vimg;
        im.krow = L.krow;
        im.qrow = L.qrow;
        im.grow = L.grow;
        im.counters = L.counters;
        im.B = B;
        im.T = T;
        im.Hq = Hq;
        im.Hkv = Hkv;
        im.nkt = nqt;
        const int64_t n_max = B * Hq * nqt * (AT * HD / 4);
        k_attn_bimg<<<dim3((unsigned)std::min<int64_t>((n_max + 255) / 256, cap), 4), 256, 0, st>>>(im);
        count_launches(1);
        // dA, a and dS per query tile (the cache is only read in this mode)
        AttnLogitArgs la;
        la.q = dout;
        la.kimg = L.vimg;
        la.cache = const_cast<float*>(static_cast<const float*>(lcache));
        la.m = nullptr;
        la.counter = L.counters;
        la.T = T;
        la.Hq = Hq;
        la.Hkv = Hkv;
        la.W = Wc;
        la.tiles_bh = a.tiles_bh;
        la.nqt = nqt;
        la.nkt = nqt;
        la.items = items;
        la.c = c;
        la.err = err;
        la.l = l;
        la.drow = L.drow;
        la.at = L.at;
        la.st = L.st;
        e = cudaFuncSetAttribute(k_attn_rows<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LG_SMEM);
        if (e != cudaSuccess)
            return e;
        k_attn_rows<true><<<(unsigned)std::min<int64_t>(num_sms(), (items + 1) / 2), LG_NT, LG_SMEM, st>>>(la);
        count_launches(1);
        // dQ per query tile
        AttnDqArgs qa;
        qa.st = L.st;
        qa.krow = L.krow;
        qa.dq = dq;
        qa.counter = L.counters + 1;
        qa.T = T;
        qa.Hq = Hq;
        qa.Hkv = Hkv;
        qa.W = Wc;
        qa.tiles_bh = a.tiles_bh;
        qa.nqt = nqt;
        qa.nkt = nqt;
        qa.items = items;
        qa.c = c;
        qa.err = err;
        e = cudaFuncSetAttribute(k_attn_bdq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DQ_SMEM);
        if (e != cudaSuccess)
            return e;
        k_attn_bdq<<<(unsigned)std::min<int64_t>(2 * (int64_t)num_sms(), items), NT, DQ_SMEM, st>>>(qa);
        count_launches(1);
        // dK and dV per key tile
        AttnDkvArgs ka;
        ka.at = L.at;
        ka.st = L.st;
        ka.qrow = L.qrow;
        ka.grow = L.grow;
        ka.dk = dk;
        ka.dv = dv;
        ka.counter = L.counters + 2;
        ka.B = B;
        ka.T = T;
        ka.Hq = Hq;
        ka.Hkv = Hkv;
        ka.W = Wc;
        ka.tiles_bh = a.tiles_bh;
        ka.nqt = nqt;
        ka.items = B * Hkv * nqt;
        ka.c = c;
        ka.err = err;
        e = cudaFuncSetAttribute(k_attn_bdkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)KV_SMEM);
        if (e != cudaSuccess)
            return e;
        k_attn_bdkv<<<(unsigned)std::min<int64_t>(num_sms(), ka.items), NT, KV_SMEM, st>>>(ka);
        count_launches(1);
        return cudaGetLastError();
    }
    e = cudaMemsetAsync(L.acc, 0, (size_t)(rows * HD * 8), st);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(k_attn_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BWD_SMEM);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((T + AT - 1) / AT), (unsigned)Hkv, (unsigned)B);
    k_attn_bwd<<<grid, NT, BWD_SMEM, st>>>(a);
    const int64_t n = rows * HD;
    int nb = num_sms() * 8;
    k_attn_dq_final<<<nb, NT, 0, st>>>(L.acc, dq, n, c);
    count_launches(2);
    return cudaGetLastError();
}

// the logit cache, then the V^T and K^T images of the tensor-core route
// (sized for Hkv = Hq, its upper bound) and the logits kernel's work counter
static size_t attn_cache_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W)
{
    const int64_t nqt = (T + AT - 1) / AT;
    return (size_t)(B * Hq * tile_prefix(nqt, W) * (AT * AT) * 4);
}

size_t attn_fwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W)
{
    const int64_t nqt = (T + AT - 1) / AT;
    return attn_cache_bytes(B, T, Hq, W) + (size_t)(B * Hq * nqt) * (VIMG_TILE + KIMG_TILE) + 16;
}

cudaError_t launch_attn_fwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                            float* o, float* m, float* l, int64_t B, int64_t T, int64_t Hq,
                            int64_t Hkv, int64_t W, void* cache, bool tc, cudaStream_t st)
{
    AttnFwdArgs a;
    a.q = q;
    a.k = k;
    a.vq = vq;
    a.s_v = s_v;
    a.o = o;
    a.m = m;
    a.l = l;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.W = W;
    a.cache = static_cast<float*>(cache);
    a.tiles_bh = tile_prefix((T + AT - 1) / AT, W);
    a.c = 1.0f / sqrtf(128.0f);   // correctly rounded sqrt and division on the host
    a.err = device_error_word();
    if (!a.err)
        return cudaErrorInvalidValue;
    if (tc && cache) {
        // the K^T and V^T images after the cache, then the two passes
        const int64_t nqt = (T + AT - 1) / AT;
        uint8_t* vimg = static_cast<uint8_t*>(cache) + attn_cache_bytes(B, T, Hq, W);
        float* kimg = reinterpret_cast<float*>(vimg + (size_t)(B * Hq * nqt) * VIMG_TILE);
        auto* counter = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(kimg) +
                                                              (size_t)(B * Hq * nqt) * KIMG_TILE);
        a.m = m;
        if (a.W > T)
            a.W = T;   // the same windows and cache layout; keeps W in 32 bits
        const int64_t vchunks = B * Hkv * nqt * 1024, kn = B * Hkv * nqt * (AT * HD / 4);
        const int64_t cap = (int64_t)num_sms() * 8;
        k_attn_vimg<<<(int)std::min<int64_t>((vchunks + 255) / 256, cap), 256, 0, st>>>(vq, vimg, T, Hkv,
                                                                                      nqt, vchunks);
        k_attn_kimg<<<(int)std::min<int64_t>((kn + 255) / 256, cap), 256, 0, st>>>(k, kimg, T, Hkv, nqt,
                                                                                  kn, counter);
        count_launches(2);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        AttnLogitArgs la;
        la.q = q;
        la.kimg = kimg;
        la.cache = a.cache;
        la.m = m;
        la.counter = counter;
        la.T = T;
        la.Hq = Hq;
        la.Hkv = Hkv;
        la.W = a.W;
        la.tiles_bh = a.tiles_bh;
        la.nqt = nqt;
        la.nkt = nqt;
        la.items = B * Hq * nqt;
        la.c = a.c;
        la.err = a.err;
        e = cudaFuncSetAttribute(k_attn_rows<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LG_SMEM);
        if (e != cudaSuccess)
            return e;
        const unsigned lgrid = (unsigned)std::min<int64_t>(num_sms(), (la.items + 1) / 2);
        k_attn_rows<false><<<lgrid, LG_NT, LG_SMEM, st>>>(la);
        count_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        AttnPVArgs pa;
        pa.f = a;
        pa.vimg = vimg;
        pa.nkt = nqt;
        e = cudaFuncSetAttribute(k_attn_pv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PV_SMEM);
        if (e != cudaSuccess)
            return e;
        k_attn_pv<<<dim3((unsigned)nqt, (unsigned)Hq, (unsigned)B), PV_NTH, PV_SMEM, st>>>(pa);
        count_launches(1);
        return cudaGetLastError();
    }
    auto kern = k_attn_fwd;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)FWD_SMEM);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((T + AT - 1) / AT), (unsigned)Hq, (unsigned)B);
    kern<<<grid, NT, FWD_SMEM, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
