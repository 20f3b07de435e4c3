// k_attn.cuh -- attention with int8 P.V: inside flash attention the P.V
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
//     passed (the default): k_attn_rows<false> (pass 1, below) and k_attn_pv
//     (pass 2, P.V on the tensor cores, k_attn_fwd.cu);
//   * otherwise k_attn_fwd (k_attn_fwd.cu): one CTA per (64-row query tile, query head,
//     sequence) runs both passes; pass 2 reads the cached logits or recomputes
//     them, and P.V runs on dp4a (exact int32).  Logits: 256 threads own 4 x 4
//     outputs each, packed f32x2 products over d with the chunk-of-64 order.
//
// This header holds what both passes share: the tile constants, e^x, the
// cache layout, and the banded-product kernel k_attn_rows (the forward's logits,
// the backward's dA / a / dS).  The forward lives in k_attn_fwd.cu, the
// backward in k_attn_bwd.cu.
#pragma once

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

// ---------------------------------------------------------------------------
// Default forward route (logit cache and tensor-core P.V), two kernels.
//
// k_attn_rows<false>: pass 1 -- every logit of the window written to the cache and
// the exact row maxima written to m -- as a banded product in the canonical
// order over d.  (k_attn_rows<true> is the backward's dA / a / dS pass: the
// same product of dO and V^, described with the backward in k_attn_bwd.cu.)
// A CTA holds two groups of 128 threads; each group takes its
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

// RN(p / l) for a packed pair of quotients, from nl = -l and y = RN(1 / l).
// q = p (x) y is within two units in the last place; one correction
// (r = p - l q, then q + r y, each with a single rounding) leaves it within
// 1/2 unit plus 2^-46 relative, so it is faithful; a second correction then
// returns the correctly rounded quotient by Markstein's theorem (P. Markstein,
// IBM J. Res. Dev. 34(1), 1990; Muller et al., Handbook of Floating-Point
// Arithmetic, chapter 5, division with a fused multiply-add), and the
// remainder it uses is exact.  Both need every intermediate normal: the
// caller takes this only for l in [2^-30, 2^30) and p = +0 or p in
// [2^-90, 2^90), where q stays in (2^-120, 2^120) and every remainder is zero
// or above 2^-114, and divides otherwise.
__device__ __forceinline__ u64 div2_rn(u64 p, u64 nl, u64 y)
{
    u64 q = fmul2_rn(p, y);
    q = ffma2_rn(ffma2_rn(nl, q, p), y, q);
    return ffma2_rn(ffma2_rn(nl, q, p), y, q);
}

constexpr uint32_t DIV_L_LO = 0x30800000u;   // 2^-30: bits of the smallest l taken
constexpr uint32_t DIV_L_SPAN = 0x1E000000u; // up to 2^30 (excluded)
constexpr uint32_t DIV_P_LO = 0x12800000u;   // 2^-90: the smallest nonzero p taken
constexpr uint32_t DIV_P_HI = 0x6C800000u;   // 2^90 (excluded)

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
        // backward: -l and RN(1 / l) of the thread's row pairs, and whether
        // all eight l admit the quotient by correction (div2_rn)
        u64 nl2[4], y2[4];
        bool l_ok = true;
        if constexpr (BWD) {
#pragma unroll
            for (int ip = 0; ip < 4; ++ip) {
                const float l0 = lrw[8 * ty + 2 * ip], l1 = lrw[8 * ty + 2 * ip + 1];
                nl2[ip] = pack2(-l0, -l1);
                y2[ip] = pack2(__frcp_rn(l0), __frcp_rn(l1));
                l_ok = l_ok && __float_as_uint(l0) - DIV_L_LO < DIV_L_SPAN &&
                       __float_as_uint(l1) - DIV_L_LO < DIV_L_SPAN;
            }
        }
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
            const int j0 = t * AT;
            // every (query, key) pair of the tile valid: no per-pair test
            const bool inner = qt.i0 + AT - 1 < T && j0 + AT - 1 <= qt.i0 && (W == 0 || j0 >= qt.i0 + AT - W);
            // A mask-edge tile may leave a warp (rows r0w .. r0w + 15) with
            // valid keys in at most 8 of its 16 four-key column blocks
            // [ca, cb]: then each such block's two 64-term chunks are summed by
            // two threads of its half-warp -- d 0..63 by the block's thread,
            // d 64..127 by one whose own block has no valid key -- and the
            // second sum is handed over; with no valid key at all the warp
            // skips the tile.  Each logit is still (chunk 0 (+) chunk 1) (x) c
            u64 t0[16], t1[16];
            bool need = true;   // this thread's own block is formed and used
            int ca = 0, cb = AT / 4 - 1;
            bool pair = false, skip = false;
            if (!inner) {
                const int r0w = qt.i0 + 16 * (lt >> 5), r1w = min(r0w + 15, T - 1);
                const int ka = max((W > 0 ? max(0, r0w - W + 1) : 0) - j0, 0);
                const int kb = min(r1w - j0, AT - 1);
                skip = r0w >= T || kb < ka;
                if (!skip) {
                    ca = ka >> 2;
                    cb = kb >> 2;
                    pair = cb - ca + 1 <= 8;
                }
            }
            if (skip) {
                need = false;
            } else if (pair) {
                const int n = cb - ca + 1;
                const bool prim = tx >= ca && tx <= cb;
                const int k = tx < ca ? tx : tx - n;       // rank among the blocks outside [ca, cb]
                const bool help = !prim && k < n;
                const int own = help ? ca + k : tx;        // the block this thread's chunk belongs to
                const int dofs = help ? 64 : 0;
                logit_chunk84(t0, Qt + dofs * PT + 8 * ty, Kc + dofs * AT + 4 * own);
                // a valid block's helper: the column outside [ca, cb] of the same rank
                const int kp = tx - ca;
                const int src = (lane & 16) | (prim ? (kp < ca ? kp : kp + n) : tx);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    t1[e] = __shfl_sync(0xffffffffu, t0[e], src);
                need = prim;
            } else {
                logit_chunk84(t0, Qt + 8 * ty, Kc + 4 * tx);
                logit_chunk84(t1, Qt + 64 * PT + 8 * ty, Kc + 64 * AT + 4 * tx);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[gp][s]);
            ++used;
            if (!need) {
                // nothing of this thread's block is valid: no logits, maxima
                // or (backward) a and dS to form
            } else if constexpr (!BWD) {
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
                // a = p (/) l_i, flushed, for the thread's 16 pairs: by
                // correction when every p and l admits it, else divided
                u64 a2[16];
                {
                    uint32_t lo = 0xffffffffu, hi = 0u;   // min of bits - 1 (+0 wraps), max of bits
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t b0 = (uint32_t)pv[e], b1 = (uint32_t)(pv[e] >> 32);
                        lo = min(lo, min(b0 - 1u, b1 - 1u));
                        hi = max(hi, max(b0, b1));
                    }
                    if (l_ok && lo >= DIV_P_LO - 1u && hi < DIV_P_HI) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            a2[e] = fadd2_ftz(div2_rn(pv[e], nl2[e >> 2], y2[e >> 2]), z);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int r0 = 8 * ty + 2 * (e >> 2);
                            float p0, p1;
                            unpack2(pv[e], p0, p1);
                            a2[e] = pack2(flush(__fdiv_rn(p0, lrw[r0])), flush(__fdiv_rn(p1, lrw[r0 + 1])));
                        }
                    }
                }
                float av[8][4], dv[8][4];   // rows 8ty + rr, keys 4tx + j
#pragma unroll
                for (int ip = 0; ip < 4; ++ip)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int e = ip * 4 + j, r0 = 8 * ty + 2 * ip;
                        float aa[2];
                        unpack2(a2[e], aa[0], aa[1]);
                        float d[2];
                        unpack2(fadd2_ftz(fmul2_rn(a2[e],
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

} // namespace
} // namespace repro
