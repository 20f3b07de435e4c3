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
// k_attn_fwd: one CTA per (64-row query tile, query head, sequence).  The row
// maximum must be exact before any p is quantised, so the key tiles of the
// window are visited twice: pass 1 computes the logits and the row maxima,
// pass 2 recomputes the same logits, forms p and the int8 codes, streams the
// row sums through the canonical-order chunk/tree stack (one thread per row)
// and accumulates P.V with dp4a (exact int32).  Logits: 256 threads own 4 x 4
// outputs each, packed f32x2 products over d with the chunk-of-64 order.
#include "common.cuh"
#include "internal.h"

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
    int64_t T, Hq, Hkv, W;
    float c;
};

constexpr size_t FWD_SMEM = (size_t)(2 * HD * PT + AT * PS) * 4 + (size_t)(AT * PP) * 4 +
                            (size_t)(AT / 4 * HD) * 4 + (size_t)(AT * (MAXL + 1)) * 4 +
                            (size_t)(3 * AT) * 4;

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

__device__ __forceinline__ int quant_p(float p)
{
    float r = rintf(fmul_flush(p, 127.0f));
    r = fminf(fmaxf(r, 0.0f), 127.0f);
    return (int)r;
}

// tile of 64 rows x 128 floats of a [.., H, 128] tensor, flushed and
// transposed into t[d][r] (pitch PT); rows outside [0, T) read as 0.
// Warp lanes cover 8 rows x 4 float4 columns per step.
__device__ __forceinline__ void load_tile_t(float* __restrict__ t, const float* __restrict__ src,
                                            int64_t row0, int64_t T, int64_t row_stride, int tid)
{
#pragma unroll
    for (int it = 0; it < (AT * HD / 4) / NT; ++it) {
        const int e = tid + it * NT;            // 2048 float4 pieces
        const int lane = e & 31, w = e >> 5;    // w: 64 groups of 8 rows x 4 columns
        const int r = (w & 7) * 8 + (lane & 7);
        const int c4 = (w >> 3) * 4 + (lane >> 3);
        const int64_t row = row0 + r;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row >= 0 && row < T)
            v = flush4(*reinterpret_cast<const float4*>(src + row * row_stride + 4 * c4));
        t[(4 * c4 + 0) * PT + r] = v.x;
        t[(4 * c4 + 1) * PT + r] = v.y;
        t[(4 * c4 + 2) * PT + r] = v.z;
        t[(4 * c4 + 3) * PT + r] = v.w;
    }
}

// the thread's 4 x 4 logits: rows 4ty..4ty+3 (as 2 packed pairs), columns
// 4tx..4tx+3; canonical order over d: two chunks of 64, then one pairwise add
__device__ __forceinline__ void logits4x4(u64 (&s)[8], const float* __restrict__ Qt,
                                          const float* __restrict__ Kt, int ty, int tx, float c)
{
    u64 t0[8];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        u64 acc[8];
#pragma unroll 4
        for (int dd = 0; dd < 64; ++dd) {
            const int d = half * 64 + dd;
            const ulonglong2 qa = *reinterpret_cast<const ulonglong2*>(Qt + d * PT + 4 * ty);
            const float4 kb = *reinterpret_cast<const float4*>(Kt + d * PT + 4 * tx);
            const u64 P[2] = {qa.x, qa.y};
            const u64 D[4] = {pack2(kb.x, kb.x), pack2(kb.y, kb.y), pack2(kb.z, kb.z),
                              pack2(kb.w, kb.w)};
#pragma unroll
            for (int ip = 0; ip < 2; ++ip)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const u64 p = fmul2_rn(P[ip], D[j]);
                    acc[ip * 4 + j] = dd == 0 ? p : fadd2_ftz(acc[ip * 4 + j], p);
                }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (half == 0)
                t0[e] = acc[e];
            else
                s[e] = fadd2_ftz(t0[e], acc[e]);
        }
    }
    const u64 cc = pack2(c, c);
#pragma unroll
    for (int e = 0; e < 8; ++e)
        s[e] = fadd2_ftz(fmul2_rn(s[e], cc), pack2(-0.0f, -0.0f));   // (x) c, flushed
}

// logit (row 4ty + 2ip + h, column 4tx + j) is lane h of s[ip*4 + j]
__device__ __forceinline__ float lane_of(const u64 (&s)[8], int ip, int j, int h)
{
    float lo, hi;
    unpack2(s[ip * 4 + j], lo, hi);
    return h ? hi : lo;
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

    load_tile_t(Qt, qbase, i0, T, qstride, tid);

    // ---------------------------------------------------------- pass 1: maxima
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for (int64_t t = t_lo; t <= t_hi; ++t) {
        const int64_t j0 = t * AT;
        __syncthreads();   // previous tile's readers are done with Kt
        load_tile_t(Kt, kbase, j0, T, kstride, tid);
        __syncthreads();
        u64 s[8];
        logits4x4(s, Qt, Kt, ty, tx, a.c);
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

    const int ri = tid >> 4, di = tid & 15;   // P.V: rows 4ri..4ri+3, d 8di..8di+7
    int acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int u = 0; u < 8; ++u)
            acc[r][u] = 0;

    for (int64_t t = t_lo; t <= t_hi; ++t) {
        const int64_t j0 = t * AT;
        __syncthreads();   // Kt, Ps, Pp, Vp free
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
            logits4x4(s, Qt, Kt, ty, tx, a.c);
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
                        word |= (uint32_t)quant_p(p) << (8 * j);
                    }
                    Pp[r * PP + tx] = (int)word;
                }
        }
        __syncthreads();
        // row sums: the valid p of this tile, left to right, through the
        // chunk-of-64 / pairwise-tree stack
        if (tid < AT && my_i < T) {
            const int64_t cb = max(my_lo, j0), ce = min(my_i, j0 + AT - 1);
            for (int64_t jj = cb; jj <= ce; ++jj) {
                const float p = Ps[tid * PS + (int)(jj - j0)];
                cs = (pos & 63) == 0 ? p : fadd_ftz(cs, p);
                ++pos;
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

} // namespace

cudaError_t launch_attn_fwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                            float* o, float* m, float* l, int64_t B, int64_t T, int64_t Hq,
                            int64_t Hkv, int64_t W, cudaStream_t st)
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
    a.c = 1.0f / sqrtf(128.0f);   // correctly rounded sqrt and division on the host
    cudaError_t e = cudaFuncSetAttribute(k_attn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)FWD_SMEM);
    if (e != cudaSuccess)
        return e;
    dim3 grid((unsigned)((T + AT - 1) / AT), (unsigned)Hq, (unsigned)B);
    k_attn_fwd<<<grid, NT, FWD_SMEM, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
