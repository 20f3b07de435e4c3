// k_attn_fwd.cu -- the attention forward (the method, its order and the
// routes are stated in k_attn.cuh): the images of K and V, the P.V pass of
// the default route, the single-kernel forward of the other route, and the
// launcher.
#include "k_attn.cuh"

namespace repro {
namespace {

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

constexpr size_t FWD_SMEM = (size_t)(2 * HD * PT + AT * PS) * 4 + (size_t)(AT * PP) * 4 +
                            (size_t)(AT / 4 * HD) * 4 + (size_t)(AT * (MAXL + 1)) * 4 +
                            (size_t)(3 * AT) * 4;

// pass 1's second key tile lives in pass 2's scratch (Ps .. stk)
static_assert(HD * PT <= AT * PS + AT * PP + AT / 4 * HD + AT * (MAXL + 1),
              "second key tile does not fit in the pass-2 scratch");

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
// k_attn_pv: pass 2 of the default route -- p, the int8 codes, the row sums and P.V -- one CTA of
// 256 threads per query tile, two CTAs per SM.  The P and V^T tiles and the p
// tile are double-buffered, so tile t + 1 is written while the MMA of tile t
// runs and the row sums of tile t are read; V^T comes from the image of the V
// codes (k_attn_vimg) by one bulk copy per tile.
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

} // namespace

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
