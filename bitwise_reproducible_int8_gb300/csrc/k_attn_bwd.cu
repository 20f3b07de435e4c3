// k_attn_bwd.cu -- the attention backward (the method, its order and the
// routes are stated in k_attn.cuh): Dr, the cached route's images and its
// dQ and dK/dV kernels, the single-kernel backward of the other route, and the
// launcher.
#include "k_attn.cuh"

namespace repro {
namespace {

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
                                // the first term is flushed as -0 (+) t, the same as t (+) -0
                                pp[r][q] = fadd2_ftz(j == jb[r] ? z : pp[r][q], pr);
                            }
                        }
                    }
                };
                if (mid_lo <= mid_hi) {
                    edge(lo_all, mid_lo - 1);
                    load(mid_lo);
#pragma unroll 4
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
#pragma unroll 7
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
                                    // the first term is flushed as -0 (+) t, the same as t (+) -0
                                    pk[r][q] = fadd2_ftz(i == ib[r] ? z : pk[r][q], xk);
                                    pv[r][q] = fadd2_ftz(i == ib[r] ? z : pv[r][q], xv);
                                }
                            }
                        }
                    };
                    if (mid_lo <= mid_hi) {
                        edge(lo_all, mid_lo - 1);
                        load(mid_lo);
#pragma unroll 4
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
                // fold the group partials, left to right over the groups; once
                // every key of the warp has started and has queries here, plain adds
                bool plain = true;
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    plain = plain && started[r] && ib[r] <= ie[r];
                if (__all_sync(0xffffffffu, plain)) {
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            fk[r][q] = fadd2_ftz(fk[r][q], pk[r][q]);
                            fv[r][q] = fadd2_ftz(fv[r][q], pv[r][q]);
                        }
                } else {
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
} // namespace repro
