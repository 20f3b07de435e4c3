// k_bwd.cu -- fp32 backward of the int8 QAT linear in canonical order.
//
//   W^[n,k] = float(Wq[n,k]) (x) s_w        X^[m,k] = float(Xq[m,k]) (x) s_x
//   dX[m,k] = canon_n( dY[m,n] (x) W^[n,k] )
//   dW[n,k] = canon_m( dY[m,n] (x) X^[m,k] )
// Fixed reduction order and explicit unfused multiply then add (Open-1B
// review, onedev.kr/papers/92, section "How it works").  canon = chunks of 64
// terms summed left to right from the first term, then the stride-doubling
// pairwise tree over chunk partials.
//
// Both products are one kernel shape: C[i,j] = canon_r( A[r,i] (x) B[r,j] )
// with A taken from dY (dX: A[r,i] = dY[i,r]; dW: A[r,i] = dY[r,i]) and B the
// dequantised int8 operand with j = k (B[r,j] = q[r,j] (x) s).
//
// Parallel over outputs only; each output's sequence of roundings is fixed:
//   * a CTA owns a 64 x 64 output tile; 256 threads own 4 x 4 outputs each;
//   * the reduction advances one 64-term chunk at a time: the chunk's A and B
//     slices are staged in shared memory (dY flushed, int8 dequantised and
//     flushed on the way in), then every thread runs the 64 steps of the chunk
//     for its 16 outputs: first product, then 63 rounded multiply + add pairs;
//   * chunk partials enter the pairwise tree through a binary-counter stack
//     kept in registers: after chunk c (counted from the segment start) it is
//     merged with the stack levels given by the trailing one bits of c, left
//     operand first, and the last chunk folds every remaining level in, lowest
//     first.  This evaluates exactly the stride-doubling tree;
//   * a segment is an aligned block of 2^k chunks (k <= 8, 256 by default, so
//     reductions up to 16384 terms need one segment).  The tree over aligned
//     power-of-two blocks is a subtree of the canonical tree, so longer
//     reductions (or a smaller k set through the launch-configuration hook)
//     write one partial per segment to the workspace and finish with pairwise
//     passes over segments -- the same bits for every k.
// No atomics: each output is written by exactly one thread.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

constexpr int BT = 64;       // output tile edge
constexpr int CH = 64;       // chunk length of the canonical order
constexpr int MAXLVL = 8;    // stack levels: up to 256 chunks per segment

struct BwdArgs {
    const float* dy;
    const int8_t* q;
    const float* scale;
    float* out;
    float* ws;
    int64_t I, J, R;   // output rows, output columns, reduction length
    int64_t ldy;       // row stride of dY (= N)
    int seg_log2;
    int nseg;
    int accumulate;
};

// A[r][i] for the chunk starting at reduction index r0 (valid rows < valid)
template <bool DW>
__device__ __forceinline__ void load_a(float (&As)[CH][BT], const BwdArgs& a, int64_t i0,
                                       int64_t r0, int valid, int tid)
{
    if (DW) {
        // A[r][i] = dY[r0 + r][i0 + i]: rows of dY, contiguous along i
        const bool vec = (a.ldy & 3) == 0;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = tid + it * 256;
            const int r = e >> 4, f = e & 15;
            const int64_t i = i0 + 4 * f;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < valid) {
                const float* src = a.dy + (r0 + r) * a.ldy + i;
                if (vec && i + 4 <= a.I) {
                    v = flush4(__ldg(reinterpret_cast<const float4*>(src)));
                } else {
                    v.x = (i + 0 < a.I) ? flush(src[0]) : 0.f;
                    v.y = (i + 1 < a.I) ? flush(src[1]) : 0.f;
                    v.z = (i + 2 < a.I) ? flush(src[2]) : 0.f;
                    v.w = (i + 3 < a.I) ? flush(src[3]) : 0.f;
                }
            }
            *reinterpret_cast<float4*>(&As[r][4 * f]) = v;
        }
    } else {
        // A[r][i] = dY[i0 + i][r0 + r]: lane <-> row i, so the transposed
        // shared-memory stores hit 32 distinct banks
        const int i = tid & 63;
        const bool row_ok = i0 + i < a.I;
        const float* src = a.dy + (i0 + i) * a.ldy + r0;
        const bool vec = (a.ldy & 3) == 0;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int f = (tid >> 6) + 4 * it;   // float4 group along r
            const int r = 4 * f;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row_ok) {
                if (vec && r + 4 <= valid) {
                    v = flush4(__ldg(reinterpret_cast<const float4*>(src + r)));
                } else {
                    v.x = (r + 0 < valid) ? flush(src[r + 0]) : 0.f;
                    v.y = (r + 1 < valid) ? flush(src[r + 1]) : 0.f;
                    v.z = (r + 2 < valid) ? flush(src[r + 2]) : 0.f;
                    v.w = (r + 3 < valid) ? flush(src[r + 3]) : 0.f;
                }
            }
            As[r + 0][i] = v.x;
            As[r + 1][i] = v.y;
            As[r + 2][i] = v.z;
            As[r + 3][i] = v.w;
        }
    }
}

// B[r][j] = float(q[r0 + r][j0 + j]) (x) s, flushed
__device__ __forceinline__ void load_b(float (&Bs)[CH][BT], const BwdArgs& a, int64_t j0,
                                       int64_t r0, int valid, float s, int tid)
{
    const int r = tid >> 2, part = tid & 3;
    const int64_t j = j0 + 16 * part;
    float v[16];
    if (r < valid) {
        const int8_t* src = a.q + (r0 + r) * a.J + j;
        if ((a.J & 15) == 0 && j + 16 <= a.J) {
            const int4 w = __ldg(reinterpret_cast<const int4*>(src));
            const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    v[4 * u + b] = dequant((int)(int8_t)(words[u] >> (8 * b)), s);
        } else {
#pragma unroll
            for (int u = 0; u < 16; ++u)
                v[u] = (j + u < a.J) ? dequant((int)src[u], s) : 0.f;
        }
    } else {
#pragma unroll
        for (int u = 0; u < 16; ++u)
            v[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
        *reinterpret_cast<float4*>(&Bs[r][16 * part + 4 * u]) =
            make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
}

template <bool DW>
__global__ void __launch_bounds__(256, 1) k_bwd(const BwdArgs a)
{
    __shared__ __align__(16) float As[CH][BT];
    __shared__ __align__(16) float Bs[CH][BT];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);   // 4 rows: 4ty .. 4ty+3
    const int tx = (warp & 1) * 8 + (lane & 7);     // 4 cols: 4tx .. 4tx+3
    const int64_t i0 = (int64_t)blockIdx.y * BT, j0 = (int64_t)blockIdx.x * BT;
    const float s = flush(*a.scale);

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));

    float S[MAXLVL][16];
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        acc[e] = 0.f;
#pragma unroll
    for (int l = 0; l < MAXLVL; ++l)
#pragma unroll
        for (int e = 0; e < 16; ++e)
            S[l][e] = 0.f;

    for (int64_t c = cbeg; c < cend; ++c) {
        const int64_t r0 = c * CH;
        const int valid = (int)min((int64_t)CH, a.R - r0);
        load_a<DW>(As, a, i0, r0, valid, tid);
        load_b(Bs, a, j0, r0, valid, s, tid);
        __syncthreads();

        {
            const float4 av = *reinterpret_cast<const float4*>(&As[0][4 * ty]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[0][4 * tx]);
            const float ar[4] = {av.x, av.y, av.z, av.w};
            const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[4 * i + j] = fmul_rn(ar[i], br[j]);
        }
        if (valid == CH) {
#pragma unroll 9
            for (int r = 1; r < CH; ++r) {
                const float4 av = *reinterpret_cast<const float4*>(&As[r][4 * ty]);
                const float4 bv = *reinterpret_cast<const float4*>(&Bs[r][4 * tx]);
                const float ar[4] = {av.x, av.y, av.z, av.w};
                const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        acc[4 * i + j] = fadd_ftz(acc[4 * i + j], fmul_rn(ar[i], br[j]));
            }
        } else {
            for (int r = 1; r < valid; ++r) {
                const float4 av = *reinterpret_cast<const float4*>(&As[r][4 * ty]);
                const float4 bv = *reinterpret_cast<const float4*>(&Bs[r][4 * tx]);
                const float ar[4] = {av.x, av.y, av.z, av.w};
                const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        acc[4 * i + j] = fadd_ftz(acc[4 * i + j], fmul_rn(ar[i], br[j]));
            }
        }
        __syncthreads();

        const int cs = (int)(c - cbeg);
        if (c + 1 < cend) {
            // push: merge with the levels named by the trailing ones of cs
            const int tz = __ffs(~cs) - 1;
#pragma unroll
            for (int t = 0; t < MAXLVL; ++t) {
                if (tz == t) {
#pragma unroll
                    for (int l = 0; l < t; ++l)
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            acc[e] = fadd_ftz(S[l][e], acc[e]);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        S[t][e] = acc[e];
                }
            }
        } else {
            // last chunk of the segment: fold the occupied levels, lowest first
#pragma unroll
            for (int l = 0; l < MAXLVL; ++l) {
                if ((cs >> l) & 1) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        acc[e] = fadd_ftz(S[l][e], acc[e]);
                }
            }
        }
    }

    // store: the final value is flushed (a one-term sum is a bare product)
    const bool vec = (a.J & 3) == 0;
    if (a.nseg == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = i0 + 4 * ty + i;
            if (row >= a.I)
                continue;
            const int64_t col = j0 + 4 * tx;
            float* dst = a.out + row * a.J + col;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = flush(acc[4 * i + j]);
            if (vec && col + 4 <= a.J) {
                if (a.accumulate) {
                    const float4 o = *reinterpret_cast<const float4*>(dst);
                    v[0] = fadd_ftz(o.x, v[0]);
                    v[1] = fadd_ftz(o.y, v[1]);
                    v[2] = fadd_ftz(o.z, v[2]);
                    v[3] = fadd_ftz(o.w, v[3]);
                }
                *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < a.J)
                        dst[j] = a.accumulate ? fadd_ftz(dst[j], v[j]) : v[j];
            }
        }
    } else {
        float* base = a.ws + (int64_t)blockIdx.z * a.I * a.J;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = i0 + 4 * ty + i;
            if (row >= a.I)
                continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t col = j0 + 4 * tx + j;
                if (col < a.J)
                    base[row * a.J + col] = acc[4 * i + j];
            }
        }
    }
}

// one level of the tree over segment partials: ws[j] <- ws[j] (+) ws[j + s]
// for every j that is a multiple of 2s with j + s < nseg
__global__ void k_seg_level(float* __restrict__ ws, int nseg, int s, int64_t count)
{
    const int npairs = (nseg - s + 2 * s - 1) / (2 * s);
    const int64_t total = (int64_t)npairs * count;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int p = (int)(t / count);
        const int64_t e = t - (int64_t)p * count;
        const int64_t j = (int64_t)p * 2 * s;
        ws[j * count + e] = fadd_ftz(ws[j * count + e], ws[(j + s) * count + e]);
    }
}

__global__ void k_seg_store(const float* __restrict__ ws, float* __restrict__ out, int64_t count,
                            int accumulate)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count;
         e += (int64_t)gridDim.x * blockDim.x) {
        const float v = flush(ws[e]);
        out[e] = accumulate ? fadd_ftz(out[e], v) : v;
    }
}

// empty reduction: the canonical sum of nothing is +0
__global__ void k_zero_sum(float* __restrict__ out, int64_t count, int accumulate)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count;
         e += (int64_t)gridDim.x * blockDim.x)
        out[e] = accumulate ? fadd_ftz(out[e], 0.f) : 0.f;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t nseg_for(int64_t R, int seg_log2)
{
    return cdiv(cdiv(R, CH), (int64_t)1 << seg_log2);
}

template <bool DW>
cudaError_t run(const float* dy, const int8_t* q, const float* scale, float* out, int64_t I,
                int64_t J, int64_t R, int64_t ldy, int seg_log2, bool accumulate, float* ws,
                cudaStream_t st)
{
    if (I == 0 || J == 0)
        return cudaSuccess;
    const int64_t count = I * J;
    const int eb = 4 * num_sms();
    if (R == 0) {
        k_zero_sum<<<eb, 256, 0, st>>>(out, count, accumulate ? 1 : 0);
        count_launches(1);
        return cudaGetLastError();
    }
    BwdArgs a;
    a.dy = dy;
    a.q = q;
    a.scale = scale;
    a.out = out;
    a.ws = ws;
    a.I = I;
    a.J = J;
    a.R = R;
    a.ldy = ldy;
    a.seg_log2 = seg_log2;
    a.nseg = (int)nseg_for(R, seg_log2);
    a.accumulate = accumulate ? 1 : 0;
    dim3 grid((unsigned)cdiv(J, BT), (unsigned)cdiv(I, BT), (unsigned)a.nseg);
    k_bwd<DW><<<grid, 256, 0, st>>>(a);
    count_launches(1);
    if (a.nseg > 1) {
        for (int s = 1; s < a.nseg; s *= 2)
        {
            k_seg_level<<<eb, 256, 0, st>>>(ws, a.nseg, s, count);
            count_launches(1);
        }
        k_seg_store<<<eb, 256, 0, st>>>(ws, out, count, a.accumulate);
        count_launches(1);
    }
    return cudaGetLastError();
}

} // namespace

size_t bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int seg_log2)
{
    const int64_t sx = nseg_for(N, seg_log2), sw = nseg_for(M, seg_log2);
    const int64_t bx = sx > 1 ? sx * M * K : 0;
    const int64_t bw = sw > 1 ? sw * N * K : 0;
    return (size_t)((bx > bw ? bx : bw) * (int64_t)sizeof(float));
}

cudaError_t launch_bwd_dx(const float* dy, const int8_t* wq, const float* s_w, float* dx,
                          int64_t M, int64_t N, int64_t K, int seg_log2, float* ws,
                          cudaStream_t st)
{
    return run<false>(dy, wq, s_w, dx, M, K, N, N, seg_log2, false, ws, st);
}

cudaError_t launch_bwd_dw(const float* dy, const int8_t* xq, const float* s_x, float* dw,
                          int64_t M, int64_t N, int64_t K, int seg_log2, bool accumulate,
                          float* ws, cudaStream_t st)
{
    return run<true>(dy, xq, s_x, dw, N, K, M, N, seg_log2, accumulate, ws, st);
}

} // namespace repro
