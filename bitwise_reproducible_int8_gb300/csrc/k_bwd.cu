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
//   * a CTA owns an output tile and each thread a block of it; the two
//     kernels (k_bwd_tma.cu, the default, for 16-byte-aligned rows, and
//     k_bwd_prefetch.cu for any rows) differ only in how operands reach the
//     products;
//   * the reduction advances one 64-term chunk at a time: the chunk's A and B
//     slices sit in shared memory (dY flushed, the int8 operand dequantised
//     and flushed), then every thread runs the 64 steps of the chunk for each
//     of its outputs: first product, then 63 rounded multiply + add pairs;
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
#include "bwd_common.cuh"
#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

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

int64_t nseg_for(int64_t R, int seg_log2)
{
    return cdiv(cdiv(R, CH), (int64_t)1 << seg_log2);
}

// kernel launched for a shape: the tensor-copy-fed kernel (8) needs
// 16-byte-aligned rows of dY (N % 4 == 0) and of the int8 operand
// (J % 16 == 0); other shapes, or the launch-configuration hook's 1, take the
// register-prefetch kernel (1)
constexpr int KERNEL_TMA = 8, KERNEL_PREFETCH = 1;

int kernel_for(int64_t ldy, int64_t J)
{
    const bool aligned = (ldy % 4) == 0 && (J % 16) == 0;
    return (aligned && launch_cfg().bwd_kernel == KERNEL_TMA) ? KERNEL_TMA : KERNEL_PREFETCH;
}

int tile_rows(int kernel) { return kernel == KERNEL_TMA ? BWD_TMA_ROWS : BT; }

// Segment size when the launch configuration leaves it open.  One CTA runs
// per SM, so a grid of tiles that is not close to a whole number of waves
// wastes SMs in its last wave; splitting the reduction into aligned segments
// multiplies the CTA count (the segment partials are then folded by the
// pairwise passes, same bits).  Picks the fewest segments (at most 8) that
// reach 95 % wave efficiency, else the most efficient split.
int auto_seg_log2(int64_t I, int64_t J, int64_t R, int kernel)
{
    const int64_t C = cdiv(R, CH);
    int kmax = 0;
    while (((int64_t)1 << kmax) < C)
        ++kmax;
    if (kmax > MAXLVL)
        kmax = MAXLVL;
    const int64_t tiles = cdiv(J, BT) * cdiv(I, tile_rows(kernel));
    const int64_t sms = num_sms();
    int best = kmax;
    double best_eff = -1.0;
    for (int k = kmax; k >= 0 && k >= kmax - 3; --k) {
        const int64_t ctas = tiles * nseg_for(R, k);
        const double eff = (double)ctas / (double)(cdiv(ctas, sms) * sms);
        if (eff >= 0.95)
            return k;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = k;
        }
    }
    return best;
}

int resolve_seg(int seg_log2, int64_t I, int64_t J, int64_t R, int64_t ldy)
{
    if (seg_log2 >= 0)
        return seg_log2;
    return auto_seg_log2(I, J, R, kernel_for(ldy, J));
}

template <bool DW>
cudaError_t run(const float* dy, const int8_t* q, const float* scale, float* out, int64_t I,
                int64_t J, int64_t R, int64_t ldy, int seg_log2, bool accumulate, float* ws,
                float* opnd, cudaStream_t st)
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
    seg_log2 = resolve_seg(seg_log2, I, J, R, ldy);
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
    a.err = device_error_word();
    cudaError_t e;
    if (kernel_for(ldy, J) == KERNEL_TMA) {
        if (!a.err || !opnd)
            return cudaErrorInvalidValue;
        dim3 gt((unsigned)cdiv(J, BT), (unsigned)cdiv(I, BWD_TMA_ROWS), (unsigned)a.nseg);
        e = launch_bwd_tma<DW>(a, q, opnd, gt, st);
    } else {
        e = launch_bwd_prefetch<DW>(a, st);
    }
    if (e != cudaSuccess)
        return e;
    count_launches(1);
    if (a.nseg > 1) {
        for (int s = 1; s < a.nseg; s *= 2) {
            k_seg_level<<<eb, 256, 0, st>>>(ws, a.nseg, s, count);
            count_launches(1);
        }
        k_seg_store<<<eb, 256, 0, st>>>(ws, out, count, a.accumulate);
        count_launches(1);
    }
    return cudaGetLastError();
}

} // namespace

// workspace: segment partials first, then (tensor-copy kernel only) the
// prepared operands, 256-byte aligned
static int64_t seg_region_bytes(int64_t M, int64_t N, int64_t K, int seg_log2)
{
    // dX: I = M, J = K, R = N, dY rows of N; dW: I = N, J = K, R = M
    const int64_t sx = nseg_for(N, resolve_seg(seg_log2, M, K, N, N));
    const int64_t sw = nseg_for(M, resolve_seg(seg_log2, N, K, M, N));
    const int64_t bx = sx > 1 ? sx * M * K : 0;
    const int64_t bw = sw > 1 ? sw * N * K : 0;
    return (bx > bw ? bx : bw) * (int64_t)sizeof(float);
}

static bool uses_operand_region(int64_t N, int64_t K)
{
    return kernel_for(N, K) == KERNEL_TMA;
}

size_t bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int seg_log2)
{
    const int64_t seg = seg_region_bytes(M, N, K, seg_log2);
    if (!uses_operand_region(N, K))
        return (size_t)seg;
    return (size_t)(((seg + 255) & ~(int64_t)255) + (int64_t)bwd_tma_operand_bytes(M, N, K));
}

static float* operand_region(float* ws, int64_t M, int64_t N, int64_t K, int seg_log2)
{
    if (!ws || !uses_operand_region(N, K))
        return nullptr;
    const int64_t seg = seg_region_bytes(M, N, K, seg_log2);
    return reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + ((seg + 255) & ~(int64_t)255));
}

cudaError_t launch_bwd_dx(const float* dy, const int8_t* wq, const float* s_w, float* dx,
                          int64_t M, int64_t N, int64_t K, int seg_log2, float* ws,
                          cudaStream_t st)
{
    return run<false>(dy, wq, s_w, dx, M, K, N, N, seg_log2, false, ws,
                      operand_region(ws, M, N, K, seg_log2), st);
}

cudaError_t launch_bwd_dw(const float* dy, const int8_t* xq, const float* s_x, float* dw,
                          int64_t M, int64_t N, int64_t K, int seg_log2, bool accumulate,
                          float* ws, cudaStream_t st)
{
    return run<true>(dy, xq, s_x, dw, N, K, M, N, seg_log2, accumulate, ws,
                     operand_region(ws, M, N, K, seg_log2), st);
}

} // namespace repro
