// k_fwd.cu -- exact int8 forward on CUDA cores (general shapes).
//
// acc[m,n] = sum_k Xq[m,k] * Wq[n,k] is an exact integer (|acc| <= 127^2 K
// fits int32 for K <= 133144), so the order of the dp4a accumulation cannot
// change it; Y = (float(acc) (x) s_x) (x) s_w with two unfused, flushed
// multiplies (int8 QAT linears: Open-1B review, onedev.kr/papers/92, section
// "How to use").  This path serves every shape; the tensor-core path takes the
// aligned shapes.
#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

constexpr int FT = 64;          // output tile edge
constexpr int KW = 16;          // 32-bit words (4 int8) per K slab -> 64 int8

__device__ __forceinline__ int load_word(const int8_t* __restrict__ p, int64_t row, int64_t rows,
                                         int64_t K, int64_t k, bool k4)
{
    if (row >= rows)
        return 0;
    const int8_t* r = p + row * K;
    if (k4) {
        if (k + 4 <= K)
            return __ldg(reinterpret_cast<const int*>(r + k));
        return 0;
    }
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (k + i < K)
            w |= (uint32_t)(uint8_t)r[k + i] << (8 * i);
    return (int)w;
}

__global__ void __launch_bounds__(256)
k_fwd_dp4a(const int8_t* __restrict__ xq, const int8_t* __restrict__ wq,
           const float* __restrict__ s_x, const float* __restrict__ s_w, float* __restrict__ y,
           int64_t M, int64_t N, int64_t K)
{
    __shared__ __align__(16) int Xs[KW][FT + 4];
    __shared__ __align__(16) int Ws[KW][FT + 4];
    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int64_t m0 = (int64_t)blockIdx.y * FT, n0 = (int64_t)blockIdx.x * FT;
    const bool k4 = (K & 3) == 0;
    int acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[i][j] = 0;

    for (int64_t k0 = 0; k0 < K; k0 += 4 * KW) {
        for (int e = tid; e < FT * KW; e += 256) {
            const int r = e / KW, w = e % KW;
            Xs[w][r] = load_word(xq, m0 + r, M, K, k0 + 4 * w, k4);
            Ws[w][r] = load_word(wq, n0 + r, N, K, k0 + 4 * w, k4);
        }
        __syncthreads();
#pragma unroll
        for (int w = 0; w < KW; ++w) {
            const int4 a = *reinterpret_cast<const int4*>(&Xs[w][ty * 4]);
            const int4 b = *reinterpret_cast<const int4*>(&Ws[w][tx * 4]);
            const int av[4] = {a.x, a.y, a.z, a.w};
            const int bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[i][j] = __dp4a(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }

    const float sx = flush(*s_x), sw = flush(*s_w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty * 4 + i;
        if (m >= M)
            continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx * 4 + j;
            if (n < N)
                y[m * N + n] = fmul_flush(fmul_flush(__int2float_rn(acc[i][j]), sx), sw);
        }
    }
}

} // namespace

cudaError_t launch_fwd_cuda_core(const int8_t* xq, const int8_t* wq, const float* s_x,
                                 const float* s_w, float* y, int64_t M, int64_t N, int64_t K,
                                 cudaStream_t st)
{
    dim3 grid((unsigned)((N + FT - 1) / FT), (unsigned)((M + FT - 1) / FT));
    k_fwd_dp4a<<<grid, 256, 0, st>>>(xq, wq, s_x, s_w, y, M, N, K);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
