// k_selftest.cu -- on-device check of the tensor-core forward's exactness.
//
// The forward feeds int8 codes as bf16 to tcgen05.mma kind::f16 and relies on
// the fp32 accumulator holding every partial sum over a 512-term K-slice
// exactly (each is an integer below 2^23).  The hardware documentation does
// not promise how the tensor core adds inside a slice, so this check runs the
// tensor-core path (both tile widths, 128 x 256 and 128 x 128) and the
// CUDA-core dp4a path (exact by construction) on
// adversarial codes -- every code at the clamp, alternating signs, a sign flip
// at the slice boundary, one small term among large ones, a slice whose
// running sum reaches 511 * 16129 = 8,241,919 (just below 2^23) before a last
// product of +-1 (so the accumulator's lowest integer bit is probed at the top
// of its range), hashed codes -- and compares the outputs bit for bit.  With
// unit scales and K = 1024 every output is an integer below 2^24, exact in
// fp32, so a wrong integer shows.
#include "internal.h"

namespace repro {
namespace {

constexpr int ST_M = 128, ST_N = 256, ST_K = 1024;

__device__ __forceinline__ int hashed_code(uint32_t r, uint32_t c)
{
    uint32_t h = r * 0x9E3779B1u ^ (c + 0x7F4A7C15u) * 0x85EBCA77u;
    h ^= h >> 15;
    h *= 0xC2B2AE3Du;
    h ^= h >> 13;
    return (int)(h % 255u) - 127;
}

__device__ __forceinline__ int x_code(int r, int c)
{
    switch (r & 7) {
    case 0: return 127;
    case 1: return (c & 1) ? -127 : 127;
    case 2: return c == r ? 1 : 127;
    case 3: return -127;
    case 5: return (c & 511) == 511 ? (((r >> 3) & 1) ? -1 : 1) : 127;
    default: return hashed_code((uint32_t)r, (uint32_t)c);
    }
}

__device__ __forceinline__ int w_code(int n, int c)
{
    switch (n & 7) {
    case 0: return 127;
    case 1: return -127;
    case 2: return (c & 1) ? 127 : -127;
    case 3: return c < 512 ? 127 : -127;
    case 5: return (c & 511) == 511 ? 1 : 127;
    default: return hashed_code((uint32_t)(n + 7919), (uint32_t)c);
    }
}

__global__ void k_selftest_fill(int8_t* __restrict__ xq, int8_t* __restrict__ wq,
                                float* __restrict__ scales, int* __restrict__ flag)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < ST_M * ST_K)
        xq[e] = (int8_t)x_code(e / ST_K, e % ST_K);
    if (e < ST_N * ST_K)
        wq[e] = (int8_t)w_code(e / ST_K, e % ST_K);
    if (e == 0) {
        scales[0] = 1.0f;
        scales[1] = 1.0f;
        *flag = 0;
    }
}

__global__ void k_selftest_compare(const float* __restrict__ a, const float* __restrict__ b,
                                   int n, int* __restrict__ flag)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < n && __float_as_uint(a[e]) != __float_as_uint(b[e]))
        atomicOr(flag, 1);
}

inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

} // namespace

size_t selftest_ws_bytes()
{
    return align256(ST_M * ST_K) + align256(ST_N * ST_K) + align256(16) +
           2 * align256((size_t)ST_M * ST_N * 4) + align256(fwd_tc_ws_bytes(ST_M, ST_N, ST_K));
}

// 0: identical, 1: a mismatch, negative: a CUDA error
int run_selftest(void* ws, cudaStream_t st)
{
    uint8_t* p = static_cast<uint8_t*>(ws);
    int8_t* xq = reinterpret_cast<int8_t*>(p);
    p += align256(ST_M * ST_K);
    int8_t* wq = reinterpret_cast<int8_t*>(p);
    p += align256(ST_N * ST_K);
    float* scales = reinterpret_cast<float*>(p);
    int* flag = reinterpret_cast<int*>(p + 8);
    p += align256(16);
    float* y_tc = reinterpret_cast<float*>(p);
    p += align256((size_t)ST_M * ST_N * 4);
    float* y_cc = reinterpret_cast<float*>(p);
    p += align256((size_t)ST_M * ST_N * 4);
    void* tc_ws = p;

    k_selftest_fill<<<(ST_M * ST_K + 255) / 256, 256, 0, st>>>(xq, wq, scales, flag);
    count_launches(1);
    if (cudaGetLastError() != cudaSuccess)
        return -1;
    if (launch_fwd_cuda_core(xq, wq, scales, scales + 1, y_cc, ST_M, ST_N, ST_K, st) != cudaSuccess)
        return -1;
    // both tensor-core tile widths (128 x 128 and 128 x 256), each against the
    // CUDA-core output
    for (int wide = 0; wide < 2; ++wide) {
        if (launch_fwd_tc(xq, wq, scales, scales + 1, y_tc, ST_M, ST_N, ST_K, tc_ws, wide != 0,
                          st) != cudaSuccess)
            return -1;
        k_selftest_compare<<<(ST_M * ST_N + 255) / 256, 256, 0, st>>>(y_tc, y_cc, ST_M * ST_N, flag);
        count_launches(1);
    }
    int h = 0;
    if (cudaMemcpyAsync(&h, flag, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return -1;
    return h != 0 ? 1 : 0;
}

} // namespace repro
