// k_quant.cu -- int8 quantiser.
//
// q = clamp(round_half_even(x (/) s), -127, 127): int8 weights and activations
// for every attention/FFN linear (Open-1B review, onedev.kr/papers/92, section
// "How to use"), deterministic rounding since stochastic rounding breaks
// bitwise reproducibility (section "Premises and limits").  The quotient is
// the correctly rounded binary32 division; it is then rounded to an integer
// with ties to even (cvt.rni), which saturates out-of-range values and maps
// NaN to 0 before the clamp.  A zero (or subnormal) scale gives q = 0.
//
// Streaming kernel: each thread converts 16 elements per step with four
// 16-byte loads and one 16-byte store; the grid is a multiple of the SM count.
#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace repro {
namespace {

__device__ __forceinline__ int quant_one(float x, float s, int qmax)
{
    const float v = __fdiv_rn(flush(x), s);
    int q = __float2int_rn(v);
    q = q > qmax ? qmax : q;
    q = q < -qmax ? -qmax : q;
    return q;
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d)
{
    return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
           ((uint32_t)(d & 0xff) << 24);
}

__global__ void __launch_bounds__(256)
k_quant(const float* __restrict__ x, int64_t n, const float* __restrict__ scale, int qmax,
        int8_t* __restrict__ q)
{
    pdl_wait();
    pdl_trigger();
    const float s = flush(*scale);
    const int64_t nv = n >> 4;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint4* q16 = reinterpret_cast<uint4*>(q);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (s == 0.f) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride)
            q16[i] = make_uint4(0, 0, 0, 0);
    } else {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
            const float4 a = ld_stream(x4 + 4 * i + 0);
            const float4 b = ld_stream(x4 + 4 * i + 1);
            const float4 c = ld_stream(x4 + 4 * i + 2);
            const float4 d = ld_stream(x4 + 4 * i + 3);
            uint4 o;
            o.x = pack4(quant_one(a.x, s, qmax), quant_one(a.y, s, qmax), quant_one(a.z, s, qmax),
                        quant_one(a.w, s, qmax));
            o.y = pack4(quant_one(b.x, s, qmax), quant_one(b.y, s, qmax), quant_one(b.z, s, qmax),
                        quant_one(b.w, s, qmax));
            o.z = pack4(quant_one(c.x, s, qmax), quant_one(c.y, s, qmax), quant_one(c.z, s, qmax),
                        quant_one(c.w, s, qmax));
            o.w = pack4(quant_one(d.x, s, qmax), quant_one(d.y, s, qmax), quant_one(d.z, s, qmax),
                        quant_one(d.w, s, qmax));
            q16[i] = o;
        }
    }
    // tail (< 16 elements)
    if (blockIdx.x == 0) {
        const int64_t i = (nv << 4) + threadIdx.x;
        if (threadIdx.x < 16 && i < n)
            q[i] = (int8_t)(s == 0.f ? 0 : quant_one(x[i], s, qmax));
    }
}

// several tensors, each with its own scale: the 16-element groups of all of
// them form one grid-stride range, tensor t owning groups [g0[t], g0[t+1])
struct QuantMulti {
    const float* x[REPRO_MAX_TENSORS_INTERNAL];
    int8_t* q[REPRO_MAX_TENSORS_INTERNAL];
    int64_t n[REPRO_MAX_TENSORS_INTERNAL];
    int64_t g0[REPRO_MAX_TENSORS_INTERNAL + 1];
    int count;
};

__global__ void __launch_bounds__(256)
k_quant_multi(const __grid_constant__ QuantMulti a, const float* __restrict__ scales, int qmax)
{
    pdl_wait();
    pdl_trigger();
    const int64_t total = a.g0[a.count];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int t = 0;
    float s = 0.f;
    int st = -1;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride) {
        while (g >= a.g0[t + 1])   // g only grows: the owning tensor only moves forward
            ++t;
        if (t != st) {
            s = flush(scales[t]);
            st = t;
        }
        const int64_t i = g - a.g0[t];
        uint4 o;
        if (s == 0.f) {
            o = make_uint4(0, 0, 0, 0);
        } else {
            const float4* x4 = reinterpret_cast<const float4*>(a.x[t]) + 4 * i;
            const float4 v0 = ld_stream(x4 + 0);
            const float4 v1 = ld_stream(x4 + 1);
            const float4 v2 = ld_stream(x4 + 2);
            const float4 v3 = ld_stream(x4 + 3);
            o.x = pack4(quant_one(v0.x, s, qmax), quant_one(v0.y, s, qmax),
                        quant_one(v0.z, s, qmax), quant_one(v0.w, s, qmax));
            o.y = pack4(quant_one(v1.x, s, qmax), quant_one(v1.y, s, qmax),
                        quant_one(v1.z, s, qmax), quant_one(v1.w, s, qmax));
            o.z = pack4(quant_one(v2.x, s, qmax), quant_one(v2.y, s, qmax),
                        quant_one(v2.z, s, qmax), quant_one(v2.w, s, qmax));
            o.w = pack4(quant_one(v3.x, s, qmax), quant_one(v3.y, s, qmax),
                        quant_one(v3.z, s, qmax), quant_one(v3.w, s, qmax));
        }
        reinterpret_cast<uint4*>(a.q[t])[i] = o;
    }
    // tails (< 16 elements): CTA t finishes tensor t
    if (blockIdx.x < (unsigned)a.count && threadIdx.x < 16) {
        const int tt = blockIdx.x;
        const int64_t i = ((a.n[tt] >> 4) << 4) + threadIdx.x;
        if (i < a.n[tt]) {
            const float sv = flush(scales[tt]);
            a.q[tt][i] = (int8_t)(sv == 0.f ? 0 : quant_one(a.x[tt][i], sv, qmax));
        }
    }
}

} // namespace

cudaError_t launch_quant_multi(const float* const* xs, const int64_t* ns, int count,
                               const float* scales, int qmax, int8_t* const* qs, int grid,
                               cudaStream_t st)
{
    QuantMulti a;
    a.count = count;
    a.g0[0] = 0;
    for (int t = 0; t < count; ++t) {
        a.x[t] = xs[t];
        a.q[t] = qs[t];
        a.n[t] = ns[t];
        a.g0[t + 1] = a.g0[t] + (ns[t] >> 4);
    }
    // at least one CTA per tensor, for the tails
    if (grid < count)
        grid = count;
    const cudaError_t e = launch_pdl(k_quant_multi, dim3(grid), dim3(256), 0, st, a, scales, qmax);
    count_launches(1);
    return e;
}

cudaError_t launch_quant(const float* x, int64_t n, const float* scale, int qmax, int8_t* q,
                         int grid, cudaStream_t st)
{
    const cudaError_t e = launch_pdl(k_quant, dim3(grid), dim3(256), 0, st, x, n, scale, qmax, q);
    count_launches(1);
    return e;
}

} // namespace repro
