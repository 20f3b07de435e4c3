// k_reduce.cu -- levels 1 and 3 of the replayed three-level gradient
// reduction (Open-1B review, onedev.kr/papers/92, section "Premises and
// limits"): micro-batch accumulation acc <- acc (+) g in micro-batch order,
// and TreeFold, which folds R replica partials in the pairing order of a
// recursive-doubling all-reduce.  Both are elementwise and HBM-bound: 16-byte
// loads and stores, grid a multiple of the SM count, one pass over all R
// inputs for TreeFold.  The output of TreeFold and of the running sum may be
// the first part itself, so that part is read on the coherent path (each
// element is read before the same thread writes it); the others, which never
// overlap the output, stream through the read-only path.
#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

__global__ void __launch_bounds__(256)
k_grad_accum(float* __restrict__ acc, const float* __restrict__ g, int64_t n)
{
    const int64_t nv = n >> 2;
    float4* a4 = reinterpret_cast<float4*>(acc);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = a4[i];
        const float4 b = ld_stream(g4 + i);
        a.x = fadd_ftz(a.x, b.x);
        a.y = fadd_ftz(a.y, b.y);
        a.z = fadd_ftz(a.z, b.z);
        a.w = fadd_ftz(a.w, b.w);
        a4[i] = a;
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t i = (nv << 2) + threadIdx.x;
        acc[i] = fadd_ftz(acc[i], g[i]);
    }
}

struct Parts {
    const float* p[REPRO_MAX_PARTS_INTERNAL];
};

__host__ __device__ constexpr int pow2_floor(int R)
{
    int p = 1;
    while (p * 2 <= R)
        p *= 2;
    return p;
}

// TF_R of one lane: survivors of the non-power-of-two pre-step, then the
// recursive-doubling pairing (survivor 0's dependency tree).
template <int R>
__device__ __forceinline__ float treefold_lane(const float (&v)[R])
{
    constexpr int P2 = pow2_floor(R);
    constexpr int RR = R - P2;
    float t[P2];
#pragma unroll
    for (int i = 0; i < P2; ++i)
        t[i] = (i < RR) ? fadd_ftz(v[2 * i], v[2 * i + 1]) : v[RR + i];
#pragma unroll
    for (int d = 1; d < P2; d *= 2)
#pragma unroll
        for (int j = 0; j < P2; j += 2 * d)
            t[j] = fadd_ftz(t[j], t[j + d]);
    return t[0];
}

template <int R>
__global__ void __launch_bounds__(256)
k_treefold(const Parts parts, int64_t n, float* out)
{
    const int64_t nv = n >> 2;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x) {
        float x[R], y[R], z[R], w[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4* src = reinterpret_cast<const float4*>(parts.p[r]) + i;
            const float4 v = r == 0 ? ld_stream_coherent(src) : ld_stream(src);
            x[r] = v.x;
            y[r] = v.y;
            z[r] = v.z;
            w[r] = v.w;
        }
        float4 o;
        if (R == 1) {
            o = make_float4(x[0], y[0], z[0], w[0]);
        } else {
            o = make_float4(treefold_lane<R>(x), treefold_lane<R>(y), treefold_lane<R>(z),
                            treefold_lane<R>(w));
        }
        // evict-first: the folded gradient leaves the step (the optimiser or
        // the host reads it next), so its lines are written back now instead
        // of lingering dirty in L2 into the next kernel's reads
        __stcs(reinterpret_cast<float4*>(out) + i, o);
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t i = (nv << 2) + threadIdx.x;
        float x[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            x[r] = parts.p[r][i];
        out[i] = (R == 1) ? x[0] : treefold_lane<R>(x);
    }
}

// any R up to the maximum: survivors in a local array, same pairing
__global__ void __launch_bounds__(256)
k_treefold_generic(const Parts parts, int R, int64_t n, float* out)
{
    int p2 = 1;
    while (p2 * 2 <= R)
        p2 *= 2;
    const int rr = R - p2;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float t[REPRO_MAX_PARTS_INTERNAL];
        for (int k = 0; k < p2; ++k)
            t[k] = (k < rr) ? fadd_ftz(parts.p[2 * k][i], parts.p[2 * k + 1][i])
                            : parts.p[rr + k][i];
        for (int d = 1; d < p2; d *= 2)
            for (int j = 0; j < p2; j += 2 * d)
                t[j] = fadd_ftz(t[j], t[j + d]);
        out[i] = (R == 1) ? parts.p[0][i] : t[0];
    }
}

// level 2: left fold of S shard partials in mesh order (first taken as it is)
template <int S>
__global__ void __launch_bounds__(256)
k_running_sum(const Parts parts, int64_t n, float* out)
{
    const int64_t nv = n >> 2;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = ld_stream_coherent(reinterpret_cast<const float4*>(parts.p[0]) + i);
#pragma unroll
        for (int s = 1; s < S; ++s) {
            const float4 b = ld_stream(reinterpret_cast<const float4*>(parts.p[s]) + i);
            a.x = fadd_ftz(a.x, b.x);
            a.y = fadd_ftz(a.y, b.y);
            a.z = fadd_ftz(a.z, b.z);
            a.w = fadd_ftz(a.w, b.w);
        }
        reinterpret_cast<float4*>(out)[i] = a;
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t i = (nv << 2) + threadIdx.x;
        float a = parts.p[0][i];
#pragma unroll
        for (int s = 1; s < S; ++s)
            a = fadd_ftz(a, parts.p[s][i]);
        out[i] = a;
    }
}

__global__ void __launch_bounds__(256)
k_running_sum_generic(const Parts parts, int S, int64_t n, float* out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        float a = parts.p[0][i];
        for (int s = 1; s < S; ++s)
            a = fadd_ftz(a, parts.p[s][i]);
        out[i] = a;
    }
}

// debug scan: any NaN or infinity among n floats ORs the non-finite bit into
// the error word (one atomic per warp that finds one).  p is 16-byte aligned
__global__ void __launch_bounds__(256) k_check_finite(const float* __restrict__ p, int64_t n, int* err)
{
    const int64_t nv = n >> 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
        const float4 v = ld_stream(reinterpret_cast<const float4*>(p) + i);
        bad = bad || !isfinite(v.x) || !isfinite(v.y) || !isfinite(v.z) || !isfinite(v.w);
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3))
        bad = bad || !isfinite(p[(nv << 2) + threadIdx.x]);
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0)
        atomicOr(err, kErrNonfiniteBit);
}

} // namespace

cudaError_t launch_running_sum(const float* const* parts, int S, int64_t n, float* out, int grid,
                               cudaStream_t st)
{
    Parts P;
    for (int r = 0; r < REPRO_MAX_PARTS_INTERNAL; ++r)
        P.p[r] = r < S ? parts[r] : nullptr;
    switch (S) {
    case 1: k_running_sum<1><<<grid, 256, 0, st>>>(P, n, out); break;
    case 2: k_running_sum<2><<<grid, 256, 0, st>>>(P, n, out); break;
    case 3: k_running_sum<3><<<grid, 256, 0, st>>>(P, n, out); break;
    case 4: k_running_sum<4><<<grid, 256, 0, st>>>(P, n, out); break;
    case 5: k_running_sum<5><<<grid, 256, 0, st>>>(P, n, out); break;
    case 6: k_running_sum<6><<<grid, 256, 0, st>>>(P, n, out); break;
    case 7: k_running_sum<7><<<grid, 256, 0, st>>>(P, n, out); break;
    case 8: k_running_sum<8><<<grid, 256, 0, st>>>(P, n, out); break;
    default: k_running_sum_generic<<<grid, 256, 0, st>>>(P, S, n, out); break;
    }
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_grad_accum(float* acc, const float* g, int64_t n, int grid, cudaStream_t st)
{
    k_grad_accum<<<grid, 256, 0, st>>>(acc, g, n);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_treefold(const float* const* parts, int R, int64_t n, float* out, int grid,
                            cudaStream_t st)
{
    Parts P;
    for (int r = 0; r < REPRO_MAX_PARTS_INTERNAL; ++r)
        P.p[r] = r < R ? parts[r] : nullptr;
    switch (R) {
    case 1: k_treefold<1><<<grid, 256, 0, st>>>(P, n, out); break;
    case 2: k_treefold<2><<<grid, 256, 0, st>>>(P, n, out); break;
    case 3: k_treefold<3><<<grid, 256, 0, st>>>(P, n, out); break;
    case 4: k_treefold<4><<<grid, 256, 0, st>>>(P, n, out); break;
    case 5: k_treefold<5><<<grid, 256, 0, st>>>(P, n, out); break;
    case 6: k_treefold<6><<<grid, 256, 0, st>>>(P, n, out); break;
    case 7: k_treefold<7><<<grid, 256, 0, st>>>(P, n, out); break;
    case 8: k_treefold<8><<<grid, 256, 0, st>>>(P, n, out); break;
    default: k_treefold_generic<<<grid, 256, 0, st>>>(P, R, n, out); break;
    }
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_check_finite(const float* p, int64_t n, int* err, cudaStream_t st)
{
    if (n <= 0)
        return cudaSuccess;
    const int64_t want = ((n >> 2) + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    k_check_finite<<<(unsigned)(want < 1 ? 1 : (want > cap ? cap : want)), 256, 0, st>>>(p, n, err);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
