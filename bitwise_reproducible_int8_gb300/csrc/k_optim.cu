// k_optim.cu -- the optimiser step after TreeFold: global-norm clip and AdamW.
//
// Recipe (Open-1B review, onedev.kr/papers/92, section "Premises and limits"):
// AdamW with beta1 0.9, beta2 0.95, eps 1e-8, decoupled weight decay 0.1,
// gradient clipping at global L2 norm 1.0.  The pages give no operation order;
// the library fixes this one (binary32, every operation rounded and flushed,
// never fused):
//   norm  = sqrt(sumsq)            sumsq = canonical sum of g_i (x) g_i
//   coef  = min(max_norm (/) (norm (+) 1e-6), 1)        g' = g (x) coef
//   b^t   = right-to-left binary exponentiation with rounded multiplies
//   m     = (b1 (x) m) (+) ((1 (-) b1) (x) g')
//   v     = (b2 (x) v) (+) ((1 (-) b2) (x) (g' (x) g'))
//   p     = (p (x) (1 (-) lr (x) wd)) (-) lr (x) ((m (/) (1 (-) b1^t)) (/)
//                                               (sqrt(v (/) (1 (-) b2^t)) (+) eps))
// Elementwise and HBM-bound: 16 B read and 12 B written per parameter, 16-byte
// accesses, grid a multiple of the SM count.  The step's scalars are
// recomputed by every thread from the hyperparameters (a few dozen operations).
#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

struct Scalars {
    float coef, b1, b2, one_b1, one_b2, bc1, bc2, decay, lr, eps;
};

__device__ __forceinline__ float pow_t(float b, int64_t t)
{
    float r = 1.0f, base = flush(b);
    while (t > 0) {
        if (t & 1)
            r = fmul_flush(r, base);
        base = fmul_flush(base, base);
        t >>= 1;
    }
    return r;
}

__device__ __forceinline__ Scalars scalars(const AdamWArgs& h, float sumsq, int64_t t)
{
    Scalars c;
    const float norm = flush(__fsqrt_rn(flush(sumsq)));
    const float coef = flush(__fdiv_rn(flush(h.max_norm), fadd_ftz(norm, 1e-6f)));
    c.coef = coef < 1.0f ? coef : 1.0f;
    c.b1 = flush(h.beta1);
    c.b2 = flush(h.beta2);
    c.one_b1 = fadd_ftz(1.0f, -c.b1);
    c.one_b2 = fadd_ftz(1.0f, -c.b2);
    c.bc1 = fadd_ftz(1.0f, -pow_t(c.b1, t));
    c.bc2 = fadd_ftz(1.0f, -pow_t(c.b2, t));
    c.lr = flush(h.lr);
    c.decay = fadd_ftz(1.0f, -fmul_flush(c.lr, flush(h.weight_decay)));
    c.eps = flush(h.eps);
    return c;
}

__device__ __forceinline__ void update(float& p, float& m, float& v, float g, const Scalars& c)
{
    const float gc = fmul_flush(flush(g), c.coef);
    const float mi = fadd_ftz(fmul_rn(c.b1, flush(m)), fmul_rn(c.one_b1, gc));
    const float vi = fadd_ftz(fmul_rn(c.b2, flush(v)), fmul_rn(c.one_b2, fmul_flush(gc, gc)));
    const float mh = flush(__fdiv_rn(mi, c.bc1));
    const float vh = flush(__fdiv_rn(vi, c.bc2));
    const float den = fadd_ftz(flush(__fsqrt_rn(vh)), c.eps);
    const float upd = fmul_flush(c.lr, flush(__fdiv_rn(mh, den)));
    p = fadd_ftz(fmul_rn(flush(p), c.decay), -upd);
    m = mi;
    v = vi;
}

__global__ void __launch_bounds__(256)
k_adamw(float* __restrict__ p, float* __restrict__ m, float* __restrict__ v,
        const float* __restrict__ g, int64_t n, const float* __restrict__ sumsq,
        const AdamWArgs h, int64_t t)
{
    const Scalars c = scalars(h, *sumsq, t);
    const int64_t nv = n >> 2;
    float4* p4 = reinterpret_cast<float4*>(p);
    float4* m4 = reinterpret_cast<float4*>(m);
    float4* v4 = reinterpret_cast<float4*>(v);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 pp = p4[i], mm = m4[i], vv = v4[i];
        const float4 gg = ld_stream(g4 + i);
        update(pp.x, mm.x, vv.x, gg.x, c);
        update(pp.y, mm.y, vv.y, gg.y, c);
        update(pp.z, mm.z, vv.z, gg.z, c);
        update(pp.w, mm.w, vv.w, gg.w, c);
        p4[i] = pp;
        m4[i] = mm;
        v4[i] = vv;
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t i = (nv << 2) + threadIdx.x;
        float pp = p[i], mm = m[i], vv = v[i];
        update(pp, mm, vv, g[i], c);
        p[i] = pp;
        m[i] = mm;
        v[i] = vv;
    }
}

} // namespace

cudaError_t launch_adamw(float* p, float* m, float* v, const float* g, int64_t n,
                         const float* sumsq, const AdamWArgs& h, int64_t t, int grid,
                         cudaStream_t st)
{
    k_adamw<<<grid, 256, 0, st>>>(p, m, v, g, n, sumsq, h, t);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
