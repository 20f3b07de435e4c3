// k_scale.cu -- per-tensor scales.
//
// Weight scale (Open-1B review, onedev.kr/papers/92, sections "How to use" and
// "Premises and limits": the step size is re-pinned from the weights every
// optimiser step as 2*mean(|w|)/sqrt(q_max)).  The sum of |w| follows the
// canonical order: chunks of 64 summed left to right, then the stride-doubling
// pairwise tree over chunk partials.  The tree over any aligned block of 2^b
// chunk partials is itself the canonical tree of that block, and the tree over
// the block results (ragged last block included) completes the canonical tree,
// so the reduction runs as one pass over HBM (phase 1: one CTA per aligned
// block of chunks) plus tiny tree passes over the block partials.
//
// Activation scale: max|x| / q_max; the maximum is exact, so any order works.
#include <float.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"

namespace repro {
namespace {

constexpr int P1_CHUNKS = 128;   // chunks (and threads) per phase-1 CTA
constexpr int P2_MAX = 1024;     // partials (and threads) per tree-pass CTA

// term of the canonical sum: |x| (weight scale) or x (x) x (squared norm); a
// subnormal x gives a term the first add reads as zero either way
template <int SQUARE>
__device__ __forceinline__ float term(float x)
{
    return SQUARE ? fmul_rn(x, x) : fabsf(x);
}

// The tensors of one call (one, or all of a step's weights): their phase-1
// blocks form one range, the blocks of tensor t being [blk0[t], blk0[t+1]).
struct MultiArgs {
    const float* x[REPRO_MAX_TENSORS_INTERNAL];
    int64_t n[REPRO_MAX_TENSORS_INTERNAL];
    int64_t blk0[REPRO_MAX_TENSORS_INTERNAL + 1];
    int count;
};

// tensor owning phase-1 block b (blk0 ascending, blk0[0] = 0)
__device__ __forceinline__ int tensor_of(const MultiArgs& a, int64_t b)
{
    int lo = 0, hi = a.count - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.blk0[mid] <= b)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte asynchronous copy global -> shared; bytes past src_bytes read as 0
__device__ __forceinline__ void cp_async16(uint32_t sdst, const void* gsrc, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(sdst), "l"(gsrc),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Thread j's chunk of a block staged in shared memory (chunk j's 16 float4
// sit XOR-swizzled at S[j*16 + (p ^ (j & 15))], so the fill and these reads
// are free of bank conflicts), copied to registers.
__device__ __forceinline__ void chunk_to_regs(const float4* __restrict__ S, int j, float4 (&v)[16])
{
#pragma unroll
    for (int p = 0; p < 16; ++p)
        v[p] = S[j * 16 + (p ^ (j & 15))];
}

// Left-to-right sum of the chunk's first len (1..64) terms, seeded with the
// first term.
template <int SQUARE>
__device__ __forceinline__ float chunk_sum(const float4 (&v)[16], int len)
{
    float a = term<SQUARE>(v[0].x);
    if (len == 64) {
        a = fadd_ftz(a, term<SQUARE>(v[0].y));
        a = fadd_ftz(a, term<SQUARE>(v[0].z));
        a = fadd_ftz(a, term<SQUARE>(v[0].w));
#pragma unroll
        for (int p = 1; p < 16; ++p) {
            a = fadd_ftz(a, term<SQUARE>(v[p].x));
            a = fadd_ftz(a, term<SQUARE>(v[p].y));
            a = fadd_ftz(a, term<SQUARE>(v[p].z));
            a = fadd_ftz(a, term<SQUARE>(v[p].w));
        }
    } else {
#pragma unroll
        for (int i = 1; i < 64; ++i) {
            const float4 q = v[i >> 2];
            const float x = (i & 3) == 0 ? q.x : (i & 3) == 1 ? q.y : (i & 3) == 2 ? q.z : q.w;
            if (i < len)
                a = fadd_ftz(a, term<SQUARE>(x));
        }
    }
    return a;
}

// The stride-doubling tree over the cnt (<= 128) chunk partials of a block,
// partial j held by thread j of the 128-thread CTA: levels 1..16 inside each
// warp with shuffles (lane j, j a multiple of 2s, adds lane j+s's partial
// when j+s < cnt -- the tree's own pairs), levels 32 and 64 by thread 0 over
// the four warps' partials in W.  Every thread must call it; the result is
// valid in thread 0.
__device__ __forceinline__ float block_tree(float a, float* __restrict__ W, int cnt)
{
    const int j = threadIdx.x, lane = j & 31;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const float o = __shfl_down_sync(0xffffffffu, a, s);
        if ((lane & (2 * s - 1)) == 0 && j + s < cnt)
            a = fadd_ftz(a, o);
    }
    if (lane == 0)
        W[j >> 5] = a;
    __syncthreads();
    float r = 0.f;
    if (j == 0) {
        r = W[0];
        float r2 = W[2];
        if (32 < cnt)
            r = fadd_ftz(r, W[1]);
        if (96 < cnt)
            r2 = fadd_ftz(r2, W[3]);
        if (64 < cnt)
            r = fadd_ftz(r, r2);
    }
    return r;
}

constexpr int P1_STAGES = 3;                                       // blocks in flight per CTA
constexpr size_t P1_SMEM = (size_t)P1_STAGES * P1_CHUNKS * 16 * sizeof(float4);   // 96 KB

// Phase 1, persistent: CTA c takes blocks c, c + G, c + 2G, ... (G CTAs, two
// per SM) of all the call's tensors.  Each block's 32 KB is copied into a
// three-stage shared-memory ring with 16-byte asynchronous copies (zero fill
// past the tensor's end).  When a block has landed, every thread moves its
// own chunk into registers and the stage is refilled at once, so three
// blocks (192 KB per SM) stay in flight while the chunk sums and the tree of
// the current block run from registers.  Writes one partial per block.
template <int SQUARE>
__global__ void __launch_bounds__(P1_CHUNKS)
k_absum_pipe(const __grid_constant__ MultiArgs a, int blk_log2, float* __restrict__ part)
{
    extern __shared__ __align__(16) float4 ring[];
    __shared__ float W[P1_CHUNKS / 32];
    pdl_wait();
    pdl_trigger();
    const int64_t total = a.blk0[a.count];
    const int nb = 1 << blk_log2;
    const int64_t step = gridDim.x;
    auto issue = [&](int64_t b, int stage) {
        if (b < total) {
            const int t = tensor_of(a, b);
            const float* x = a.x[t];
            const int64_t n = a.n[t];
            const int64_t e0 = (b - a.blk0[t]) * (int64_t)nb * 64;
            float4* S = ring + stage * (P1_CHUNKS * 16);
            if (nb == P1_CHUNKS && e0 + P1_CHUNKS * 64 <= n) {
                // a full block: float4 g = tid + 128u is chunk (tid >> 4) + 8u,
                // part tid & 15, so only the swizzle's parity in u varies
                const int ch0 = threadIdx.x >> 4, p = threadIdx.x & 15;
                const float* src = x + e0 + 4 * threadIdx.x;
                const uint32_t d0 = smem_u32(S + ch0 * 16 + (p ^ ch0));
                const uint32_t d1 = smem_u32(S + ch0 * 16 + (p ^ (ch0 + 8)));
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    cp_async16((u & 1 ? d1 : d0) + (uint32_t)(u * 128 * 16), src + 512 * u, 16);
                cp_async_commit();
                return;
            }
            for (int g = threadIdx.x; g < nb * 16; g += P1_CHUNKS) {
                const int ch = g >> 4, p = g & 15;
                const int64_t e = e0 + (int64_t)g * 4;
                const int bytes = e >= n ? 0 : (int)min((int64_t)16, (n - e) * 4);
                cp_async16(smem_u32(&S[ch * 16 + (p ^ (ch & 15))]),
                           bytes ? static_cast<const void*>(x + e) : static_cast<const void*>(x),
                           bytes);
            }
        }
        cp_async_commit();   // one group per block, empty past the end
    };
    int64_t b = blockIdx.x;
#pragma unroll
    for (int s0 = 0; s0 < P1_STAGES; ++s0)
        issue(b + s0 * step, s0);
    for (int i = 0; b < total; b += step, ++i) {
        cp_async_wait<P1_STAGES - 1>();   // this thread's copies of block b have landed
        __syncthreads();                  // everyone's have
        const int stage = i % P1_STAGES;
        const int j = threadIdx.x;
        float4 v[16];
        chunk_to_regs(ring + stage * (P1_CHUNKS * 16), j, v);
        __syncthreads();                  // everyone has read the stage: refill it
        issue(b + P1_STAGES * step, stage);
        const int t = tensor_of(a, b);
        const int64_t n = a.n[t];
        const int64_t c0 = (b - a.blk0[t]) * nb;
        const int cnt = (int)min((int64_t)nb, ((n + 63) >> 6) - c0);
        float sum = 0.f;
        if (j < cnt)
            sum = chunk_sum<SQUARE>(v, (int)min((int64_t)64, n - (c0 + j) * 64));
        const float r = block_tree(sum, W, cnt);
        if (j == 0)
            part[b] = r;
    }
    cp_async_wait<0>();
}

// s_w = (2 (x) (S (/) float(n))) (/) sqrt(float(q_max)); every operand and
// result flushed
__device__ float weight_scale_from_sum(float S, int64_t n, int qmax)
{
    const float mean = flush(__fdiv_rn(flush(S), __ll2float_rn(n)));
    const float twice = fmul_flush(2.0f, mean);
    const float root = flush(__fsqrt_rn(__int2float_rn(qmax)));
    return flush(__fdiv_rn(twice, root));
}

// Tree pass: CTA b reduces partials [b*2^k, (b+1)*2^k) of `in` with the
// stride-doubling tree.  With one CTA left it finishes the weight scale.
__global__ void __launch_bounds__(P2_MAX)
k_tree_pass(const float* __restrict__ in, int64_t cnt_total, int blk_log2,
            float* __restrict__ out, int final_pass, int64_t n, int qmax,
            float* __restrict__ scale_out)
{
    __shared__ float T[P2_MAX];
    pdl_wait();
    pdl_trigger();
    const int nb = 1 << blk_log2;
    const int64_t b0 = (int64_t)blockIdx.x * nb;
    const int cnt = (int)min((int64_t)nb, cnt_total - b0);
    for (int j = threadIdx.x; j < cnt; j += blockDim.x)
        T[j] = in[b0 + j];
    __syncthreads();
    for (int s = 1; s < cnt; s <<= 1) {
        for (int j = threadIdx.x * 2 * s; j + s < cnt; j += blockDim.x * 2 * s)
            T[j] = fadd_ftz(T[j], T[j + s]);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (final_pass == 1)
            scale_out[0] = weight_scale_from_sum(T[0], n, qmax);
        else if (final_pass == 2)
            scale_out[0] = flush(T[0]);      // the canonical sum itself
        else
            out[blockIdx.x] = T[0];
    }
}

// ---------------------------------------------------------------- amax

__device__ __forceinline__ float absflush(float v)
{
    v = fabsf(v);
    return v < FLT_MIN ? 0.f : v;
}

__global__ void __launch_bounds__(256)
k_amax_partial(const float* __restrict__ x, int64_t n, float* __restrict__ part)
{
    pdl_wait();
    pdl_trigger();
    float m = 0.f;
    const int64_t nv = n >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // four independent loads in flight per step (the maximum is order-free)
    for (; i + 3 * stride < nv; i += 4 * stride) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            v[u] = ld_stream(x4 + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            m = fmaxf(m, fmaxf(fmaxf(absflush(v[u].x), absflush(v[u].y)),
                               fmaxf(absflush(v[u].z), absflush(v[u].w))));
    }
    for (; i < nv; i += stride) {
        const float4 v = ld_stream(x4 + i);
        m = fmaxf(m, fmaxf(fmaxf(absflush(v.x), absflush(v.y)), fmaxf(absflush(v.z), absflush(v.w))));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3))
        m = fmaxf(m, absflush(x[(nv << 2) + threadIdx.x]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float W[8];
    if ((threadIdx.x & 31) == 0)
        W[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            m = fmaxf(m, W[w]);
        part[blockIdx.x] = m;
    }
}

__global__ void __launch_bounds__(1024)
k_amax_final(const float* __restrict__ part, int cnt, int qmax, float* __restrict__ scale_out)
{
    pdl_wait();
    float m = 0.f;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x)
        m = fmaxf(m, part[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float W[32];
    if ((threadIdx.x & 31) == 0)
        W[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            m = fmaxf(m, W[w]);
        scale_out[0] = flush(__fdiv_rn(m, __int2float_rn(qmax)));
    }
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------- several tensors

constexpr int TREE_MULTI_MAX = 8192;   // block partials one tree CTA holds (1024 x 8)

// one CTA of 1024 threads per tensor: the stride-doubling tree over the
// tensor's block partials, then its weight scale.  Thread t holds partials
// 8t .. 8t+7 and takes levels 1, 2, 4 in registers; levels 8 .. 128 run across
// the lanes of a warp with shuffles, levels 256 .. 4096 across the warps'
// partials in warp 0 -- at every level partial j (j a multiple of 2s) adds
// partial j + s when j + s < cnt, as the tree defines.
__global__ void __launch_bounds__(1024)
k_tree_multi(const __grid_constant__ MultiArgs a, const float* __restrict__ part, int qmax,
             float* __restrict__ scales)
{
    __shared__ float W[32];
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    const int64_t b0 = a.blk0[t];
    const int cnt = (int)(a.blk0[t + 1] - b0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        v[r] = 8 * tid + r < cnt ? part[b0 + 8 * tid + r] : 0.f;
#pragma unroll
    for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int r = 0; r < 8; r += 2 * s)
            if (8 * tid + r + s < cnt)
                v[r] = fadd_ftz(v[r], v[r + s]);
    float x = v[0];
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {   // element stride 8s
        const float o = __shfl_down_sync(0xffffffffu, x, s);
        if ((lane & (2 * s - 1)) == 0 && 8 * (tid + s) < cnt)
            x = fadd_ftz(x, o);
    }
    if (lane == 0)
        W[warp] = x;
    __syncthreads();
    if (warp == 0) {
        x = W[lane];
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {   // element stride 256s
            const float o = __shfl_down_sync(0xffffffffu, x, s);
            if ((lane & (2 * s - 1)) == 0 && 256 * (lane + s) < cnt)
                x = fadd_ftz(x, o);
        }
        if (lane == 0)
            scales[t] = weight_scale_from_sum(x, a.n[t], qmax);
    }
}

constexpr int AMAX_BLOCK = 8192;   // elements per phase-1 CTA of the multi amax

__global__ void __launch_bounds__(256)
k_amax_multi(const __grid_constant__ MultiArgs a, float* __restrict__ part)
{
    pdl_wait();
    pdl_trigger();
    const int t = tensor_of(a, blockIdx.x);
    const float* x = a.x[t];
    const int64_t n = a.n[t];
    const int64_t e0 = (int64_t)(blockIdx.x - a.blk0[t]) * AMAX_BLOCK;
    float m = 0.f;
    if (e0 + AMAX_BLOCK <= n) {
        const float4* x4 = reinterpret_cast<const float4*>(x + e0);
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            v[u] = ld_stream(x4 + threadIdx.x + u * 256);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            m = fmaxf(m, fmaxf(fmaxf(absflush(v[u].x), absflush(v[u].y)),
                               fmaxf(absflush(v[u].z), absflush(v[u].w))));
    } else {
        for (int64_t e = e0 + threadIdx.x; e < n; e += 256)
            m = fmaxf(m, absflush(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float W[8];
    if ((threadIdx.x & 31) == 0)
        W[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 8; ++w)
            m = fmaxf(m, W[w]);
        part[blockIdx.x] = m;
    }
}

__global__ void __launch_bounds__(1024)
k_amax_final_multi(const __grid_constant__ MultiArgs a, const float* __restrict__ part, int qmax,
                   float* __restrict__ scales)
{
    pdl_wait();
    const int t = blockIdx.x;
    float m = 0.f;
    for (int64_t i = a.blk0[t] + threadIdx.x; i < a.blk0[t + 1]; i += blockDim.x)
        m = fmaxf(m, part[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float W[32];
    if ((threadIdx.x & 31) == 0)
        W[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 32; ++w)
            m = fmaxf(m, W[w]);
        scales[t] = flush(__fdiv_rn(m, __int2float_rn(qmax)));
    }
}

} // namespace

// Phase-1 block of 2^min(k,7) chunks, tree passes of 2^max(k,1) partials
// (capped at 1024).  Workspace: phase-1 partials, then the first tree pass's
// output; later passes ping-pong between the two regions (they only shrink).
static void split_blocks(int block_log2, int& p1_log2, int& p2_log2)
{
    if (block_log2 < 0) {   // default: 128-chunk CTAs, 1024-partial tree passes
        p1_log2 = 7;
        p2_log2 = 10;
        return;
    }
    p1_log2 = block_log2 < 7 ? block_log2 : 7;
    p2_log2 = block_log2 < 1 ? 1 : (block_log2 > 10 ? 10 : block_log2);
}

size_t wscale_ws_bytes(int64_t n, int block_log2)
{
    int p1, p2;
    split_blocks(block_log2, p1, p2);
    const int64_t C = cdiv(n, 64);
    const int64_t c1 = cdiv(C, (int64_t)1 << p1);
    const int64_t c2 = cdiv(c1, (int64_t)1 << p2);
    return (size_t)(c1 + c2 + 64) * sizeof(float);
}

// phase 1 over the blocks of a.count tensors (a.blk0 filled): one block
// partial per block into part
static cudaError_t launch_phase1(const MultiArgs& a, int square, int p1, float* part,
                                 cudaStream_t st)
{
    auto kern = square ? k_absum_pipe<1> : k_absum_pipe<0>;
    // the 96 KB ring needs the opt-in shared-memory size, set once per device
    // and kernel (a host call that takes microseconds, kept off every launch)
    constexpr int kMaxDev = 64;
    static std::atomic<int> opted[2][kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDev || opted[square][dev].load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P1_SMEM);
        if (e != cudaSuccess)
            return e;
        if (dev < kMaxDev)
            opted[square][dev].store(1, std::memory_order_release);
    }
    const int64_t blocks = a.blk0[a.count];
    // two 97 KB CTAs per SM, unless the launch-configuration hook sets the grid
    const int64_t cap = launch_cfg().elementwise_blocks > 0 ? launch_cfg().elementwise_blocks
                                                            : 2 * (int64_t)num_sms();
    const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
    e = launch_pdl(kern, dim3(grid), dim3(P1_CHUNKS), P1_SMEM, st, a, p1, part);
    if (e == cudaErrorInvalidValue) {
        // the opt-in was lost (the device was reset since): set it again
        (void)cudaGetLastError();
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P1_SMEM);
        if (e == cudaSuccess)
            e = launch_pdl(kern, dim3(grid), dim3(P1_CHUNKS), P1_SMEM, st, a, p1, part);
    }
    count_launches(1);
    return e;
}

// canonical sum of |x_i| (square = 0) or x_i (x) x_i (square = 1); with
// square = 0 the last pass turns the sum into the weight scale, with
// square = 1 it stores the sum
static cudaError_t canonical_sum(const float* x, int64_t n, int square, int qmax, float* out,
                                 void* ws, int block_log2, cudaStream_t st)
{
    int p1, p2;
    split_blocks(block_log2, p1, p2);
    const int64_t C = cdiv(n, 64);
    int64_t cnt = cdiv(C, (int64_t)1 << p1);
    float* regA = static_cast<float*>(ws);
    float* regB = regA + cnt + 32;
    float* scale_out = out;
    MultiArgs a;
    a.count = 1;
    a.x[0] = x;
    a.n[0] = n;
    a.blk0[0] = 0;
    a.blk0[1] = cnt;
    cudaError_t e = launch_phase1(a, square, p1, regA, st);
    if (e != cudaSuccess)
        return e;
    float* src = regA;
    float* dst = regB;
    for (;;) {
        const int64_t grid = cdiv(cnt, (int64_t)1 << p2);
        const int final_pass = grid == 1 ? (square ? 2 : 1) : 0;
        e = launch_pdl(k_tree_pass, dim3((unsigned)grid), dim3(P2_MAX), 0, st, src, cnt, p2, dst,
                       final_pass, n, qmax, scale_out);
        count_launches(1);
        if (e != cudaSuccess)
            return e;
        if (final_pass)
            break;
        cnt = grid;
        float* t = src;
        src = dst;
        dst = t;
    }
    return cudaGetLastError();
}

cudaError_t launch_wscale_meanabs(const float* x, int64_t n, int qmax, float* scale_out,
                                  void* ws, int block_log2, cudaStream_t st)
{
    return canonical_sum(x, n, 0, qmax, scale_out, ws, block_log2, st);
}

cudaError_t launch_sumsq(const float* x, int64_t n, float* out, void* ws, int block_log2,
                         cudaStream_t st)
{
    return canonical_sum(x, n, 1, 0, out, ws, block_log2, st);
}

int amax_grid(int64_t n)
{
    const int64_t want = cdiv(n, 256 * 4 * 4);
    const int64_t cap = (int64_t)num_sms() * 4;
    return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

// phase-1 blocks per tensor for the multi-tensor calls: 2^p1 chunks each
// (weight scale) or AMAX_BLOCK elements (activation scale)
static int64_t multi_blocks(int64_t n, int mode, int p1)
{
    return mode == 0 ? cdiv(cdiv(n, 64), (int64_t)1 << p1) : cdiv(n, AMAX_BLOCK);
}

size_t wscale_multi_ws_bytes(const int64_t* ns, int count)
{
    // the block partials of every tensor at the finest split (one chunk per
    // block, the launch-configuration hook's smallest), or one tensor's
    // workspace on the multi-pass path, whichever is larger
    int64_t total = 0, single = 0;
    for (int t = 0; t < count; ++t) {
        total += cdiv(ns[t], 64) + 64;
        const int64_t one = (int64_t)(wscale_ws_bytes(ns[t], 0) / sizeof(float));
        single = one > single ? one : single;
    }
    return (size_t)((total > single ? total : single) + 64) * sizeof(float);
}

cudaError_t launch_wscale_multi(const float* const* xs, const int64_t* ns, int count, int mode,
                                int qmax, float* scales, void* ws, int block_log2,
                                cudaStream_t st)
{
    int p1, p2;
    split_blocks(block_log2, p1, p2);
    MultiArgs a;
    a.count = count;
    a.blk0[0] = 0;
    bool one_pass = true;
    for (int t = 0; t < count; ++t) {
        a.x[t] = xs[t];
        a.n[t] = ns[t];
        const int64_t nb = multi_blocks(ns[t], mode, p1);
        a.blk0[t + 1] = a.blk0[t] + nb;
        if (mode == 0 && nb > TREE_MULTI_MAX)
            one_pass = false;
    }
    if (!one_pass) {
        // a tensor too large for one tree CTA: each tensor on its own,
        // through the single-tensor passes (same bits)
        for (int t = 0; t < count; ++t) {
            cudaError_t e = canonical_sum(xs[t], ns[t], 0, qmax, scales + t, ws, block_log2, st);
            if (e != cudaSuccess)
                return e;
        }
        return cudaSuccess;
    }
    float* part = static_cast<float*>(ws);
    const unsigned grid = (unsigned)a.blk0[count];
    cudaError_t e;
    if (mode == 0) {
        e = launch_phase1(a, 0, p1, part, st);
        if (e == cudaSuccess)
            e = launch_pdl(k_tree_multi, dim3((unsigned)count), dim3(1024), 0, st, a,
                           (const float*)part, qmax, scales);
        count_launches(1);
    } else {
        e = launch_pdl(k_amax_multi, dim3(grid), dim3(256), 0, st, a, part);
        if (e == cudaSuccess)
            e = launch_pdl(k_amax_final_multi, dim3((unsigned)count), dim3(1024), 0, st, a,
                           (const float*)part, qmax, scales);
        count_launches(2);
    }
    return e;
}

cudaError_t launch_wscale_amax(const float* x, int64_t n, int qmax, float* scale_out, void* ws,
                               int grid, cudaStream_t st)
{
    float* part = static_cast<float*>(ws);
    cudaError_t e = launch_pdl(k_amax_partial, dim3(grid), dim3(256), 0, st, x, n, part);
    if (e == cudaSuccess)
        e = launch_pdl(k_amax_final, dim3(1), dim3(1024), 0, st, part, grid, qmax, scale_out);
    count_launches(2);
    return e;
}

} // namespace repro
