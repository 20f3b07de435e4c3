// k_bwd_prefetch.cu -- the backward kernel for shapes whose rows are not
// 16-byte aligned (dY rows with N % 4 != 0, or int8 rows with K % 16 != 0),
// where the tensor-copy-fed default kernel (k_bwd_tma.cu) cannot take its
// tiles.  It computes the same
//   C[i,j] = canon_r( A[r,i] (x) B[r,j] )
// with A from dY (flushed) and B the dequantised int8 operand: chunks of 64
// terms summed left to right from the first term, then the stride-doubling
// pairwise tree over chunk partials, each product rounded and each add
// flushed, never fused (Open-1B review, onedev.kr/papers/92, section "How it
// works").  Only the data movement differs from the default kernel:
//   * 64 x 64 output tile per CTA, 256 threads, 4 x 4 outputs per thread as
//     packed f32x2 pairs (two adjacent rows share one mul.rn.f32x2 and one
//     add.rn.ftz.f32x2; each lane rounds exactly like the scalar form);
//   * B is stored duplicated -- (b_j, b_j, b_j+1, b_j+1) and
//     (b_j+2, b_j+2, b_j+3, b_j+3) -- so the packed operand pairs come
//     straight out of two 16-byte shared loads;
//   * double buffering: chunk c+1 is fetched from global memory into
//     registers (element-wise at ragged edges) while chunk c is computed,
//     then flushed / dequantised into the other shared-memory stage; one
//     barrier per chunk;
//   * all eight tree levels in registers.
#include "bwd_common.cuh"
#include "bwd_tile.cuh"
#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

constexpr int STAGE_FLOATS = 3 * CH * BT;                       // A, B dup lo, B dup hi
constexpr size_t PREFETCH_SMEM = 2 * STAGE_FLOATS * sizeof(float);  // 96 KB

template <bool DW>
__device__ __forceinline__ void fetch_a(float4 (&v)[4], const BwdArgs& a, int64_t i0, int64_t r0,
                                        int valid, int tid)
{
    const bool vec = (a.ldy & 3) == 0;
    if (DW) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = tid + it * 256;
            const int r = e >> 4, f = e & 15;
            const int64_t i = i0 + 4 * f;
            v[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < valid) {
                const float* src = a.dy + (r0 + r) * a.ldy + i;
                if (vec && i + 4 <= a.I) {
                    v[it] = __ldg(reinterpret_cast<const float4*>(src));
                } else {
                    if (i + 0 < a.I) v[it].x = src[0];
                    if (i + 1 < a.I) v[it].y = src[1];
                    if (i + 2 < a.I) v[it].z = src[2];
                    if (i + 3 < a.I) v[it].w = src[3];
                }
            }
        }
    } else {
        const int i = tid & 63;
        const bool row_ok = i0 + i < a.I;
        const float* src = a.dy + (i0 + i) * a.ldy + r0;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = 4 * ((tid >> 6) + 4 * it);
            v[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row_ok) {
                if (vec && r + 4 <= valid) {
                    v[it] = __ldg(reinterpret_cast<const float4*>(src + r));
                } else {
                    if (r + 0 < valid) v[it].x = src[r + 0];
                    if (r + 1 < valid) v[it].y = src[r + 1];
                    if (r + 2 < valid) v[it].z = src[r + 2];
                    if (r + 3 < valid) v[it].w = src[r + 3];
                }
            }
        }
    }
}

template <bool DW>
__device__ __forceinline__ void store_a(float* __restrict__ As, const float4 (&v)[4], int tid)
{
    if (DW) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = tid + it * 256;
            *reinterpret_cast<float4*>(&As[(e >> 4) * BT + 4 * (e & 15)]) = flush4(v[it]);
        }
    } else {
        const int i = tid & 63;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = 4 * ((tid >> 6) + 4 * it);
            As[(r + 0) * BT + i] = flush(v[it].x);
            As[(r + 1) * BT + i] = flush(v[it].y);
            As[(r + 2) * BT + i] = flush(v[it].z);
            As[(r + 3) * BT + i] = flush(v[it].w);
        }
    }
}

// 16 int8 codes of row (tid >> 2), columns 16*(tid & 3) .. +15 of the tile,
// packed little-endian; codes outside the tensor read as 0
__device__ __forceinline__ int4 fetch_b(const BwdArgs& a, int64_t j0, int64_t r0, int valid,
                                        int tid)
{
    const int r = tid >> 2, part = tid & 3;
    const int64_t j = j0 + 16 * part;
    int4 w = make_int4(0, 0, 0, 0);
    if (r < valid) {
        const int8_t* src = a.q + (r0 + r) * a.J + j;
        if ((a.J & 15) == 0 && j + 16 <= a.J) {
            w = __ldg(reinterpret_cast<const int4*>(src));
        } else {
            uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (j + u < a.J)
                    words[u >> 2] |= (uint32_t)(uint8_t)src[u] << (8 * (u & 3));
            w = make_int4((int)words[0], (int)words[1], (int)words[2], (int)words[3]);
        }
    }
    return w;
}

__device__ __forceinline__ void store_b(float* __restrict__ B0, float* __restrict__ B1, int4 w,
                                        float s, int tid)
{
    const int r = tid >> 2, part = tid & 3;
    const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float b0 = dequant((int)(int8_t)(words[u]), s);
        const float b1 = dequant((int)(int8_t)(words[u] >> 8), s);
        const float b2 = dequant((int)(int8_t)(words[u] >> 16), s);
        const float b3 = dequant((int)(int8_t)(words[u] >> 24), s);
        const int col = 4 * (4 * part + u);
        *reinterpret_cast<float4*>(&B0[r * BT + col]) = make_float4(b0, b0, b1, b1);
        *reinterpret_cast<float4*>(&B1[r * BT + col]) = make_float4(b2, b2, b3, b3);
    }
}

// one reduction step r of the chunk for the thread's 4 x 4 outputs, as 8 pairs
// acc[2*... ]: acc[ip*4 + j] = (out(4ty+2ip, 4tx+j), out(4ty+2ip+1, 4tx+j))
template <bool FIRST>
__device__ __forceinline__ void step2(u64 (&acc)[8], const float* __restrict__ Ar,
                                      const float* __restrict__ B0r, const float* __restrict__ B1r)
{
    const ulonglong2 av = *reinterpret_cast<const ulonglong2*>(Ar);
    const ulonglong2 b01 = *reinterpret_cast<const ulonglong2*>(B0r);
    const ulonglong2 b23 = *reinterpret_cast<const ulonglong2*>(B1r);
    const u64 A[2] = {av.x, av.y};
    const u64 B[4] = {b01.x, b01.y, b23.x, b23.y};
#pragma unroll
    for (int ip = 0; ip < 2; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const u64 p = fmul2_rn(A[ip], B[j]);
            acc[ip * 4 + j] = FIRST ? p : fadd2_ftz(acc[ip * 4 + j], p);
        }
}

template <bool DW>
__global__ void __launch_bounds__(256, 1) k_bwd_prefetch(const BwdArgs a)
{
    extern __shared__ __align__(16) float smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);
    const int tx = (warp & 1) * 8 + (lane & 7);
    const int64_t i0 = (int64_t)blockIdx.y * BT, j0 = (int64_t)blockIdx.x * BT;
    const float s = flush(*a.scale);

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));

    u64 S[MAXLVL][8];
    u64 acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        acc[e] = 0ull;
#pragma unroll
    for (int l = 0; l < MAXLVL; ++l)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            S[l][e] = 0ull;

    float4 pa[4];
    int4 pb;
    {
        const int valid = (int)min((int64_t)CH, a.R - cbeg * CH);
        fetch_a<DW>(pa, a, i0, cbeg * CH, valid, tid);
        pb = fetch_b(a, j0, cbeg * CH, valid, tid);
        store_a<DW>(smem, pa, tid);
        store_b(smem + CH * BT, smem + 2 * CH * BT, pb, s, tid);
    }
    __syncthreads();

    for (int64_t c = cbeg; c < cend; ++c) {
        const int stage = (int)((c - cbeg) & 1);
        const float* As = smem + stage * STAGE_FLOATS;
        const float* B0 = As + CH * BT;
        const float* B1 = As + 2 * CH * BT;
        const int64_t r0 = c * CH;
        const int valid = (int)min((int64_t)CH, a.R - r0);
        const bool more = c + 1 < cend;
        if (more) {
            const int nvalid = (int)min((int64_t)CH, a.R - r0 - CH);
            fetch_a<DW>(pa, a, i0, r0 + CH, nvalid, tid);
            pb = fetch_b(a, j0, r0 + CH, nvalid, tid);
        }

        const float* Ar = As + 4 * ty;
        const float* B0r = B0 + 4 * tx;
        const float* B1r = B1 + 4 * tx;
        step2<true>(acc, Ar, B0r, B1r);
        if (valid == CH) {
#pragma unroll 9
            for (int r = 1; r < CH; ++r)
                step2<false>(acc, Ar + r * BT, B0r + r * BT, B1r + r * BT);
        } else {
            for (int r = 1; r < valid; ++r)
                step2<false>(acc, Ar + r * BT, B0r + r * BT, B1r + r * BT);
        }

        if (more) {
            float* Ns = smem + (stage ^ 1) * STAGE_FLOATS;
            store_a<DW>(Ns, pa, tid);
            store_b(Ns + CH * BT, Ns + 2 * CH * BT, pb, s, tid);
        }

        const int cs = (int)(c - cbeg);
        if (more) {
            const int tz = __ffs(~cs) - 1;
#pragma unroll
            for (int t = 0; t < MAXLVL; ++t) {
                if (tz == t) {
#pragma unroll
                    for (int l = 0; l < t; ++l)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            acc[e] = fadd2_ftz(S[l][e], acc[e]);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        S[t][e] = acc[e];
                }
            }
        } else {
#pragma unroll
            for (int l = 0; l < MAXLVL; ++l) {
                if ((cs >> l) & 1) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        acc[e] = fadd2_ftz(S[l][e], acc[e]);
                }
            }
        }
        __syncthreads();
    }

    // unpack: row 4ty + 2ip + h, column 4tx + j is lane h of acc[ip*4 + j]
    float o[4][4];
#pragma unroll
    for (int ip = 0; ip < 2; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float lo, hi;
            unpack2(acc[ip * 4 + j], lo, hi);
            o[2 * ip][j] = lo;
            o[2 * ip + 1][j] = hi;
        }
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
                v[j] = flush(o[i][j]);
            if (vec && col + 4 <= a.J) {
                if (a.accumulate) {
                    const float4 old = *reinterpret_cast<const float4*>(dst);
                    v[0] = fadd_ftz(old.x, v[0]);
                    v[1] = fadd_ftz(old.y, v[1]);
                    v[2] = fadd_ftz(old.z, v[2]);
                    v[3] = fadd_ftz(old.w, v[3]);
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
                    base[row * a.J + col] = o[i][j];
            }
        }
    }
}

} // namespace

template <bool DW>
cudaError_t launch_bwd_prefetch(const BwdArgs& a, cudaStream_t st)
{
    // opt in to 96 KB of dynamic shared memory (on the current device)
    cudaError_t e = cudaFuncSetAttribute(k_bwd_prefetch<DW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)PREFETCH_SMEM);
    if (e != cudaSuccess)
        return e;
    k_bwd_prefetch<DW><<<dim3((unsigned)cdiv(a.J, BT), (unsigned)cdiv(a.I, BT), (unsigned)a.nseg),
                         256, PREFETCH_SMEM, st>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_bwd_prefetch<false>(const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_prefetch<true>(const BwdArgs&, cudaStream_t);

} // namespace repro
