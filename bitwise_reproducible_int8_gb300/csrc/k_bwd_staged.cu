// k_bwd_staged.cu -- backward kernel variants 0-5, which stage and transform
// their operands inside every CTA (k_bwd.cu dispatches; variants 6-8 are in
// k_bwd_ws.cu and k_bwd_tma.cu).  All compute
//   C[i,j] = canon_r( A[r,i] (x) B[r,j] )
// with A from dY (flushed) and B the dequantised int8 operand, chunks of 64
// terms left to right from the first term and the stride-doubling pairwise
// tree over chunk partials (Open-1B review, onedev.kr/papers/92, section "How
// it works"); they differ only in how operands reach the products:
//   0 k_bwd   64 x 64 tile, 4 x 4 scalar outputs a thread, two barriers a chunk;
//   1 k_bwd2  4 x 4 packed f32x2 pairs (B duplicated in shared memory),
//             register-prefetched chunk loads; any row alignment;
//   2 k_bwd3  cp.async raw staging + transform pass, tree levels 4-7 in
//             shared memory;
//   3 k_bwd4  128 x 64 tile, 8 x 4 outputs a thread (B pairs by register move);
//   4 k_bwd5  as 3, double-buffered, tree levels 2-7 in tensor memory;
//   5 k_bwd6  twelve warps, 192 x 64 tile.
// 2-5 need 16-byte-aligned rows (dY rows N % 4 == 0, int8 rows J % 16 == 0).
#include <float.h>

#include "bwd_common.cuh"
#include "bwd_tile.cuh"
#include "common.cuh"
#include "internal.h"

namespace repro {
namespace {

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

// ---------------------------------------------------------------------------
// Pipelined variant (default).  Same tile, same per-output order, same tree
// stack; three changes that alter no rounding:
//   * packed arithmetic: two adjacent output rows share one mul.rn.f32x2 and
//     one add.rn.ftz.f32x2 (each lane rounds exactly like the scalar form),
//     halving the issue slots spent on arithmetic;
//   * B is stored duplicated -- (b_j, b_j, b_j+1, b_j+1) and
//     (b_j+2, b_j+2, b_j+3, b_j+3) -- so the packed operand pairs come
//     straight out of two 16-byte shared loads;
//   * double buffering: chunk c+1 is fetched from global memory into
//     registers while chunk c is computed, then dequantised/flushed into the
//     other shared-memory stage; one barrier per chunk.
// ---------------------------------------------------------------------------

constexpr int STAGE_FLOATS = 3 * CH * BT;                       // A, B dup lo, B dup hi
constexpr size_t BWD2_SMEM = 2 * STAGE_FLOATS * sizeof(float);  // 96 KB

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
__global__ void __launch_bounds__(256, 1) k_bwd2(const BwdArgs a)
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

// ---------------------------------------------------------------------------
// Staged variant (default for aligned shapes: rows of dY and of the int8
// operand start on 16-byte boundaries).  Same tile, per-output order, packed
// arithmetic and tree as k_bwd2; the data movement changes:
//   * the next chunk's raw bytes are copied global -> shared with cp.async
//     (16-byte pieces, zero-filled outside the tensor) while the current chunk
//     is computed, so no registers wait on global memory;
//   * after a barrier, a transform pass turns the raw chunk into the compute
//     layout: dY flushed (and transposed for dX, through a raw layout padded
//     to 68 floats per row so the transposing reads are conflict-free), the
//     int8 operand dequantised into the duplicated pair layout;
//   * stack levels 0-3 stay in registers, levels 4-7 (merged at most once per
//     16 chunks) live in a per-thread slice of shared memory, which frees 64
//     registers for a one-step-ahead prefetch of the shared-memory fragments.
// ---------------------------------------------------------------------------

constexpr int RAW_A_LD = 68;                                   // floats per raw A row
constexpr int RAW_A_BYTES = CH * RAW_A_LD * 4;                 // 17408
constexpr int RAW_B_BYTES = CH * BT;                           // 4096 int8
constexpr int COMP_BYTES = 3 * CH * BT * 4;                    // 49152
constexpr int REG_LVL = 4;                                     // levels kept in registers
constexpr int EXT_BYTES = (MAXLVL - REG_LVL) * 8 * 256 * 8;    // 65536
constexpr size_t BWD3_SMEM = (size_t)RAW_A_BYTES + RAW_B_BYTES + COMP_BYTES + EXT_BYTES;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// raw copy of chunk r0: A as 64 rows x 64 floats (DW: rows = reduction index,
// columns = i; DX: rows = i, columns = reduction index), B as 64 rows x 64 int8
template <bool DW>
__device__ __forceinline__ void issue_raw(float* __restrict__ rawA, int8_t* __restrict__ rawB,
                                          const BwdArgs& a, int64_t i0, int64_t j0, int64_t r0,
                                          int valid, int tid)
{
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int p = tid + it * 256;
        const int row = p >> 4, f = p & 15;
        const float* src;
        bool ok;
        if (DW) {
            src = a.dy + (r0 + row) * a.ldy + i0 + 4 * f;
            ok = row < valid && i0 + 4 * f < a.I;
        } else {
            src = a.dy + (i0 + row) * a.ldy + r0 + 4 * f;
            ok = i0 + row < a.I && 4 * f < valid;
        }
        cp_async16(rawA + row * RAW_A_LD + 4 * f, ok ? src : a.dy, ok ? 16u : 0u);
    }
    {
        const int row = tid >> 2, part = tid & 3;
        const bool ok = row < valid && j0 + 16 * part < a.J;
        const int8_t* src = ok ? a.q + (r0 + row) * a.J + j0 + 16 * part : a.q;
        cp_async16(rawB + row * BT + 16 * part, src, ok ? 16u : 0u);
    }
    cp_async_commit();
}

template <bool DW>
__device__ __forceinline__ void transform(float* __restrict__ As, float* __restrict__ B0,
                                          float* __restrict__ B1, const float* __restrict__ rawA,
                                          const int8_t* __restrict__ rawB, float s, int tid)
{
    if (DW) {
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = tid + it * 256;
            const int r = e >> 4, f = e & 15;
            const float4 v = *reinterpret_cast<const float4*>(rawA + r * RAW_A_LD + 4 * f);
            *reinterpret_cast<float4*>(&As[r * BT + 4 * f]) = flush4(v);
        }
    } else {
        const int i = tid & 63;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int f = (tid >> 6) + 4 * it;
            const float4 v = *reinterpret_cast<const float4*>(rawA + i * RAW_A_LD + 4 * f);
            As[(4 * f + 0) * BT + i] = flush(v.x);
            As[(4 * f + 1) * BT + i] = flush(v.y);
            As[(4 * f + 2) * BT + i] = flush(v.z);
            As[(4 * f + 3) * BT + i] = flush(v.w);
        }
    }
    const int4 w = *reinterpret_cast<const int4*>(rawB + (tid >> 2) * BT + 16 * (tid & 3));
    store_b(B0, B1, w, s, tid);
}

template <bool DW>
__global__ void __launch_bounds__(256, 1) k_bwd3(const BwdArgs a)
{
    extern __shared__ __align__(16) uint8_t smem3[];
    float* rawA = reinterpret_cast<float*>(smem3);
    int8_t* rawB = reinterpret_cast<int8_t*>(smem3 + RAW_A_BYTES);
    float* As = reinterpret_cast<float*>(smem3 + RAW_A_BYTES + RAW_B_BYTES);
    float* B0 = As + CH * BT;
    float* B1 = As + 2 * CH * BT;
    u64* ext = reinterpret_cast<u64*>(smem3 + RAW_A_BYTES + RAW_B_BYTES + COMP_BYTES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);
    const int tx = (warp & 1) * 8 + (lane & 7);
    const int64_t i0 = (int64_t)blockIdx.y * BT, j0 = (int64_t)blockIdx.x * BT;
    const float s = flush(*a.scale);

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));

    // level l >= REG_LVL, pair e of this thread
    auto X = [&](int l, int e) -> u64& { return ext[((l - REG_LVL) * 8 + e) * 256 + tid]; };

    u64 S[REG_LVL][8];
    u64 acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        acc[e] = 0ull;
#pragma unroll
    for (int l = 0; l < REG_LVL; ++l)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            S[l][e] = 0ull;

    issue_raw<DW>(rawA, rawB, a, i0, j0, cbeg * CH, (int)min((int64_t)CH, a.R - cbeg * CH), tid);
    cp_async_wait_all();
    __syncthreads();
    transform<DW>(As, B0, B1, rawA, rawB, s, tid);
    __syncthreads();

    const float* Ar = As + 4 * ty;
    const float* B0r = B0 + 4 * tx;
    const float* B1r = B1 + 4 * tx;

    for (int64_t c = cbeg; c < cend; ++c) {
        const int64_t r0 = c * CH;
        const int valid = (int)min((int64_t)CH, a.R - r0);
        const bool more = c + 1 < cend;
        if (more)
            issue_raw<DW>(rawA, rawB, a, i0, j0, r0 + CH, (int)min((int64_t)CH, a.R - r0 - CH),
                          tid);

        // the chunk, with the next step's fragments loaded one step ahead
        ulonglong2 av = *reinterpret_cast<const ulonglong2*>(Ar);
        ulonglong2 b01 = *reinterpret_cast<const ulonglong2*>(B0r);
        ulonglong2 b23 = *reinterpret_cast<const ulonglong2*>(B1r);
        {
            const u64 A_[2] = {av.x, av.y};
            const u64 B_[4] = {b01.x, b01.y, b23.x, b23.y};
            if (valid > 1) {
                av = *reinterpret_cast<const ulonglong2*>(Ar + BT);
                b01 = *reinterpret_cast<const ulonglong2*>(B0r + BT);
                b23 = *reinterpret_cast<const ulonglong2*>(B1r + BT);
            }
#pragma unroll
            for (int ip = 0; ip < 2; ++ip)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    acc[ip * 4 + j] = fmul2_rn(A_[ip], B_[j]);
        }
        if (valid == CH) {
#pragma unroll 7
            for (int r = 1; r < CH; ++r) {
                const u64 A_[2] = {av.x, av.y};
                const u64 B_[4] = {b01.x, b01.y, b23.x, b23.y};
                const int rn = r + 1 < CH ? r + 1 : r;
                av = *reinterpret_cast<const ulonglong2*>(Ar + rn * BT);
                b01 = *reinterpret_cast<const ulonglong2*>(B0r + rn * BT);
                b23 = *reinterpret_cast<const ulonglong2*>(B1r + rn * BT);
#pragma unroll
                for (int ip = 0; ip < 2; ++ip)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        acc[ip * 4 + j] = fadd2_ftz(acc[ip * 4 + j], fmul2_rn(A_[ip], B_[j]));
            }
        } else {
            for (int r = 1; r < valid; ++r) {
                const u64 A_[2] = {av.x, av.y};
                const u64 B_[4] = {b01.x, b01.y, b23.x, b23.y};
                const int rn = r + 1 < valid ? r + 1 : r;
                av = *reinterpret_cast<const ulonglong2*>(Ar + rn * BT);
                b01 = *reinterpret_cast<const ulonglong2*>(B0r + rn * BT);
                b23 = *reinterpret_cast<const ulonglong2*>(B1r + rn * BT);
#pragma unroll
                for (int ip = 0; ip < 2; ++ip)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        acc[ip * 4 + j] = fadd2_ftz(acc[ip * 4 + j], fmul2_rn(A_[ip], B_[j]));
            }
        }

        // tree: push (merge the levels named by the trailing ones of cs) or,
        // after the segment's last chunk, fold every occupied level
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
                            acc[e] = fadd2_ftz(l < REG_LVL ? S[l < REG_LVL ? l : 0][e] : X(l, e), acc[e]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (t < REG_LVL)
                            S[t < REG_LVL ? t : 0][e] = acc[e];
                        else
                            X(t, e) = acc[e];
                    }
                }
            }
        } else {
#pragma unroll
            for (int l = 0; l < MAXLVL; ++l) {
                if ((cs >> l) & 1) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        acc[e] = fadd2_ftz(l < REG_LVL ? S[l < REG_LVL ? l : 0][e] : X(l, e), acc[e]);
                }
            }
        }

        if (more) {
            cp_async_wait_all();
            __syncthreads();            // comp reads done, raw chunk visible
            transform<DW>(As, B0, B1, rawA, rawB, s, tid);
            __syncthreads();            // comp ready
        }
    }

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
    if (a.nseg == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = i0 + 4 * ty + i;
            if (row >= a.I)
                continue;
            const int64_t col = j0 + 4 * tx;
            if (col >= a.J)
                continue;
            float* dst = a.out + row * a.J + col;     // J % 16 == 0: whole float4 inside
            float v0 = flush(o[i][0]), v1 = flush(o[i][1]), v2 = flush(o[i][2]), v3 = flush(o[i][3]);
            if (a.accumulate) {
                const float4 old = *reinterpret_cast<const float4*>(dst);
                v0 = fadd_ftz(old.x, v0);
                v1 = fadd_ftz(old.y, v1);
                v2 = fadd_ftz(old.z, v2);
                v3 = fadd_ftz(old.w, v3);
            }
            *reinterpret_cast<float4*>(dst) = make_float4(v0, v1, v2, v3);
        }
    } else {
        float* base = a.ws + (int64_t)blockIdx.z * a.I * a.J;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = i0 + 4 * ty + i;
            const int64_t col = j0 + 4 * tx;
            if (row < a.I && col < a.J)
                *reinterpret_cast<float4*>(base + row * a.J + col) =
                    make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
        }
    }
}

// ---------------------------------------------------------------------------
// Wide-tile variant (default for aligned shapes).  Shared-memory bandwidth
// bounds the 4 x 4 thread tile: every 16-byte shared load costs one wavefront
// per quarter-warp however many lanes share its address, so the cost is one
// wavefront per warp per float a thread loads.  A thread of this kernel owns
// 8 x 4 outputs (0.375 loaded floats per output instead of 0.75), and builds
// the packed (b, b) pairs with a register move instead of a duplicated
// shared-memory copy.  CTA tile 128 (i) x 64 (j), 256 threads; cp.async
// staging and transform pass as in k_bwd3; tree levels 0-3 in registers,
// 4-7 in 128 KB of per-thread shared memory.  Same per-output arithmetic.
// ---------------------------------------------------------------------------

constexpr int BI4 = BWD_WIDE_ROWS;                            // tile rows (i)
constexpr int RAW4_A_BYTES = 128 * 68 * 4;                    // 34816 (DX; DW needs 64 x 132)
constexpr int RAW4_B_BYTES = CH * BT;                         // 4096
constexpr int COMP4_A_BYTES = CH * BI4 * 4;                   // 32768
constexpr int COMP4_B_BYTES = CH * BT * 4;                    // 16384
constexpr int EXT4_BYTES = (MAXLVL - REG_LVL) * 16 * 256 * 8; // 131072
constexpr size_t BWD4_SMEM =
    (size_t)RAW4_A_BYTES + RAW4_B_BYTES + COMP4_A_BYTES + COMP4_B_BYTES + EXT4_BYTES;

template <bool DW>
__device__ __forceinline__ void issue_raw4(float* __restrict__ rawA, int8_t* __restrict__ rawB,
                                           const BwdArgs& a, int64_t i0, int64_t j0, int64_t r0,
                                           int valid, int tid)
{
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int p = tid + it * 256;
        const float* src;
        float* dst;
        bool ok;
        if (DW) {   // 64 rows (reduction) x 128 floats (i), row pitch 132
            const int row = p >> 5, f = p & 31;
            src = a.dy + (r0 + row) * a.ldy + i0 + 4 * f;
            ok = row < valid && i0 + 4 * f < a.I;
            dst = rawA + row * 132 + 4 * f;
        } else {    // 128 rows (i) x 64 floats (reduction), row pitch 68
            const int row = p >> 4, f = p & 15;
            src = a.dy + (i0 + row) * a.ldy + r0 + 4 * f;
            ok = i0 + row < a.I && 4 * f < valid;
            dst = rawA + row * 68 + 4 * f;
        }
        cp_async16(dst, ok ? src : a.dy, ok ? 16u : 0u);
    }
    {
        const int row = tid >> 2, part = tid & 3;
        const bool ok = row < valid && j0 + 16 * part < a.J;
        const int8_t* src = ok ? a.q + (r0 + row) * a.J + j0 + 16 * part : a.q;
        cp_async16(rawB + row * BT + 16 * part, src, ok ? 16u : 0u);
    }
    cp_async_commit();
}

template <bool DW>
__device__ __forceinline__ void transform4(float* __restrict__ As, float* __restrict__ Bs,
                                           const float* __restrict__ rawA,
                                           const int8_t* __restrict__ rawB, float s, int tid)
{
    if (DW) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int e = tid + it * 256;
            const int r = e >> 5, f = e & 31;
            const float4 v = *reinterpret_cast<const float4*>(rawA + r * 132 + 4 * f);
            *reinterpret_cast<float4*>(&As[r * BI4 + 4 * f]) = flush4(v);
        }
    } else {
        const int i = tid & 127;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int f = (tid >> 7) + 2 * it;
            const float4 v = *reinterpret_cast<const float4*>(rawA + i * 68 + 4 * f);
            As[(4 * f + 0) * BI4 + i] = flush(v.x);
            As[(4 * f + 1) * BI4 + i] = flush(v.y);
            As[(4 * f + 2) * BI4 + i] = flush(v.z);
            As[(4 * f + 3) * BI4 + i] = flush(v.w);
        }
    }
    const int row = tid >> 2, part = tid & 3;
    const int4 w = *reinterpret_cast<const int4*>(rawB + row * BT + 16 * part);
    const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
        *reinterpret_cast<float4*>(&Bs[row * BT + 16 * part + 4 * u]) =
            make_float4(dequant((int)(int8_t)(words[u]), s), dequant((int)(int8_t)(words[u] >> 8), s),
                        dequant((int)(int8_t)(words[u] >> 16), s),
                        dequant((int)(int8_t)(words[u] >> 24), s));
}

template <bool DW>
__global__ void __launch_bounds__(256, 1) k_bwd4(const BwdArgs a)
{
    extern __shared__ __align__(16) uint8_t smem4[];
    float* rawA = reinterpret_cast<float*>(smem4);
    int8_t* rawB = reinterpret_cast<int8_t*>(smem4 + RAW4_A_BYTES);
    float* As = reinterpret_cast<float*>(smem4 + RAW4_A_BYTES + RAW4_B_BYTES);
    float* Bs = reinterpret_cast<float*>(smem4 + RAW4_A_BYTES + RAW4_B_BYTES + COMP4_A_BYTES);
    u64* ext = reinterpret_cast<u64*>(smem4 + RAW4_A_BYTES + RAW4_B_BYTES + COMP4_A_BYTES +
                                      COMP4_B_BYTES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);   // rows 8ty .. 8ty+7
    const int tx = (warp & 1) * 8 + (lane & 7);     // cols 4tx .. 4tx+3
    const int64_t i0 = (int64_t)blockIdx.y * BI4, j0 = (int64_t)blockIdx.x * BT;
    const float s = flush(*a.scale);

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));

    auto X = [&](int l, int e) -> u64& { return ext[((l - REG_LVL) * 16 + e) * 256 + tid]; };

    u64 S[REG_LVL][16];
    u64 acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        acc[e] = 0ull;
#pragma unroll
    for (int l = 0; l < REG_LVL; ++l)
#pragma unroll
        for (int e = 0; e < 16; ++e)
            S[l][e] = 0ull;

    issue_raw4<DW>(rawA, rawB, a, i0, j0, cbeg * CH, (int)min((int64_t)CH, a.R - cbeg * CH), tid);
    cp_async_wait_all();
    __syncthreads();
    transform4<DW>(As, Bs, rawA, rawB, s, tid);
    __syncthreads();

    const float* Ar = As + 8 * ty;
    const float* Br = Bs + 4 * tx;

    for (int64_t c = cbeg; c < cend; ++c) {
        const int64_t r0 = c * CH;
        const int valid = (int)min((int64_t)CH, a.R - r0);
        const bool more = c + 1 < cend;
        if (more)
            issue_raw4<DW>(rawA, rawB, a, i0, j0, r0 + CH,
                           (int)min((int64_t)CH, a.R - r0 - CH), tid);

        ulonglong2 a03 = *reinterpret_cast<const ulonglong2*>(Ar);
        ulonglong2 a47 = *reinterpret_cast<const ulonglong2*>(Ar + 4);
        float4 b = *reinterpret_cast<const float4*>(Br);
        {
            const ulonglong2 c03 = a03, c47 = a47;
            const float4 cb = b;
            if (valid > 1) {
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + BI4);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + BI4 + 4);
                b = *reinterpret_cast<const float4*>(Br + BT);
            }
            step<true>(acc, c03, c47, cb);
        }
        if (valid == CH) {
#pragma unroll 7
            for (int r = 1; r < CH; ++r) {
                const ulonglong2 c03 = a03, c47 = a47;
                const float4 cb = b;
                const int rn = r + 1 < CH ? r + 1 : r;
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4 + 4);
                b = *reinterpret_cast<const float4*>(Br + rn * BT);
                step<false>(acc, c03, c47, cb);
            }
        } else {
            for (int r = 1; r < valid; ++r) {
                const ulonglong2 c03 = a03, c47 = a47;
                const float4 cb = b;
                const int rn = r + 1 < valid ? r + 1 : r;
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4 + 4);
                b = *reinterpret_cast<const float4*>(Br + rn * BT);
                step<false>(acc, c03, c47, cb);
            }
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
                        for (int e = 0; e < 16; ++e)
                            acc[e] = fadd2_ftz(l < REG_LVL ? S[l < REG_LVL ? l : 0][e] : X(l, e), acc[e]);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (t < REG_LVL)
                            S[t < REG_LVL ? t : 0][e] = acc[e];
                        else
                            X(t, e) = acc[e];
                    }
                }
            }
        } else {
#pragma unroll
            for (int l = 0; l < MAXLVL; ++l) {
                if ((cs >> l) & 1) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        acc[e] = fadd2_ftz(l < REG_LVL ? S[l < REG_LVL ? l : 0][e] : X(l, e), acc[e]);
                }
            }
        }

        if (more) {
            cp_async_wait_all();
            __syncthreads();
            transform4<DW>(As, Bs, rawA, rawB, s, tid);
            __syncthreads();
        }
    }

    // row 8ty + 2ip + h, column 4tx + j is lane h of acc[ip*4 + j]
    const int64_t col = j0 + 4 * tx;
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = i0 + 8 * ty + 2 * ip + h;
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo, hi;
                unpack2(acc[ip * 4 + j], lo, hi);
                o[j] = h ? hi : lo;
            }
            if (row >= a.I || col >= a.J)
                continue;
            if (a.nseg == 1) {
                float* dst = a.out + row * a.J + col;    // J % 16 == 0: whole float4 inside
                float v0 = flush(o[0]), v1 = flush(o[1]), v2 = flush(o[2]), v3 = flush(o[3]);
                if (a.accumulate) {
                    const float4 old = *reinterpret_cast<const float4*>(dst);
                    v0 = fadd_ftz(old.x, v0);
                    v1 = fadd_ftz(old.y, v1);
                    v2 = fadd_ftz(old.z, v2);
                    v3 = fadd_ftz(old.w, v3);
                }
                *reinterpret_cast<float4*>(dst) = make_float4(v0, v1, v2, v3);
            } else {
                float* base = a.ws + (int64_t)blockIdx.z * a.I * a.J;
                *reinterpret_cast<float4*>(base + row * a.J + col) = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Tensor-memory variant.  k_bwd4's tile and arithmetic, with the resources the
// backward leaves idle put to work:
//   * tree levels 2-7 live in tensor memory (unused by this kernel): each
//     thread owns one TMEM lane (32*(warp%4) + lane) and a 256-column slice
//     ((warp/4)*256), one 32-column block per level, written and read with
//     tcgen05.st / tcgen05.ld 32x32b.x32 at chunk boundaries only;
//   * the shared memory this frees double-buffers both the raw (cp.async) and
//     the compute stages, so each chunk needs one barrier: after it, a thread
//     transforms chunk c+1 into the other compute buffer and then computes
//     chunk c, overlapping other warps' transforms with its arithmetic;
//   * the registers it frees let each reduction step issue its 16 products
//     before its 16 additions.
// The CTA allocates all 512 TMEM columns (one CTA per SM) and frees them
// before it exits.
// ---------------------------------------------------------------------------

constexpr int RAW5_STAGE = RAW4_A_BYTES + RAW4_B_BYTES;          // 38912
constexpr int COMP5_STAGE = COMP4_A_BYTES + COMP4_B_BYTES;       // 49152
constexpr size_t BWD5_SMEM = 2 * (size_t)RAW5_STAGE + 2 * (size_t)COMP5_STAGE + 16;
constexpr int REG5 = 2;                                          // levels in registers

__device__ __forceinline__ void tmem_ld32_u64(uint32_t taddr, u64 (&v)[16])
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
    for (int e = 0; e < 16; ++e)
        v[e] = (u64)w[2 * e] | ((u64)w[2 * e + 1] << 32);
}

// 16-column halves (8 pairs) of a level, to keep the transient register peak low
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const u64* v)
{
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        w[2 * e] = (uint32_t)(v[e] & 0xffffffffull);
        w[2 * e + 1] = (uint32_t)(v[e] >> 32);
    }
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// acc[e] <- level[e] (+) acc[e] for the 8 pairs of one half
__device__ __forceinline__ void tmem_fold16(uint32_t taddr, u64* acc)
{
    uint32_t w[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
          "=r"(w[7]), "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]),
          "=r"(w[14]), "=r"(w[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 8; ++e)
        acc[e] = fadd2_ftz((u64)w[2 * e] | ((u64)w[2 * e + 1] << 32), acc[e]);
}

template <bool FIRST>
__device__ __forceinline__ void step5(u64 (&acc)[16], const ulonglong2& a03, const ulonglong2& a47,
                                      const float4& b)
{
    const u64 P[4] = {a03.x, a03.y, a47.x, a47.y};
    const u64 D[4] = {pack2(b.x, b.x), pack2(b.y, b.y), pack2(b.z, b.z), pack2(b.w, b.w)};
    u64 prod[16];
#pragma unroll
    for (int ip = 0; ip < 4; ++ip)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            prod[ip * 4 + j] = fmul2_rn(P[ip], D[j]);
#pragma unroll
    for (int e = 0; e < 16; ++e)
        acc[e] = FIRST ? prod[e] : fadd2_ftz(acc[e], prod[e]);
}

template <bool DW>
__global__ void __launch_bounds__(256, 1) k_bwd5(const BwdArgs a)
{
    extern __shared__ __align__(16) uint8_t smem5[];
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem5 + 2 * RAW5_STAGE + 2 * COMP5_STAGE);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);
    const int tx = (warp & 1) * 8 + (lane & 7);
    const int64_t i0 = (int64_t)blockIdx.y * BI4, j0 = (int64_t)blockIdx.x * BT;
    const float s = flush(*a.scale);

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // this thread's slice: lane 32*(warp%4)+lane, columns (warp/4)*256 + 32*(level-2)
    const uint32_t tbase = *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));

    auto rawA = [&](int b) { return reinterpret_cast<float*>(smem5 + b * RAW5_STAGE); };
    auto rawB = [&](int b) { return reinterpret_cast<int8_t*>(smem5 + b * RAW5_STAGE + RAW4_A_BYTES); };
    auto compA = [&](int b) { return reinterpret_cast<float*>(smem5 + 2 * RAW5_STAGE + b * COMP5_STAGE); };
    auto compB = [&](int b) {
        return reinterpret_cast<float*>(smem5 + 2 * RAW5_STAGE + b * COMP5_STAGE + COMP4_A_BYTES);
    };
    auto valid_of = [&](int64_t c) { return (int)min((int64_t)CH, a.R - c * CH); };

    u64 S[REG5][16];
    u64 acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        acc[e] = 0ull;
#pragma unroll
    for (int l = 0; l < REG5; ++l)
#pragma unroll
        for (int e = 0; e < 16; ++e)
            S[l][e] = 0ull;

    // prologue: chunk cbeg transformed into compute buffer 0; chunk cbeg+1's
    // raw copy in flight into raw buffer 1
    issue_raw4<DW>(rawA(0), rawB(0), a, i0, j0, cbeg * CH, valid_of(cbeg), tid);
    if (cbeg + 1 < cend)
        issue_raw4<DW>(rawA(1), rawB(1), a, i0, j0, (cbeg + 1) * CH, valid_of(cbeg + 1), tid);
    if (cbeg + 1 < cend)
        asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
        cp_async_wait_all();
    __syncthreads();
    transform4<DW>(compA(0), compB(0), rawA(0), rawB(0), s, tid);

    for (int64_t c = cbeg; c < cend; ++c) {
        const int cs = (int)(c - cbeg);
        const int buf = cs & 1;
        const bool more = c + 1 < cend;
        // raw(c+1) has landed (this thread's pieces); after the barrier every
        // thread's pieces are visible, compute buffer `buf` is complete, and
        // every thread is done with raw buffer `buf` and compute buffer buf^1
        cp_async_wait_all();
        __syncthreads();
        if (c + 2 < cend)
            issue_raw4<DW>(rawA(buf), rawB(buf), a, i0, j0, (c + 2) * CH, valid_of(c + 2), tid);
        if (more)
            transform4<DW>(compA(buf ^ 1), compB(buf ^ 1), rawA(buf ^ 1), rawB(buf ^ 1), s, tid);

        const int valid = valid_of(c);
        const float* Ar = compA(buf) + 8 * ty;
        const float* Br = compB(buf) + 4 * tx;
        ulonglong2 a03 = *reinterpret_cast<const ulonglong2*>(Ar);
        ulonglong2 a47 = *reinterpret_cast<const ulonglong2*>(Ar + 4);
        float4 b = *reinterpret_cast<const float4*>(Br);
        {
            const ulonglong2 c03 = a03, c47 = a47;
            const float4 cb = b;
            if (valid > 1) {
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + BI4);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + BI4 + 4);
                b = *reinterpret_cast<const float4*>(Br + BT);
            }
            step5<true>(acc, c03, c47, cb);
        }
        if (valid == CH) {
#pragma unroll 7
            for (int r = 1; r < CH; ++r) {
                const ulonglong2 c03 = a03, c47 = a47;
                const float4 cb = b;
                const int rn = r + 1 < CH ? r + 1 : r;
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4 + 4);
                b = *reinterpret_cast<const float4*>(Br + rn * BT);
                step5<false>(acc, c03, c47, cb);
            }
        } else {
            for (int r = 1; r < valid; ++r) {
                const ulonglong2 c03 = a03, c47 = a47;
                const float4 cb = b;
                const int rn = r + 1 < valid ? r + 1 : r;
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI4 + 4);
                b = *reinterpret_cast<const float4*>(Br + rn * BT);
                step5<false>(acc, c03, c47, cb);
            }
        }

        // tree over chunk partials; levels >= REG5 go through tensor memory
        if (more) {
            const int tz = __ffs(~cs) - 1;
#pragma unroll
            for (int t = 0; t < MAXLVL; ++t) {
                if (tz == t) {
#pragma unroll
                    for (int l = 0; l < t; ++l) {
                        if (l < REG5) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                acc[e] = fadd2_ftz(S[l < REG5 ? l : 0][e], acc[e]);
                        } else {
                            u64 v[16];
                            tmem_ld32_u64(tbase + (uint32_t)(32 * (l - REG5)), v);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                acc[e] = fadd2_ftz(v[e], acc[e]);
                        }
                    }
                    if (t < REG5) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            S[t < REG5 ? t : 0][e] = acc[e];
                    } else {
                        tmem_st32(tbase + (uint32_t)(32 * (t - REG5)), acc);
                    }
                }
            }
        } else {
#pragma unroll
            for (int l = 0; l < MAXLVL; ++l) {
                if ((cs >> l) & 1) {
                    if (l < REG5) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            acc[e] = fadd2_ftz(S[l < REG5 ? l : 0][e], acc[e]);
                    } else {
                        u64 v[16];
                        tmem_ld32_u64(tbase + (uint32_t)(32 * (l - REG5)), v);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            acc[e] = fadd2_ftz(v[e], acc[e]);
                    }
                }
            }
        }
    }

    const int64_t col = j0 + 4 * tx;
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = i0 + 8 * ty + 2 * ip + h;
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo, hi;
                unpack2(acc[ip * 4 + j], lo, hi);
                o[j] = h ? hi : lo;
            }
            if (row >= a.I || col >= a.J)
                continue;
            if (a.nseg == 1) {
                float* dst = a.out + row * a.J + col;
                float v0 = flush(o[0]), v1 = flush(o[1]), v2 = flush(o[2]), v3 = flush(o[3]);
                if (a.accumulate) {
                    const float4 old = *reinterpret_cast<const float4*>(dst);
                    v0 = fadd_ftz(old.x, v0);
                    v1 = fadd_ftz(old.y, v1);
                    v2 = fadd_ftz(old.z, v2);
                    v3 = fadd_ftz(old.w, v3);
                }
                *reinterpret_cast<float4*>(dst) = make_float4(v0, v1, v2, v3);
            } else {
                float* base = a.ws + (int64_t)blockIdx.z * a.I * a.J;
                *reinterpret_cast<float4*>(base + row * a.J + col) = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(*tmem_slot)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Twelve-warp variant: k_bwd4's 8 x 4 thread tile on 384 threads (CTA tile
// 192 x 64) so that three warps per SM sub-partition hide each other's
// fixed-latency waits.  To fit 170 registers per thread, tree levels 0-1 stay
// in registers, levels 2-6 live in tensor memory (warp w: lanes 32*(w%4)..,
// a 160-column slice at (w/4)*160) and level 7 in shared memory.  Staging as
// in k_bwd4 (cp.async raw copy, transform pass, two barriers per chunk).
// ---------------------------------------------------------------------------

constexpr int NT6 = 384;
constexpr int BI6 = BWD_WIDE12_ROWS;
constexpr int RAW6_A_BYTES = BI6 * 68 * 4;                     // 52224 (DX; DW: 64 x 196)
constexpr int RAW6_B_BYTES = CH * BT;                          // 4096
constexpr int COMP6_A_BYTES = CH * BI6 * 4;                    // 49152
constexpr int COMP6_B_BYTES = CH * BT * 4;                     // 16384
constexpr int EXT6_BYTES = 16 * NT6 * 8;                       // 49152: level 7
constexpr size_t BWD6_SMEM = (size_t)RAW6_A_BYTES + RAW6_B_BYTES + COMP6_A_BYTES +
                             COMP6_B_BYTES + EXT6_BYTES + 16;

template <bool DW>
__device__ __forceinline__ void issue_raw6(float* __restrict__ rawA, int8_t* __restrict__ rawB,
                                           const BwdArgs& a, int64_t i0, int64_t j0, int64_t r0,
                                           int valid, int tid)
{
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int p = tid + it * NT6;
        const float* src;
        float* dst;
        bool ok;
        if (DW) {   // 64 rows (reduction) x 192 floats (i), pitch 196
            const int row = p / 48, f = p % 48;
            src = a.dy + (r0 + row) * a.ldy + i0 + 4 * f;
            ok = row < valid && i0 + 4 * f < a.I;
            dst = rawA + row * 196 + 4 * f;
        } else {    // 192 rows (i) x 64 floats (reduction), pitch 68
            const int row = p >> 4, f = p & 15;
            src = a.dy + (i0 + row) * a.ldy + r0 + 4 * f;
            ok = i0 + row < a.I && 4 * f < valid;
            dst = rawA + row * 68 + 4 * f;
        }
        cp_async16(dst, ok ? src : a.dy, ok ? 16u : 0u);
    }
    if (tid < 256) {
        const int row = tid >> 2, part = tid & 3;
        const bool ok = row < valid && j0 + 16 * part < a.J;
        const int8_t* src = ok ? a.q + (r0 + row) * a.J + j0 + 16 * part : a.q;
        cp_async16(rawB + row * BT + 16 * part, src, ok ? 16u : 0u);
    }
    cp_async_commit();
}

template <bool DW>
__device__ __forceinline__ void transform6(float* __restrict__ As, float* __restrict__ Bs,
                                           const float* __restrict__ rawA,
                                           const int8_t* __restrict__ rawB, float s, int tid)
{
    if (DW) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int e = tid + it * NT6;
            const int r = e / 48, f = e % 48;
            const float4 v = *reinterpret_cast<const float4*>(rawA + r * 196 + 4 * f);
            *reinterpret_cast<float4*>(&As[r * BI6 + 4 * f]) = flush4(v);
        }
    } else {
        const int i = tid % BI6, fg = tid / BI6;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int f = fg + 2 * it;
            const float4 v = *reinterpret_cast<const float4*>(rawA + i * 68 + 4 * f);
            As[(4 * f + 0) * BI6 + i] = flush(v.x);
            As[(4 * f + 1) * BI6 + i] = flush(v.y);
            As[(4 * f + 2) * BI6 + i] = flush(v.z);
            As[(4 * f + 3) * BI6 + i] = flush(v.w);
        }
    }
    if (tid < 256) {
        const int row = tid >> 2, part = tid & 3;
        const int4 w = *reinterpret_cast<const int4*>(rawB + row * BT + 16 * part);
        const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
            *reinterpret_cast<float4*>(&Bs[row * BT + 16 * part + 4 * u]) = make_float4(
                dequant((int)(int8_t)(words[u]), s), dequant((int)(int8_t)(words[u] >> 8), s),
                dequant((int)(int8_t)(words[u] >> 16), s), dequant((int)(int8_t)(words[u] >> 24), s));
    }
}

template <bool DW>
__global__ void __launch_bounds__(NT6, 1) k_bwd6(const BwdArgs a)
{
    extern __shared__ __align__(16) uint8_t smem6[];
    float* rawA = reinterpret_cast<float*>(smem6);
    int8_t* rawB = reinterpret_cast<int8_t*>(smem6 + RAW6_A_BYTES);
    float* As = reinterpret_cast<float*>(smem6 + RAW6_A_BYTES + RAW6_B_BYTES);
    float* Bs = reinterpret_cast<float*>(smem6 + RAW6_A_BYTES + RAW6_B_BYTES + COMP6_A_BYTES);
    u64* ext7 = reinterpret_cast<u64*>(smem6 + RAW6_A_BYTES + RAW6_B_BYTES + COMP6_A_BYTES +
                                       COMP6_B_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem6 + RAW6_A_BYTES + RAW6_B_BYTES +
                                                      COMP6_A_BYTES + COMP6_B_BYTES + EXT6_BYTES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);   // rows 8ty .. 8ty+7 (ty < 24)
    const int tx = (warp & 1) * 8 + (lane & 7);     // cols 4tx .. 4tx+3
    const int64_t i0 = (int64_t)blockIdx.y * BI6, j0 = (int64_t)blockIdx.x * BT;
    const float s = flush(*a.scale);

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         (uint32_t)__cvta_generic_to_shared(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) +
                           (uint32_t)((warp >> 2) * 160);

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));

    u64 S[2][16];
    u64 acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        acc[e] = 0ull;
#pragma unroll
    for (int l = 0; l < 2; ++l)
#pragma unroll
        for (int e = 0; e < 16; ++e)
            S[l][e] = 0ull;

    issue_raw6<DW>(rawA, rawB, a, i0, j0, cbeg * CH, (int)min((int64_t)CH, a.R - cbeg * CH), tid);
    cp_async_wait_all();
    __syncthreads();
    transform6<DW>(As, Bs, rawA, rawB, s, tid);
    __syncthreads();

    const float* Ar = As + 8 * ty;
    const float* Br = Bs + 4 * tx;

    for (int64_t c = cbeg; c < cend; ++c) {
        const int64_t r0 = c * CH;
        const int valid = (int)min((int64_t)CH, a.R - r0);
        const bool more = c + 1 < cend;
        if (more)
            issue_raw6<DW>(rawA, rawB, a, i0, j0, r0 + CH, (int)min((int64_t)CH, a.R - r0 - CH),
                           tid);

        ulonglong2 a03 = *reinterpret_cast<const ulonglong2*>(Ar);
        ulonglong2 a47 = *reinterpret_cast<const ulonglong2*>(Ar + 4);
        float4 b = *reinterpret_cast<const float4*>(Br);
        {
            const ulonglong2 c03 = a03, c47 = a47;
            const float4 cb = b;
            if (valid > 1) {
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + BI6);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + BI6 + 4);
                b = *reinterpret_cast<const float4*>(Br + BT);
            }
            step<true>(acc, c03, c47, cb);
        }
        if (valid == CH) {
#pragma unroll 7
            for (int r = 1; r < CH; ++r) {
                const ulonglong2 c03 = a03, c47 = a47;
                const float4 cb = b;
                const int rn = r + 1 < CH ? r + 1 : r;
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI6);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI6 + 4);
                b = *reinterpret_cast<const float4*>(Br + rn * BT);
                step<false>(acc, c03, c47, cb);
            }
        } else {
            for (int r = 1; r < valid; ++r) {
                const ulonglong2 c03 = a03, c47 = a47;
                const float4 cb = b;
                const int rn = r + 1 < valid ? r + 1 : r;
                a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI6);
                a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * BI6 + 4);
                b = *reinterpret_cast<const float4*>(Br + rn * BT);
                step<false>(acc, c03, c47, cb);
            }
        }

        // tree: levels 0-1 registers, 2-6 tensor memory, 7 shared memory
        const int cs = (int)(c - cbeg);
        if (more) {
            const int tz = __ffs(~cs) - 1;
#pragma unroll
            for (int t = 0; t < MAXLVL; ++t) {
                if (tz == t) {
#pragma unroll
                    for (int l = 0; l < t; ++l) {
                        if (l < 2) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                acc[e] = fadd2_ftz(S[l < 2 ? l : 0][e], acc[e]);
                        } else {
                            tmem_fold16(tbase + (uint32_t)(32 * (l - 2)), acc);
                            tmem_fold16(tbase + (uint32_t)(32 * (l - 2) + 16), acc + 8);
                        }
                    }
                    if (t < 2) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            S[t < 2 ? t : 0][e] = acc[e];
                    } else if (t < 7) {
                        tmem_st16(tbase + (uint32_t)(32 * (t - 2)), acc);
                        tmem_st16(tbase + (uint32_t)(32 * (t - 2) + 16), acc + 8);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            ext7[e * NT6 + tid] = acc[e];
                    }
                }
            }
        } else {
#pragma unroll
            for (int l = 0; l < MAXLVL; ++l) {
                if ((cs >> l) & 1) {
                    if (l < 2) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            acc[e] = fadd2_ftz(S[l < 2 ? l : 0][e], acc[e]);
                    } else if (l < 7) {
                        tmem_fold16(tbase + (uint32_t)(32 * (l - 2)), acc);
                        tmem_fold16(tbase + (uint32_t)(32 * (l - 2) + 16), acc + 8);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            acc[e] = fadd2_ftz(ext7[e * NT6 + tid], acc[e]);
                    }
                }
            }
        }

        if (more) {
            cp_async_wait_all();
            __syncthreads();
            transform6<DW>(As, Bs, rawA, rawB, s, tid);
            __syncthreads();
        }
    }

    const int64_t col = j0 + 4 * tx;
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = i0 + 8 * ty + 2 * ip + h;
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo, hi;
                unpack2(acc[ip * 4 + j], lo, hi);
                o[j] = h ? hi : lo;
            }
            if (row >= a.I || col >= a.J)
                continue;
            if (a.nseg == 1) {
                float* dst = a.out + row * a.J + col;
                float v0 = flush(o[0]), v1 = flush(o[1]), v2 = flush(o[2]), v3 = flush(o[3]);
                if (a.accumulate) {
                    const float4 old = *reinterpret_cast<const float4*>(dst);
                    v0 = fadd_ftz(old.x, v0);
                    v1 = fadd_ftz(old.y, v1);
                    v2 = fadd_ftz(old.z, v2);
                    v3 = fadd_ftz(old.w, v3);
                }
                *reinterpret_cast<float4*>(dst) = make_float4(v0, v1, v2, v3);
            } else {
                float* base = a.ws + (int64_t)blockIdx.z * a.I * a.J;
                *reinterpret_cast<float4*>(base + row * a.J + col) = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(*tmem_slot)
                     : "memory");
    }
}

} // namespace

template <bool DW>
cudaError_t launch_bwd_staged(int kernel, const BwdArgs& a, cudaStream_t st)
{
    const unsigned gx = (unsigned)cdiv(a.J, BT), gz = (unsigned)a.nseg;
    cudaError_t e = cudaSuccess;
    switch (kernel) {
    case 0:
        k_bwd<DW><<<dim3(gx, (unsigned)cdiv(a.I, BT), gz), 256, 0, st>>>(a);
        break;
    case 2:
        e = cudaFuncSetAttribute(k_bwd3<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)BWD3_SMEM);
        if (e == cudaSuccess)
            k_bwd3<DW><<<dim3(gx, (unsigned)cdiv(a.I, BT), gz), 256, BWD3_SMEM, st>>>(a);
        break;
    case 3:
        e = cudaFuncSetAttribute(k_bwd4<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)BWD4_SMEM);
        if (e == cudaSuccess)
            k_bwd4<DW><<<dim3(gx, (unsigned)cdiv(a.I, BI4), gz), 256, BWD4_SMEM, st>>>(a);
        break;
    case 4:
        e = cudaFuncSetAttribute(k_bwd5<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)BWD5_SMEM);
        if (e == cudaSuccess)
            k_bwd5<DW><<<dim3(gx, (unsigned)cdiv(a.I, BI4), gz), 256, BWD5_SMEM, st>>>(a);
        break;
    case 5:
        e = cudaFuncSetAttribute(k_bwd6<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)BWD6_SMEM);
        if (e == cudaSuccess)
            k_bwd6<DW><<<dim3(gx, (unsigned)cdiv(a.I, BI6), gz), NT6, BWD6_SMEM, st>>>(a);
        break;
    default:
        // opt in to 96 KB of dynamic shared memory (on the current device)
        e = cudaFuncSetAttribute(k_bwd2<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)BWD2_SMEM);
        if (e == cudaSuccess)
            k_bwd2<DW><<<dim3(gx, (unsigned)cdiv(a.I, BT), gz), 256, BWD2_SMEM, st>>>(a);
        break;
    }
    return e;
}

template cudaError_t launch_bwd_staged<false>(int, const BwdArgs&, cudaStream_t);
template cudaError_t launch_bwd_staged<true>(int, const BwdArgs&, cudaStream_t);

} // namespace repro
