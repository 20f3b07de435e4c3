// k_bwd_ws.cu -- warp-specialised fp32 backward of the int8 QAT linear.
//
//   dX[m,k] = canon_n( dY[m,n] (x) W^[n,k] )     W^ = float(Wq) (x) s_w
//   dW[n,k] = canon_m( dY[m,n] (x) X^[m,k] )     X^ = float(Xq) (x) s_x
// with the fixed reduction order and explicit unfused multiply then add of the
// Open-1B review (onedev.kr/papers/92, section "How it works"): chunks of 64
// terms summed left to right from the first term, then the stride-doubling
// pairwise tree over chunk partials.  Same per-output arithmetic, tile and
// tree as the wide-tile kernel of k_bwd.cu (k_bwd4); only the division of
// labour changes, so the bits are the same.
//
// The single-role kernels stop every warp twice per 64-term chunk (a CTA
// barrier before and after the pass that turns the raw chunk into the compute
// layout).  Here the roles are split:
//   * 4 producer warps copy raw chunks global -> shared with cp.async (two raw
//     stages, one chunk ahead), then flush dY (transposing it for dX) and
//     dequantise the int8 operand into one of two compute stages; they sync
//     among themselves with a named barrier only;
//   * 8 compute warps own the 128 x 64 output tile (8 x 4 outputs per thread,
//     packed f32x2 multiply and add) and meet the producers only through a
//     full/empty mbarrier pair per compute stage, so a warp that finishes a
//     chunk early starts the next one at once;
//   * tree level 0 stays in registers, levels 1-7 live in tensor memory
//     (thread: lane 32*(warp%4) + lane, columns (warp/4)*256 + 32*(level-1)),
//     touched at most once every other chunk.
// Every wait is bounded: past the limit the CTA records a failure in the
// device error word, lets its copies land, frees its tensor memory and exits.
#include "bwd_common.cuh"
#include "bwd_tile.cuh"
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace repro {
namespace {

constexpr int NC = 256;                              // compute threads (warps 0-7)
constexpr int NP = 128;                              // producer threads (warps 8-11)
constexpr int NTH = NC + NP;
constexpr int TI = BWD_WS_ROWS;                      // 128 tile rows (i)
constexpr int RAWA_BYTES = TI * 68 * 4;              // DX: 128 rows x pitch 68; DW: 64 x 132
constexpr int RAWB_BYTES = CH * BT;                  // 64 rows x 64 int8
constexpr int RAW_STAGE = RAWA_BYTES + RAWB_BYTES;   // 38912
constexpr int COMPA_BYTES = CH * TI * 4;             // A[r][i], 32768
constexpr int COMPB_BYTES = CH * BT * 4;             // B[r][j], 16384
constexpr int COMP_STAGE = COMPA_BYTES + COMPB_BYTES;
constexpr int CTRL_OFF = 2 * RAW_STAGE + 2 * COMP_STAGE;
constexpr size_t SMEM_BYTES = (size_t)CTRL_OFF + 64;
constexpr int REGL = 1;                              // tree levels kept in registers

__device__ __forceinline__ void producer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NP) : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(su32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

// raw copy of the chunk starting at reduction index r0 by producer thread p:
// DW: A = 64 rows (reduction) x 128 floats (i), pitch 132;
// DX: A = 128 rows (i) x 64 floats (reduction), pitch 68;
// B = 64 rows (reduction) x 64 int8 (j).  Pieces outside the tensor are
// zero-filled (the shapes guarantee a 16-byte piece is wholly in or out).
template <bool DW>
__device__ __forceinline__ void issue_raw(float* __restrict__ rawA, int8_t* __restrict__ rawB,
                                          const BwdArgs& a, int64_t i0, int64_t j0, int64_t r0,
                                          int valid, int p)
{
#pragma unroll
    for (int it = 0; it < 16; ++it) {
        const int e = p + it * NP;
        const float* src;
        float* dst;
        bool ok;
        if (DW) {
            const int row = e >> 5, f = e & 31;
            src = a.dy + (r0 + row) * a.ldy + i0 + 4 * f;
            ok = row < valid && i0 + 4 * f < a.I;
            dst = rawA + row * 132 + 4 * f;
        } else {
            const int row = e >> 4, f = e & 15;
            src = a.dy + (i0 + row) * a.ldy + r0 + 4 * f;
            ok = i0 + row < a.I && 4 * f < valid;
            dst = rawA + row * 68 + 4 * f;
        }
        cp_async16(dst, ok ? src : a.dy, ok ? 16u : 0u);
    }
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int e = p + it * NP;
        const int row = e >> 2, part = e & 3;
        const bool ok = row < valid && j0 + 16 * part < a.J;
        const int8_t* src = ok ? a.q + (r0 + row) * a.J + j0 + 16 * part : a.q;
        cp_async16(rawB + row * BT + 16 * part, src, ok ? 16u : 0u);
    }
}

// raw chunk -> compute layout: A[r][i] = flush(dY), B[r][j] = float(q) (x) s, flushed
template <bool DW>
__device__ __forceinline__ void transform(float* __restrict__ As, float* __restrict__ Bs,
                                          const float* __restrict__ rawA,
                                          const int8_t* __restrict__ rawB, float s, int p)
{
    if (DW) {
#pragma unroll
        for (int it = 0; it < 16; ++it) {
            const int e = p + it * NP;
            const int r = e >> 5, f = e & 31;
            const float4 v = *reinterpret_cast<const float4*>(rawA + r * 132 + 4 * f);
            *reinterpret_cast<float4*>(&As[r * TI + 4 * f]) = flush4(v);
        }
    } else {
        const int i = p;   // one tile row per producer thread
#pragma unroll
        for (int f = 0; f < 16; ++f) {
            const float4 v = *reinterpret_cast<const float4*>(rawA + i * 68 + 4 * f);
            As[(4 * f + 0) * TI + i] = flush(v.x);
            As[(4 * f + 1) * TI + i] = flush(v.y);
            As[(4 * f + 2) * TI + i] = flush(v.z);
            As[(4 * f + 3) * TI + i] = flush(v.w);
        }
    }
    const int row = p >> 1, half = p & 1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int4 w = *reinterpret_cast<const int4*>(rawB + row * BT + 32 * half + 16 * h);
        const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
            *reinterpret_cast<float4*>(&Bs[row * BT + 32 * half + 16 * h + 4 * u]) =
                make_float4(dequant((int)(int8_t)(words[u]), s),
                            dequant((int)(int8_t)(words[u] >> 8), s),
                            dequant((int)(int8_t)(words[u] >> 16), s),
                            dequant((int)(int8_t)(words[u] >> 24), s));
    }
}

// the chunk's left-to-right sums for this thread's 32 outputs
__device__ __forceinline__ void chunk_sum(u64 (&acc)[16], const float* __restrict__ Ar,
                                          const float* __restrict__ Br, int valid)
{
    ulonglong2 a03 = *reinterpret_cast<const ulonglong2*>(Ar);
    ulonglong2 a47 = *reinterpret_cast<const ulonglong2*>(Ar + 4);
    float4 b = *reinterpret_cast<const float4*>(Br);
    {
        const ulonglong2 c03 = a03, c47 = a47;
        const float4 cb = b;
        if (valid > 1) {
            a03 = *reinterpret_cast<const ulonglong2*>(Ar + TI);
            a47 = *reinterpret_cast<const ulonglong2*>(Ar + TI + 4);
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
            a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI);
            a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI + 4);
            b = *reinterpret_cast<const float4*>(Br + rn * BT);
            step<false>(acc, c03, c47, cb);
        }
    } else {
        for (int r = 1; r < valid; ++r) {
            const ulonglong2 c03 = a03, c47 = a47;
            const float4 cb = b;
            const int rn = r + 1 < valid ? r + 1 : r;
            a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI);
            a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI + 4);
            b = *reinterpret_cast<const float4*>(Br + rn * BT);
            step<false>(acc, c03, c47, cb);
        }
    }
}

template <bool DW>
__global__ void __launch_bounds__(NTH, 1) k_bwd_ws(const BwdArgs a)
{
    extern __shared__ __align__(128) uint8_t smw[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smw + CTRL_OFF);   // [2], producers -> compute
    uint64_t* empty = full + 2;                                     // [2], compute -> producers
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty + 2);
    int* prod_fail = reinterpret_cast<int*>(tmem_slot + 1);
    int* comp_fail = prod_fail + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t i0 = (int64_t)blockIdx.y * TI, j0 = (int64_t)blockIdx.x * BT;

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));
    const int n = (int)(cend - cbeg);

    auto rawA = [&](int b) { return reinterpret_cast<float*>(smw + b * RAW_STAGE); };
    auto rawB = [&](int b) { return reinterpret_cast<int8_t*>(smw + b * RAW_STAGE + RAWA_BYTES); };
    auto compA = [&](int b) { return reinterpret_cast<float*>(smw + 2 * RAW_STAGE + b * COMP_STAGE); };
    auto compB = [&](int b) {
        return reinterpret_cast<float*>(smw + 2 * RAW_STAGE + b * COMP_STAGE + COMPA_BYTES);
    };
    auto valid_of = [&](int cs) { return (int)min((int64_t)CH, a.R - (cbeg + cs) * CH); };

    if (tid == 0) {
        mbar_init(&full[0], NP);
        mbar_init(&full[1], NP);
        mbar_init(&empty[0], NC);
        mbar_init(&empty[1], NC);
        *prod_fail = 0;
        *comp_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         su32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    if (warp >= NC / 32) {
        // ------------------------------------------------------------ producers
        const int p = tid - NC;
        const float s = flush(*a.scale);
        issue_raw<DW>(rawA(0), rawB(0), a, i0, j0, cbeg * CH, valid_of(0), p);
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (n > 1)
            issue_raw<DW>(rawA(1), rawB(1), a, i0, j0, (cbeg + 1) * CH, valid_of(1), p);
        asm volatile("cp.async.commit_group;" ::: "memory");
        for (int cs = 0; cs < n; ++cs) {
            const int st = cs & 1;
            // groups committed so far: cs + 2; all but the newest hold chunk cs
            asm volatile("cp.async.wait_group 1;" ::: "memory");
            if (cs >= 2 && p == 0 && !mbar_wait(&empty[st], ((cs >> 1) - 1) & 1))
                *prod_fail = 1;
            producer_sync();   // raw chunk cs visible; compute stage st released
            if (*prod_fail)
                break;
            transform<DW>(compA(st), compB(st), rawA(st), rawB(st), s, p);
            mbar_arrive(&full[st]);
            producer_sync();   // every producer is done reading raw stage st
            if (cs + 2 < n)
                issue_raw<DW>(rawA(st), rawB(st), a, i0, j0, (cbeg + cs + 2) * CH, valid_of(cs + 2), p);
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    } else {
        // -------------------------------------------------------------- compute
        const int ty = (warp >> 1) * 4 + (lane >> 3);   // rows 8ty .. 8ty+7
        const int tx = (warp & 1) * 8 + (lane & 7);     // cols 4tx .. 4tx+3
        const uint32_t tbase =
            *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);

        u64 S[REGL][16];
        u64 acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            acc[e] = 0ull;
#pragma unroll
        for (int l = 0; l < REGL; ++l)
#pragma unroll
            for (int e = 0; e < 16; ++e)
                S[l][e] = 0ull;

        bool ok = true;
        for (int cs = 0; cs < n; ++cs) {
            const int st = cs & 1;
            const bool got = mbar_wait(&full[st], (cs >> 1) & 1);
            if (__any_sync(0xffffffffu, !got)) {
                ok = false;
                if (lane == 0)
                    *comp_fail = 1;
                break;
            }
            chunk_sum(acc, compA(st) + 8 * ty, compB(st) + 4 * tx, valid_of(cs));
            mbar_arrive(&empty[st]);

            // tree over chunk partials (cs counted from the segment start)
            if (cs + 1 < n) {
                const int tz = __ffs(~cs) - 1;
#pragma unroll
                for (int t = 0; t < MAXLVL; ++t) {
                    if (tz == t) {
#pragma unroll
                        for (int l = 0; l < t; ++l) {
                            if (l < REGL) {
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    acc[e] = fadd2_ftz(S[l < REGL ? l : 0][e], acc[e]);
                            } else {
                                tmem_fold32(tbase + (uint32_t)(32 * (l - REGL)), acc);
                            }
                        }
                        if (t < REGL) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                S[t < REGL ? t : 0][e] = acc[e];
                        } else {
                            tmem_st32(tbase + (uint32_t)(32 * (t - REGL)), acc);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int l = 0; l < MAXLVL; ++l) {
                    if ((cs >> l) & 1) {
                        if (l < REGL) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                acc[e] = fadd2_ftz(S[l < REGL ? l : 0][e], acc[e]);
                        } else {
                            tmem_fold32(tbase + (uint32_t)(32 * (l - REGL)), acc);
                        }
                    }
                }
            }
        }

        if (ok) {
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
                        float* dst = a.out + row * a.J + col;   // J % 16 == 0: whole float4 inside
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
                        *reinterpret_cast<float4*>(base + row * a.J + col) =
                            make_float4(o[0], o[1], o[2], o[3]);
                    }
                }
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
    if (tid == 0 && (*prod_fail || *comp_fail))
        atomicExch(a.err, 1);
}

} // namespace

template <bool DW>
cudaError_t launch_bwd_ws(const BwdArgs& a, dim3 grid, cudaStream_t st)
{
    cudaError_t e =
        cudaFuncSetAttribute(k_bwd_ws<DW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    k_bwd_ws<DW><<<grid, NTH, SMEM_BYTES, st>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_bwd_ws<false>(const BwdArgs&, dim3, cudaStream_t);
template cudaError_t launch_bwd_ws<true>(const BwdArgs&, dim3, cudaStream_t);

} // namespace repro
