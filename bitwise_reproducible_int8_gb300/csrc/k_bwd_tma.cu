// k_bwd_tma.cu -- fp32 backward of the int8 QAT linear fed by the tensor
// memory accelerator, with the operand preparation done once per call.
//
//   dX[m,k] = canon_n( dY[m,n] (x) W^[n,k] )     W^ = float(Wq) (x) s_w, flushed
//   dW[n,k] = canon_m( dY[m,n] (x) X^[m,k] )     X^ = float(Xq) (x) s_x, flushed
// with the fixed reduction order and explicit unfused multiply then add of the
// Open-1B review (onedev.kr/papers/92, section "How it works"): chunks of 64
// terms summed left to right from the first term, then the stride-doubling
// pairwise tree over chunk partials; subnormal operands read as zero.
//
// The single-pass kernels flush dY and dequantise the int8 operand inside
// every CTA that reads a tile, so the same element is transformed once per
// CTA row (128 times for the weight of a 16,384-token micro-batch), on the
// same pipes as the products.  Here the operands are prepared once, into the
// caller's workspace, by streaming kernels:
//   * dY flushed, in its own layout (dW: A[r=m][i=n]) or transposed
//     (dX: A[r=n][i=m], rows padded to a multiple of 4 floats);
//   * the int8 operand dequantised to fp32 (B[r][j]).
// The values are exactly the ones the single-pass kernels build in shared
// memory, so the bits of dX and dW are unchanged.
//
// The main kernel then only moves bytes and computes:
//   * 8 warps own the 128 x 64 output tile, 8 x 4 outputs per thread, packed
//     f32x2 multiply and add, reading a 4-stage shared-memory ring in place;
//   * thread 0 also issues the copies: two 2D tensor copies per 64-term chunk
//     (A: 64 x 128 floats, B: 64 x 64 floats, zero fill outside the tensor),
//     the ring guarded by full/empty mbarriers.  The prologue fills the four
//     stages; at the start of chunk c it refills the stage that every warp
//     released at the end of chunk c - 2 with chunk c + 2, so no warp runs
//     more than two chunks ahead of warp 0 and every wait ends;
//   * with 8 warps a thread may hold 255 registers: tree level 0 (RL = 1)
//     stays in registers, beside the products formed two row pairs ahead of
//     their adds, and the rest live in tensor memory (thread: lane
//     32*(warp%4) + lane, columns (warp/4)*256 + 32*(level-RL)), touched once
//     every 2 chunks.
// Every wait is bounded: past the limit the CTA records a failure in the
// device error word, lets its copies land, frees its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "bwd_common.cuh"
#include "bwd_tile.cuh"
#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace repro {
namespace {

constexpr int NC = 256;                        // threads (8 warps)
constexpr int RL = 1;                          // tree levels kept in registers
constexpr int TI = BWD_TMA_ROWS;               // 128 tile rows (i)
constexpr int STG = 4;                         // ring stages
constexpr int A_BYTES = CH * TI * 4;           // 32768: A[r][i]
constexpr int B_BYTES = CH * BT * 4;           // 16384: B[r][j]
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CTRL_OFF = STG * STAGE_BYTES;
constexpr size_t SMEM_BYTES = 1024 + (size_t)CTRL_OFF + 128;   // + alignment slack

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
        step_ahead2<true>(acc, c03, c47, cb);
    }
    if (valid == CH) {
#pragma unroll 21
        for (int r = 1; r < CH; ++r) {
            const ulonglong2 c03 = a03, c47 = a47;
            const float4 cb = b;
            const int rn = r + 1 < CH ? r + 1 : r;
            a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI);
            a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI + 4);
            b = *reinterpret_cast<const float4*>(Br + rn * BT);
            step_ahead2<false>(acc, c03, c47, cb);
        }
    } else {
        for (int r = 1; r < valid; ++r) {
            const ulonglong2 c03 = a03, c47 = a47;
            const float4 cb = b;
            const int rn = r + 1 < valid ? r + 1 : r;
            a03 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI);
            a47 = *reinterpret_cast<const ulonglong2*>(Ar + rn * TI + 4);
            b = *reinterpret_cast<const float4*>(Br + rn * BT);
            step_ahead2<false>(acc, c03, c47, cb);
        }
    }
}

// rows 0 .. CH-2 of a full chunk with row 0 already in (a03, a47, b); on
// return (a03, a47, b) hold row CH-1, loaded but not yet multiplied
__device__ __forceinline__ void chunk_head(u64 (&acc)[16], const float* __restrict__ Ar,
                                           const float* __restrict__ Br, ulonglong2& a03,
                                           ulonglong2& a47, float4& b)
{
    {
        const ulonglong2 c03 = a03, c47 = a47;
        const float4 cb = b;
        a03 = *reinterpret_cast<const ulonglong2*>(Ar + TI);
        a47 = *reinterpret_cast<const ulonglong2*>(Ar + TI + 4);
        b = *reinterpret_cast<const float4*>(Br + BT);
        step_ahead2<true>(acc, c03, c47, cb);
    }
#pragma unroll 31
    for (int r = 1; r < CH - 1; ++r) {
        const ulonglong2 c03 = a03, c47 = a47;
        const float4 cb = b;
        a03 = *reinterpret_cast<const ulonglong2*>(Ar + (r + 1) * TI);
        a47 = *reinterpret_cast<const ulonglong2*>(Ar + (r + 1) * TI + 4);
        b = *reinterpret_cast<const float4*>(Br + (r + 1) * BT);
        step_ahead2<false>(acc, c03, c47, cb);
    }
}

template <bool DW>
__global__ void __launch_bounds__(NC, 1)
    k_bwd_tma(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
              const BwdArgs a)
{
    extern __shared__ uint8_t smt_raw[];
    // tensor copies want 128-byte aligned destinations; align the ring to 1024
    uint8_t* smt = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smt_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smt + CTRL_OFF);   // [STG], copies landed
    uint64_t* empty = full + STG;                                   // [STG], stage released
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(empty + STG);
    int* prod_fail = reinterpret_cast<int*>(tmem_slot + 1);
    int* comp_fail = prod_fail + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t i0 = (int64_t)blockIdx.y * TI, j0 = (int64_t)blockIdx.x * BT;

    const int64_t C = (a.R + CH - 1) / CH;
    const int64_t cbeg = (int64_t)blockIdx.z << a.seg_log2;
    const int64_t cend = min(C, cbeg + ((int64_t)1 << a.seg_log2));
    const int n = (int)(cend - cbeg);

    auto stA = [&](int s) { return reinterpret_cast<float*>(smt + s * STAGE_BYTES); };
    auto stB = [&](int s) { return reinterpret_cast<float*>(smt + s * STAGE_BYTES + A_BYTES); };
    auto valid_of = [&](int cs) { return (int)min((int64_t)CH, a.R - (cbeg + cs) * CH); };
    auto issue = [&](int cs) {
        const int s = cs % STG;
        const int r0 = (int)((cbeg + cs) * CH);
        mbar_expect_tx(&full[s], STAGE_BYTES);
        tma_load_2d(stA(s), &map_a, (int)i0, r0, &full[s]);
        tma_load_2d(stB(s), &map_b, (int)j0, r0, &full[s]);
    };
    // the last copy into every stage has landed (bounded); false on a timeout
    auto drain = [&](int issued) {
        bool fine = true;
        for (int cs = issued - 1; cs >= 0 && cs >= issued - STG; --cs)
            if (!mbar_wait(&full[cs % STG], (cs / STG) & 1))
                fine = false;
        return fine;
    };

    if (tid == 0) {
        for (int s = 0; s < STG; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NC / 32);   // one arrival per compute warp
        }
        *prod_fail = 0;
        *comp_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
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

    {
        const int ty = (warp >> 1) * 4 + (lane >> 3);   // rows 8ty .. 8ty+7
        const int tx = (warp & 1) * 8 + (lane & 7);     // cols 4tx .. 4tx+3
        const uint32_t tbase =
            *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);

        const bool issuer = tid == 0;
        int issued = 0;
        if (issuer) {
            for (; issued < n && issued < STG; ++issued)
                issue(issued);
        }

        u64 S[RL][16];
        u64 acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            acc[e] = 0ull;
#pragma unroll
        for (int l = 0; l < RL; ++l)
#pragma unroll
            for (int e = 0; e < 16; ++e)
                S[l][e] = 0ull;

        bool ok = true;
        // the next chunk's full wait and its row-0 loads are made before the
        // current chunk's last row is multiplied, so they overlap it
        ulonglong2 n03 = {0ull, 0ull}, n47 = {0ull, 0ull};
        float4 nb = make_float4(0.f, 0.f, 0.f, 0.f);
        auto wait_full = [&](int c) {
            const bool got = mbar_wait(&full[c % STG], (c / STG) & 1);
            return !__any_sync(0xffffffffu, !got);
        };
        auto load_row0 = [&](int c) {
            const float* Ar = stA(c % STG) + 8 * ty;
            n03 = *reinterpret_cast<const ulonglong2*>(Ar);
            n47 = *reinterpret_cast<const ulonglong2*>(Ar + 4);
            nb = *reinterpret_cast<const float4*>(stB(c % STG) + 4 * tx);
        };
        if (n > 0) {
            if (wait_full(0)) {
                load_row0(0);
            } else {
                ok = false;
                if (lane == 0)
                    *comp_fail = 1;
            }
        }
        for (int cs = 0; ok && cs < n; ++cs) {
            const int s = cs % STG;
            if (warp == 0) {
                // refill the stage every warp released two chunks ago
                if (lane == 0 && issued == cs + 2 && issued < n) {
                    const int rc = issued - STG;
                    if (mbar_wait(&empty[rc % STG], (rc / STG) & 1)) {
                        issue(issued);
                        ++issued;
                    } else {
                        *prod_fail = 1;
                    }
                }
                __syncwarp();
            }
            const int valid = valid_of(cs);
            if (valid == CH) {
                chunk_head(acc, stA(s) + 8 * ty, stB(s) + 4 * tx, n03, n47, nb);
                const ulonglong2 l03 = n03, l47 = n47;
                const float4 lb = nb;
                bool next_ok = true;
                if (cs + 1 < n) {
                    next_ok = wait_full(cs + 1);
                    if (next_ok)
                        load_row0(cs + 1);
                }
                __syncwarp();   // every lane's reads of stage s precede lane 0's release
                if (lane == 0)
                    mbar_arrive(&empty[s]);
                step_ahead2<false>(acc, l03, l47, lb);
                if (!next_ok) {
                    ok = false;
                    if (lane == 0)
                        *comp_fail = 1;
                    break;
                }
            } else {
                // only the reduction's last chunk is partial, and its full
                // wait was made at the end of the chunk before
                chunk_sum(acc, stA(s) + 8 * ty, stB(s) + 4 * tx, valid);
                __syncwarp();   // every lane's reads of stage s precede lane 0's release
                if (lane == 0)
                    mbar_arrive(&empty[s]);
            }

            // tree over chunk partials (cs counted from the segment start)
            if (cs + 1 < n) {
                const int tz = __ffs(~cs) - 1;
#pragma unroll
                for (int t = 0; t < MAXLVL; ++t) {
                    if (tz == t) {
#pragma unroll
                        for (int l = 0; l < t; ++l) {
                            if (l < RL) {
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    acc[e] = fadd2_ftz(S[l < RL ? l : 0][e], acc[e]);
                            } else {
                                tmem_fold32(tbase + (uint32_t)(32 * (l - RL)), acc);
                            }
                        }
                        if (t < RL) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                S[t < RL ? t : 0][e] = acc[e];
                        } else {
                            tmem_st32(tbase + (uint32_t)(32 * (t - RL)), acc);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int l = 0; l < MAXLVL; ++l) {
                    if ((cs >> l) & 1) {
                        if (l < RL) {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                acc[e] = fadd2_ftz(S[l < RL ? l : 0][e], acc[e]);
                        } else {
                            tmem_fold32(tbase + (uint32_t)(32 * (l - RL)), acc);
                        }
                    }
                }
            }
        }

        if (issuer && !drain(issued))
            *prod_fail = 1;

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

// ---------------------------------------------------------------- wait probe

// One thread waits, with the pipeline's bounded wait, on a barrier phase that
// completes only if `arrive` is set.  Without the arrival the wait gives up
// after WAIT_CYCLES, the error word is set exactly as a stalled pipeline sets
// it, and the kernel returns.
__global__ void __launch_bounds__(32) k_wait_probe(int* err, int arrive)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0)
        return;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (arrive)
        mbar_arrive(&bar);
    if (!mbar_wait(&bar, 0))
        atomicExch(err, 1);
}

// ---------------------------------------------------------------- operand prep

// 16 codes -> 4 float4 of dequantised, flushed values
__device__ __forceinline__ void dequant16(const int4 w, float s, float4* o)
{
    const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
        o[u] = make_float4(dequant((int)(int8_t)(words[u]), s), dequant((int)(int8_t)(words[u] >> 8), s),
                           dequant((int)(int8_t)(words[u] >> 16), s),
                           dequant((int)(int8_t)(words[u] >> 24), s));
}

// out[e] = float(q[e]) (x) s, flushed; 16 codes per thread per load, four
// loads in flight per step
__global__ void __launch_bounds__(256)
    k_dequant_f32(const int8_t* __restrict__ q, const float* __restrict__ scale,
                  float* __restrict__ out, int64_t n)
{
    const float s = flush(*scale);
    const int64_t nv = n >> 4;
    const int4* q16 = reinterpret_cast<const int4*>(q);
    float4* o = reinterpret_cast<float4*>(out);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < nv; i += 4 * stride) {
        int4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            w[u] = ld_stream(q16 + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            dequant16(w[u], s, o + 4 * (i + u * stride));
    }
    for (; i < nv; i += stride)
        dequant16(ld_stream(q16 + i), s, o + 4 * i);
    if (blockIdx.x == 0) {
        const int64_t i = (nv << 4) + threadIdx.x;
        if (threadIdx.x < 16 && i < n)
            out[i] = dequant((int)q[i], s);
    }
}

// out[e] = flush(x[e]), n % 4 == 0
__global__ void __launch_bounds__(256)
    k_flush_copy(const float* __restrict__ x, float* __restrict__ out, int64_t n)
{
    const int64_t nv = n >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float4* o4 = reinterpret_cast<float4*>(out);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x)
        o4[i] = flush4(ld_stream(x4 + i));
}

// out[c][r] = flush(x[r][c]) for x [rows x cols]; out row pitch ldo floats.
// 32 x 32 tiles through shared memory (padded: conflict-free both ways),
// tiles visited grid-stride.  (Moving four tiles per step, for more loads in
// flight, made it slower on GB300: 184 vs 131 us per block-workload launch.)
__global__ void __launch_bounds__(256)
    k_flush_transpose(const float* __restrict__ x, float* __restrict__ out, int64_t rows,
                      int64_t cols, int64_t ldo)
{
    __shared__ float t[32][33];
    const int64_t tr = (rows + 31) / 32, tc = (cols + 31) / 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    for (int64_t tile = blockIdx.x; tile < tr * tc; tile += gridDim.x) {
        const int64_t r0 = (tile / tc) * 32, c0 = (tile % tc) * 32;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t r = r0 + ty + 8 * k, c = c0 + tx;
            t[ty + 8 * k][tx] = (r < rows && c < cols) ? flush(x[r * cols + c]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = c0 + ty + 8 * k, r = r0 + tx;
            if (c < cols && r < rows)
                out[c * ldo + r] = t[tx][ty + 8 * k];
        }
        __syncthreads();
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// fp32 [rows x cols] with row pitch ld floats; box box_c (columns) x 64 rows, no swizzle
bool make_map(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld,
              int box_c)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    cuuint32_t box[2] = {(cuuint32_t)box_c, (cuuint32_t)CH};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

inline int64_t align256(int64_t b) { return (b + 255) & ~(int64_t)255; }
inline int64_t pad4(int64_t v) { return (v + 3) & ~(int64_t)3; }

} // namespace

size_t bwd_tma_operand_bytes(int64_t M, int64_t N, int64_t K)
{
    // dX: dY^T [N x pad4(M)] + W^ [N x K]; dW: dY [M x N] + X^ [M x K]; the two
    // calls run in stream order and share the region
    const int64_t dx = align256(N * pad4(M) * 4) + align256(N * K * 4);
    const int64_t dw = align256(M * N * 4) + align256(M * K * 4);
    return (size_t)(dx > dw ? dx : dw);
}

template <bool DW>
cudaError_t launch_bwd_tma(const BwdArgs& a0, const int8_t* q, float* opnd, dim3 grid,
                           cudaStream_t st)
{
    BwdArgs a = a0;
    const int eb = 8 * num_sms();
    // a.I x a.J outputs, reduction a.R; dY is [M x N] with ldy = N
    float* Aop = opnd;
    int64_t lda;
    float* Bop;
    if (DW) {
        // A[r=m][i=n] = flush(dY[m][n]): I = N, R = M
        lda = a.I;
        Bop = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(opnd) + align256(a.R * a.I * 4));
        k_flush_copy<<<eb, 256, 0, st>>>(a.dy, Aop, a.R * a.I);
    } else {
        // A[r=n][i=m] = flush(dY[m][n]): I = M, R = N, rows padded to 4 floats
        lda = pad4(a.I);
        Bop = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(opnd) + align256(a.R * lda * 4));
        k_flush_transpose<<<eb, 256, 0, st>>>(a.dy, Aop, a.I, a.R, lda);
    }
    k_dequant_f32<<<eb, 256, 0, st>>>(q, a.scale, Bop, a.R * a.J);
    count_launches(2);
    CUtensorMap ma, mb;
    if (!make_map(&ma, Aop, a.R, a.I, lda, TI) || !make_map(&mb, Bop, a.R, a.J, a.J, BT))
        return cudaErrorInvalidValue;
    auto kern = k_bwd_tma<DW>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, NC, SMEM_BYTES, st>>>(ma, mb, a);
    return cudaGetLastError();
}

template cudaError_t launch_bwd_tma<false>(const BwdArgs&, const int8_t*, float*, dim3,
                                           cudaStream_t);
template cudaError_t launch_bwd_tma<true>(const BwdArgs&, const int8_t*, float*, dim3,
                                          cudaStream_t);

cudaError_t launch_wait_probe(int arrive, cudaStream_t st)
{
    k_wait_probe<<<1, 32, 0, st>>>(device_error_word(), arrive);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
