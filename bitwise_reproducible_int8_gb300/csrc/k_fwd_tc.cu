// k_fwd_tc.cu -- exact int8 forward on the 5th-generation tensor cores.
//
// acc[m,n] = sum_k Xq[m,k] * Wq[n,k] must be the exact integer (int8 QAT
// linears: Open-1B review, onedev.kr/papers/92, section "How to use").  sm_103a
// has no tcgen05 int8 kind, so the codes are fed as bf16, which holds every
// integer in [-127, 127] exactly, to tcgen05.mma kind::f16 with fp32
// accumulation in tensor memory.  Each product is an integer of magnitude at
// most 16129 and every partial sum over a K-slice of 512 is an integer of
// magnitude at most 8,258,048 < 2^23, so each slice's fp32 accumulator holds
// its integer exactly; the epilogue converts every slice to int32 and adds the
// slices exactly.  Y = (float(acc) (x) s_x) (x) s_w, two flushed multiplies.
//
// Kernel structure (one 128 x 128 output tile per CTA, two CTAs per SM):
//   warp 0      TMA producer: bf16 A/B tiles of 128 rows x 64 K, 128-byte
//               swizzle, 3-stage ring (full/empty mbarriers);
//   warp 1      allocates 256 TMEM columns (two 128-column fp32 accumulators)
//               and one thread issues the MMAs (M=128, N=128, K=16), committing
//               each stage back to the producer and each K-slice to the
//               epilogue;
//   warps 2-5   epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its rows),
//               converts the slice to int32 and accumulates in registers, then
//               frees the accumulator for the slice after next.
// Every wait is bounded (about two seconds of clock64); on expiry the kernel
// records an error in the device error word, lets in-flight copies land,
// frees tensor memory and returns.  repro_device_check reports it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "pipeline.cuh"

namespace repro {
namespace {

constexpr int TM = 128;            // tile rows (M)
constexpr int TN = 128;            // tile columns (N)
constexpr int TK = 64;             // K per stage: one 128-byte swizzle row of bf16
constexpr int STAGES = 3;
constexpr int SLICE_KB = 8;        // k-blocks per exact slice: 8 * 64 = 512
constexpr int TILE_BYTES = TM * TK * 2;   // 16 KB, the same for A and B
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;
constexpr size_t SMEM_BYTES = 1024 + 2 * STAGES * TILE_BYTES + 256;
constexpr int EPI_PITCH = TN + 4;  // floats per staged output row (conflict-free both ways)
static_assert(4 * 32 * EPI_PITCH * 4 <= 2 * STAGES * TILE_BYTES,
              "the epilogue staging must fit in the operand ring");

struct Smem {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t dfull[2];
    uint64_t dempty[2];
    uint64_t done;
    uint32_t tmem_base;
    int failed;
};

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 128, M = 128
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TN >> 3) << 17) |
                           ((uint32_t)(TM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(a), "l"(b), "r"(IDESC), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            su32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define R8(i) "=r"(v[i + 0]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), \
              "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : R8(0), R8(8), R8(16), R8(24)
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
#undef R8

__global__ void __launch_bounds__(THREADS, 2)
k_fwd_tc(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
         const float* __restrict__ s_x, const float* __restrict__ s_w, float* __restrict__ y,
         int M, int N, int K, int* __restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled tiles need 1024-byte alignment in the shared window
    uint8_t* base = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
    uint8_t* A = base;                                   // STAGES x 16 KB
    uint8_t* B = base + STAGES * TILE_BYTES;             // STAGES x 16 KB
    Smem* sm = reinterpret_cast<Smem*>(base + 2 * STAGES * TILE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
    const int KB = (K + TK - 1) / TK;
    const int NS = (KB + SLICE_KB - 1) / SLICE_KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(&sm->dfull[d], 1);
            mbar_init(&sm->dempty[d], 4);
        }
        mbar_init(&sm->done, 1);
        sm->failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(&sm->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = sm->tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(&sm->empty[s], ((kb / STAGES) - 1) & 1)) {
                    sm->failed = 1;
                    break;
                }
                if (*(volatile int*)&sm->failed)
                    break;
                mbar_expect_tx(&sm->full[s], 2 * TILE_BYTES);
                tma_load_2d(A + s * TILE_BYTES, &map_a, kb * TK, m0, &sm->full[s]);
                tma_load_2d(B + s * TILE_BYTES, &map_b, kb * TK, n0, &sm->full[s]);
                issued = kb + 1;
            }
            // let the last copy into every stage land before the CTA can exit
            for (int kb = issued - 1; kb >= 0 && kb >= issued - STAGES; --kb)
                if (!mbar_wait(&sm->full[kb % STAGES], (kb / STAGES) & 1))
                    sm->failed = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            for (int kb = 0; kb < KB && ok; ++kb) {
                const int s = kb % STAGES;
                const int sl = kb / SLICE_KB, d = sl & 1;
                if (kb % SLICE_KB == 0 && sl >= 2 && !mbar_wait(&sm->dempty[d], ((sl >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (!mbar_wait(&sm->full[s], (kb / STAGES) & 1)) {
                    ok = false;
                    break;
                }
                fence_after();
                const uint64_t a0 = sdesc(su32(A + s * TILE_BYTES));
                const uint64_t b0 = sdesc(su32(B + s * TILE_BYTES));
#pragma unroll
                for (int k = 0; k < TK / 16; ++k)
                    mma_bf16(tmem + (uint32_t)(d * TN), a0 + 2 * k, b0 + 2 * k,
                             (kb % SLICE_KB != 0 || k != 0) ? 1u : 0u);
                mma_commit(&sm->empty[s]);
                if (kb % SLICE_KB == SLICE_KB - 1 || kb == KB - 1)
                    mma_commit(&sm->dfull[d]);
            }
            if (!ok)
                sm->failed = 1;
            // all MMAs issued by this thread have completed once `done` fires
            mma_commit(&sm->done);
            if (!mbar_wait(&sm->done, 0))
                sm->failed = 1;
        }
    } else {
        // epilogue: rows m0 + 32*q + lane, columns n0 .. n0+127
        const int q = warp & 3;
        int acc[TN];
#pragma unroll
        for (int j = 0; j < TN; ++j)
            acc[j] = 0;
        bool ok = true;
        for (int sl = 0; sl < NS; ++sl) {
            const int d = sl & 1;
            if (!mbar_wait(&sm->dfull[d], (sl >> 1) & 1)) {
                ok = false;
                break;
            }
            fence_after();
#pragma unroll
            for (int c = 0; c < TN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * TN + 32 * c), v);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    acc[32 * c + e] += __float2int_rn(__uint_as_float(v[e]));
            }
            fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm->dempty[d]);
        }
        if (!ok) {
            if (lane == 0)
                sm->failed = 1;
        } else {
            const float sx = flush(*s_x), sw = flush(*s_w);
            const int row = m0 + 32 * q + lane;
            if ((N & 3) == 0 && n0 + TN <= N) {
                // every MMA has completed (the last slice's barrier), so no copy or
                // MMA touches the operand ring any more: each warp stages its 32 x
                // 128 block there (pitch EPI_PITCH) and stores whole rows, 512
                // contiguous bytes per warp instruction
                float* stg = reinterpret_cast<float*>(base) + q * (32 * EPI_PITCH);
#pragma unroll
                for (int j = 0; j < TN; j += 4) {
                    float4 o;
                    o.x = fmul_flush(fmul_flush(__int2float_rn(acc[j + 0]), sx), sw);
                    o.y = fmul_flush(fmul_flush(__int2float_rn(acc[j + 1]), sx), sw);
                    o.z = fmul_flush(fmul_flush(__int2float_rn(acc[j + 2]), sx), sw);
                    o.w = fmul_flush(fmul_flush(__int2float_rn(acc[j + 3]), sx), sw);
                    *reinterpret_cast<float4*>(stg + lane * EPI_PITCH + j) = o;
                }
                __syncwarp();
                const int rows = min(32, M - (m0 + 32 * q));
                for (int r = 0; r < rows; ++r) {
                    const float4 v = *reinterpret_cast<const float4*>(stg + r * EPI_PITCH + 4 * lane);
                    *reinterpret_cast<float4*>(y + (int64_t)(m0 + 32 * q + r) * N + n0 + 4 * lane) = v;
                }
            } else if (row < M) {
                float* dst = y + (int64_t)row * N + n0;
                {
#pragma unroll
                    for (int j = 0; j < TN; ++j)
                        if (n0 + j < N)
                            dst[j] = fmul_flush(fmul_flush(__int2float_rn(acc[j]), sx), sw);
                }
            }
        }
    }

    fence_before();
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
    if (threadIdx.x == 0 && sm->failed)
        atomicExch(err, 1);
}

// int8 codes -> bf16 (exact for |q| <= 256), 16 per thread per step
__global__ void __launch_bounds__(256)
k_i8_to_bf16(const int8_t* __restrict__ q, __nv_bfloat16* __restrict__ out, int64_t n)
{
    const int64_t nv = n >> 4;
    const int4* q16 = reinterpret_cast<const int4*>(q);
    uint4* o = reinterpret_cast<uint4*>(out);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int4 w = __ldg(q16 + i);
        const int words[4] = {w.x, w.y, w.z, w.w};
        uint32_t h[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn((float)(int8_t)(words[u]),
                                                            (float)(int8_t)(words[u] >> 8));
            const __nv_bfloat162 hi = __floats2bfloat162_rn((float)(int8_t)(words[u] >> 16),
                                                            (float)(int8_t)(words[u] >> 24));
            h[2 * u] = *reinterpret_cast<const uint32_t*>(&lo);
            h[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&hi);
        }
        o[2 * i] = make_uint4(h[0], h[1], h[2], h[3]);
        o[2 * i + 1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
    if (blockIdx.x == 0) {
        const int64_t i = (nv << 4) + threadIdx.x;
        if (threadIdx.x < 16 && i < n)
            out[i] = __float2bfloat16_rn((float)q[i]);
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

// [rows x K] bf16, row-major; box 64 (K) x 128 (rows), 128-byte swizzle
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)TK, (cuuint32_t)TM};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

inline int64_t align256(int64_t b) { return (b + 255) & ~(int64_t)255; }

} // namespace

bool fwd_tc_supported(int64_t M, int64_t N, int64_t K)
{
    return M > 0 && N > 0 && K > 0 && (K % 8) == 0 && M <= 0x7fffffff / 2 &&
           N <= 0x7fffffff / 2 && K <= 133144;
}

size_t fwd_tc_ws_bytes(int64_t M, int64_t N, int64_t K)
{
    return (size_t)(align256(2 * M * K) + align256(2 * N * K));
}

cudaError_t launch_fwd_tc(const int8_t* xq, const int8_t* wq, const float* s_x, const float* s_w,
                          float* y, int64_t M, int64_t N, int64_t K, void* ws, cudaStream_t st)
{
    __nv_bfloat16* xa = static_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* wb = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) +
                                                          align256(2 * M * K));
    const int grid_c = num_sms() * 8;
    k_i8_to_bf16<<<grid_c, 256, 0, st>>>(xq, xa, M * K);
    k_i8_to_bf16<<<grid_c, 256, 0, st>>>(wq, wb, N * K);
    count_launches(2);
    CUtensorMap ma, mb;
    if (!make_map(&ma, xa, M, K) || !make_map(&mb, wb, N, K))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    int* err = device_error_word();
    if (!err)
        return cudaErrorInvalidValue;
    dim3 grid((unsigned)((N + TN - 1) / TN), (unsigned)((M + TM - 1) / TM));
    k_fwd_tc<<<grid, THREADS, SMEM_BYTES, st>>>(ma, mb, s_x, s_w, y, (int)M, (int)N, (int)K, err);
    count_launches(1);
    return cudaGetLastError();
}

} // namespace repro
