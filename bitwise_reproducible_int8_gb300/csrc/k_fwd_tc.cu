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
// Kernel structure: persistent, one CTA per SM, each CTA walking output tiles
// of 128 rows x TN columns (TN = 128 or 256) in a fixed round-robin order:
//   warp 0      TMA producer: bf16 A (128 x 64 K) and B (TN x 64 K) tiles,
//               128-byte swizzle, a ring of 192 KB of stages (full/empty
//               mbarriers), running straight on into the next tile;
//   warp 1      allocates all 512 TMEM columns as 512/TN fp32 accumulators of
//               TN columns, used in turn by consecutive K-slices of consecutive
//               tiles; one thread issues the MMAs (M=128, N=TN, K=16),
//               committing each stage back to the producer and each K-slice to
//               the epilogue, so the next tile's products start while the
//               epilogue is still converting and storing the last one;
//   warps 2..   epilogue, TN/32 warps: warp w reads TMEM lanes 32*(w%4) .. +31
//               (its rows) and 128 of the tile's columns, converts each slice
//               to int32 and accumulates in registers, frees the accumulator,
//               and at the tile's end scales, stages 32 x 32 blocks in its own
//               128-byte-swizzled shared buffer and writes them with TMA tensor
//               stores that drain while the next tile computes.
// Every wait is bounded (about two seconds of clock64); on expiry the kernel
// records an error in the device error word, lets in-flight copies land,
// frees tensor memory and returns.  repro_device_check reports it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "launch.cuh"
#include "pipeline.cuh"
#include "umma.cuh"

namespace repro {
namespace {

constexpr int TM = 128;            // tile rows (M)
constexpr int TK = 64;             // K per stage: one 128-byte swizzle row of bf16
constexpr int SLICE_KB = 8;        // k-blocks per exact slice: 8 * 64 = 512
constexpr int A_BYTES = TM * TK * 2;   // 16 KB
constexpr int RING_BYTES = 192 * 1024;
constexpr int STG_BYTES = 32 * 32 * 4;  // one epilogue warp's 32 x 32 fp32 staging block
constexpr uint32_t TMEM_COLS = 512;

// tile width TN = 128 (6 stages, 4 accumulators, 4 epilogue warps) or 256
// (4 stages, 2 accumulators, 8 epilogue warps, a quarter fewer operand bytes
// per multiply); each epilogue warp owns 32 rows x 128 columns of a tile
template <int TN>
struct Cfg {
    static constexpr int B_BYTES = TN * TK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = RING_BYTES / STAGE_BYTES;
    static constexpr int NBUF = (int)TMEM_COLS / TN;
    static constexpr int EPI_WARPS = TN / 32;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr size_t SMEM_BYTES = 1024 + (size_t)RING_BYTES + EPI_WARPS * STG_BYTES + 256;
    static_assert(STAGES * STAGE_BYTES == RING_BYTES, "whole stages");
    static_assert(SMEM_BYTES <= 227 * 1024, "fits one SM's shared memory");
};

constexpr int MAX_STAGES = 6, MAX_BUF = 4;
struct Smem {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t dfull[MAX_BUF];
    uint64_t dempty[MAX_BUF];
    uint64_t done;
    uint32_t tmem_base;
    int failed;
};


// 32 x 32 fp32 block from shared memory (128-byte swizzle) to Y at column x,
// row yr; the tensor map clips the parts beyond M and N
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int yr)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(yr), "r"(su32(src))
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// tile t of the CTA's round-robin walk, row-major over (row block, column block)
__device__ __forceinline__ void tile_origin(int t, int tiles_n, int tn, int& m0, int& n0)
{
    m0 = (t / tiles_n) * TM;
    n0 = (t % tiles_n) * tn;
}

// shared memory admits one CTA per SM; the second bound only caps the narrow
// tile's registers at the wide tile's 168, which keeps both free of spills
template <int TN>
__global__ void __launch_bounds__(Cfg<TN>::THREADS, TN == 128 ? 2 : 1)
k_fwd_tc(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
         const __grid_constant__ CUtensorMap map_y, int y_tma, const float* __restrict__ s_x,
         const float* __restrict__ s_w, float* __restrict__ y, int M, int N, int K,
         int* __restrict__ err)
{
    using C = Cfg<TN>;
    constexpr int STAGES = C::STAGES, NBUF = C::NBUF;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled tiles need 1024-byte alignment in the shared window
    uint8_t* base = smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u);
    uint8_t* A = base;                                   // STAGES x 16 KB
    uint8_t* B = base + STAGES * A_BYTES;                // STAGES x TN/128 x 16 KB
    uint8_t* STG = base + RING_BYTES;                    // EPI_WARPS x 4 KB
    Smem* sm = reinterpret_cast<Smem*>(STG + C::EPI_WARPS * STG_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = (N + TN - 1) / TN;
    const int tiles = ((M + TM - 1) / TM) * tiles_n;
    const int KB = (K + TK - 1) / TK;
    const int NS = (KB + SLICE_KB - 1) / SLICE_KB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->empty[s], 1);
        }
        for (int d = 0; d < NBUF; ++d) {
            mbar_init(&sm->dfull[d], 1);
            mbar_init(&sm->dempty[d], C::EPI_WARPS);
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
    // the set-up above touches no global memory; everything below may read
    // what the kernels before this one on the stream wrote
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            int g = 0;   // k-blocks issued over all of this CTA's tiles
            for (int t = blockIdx.x; t < tiles && !*(volatile int*)&sm->failed; t += gridDim.x) {
                int m0, n0;
                tile_origin(t, tiles_n, TN, m0, n0);
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int s = g % STAGES;
                    if (g >= STAGES && !mbar_wait(&sm->empty[s], ((g / STAGES) - 1) & 1)) {
                        sm->failed = 1;
                        break;
                    }
                    if (*(volatile int*)&sm->failed)
                        break;
                    mbar_expect_tx(&sm->full[s], C::STAGE_BYTES);
                    tma_load_2d(A + s * A_BYTES, &map_a, kb * TK, m0, &sm->full[s]);
                    tma_load_2d(B + s * C::B_BYTES, &map_b, kb * TK, n0, &sm->full[s]);
                }
                if (*(volatile int*)&sm->failed)
                    break;
            }
            // let the last copy into every stage land before the CTA can exit
            for (int h = g - 1; h >= 0 && h >= g - STAGES; --h)
                if (!mbar_wait(&sm->full[h % STAGES], (h / STAGES) & 1))
                    sm->failed = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            bool ok = true;
            int g = 0, sg = 0;   // k-blocks and K-slices consumed over all tiles
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb, ++g) {
                    const int s = g % STAGES;
                    const int d = sg % NBUF;
                    if (kb % SLICE_KB == 0 && sg >= NBUF &&
                        !mbar_wait(&sm->dempty[d], ((sg / NBUF) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&sm->full[s], (g / STAGES) & 1)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint64_t a0 = sdesc(su32(A + s * A_BYTES));
                    const uint64_t b0 = sdesc(su32(B + s * C::B_BYTES));
#pragma unroll
                    for (int k = 0; k < TK / 16; ++k)
                        mma_bf16<TN>(tmem + (uint32_t)(d * TN), a0 + 2 * k, b0 + 2 * k,
                                     (kb % SLICE_KB != 0 || k != 0) ? 1u : 0u);
                    mma_commit(&sm->empty[s]);
                    if (kb % SLICE_KB == SLICE_KB - 1 || kb == KB - 1) {
                        mma_commit(&sm->dfull[d]);
                        ++sg;
                    }
                }
            }
            if (!ok)
                sm->failed = 1;
            // all MMAs issued by this thread have completed once `done` fires
            mma_commit(&sm->done);
            if (!mbar_wait(&sm->done, 0))
                sm->failed = 1;
        }
    } else {
        // epilogue: rows m0 + 32*q + lane, columns n0 + 128*h .. + 127
        const int q = warp & 3;
        const int ew = warp - 2;              // epilogue warp 0 .. EPI_WARPS-1
        const int h = ew >> 2;                // column half (TN = 256)
        const float sx = flush(*s_x), sw = flush(*s_w);
        float* stg = reinterpret_cast<float*>(STG + ew * STG_BYTES);
        bool ok = true;
        int sg = 0;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
            int m0, n0;
            tile_origin(t, tiles_n, TN, m0, n0);
            const int nc = n0 + 128 * h;
            int acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j)
                acc[j] = 0;
            for (int sl = 0; sl < NS; ++sl, ++sg) {
                const int d = sg % NBUF;
                if (!mbar_wait(&sm->dfull[d], (sg / NBUF) & 1)) {
                    ok = false;
                    break;
                }
                fence_after();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t v[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * TN + 128 * h + 16 * c), v);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        acc[16 * c + e] += __float2int_rn(__uint_as_float(v[e]));
                }
                fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sm->dempty[d]);
            }
            if (!ok)
                break;
            const int r0 = m0 + 32 * q;
            if (y_tma) {
                // 32 x 32 blocks: lane writes its row's eight 16-byte chunks at
                // the 128-byte-swizzled positions (chunk k of row r at k ^ (r % 8)),
                // then one TMA store writes the block; the buffer is reused once
                // the previous store has read it
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (r0 < M && nc + 32 * c < N) {   // warp-uniform
                        if (lane == 0)
                            bulk_wait_read();
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int j = 32 * c + 4 * k;
                            float4 o;
                            o.x = fmul_flush(fmul_flush(__int2float_rn(acc[j + 0]), sx), sw);
                            o.y = fmul_flush(fmul_flush(__int2float_rn(acc[j + 1]), sx), sw);
                            o.z = fmul_flush(fmul_flush(__int2float_rn(acc[j + 2]), sx), sw);
                            o.w = fmul_flush(fmul_flush(__int2float_rn(acc[j + 3]), sx), sw);
                            *reinterpret_cast<float4*>(stg + lane * 32 + 4 * (k ^ (lane & 7))) = o;
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0)
                            tma_store_2d(&map_y, stg, nc + 32 * c, r0);
                    }
                }
            } else if (r0 + lane < M) {
                float* dst = y + (int64_t)(r0 + lane) * N + nc;
#pragma unroll
                for (int j = 0; j < 128; ++j)
                    if (nc + j < N)
                        dst[j] = fmul_flush(fmul_flush(__int2float_rn(acc[j]), sx), sw);
            }
        }
        if (!ok && lane == 0)
            sm->failed = 1;
        if (lane == 0)
            bulk_wait_all();
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
    pdl_wait();
    pdl_trigger();
    const int64_t nv = n >> 4;
    const int4* q16 = reinterpret_cast<const int4*>(q);
    uint4* o = reinterpret_cast<uint4*>(out);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int4 w = ld_stream(q16 + i);
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

// [rows x K] bf16, row-major; box 64 (K) x box_rows, 128-byte swizzle
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)TK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

inline int64_t align256(int64_t b) { return (b + 255) & ~(int64_t)255; }

// Y [M x N] fp32, row-major; box 32 x 32, 128-byte swizzle (the epilogue's
// staging layout); needs a row pitch that is a multiple of 16 bytes
bool make_y_map(CUtensorMap* map, float* y, int64_t M, int64_t N)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)N * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TN>
cudaError_t run_tile(const __nv_bfloat16* xa, const __nv_bfloat16* wb, const float* s_x,
                     const float* s_w, float* y, int64_t M, int64_t N, int64_t K, int* err,
                     cudaStream_t st)
{
    using C = Cfg<TN>;
    CUtensorMap ma, mb, my;
    memset(&my, 0, sizeof(my));
    if (!make_map(&ma, xa, M, K, TM) || !make_map(&mb, wb, N, K, TN))
        return cudaErrorInvalidValue;
    const int y_tma = (N % 4) == 0;
    if (y_tma && !make_y_map(&my, y, M, N))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_fwd_tc<TN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    const int64_t tiles = ((M + TM - 1) / TM) * ((N + TN - 1) / TN);
    const unsigned grid = (unsigned)std::min<int64_t>(tiles, num_sms());
    e = launch_pdl(k_fwd_tc<TN>, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, st, ma, mb, my, y_tma,
                   s_x, s_w, y, (int)M, (int)N, (int)K, err);
    count_launches(1);
    return e;
}

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
                          float* y, int64_t M, int64_t N, int64_t K, void* ws, bool wide,
                          cudaStream_t st)
{
    __nv_bfloat16* xa = static_cast<__nv_bfloat16*>(ws);
    __nv_bfloat16* wb = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) +
                                                          align256(2 * M * K));
    const int grid_c = num_sms() * 8;
    cudaError_t e = launch_pdl(k_i8_to_bf16, dim3(grid_c), dim3(256), 0, st, xq, xa, M * K);
    if (e == cudaSuccess)
        e = launch_pdl(k_i8_to_bf16, dim3(grid_c), dim3(256), 0, st, wq, wb, N * K);
    count_launches(2);
    if (e != cudaSuccess)
        return e;
    int* err = device_error_word();
    if (!err)
        return cudaErrorInvalidValue;
    return wide ? run_tile<256>(xa, wb, s_x, s_w, y, M, N, K, err, st)
                : run_tile<128>(xa, wb, s_x, s_w, y, M, N, K, err, st);
}

} // namespace repro
