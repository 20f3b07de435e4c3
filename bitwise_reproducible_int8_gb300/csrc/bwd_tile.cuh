// bwd_tile.cuh -- the 8 x 4 packed thread tile of the default backward kernel
// (k_bwd_tma.cu): one reduction step of rounded multiplies and flushed adds,
// and the tree levels kept in tensor memory.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace repro {

typedef unsigned long long u64;

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const u64 (&v)[16])
{
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        w[2 * e] = (uint32_t)(v[e] & 0xffffffffull);
        w[2 * e + 1] = (uint32_t)(v[e] >> 32);
    }
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]),
        "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]),
        "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// acc[e] <- level[e] (+) acc[e]: the level holds the left operand
__device__ __forceinline__ void tmem_fold32(uint32_t taddr, u64 (&acc)[16])
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
        acc[e] = fadd2_ftz((u64)w[2 * e] | ((u64)w[2 * e + 1] << 32), acc[e]);
}

// one reduction step: rows 8ty..8ty+7 as 4 pairs, columns 4tx..4tx+3.  The
// products of row pair ip+1 are formed before the adds of row pair ip, so no
// add waits on the multiply just issued; every accumulator still sees its
// own product, then its one add, in the same order
template <bool FIRST>
__device__ __forceinline__ void step(u64 (&acc)[16], const ulonglong2& a03, const ulonglong2& a47,
                                     const float4& b)
{
    const u64 P[4] = {a03.x, a03.y, a47.x, a47.y};
    const u64 D[4] = {pack2(b.x, b.x), pack2(b.y, b.y), pack2(b.z, b.z), pack2(b.w, b.w)};
    u64 cur[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        cur[j] = fmul2_rn(P[0], D[j]);
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
        u64 nxt[4];
        if (ip + 1 < 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                nxt[j] = fmul2_rn(P[ip + 1], D[j]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[ip * 4 + j] = FIRST ? cur[j] : fadd2_ftz(acc[ip * 4 + j], cur[j]);
        if (ip + 1 < 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                cur[j] = nxt[j];
        }
    }
}

// the same step with the products two row pairs ahead of their adds
template <bool FIRST>
__device__ __forceinline__ void step_ahead2(u64 (&acc)[16], const ulonglong2& a03, const ulonglong2& a47,
                                            const float4& b)
{
    const u64 P[4] = {a03.x, a03.y, a47.x, a47.y};
    const u64 D[4] = {pack2(b.x, b.x), pack2(b.y, b.y), pack2(b.z, b.z), pack2(b.w, b.w)};
    u64 c0[4], c1[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        c0[j] = fmul2_rn(P[0], D[j]);
        c1[j] = fmul2_rn(P[1], D[j]);
    }
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
        u64 nx[4];
        if (ip + 2 < 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                nx[j] = fmul2_rn(P[ip + 2], D[j]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            acc[ip * 4 + j] = FIRST ? c0[j] : fadd2_ftz(acc[ip * 4 + j], c0[j]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c0[j] = c1[j];
            if (ip + 2 < 4)
                c1[j] = nx[j];
        }
    }
}

} // namespace repro
