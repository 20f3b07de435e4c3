// common.cuh -- device arithmetic of the reproducible path and small helpers.
//
// Arithmetic model (Open-1B review, onedev.kr/papers/92, section "How it
// works": fixed order, explicit unfused multiply and add, subnormals flushed on
// every backend):
//   * a product is `mul.rn.f32` -- IEEE round-to-nearest-even with gradual
//     underflow, no flush.  Every product is consumed by an `add.rn.ftz.f32`
//     (which reads a subnormal operand as a signed zero) or passed through
//     flush() before it is stored, so the flush happens exactly once, after
//     IEEE rounding, as the oracle defines it.  This keeps the result
//     independent of how a hardware flush treats results that round up to the
//     smallest normal.
//   * a sum is `add.rn.ftz.f32`: operands flushed, IEEE sum, subnormal result
//     flushed.  A sum of two values on the 2^-149 grid is exact whenever it is
//     subnormal, so this flush is unambiguous.
//   * flush(x) = x (+) -0 with the same instruction: the identity on every
//     normal value and on both zeros, and the signed zero for a subnormal.
// All inline asm is non-volatile: the operations are pure, the compiler may
// schedule them, and explicit rounding modifiers forbid any contraction.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace repro {

__device__ __forceinline__ float fmul_rn(float a, float b)
{
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float fadd_ftz(float a, float b)
{
    float r;
    asm("add.rn.ftz.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float flush(float x)
{
    return fadd_ftz(x, -0.0f);
}

// product stored or reused as an operand: round, then flush
__device__ __forceinline__ float fmul_flush(float a, float b)
{
    return flush(fmul_rn(a, b));
}

// Packed pairs (sm_100 family): two independent lanes per instruction, same
// rounding as the scalar forms.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(unsigned long long v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ unsigned long long fmul2_rn(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ unsigned long long fadd2_ftz(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// a * b + c with one rounding, gradual underflow.  Not an operation of the
// method: only for computing a correctly rounded quotient (k_attn.cuh)
__device__ __forceinline__ unsigned long long ffma2_rn(unsigned long long a, unsigned long long b,
                                                       unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// dequantised operand: float(q) (x) s, flushed (q is an exact small integer)
__device__ __forceinline__ float dequant(int q, float s)
{
    return fmul_flush(__int2float_rn(q), s);
}

// streaming 16-byte loads of data no thread writes during the kernel: the
// read-only (non-coherent) path, no L1 allocation, 256-byte L2 fetches.  On
// GB300 this took the activation-scale pass over 369 MB from 4.83 to 5.66 TB/s.
__device__ __forceinline__ float4 ld_stream(const float4* p)
{
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int4 ld_stream(const int4* p)
{
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// the same streaming hints on the coherent path, for data the kernel may also
// write (an input that aliases the output): .nc is defined only for memory
// that stays read-only for the kernel's whole lifetime
__device__ __forceinline__ float4 ld_stream_coherent(const float4* p)
{
    float4 v;
    asm volatile("ld.global.L1::no_allocate.L2::256B.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 flush4(float4 v)
{
    return make_float4(flush(v.x), flush(v.y), flush(v.z), flush(v.w));
}

} // namespace repro
