// bwd_common.cuh -- argument block and tile constants shared by the backward
// kernels (k_bwd.cu: dispatch, segments and workspace; k_bwd_tma.cu: the
// tensor-copy-fed default kernel; k_bwd_prefetch.cu: the kernel for rows that
// are not 16-byte aligned).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace repro {

constexpr int BT = 64;       // output tile width (j) and the square tile edge
constexpr int CH = 64;       // chunk length of the canonical order
constexpr int MAXLVL = 8;    // tree stack levels: up to 256 chunks per segment

// C[i,j] = canon_r( A[r,i] (x) B[r,j] ), A from dY, B = q (x) s
struct BwdArgs {
    const float* dy;
    const int8_t* q;
    const float* scale;
    float* out;
    float* ws;
    int64_t I, J, R;   // output rows, output columns, reduction length
    int64_t ldy;       // row stride of dY (= N)
    int seg_log2;
    int nseg;
    int accumulate;
    int* err;          // device error word (bounded waits)
};

// tensor-copy-fed kernel (k_bwd_tma.cu): 128 x 64 output tile per CTA, needs
// 16-byte-aligned rows (ldy % 4 == 0, J % 16 == 0); prepares its operands (flushed dY, dequantised int8
// operand) in `opnd`, a 256-byte aligned workspace region of
// bwd_tma_operand_bytes(M, N, K) bytes
constexpr int BWD_TMA_ROWS = 128;
size_t bwd_tma_operand_bytes(int64_t M, int64_t N, int64_t K);
template <bool DW>
cudaError_t launch_bwd_tma(const BwdArgs& a, const int8_t* q, float* opnd, dim3 grid,
                           cudaStream_t st);

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// register-prefetch kernel (k_bwd_prefetch.cu): 64 x 64 output tile per CTA,
// any row alignment; grid (J tiles, I tiles, segments)
template <bool DW>
cudaError_t launch_bwd_prefetch(const BwdArgs& a, cudaStream_t st);

} // namespace repro
