// bwd_common.cuh -- argument block and tile constants shared by the backward
// kernels (k_bwd.cu: single-role kernels; k_bwd_ws.cu: warp-specialised kernel;
// k_bwd_tma.cu: tensor-copy-fed kernel).
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

// warp-specialised kernel (k_bwd_ws.cu): 128 x 64 output tile per CTA, needs
// 16-byte-aligned rows (ldy % 4 == 0, J % 16 == 0)
constexpr int BWD_WS_ROWS = 128;
template <bool DW>
cudaError_t launch_bwd_ws(const BwdArgs& a, dim3 grid, cudaStream_t st);

// tensor-copy-fed kernel (k_bwd_tma.cu): 128 x 64 output tile per CTA, same
// alignment needs; prepares its operands (flushed dY, dequantised int8
// operand) in `opnd`, a 256-byte aligned workspace region of
// bwd_tma_operand_bytes(M, N, K) bytes.  self_issue: the compute warps issue
// the copies themselves (no producer warp, three tree levels in registers)
constexpr int BWD_TMA_ROWS = 128;
size_t bwd_tma_operand_bytes(int64_t M, int64_t N, int64_t K);
template <bool DW>
cudaError_t launch_bwd_tma(const BwdArgs& a, const int8_t* q, float* opnd, dim3 grid,
                           bool self_issue, cudaStream_t st);

// tile heights of the staged wide variants (k_bwd_staged.cu): 3 and 4, and 5
constexpr int BWD_WIDE_ROWS = 128;
constexpr int BWD_WIDE12_ROWS = 192;

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// variants 0-5 (k_bwd_staged.cu): launches variant `kernel` over a's outputs,
// grid (J tiles, I tiles, segments)
template <bool DW>
cudaError_t launch_bwd_staged(int kernel, const BwdArgs& a, cudaStream_t st);

} // namespace repro
