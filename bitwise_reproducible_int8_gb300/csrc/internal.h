// internal.h -- launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments are already validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <initializer_list>

#define REPRO_MAX_PARTS_INTERNAL 64
#define REPRO_MAX_TENSORS_INTERNAL 64

namespace repro {

struct LaunchCfg {
    int bwd_segment_log2;   // chunks per backward reduction segment = 2^k (0..8)
    int reduce_block_log2;  // chunk partials per block in the scale reduction (0..10)
    int fwd_path;           // 0: CUDA-core exact path, 1: tensor cores 128 x 256 tiles, 2: 128 x 128
    int elementwise_blocks; // 0: default grid for streaming kernels
    int bwd_kernel;         // 8: tensor-copy-fed kernel (default), 1: register-prefetch kernel
    int fwd_selftest;       // -1: gate the tensor-core forward on its self-test; 1: treat it as failed
};

const LaunchCfg& launch_cfg();
// debug mode (repro_set_debug): the scans of a call's float inputs, enqueued
// before its kernels; REPRO_OK, or REPRO_ERR_LAUNCH if one could not be enqueued
struct FloatSpan {
    const float* p;
    int64_t n;
};
int scan_inputs(void* stream, std::initializer_list<FloatSpan> spans);
int num_sms();
int* device_error_word();   // device address of the error word: bit 0 a bounded wait gave up,
                            // bit 1 the debug scan found a non-finite input
constexpr int kErrTimeoutBit = 1, kErrNonfiniteBit = 2;
int arch_status();          // REPRO_OK when the current device is a GB300
void count_launches(int k); // adds k to the process-wide launch counter
// status code of a CUDA runtime result, the same for every entry point
inline int status_of(cudaError_t e) { return e == cudaSuccess ? 0 : -5; }   // REPRO_OK / REPRO_ERR_LAUNCH

// ---- scale (k_scale.cu)
size_t wscale_ws_bytes(int64_t n, int block_log2);
cudaError_t launch_wscale_meanabs(const float* x, int64_t n, int qmax, float* scale_out,
                                  void* ws, int block_log2, cudaStream_t st);
cudaError_t launch_wscale_amax(const float* x, int64_t n, int qmax, float* scale_out,
                               void* ws, int grid, cudaStream_t st);
int amax_grid(int64_t n);
// several tensors in one pass: scales[t] of xs[t] (mode 0 weight, 1 activation)
size_t wscale_multi_ws_bytes(const int64_t* ns, int count);
cudaError_t launch_wscale_multi(const float* const* xs, const int64_t* ns, int count, int mode,
                                int qmax, float* scales, void* ws, int block_log2,
                                cudaStream_t st);

cudaError_t launch_sumsq(const float* x, int64_t n, float* out, void* ws, int block_log2,
                         cudaStream_t st);

// ---- optimiser (k_optim.cu)
struct AdamWArgs {
    float lr, beta1, beta2, eps, weight_decay, max_norm;
};
cudaError_t launch_adamw(float* p, float* m, float* v, const float* g, int64_t n,
                         const float* sumsq, const AdamWArgs& h, int64_t t, int grid,
                         cudaStream_t st);

// ---- quantiser (k_quant.cu)
cudaError_t launch_quant(const float* x, int64_t n, const float* scale, int qmax, int8_t* q,
                         int grid, cudaStream_t st);
cudaError_t launch_quant_multi(const float* const* xs, const int64_t* ns, int count,
                               const float* scales, int qmax, int8_t* const* qs, int grid,
                               cudaStream_t st);

// ---- forward (k_fwd.cu)
cudaError_t launch_fwd_cuda_core(const int8_t* xq, const int8_t* wq, const float* s_x,
                                 const float* s_w, float* y, int64_t M, int64_t N, int64_t K,
                                 cudaStream_t st);

// ---- forward on tensor cores (k_fwd_tc.cu)
bool fwd_tc_supported(int64_t M, int64_t N, int64_t K);
size_t fwd_tc_ws_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_fwd_tc(const int8_t* xq, const int8_t* wq, const float* s_x, const float* s_w,
                          float* y, int64_t M, int64_t N, int64_t K, void* ws, bool wide,
                          cudaStream_t st);

// ---- backward (k_bwd.cu)
size_t bwd_ws_bytes(int64_t M, int64_t N, int64_t K, int seg_log2);
cudaError_t launch_bwd_dx(const float* dy, const int8_t* wq, const float* s_w, float* dx,
                          int64_t M, int64_t N, int64_t K, int seg_log2, float* ws,
                          cudaStream_t st);
cudaError_t launch_bwd_dw(const float* dy, const int8_t* xq, const float* s_x, float* dw,
                          int64_t M, int64_t N, int64_t K, int seg_log2, bool accumulate,
                          float* ws, cudaStream_t st);

// ---- reductions (k_reduce.cu)
cudaError_t launch_grad_accum(float* acc, const float* g, int64_t n, int grid, cudaStream_t st);
cudaError_t launch_running_sum(const float* const* parts, int S, int64_t n, float* out, int grid,
                               cudaStream_t st);
cudaError_t launch_treefold(const float* const* parts, int R, int64_t n, float* out, int grid,
                            cudaStream_t st);

// ---- attention with int8 P.V (k_attn_fwd.cu, k_attn_bwd.cu)
size_t attn_fwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W);
cudaError_t launch_attn_fwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                            float* o, float* m, float* l, int64_t B, int64_t T, int64_t Hq,
                            int64_t Hkv, int64_t W, void* cache, bool tc, cudaStream_t st);

size_t attn_bwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W);   // W = -1: without the cache
cudaError_t launch_attn_bwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                            const float* o, const float* dout, const float* m, const float* l,
                            float* dq, float* dk, float* dv, int64_t B, int64_t T, int64_t Hq,
                            int64_t Hkv, int64_t W, void* ws, const void* lcache,
                            cudaStream_t st);

// ---- bounded-wait probe (k_bwd_tma.cu)
cudaError_t launch_wait_probe(int arrive, cudaStream_t st);
// debug mode: ORs kErrNonfiniteBit into *err if any of the n floats at p is a
// NaN or an infinity
cudaError_t launch_check_finite(const float* p, int64_t n, int* err, cudaStream_t st);

// ---- forward exactness self-test (k_selftest.cu)
size_t selftest_ws_bytes();
int run_selftest(void* ws, cudaStream_t st);

// ---- state hash (k_hash.cu)
int64_t hash_leaf_count(const int64_t* nbytes, int nbuf, int64_t leaf_bytes);
size_t hash_ws_bytes(int64_t nleaves);
cudaError_t launch_state_hash(const void* const* bufs, const int64_t* nbytes, int nbuf,
                              int64_t leaf_bytes, uint8_t* digest, void* ws, cudaStream_t st);

} // namespace repro
