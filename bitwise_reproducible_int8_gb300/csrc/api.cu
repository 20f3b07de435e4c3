// api.cu -- the C ABI declared in include/repro.h: argument validation,
// architecture check, workspace sizing and dispatch to the kernels.  No call
// allocates device memory; every call enqueues on the caller's stream.
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <initializer_list>

#include "internal.h"
#include "repro.h"

namespace repro {

namespace {

constexpr int kDefaultBwdKernel = 8;   // operand prep + tensor-copy-fed kernel
LaunchCfg g_cfg = {-1, -1, -1, 0, kDefaultBwdKernel, -1};

constexpr int kMaxDevices = 64;
int g_arch_ok[kMaxDevices];   // 0 unknown, 1 GB300, -1 other
int g_sms[kMaxDevices];

__device__ int g_device_error;   // set by bounded device-side waits

// exactness of the tensor-core forward on each device: 0 not checked yet,
// 1 the self-test passed, -1 it failed (every forward then takes the exact
// CUDA-core path); and a failure that repro_device_check has not reported yet
std::atomic<int> g_tc_state[kMaxDevices];
std::atomic<int> g_tc_notice[kMaxDevices];

unsigned long long g_launches;    // kernels enqueued by this library

std::atomic<int> g_debug{0};      // repro_set_debug flags

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    return dev;
}

} // namespace

const LaunchCfg& launch_cfg() { return g_cfg; }

int num_sms()
{
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices)
        return 152;
    if (g_sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 152;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

void count_launches(int k) { __atomic_fetch_add(&g_launches, (unsigned long long)k, __ATOMIC_RELAXED); }

int scan_inputs(void* stream, std::initializer_list<FloatSpan> spans)
{
    if ((g_debug.load(std::memory_order_relaxed) & REPRO_DEBUG_CHECK_FINITE) == 0)
        return REPRO_OK;
    int* err = device_error_word();
    if (!err)
        return REPRO_ERR_LAUNCH;
    for (const FloatSpan& f : spans)
        if (f.p && f.n > 0 &&
            launch_check_finite(f.p, f.n, err, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return REPRO_ERR_LAUNCH;
    return REPRO_OK;
}

int* device_error_word()
{
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess)
        return nullptr;
    return static_cast<int*>(p);
}

} // namespace repro

using namespace repro;

namespace {

int check_arch()
{
    const int dev = current_device();
    if (dev < 0)
        return REPRO_ERR_LAUNCH;
    if (dev >= kMaxDevices)
        return REPRO_ERR_ARCH;
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return REPRO_ERR_LAUNCH;
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_arch_ok[dev] == 1 ? REPRO_OK : REPRO_ERR_ARCH;
}

// output rows are tiled 64 per CTA along grid.y (at most 65535 tiles)
constexpr int64_t kMaxRows = 65535LL * 64;

inline bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline bool al4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

inline bool overlap(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0)
        return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// grid of a streaming kernel: one 256-thread CTA per 256 work items, at most
// ctas_per_sm per SM (the launch-configuration hook overrides it)
int stream_grid(int64_t work_items, int ctas_per_sm = 8)
{
    const int cfg = g_cfg.elementwise_blocks;
    if (cfg > 0)
        return cfg;
    const int64_t cap = (int64_t)num_sms() * ctas_per_sm;
    const int64_t want = (work_items + 255) / 256;
    return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

// -1: chosen per shape by the backward launcher
int seg_log2() { return g_cfg.bwd_segment_log2; }

// tensor-core forward for every supported shape unless the launch
// configuration asks for the CUDA-core path
bool use_tc(int64_t M, int64_t N, int64_t K)
{
    return g_cfg.fwd_path != 0 && fwd_tc_supported(M, N, K);
}

// 1 when the current device's exactness check has passed (the test hook's
// forced failure aside), else 0; never runs the check
int tc_state_passed()
{
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices || g_cfg.fwd_selftest == 1)
        return 0;
    return g_tc_state[dev].load() > 0 ? 1 : 0;
}

// Whether a default-path forward may use the tensor cores on the current
// device: 1 yes, 0 take the CUDA-core path, negative a CUDA error.  The first
// call on a device runs the exactness self-test in `ws` (at least
// selftest_ws_bytes()) and synchronises `stream`; a call made while `stream`
// is being captured cannot, so before the check has run it takes the exact
// CUDA-core path.
int tc_gate(void* ws, cudaStream_t stream)
{
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices)
        return -1;
    if (g_cfg.fwd_selftest == 1) {   // test hook: act as if the check had failed
        g_tc_notice[dev].store(1);
        return 0;
    }
    const int state = g_tc_state[dev].load();
    if (state != 0)
        return state > 0 ? 1 : 0;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess)
        return -1;
    if (cs != cudaStreamCaptureStatusNone)
        return 0;
    const int r = run_selftest(ws, stream);
    if (r < 0)
        return -1;
    g_tc_state[dev].store(r == 0 ? 1 : -1);
    if (r != 0)
        g_tc_notice[dev].store(1);
    return r == 0 ? 1 : 0;
}

} // namespace

namespace repro {
int arch_status() { return check_arch(); }
} // namespace repro

extern "C" {

const char* repro_status_str(int s)
{
    switch (s) {
    case REPRO_OK: return "ok";
    case REPRO_ERR_ARG: return "invalid argument (null pointer, mode, flag, q_max or R)";
    case REPRO_ERR_SHAPE: return "invalid shape";
    case REPRO_ERR_ALIGN: return "device pointer not aligned (16 bytes for tensors, 4 for scales)";
    case REPRO_ERR_ARCH: return "current device is not a GB300 (compute capability 10.3)";
    case REPRO_ERR_LAUNCH: return "CUDA runtime error while enqueueing";
    case REPRO_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case REPRO_ERR_WORKSPACE: return "workspace missing or too small";
    case REPRO_ERR_ALIAS: return "buffers that must not overlap do";
    case REPRO_ERR_SELFTEST: return "the tensor-core forward differs from the exact CUDA-core forward";
    case REPRO_ERR_NONFINITE: return "debug mode: a float input held a NaN or an infinity";
    default: return "unknown status";
    }
}

int repro_version(void) { return REPRO_VERSION; }

uint64_t repro_launch_count(void) { return (uint64_t)__atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

int repro_set_debug(int flags)
{
    if (flags & ~REPRO_DEBUG_CHECK_FINITE)
        return REPRO_ERR_ARG;
    g_debug.store(flags, std::memory_order_relaxed);
    return REPRO_OK;
}

int repro_set_launch_cfg(const repro_launch_cfg* cfg)
{
    if (!cfg) {
        g_cfg = LaunchCfg{-1, -1, -1, 0, kDefaultBwdKernel, -1};
        return REPRO_OK;
    }
    if (cfg->bwd_segment_log2 < -1 || cfg->bwd_segment_log2 > 8)
        return REPRO_ERR_ARG;
    if (cfg->reduce_block_log2 < -1 || cfg->reduce_block_log2 > 10)
        return REPRO_ERR_ARG;
    if (cfg->fwd_path < -1 || cfg->fwd_path > 2)
        return REPRO_ERR_ARG;
    if (cfg->elementwise_blocks < -1 || cfg->elementwise_blocks > (1 << 20))
        return REPRO_ERR_ARG;
    if (cfg->bwd_kernel != -1 && cfg->bwd_kernel != 1 && cfg->bwd_kernel != 8)
        return REPRO_ERR_ARG;
    if (cfg->fwd_selftest != -1 && cfg->fwd_selftest != 1)
        return REPRO_ERR_ARG;
    g_cfg.bwd_segment_log2 = cfg->bwd_segment_log2;
    g_cfg.reduce_block_log2 = cfg->reduce_block_log2;
    g_cfg.fwd_path = cfg->fwd_path;
    g_cfg.elementwise_blocks = cfg->elementwise_blocks < 0 ? 0 : cfg->elementwise_blocks;
    g_cfg.bwd_kernel = cfg->bwd_kernel < 0 ? kDefaultBwdKernel : cfg->bwd_kernel;
    g_cfg.fwd_selftest = cfg->fwd_selftest;
    return REPRO_OK;
}

size_t repro_selftest_ws_bytes(void)
{
    return selftest_ws_bytes();
}

int repro_selftest(void* ws, size_t ws_bytes, void* stream)
{
    if (!ws || ws_bytes < selftest_ws_bytes())
        return REPRO_ERR_WORKSPACE;
    if (!al16(ws))
        return REPRO_ERR_ALIGN;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    const int r = run_selftest(ws, as_stream(stream));
    if (r < 0)
        return REPRO_ERR_LAUNCH;
    const int dev = current_device();
    if (dev >= 0 && dev < kMaxDevices)
        g_tc_state[dev].store(r == 0 ? 1 : -1);   // the forward's gate uses this result
    return r == 0 ? REPRO_OK : REPRO_ERR_SELFTEST;
}

int repro_wait_probe(int arrive, void* stream)
{
    if (arrive != 0 && arrive != 1)
        return REPRO_ERR_ARG;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    return launch_wait_probe(arrive, as_stream(stream)) == cudaSuccess ? REPRO_OK
                                                                       : REPRO_ERR_LAUNCH;
}

int repro_device_check(void* stream)
{
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess)
        return REPRO_ERR_LAUNCH;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess)
        return REPRO_ERR_LAUNCH;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess)
            return REPRO_ERR_LAUNCH;
        return (v & kErrTimeoutBit) || !(v & kErrNonfiniteBit) ? REPRO_ERR_TIMEOUT : REPRO_ERR_NONFINITE;
    }
    const int dev = current_device();
    if (dev >= 0 && dev < kMaxDevices && g_tc_notice[dev].exchange(0) != 0)
        return REPRO_ERR_SELFTEST;
    return REPRO_OK;
}

size_t repro_wscale_ws_bytes(int64_t n)
{
    if (n <= 0)
        return 0;
    return wscale_ws_bytes(n, 0);   // the largest over every launch configuration
}

int repro_wscale(const float* x, int64_t n, int mode, int qmax, float* scale_out, void* ws,
                 size_t ws_bytes, void* stream)
{
    if (!x || !scale_out)
        return REPRO_ERR_ARG;
    if (mode != REPRO_SCALE_WEIGHT_MEANABS && mode != REPRO_SCALE_ACT_AMAX)
        return REPRO_ERR_ARG;
    if (qmax != REPRO_QMAX)
        return REPRO_ERR_ARG;
    if (n <= 0)
        return REPRO_ERR_SHAPE;
    if (!al16(x) || !al4(scale_out))
        return REPRO_ERR_ALIGN;
    if (!ws || ws_bytes < repro_wscale_ws_bytes(n))
        return REPRO_ERR_WORKSPACE;
    if (!al16(ws))
        return REPRO_ERR_ALIGN;
    if (overlap(ws, ws_bytes, x, (size_t)n * 4) || overlap(ws, ws_bytes, scale_out, 4))
        return REPRO_ERR_ALIAS;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{x, n}})) != REPRO_OK)
        return st;
    if (mode == REPRO_SCALE_WEIGHT_MEANABS)
        return status_of(launch_wscale_meanabs(x, n, qmax, scale_out, ws, g_cfg.reduce_block_log2,
                                               as_stream(stream)));
    // the launch-configuration hook may set the grid; the workspace holds at
    // least ceil(n / 64) + 64 per-CTA partials, so the grid is capped there
    int grid = amax_grid(n);
    if (g_cfg.elementwise_blocks > 0) {
        const int64_t cap = (n + 63) / 64 + 64;
        grid = (int)(g_cfg.elementwise_blocks < cap ? g_cfg.elementwise_blocks : cap);
    }
    return status_of(launch_wscale_amax(x, n, qmax, scale_out, ws, grid, as_stream(stream)));
}

int repro_quant_i8(const float* x, int64_t n, const float* scale, int qmax, int8_t* q_out,
                   void* stream)
{
    if (qmax != REPRO_QMAX)
        return REPRO_ERR_ARG;
    if (n < 0)
        return REPRO_ERR_SHAPE;
    if (n == 0)
        return REPRO_OK;
    if (!x || !scale || !q_out)
        return REPRO_ERR_ARG;
    if (!al16(x) || !al16(q_out) || !al4(scale))
        return REPRO_ERR_ALIGN;
    if (overlap(q_out, (size_t)n, x, (size_t)n * 4) || overlap(q_out, (size_t)n, scale, 4))
        return REPRO_ERR_ALIAS;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{x, n}, {scale, 1}})) != REPRO_OK)
        return st;
    // up to 32 CTAs per SM: on GB300 the quantiser streams 92M elements in 78.5 us
    // this way against 90.8 us with the grid capped at one resident wave
    return status_of(launch_quant(x, n, scale, qmax, q_out, stream_grid(n / 16, 32),
                                  as_stream(stream)));
}

size_t repro_wscale_multi_ws_bytes(const int64_t* ns, int count)
{
    if (!ns || count < 1 || count > REPRO_MAX_TENSORS)
        return 0;
    for (int t = 0; t < count; ++t)
        if (ns[t] <= 0)
            return 0;
    return wscale_multi_ws_bytes(ns, count);
}

int repro_wscale_multi(const float* const* xs, const int64_t* ns, int count, int mode, int qmax,
                       float* scales_out, void* ws, size_t ws_bytes, void* stream)
{
    if (!xs || !ns || !scales_out || count < 1 || count > REPRO_MAX_TENSORS)
        return REPRO_ERR_ARG;
    if (mode != REPRO_SCALE_WEIGHT_MEANABS && mode != REPRO_SCALE_ACT_AMAX)
        return REPRO_ERR_ARG;
    if (qmax != REPRO_QMAX)
        return REPRO_ERR_ARG;
    for (int t = 0; t < count; ++t) {
        if (!xs[t])
            return REPRO_ERR_ARG;
        if (ns[t] <= 0)
            return REPRO_ERR_SHAPE;
        if (!al16(xs[t]))
            return REPRO_ERR_ALIGN;
    }
    if (!al4(scales_out))
        return REPRO_ERR_ALIGN;
    const size_t need = wscale_multi_ws_bytes(ns, count);
    if (!ws || ws_bytes < need)
        return REPRO_ERR_WORKSPACE;
    if (!al16(ws))
        return REPRO_ERR_ALIGN;
    const size_t sb = (size_t)count * 4;
    if (overlap(ws, ws_bytes, scales_out, sb))
        return REPRO_ERR_ALIAS;
    for (int t = 0; t < count; ++t)
        if (overlap(ws, ws_bytes, xs[t], (size_t)ns[t] * 4) ||
            overlap(scales_out, sb, xs[t], (size_t)ns[t] * 4))
            return REPRO_ERR_ALIAS;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    for (int t = 0; t < count; ++t)
        if ((st = scan_inputs(stream, {{xs[t], ns[t]}})) != REPRO_OK)
            return st;
    return status_of(launch_wscale_multi(xs, ns, count, mode, qmax, scales_out, ws,
                                         g_cfg.reduce_block_log2, as_stream(stream)));
}

int repro_quant_i8_multi(const float* const* xs, const int64_t* ns, int count,
                         const float* scales, int qmax, int8_t* const* q_outs, void* stream)
{
    if (!xs || !ns || !q_outs || !scales || count < 1 || count > REPRO_MAX_TENSORS)
        return REPRO_ERR_ARG;
    if (qmax != REPRO_QMAX)
        return REPRO_ERR_ARG;
    int64_t total = 0;
    for (int t = 0; t < count; ++t) {
        if (ns[t] < 0)
            return REPRO_ERR_SHAPE;
        if (ns[t] == 0)
            continue;
        if (!xs[t] || !q_outs[t])
            return REPRO_ERR_ARG;
        if (!al16(xs[t]) || !al16(q_outs[t]))
            return REPRO_ERR_ALIGN;
        total += ns[t];
    }
    if (!al4(scales))
        return REPRO_ERR_ALIGN;
    const size_t sb = (size_t)count * 4;
    for (int t = 0; t < count; ++t) {
        if (ns[t] == 0)
            continue;
        if (overlap(q_outs[t], (size_t)ns[t], scales, sb))
            return REPRO_ERR_ALIAS;
        for (int u = 0; u < count; ++u) {
            if (ns[u] == 0)
                continue;
            if (overlap(q_outs[t], (size_t)ns[t], xs[u], (size_t)ns[u] * 4) ||
                (u != t && overlap(q_outs[t], (size_t)ns[t], q_outs[u], (size_t)ns[u])))
                return REPRO_ERR_ALIAS;
        }
    }
    if (total == 0)
        return REPRO_OK;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    for (int t = 0; t < count; ++t)
        if ((st = scan_inputs(stream, {{xs[t], ns[t]}})) != REPRO_OK)
            return st;
    if ((st = scan_inputs(stream, {{scales, count}})) != REPRO_OK)
        return st;
    return status_of(launch_quant_multi(xs, ns, count, scales, qmax, q_outs,
                                        stream_grid(total / 16, 32), as_stream(stream)));
}

// tensor-core shapes: the bf16 copies, and room for the once-per-device
// exactness check that may run first
static size_t fwd_ws_need(int64_t M, int64_t N, int64_t K)
{
    const size_t a = fwd_tc_ws_bytes(M, N, K), b = selftest_ws_bytes();
    return a > b ? a : b;
}

size_t repro_linear_fwd_ws_bytes(int64_t M, int64_t N, int64_t K)
{
    if (!use_tc(M, N, K))
        return 0;
    return fwd_ws_need(M, N, K);
}

int repro_linear_fwd(const int8_t* xq, const int8_t* wq, const float* s_x, const float* s_w,
                     float* y, int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes,
                     void* stream)
{
    if (M < 0 || N < 0 || K < 0 || K > 133144 || M > kMaxRows || N > kMaxRows)
        return REPRO_ERR_SHAPE;
    if (M == 0 || N == 0)
        return REPRO_OK;
    if (!y || !s_x || !s_w || (K > 0 && (!xq || !wq)))
        return REPRO_ERR_ARG;
    if (!al16(y) || (xq && !al16(xq)) || (wq && !al16(wq)) || !al4(s_x) || !al4(s_w))
        return REPRO_ERR_ALIGN;
    const size_t ybytes = (size_t)(M * N) * 4;
    if (overlap(y, ybytes, xq, (size_t)(M * K)) || overlap(y, ybytes, wq, (size_t)(N * K)) ||
        overlap(y, ybytes, s_x, 4) || overlap(y, ybytes, s_w, 4))
        return REPRO_ERR_ALIAS;
    bool tc = use_tc(M, N, K);
    if (tc) {
        const size_t need = fwd_ws_need(M, N, K);
        if (!ws || ws_bytes < need)
            return REPRO_ERR_WORKSPACE;
        if (!al16(ws))
            return REPRO_ERR_ALIGN;
        if (overlap(ws, ws_bytes, y, ybytes) || overlap(ws, ws_bytes, xq, (size_t)(M * K)) ||
            overlap(ws, ws_bytes, wq, (size_t)(N * K)) || overlap(ws, ws_bytes, s_x, 4) ||
            overlap(ws, ws_bytes, s_w, 4))
            return REPRO_ERR_ALIAS;
    }
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{s_x, 1}, {s_w, 1}})) != REPRO_OK)
        return st;
    if (tc && g_cfg.fwd_path < 1) {   // the default path is gated; explicit tile paths are not
        const int gate = tc_gate(ws, as_stream(stream));
        if (gate < 0)
            return REPRO_ERR_LAUNCH;
        tc = gate == 1;
    }
    if (tc)
        return status_of(launch_fwd_tc(xq, wq, s_x, s_w, y, M, N, K, ws, g_cfg.fwd_path != 2,
                                       as_stream(stream)));
    return status_of(launch_fwd_cuda_core(xq, wq, s_x, s_w, y, M, N, K, as_stream(stream)));
}

size_t repro_linear_bwd_ws_bytes(int64_t M, int64_t N, int64_t K)
{
    if (M <= 0 || N <= 0 || K <= 0)
        return 0;
    return bwd_ws_bytes(M, N, K, seg_log2());
}

int repro_linear_bwd(const float* dy, const int8_t* xq, const int8_t* wq, const float* s_x,
                     const float* s_w, float* dx, float* dw, int64_t M, int64_t N, int64_t K,
                     int flags, void* ws, size_t ws_bytes, void* stream)
{
    if (flags & ~REPRO_BWD_DW_ACCUMULATE)
        return REPRO_ERR_ARG;
    if (M < 0 || N < 0 || K < 0 || M > kMaxRows || N > kMaxRows || K > kMaxRows * 64)
        return REPRO_ERR_SHAPE;
    if (!dx && !dw)
        return REPRO_ERR_ARG;
    const bool want_dx = dx && M > 0 && K > 0;
    const bool want_dw = dw && N > 0 && K > 0;
    if (!want_dx && !want_dw)
        return REPRO_OK;
    if ((want_dx && N > 0 && (!dy || !wq || !s_w)) || (want_dw && M > 0 && (!dy || !xq || !s_x)))
        return REPRO_ERR_ARG;
    if ((dy && !al16(dy)) || (xq && !al16(xq)) || (wq && !al16(wq)) || (dx && !al16(dx)) ||
        (dw && !al16(dw)) || (s_x && !al4(s_x)) || (s_w && !al4(s_w)))
        return REPRO_ERR_ALIGN;
    const size_t dyb = (size_t)(M * N) * 4, xqb = (size_t)(M * K), wqb = (size_t)(N * K);
    const size_t dxb = want_dx ? (size_t)(M * K) * 4 : 0, dwb = want_dw ? (size_t)(N * K) * 4 : 0;
    if (overlap(dx, dxb, dy, dyb) || overlap(dx, dxb, xq, xqb) || overlap(dx, dxb, wq, wqb) ||
        overlap(dw, dwb, dy, dyb) || overlap(dw, dwb, xq, xqb) || overlap(dw, dwb, wq, wqb) ||
        overlap(dx, dxb, dw, dwb) || overlap(dx, dxb, s_x, 4) || overlap(dx, dxb, s_w, 4) ||
        overlap(dw, dwb, s_x, 4) || overlap(dw, dwb, s_w, 4))
        return REPRO_ERR_ALIAS;
    const int sl = seg_log2();
    const size_t need = bwd_ws_bytes(M, N, K, sl);
    if (need > 0) {
        if (!ws || ws_bytes < need)
            return REPRO_ERR_WORKSPACE;
        if (!al16(ws))
            return REPRO_ERR_ALIGN;
        if (overlap(ws, ws_bytes, dx, dxb) || overlap(ws, ws_bytes, dw, dwb) ||
            overlap(ws, ws_bytes, dy, dyb) || overlap(ws, ws_bytes, xq, xqb) ||
            overlap(ws, ws_bytes, wq, wqb) || overlap(ws, ws_bytes, s_x, 4) ||
            overlap(ws, ws_bytes, s_w, 4))
            return REPRO_ERR_ALIAS;
    }
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{dy, M * N}, {want_dw ? s_x : nullptr, 1}, {want_dx ? s_w : nullptr, 1}})) != REPRO_OK)
        return st;
    cudaStream_t s = as_stream(stream);
    if (want_dx) {
        cudaError_t e = launch_bwd_dx(dy, wq, s_w, dx, M, N, K, sl, static_cast<float*>(ws), s);
        if (e != cudaSuccess)
            return REPRO_ERR_LAUNCH;
    }
    if (want_dw) {
        cudaError_t e = launch_bwd_dw(dy, xq, s_x, dw, M, N, K, sl,
                                      (flags & REPRO_BWD_DW_ACCUMULATE) != 0,
                                      static_cast<float*>(ws), s);
        if (e != cudaSuccess)
            return REPRO_ERR_LAUNCH;
    }
    return REPRO_OK;
}

int repro_grad_accum(float* acc, const float* g, int64_t n, void* stream)
{
    if (n < 0)
        return REPRO_ERR_SHAPE;
    if (n == 0)
        return REPRO_OK;
    if (!acc || !g)
        return REPRO_ERR_ARG;
    if (!al16(acc) || !al16(g))
        return REPRO_ERR_ALIGN;
    if (overlap(acc, (size_t)n * 4, g, (size_t)n * 4))
        return REPRO_ERR_ALIAS;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{acc, n}, {g, n}})) != REPRO_OK)
        return st;
    return status_of(launch_grad_accum(acc, g, n, stream_grid(n / 4), as_stream(stream)));
}

size_t repro_sumsq_ws_bytes(int64_t n)
{
    if (n <= 0)
        return 0;
    return wscale_ws_bytes(n, 0);
}

int repro_sumsq(const float* g, int64_t n, float* out, void* ws, size_t ws_bytes, void* stream)
{
    if (!g || !out)
        return REPRO_ERR_ARG;
    if (n <= 0)
        return REPRO_ERR_SHAPE;
    if (!al16(g) || !al4(out))
        return REPRO_ERR_ALIGN;
    if (!ws || ws_bytes < repro_sumsq_ws_bytes(n))
        return REPRO_ERR_WORKSPACE;
    if (!al16(ws))
        return REPRO_ERR_ALIGN;
    if (overlap(ws, ws_bytes, g, (size_t)n * 4) || overlap(ws, ws_bytes, out, 4))
        return REPRO_ERR_ALIAS;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{g, n}})) != REPRO_OK)
        return st;
    return status_of(launch_sumsq(g, n, out, ws, g_cfg.reduce_block_log2, as_stream(stream)));
}

int repro_adamw_step(float* p, float* m, float* v, const float* g, int64_t n, const float* sumsq,
                     const repro_adamw_hparams* hp, int64_t t, void* stream)
{
    if (!hp || t < 1)
        return REPRO_ERR_ARG;
    if (n < 0)
        return REPRO_ERR_SHAPE;
    if (n == 0)
        return REPRO_OK;
    if (!p || !m || !v || !g || !sumsq)
        return REPRO_ERR_ARG;
    if (!al16(p) || !al16(m) || !al16(v) || !al16(g) || !al4(sumsq))
        return REPRO_ERR_ALIGN;
    const size_t nb = (size_t)n * 4;
    if (overlap(p, nb, m, nb) || overlap(p, nb, v, nb) || overlap(m, nb, v, nb) ||
        overlap(g, nb, p, nb) || overlap(g, nb, m, nb) || overlap(g, nb, v, nb) ||
        overlap(sumsq, 4, p, nb) || overlap(sumsq, 4, m, nb) || overlap(sumsq, 4, v, nb))
        return REPRO_ERR_ALIAS;
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{p, n}, {m, n}, {v, n}, {g, n}, {sumsq, 1}})) != REPRO_OK)
        return st;
    AdamWArgs h{hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_norm};
    return status_of(launch_adamw(p, m, v, g, n, sumsq, h, t, stream_grid(n / 4), as_stream(stream)));
}

// shared checks of the multi-input folds (running sum, TreeFold)
static int check_parts(const float* const* parts, int count, int64_t n, const float* out)
{
    if (!parts || count < 1 || count > REPRO_MAX_REPLICAS)
        return REPRO_ERR_ARG;
    if (n < 0)
        return REPRO_ERR_SHAPE;
    if (!out)
        return REPRO_ERR_ARG;
    for (int r = 0; r < count; ++r) {
        if (!parts[r])
            return REPRO_ERR_ARG;
        if (!al16(parts[r]))
            return REPRO_ERR_ALIGN;
    }
    if (!al16(out))
        return REPRO_ERR_ALIGN;
    const size_t nb = (size_t)n * 4;
    for (int r = 0; r < count; ++r) {
        if (r == 0 && parts[0] == out)
            continue;
        if (overlap(out, nb, parts[r], nb))
            return REPRO_ERR_ALIAS;
    }
    return REPRO_OK;
}

int repro_running_sum(const float* const* parts, int S, int64_t n, float* out, void* stream)
{
    int st = check_parts(parts, S, n, out);
    if (st != REPRO_OK || n == 0)
        return st;
    st = check_arch();
    if (st != REPRO_OK)
        return st;
    for (int r = 0; r < S; ++r)
        if ((st = scan_inputs(stream, {{parts[r], n}})) != REPRO_OK)
            return st;
    return status_of(launch_running_sum(parts, S, n, out, stream_grid(n / 4), as_stream(stream)));
}

int repro_treefold(const float* const* parts, int R, int64_t n, float* out, void* stream)
{
    if (!parts || R < 1 || R > REPRO_MAX_REPLICAS)
        return REPRO_ERR_ARG;
    if (n < 0)
        return REPRO_ERR_SHAPE;
    if (!out)
        return REPRO_ERR_ARG;
    for (int r = 0; r < R; ++r) {
        if (!parts[r])
            return REPRO_ERR_ARG;
        if (!al16(parts[r]))
            return REPRO_ERR_ALIGN;
    }
    if (!al16(out))
        return REPRO_ERR_ALIGN;
    if (n == 0)
        return REPRO_OK;
    const size_t nb = (size_t)n * 4;
    for (int r = 0; r < R; ++r) {
        if (r == 0 && parts[0] == out)
            continue;
        if (overlap(out, nb, parts[r], nb))
            return REPRO_ERR_ALIAS;
    }
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    for (int r = 0; r < R; ++r)
        if ((st = scan_inputs(stream, {{parts[r], n}})) != REPRO_OK)
            return st;
    return status_of(launch_treefold(parts, R, n, out, stream_grid(n / 4), as_stream(stream)));
}

size_t repro_attn_fwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W)
{
    if (B <= 0 || T <= 0 || Hq <= 0 || W < 0 || T > REPRO_ATTN_MAX_T)
        return 0;
    return attn_fwd_ws_bytes(B, T, Hq, W);
}

int repro_attn_fwd(const float* q, const float* k, const int8_t* vq, const float* s_v, float* o,
                   float* m, float* l, int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                   int64_t W, void* ws, size_t ws_bytes, void* stream)
{
    if (B < 0 || T < 0 || Hq < 1 || Hkv < 1 || W < 0)
        return REPRO_ERR_SHAPE;
    if (D != REPRO_ATTN_HEAD_DIM || Hq % Hkv != 0 || T > REPRO_ATTN_MAX_T || Hq > 65535 ||
        B > 65535)
        return REPRO_ERR_SHAPE;
    if (!q || !k || !vq || !s_v || !o || !m || !l)
        return REPRO_ERR_ARG;
    if (!al16(q) || !al16(k) || !al16(vq) || !al16(o) || !al4(s_v) || !al4(m) || !al4(l))
        return REPRO_ERR_ALIGN;
    if (B == 0 || T == 0)
        return REPRO_OK;
    const size_t nq = (size_t)(B * T * Hq * D) * 4, nk = (size_t)(B * T * Hkv * D);
    const size_t nr = (size_t)(B * T * Hq) * 4;
    if (overlap(o, nq, q, nq) || overlap(o, nq, k, nk * 4) || overlap(o, nq, vq, nk) ||
        overlap(m, nr, o, nq) || overlap(l, nr, o, nq) || overlap(m, nr, l, nr) ||
        overlap(m, nr, q, nq) || overlap(l, nr, q, nq) || overlap(m, nr, k, nk * 4) ||
        overlap(l, nr, k, nk * 4) || overlap(m, nr, vq, nk) || overlap(l, nr, vq, nk) ||
        overlap(o, nq, s_v, 4) || overlap(m, nr, s_v, 4) || overlap(l, nr, s_v, 4))
        return REPRO_ERR_ALIAS;
    if (ws) {
        const size_t need = attn_fwd_ws_bytes(B, T, Hq, W);
        if (ws_bytes < need)
            return REPRO_ERR_WORKSPACE;
        if (!al16(ws))
            return REPRO_ERR_ALIGN;
        const void* bufs[7] = {q, k, vq, s_v, o, m, l};
        const size_t sz[7] = {nq, nk * 4, nk, 4, nq, nr, nr};
        for (int x = 0; x < 7; ++x)
            if (overlap(ws, need, bufs[x], sz[x]))
                return REPRO_ERR_ALIAS;
    }
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{q, B * T * Hq * D}, {k, B * T * Hkv * D}, {s_v, 1}})) != REPRO_OK)
        return st;
    // P.V on the tensor cores needs the logit cache and a device whose exactness
    // check has passed (run here, in the cache's space, if it has not run yet)
    bool tc = false;
    if (ws && g_cfg.fwd_path != 0) {
        const int gate = ws_bytes >= selftest_ws_bytes() ? tc_gate(ws, as_stream(stream))
                                                         : tc_state_passed();
        if (gate < 0)
            return REPRO_ERR_LAUNCH;
        tc = gate == 1;
    }
    return status_of(
        launch_attn_fwd(q, k, vq, s_v, o, m, l, B, T, Hq, Hkv, W, ws, tc, as_stream(stream)));
}

size_t repro_attn_bwd_ws_bytes(int64_t B, int64_t T, int64_t Hq, int64_t W)
{
    if (B <= 0 || T <= 0 || Hq <= 0 || W < -1 || T > REPRO_ATTN_MAX_T)
        return 0;
    return attn_bwd_ws_bytes(B, T, Hq, W);
}

int repro_attn_bwd(const float* q, const float* k, const int8_t* vq, const float* s_v,
                   const float* o, const float* dout, const float* m, const float* l, float* dq,
                   float* dk, float* dv, int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t D,
                   int64_t W, void* ws, size_t ws_bytes, const void* fwd_ws, size_t fwd_ws_bytes,
                   void* stream)
{
    if (B < 0 || T < 0 || Hq < 1 || Hkv < 1 || W < 0)
        return REPRO_ERR_SHAPE;
    if (D != REPRO_ATTN_HEAD_DIM || Hq % Hkv != 0 || T > REPRO_ATTN_MAX_T || Hkv > 65535 ||
        B > 65535)
        return REPRO_ERR_SHAPE;
    if (!q || !k || !vq || !s_v || !o || !dout || !m || !l || !dq || !dk || !dv)
        return REPRO_ERR_ARG;
    if (!al16(q) || !al16(k) || !al16(vq) || !al16(o) || !al16(dout) || !al16(dq) || !al16(dk) ||
        !al16(dv) || !al4(s_v) || !al4(m) || !al4(l))
        return REPRO_ERR_ALIGN;
    if (B == 0 || T == 0)
        return REPRO_OK;
    const size_t nq = (size_t)(B * T * Hq * D) * 4, nk = (size_t)(B * T * Hkv * D);
    const size_t nr = (size_t)(B * T * Hq) * 4;
    const void* ins[8] = {q, k, vq, s_v, o, dout, m, l};
    const size_t insz[8] = {nq, nk * 4, nk, 4, nq, nq, nr, nr};
    void* outs[3] = {dq, dk, dv};
    const size_t outsz[3] = {nq, nk * 4, nk * 4};
    for (int x = 0; x < 3; ++x) {
        for (int y = 0; y < 8; ++y)
            if (overlap(outs[x], outsz[x], ins[y], insz[y]))
                return REPRO_ERR_ALIAS;
        for (int y = x + 1; y < 3; ++y)
            if (overlap(outs[x], outsz[x], outs[y], outsz[y]))
                return REPRO_ERR_ALIAS;
    }
    // the cached route keeps its tiles and copies in ws too
    const size_t need = attn_bwd_ws_bytes(B, T, Hq, fwd_ws ? W : -1);
    if (!ws || ws_bytes < need)
        return REPRO_ERR_WORKSPACE;
    if (!al16(ws))
        return REPRO_ERR_ALIGN;
    for (int y = 0; y < 8; ++y)
        if (overlap(ws, need, ins[y], insz[y]))
            return REPRO_ERR_ALIAS;
    for (int x = 0; x < 3; ++x)
        if (overlap(ws, need, outs[x], outsz[x]))
            return REPRO_ERR_ALIAS;
    if (fwd_ws) {
        const size_t fneed = attn_fwd_ws_bytes(B, T, Hq, W);
        if (fwd_ws_bytes < fneed)
            return REPRO_ERR_WORKSPACE;
        if (!al16(fwd_ws))
            return REPRO_ERR_ALIGN;
        if (overlap(fwd_ws, fneed, ws, need))
            return REPRO_ERR_ALIAS;
        for (int x = 0; x < 3; ++x)
            if (overlap(fwd_ws, fneed, outs[x], outsz[x]))
                return REPRO_ERR_ALIAS;
    }
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{q, B * T * Hq * D}, {k, B * T * Hkv * D}, {s_v, 1}, {o, B * T * Hq * D},
                                   {dout, B * T * Hq * D}, {m, B * T * Hq}, {l, B * T * Hq}})) != REPRO_OK)
        return st;
    return status_of(launch_attn_bwd(q, k, vq, s_v, o, dout, m, l, dq, dk, dv, B, T, Hq, Hkv, W,
                                     ws, fwd_ws, as_stream(stream)));
}

size_t repro_state_hash_ws_bytes(const int64_t* nbytes, int nbuf)
{
    if (nbuf < 0 || nbuf > REPRO_HASH_MAX_BUFFERS || (nbuf > 0 && !nbytes))
        return 0;
    for (int b = 0; b < nbuf; ++b)
        if (nbytes[b] < 0)
            return 0;
    return hash_ws_bytes(hash_leaf_count(nbytes, nbuf, REPRO_HASH_LEAF_BYTES));
}

int repro_state_hash(const void* const* bufs, const int64_t* nbytes, int nbuf, uint8_t* digest,
                     void* ws, size_t ws_bytes, void* stream)
{
    if (nbuf < 0 || nbuf > REPRO_HASH_MAX_BUFFERS || !digest)
        return REPRO_ERR_ARG;
    if (nbuf > 0 && (!bufs || !nbytes))
        return REPRO_ERR_ARG;
    for (int b = 0; b < nbuf; ++b) {
        if (nbytes[b] < 0)
            return REPRO_ERR_SHAPE;
        if (nbytes[b] > 0 && !bufs[b])
            return REPRO_ERR_ARG;
        if (nbytes[b] > 0 && !al16(bufs[b]))
            return REPRO_ERR_ALIGN;
    }
    if (!al16(digest))
        return REPRO_ERR_ALIGN;
    const size_t need = hash_ws_bytes(hash_leaf_count(nbytes, nbuf, REPRO_HASH_LEAF_BYTES));
    if (need > 0) {
        if (!ws || ws_bytes < need)
            return REPRO_ERR_WORKSPACE;
        if (!al16(ws))
            return REPRO_ERR_ALIGN;
        if (overlap(ws, need, digest, 32))
            return REPRO_ERR_ALIAS;
        for (int b = 0; b < nbuf; ++b)
            if (overlap(ws, need, bufs[b], (size_t)nbytes[b]))
                return REPRO_ERR_ALIAS;
    }
    int st = check_arch();
    if (st != REPRO_OK)
        return st;
    return status_of(launch_state_hash(bufs, nbytes, nbuf, REPRO_HASH_LEAF_BYTES, digest, ws,
                                       as_stream(stream)));
}

} // extern "C"
