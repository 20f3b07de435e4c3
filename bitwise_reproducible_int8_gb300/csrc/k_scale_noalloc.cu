// k_scale_noalloc.cu -- the scale reduction for callers that cannot allocate
// device memory.
//
// repro_wscale needs a small scratch buffer for its per-block partial sums and
// takes it from the caller.  Some callers have no way to provide one: code
// running where every device allocation is owned by someone else (a host
// application's private memory pool, a plugin with no allocator hooks), or a
// loop that must never call cudaMalloc because it would synchronise the
// device.  repro_wscale_noalloc serves them with a fixed scratch array that
// lives in this library's own device memory.
//
// The array (REPRO_NOALLOC_SCRATCH_FLOATS floats, 256 KB) is a static
// __device__ variable: every GPU that loads the library holds it until the
// process exits.  Host code cannot use its name as a device address, so each
// call looks the address up with cudaGetSymbolAddress, with the call's device
// current, and keeps it per device.  A call made while its stream is being
// captured into a CUDA graph uses the kept address instead (a lookup may not
// be legal then), so the first call on a device must come before any stream
// capture; calls outside capture look it up again, which also picks up the
// new address after a cudaDeviceReset.  All calls share the one array and it
// keeps whatever the last call left there; the kernels overwrite every
// partial before reading it, so nothing needs clearing.  Two calls whose work
// overlaps on the GPU (for example on two streams of the same device) race on
// the array: serialise them.
#include <atomic>

#include "internal.h"
#include "repro.h"

namespace repro {
namespace {

static __device__ __align__(256) float g_noalloc_scratch[REPRO_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDev = 64;
std::atomic<float*> g_scratch_addr[kMaxDev];   // last looked-up address per device

// the array's device address on device `dev` (current), or nullptr
float* scratch_address(int dev, cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess)
        return nullptr;
    if (cs != cudaStreamCaptureStatusNone)
        return g_scratch_addr[dev].load(std::memory_order_acquire);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
        return nullptr;
    g_scratch_addr[dev].store(static_cast<float*>(p), std::memory_order_release);
    return static_cast<float*>(p);
}

} // namespace
} // namespace repro

using namespace repro;

extern "C" int repro_wscale_noalloc(const float* x, int64_t n, int mode, int qmax,
                                    float* scale_out, void* stream)
{
    if (!x || !scale_out)
        return REPRO_ERR_ARG;
    if (mode != REPRO_SCALE_WEIGHT_MEANABS && mode != REPRO_SCALE_ACT_AMAX)
        return REPRO_ERR_ARG;
    if (qmax != REPRO_QMAX)
        return REPRO_ERR_ARG;
    if (n <= 0 || n > REPRO_NOALLOC_MAX_N)
        return REPRO_ERR_SHAPE;
    if (((uintptr_t)x & 15u) != 0 || ((uintptr_t)scale_out & 3u) != 0)
        return REPRO_ERR_ALIGN;
    int st = arch_status();
    if (st != REPRO_OK)
        return st;
    if ((st = scan_inputs(stream, {{x, n}})) != REPRO_OK)
        return st;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return REPRO_ERR_LAUNCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* scratch = scratch_address(dev, s);
    if (!scratch)
        return REPRO_ERR_LAUNCH;   // no lookup possible (e.g. first call inside a capture)
    if (mode == REPRO_SCALE_WEIGHT_MEANABS) {
        // the default block split always: its partials fit the array for every
        // n up to REPRO_NOALLOC_MAX_N
        if (wscale_ws_bytes(n, -1) > sizeof(float) * REPRO_NOALLOC_SCRATCH_FLOATS)
            return REPRO_ERR_SHAPE;
        return status_of(launch_wscale_meanabs(x, n, qmax, scale_out, scratch, -1, s));
    }
    return status_of(launch_wscale_amax(x, n, qmax, scale_out, scratch, amax_grid(n), s));
}
