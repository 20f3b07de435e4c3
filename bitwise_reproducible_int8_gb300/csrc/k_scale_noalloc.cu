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
// process exits.  Host code cannot use its name as a device address, so the
// first call on each device, with that device current, looks the address up
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.  All calls share the one array and it keeps whatever the
// last call left there; the kernels overwrite every partial before reading it,
// so nothing needs clearing.  Two calls whose work overlaps on the GPU (for
// example on two streams of the same device) race on the array: serialise
// them.
#include "internal.h"
#include "repro.h"

namespace repro {
namespace {

static __device__ __align__(256) float g_noalloc_scratch[REPRO_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDev = 64;
float* g_scratch_addr[kMaxDev];

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
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
        return REPRO_ERR_LAUNCH;
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return REPRO_ERR_LAUNCH;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == REPRO_SCALE_WEIGHT_MEANABS) {
        // the default block split always: its partials fit the array for every
        // n up to REPRO_NOALLOC_MAX_N
        if (wscale_ws_bytes(n, -1) > sizeof(float) * REPRO_NOALLOC_SCRATCH_FLOATS)
            return REPRO_ERR_SHAPE;
        e = launch_wscale_meanabs(x, n, qmax, scale_out, g_scratch_addr[dev], -1, s);
    } else {
        e = launch_wscale_amax(x, n, qmax, scale_out, g_scratch_addr[dev], amax_grid(n), s);
    }
    return e == cudaSuccess ? REPRO_OK : REPRO_ERR_LAUNCH;
}
