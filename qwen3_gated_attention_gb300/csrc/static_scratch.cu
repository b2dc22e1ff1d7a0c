// static_scratch.cu -- dequantizing a projection without allocating.
//
// gattn_layer_dequant_device stages the layer's tile-layout rows through a
// buffer it obtains with cudaMalloc on every call, and synchronizes.  Some
// callers cannot do that: code recording a CUDA graph in global capture mode
// (where cudaMalloc, cudaFree and synchronization are refused), code running
// inside a framework that owns the whole device memory budget through its own
// pool, or latency-sensitive paths where cudaMalloc/cudaFree may synchronize
// the device.  gattn_layer_dequant_device_static does the same work with its
// staging buffer in the file-scope device array below: it allocates nothing
// and returns without waiting for the GPU.
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gattn.h"
#include "kernels.cuh"

namespace {

// The staging area: 16 MiB, held by every GPU that loads the library until the
// process exits.  A projection fits when the 128-row blocks spanning it, times
// K, are at most kStaticScratchFloats floats.
constexpr size_t kStaticScratchFloats = size_t(4) << 20;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

// Device address of g_static_scratch per device, remembered together with the
// CUDA context it was resolved in.  In host code the symbol's name is only a
// host-side stand-in, not a device address, so it is looked up with
// cudaGetSymbolAddress with the device current.  A context that is destroyed
// and created again (cudaDeviceReset, or the primary context released and
// retained again) reloads the module, and the array may then sit elsewhere:
// the cached address is used only while the current context's unique id is
// the one it was resolved under, and is looked up again otherwise.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float *g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);

// Unique id of the calling thread's current context (driver entry points
// resolved once through the runtime, so the library needs no libcuda link).
cudaError_t current_context_id(unsigned long long *id)
{
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static cudaError_t resolved = cudaErrorUnknown;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000,
                                                         cudaEnableDefault, &q1);
        if (e == cudaSuccess)
            e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
        if (e == cudaSuccess && (q1 != cudaDriverEntryPointSuccess || !f1 ||
                                 q2 != cudaDriverEntryPointSuccess || !f2))
            e = cudaErrorSymbolNotFound;
        get_current = reinterpret_cast<PfnCtxGetCurrent>(f1);
        get_id = reinterpret_cast<PfnCtxGetId>(f2);
        resolved = e;
    });
    if (resolved != cudaSuccess)
        return resolved;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    return cudaSuccess;
}

gattn_status scratch_for_current_device(float **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        gattn_set_error(cudaGetErrorString(e));
        return GATTN_E_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        gattn_set_error("device index beyond the static scratch table");
        return GATTN_E_UNSUPPORTED;
    }
    // the thread's current context; before the runtime has bound one to this
    // thread there is none (id 0), and the symbol lookup below binds it
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != cudaSuccess)
        ctx = 0;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        float *p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_scratch);
        if (e == cudaSuccess && ctx == 0)
            e = current_context_id(&ctx);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s",
                     cudaGetErrorString(e));
            gattn_set_error(msg);
            return GATTN_E_CUDA;
        }
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return GATTN_OK;
}

}  // namespace

extern "C" gattn_status gattn_layer_dequant_device_static(gattn_layer *layer, int32_t proj,
                                                          float *w, gattn_stream stream)
{
    using namespace gattn;
    if (!layer || !w || proj < 0 || proj > 3) {
        gattn_set_error("bad dequant arguments");
        return GATTN_E_INVALID_ARG;
    }
    ProjTiles t;
    if (!layer_proj_tiles(layer, proj, &t)) {
        gattn_set_error("set_weights has not been called");
        return GATTN_E_STATE;
    }
    const int rb0 = t.row0 / kRBR, rb1 = (t.row0 + t.rows + kRBR - 1) / kRBR;
    const size_t need = (size_t)(rb1 - rb0) * kRBR * (size_t)t.K;
    if (need > kStaticScratchFloats) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "projection %d needs %zu floats of staging; the static scratch holds %zu "
                 "(use gattn_layer_dequant_device)",
                 (int)proj, need, kStaticScratchFloats);
        gattn_set_error(msg);
        return GATTN_E_UNSUPPORTED;
    }
    float *scratch = nullptr;
    gattn_status st = scratch_for_current_device(&scratch);
    if (st != GATTN_OK)
        return st;
    // every staged element is written by the kernel before it is copied out,
    // so nothing has to be cleared first
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *wsub = t.w + (size_t)rb0 * t.nku * t.step_bytes;
    cudaError_t e = launch_dequant_tiles(wsub, (rb1 - rb0) * kRBR, t.K, t.bits, t.group, rb1 - rb0,
                                         scratch, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(w, scratch + (size_t)(t.row0 - rb0 * kRBR) * t.K,
                            (size_t)t.rows * t.K * sizeof(float), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) {
        gattn_set_error(cudaGetErrorString(e));
        return GATTN_E_CUDA;
    }
    return GATTN_OK;
}
