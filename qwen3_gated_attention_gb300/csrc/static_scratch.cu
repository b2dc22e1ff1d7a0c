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

#include <cuda_runtime.h>

#include "gattn.h"
#include "kernels.cuh"

namespace {

// The staging area: 16 MiB, held by every GPU that loads the library until the
// process exits.  A projection fits when the 128-row blocks spanning it, times
// K, are at most kStaticScratchFloats floats.
constexpr size_t kStaticScratchFloats = size_t(4) << 20;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

// Device address of g_static_scratch per device.  In host code the symbol's
// name is only a host-side stand-in, not a device address, so it is looked up
// with cudaGetSymbolAddress once per device (with that device current).
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float *g_scratch_ptr[kMaxDevices] = {};

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
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        float *p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_static_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s",
                     cudaGetErrorString(e));
            gattn_set_error(msg);
            return GATTN_E_CUDA;
        }
        g_scratch_ptr[dev] = p;
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
