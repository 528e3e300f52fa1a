// static_ws.cu -- conv_fprop for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: a plugin whose host
// framework owns every device allocation and exposes none to the plugin, or
// a latency-critical loop that must not call cudaMalloc (it can synchronise
// the device and its cost is unbounded).  conv_fprop_static_workspace serves
// them with scratch that lives in this file-scope device array instead.  The
// array is part of the module: every GPU that loads the library holds it
// until the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"

namespace i8c {
namespace {

// Scratch for the repacked filter and the channels-last image copy of the
// tensor-core path.
__device__ __align__(256) uint8_t g_static_workspace[CONV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_static_ptr[kMaxDevices];

// Device address of this device's copy of the array.  In host code the
// array's name is only a host-side stand-in, so the address comes from the
// runtime, once per device, with that device current.
conv_status static_workspace_ptr(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CONV_ERR_UNSUPPORTED_DEVICE;
    void *p = g_static_ptr[dev].load();
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return CONV_ERR_CUDA;
        g_static_ptr[dev].store(p);
    }
    *out = p;
    return CONV_OK;
}

}  // namespace
}  // namespace i8c

using namespace i8c;

extern "C" conv_status conv_fprop_static_workspace(const conv_tensor_desc *x, const int8_t *x_dev,
                                                   const conv_tensor_desc *w, const int8_t *w_dev,
                                                   const conv_tensor_desc *y, void *y_dev,
                                                   const int32_t *bias_dev, const conv_fprop_params *p,
                                                   void *stream) {
    size_t need = 0;
    conv_status st = conv_fprop_workspace_size_for(x, x_dev, w, y, p, &need);
    if (st) return st;
    if (need > (size_t)CONV_STATIC_WORKSPACE_BYTES) return CONV_ERR_STATIC_WORKSPACE_LIMIT;
    if ((st = check_device())) return st;
    void *ws = nullptr;
    if (need > 0 && (st = static_workspace_ptr(&ws))) return st;
    // every byte of scratch the kernels read is written earlier in the same
    // call (filter blocks including their zero padding, the image copy
    // including its zero channels), so nothing needs clearing first
    return conv_fprop(x, x_dev, w, w_dev, y, y_dev, bias_dev, p, ws, need > 0 ? (size_t)CONV_STATIC_WORKSPACE_BYTES : 0,
                      stream);
}
