// moe_layer_noalloc: the whole layer without a caller-provided workspace.
//
// Some callers cannot allocate device memory at all -- e.g. code that runs
// inside another framework's memory pool with allocation disabled, or a
// runtime that must never call cudaMalloc after start-up -- yet still own
// their inputs and outputs.  For them the layer's scratch (the routing maps,
// the MXFP8 activations, the intermediate and the FC2 rows) lives in one
// file-scope device array of a fixed size, which every GPU that loads this
// library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device.  In host code the array's
// name only stands in for the symbol; the kernels need the address that
// cudaGetSymbolAddress returns with that device current.  It is looked up on
// each call (a device reset that reloads the module moves it), except while
// the stream is capturing, when the lookup, which may load the module, is
// skipped and the last address seen on the device is used.
constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(void** out, bool capturing) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!capturing) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    if (!g_scratch_ptr[dev]) return MOE_ERR_CUDA;  // the first call on a device was made during capture
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_layer_noalloc(const moe_shape* shape, const float* logits, const uint16_t* shared_logit,
                                 const uint16_t* x, const moe_weights* weights, int32_t* topk_ids, float* topk_w,
                                 uint16_t* out, moe_stream_t stream) {
    if (!shape) return MOE_ERR_NULL;
    if (!moe_is_supported(shape)) return MOE_ERR_SHAPE;
    size_t need = 0;
    int rc = moe_workspace_bytes(shape, &need);
    if (rc != MOE_OK) return rc;
    if (need > moe::kStaticScratchBytes) return MOE_ERR_WORKSPACE;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) != cudaSuccess) return MOE_ERR_CUDA;
    void* scratch = nullptr;
    if ((rc = moe::scratch_for_current_device(&scratch, cs != cudaStreamCaptureStatusNone)) != MOE_OK) return rc;
    // Nothing in the scratch has to start at zero: the sort rewrites the
    // maps, counters and status word on every call, and later kernels read
    // only what this call wrote (rows past a tile reach only accumulator lanes
    // that are never read).
    return moe_layer(shape, logits, shared_logit, x, weights, topk_ids, topk_w, scratch, moe::kStaticScratchBytes,
                     out, stream);
}

// The status word of the current device's scratch array (the header of the
// workspace carved from it), read after the caller's stream has finished.
extern "C" int moe_noalloc_get_status(int32_t* status, int32_t* detail) {
    if (!status || !detail) return MOE_ERR_NULL;
    void* scratch = nullptr;
    int rc = moe::scratch_for_current_device(&scratch, false);
    if (rc != MOE_OK) return rc;
    return moe_get_status(scratch, status, detail);
}
