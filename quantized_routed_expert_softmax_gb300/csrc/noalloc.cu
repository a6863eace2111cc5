// noalloc.cu -- moe_layer_forward_noalloc: the layer forward for callers that cannot
// allocate device memory.
//
// Some callers are handed only their input and output buffers and a stream (a plugin
// inside another engine that owns every allocation), or must not allocate once serving
// has started (an allocation can synchronise the device, and allocating while a stream
// is being captured into a graph is not allowed).  They cannot provide the workspace
// moe_layer_forward needs.  This entry point runs the same forward with its scratch in a
// fixed-size array that is part of the library itself: every GPU that loads libmoe holds
// MOE_NOALLOC_SCRATCH_BYTES of device memory for it until the process exits.
#include <mutex>

#include "common.cuh"

namespace {

// The scratch.  In host code `g_noalloc_scratch` names a host-side stand-in, not a device
// address; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch, looked up once per device with that device current.
void* scratch_address(moe_status* st) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *st = MOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            *st = MOE_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    *st = MOE_OK;
    return addr[dev];
}

}  // namespace

extern "C" moe_status moe_layer_forward_noalloc(const moe_layer_desc* desc, const void* x, moe_dtype xt, int64_t T,
                                                const int32_t* idx_in, const float* w_in, float* out,
                                                moe_stream_t stream) {
    if (!desc) return MOE_ERR_INVALID_ARG;
    if (T == 0) return moe_layer_forward(desc, x, xt, T, idx_in, w_in, out, nullptr, 0, nullptr, stream);
    const size_t need = moe_layer_workspace_bytes(desc, T);
    if (need == 0) return moe_layer_forward(desc, x, xt, T, idx_in, w_in, out, nullptr, 0, nullptr, stream);
    if (need > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;   // beyond the fixed scratch
    moe_status st = MOE_OK;
    void* scratch = scratch_address(&st);
    if (st != MOE_OK) return st;
    // The scratch's control region (the error word, the barrier and row-tile counters, at the
    // same offsets for every layer shape) must start at zero.  It is cleared on every call, so
    // a counter left behind by an earlier call (one that overlapped this on another stream, or
    // one whose kernel stopped at a timed-out wait) cannot carry over into this one.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, moe::workspace_control_bytes(), s) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_layer_forward(desc, x, xt, T, idx_in, w_in, out, scratch, MOE_NOALLOC_SCRATCH_BYTES, nullptr, stream);
}

extern "C" moe_status moe_layer_forward_noalloc_status(moe_stream_t stream, int32_t* device_code) {
    moe_status st = MOE_OK;
    void* scratch = scratch_address(&st);
    if (st != MOE_OK) return st;
    return moe_get_device_status(scratch, stream, device_code);
}
