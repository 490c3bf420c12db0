// conv_noalloc.cu -- conv_fwd for callers that cannot allocate device memory.
//
// conv_fwd takes its split-K scratch from the caller.  Some callers cannot
// provide one: code that must not call cudaMalloc at run time (engines that
// reserve all device memory up front, or latency-bound code that cannot
// afford cudaMalloc's implicit device synchronisation).  conv_fwd_noalloc
// runs the same plan with the split-K partials in a fixed static device
// array instead.  It allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds kNoallocScratchBytes of it until the process exits.  Host
// code cannot use the symbol's name as a device address, so the address is
// fetched with cudaGetSymbolAddress once per device (on that device's first
// call) and passed down as the workspace pointer.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "conv3d.h"
#include "internal.h"

namespace c3d {
namespace {

constexpr size_t kNoallocScratchBytes = CONV_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (first call per
// device looks it up).
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        set_last_error("cudaGetDevice failed");
        return CONV_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error("device ordinal out of range");
        return CONV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            set_last_error("cudaGetSymbolAddress of the static scratch failed");
            return CONV_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CONV_OK;
}

}  // namespace
}  // namespace c3d

extern "C" int conv_fwd_noalloc(const void* x, const int64_t x_dims[5], const void* w,
                                const int64_t w_dims[5], const int stride[3], const int pad[3],
                                const int dil[3], int dtype, const float* scale_x,
                                const float* scale_w, void* out, cudaStream_t stream) {
    int rc = conv_fwd_plan(x_dims, w_dims, stride, pad, dil, dtype, 0, nullptr, nullptr, nullptr,
                           nullptr, nullptr, nullptr, nullptr);
    if (rc != CONV_OK) return rc;
    // the split-K partials must fit; optional operand copies that do not fit
    // are skipped by conv_fwd itself, and a patch-class problem whose
    // gathered rows do not fit is rejected there
    const size_t need = c3d::splitk_workspace_bytes(x_dims, w_dims, stride, pad, dil, dtype);
    if (need > c3d::kNoallocScratchBytes) {
        char msg[160];
        std::snprintf(msg, sizeof msg,
                      "split-K scratch of %zu bytes exceeds the %zu-byte static scratch of "
                      "conv_fwd_noalloc",
                      need, c3d::kNoallocScratchBytes);
        c3d::set_last_error(msg);
        return CONV_ERR_INVALID;
    }
    void* scratch = nullptr;
    if ((rc = c3d::scratch_address(&scratch)) != CONV_OK) return rc;
    // The split-K partials are written in full before the reduce reads them,
    // so nothing in the scratch needs clearing between calls.
    return conv_fwd(x, x_dims, w, w_dims, stride, pad, dil, dtype, scale_x, scale_w, out, scratch,
                    c3d::kNoallocScratchBytes, stream);
}
