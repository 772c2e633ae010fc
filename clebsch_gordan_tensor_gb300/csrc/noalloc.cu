// Fused-convolution gradient for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at the point where they
// need the gradient: a host framework that owns all device memory through its
// own pool and forbids allocations behind its back, a plugin running inside
// another application under a fixed memory budget, or a latency-critical loop
// that cannot afford the implicit device synchronisation of cudaMalloc /
// cudaFree.  cgtp_conv_backward_ws asks them for scratch memory when the plan
// shares one weight row between all edges (the weight gradient is summed from
// per-CTA partial rows).  cgtp_conv_backward_noalloc takes that scratch from a
// fixed array compiled into the library instead, so the caller passes only its
// inputs and outputs.
//
// The array, g_noalloc_scratch, is a file-scope __device__ array of
// kNoAllocScratchBytes (8 MiB): every GPU that loads this library holds it
// until the process exits.  Host code must not use its name as an address (on
// the host the name is only a stand-in); the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the first
// call of the entry point on that device.  That first call also loads the
// plan's remaining kernels and the reduction kernels into the device's context
// (set-up that may allocate code memory); later calls allocate nothing.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <string>

#include "cgtp.h"
#include "internal.hpp"

namespace cgtp {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
// Partial weight-gradient rows the array must hold at least: the most that one
// CTA of any kernel writes (the non-staged kernels write one per work slot, at
// most 128), so a weight row may take up to 8 MiB / 128 = 64 KiB.
constexpr int64_t kNoAllocMinRows = 128;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static std::map<int, void*> g_noalloc_addr;  // device -> address of the array

// Device address of the array on device dev, the current device (looked up on
// the first call there).
static cgtp_status noalloc_scratch(int dev, void** out) {
    cudaError_t e;
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    auto it = g_noalloc_addr.find(dev);
    if (it != g_noalloc_addr.end()) {
        *out = it->second;
        return CGTP_OK;
    }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
        set_cuda_error(e);
        set_error_message(std::string("cudaGetSymbolAddress(no-alloc scratch): ") +
                          cudaGetErrorString(e));
        return CGTP_E_CUDA;
    }
    g_noalloc_addr[dev] = ptr;
    *out = ptr;
    return CGTP_OK;
}

}  // namespace cgtp

extern "C" cgtp_status cgtp_conv_backward_noalloc(
    cgtp_plan plan, int64_t N, int64_t E, const int32_t* rowptr, const int32_t* sender,
    const int32_t* s_rowptr, const int32_t* s_perm, const int32_t* s_recv, const void* x,
    const void* y, const void* w, double scale, const void* grad_out, void* grad_x, void* grad_y,
    void* grad_w, cgtp_stream stream) {
    try {
        (void)rowptr;
        (void)sender;
        if (!plan) {
            cgtp::set_error_message("plan is NULL");
            return CGTP_E_ARG;
        }
        // A shared weight row's gradient is summed from partial rows: at least
        // kNoAllocMinRows of them (the most one CTA of any kernel writes) must fit.
        const int64_t row = cgtp::plan_weight_row_bytes(plan);
        if (cgtp::plan_shared_weights(plan) && grad_w &&
            row > (int64_t)(cgtp::kNoAllocScratchBytes / cgtp::kNoAllocMinRows)) {
            cgtp::set_error_message("weight row of " + std::to_string(row) +
                                    " bytes is larger than the no-allocation limit of " +
                                    std::to_string(cgtp::kNoAllocScratchBytes /
                                                   cgtp::kNoAllocMinRows) +
                                    " bytes");
            return CGTP_E_ARG;
        }
        if (!cgtp::plan_module_loaded(plan, -1)) {
            cgtp::set_error_message(
                "the plan's kernels have not run on any device yet (loading them allocates "
                "device memory): make one call through another entry point first");
            return CGTP_E_ARG;
        }
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) {
            cgtp::set_cuda_error(e);
            cgtp::set_error_message(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
            return CGTP_E_CUDA;
        }
        if (!cgtp::plan_module_loaded(plan, dev)) {
            cgtp::set_error_message(
                "the plan's kernels have not run on device " + std::to_string(dev) +
                " yet (loading them there allocates device memory): make one call through "
                "another entry point on this device first");
            return CGTP_E_ARG;
        }
        void* scratch = nullptr;
        cgtp_status st = cgtp::noalloc_scratch(dev, &scratch);
        if (st != CGTP_OK) return st;
        if ((st = cgtp::plan_preload_kernels(plan, dev)) != CGTP_OK) return st;
        return cgtp::conv_backward_into_scratch(plan, N, E, s_rowptr, s_perm, s_recv, x, y, w,
                                                scale, grad_out, grad_x, grad_y, grad_w, scratch,
                                                cgtp::kNoAllocScratchBytes,
                                                reinterpret_cast<cudaStream_t>(stream));
    } catch (...) {
        cgtp::set_error_message("unexpected internal exception");
        return CGTP_E_ARG;
    }
}
