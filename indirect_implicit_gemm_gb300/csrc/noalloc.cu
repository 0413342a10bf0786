// noalloc.cu -- conv2d_fwd_noalloc: the gather-path convolution for callers
// that cannot hand the library a workspace.
//
// conv2d_fwd needs scratch device memory for its indirection buffer, and the
// caller normally provides it (allocated with cudaMalloc or a framework
// allocator).  Some callers cannot do that: code whose device memory is
// planned and owned by a host framework that gives plugins no allocation
// hook, and latency-critical loops that must never trigger cudaMalloc or
// cudaFree (both can synchronise the whole device).  This entry point keeps
// its scratch in a fixed array that is part of the library's device image
// instead, so it allocates nothing at call time.
//
// The array is kNoAllocScratchBytes (4 MiB) of device memory on every GPU that
// loads the library, held until the process exits.  Every call shares it:
// calls that may overlap on the GPU (different streams, or different host
// threads) race on it and must be serialised by the caller.  Each call
// rewrites every entry it reads, so nothing needs clearing between calls.
#include <mutex>

#include "internal.h"

namespace convgb {
namespace {

// Largest indirection buffer the static scratch holds: 4 MiB, i.e.
// H_out*W_out*KH*KW <= 1,048,576 entries.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

// Static scratch for the indirection buffer.  In host code this name is only a
// stand-in for the symbol, never a device address: host code reaches the
// memory through cudaGetSymbolAddress() (see scratch_on_current_device()).
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached; nullptr on failure.
int32_t* scratch_on_current_device()
{
    static int32_t* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();  // leave no error of this call for the caller's next check
            return nullptr;
        }
        addr[dev] = static_cast<int32_t*>(p);
    }
    return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace convgb

extern "C" convgb_status conv2d_fwd_noalloc(const void* x, const void* w, const void* bias, int N,
                                            int C_in, int H, int W, int C_out, int KH, int KW,
                                            int stride, int pad, int dilation, void* y,
                                            int y_dtype, void* stream)
{
    using namespace convgb;
    // Every check, and the whole plan of the GEMM, happens before the first
    // launch: a call that fails queues nothing and leaves the array untouched.
    int H_out = 0, W_out = 0;
    if (convgb_output_dims(H, W, KH, KW, stride, pad, dilation, &H_out, &W_out) != CONVGB_OK)
        return CONVGB_ERR_INVALID_ARG;
    if (N < 1 || C_in < 1 || C_out < 1) return CONVGB_ERR_INVALID_ARG;
    if (!x || !w || !y) return CONVGB_ERR_INVALID_ARG;
    if (y_dtype != CONVGB_BF16 && y_dtype != CONVGB_F32) return CONVGB_ERR_INVALID_ARG;
    if (convgb_select_path(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation) < 0)
        return CONVGB_ERR_UNSUPPORTED;  // index limits exceeded
    if (C_in % 8 != 0) return CONVGB_ERR_UNSUPPORTED;  // gather path only
    const size_t need = convgb_indirection_buffer_bytes(H, W, KH, KW, stride, pad, dilation);
    if (need == 0) return CONVGB_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return CONVGB_ERR_WORKSPACE;  // beyond the static scratch
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)))
        return CONVGB_ERR_ALIGNMENT;
    int32_t* scratch = scratch_on_current_device();
    if (scratch == nullptr) return CONVGB_ERR_CUDA;

    return conv_indirect(x, w, bias, N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, scratch,
                         kNoAllocScratchBytes, 1, y, y_dtype, stream);
}
