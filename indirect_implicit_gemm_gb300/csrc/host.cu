// host.cu -- conv2d_fwd from and to host memory, with the copies pipelined
// against the convolution.
//
// The batch is cut into up to four chunks of whole images.  Three streams of
// the library's own (created once per device) carry the host-to-device copies,
// the convolutions and the device-to-host copies; events order them so that
// chunk k+1's input copy, chunk k's convolution and chunk k-1's output copy
// run at the same time.  Each chunk's input and output live in one of two
// slots of the caller's device scratch, so a slot is refilled only after the
// work that read it has finished.  The three streams wait for the caller's
// stream before the first copy, and the caller's stream waits for them after
// the last, so to the caller the call behaves like work queued on `stream`.
// The convolution of each chunk is conv2d_fwd itself on device memory.

#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "convgb.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 4;
constexpr size_t kAlign = 256;

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Scratch layout of one call: weights, bias, two input slots, two output slots
// and the convolution's workspace for the largest chunk.
struct HostPlan {
    int chunks = 0, per_chunk = 0;
    size_t x_img = 0, y_img = 0;  // bytes of one image of x and of y
    size_t off_w = 0, off_b = 0, off_x[2] = {0, 0}, off_y[2] = {0, 0}, off_ws = 0;
    size_t ws_bytes = 0, total = 0;
};

bool host_plan(int N, int C_in, int H, int W, int C_out, int KH, int KW, int stride, int pad,
               int dilation, int y_dtype, bool has_bias, HostPlan* hp)
{
    if (N < 1 || C_in < 1 || C_out < 1) return false;
    if (y_dtype != CONVGB_BF16 && y_dtype != CONVGB_F32) return false;
    int Ho = 0, Wo = 0;
    if (convgb_output_dims(H, W, KH, KW, stride, pad, dilation, &Ho, &Wo) != CONVGB_OK)
        return false;
    HostPlan p;
    p.chunks = N < kMaxChunks ? N : kMaxChunks;
    p.per_chunk = (N + p.chunks - 1) / p.chunks;
    p.chunks = (N + p.per_chunk - 1) / p.per_chunk;
    p.x_img = static_cast<size_t>(H) * W * C_in * 2;
    p.y_img = static_cast<size_t>(Ho) * Wo * C_out * (y_dtype == CONVGB_F32 ? 4 : 2);
    const int last = N - (p.chunks - 1) * p.per_chunk;
    const size_t ws_full = convgb_conv2d_fwd_workspace_size(p.per_chunk, C_in, H, W, C_out, KH,
                                                            KW, stride, pad, dilation);
    const size_t ws_last =
        convgb_conv2d_fwd_workspace_size(last, C_in, H, W, C_out, KH, KW, stride, pad, dilation);
    p.ws_bytes = ws_full > ws_last ? ws_full : ws_last;
    size_t off = 0;
    p.off_w = off;
    off += round_up(static_cast<size_t>(C_out) * KH * KW * C_in * 2);
    p.off_b = off;
    off += has_bias ? round_up(static_cast<size_t>(C_out) * 2) : 0;
    for (int s = 0; s < 2; ++s) {
        p.off_x[s] = off;
        off += round_up(p.x_img * p.per_chunk);
    }
    for (int s = 0; s < 2; ++s) {
        p.off_y[s] = off;
        off += round_up(p.y_img * p.per_chunk);
    }
    p.off_ws = off;
    off += round_up(p.ws_bytes);
    p.total = off;
    *hp = p;
    return true;
}

// The library's three streams and the events that order them, per device.
struct Pipeline {
    cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done[3] = {nullptr, nullptr, nullptr};
    cudaEvent_t in_ready[2] = {nullptr, nullptr}, computed[2] = {nullptr, nullptr},
                out_read[2] = {nullptr, nullptr};
    bool ready = false;
    std::mutex mu;  // one call's queueing at a time per device
};

Pipeline* pipeline_for(int dev)
{
    static Pipeline pipes[kMaxDevices];
    static std::mutex mu;
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    Pipeline& pl = pipes[dev];
    if (!pl.ready) {
        const unsigned sf = cudaStreamNonBlocking;
        const unsigned ef = cudaEventDisableTiming;
        bool ok = cudaStreamCreateWithFlags(&pl.h2d, sf) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&pl.comp, sf) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&pl.d2h, sf) == cudaSuccess &&
                  cudaEventCreateWithFlags(&pl.start, ef) == cudaSuccess;
        for (int i = 0; ok && i < 3; ++i) ok = cudaEventCreateWithFlags(&pl.done[i], ef) == cudaSuccess;
        for (int s = 0; ok && s < 2; ++s)
            ok = cudaEventCreateWithFlags(&pl.in_ready[s], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&pl.computed[s], ef) == cudaSuccess &&
                 cudaEventCreateWithFlags(&pl.out_read[s], ef) == cudaSuccess;
        if (!ok) {  // undo a partial setup; the next call tries again
            for (cudaStream_t* st : {&pl.h2d, &pl.comp, &pl.d2h})
                if (*st) cudaStreamDestroy(*st), *st = nullptr;
            for (cudaEvent_t* ev : {&pl.start, &pl.done[0], &pl.done[1], &pl.done[2], &pl.in_ready[0],
                                    &pl.in_ready[1], &pl.computed[0], &pl.computed[1],
                                    &pl.out_read[0], &pl.out_read[1]})
                if (*ev) cudaEventDestroy(*ev), *ev = nullptr;
            return nullptr;
        }
        pl.ready = true;
    }
    return &pl;
}

}  // namespace

extern "C" {

size_t convgb_conv2d_fwd_host_scratch_size(int N, int C_in, int H, int W, int C_out, int KH,
                                           int KW, int stride, int pad, int dilation,
                                           int y_dtype, int has_bias)
{
    HostPlan p;
    if (!host_plan(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, y_dtype, has_bias != 0,
                   &p))
        return 0;
    return p.total;
}

convgb_status conv2d_fwd_host(const void* x_host, const void* w_host, const void* bias_host,
                              int N, int C_in, int H, int W, int C_out, int KH, int KW,
                              int stride, int pad, int dilation, void* y_host, int y_dtype,
                              void* scratch, size_t scratch_bytes, void* stream)
{
    // Everything is checked before the first CUDA call.
    if (!x_host || !w_host || !y_host || !scratch) return CONVGB_ERR_INVALID_ARG;
    HostPlan p;
    if (!host_plan(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, y_dtype,
                   bias_host != nullptr, &p))
        return CONVGB_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(scratch) & 15u) != 0) return CONVGB_ERR_ALIGNMENT;
    if (scratch_bytes < p.total) return CONVGB_ERR_WORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONVGB_ERR_CUDA;
    Pipeline* pl = pipeline_for(dev);
    if (!pl) return CONVGB_ERR_CUDA;
    std::lock_guard<std::mutex> lock(pl->mu);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    uint8_t* sb = static_cast<uint8_t*>(scratch);
    const uint8_t* xh = static_cast<const uint8_t*>(x_host);
    uint8_t* yh = static_cast<uint8_t*>(y_host);
    void* wd = sb + p.off_w;
    void* bd = bias_host ? sb + p.off_b : nullptr;
    void* ws = p.ws_bytes ? sb + p.off_ws : nullptr;

    convgb_status status = CONVGB_OK;
    bool cuda_ok = cudaEventRecord(pl->start, cs) == cudaSuccess &&
                   cudaStreamWaitEvent(pl->h2d, pl->start, 0) == cudaSuccess &&
                   cudaStreamWaitEvent(pl->comp, pl->start, 0) == cudaSuccess &&
                   cudaStreamWaitEvent(pl->d2h, pl->start, 0) == cudaSuccess;
    if (cuda_ok) {
        cuda_ok = cudaMemcpyAsync(wd, w_host, static_cast<size_t>(C_out) * KH * KW * C_in * 2,
                                  cudaMemcpyHostToDevice, pl->h2d) == cudaSuccess;
        if (cuda_ok && bias_host)
            cuda_ok = cudaMemcpyAsync(bd, bias_host, static_cast<size_t>(C_out) * 2,
                                      cudaMemcpyHostToDevice, pl->h2d) == cudaSuccess;
    }
    for (int k = 0; cuda_ok && status == CONVGB_OK && k < p.chunks; ++k) {
        const int s = k & 1;
        const int n0 = k * p.per_chunk;
        const int nk = (N - n0) < p.per_chunk ? (N - n0) : p.per_chunk;
        void* xd = sb + p.off_x[s];
        void* yd = sb + p.off_y[s];
        // input slot s is free once the convolution two chunks back has read it
        if (k >= 2) cuda_ok = cudaStreamWaitEvent(pl->h2d, pl->computed[s], 0) == cudaSuccess;
        cuda_ok = cuda_ok &&
                  cudaMemcpyAsync(xd, xh + static_cast<size_t>(n0) * p.x_img,
                                  static_cast<size_t>(nk) * p.x_img, cudaMemcpyHostToDevice,
                                  pl->h2d) == cudaSuccess &&
                  cudaEventRecord(pl->in_ready[s], pl->h2d) == cudaSuccess;
        // output slot s is free once the copy-out two chunks back has read it
        cuda_ok = cuda_ok && cudaStreamWaitEvent(pl->comp, pl->in_ready[s], 0) == cudaSuccess;
        if (cuda_ok && k >= 2)
            cuda_ok = cudaStreamWaitEvent(pl->comp, pl->out_read[s], 0) == cudaSuccess;
        if (!cuda_ok) break;
        status = conv2d_fwd(xd, wd, bd, nk, C_in, H, W, C_out, KH, KW, stride, pad, dilation, yd,
                            y_dtype, ws, p.ws_bytes, pl->comp);
        if (status != CONVGB_OK) break;
        cuda_ok = cudaEventRecord(pl->computed[s], pl->comp) == cudaSuccess &&
                  cudaStreamWaitEvent(pl->d2h, pl->computed[s], 0) == cudaSuccess &&
                  cudaMemcpyAsync(yh + static_cast<size_t>(n0) * p.y_img, yd,
                                  static_cast<size_t>(nk) * p.y_img, cudaMemcpyDeviceToHost,
                                  pl->d2h) == cudaSuccess &&
                  cudaEventRecord(pl->out_read[s], pl->d2h) == cudaSuccess;
    }
    // Join whatever was queued back into the caller's stream, also on failure.
    bool joined = cudaEventRecord(pl->done[0], pl->h2d) == cudaSuccess &&
                  cudaEventRecord(pl->done[1], pl->comp) == cudaSuccess &&
                  cudaEventRecord(pl->done[2], pl->d2h) == cudaSuccess;
    for (int i = 0; joined && i < 3; ++i)
        joined = cudaStreamWaitEvent(cs, pl->done[i], 0) == cudaSuccess;
    if (status != CONVGB_OK) return status;
    return (cuda_ok && joined) ? CONVGB_OK : CONVGB_ERR_CUDA;
}

}  // extern "C"
