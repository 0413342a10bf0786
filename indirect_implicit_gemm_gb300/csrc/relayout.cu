// relayout.cu -- the two memory-bound re-layout kernels and the stem's
// channel padding.
//
//  * build_indirection: the indirection buffer of "The Indirect Convolution
//    Algorithm" (Abstract), one int32 element offset per (output pixel, tap).
//  * im2win: the window-order buffer of "Im2win: An Efficient Convolution
//    Paradigm on GPU" (Abstract), win[n][ho][wc][kh][ci].
//  * pack_padded_weights: the stem path's weight matrix with every tap's
//    channels padded to the gather granule (zero weights on the padding).
//
// All three are bandwidth kernels: grid-stride loops over the output, 16-byte
// vector accesses where the layout allows, grids sized in whole waves of the
// SM count.
#include "fastdiv.h"
#include "internal.h"

namespace convgb {
namespace {

constexpr int kThreads = 256;

int grid_for(long long work_items, int per_thread)
{
    long long blocks = (work_items + (long long)kThreads * per_thread - 1) /
                       ((long long)kThreads * per_thread);
    long long cap = (long long)num_sms() * 8;  // 8 resident 256-thread CTAs per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

// ibuf[pix][tap] = ((h*W)+w)*C_in, or -1 in the padding.
__global__ void __launch_bounds__(kThreads) build_indirection_kernel(
    int32_t* __restrict__ ibuf, int total, FastDiv taps, FastDiv kw_div, FastDiv wo_div, int H,
    int W, int C_in, int s, int p, int d)
{
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < (uint32_t)total;
         e += gridDim.x * blockDim.x) {
        uint32_t pix, tap, ho, wo, kh, kw;
        taps.divmod(e, pix, tap);
        wo_div.divmod(pix, ho, wo);
        kw_div.divmod(tap, kh, kw);
        int h = (int)ho * s + (int)kh * d - p;
        int w = (int)wo * s + (int)kw * d - p;
        int32_t v = -1;
        if (h >= 0 && h < H && w >= 0 && w < W) v = (h * W + w) * C_in;
        ibuf[e] = v;
    }
}

// One 16-byte vector (8 channels) of win per loop trip; C_in % 8 == 0.
__global__ void __launch_bounds__(kThreads) im2win_vec_kernel(
    const uint4* __restrict__ x, uint4* __restrict__ win, int total, FastDiv cv_div,
    FastDiv kh_div, FastDiv wu_div, FastDiv ho_div, int H, int W, int s, int p, int d)
{
    const uint32_t CV = cv_div.d;
    // v = (((n*H_out + ho)*W_used + wc)*KH + kh)*CV + cv; total < 2^31 (checked on the host).
    for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < (uint32_t)total;
         v += gridDim.x * blockDim.x) {
        uint32_t r0, cv, r1, kh, r2, wc, n, ho;
        cv_div.divmod(v, r0, cv);
        kh_div.divmod(r0, r1, kh);
        wu_div.divmod(r1, r2, wc);
        ho_div.divmod(r2, n, ho);
        int h = (int)ho * s + (int)kh * d - p;
        int w = (int)wc - p;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (h >= 0 && h < H && w >= 0 && w < W)
            val = __ldg(&x[(((long long)n * H + h) * W + w) * CV + cv]);
        win[v] = val;
    }
}

// Element-wise fallback for C_in not a multiple of 8.
__global__ void __launch_bounds__(kThreads) im2win_elem_kernel(
    const uint16_t* __restrict__ x, uint16_t* __restrict__ win, int total, FastDiv ci_div,
    FastDiv kh_div, FastDiv wu_div, FastDiv ho_div, int H, int W, int s, int p, int d)
{
    const int C_in = (int)ci_div.d;
    for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < (uint32_t)total;
         v += gridDim.x * blockDim.x) {
        uint32_t r0, ci, r1, kh, r2, wc, n, ho;
        ci_div.divmod(v, r0, ci);
        kh_div.divmod(r0, r1, kh);
        wu_div.divmod(r1, r2, wc);
        ho_div.divmod(r2, n, ho);
        int h = (int)ho * s + (int)kh * d - p;
        int w = (int)wc - p;
        uint16_t val = 0;
        if (h >= 0 && h < H && w >= 0 && w < W)
            val = x[(((long long)n * H + h) * W + w) * C_in + ci];
        win[v] = val;
    }
}

// Weights [C_out][T][C_in] -> [C_out][k_pad] with each tap's channels padded
// to cp (zero weights on the padding) and the row padded with zeros from
// T*cp to k_pad: wp[co][t*cp + c] = w[co][t][c] for c < C_in.
__global__ void __launch_bounds__(kThreads) pack_padded_weights_kernel(
    const uint16_t* __restrict__ w, uint16_t* __restrict__ wp, int total, FastDiv kpad_div,
    int taps, int C_in, int cp)
{
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < (uint32_t)total;
         e += gridDim.x * blockDim.x) {
        uint32_t co, k;
        kpad_div.divmod(e, co, k);
        const int t = (int)k / cp, c = (int)k - t * cp;
        uint16_t v = 0;
        if (t < taps && c < C_in) v = w[((long long)co * taps + t) * C_in + c];
        wp[e] = v;
    }
}

// Window-order re-layout with each column's (kh, ci) vector padded to KC
// elements (a multiple of 8), for small C_in.  One CTA per output row
// g = n*H_out + ho stages that row's KH input rows in shared memory (zeros
// outside the image), then each thread builds whole columns
//   win[g][wc][kc] = x[n][ho*s - p + kh][wc - p][ci],  kc = kh*C_in + ci < KH*C_in
// and 0 for KH*C_in <= kc < KC, wc in [0, W_used), in shared memory (the
// (kh, ci) walk needs no division), and the CTA copies the row's contiguous
// W_used*KC block out with coalesced 16-byte stores.
__global__ void __launch_bounds__(kThreads) im2win_padded_kernel(
    const uint16_t* __restrict__ x, uint16_t* __restrict__ win, int H, int W, int C_in, int KH,
    int s, int p, int H_out, int W_used, int KC)
{
    extern __shared__ uint4 smem_v[];  // output block [W_used][KC], then rows [KH][W*C_in]
    const int out_vecs = W_used * KC / 8;
    uint4* outs = smem_v;
    uint16_t* rows = reinterpret_cast<uint16_t*>(smem_v + out_vecs);
    const int g = blockIdx.x;
    const int n = g / H_out, ho = g - n * H_out;
    const int rowlen = W * C_in;
    for (int kh = 0; kh < KH; ++kh) {
        const int h = ho * s - p + kh;
        uint16_t* dst = rows + kh * rowlen;
        if (h < 0 || h >= H) {
            for (int i = threadIdx.x; i < rowlen; i += blockDim.x) dst[i] = 0;
            continue;
        }
        const uint16_t* src = x + (static_cast<long long>(n) * H + h) * rowlen;
        if ((rowlen & 7) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
            for (int i = threadIdx.x; i < rowlen / 8; i += blockDim.x)
                reinterpret_cast<uint4*>(dst)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
        } else {
            for (int i = threadIdx.x; i < rowlen; i += blockDim.x) dst[i] = src[i];
        }
    }
    __syncthreads();
    const int kcv = KC / 8;
    for (int wc = threadIdx.x; wc < W_used; wc += blockDim.x) {
        const int w = wc - p;
        const bool inside = w >= 0 && w < W;
        uint4* col = outs + wc * kcv;
        const uint16_t* rp = rows + (inside ? w * C_in : 0);
        int kh = 0, ci = 0;  // (kh, ci) of the next element, walked
        for (int vec = 0; vec < kcv; ++vec) {
            uint32_t a[4];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t v = 0;
                if (kh < KH) {
                    if (inside) v = rp[kh * rowlen + ci];
                    if (++ci == C_in) {
                        ci = 0;
                        ++kh;
                    }
                }
                if (q & 1)
                    a[q >> 1] |= v << 16;
                else
                    a[q >> 1] = v;
            }
            col[vec] = make_uint4(a[0], a[1], a[2], a[3]);
        }
    }
    __syncthreads();
    uint4* out = reinterpret_cast<uint4*>(win + static_cast<long long>(g) * W_used * KC);
    for (int v = threadIdx.x; v < out_vecs; v += blockDim.x) out[v] = outs[v];
}

// The same re-layout for compile-time KH and C_in (the 3-channel stems): each
// thread assembles one column's KC values in registers, all indices static,
// and writes it with 16-byte stores; the output needs no shared memory.
// Small CTAs keep many output rows' input loads in flight per SM (measured on
// the 7x7 stem: 32/64/128/256 threads -> 99/96/93/106 us for the whole call).
constexpr int kRowThreads = 128;

template <int KH_, int C_>
__global__ void __launch_bounds__(kRowThreads) im2win_padded_fixed_kernel(
    const uint16_t* __restrict__ x, uint16_t* __restrict__ win, int H, int W, int s, int p,
    int H_out, int W_used)
{
    constexpr int KC = (KH_ * C_ + 7) / 8 * 8;
    extern __shared__ uint4 smem_v[];  // rows [KH_][W*C_]
    uint16_t* rows = reinterpret_cast<uint16_t*>(smem_v);
    const int g = blockIdx.x;
    const int n = g / H_out, ho = g - n * H_out;
    const int rowlen = W * C_;
    bool row_in[KH_];
#pragma unroll
    for (int kh = 0; kh < KH_; ++kh) {
        const int h = ho * s - p + kh;
        row_in[kh] = h >= 0 && h < H;
        if (!row_in[kh]) continue;
        const uint16_t* src = x + (static_cast<long long>(n) * H + h) * rowlen;
        uint16_t* dst = rows + kh * rowlen;
        if ((rowlen & 7) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
            for (int i = threadIdx.x; i < rowlen / 8; i += blockDim.x)
                reinterpret_cast<uint4*>(dst)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
        } else {
            for (int i = threadIdx.x; i < rowlen; i += blockDim.x) dst[i] = src[i];
        }
    }
    __syncthreads();
    uint4* out = reinterpret_cast<uint4*>(win + static_cast<long long>(g) * W_used * KC);
    for (int wc = threadIdx.x; wc < W_used; wc += blockDim.x) {
        const int w = wc - p;
        const bool inside = w >= 0 && w < W;
        uint32_t e[KC / 2];
#pragma unroll
        for (int i = 0; i < KC / 2; ++i) e[i] = 0u;
        if (inside) {
#pragma unroll
            for (int kh = 0; kh < KH_; ++kh) {
                if (!row_in[kh]) continue;
                const uint16_t* rp = rows + kh * rowlen + w * C_;
#pragma unroll
                for (int ci = 0; ci < C_; ++ci) {
                    const int k = kh * C_ + ci;
                    e[k / 2] |= static_cast<uint32_t>(rp[ci]) << (16 * (k & 1));
                }
            }
        }
        uint4* col = out + wc * (KC / 8);
#pragma unroll
        for (int v = 0; v < KC / 8; ++v)
            col[v] = make_uint4(e[4 * v], e[4 * v + 1], e[4 * v + 2], e[4 * v + 3]);
    }
}

// Weights [C_out][KH][KW][C_in] -> [C_out][KW*KC] in the im2win path's K order
// (kw, kh, ci), each kw slice padded with zeros from KH*C_in to KC.
__global__ void __launch_bounds__(kThreads) pack_im2win_weights_kernel(
    const uint16_t* __restrict__ w, uint16_t* __restrict__ wp, int total, FastDiv kpad_div,
    FastDiv kc_div, int KH, int KW, int C_in)
{
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < (uint32_t)total;
         e += gridDim.x * blockDim.x) {
        uint32_t co, k, kw, kc;
        kpad_div.divmod(e, co, k);
        kc_div.divmod(k, kw, kc);
        const int kh = static_cast<int>(kc) / C_in, ci = static_cast<int>(kc) - kh * C_in;
        uint16_t v = 0;
        if (kh < KH)
            v = w[((static_cast<long long>(co) * KH + kh) * KW + kw) * C_in + ci];
        wp[e] = v;
    }
}

}  // namespace

cudaError_t launch_im2win_padded(const ConvShape& c, int KC, const uint16_t* x, uint16_t* win,
                                 cudaStream_t st)
{
    const int W_used = (c.W_out - 1) * c.s + (c.KW - 1) * c.d + 1;
    const int rows_smem = (c.KH * c.W * c.C_in * 2 + 15) / 16 * 16;
    if (c.C_in == 3 && (c.KH == 7 || c.KH == 11)) {
        if (c.KH == 7)
            im2win_padded_fixed_kernel<7, 3><<<c.N * c.H_out, kRowThreads, rows_smem, st>>>(
                x, win, c.H, c.W, c.s, c.p, c.H_out, W_used);
        else
            im2win_padded_fixed_kernel<11, 3><<<c.N * c.H_out, kRowThreads, rows_smem, st>>>(
                x, win, c.H, c.W, c.s, c.p, c.H_out, W_used);
        return cudaGetLastError();
    }
    const int smem = W_used * KC * 2 + rows_smem;
    im2win_padded_kernel<<<c.N * c.H_out, kThreads, smem, st>>>(x, win, c.H, c.W, c.C_in, c.KH,
                                                                c.s, c.p, c.H_out, W_used, KC);
    return cudaGetLastError();
}

cudaError_t launch_pack_im2win_weights(const uint16_t* w, uint16_t* wp, int C_out, int KH, int KW,
                                       int C_in, int KC, cudaStream_t st)
{
    const int total = C_out * KW * KC;
    pack_im2win_weights_kernel<<<grid_for(total, 4), kThreads, 0, st>>>(
        w, wp, total, FastDiv(KW * KC), FastDiv(KC), KH, KW, C_in);
    return cudaGetLastError();
}

cudaError_t launch_build_indirection(const ConvShape& c, int32_t* ibuf, cudaStream_t st)
{
    int taps = c.KH * c.KW;
    int total = c.H_out * c.W_out * taps;
    build_indirection_kernel<<<grid_for(total, 4), kThreads, 0, st>>>(
        ibuf, total, FastDiv(taps), FastDiv(c.KW), FastDiv(c.W_out), c.H, c.W, c.C_in, c.s,
        c.p, c.d);
    return cudaGetLastError();
}

// The caller guarantees the element count of win (vector count when C_in % 8 == 0) is < 2^31.
cudaError_t launch_im2win(const ConvShape& c, const uint16_t* x, uint16_t* win, cudaStream_t st)
{
    int W_used = (c.W_out - 1) * c.s + (c.KW - 1) * c.d + 1;
    if (c.C_in % 8 == 0) {
        int total = (int)((long long)c.N * c.H_out * W_used * c.KH * (c.C_in / 8));
        im2win_vec_kernel<<<grid_for(total, 4), kThreads, 0, st>>>(
            reinterpret_cast<const uint4*>(x), reinterpret_cast<uint4*>(win), total,
            FastDiv(c.C_in / 8), FastDiv(c.KH), FastDiv(W_used), FastDiv(c.H_out), c.H, c.W,
            c.s, c.p, c.d);
    } else {
        int total = (int)((long long)c.N * c.H_out * W_used * c.KH * c.C_in);
        im2win_elem_kernel<<<grid_for(total, 4), kThreads, 0, st>>>(
            x, win, total, FastDiv(c.C_in), FastDiv(c.KH), FastDiv(W_used), FastDiv(c.H_out), c.H, c.W,
            c.s, c.p, c.d);
    }
    return cudaGetLastError();
}

cudaError_t launch_pack_padded_weights(const uint16_t* w, uint16_t* wp, int C_out, int taps,
                                       int C_in, int cp, int k_pad, cudaStream_t st)
{
    int total = C_out * k_pad;
    pack_padded_weights_kernel<<<grid_for(total, 4), kThreads, 0, st>>>(
        w, wp, total, FastDiv(k_pad), taps, C_in, cp);
    return cudaGetLastError();
}

}  // namespace convgb
