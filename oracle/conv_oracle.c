/*
 * conv_oracle.c -- CPU oracle for the forward 2D convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; it exists so that tests and the benchmark's CPU baseline
 * have a plain, slow, obviously correct statement of what the GPU library
 * computes.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes ("Unifying Convolutions and GEMM", section 1, the naive
 * 7-loop convolution; the same page's section 5 adds zero padding and a
 * per-channel bias, and "The Indirect Convolution Algorithm", Abstract, names
 * dilation among the parameters the method handles):
 *
 *   Y[n,co,ho,wo] = bias[co]
 *                 + sum_{ci,kh,kw} X[n,ci,ho*s+kh*d-p, wo*s+kw*d-p] * W[co,ci,kh,kw]
 *
 * with X taken as 0 outside [0,H) x [0,W).  Every product and sum is formed
 * in IEEE double from the bf16 inputs, each of which is exactly
 * representable in double, so the only rounding is that of the fp64 sum.
 *
 * The loops run in the page's printed order (n, co, ho, wo, ci, kh, kw);
 * the section-1 listing omits padding, dilation, bias and the initialisation
 * of Y, and the readings used here are: Y starts at bias[co] (or 0 when no
 * bias is given: section 5 makes the bias optional), padding contributes
 * zeros (section 5 pads with zeros before unfolding), and tap kh sits d*kh rows
 * from the window origin (the usual meaning of dilation d; d = 1 gives the
 * listing's ho*stride+kh).
 *
 * Alongside Y the oracle also forms B[n,co,ho,wo] = |bias[co]| +
 * sum |X*W| over the same terms: the scale of the per-element error bound
 * used to judge a reduced-precision result.
 *
 * Storage is reached only through the index functions below.  The input
 * arrays hold raw bf16 bit patterns (uint16), in the channels-last layouts
 * the library uses: X as [N][H][W][C_in], W as [C_out][KH][KW][C_in], the
 * outputs as [N][H_out][W_out][C_out] doubles.  Changing an index function
 * changes the layout and nothing else.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC conv_oracle.c -o _liboracle.so
 * (the OpenMP pragma is the only parallelism; without -fopenmp it is serial).
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double: the bf16 bits are the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Output size along one spatial axis: floor((L + 2p - d(K-1) - 1)/s) + 1.
 * With d = 1 this reduces to the undilated extent section 5 gives. */
long oracle_output_size(long L, long K, long s, long p, long d)
{
    long span = L + 2 * p - d * (K - 1) - 1;
    if (s <= 0 || span < 0)
        return 0;
    return span / s + 1;
}

struct geom {
    long N, C_in, H, W, C_out, KH, KW, s, p, d, H_out, W_out;
};

/* Index functions: the only place the storage order appears. */
static size_t idx_x(const struct geom* g, long n, long ci, long h, long w)
{
    return (size_t)(((n * g->H + h) * g->W + w) * g->C_in + ci);
}
static size_t idx_w(const struct geom* g, long co, long ci, long kh, long kw)
{
    return (size_t)(((co * g->KH + kh) * g->KW + kw) * g->C_in + ci);
}
static size_t idx_y(const struct geom* g, long n, long co, long ho, long wo)
{
    return (size_t)(((n * g->H_out + ho) * g->W_out + wo) * g->C_out + co);
}

/* One output element: the innermost three loops of the 7-loop listing. */
static void one_output(const struct geom* g, const uint16_t* x, const uint16_t* wt,
                       const uint16_t* bias, long n, long co, long ho, long wo,
                       double* out, double* out_abs)
{
    double acc = 0.0, mag = 0.0;
    if (bias) {
        acc = bf16_to_double(bias[co]);
        mag = acc < 0 ? -acc : acc;
    }
    for (long ci = 0; ci < g->C_in; ++ci)
        for (long kh = 0; kh < g->KH; ++kh)
            for (long kw = 0; kw < g->KW; ++kw) {
                long h = ho * g->s + kh * g->d - g->p;
                long w = wo * g->s + kw * g->d - g->p;
                if (h < 0 || h >= g->H || w < 0 || w >= g->W)
                    continue; /* zero padding contributes nothing */
                double prod = bf16_to_double(x[idx_x(g, n, ci, h, w)]) *
                              bf16_to_double(wt[idx_w(g, co, ci, kh, kw)]);
                acc += prod;
                mag += prod < 0 ? -prod : prod;
            }
    *out = acc;
    if (out_abs)
        *out_abs = mag;
}

static int fill_geom(struct geom* g, long N, long C_in, long H, long W, long C_out,
                     long KH, long KW, long s, long p, long d)
{
    g->N = N; g->C_in = C_in; g->H = H; g->W = W; g->C_out = C_out;
    g->KH = KH; g->KW = KW; g->s = s; g->p = p; g->d = d;
    if (N < 0 || C_in < 1 || H < 1 || W < 1 || C_out < 1 || KH < 1 || KW < 1 ||
        s < 1 || p < 0 || d < 1)
        return -1;
    g->H_out = oracle_output_size(H, KH, s, p, d);
    g->W_out = oracle_output_size(W, KW, s, p, d);
    if (g->H_out < 1 || g->W_out < 1)
        return -1;
    return 0;
}

/* Full convolution.  y and y_abs (nullable) hold N*H_out*W_out*C_out doubles.
 * Returns 0, or -1 for an invalid geometry. */
int oracle_conv2d_direct(const uint16_t* x, const uint16_t* wt, const uint16_t* bias,
                         long N, long C_in, long H, long W, long C_out, long KH, long KW,
                         long s, long p, long d, double* y, double* y_abs)
{
    struct geom g;
    if (fill_geom(&g, N, C_in, H, W, C_out, KH, KW, s, p, d))
        return -1;
    long nco = g.N * g.C_out;
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < nco; ++t) {
        long n = t / g.C_out, co = t % g.C_out;
        for (long ho = 0; ho < g.H_out; ++ho)
            for (long wo = 0; wo < g.W_out; ++wo) {
                size_t o = idx_y(&g, n, co, ho, wo);
                one_output(&g, x, wt, bias, n, co, ho, wo, &y[o], y_abs ? &y_abs[o] : NULL);
            }
    }
    return 0;
}

/* Selected outputs only.  pts holds count quadruples (n, co, ho, wo); out and
 * out_abs (nullable) receive one double per point.  Returns 0, -1 for an
 * invalid geometry, -2 for a point outside the output. */
int oracle_conv2d_points(const uint16_t* x, const uint16_t* wt, const uint16_t* bias,
                         long N, long C_in, long H, long W, long C_out, long KH, long KW,
                         long s, long p, long d, const int64_t* pts, long count,
                         double* out, double* out_abs)
{
    struct geom g;
    if (fill_geom(&g, N, C_in, H, W, C_out, KH, KW, s, p, d))
        return -1;
    for (long i = 0; i < count; ++i) {
        const int64_t* q = pts + 4 * i;
        if (q[0] < 0 || q[0] >= g.N || q[1] < 0 || q[1] >= g.C_out || q[2] < 0 ||
            q[2] >= g.H_out || q[3] < 0 || q[3] >= g.W_out)
            return -2;
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (long i = 0; i < count; ++i) {
        const int64_t* q = pts + 4 * i;
        one_output(&g, x, wt, bias, q[0], q[1], q[2], q[3], &out[i],
                   out_abs ? &out_abs[i] : NULL);
    }
    return 0;
}

/* Threads the parallel loops above will use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
