// api.cu -- the C ABI (include/convgb.h): argument checks, shape derivation,
// path choice, workspace layout, TMA descriptors and launches.
//
// Nothing here computes on the host: every element of every output is
// produced by the kernels in igemm.cu and relayout.cu.
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"

namespace convgb {

namespace {

__device__ unsigned g_device_error;  // first device-side failure since the last check

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;  // alignment of each workspace region

std::atomic<unsigned long long> g_timeout_ns{4000000000ull};
// Planner overrides for tuning and ablation studies (convgb_set_tuning); 0 =
// the planner's own choice.
std::atomic<int> g_tune_bn{0};
std::atomic<int> g_tune_stages{0};
std::atomic<int> g_tune_stream_k{0};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_device()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

// Output extent along one axis; 0 when the window does not fit.
long long out_extent(long long L, long long K, long long s, long long p, long long d)
{
    long long span = L + 2 * p - d * (K - 1) - 1;
    if (span < 0) return 0;
    return span / s + 1;
}

// Validates a shape and fills the derived extents.  INVALID_ARG for bad
// parameters or an empty output, UNSUPPORTED when an index limit is exceeded.
convgb_status make_shape(int N, int C_in, int H, int W, int C_out, int KH, int KW, int s, int p,
                         int d, ConvShape* c)
{
    if (N < 1 || C_in < 1 || H < 1 || W < 1 || C_out < 1 || KH < 1 || KW < 1 || s < 1 || p < 0 ||
        d < 1)
        return CONVGB_ERR_INVALID_ARG;
    long long Ho = out_extent(H, KH, s, p, d), Wo = out_extent(W, KW, s, p, d);
    if (Ho < 1 || Wo < 1) return CONVGB_ERR_INVALID_ARG;
    const long long lim = (1ll << 31) - 1;
    long long x_elems = (long long)N * H * W * C_in;
    long long y_elems = (long long)N * Ho * Wo * C_out;
    long long w_elems = (long long)C_out * KH * KW * C_in;
    if (x_elems > lim || y_elems > lim || w_elems > lim) return CONVGB_ERR_UNSUPPORTED;
    if (Ho * Wo * KH * KW > lim) return CONVGB_ERR_UNSUPPORTED;      // indirection entries
    c->N = N; c->C_in = C_in; c->H = H; c->W = W; c->C_out = C_out;
    c->KH = KH; c->KW = KW; c->s = s; c->p = p; c->d = d;
    c->H_out = (int)Ho; c->W_out = (int)Wo;
    c->M = (long long)N * Ho * Wo;
    c->K = (long long)KH * KW * C_in;
    return CONVGB_OK;
}

bool is_pointwise(const ConvShape& c)
{
    return c.KH == 1 && c.KW == 1 && c.s == 1 && c.p == 0;
}

// 1x1 unpadded layers with stride > 1 read only every s-th pixel of every s-th
// row: a 4-D TMA box with element strides (1, s, s, 1) loads exactly those.  A
// tile is R whole output rows of one image (R divides H_out), so the box
// traverses W_out*s pixels and R*s rows, each at most 256.
int strided_rows(const ConvShape& c)
{
    if (!(c.KH == 1 && c.KW == 1 && c.p == 0 && c.s > 1 && c.s <= 8 && c.C_in % 8 == 0))
        return 0;
    if (c.W_out > 128 || c.W_out * c.s > 256) return 0;
    for (int r = 128 / c.W_out; r >= 1; --r)
        if (c.H_out % r == 0 && r * c.s <= 256) return r;
    return 0;
}

bool is_full_spatial(const ConvShape& c)
{
    return c.KH == c.H && c.KW == c.W && c.p == 0 && c.d == 1;  // H_out = W_out = 1
}

// Window mode geometry: stride-1 layers whose 64-channel blocks stay inside
// one tap and whose output rows, padded by the tap spill, fit a 128-row tile.
bool window_geometry(const ConvShape& c)
{
    const int wv = c.W_out + (c.KW - 1) * c.d;
    return c.s == 1 && c.C_in % 64 == 0 && wv <= 128 && (c.KW - 1) * c.d <= 8;
}

// Narrow-window stem geometry: small C_in, undilated, output rows that fit a
// 128-row tile, input rows whose byte length keeps bulk copies 16-byte aligned.
bool narrow_window_geometry(const ConvShape& c)
{
    return c.C_in % 8 != 0 && c.C_in < 16 && c.d == 1 && c.W_out <= 128 &&
           ((long long)c.W * c.C_in * 2) % 16 == 0;
}

// Staged-row layout of the narrow window (bytes): the row's data starts at a0
// (16-byte aligned, at least p*C_in*2 in so pixel -p has room), and each row
// holds every element an A slice of the last output column can read.
struct NarrowRows {
    int kwc, kwcp, a0, rb, rows, slot;
};
NarrowRows narrow_rows(const ConvShape& c)
{
    NarrowRows r;
    r.kwc = c.KW * c.C_in;
    r.kwcp = (r.kwc + 7) / 8 * 8;
    r.a0 = (c.p * c.C_in * 2 + 15) / 16 * 16;
    const int lead = r.a0 - c.p * c.C_in * 2;  // byte of pixel -p
    const int data_end = r.a0 + c.W * c.C_in * 2;
    const int read_end = lead + ((c.W_out - 1) * c.s * c.C_in + r.kwcp) * 2 + 4;
    r.rb = ((data_end > read_end ? data_end : read_end) + 15) / 16 * 16;
    r.rows = 128 / c.W_out;  // output rows per tile
    r.slot = (r.rows * c.KH * r.rb + 511) / 512 * 512;  // two slots keep 1024-byte alignment
    return r;
}

// im2win path: each column of the window-order buffer holds the KH*C_in values
// (kh, ci) of one input column, padded to KC (a multiple of 8) so that rows of
// the buffer stay 16-byte aligned for TMA; W_used columns per output row.
struct Im2winGeom {
    int KC = 0, W_used = 0, R = 0;
    long long buf_bytes = 0;
};
Im2winGeom im2win_geom(const ConvShape& c)
{
    Im2winGeom g;
    g.KC = (c.KH * c.C_in + 7) / 8 * 8;
    g.W_used = (c.W_out - 1) * c.s + (c.KW - 1) * c.d + 1;
    g.R = c.W_out <= 128 ? 128 / c.W_out : 0;
    g.buf_bytes = (long long)c.N * c.H_out * g.W_used * g.KC * 2;
    return g;
}

// Small C_in, undilated, output rows that fit a 128-row tile, one output row's
// block and its input rows within the re-layout kernel's 48 KB of shared
// memory, and a buffer under half of im2col.
bool im2win_applies(const ConvShape& c)
{
    if (c.C_in >= 16 || c.d != 1 || c.W_out > 128) return false;
    const Im2winGeom g = im2win_geom(c);
    // the re-layout kernel's shared memory: one output row's block and its input rows
    if ((long long)g.W_used * g.KC * 2 + c.KH * c.W * c.C_in * 2 + 16 > 48 * 1024) return false;
    if (g.buf_bytes / 2 >= (1LL << 31)) return false;
    return g.buf_bytes < c.M * c.K * 2 / 2;
}

// Staged-window stem geometry.  For stride s in {1, 2, 4} and C_in = 3, each
// 128-byte row r of a shared-memory stage holds the s input columns
// s*r - p .. s*r - p + s - 1 of one output row, KC = 64/s values (kh, ci) per
// column (khg = KC / C_in kernel rows of a group, the rest zero).  Output pixel
// wo then reads its K block kb (columns s*(wo+kb) - p ..) from row wo + kb, so
// the MMA takes every K block of a stage from the same rows at shifted
// descriptor starts, as the window path does for its taps.  A tile is R
// output rows, each a segment of seg = W_out + nkb - 1 stage rows.
struct StemWinGeom {
    bool ok = false;
    int KC = 0, khg = 0, groups = 0, nkb = 0, seg = 0, R = 0, last_steps = 0;
    int a0 = 0, rb = 0, slot = 0;  // staged input rows, as the narrow window lays them out
    long long wbytes = 0;          // raw weights [C_out][KH*KW*C_in], bf16
};
StemWinGeom stemwin_geom(const ConvShape& c)
{
    StemWinGeom g;
    if (c.C_in != 3 || c.d != 1 || c.KH > 31) return g;
    if (c.s != 1 && c.s != 2 && c.s != 4) return g;
    if (((long long)c.W * c.C_in * 2) % 16 != 0) return g;  // bulk copies of whole rows
    g.wbytes = (long long)c.C_out * c.KH * c.KW * c.C_in * 2;
    if (g.wbytes % 16 != 0) return g;  // one bulk copy of the raw weights
    g.KC = 64 / c.s;
    g.khg = g.KC / c.C_in;
    g.groups = (c.KH + g.khg - 1) / g.khg;
    g.nkb = (c.KW + c.s - 1) / c.s;
    g.seg = c.W_out + g.nkb - 1;
    if (g.seg > 128) return g;
    g.R = 128 / g.seg;
    g.last_steps = ((c.KW - c.s * (g.nkb - 1)) * g.KC + 15) / 16;
    if ((g.nkb - 1) * 4 + g.last_steps > 16) return g;  // the kernel's unrolled MMA sequence
    g.a0 = (c.p * c.C_in * 2 + 15) / 16 * 16;
    const int lead = g.a0 - c.p * c.C_in * 2;  // byte of pixel -p
    const int data_end = g.a0 + c.W * c.C_in * 2;
    const int read_end = lead + c.s * g.seg * c.C_in * 2;  // past the last column a row reads
    g.rb = (std::max(data_end, read_end) + 15) / 16 * 16;
    g.slot = (g.R * c.KH * g.rb + 511) / 512 * 512;
    g.ok = true;
    return g;
}

// Folded-window geometry (C_in = 32, stride 1).  A segment is 32 consecutive
// input columns inside the image row; with the KW taps folded into the MMA's
// columns it yields G = 32 - (KW-1)*d output pixels of an output row (the rest
// of its columns only feed its neighbours' sums).  spr segments cover an output
// row.  A tile is one segment of four consecutive output rows (HB = ceil(H_out
// / 4) row blocks per image), whose R = 4 + (KH-1)*d input rows one TMA box
// stages.  The MMA is KW*C_out columns wide and the weights of all KH blocks
// stay resident.
struct FoldGeom {
    bool ok = false;
    int G = 0, spr = 0, HB = 0, R = 0, n_mma = 0, b_bytes = 0;
    int U = 0;  // output rows per work unit: 4, or 8 (two tiles) for 3x3-sized kernels
                // whose MMA fits 128 columns
    long long tiles = 0;
};
FoldGeom fold_geom(const ConvShape& c)
{
    FoldGeom f;
    if (c.s != 1 || c.C_in != 32 || c.C_out % 32 != 0) return f;
    if (c.KW > kFoldMaxKW || c.KH > kFoldMaxKH) return f;
    // segments are 32 columns inside the row; a box spans R rows
    if (c.W < 32) return f;
    const bool pair = c.KW <= kFold3MaxK && c.KH <= kFold3MaxK && c.KW * c.C_out <= 128;
    f.U = pair ? 2 * kFoldRows : kFoldRows;
    f.R = f.U + (c.KH - 1) * c.d;
    if (f.R > 256) return f;
    f.G = 32 - (c.KW - 1) * c.d;
    if (f.G < 8) return f;
    f.n_mma = c.KW * c.C_out;
    if (f.n_mma > 256 || f.n_mma % 16 != 0) return f;
    f.spr = (c.W_out + f.G - 1) / f.G;
    f.HB = (c.H_out + f.U - 1) / f.U;
    f.tiles = (long long)c.N * f.HB * f.spr;
    if (f.tiles >= (1LL << 31)) return f;
    f.b_bytes = (c.KH * f.n_mma * 64 + 1023) / 1024 * 1024;
    f.ok = true;
    return f;
}

struct GemmPlan;
GemmPlan plan_gemm(int path, const ConvShape& c, int y_f32 = 0);
bool fold_applies(const ConvShape& c);
bool stemwin_applies(const ConvShape& c);
bool window_applies(const ConvShape& c);
bool plane_applies(const ConvShape& c);

// Whether `path` can compute this shape.
bool path_supports(int path, const ConvShape& c)
{
    switch (path) {
    case CONVGB_PATH_WINDOW: return window_applies(c);
    case CONVGB_PATH_PLANE: return plane_applies(c);
    case CONVGB_PATH_IM2WIN: return im2win_applies(c);
    case CONVGB_PATH_GATHER: return c.C_in % 8 == 0;
    case CONVGB_PATH_DENSE:
        return c.C_in % 8 == 0 && (is_pointwise(c) || is_full_spatial(c) || strided_rows(c) > 0);
    case CONVGB_PATH_STEM: return c.C_in % 8 != 0;
    case CONVGB_PATH_STEMWIN: return stemwin_applies(c);
    case CONVGB_PATH_WINFOLD: return fold_applies(c);
    default: return false;
    }
}

int select_path(const ConvShape& c)
{
    if (path_supports(CONVGB_PATH_DENSE, c)) return CONVGB_PATH_DENSE;
    if (c.C_in % 8 != 0)
        return stemwin_applies(c)  ? CONVGB_PATH_STEMWIN
               : im2win_applies(c) ? CONVGB_PATH_IM2WIN
                                   : CONVGB_PATH_STEM;
    if (path_supports(CONVGB_PATH_WINDOW, c)) return CONVGB_PATH_WINDOW;
    // The folded window when its segments are mostly output pixels: with fewer
    // than 12 real pixels per 32-row segment the gather path's full 128-row
    // tiles of narrow MMAs cost less.
    if (fold_applies(c)) {
        const FoldGeom f = fold_geom(c);
        if (c.W_out >= 12 * f.spr) return CONVGB_PATH_WINFOLD;
    }
    return CONVGB_PATH_GATHER;
}

// Stem path: channels per tap in the packed K order (4 when C_in <= 4, else the
// next multiple of 8), and the packed row length rounded to 8 elements so the
// weight rows stay 16-byte aligned for TMA.
int stem_cp(const ConvShape& c) { return c.C_in <= 4 ? 4 : (c.C_in + 7) / 8 * 8; }
long long stem_kpad(const ConvShape& c)
{
    return ((long long)c.KH * c.KW * stem_cp(c) + 7) / 8 * 8;
}

// ------------------------------------------------------------ driver entry point
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Row-major bf16 matrix [rows][cols] (cols contiguous), box [box_rows][64 cols],
// 128-byte swizzle: exactly the K-major operand tile the MMA descriptors expect.
bool encode_kmajor(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows,
                   bool narrow = false)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    // narrow: boxes of 32 columns (64-byte rows, 64-byte swizzle)
    cuuint32_t box[2] = {narrow ? 32u : 64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     narrow ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// x [N][H][W][C_in] as a 4-D tensor, box = 64 channels x `wv` pixels of one
// row, 128-byte swizzle: one staged input row of the window mode.
bool encode_window(CUtensorMap* m, const void* x, int N, int H, int W, int C_in, int wv)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)C_in, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
    cuuint64_t strides[3] = {(cuuint64_t)C_in * 2, (cuuint64_t)W * C_in * 2,
                             (cuuint64_t)H * W * C_in * 2};
    cuuint32_t box[4] = {64u, (cuuint32_t)wv, 1u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The im2win buffer [N*H_out][W_used][KC] as A: row (wo, g) is the K = KW*KC
// contiguous elements from column wo*s of output row g, so consecutive rows
// overlap (row pitch s*KC elements).  Box: 64 K x W_out pixels x R output rows,
// 128-byte swizzle, landing as R*W_out consecutive 128-byte tile rows.
bool encode_im2win(CUtensorMap* m, const void* win, const ConvShape& c, int KC, int W_used, int R)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)c.KW * KC, (cuuint64_t)c.W_out,
                          (cuuint64_t)c.N * c.H_out};
    cuuint64_t strides[2] = {(cuuint64_t)c.s * KC * 2, (cuuint64_t)W_used * KC * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)c.W_out, (cuuint32_t)R};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(win), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// x [N][H][W][C_in] with element strides (1, s, s, 1): box = 64 channels x
// W_out pixels x R rows of one image (traversing W_out*s pixels and R*s rows).
bool encode_strided(CUtensorMap* m, const void* x, const ConvShape& c, int R)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)c.C_in, (cuuint64_t)c.W, (cuuint64_t)c.H, (cuuint64_t)c.N};
    cuuint64_t strides[3] = {(cuuint64_t)c.C_in * 2, (cuuint64_t)c.W * c.C_in * 2,
                             (cuuint64_t)c.H * c.W * c.C_in * 2};
    cuuint32_t box[4] = {64u, (cuuint32_t)(c.W_out * c.s), (cuuint32_t)(R * c.s), 1u};
    cuuint32_t estr[4] = {1u, (cuuint32_t)c.s, (cuuint32_t)c.s, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Folded window: x [N][H][W][32] as a 4-D tensor; a box of 32 channels x 32
// columns x R rows is one tile's staging: R consecutive input rows of one
// segment (64-byte swizzle, 2 KB per row).  The segments' columns always lie
// inside the row, so the column bounds never apply; rows outside the image read
// as zero.
bool encode_fold_x(CUtensorMap* m, const void* x, const ConvShape& c, int R)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {32u, (cuuint64_t)c.W, (cuuint64_t)c.H, (cuuint64_t)c.N};
    cuuint64_t strides[3] = {64u, (cuuint64_t)c.W * 64, (cuuint64_t)c.H * c.W * 64};
    cuuint32_t box[4] = {32u, 32u, (cuuint32_t)R, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Folded window: w [C_out][KH][KW][32] as a 4-D tensor (32 channels, kw, kh,
// co), box = 32 channels x all C_out for one (kh, kw): the C_out rows of tap
// kw in weight block kh, 64-byte swizzle.
bool encode_fold_w(CUtensorMap* m, const void* w, const ConvShape& c)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {32u, (cuuint64_t)c.KW, (cuuint64_t)c.KH, (cuuint64_t)c.C_out};
    cuuint64_t strides[3] = {64u, (cuuint64_t)c.KW * 64, (cuuint64_t)c.KH * c.KW * 64};
    cuuint32_t box[4] = {32u, 1u, 1u, (cuuint32_t)c.C_out};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int pick_bn(int C_out)
{
    const int forced = g_tune_bn.load(std::memory_order_relaxed);
    if (forced) return forced;
    if (C_out <= 32) return 32;
    if (C_out <= 64) return 64;
    if (C_out <= 128) return 128;
    return 256;
}

// How one convolution maps onto the implicit-GEMM kernel.
struct GemmPlan {
    int amode = kADense;
    int bn = 128;
    int splits = 1;
    int stages = 0;  // shared-memory ring depth
    int bres = 0;    // weights resident in shared memory
    int m_step = 128;
    int a_stage_bytes = 128 * 64 * 2;
    int b_per_stage = 1;
    int win_wv = 0, win_rows = 0;  // row-tile geometry (window and narrow window)
    int extra_smem = 0;            // narrow window: staged-row slots
    int nw_slots = 0;
    int tma_store = 0;             // epilogue through a staging tile and TMA stores
    int epi_bufs = 1;              // staging tiles of that epilogue
    int epi_c32 = 0;               // 1: 32-column chunks, 8 KB staging tiles
    int pl_u = 1, pl_nacc = 0, b_stages = 0;  // plane mode: sub-tiles, accumulators, B slots
    int pair = 0;                  // window mode on a CTA pair (each CTA holds bn/2 columns of B)
    int min_stages = 2;            // shallowest ring the mode runs with (a tuning cap stops here)
    int sk = 0;                    // stream-K: CTAs share out all (unit, K block) iterations
    long long M = 0, K = 0;
    int num_kb = 0, m_tiles = 0, n_tiles = 0;
};

// K partitions per output tile.  When the output tiles alone leave SMs idle,
// the K loop is split so more CTAs work at once (partial sums meet in an fp32
// buffer).  Planned for a nominal 148 SMs so that workspace sizes do not
// depend on the device; a split must cut the estimated time (waves of work
// per CTA) by a quarter, keep >= 4 K blocks per CTA, and its fp32 buffer must
// fit under `partial_cap` bytes.
int choose_splits(long long tiles, int num_kb, long long partial_bytes, long long partial_cap)
{
    constexpr int kNominalSms = 148;
    if (tiles >= 2 * kNominalSms || partial_bytes >= partial_cap) return 1;
    auto cost = [&](int sp) {
        return (double)((tiles * sp + kNominalSms - 1) / kNominalSms) / sp;
    };
    int best = 1;
    double best_cost = cost(1);
    for (int sp = 2; sp <= 16 && num_kb / sp >= 4; ++sp) {
        double c = cost(sp);
        if (c < best_cost - 1e-9) {
            best = sp;
            best_cost = c;
        }
    }
    return best_cost <= 0.75 * cost(1) ? best : 1;
}

// Turns on the TMA-store epilogue when the output allows it (bf16, rows 16-byte
// aligned, no split) and the ring still has two stages with its staging tile.
void plan_epilogue(GemmPlan& g, const ConvShape& c, int y_f32)
{
    if (is_fold(g.amode)) return;  // stores straight from the shuffle sums
    if (y_f32 || c.C_out % 8 != 0 || g.splits != 1 || g.sk || g.bn < 64 || g.stages < 2) return;
    const int kb_res = g.bres ? (int)((g.K + 63) / 64) : g.num_kb;
    const int bnb = g.pair ? g.bn / 2 : g.bn;
    const int s = igemm_pick_stages(bnb, g.bres, kb_res, g.a_stage_bytes, g.b_per_stage,
                                    g.extra_smem + kEpiStageBytes);
    const bool turns = g.amode == kATmaGather || g.amode == kATmaGatherPair;
    if (s < (turns ? kMinGatherTurnStages : 2)) return;
    g.stages = s;
    g.tma_store = 1;
    g.epi_bufs = 1;
    // A second staging tile when it costs at most one ring stage and leaves four.
    const int s2 = igemm_pick_stages(bnb, g.bres, kb_res, g.a_stage_bytes, g.b_per_stage,
                                     g.extra_smem + kEpiStageBytes + kEpiTileBytes);
    if (s2 >= 4 && s2 >= s - 1) {
        g.stages = s2;
        g.epi_bufs = 2;
        return;
    }
    // A staging tile of 32-column chunks (half the bytes) when that buys one
    // more ring stage and the tile's MMAs take long enough to hide the four
    // serialised chunk stores (eight-warp epilogue modes only).  Measured: the
    // 128-channel 3x3 layer at 56x56 (72 MMAs per tile, three to four stages)
    // goes from 90.8 to 84.8 us; the 64->128 layer (36 MMAs per tile) slows
    // from 17.1 to 18.4 us, so tiles below 64 MMAs keep 64-column chunks.
    const bool window = g.amode == kAWindow || g.amode == kAWindowPair;
    const bool epi8 = window || g.amode == kADense || g.amode == kAIm2win || g.amode == kAStrided;
    const int mmas_per_tile = 4 * g.num_kb * (window ? c.KW : 1);
    const int s3 = (epi8 && mmas_per_tile >= 64)
                       ? igemm_pick_stages(bnb, g.bres, kb_res, g.a_stage_bytes, g.b_per_stage,
                                           g.extra_smem + kEpiNarrowStageBytes)
                       : 0;
    if (s3 > s) {
        g.stages = s3;
        g.epi_c32 = 1;
    }
}

GemmPlan plan_gemm_ring(int path, const ConvShape& c);
GemmPlan plan_plane(const ConvShape& c, int y_f32);

// A ring-depth cap from convgb_set_tuning applies to the finished plan, so
// that every other choice (resident weights, epilogue staging) stays the
// planner's own.
void cap_stages(GemmPlan& g)
{
    int cap = g_tune_stages.load(std::memory_order_relaxed);
    if (cap == 0) return;
    // The TMA-gather warps fill the ring by turns, one stage in four each: a
    // ring of fewer than four stages would let a warp's wait on a stage's
    // release run two phases ahead, where the barrier's parity cannot tell
    // them apart.
    if (g.amode == kATmaGather || g.amode == kATmaGatherPair) cap = std::max(cap, kMinGatherTurnStages);
    cap = std::max(cap, g.min_stages);
    if (g.stages > cap) g.stages = cap;
}

// Stream-K for layers whose work units fill less than one wave of the GPU
// (e.g. 64 pairs of 512-channel 3x3 tiles at 7x7 on 76 SM pairs): every CTA
// (pair) takes an equal share of all (unit, K block) iterations instead of
// whole units, and the units split between CTAs meet in the fp32 partial-sum
// buffer, which a finishing pass turns into y.  Eligible when at least a tenth
// of the CTAs would otherwise idle and the sums stay small enough to live in
// L2.  Taken only when asked for (convgb_set_tuning): on the 512-channel 3x3
// layer at 7x7 it measured 45.7 us against 35.7 us for whole units (the fp32
// round trip and its atomics cost more than the idle pairs; that layer is
// bound by streaming its weights through L2).
void plan_stream_k(GemmPlan& g, const ConvShape& c)
{
    if (g_tune_stream_k.load(std::memory_order_relaxed) != 1) return;
    const bool mode = g.amode == kAWindow || g.amode == kAWindowPair;  // built there only
    if (!mode || g.splits != 1 || (g.bres && g.n_tiles > 1) || g.stages < 2) return;
    constexpr int kNominalSms = 148;
    const long long units = (long long)(g.pair ? (g.m_tiles + 1) / 2 : g.m_tiles) * g.n_tiles;
    const int ctas = g.pair ? kNominalSms / 2 : kNominalSms;
    if (units >= ctas || (double)units >= 0.9 * ctas) return;
    const long long partial = c.M * c.C_out * 4;
    if (partial > (32LL << 20) || partial >= c.M * c.K * 2 / 2) return;
    if ((long long)g.num_kb * units < 2LL * ctas) return;  // too few iterations to share
    g.sk = 1;
}

GemmPlan plan_gemm(int path, const ConvShape& c, int y_f32)
{
    GemmPlan g = path == CONVGB_PATH_PLANE ? plan_plane(c, y_f32) : plan_gemm_ring(path, c);
    if (path != CONVGB_PATH_PLANE) plan_stream_k(g, c);
    if (path != CONVGB_PATH_PLANE) plan_epilogue(g, c, y_f32);
    cap_stages(g);
    // the window mode's common plan runs on the kernel built for it
    if (g.amode == kAWindow && g.bres && g.tma_store && !g.epi_c32 && g.splits == 1 && !g.sk &&
        c.KW == 3 && g.n_tiles == 1)
        g.amode = kAWindowT;
    return g;
}

// Plane mode.  With stride 1 the padded images stacked along H form one tall
// image of N*(H+2p) rows of W+2p pixels; every output pixel (n, ho, wo) is
// virtual pixel (n*(H+2p) + ho, wo) of it, and tap (kh, kw) of virtual pixel
// (v, w) reads padded pixel (v + kh*d, w + kw*d).  A tile holds R = 128 / (W+2p)
// whole virtual rows per sub-tile, so in the row-major staging of its padded
// rows every tap is the same 128-row window shifted by kh*d*(W+2p) + kw*d rows.
// Virtual pixels in the padding border (wo >= W_out, ho >= H_out) are computed
// and discarded.  Candidates differ in sub-tiles per tile (1 or 2, sharing each
// weight block), the column-tile width and whether the weights stay resident;
// the one with the least estimated time wins.  The estimate per tile is the
// larger of its tensor-core time and its L2-to-SM bytes at a per-SM share of
// L2 bandwidth, times the waves of tiles over the SMs.
GemmPlan plan_plane(const ConvShape& c, int y_f32)
{
    GemmPlan best;
    best.amode = kAPlane;
    if (!window_geometry(c)) return best;  // stages == 0: not applicable
    const int wv = c.W + 2 * c.p;
    const int hp = c.H + 2 * c.p;
    const int R = 128 / wv;
    const long long vrows = (long long)c.N * hp - (long long)(c.KH - 1) * c.d;
    if ((long long)c.N * hp * wv >= (1LL << 31)) return best;
    const int cc = c.C_in / 64;
    const int taps = c.KH * c.KW;
    const int kb_total = taps * cc;
    const int limit = smem_limit();
    const bool epi_ok = !y_f32 && c.C_out % 8 == 0;
    constexpr double kSmClock = 1.9e9, kL2PerSm = 50e9;
    constexpr int kNominalSms = 148;
    double best_cost = 1e30;
    const int bn_top = pick_bn(c.C_out);
    for (int bn = bn_top; bn >= 64 || bn == bn_top; bn /= 2) {
        const int n_tiles = (c.C_out + bn - 1) / bn;
        for (int u = 1; u <= 2; ++u) {
            if (u * bn > 256) continue;  // at least two accumulators in tensor memory
            const int rows = ((u - 1) * R + (c.KH - 1) * c.d) * wv + (c.KW - 1) * c.d + 128;
            const int ast = (rows * 128 + 1023) / 1024 * 1024;
            const long long m_tiles = (vrows + u * R - 1) / (u * R);
            for (int bres = (n_tiles == 1) ? 1 : 0; bres >= 0; --bres) {
                for (int epi = (epi_ok && bn >= 64) ? 1 : 0; epi >= 0; --epi) {
                    const int extra = epi ? kEpiStageBytes : 0;
                    int sa = 0, sb = 0;
                    if (bres) {
                        for (int s = 8; s >= 2 && !sa; --s)
                            if (plane_smem_bytes(bn, s, ast, kb_total, extra) <= limit) sa = s;
                    } else {
                        for (int s = 3; s >= 2 && !sa; --s)
                            for (int b = 8; b >= 3 && !sb; --b)
                                if (plane_smem_bytes(bn, s, ast, b, extra) <= limit) {
                                    sa = s;
                                    sb = b;
                                }
                        if (sa == 3 && sb < 6) {  // prefer a deeper weight ring
                            for (int b = 8; b >= 3; --b)
                                if (plane_smem_bytes(bn, 2, ast, b, extra) <= limit) {
                                    if (b > sb) {
                                        sa = 2;
                                        sb = b;
                                    }
                                    break;
                                }
                        }
                    }
                    if (sa < 2) continue;
                    const double mma_cyc = (double)cc * taps * u * 4 * (bn / 2 > 48 ? bn / 2 : 48);
                    const double l2 = (double)cc * (u * R + (c.KH - 1) * c.d) * wv * 128 +
                                      (bres ? 0.0 : (double)cc * taps * bn * 128);
                    const double t_tile = std::max(mma_cyc / kSmClock, l2 / kL2PerSm);
                    const long long tiles = m_tiles * n_tiles;
                    const double cost =
                        (double)((tiles + kNominalSms - 1) / kNominalSms) * t_tile;
                    if (cost < best_cost * 0.98) {
                        best_cost = cost;
                        GemmPlan g;
                        g.amode = kAPlane;
                        g.M = c.M;
                        g.K = c.K;
                        g.bn = bn;
                        g.win_wv = wv;
                        g.win_rows = R;
                        g.pl_u = u;
                        g.m_step = u * R;
                        g.m_tiles = (int)m_tiles;
                        g.n_tiles = n_tiles;
                        g.num_kb = cc;
                        g.a_stage_bytes = ast;
                        g.bres = bres;
                        g.stages = sa;
                        g.b_stages = bres ? 0 : sb;
                        g.pl_nacc = std::min(4, 512 / (u * bn));
                        g.tma_store = epi;
                        best = g;
                    }
                    break;  // the epilogue staging tile is used whenever it fits
                }
            }
        }
        if (bn <= 32) break;
    }
    if (best.stages >= 2) {
        if (c.KH == 3 && c.KW == 3) best.amode = best.pl_u == 2 ? kAPlane3U2 : kAPlane3;
        const long long im2col = c.M * c.K * 2;
        const long long partial = c.M * c.C_out * 4;
        best.splits = choose_splits((long long)best.m_tiles * best.n_tiles, best.num_kb, partial,
                                    im2col / 2);
        if (best.splits > 1) best.tma_store = 0;
    }
    return best;
}

bool plane_applies(const ConvShape& c) { return plan_plane(c, 0).stages >= 2; }

bool fold_applies(const ConvShape& c)
{
    return fold_geom(c).ok && plan_gemm_ring(CONVGB_PATH_WINFOLD, c).stages >= 2;
}

bool stemwin_applies(const ConvShape& c)
{
    if (!stemwin_geom(c).ok) return false;
    const GemmPlan g = plan_gemm_ring(CONVGB_PATH_STEMWIN, c);
    return g.stages >= 2;
}

// Operand producers, tiles, splits and the shared-memory ring.
GemmPlan plan_gemm_ring(int path, const ConvShape& c)
{
    GemmPlan g;
    if (path == CONVGB_PATH_WINDOW && window_geometry(c)) {
        g.amode = kAWindow;
        g.M = c.M;
        g.K = c.K;
        g.win_wv = c.W_out + (c.KW - 1) * c.d;
        g.win_rows = 128 / g.win_wv;
        g.m_step = g.win_rows;
        // A slot = the staged rows only; the MMAs' reads past them (for discarded
        // outputs) land in the next slot or, after the last, in a pad of
        // extra_smem bytes.  On the 64->128 3x3 layer at 56x56 this makes room
        // for a fourth slot beside 144 KB of resident weights.
        g.a_stage_bytes = (g.win_rows * g.win_wv * 128 + 1023) / 1024 * 1024;
        g.extra_smem = std::max(0, window_stage_rows(c.KW, c.d) * 128 - g.a_stage_bytes);
        g.num_kb = c.KH * (c.C_in / 64);  // one K block per (kh, 64-channel block)
        g.m_tiles = (int)(((long long)c.N * c.H_out + g.win_rows - 1) / g.win_rows);
        g.bn = pick_bn(c.C_out);
        g.n_tiles = (c.C_out + g.bn - 1) / g.bn;
        // Two CTAs per MMA (256 rows) for 256-wide column tiles: each holds half
        // of the weight columns, so each SM reads half of B per MMA and a slot of
        // streamed weights takes half the shared memory.  128-wide tiles go to a
        // pair only when one CTA could not keep the weights resident (measured:
        // 97 -> 92 us on the 128-channel 3x3 layer at 56x56; with the weights
        // resident on one CTA, as on the 64->128 layer, the pair is slower).
        const int all_kb = c.KH * c.KW * (c.C_in / 64);
        const bool solo_bres =
            g.n_tiles == 1 &&
            igemm_pick_stages(g.bn, 1, all_kb, g.a_stage_bytes, 1, g.extra_smem) >= 3;
        g.pair = (g.m_tiles >= 2 && (g.bn == 256 || (g.bn == 128 && !solo_bres))) ? 1 : 0;
        auto bnb = [&] { return g.pair ? g.bn / 2 : g.bn; };
        if (g.n_tiles == 1 &&
            igemm_pick_stages(bnb(), 1, all_kb, g.a_stage_bytes, 1, g.extra_smem) >= 3) {
            g.bres = 1;
            g.b_per_stage = 1;
            g.stages = igemm_pick_stages(bnb(), 1, all_kb, g.a_stage_bytes, 1, g.extra_smem);
        } else {
            // Streamed weights: a slot holds the KW blocks of one (kh, cc).  A
            // 256-wide column tile only on a pair with three slots beside the
            // epilogue's staging tile; otherwise 128 so that enough slots fit.
            if (g.bn > 128 && !(g.pair && igemm_pick_stages(g.bn / 2, 0, 0, g.a_stage_bytes, c.KW,
                                                            g.extra_smem + kEpiStageBytes) >= 3)) {
                g.bn = 128;
                g.n_tiles = (c.C_out + 127) / 128;
                g.pair = 0;
            }
            g.b_per_stage = c.KW;
            g.stages = igemm_pick_stages(bnb(), 0, 0, g.a_stage_bytes, c.KW, g.extra_smem);
        }
        if (g.pair) g.amode = kAWindowPair;
        const long long im2col = c.M * c.K * 2;
        const long long partial = c.M * c.C_out * 4;
        g.splits = choose_splits((long long)g.m_tiles * g.n_tiles, g.num_kb, partial, im2col / 2);
        return g;  // stages == 0 (nothing fits): see window_applies()
    }
    if (path == CONVGB_PATH_DENSE && strided_rows(c) > 0) {
        // 1x1 stride s: A straight from x by element-strided boxes, tiles of R
        // whole output rows of one image.
        const int R = strided_rows(c);
        g.amode = kAStrided;
        g.M = c.M;
        g.K = c.C_in;
        g.num_kb = (int)((g.K + 63) / 64);
        g.win_wv = c.W_out;
        g.win_rows = R;
        g.m_step = R;
        g.m_tiles = (int)((long long)c.N * c.H_out / R);
        g.bn = pick_bn(c.C_out);
        g.n_tiles = (c.C_out + g.bn - 1) / g.bn;
        // Weights resident: the whole matrix, or with several column tiles the
        // CTA's own one (each CTA then takes the tiles of one column tile only)
        // when it leaves a 4-deep ring beside the epilogue's staging.
        if ((g.n_tiles == 1 && igemm_pick_stages(g.bn, 1, g.num_kb, g.a_stage_bytes, 1) >= 4) ||
            igemm_pick_stages(g.bn, 1, g.num_kb, g.a_stage_bytes, 1, kEpiStageBytes) >= 4)
            g.bres = 1;
        g.stages = igemm_pick_stages(g.bn, g.bres, g.num_kb, g.a_stage_bytes, 1);
        return g;
    }
    if (path == CONVGB_PATH_WINFOLD) {
        // One A stage per tile: the R staged input rows of its segment.
        // Accumulator slots of 128 columns (256 when the MMA is wider).
        const FoldGeom f = fold_geom(c);
        g.amode = (c.KW <= kFold3MaxK && c.KH <= kFold3MaxK) ? kAWinFold3 : kAWinFold;
        if (!f.ok) return g;  // stages == 0: not applicable
        g.M = c.M;
        g.K = (long long)c.KH * 32;
        g.num_kb = 1;
        g.m_step = 1;
        g.m_tiles = (int)f.tiles;
        g.bn = f.n_mma <= 128 ? 128 : 256;
        g.n_tiles = 1;
        g.bres = 1;
        g.a_stage_bytes = f.R * kFoldRowBytes;
        // one stage per accumulator slot (four of 128 columns, two of 256; two
        // pairs of 128 for units of two tiles): a unit's one commit frees both
        const int st = f.U == 2 * kFoldRows ? 2 : g.bn == 128 ? 4 : 2;
        g.stages = fold_smem_bytes(f.b_bytes, st, g.a_stage_bytes) <= smem_limit() ? st : 0;
        g.min_stages = st;
        return g;
    }
    if (path == CONVGB_PATH_STEMWIN) {
        // A stages built in shared memory from staged input rows; one stage per
        // kernel-row group, each feeding nkb K blocks; weights packed by the
        // kernel into resident tiles.
        const StemWinGeom sg = stemwin_geom(c);
        g.amode = stemwin_amode(c.s);
        if (!sg.ok) return g;  // stages == 0: not applicable
        g.M = c.M;
        g.K = (long long)sg.groups * sg.nkb * 64;
        g.num_kb = sg.groups;
        g.win_wv = sg.seg;
        g.win_rows = sg.R;
        g.m_step = sg.R;
        g.m_tiles = (int)(((long long)c.N * c.H_out + sg.R - 1) / sg.R);
        g.bn = pick_bn(c.C_out);
        g.n_tiles = (c.C_out + g.bn - 1) / g.bn;
        if (g.n_tiles != 1) return g;  // the packed weights are one resident column tile
        g.bres = 1;
        g.a_stage_bytes = ((128 + sg.nkb - 1) * 128 + 1023) / 1024 * 1024;
        const int kbt = (int)(g.K / 64);
        for (int slots = 4; slots >= 2; slots -= 2) {
            g.nw_slots = slots;
            g.extra_smem = slots * sg.slot;
            if (igemm_pick_stages(g.bn, 1, kbt, g.a_stage_bytes, 1, g.extra_smem + kEpiStageBytes) >=
                4)
                break;
        }
        g.stages = igemm_pick_stages(g.bn, 1, kbt, g.a_stage_bytes, 1, g.extra_smem);
        // the raw weights land in the A stages before they are packed
        g.min_stages = std::max(2, (int)((sg.wbytes + g.a_stage_bytes - 1) / g.a_stage_bytes));
        if (g.stages < g.min_stages) g.stages = 0;
        return g;
    }
    if (path == CONVGB_PATH_IM2WIN) {
        // A by TMA from the window-order buffer: tiles of R whole output rows,
        // K ordered (kw, kh, ci) with each kw slice padded to KC.
        const Im2winGeom ig = im2win_geom(c);
        g.amode = kAIm2win;
        g.M = c.M;
        g.K = (long long)c.KW * ig.KC;
        g.num_kb = (int)((g.K + 63) / 64);
        g.win_wv = c.W_out;
        g.win_rows = ig.R;
        g.m_step = ig.R;
        g.m_tiles = (int)(((long long)c.N * c.H_out + ig.R - 1) / ig.R);
        g.bn = pick_bn(c.C_out);
        g.n_tiles = (c.C_out + g.bn - 1) / g.bn;
        const long long im2col = c.M * c.K * 2;
        const long long partial = c.M * c.C_out * 4;
        g.splits = choose_splits((long long)g.m_tiles * g.n_tiles, g.num_kb, partial, im2col / 2);
        if (g.n_tiles == 1 && g.splits == 1 &&
            igemm_pick_stages(g.bn, 1, g.num_kb, g.a_stage_bytes, 1) >= 4)
            g.bres = 1;
        g.stages = igemm_pick_stages(g.bn, g.bres, g.num_kb, g.a_stage_bytes, 1);
        return g;
    }
    // Gather path: TMA gather4 when a 64-column K block stays inside one tap's
    // channels, 16-byte cp.async otherwise.
    if (path == CONVGB_PATH_STEM && narrow_window_geometry(c)) {
        // Whole input rows staged per tile; weights resident (one column tile).
        const NarrowRows nr = narrow_rows(c);
        GemmPlan n;
        n.amode = kANarrowWin;
        n.M = c.M;
        n.K = (long long)c.KH * nr.kwcp;
        n.bn = pick_bn(c.C_out);
        n.num_kb = (int)((n.K + 63) / 64);
        n.win_wv = c.W_out;
        n.win_rows = nr.rows;
        n.m_step = nr.rows;
        n.m_tiles = (int)(((long long)c.N * c.H_out + nr.rows - 1) / nr.rows);
        n.n_tiles = (c.C_out + n.bn - 1) / n.bn;
        n.bres = 1;
        // Four staged-row slots when they still leave a 4-deep A ring beside the
        // epilogue's staging tile, else two.
        for (int slots = 4; slots >= 2; slots -= 2) {
            n.nw_slots = slots;
            n.extra_smem = slots * nr.slot;
            if (igemm_pick_stages(n.bn, 1, n.num_kb, n.a_stage_bytes, 1,
                                  n.extra_smem + kEpiStageBytes) >= 4)
                break;
        }
        n.stages = igemm_pick_stages(n.bn, 1, n.num_kb, n.a_stage_bytes, 1, n.extra_smem);
        if (n.n_tiles == 1 && n.stages >= 2) return n;
    }
    g.amode = path == CONVGB_PATH_DENSE  ? kADense
              : path == CONVGB_PATH_STEM ? kANarrow
              : c.C_in % 64 == 0         ? kATmaGather
                                         : kAGather;
    g.M = c.M;
    g.K = path == CONVGB_PATH_STEM ? stem_kpad(c) : c.K;
    g.bn = pick_bn(c.C_out);
    g.num_kb = (int)((g.K + 63) / 64);
    g.m_tiles = (int)((g.M + 127) / 128);
    g.n_tiles = (c.C_out + g.bn - 1) / g.bn;
    const long long im2col = c.M * c.K * 2;
    const long long partial = c.M * c.C_out * 4;
    g.splits = choose_splits((long long)g.m_tiles * g.n_tiles, g.num_kb, partial, im2col / 2);
    // TMA gather with 256-wide column tiles: two CTAs per MMA, each streaming
    // half of the weight columns (as on the window path).
    if (g.amode == kATmaGather && g.bn == 256 && g.m_tiles >= 2 && g.splits == 1) {
        g.amode = kATmaGatherPair;
        g.pair = 1;
    }
    const int bnb = g.pair ? g.bn / 2 : g.bn;
    // Layers whose whole weight matrix is one column tile: keep it in shared
    // memory for the CTA's lifetime when that still leaves a 4-deep A ring.
    // With several column tiles, a CTA keeps its own column tile's weights when
    // they leave that ring beside the epilogue's staging: the launch makes the
    // grid a multiple of the column tiles, so each CTA's tiles share one.
    if (g.splits == 1 &&
        ((g.n_tiles == 1 && igemm_pick_stages(bnb, 1, g.num_kb, g.a_stage_bytes, 1) >= 4) ||
         (g.n_tiles > 1 && !g.pair &&
          igemm_pick_stages(bnb, 1, g.num_kb, g.a_stage_bytes, 1, kEpiStageBytes) >= 4)))
        g.bres = 1;
    g.stages = igemm_pick_stages(bnb, g.bres, g.num_kb, g.a_stage_bytes, 1);
    if ((g.amode == kATmaGather || g.amode == kATmaGatherPair) &&
        g.stages < kMinGatherTurnStages) {
        // too shallow a ring for the gather warps' turns: 16-byte cp.async instead
        g.amode = kAGather;
        g.pair = 0;
        g.bres = 0;
        if (g.n_tiles == 1 && g.splits == 1 &&
            igemm_pick_stages(g.bn, 1, g.num_kb, g.a_stage_bytes, 1) >= 4)
            g.bres = 1;
        g.stages = igemm_pick_stages(g.bn, g.bres, g.num_kb, g.a_stage_bytes, 1);
    }
    return g;
}

// The window path also needs two ring slots (staged rows plus, unless the
// weights stay resident, the KW weight blocks of one (kh, cc)) to fit.
bool window_applies(const ConvShape& c)
{
    return window_geometry(c) && plan_gemm(CONVGB_PATH_WINDOW, c).stages >= 2;
}

// The gather path's plan without split K (conv2d_fwd_indirect and
// conv2d_fwd_noalloc have nowhere to keep partial sums).
GemmPlan plan_indirect(const ConvShape& c, int y_f32)
{
    GemmPlan plan = plan_gemm_ring(CONVGB_PATH_GATHER, c);
    plan.splits = 1;
    plan_epilogue(plan, c, y_f32);
    cap_stages(plan);
    return plan;
}

// Workspace regions of each path, in order; every region starts 256-byte aligned.
struct WsLayout {
    size_t win_off = 0, win_bytes = 0;  // im2win path: window-order input
    size_t ibuf_off = 0, ibuf_bytes = 0;
    size_t wpad_off = 0, wpad_bytes = 0;
    size_t part_off = 0, part_bytes = 0;
    size_t total = 0;
};

WsLayout workspace_layout(int path, const ConvShape& c)
{
    WsLayout L;
    size_t at = 0;
    const GemmPlan g = plan_gemm(path, c);
    if (g.amode == kAGather || g.amode == kATmaGather || g.amode == kATmaGatherPair ||
        g.amode == kANarrow) {
        L.ibuf_off = at;
        L.ibuf_bytes = (size_t)c.H_out * c.W_out * c.KH * c.KW * sizeof(int32_t);
        at = align_up(at + L.ibuf_bytes, kAlign);
    }
    if (path == CONVGB_PATH_IM2WIN) {
        L.win_off = at;
        L.win_bytes = (size_t)im2win_geom(c).buf_bytes;
        at = align_up(at + L.win_bytes, kAlign);
    }
    if (path == CONVGB_PATH_STEM || path == CONVGB_PATH_IM2WIN) {
        L.wpad_off = at;
        L.wpad_bytes = (size_t)c.C_out * g.K * 2;
        at = align_up(at + L.wpad_bytes, kAlign);
    }
    if (g.splits > 1 || g.sk) {
        L.part_off = at;
        L.part_bytes = (size_t)c.M * c.C_out * sizeof(float);
        at = align_up(at + L.part_bytes, kAlign);
    }
    L.total = at;
    return L;
}

struct IgemmArgs {
    const void* a_dense = nullptr;  // dense mode: [M][K] bf16
    const uint16_t* x = nullptr;    // gather modes
    const int32_t* ibuf = nullptr;
    const void* w = nullptr;        // [C_out][K] bf16
    const void* bias = nullptr;
    void* y = nullptr;
    float* partial = nullptr;       // split-K sums (plan.splits > 1)
    int y_f32 = 0;
    int C_out = 0, C_in = 1, cp = 1, taps = 1, HWo = 1;
    long long k_valid = 0, img_elems = 0;
    int img_rows = 0;    // H*W
    long long x_rows = 0;  // N*H*W
    const ConvShape* shape = nullptr;  // window mode geometry
    int pack_taps = 0, pack_cin = 0, pack_cp = 0;  // stem weight packing
};

// Tensor maps and kernel parameters, all host-side: nothing is launched here,
// so every failure is reported before the first launch of a call.
struct PreparedGemm {
    CUtensorMap ta, tb, ty;
    IgemmParams p;
    GemmPlan plan;
};

convgb_status prepare_gemm(const GemmPlan& g, const IgemmArgs& a, PreparedGemm* out)
{
    if (g.K % 8 != 0) return CONVGB_ERR_UNSUPPORTED;  // TMA row pitch must be 16-byte aligned
    memset(out, 0, sizeof *out);
    out->plan = g;
    // (the staged-window stem packs its weights in the kernel: no weight map;
    // the folded window reads them through its own 4-D map)
    if (!is_stemwin(g.amode) && !is_fold(g.amode) &&
        !encode_kmajor(&out->tb, a.w, a.C_out, g.K, g.pair ? g.bn / 2 : g.bn))
        return CONVGB_ERR_CUDA;
    if (is_fold(g.amode) &&
        (!encode_fold_x(&out->ta, a.x, *a.shape, fold_geom(*a.shape).R) ||
         !encode_fold_w(&out->tb, a.w, *a.shape)))
        return CONVGB_ERR_CUDA;
    if (g.amode == kADense && !encode_kmajor(&out->ta, a.a_dense, g.M, g.K, 128))
        return CONVGB_ERR_CUDA;
    if (g.amode == kAIm2win) {
        const Im2winGeom ig = im2win_geom(*a.shape);
        if (!encode_im2win(&out->ta, a.a_dense, *a.shape, ig.KC, ig.W_used, ig.R))
            return CONVGB_ERR_CUDA;
    }
    if (g.amode == kAStrided && !encode_strided(&out->ta, a.a_dense, *a.shape, g.win_rows))
        return CONVGB_ERR_CUDA;
    // TMA gather: x as [N*H*W][C_in], one-row boxes of 64 channels.
    if ((g.amode == kATmaGather || g.amode == kATmaGatherPair) &&
        !encode_kmajor(&out->ta, a.x, a.x_rows, a.C_in, 1))
        return CONVGB_ERR_CUDA;
    const bool plane = g.amode == kAPlane || g.amode == kAPlane3 || g.amode == kAPlane3U2;
    const bool window = is_window(g.amode);
    if (window || plane) {
        const ConvShape& c = *a.shape;
        if (!encode_window(&out->ta, a.x, c.N, c.H, c.W, c.C_in, g.win_wv)) return CONVGB_ERR_CUDA;
    }
    // TMA-store epilogue: y as [M][C_out], boxes of 64 channels x (one output row
    // for row tiles, 128 rows otherwise).
    if (g.tma_store) {
        // row tiles: the tile's win_rows output rows, consecutive in y; plane
        // tiles: one output row per box (their rows are not consecutive)
        const int box_rows = (window || g.amode == kANarrowWin || g.amode == kAIm2win ||
                              g.amode == kAStrided || is_stemwin(g.amode))
                                 ? g.win_rows * a.shape->W_out
                             : plane                             ? a.shape->W_out
                                                                 : 128;
        if (!encode_kmajor(&out->ty, a.y, g.M, a.C_out, box_rows, g.epi_c32 != 0))
            return CONVGB_ERR_CUDA;
    }
    unsigned* err = device_error_word();
    if (!err) return CONVGB_ERR_CUDA;
    IgemmParams& p = out->p;
    p.x = a.x;
    p.ibuf = a.ibuf;
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.y = a.y;
    p.M = (int)g.M;
    p.K = (int)g.K;
    p.C_out = a.C_out;
    p.C_in = a.C_in;
    p.cp = a.cp;
    p.k_valid = (int)a.k_valid;
    p.taps = a.taps;
    p.cin_div = FastDiv((uint32_t)(g.amode == kANarrow ? a.cp : a.C_in));
    p.hwo_div = FastDiv((uint32_t)a.HWo);
    p.img_elems = a.img_elems;
    p.img_rows = a.img_rows;
    p.oob_row = (int)a.x_rows;
    p.num_kb = g.num_kb;
    p.kb_total = (int)((g.K + 63) / 64);
    p.m_tiles = g.pair ? (g.m_tiles + 1) / 2 : g.m_tiles;  // work units: pairs of tiles
    p.n_tiles = g.n_tiles;
    p.splits = g.splits;
    p.split_div = FastDiv((uint32_t)g.splits);
    p.sk = g.sk;
    p.sk_iters = (long long)(g.pair ? (g.m_tiles + 1) / 2 : g.m_tiles) * g.n_tiles * g.num_kb;
    p.sk_ctas = 1;  // set at launch
    p.ntile_div = FastDiv((uint32_t)g.n_tiles);
    p.tma_store = g.tma_store;
    p.epi_bufs = g.epi_bufs;
    p.epi_c32 = g.epi_c32;
    p.stages = g.stages;
    p.bres = g.bres;
    p.m_step = g.m_step;
    p.a_stage_bytes = g.a_stage_bytes;
    p.b_per_stage = g.b_per_stage;
    if (g.amode == kANarrowWin) {
        const ConvShape& c = *a.shape;
        const NarrowRows nr = narrow_rows(c);
        p.win_wv = g.win_wv;
        p.win_rows = g.win_rows;
        p.win_groups = c.N * c.H_out;
        p.win_wout = c.W_out;
        p.ho_div = FastDiv((uint32_t)c.H_out);
        p.nw_H = c.H;
        p.nw_W = c.W;
        p.nw_KH = c.KH;
        p.nw_s = c.s;
        p.nw_p = c.p;
        p.nw_cin = c.C_in;
        p.nw_rb = nr.rb;
        p.nw_a0 = nr.a0;
        p.nw_kwc = nr.kwc;
        p.nw_kwcp = nr.kwcp;
        p.nw_slot_bytes = nr.slot;
        p.nw_slots = g.nw_slots;
    }
    if (is_stemwin(g.amode)) {
        const ConvShape& c = *a.shape;
        const StemWinGeom sg = stemwin_geom(c);
        p.w = static_cast<const uint16_t*>(a.w);
        p.win_wv = sg.seg;
        p.win_rows = sg.R;
        p.win_groups = c.N * c.H_out;
        p.win_wout = c.W_out;
        p.ho_div = FastDiv((uint32_t)c.H_out);
        p.nw_H = c.H;
        p.nw_W = c.W;
        p.nw_KH = c.KH;
        p.nw_s = c.s;
        p.nw_p = c.p;
        p.nw_cin = c.C_in;
        p.nw_rb = sg.rb;
        p.nw_a0 = sg.a0;
        p.nw_slot_bytes = sg.slot;
        p.nw_slots = g.nw_slots;
        p.sw_kc = sg.KC;
        p.sw_khg = sg.khg;
        p.sw_nkb = sg.nkb;
        p.sw_last = sg.last_steps;
        p.sw_steps = (sg.nkb - 1) * 4 + sg.last_steps;
        p.sw_kw = c.KW;
        p.sw_wbytes = (int)sg.wbytes;
    }
    if (g.amode == kAIm2win || g.amode == kAStrided) {
        const ConvShape& c = *a.shape;
        p.win_wv = c.W_out;
        p.win_rows = g.win_rows;
        p.win_groups = c.N * c.H_out;
        p.win_wout = c.W_out;
        p.ho_div = FastDiv((uint32_t)c.H_out);
        p.st_s = c.s;
    }
    if (is_fold(g.amode)) {
        const ConvShape& c = *a.shape;
        const FoldGeom f = fold_geom(c);
        p.win_wout = c.W_out;
        p.win_kw = c.KW;
        p.win_d = c.d;
        p.win_pad = c.p;
        p.x_KH = c.KH;
        p.x_W = c.W;
        p.ho_div = FastDiv((uint32_t)c.H_out);
        p.fold_g = f.G;
        p.fold_hout = c.H_out;
        p.fold_hb_div = FastDiv((uint32_t)f.HB);
        p.fold_n = f.n_mma;
        p.fold_bbytes = f.b_bytes;
        p.fold_spr_div = FastDiv((uint32_t)f.spr);
    }
    if (window) {
        const ConvShape& c = *a.shape;
        p.win_wv = g.win_wv;
        p.win_rows = g.win_rows;
        p.win_groups = c.N * c.H_out;
        p.win_wout = c.W_out;
        p.win_kw = c.KW;
        p.win_d = c.d;
        p.win_pad = c.p;
        p.win_cc = c.C_in / 64;
        p.win_tail = g.extra_smem;
        p.ho_div = FastDiv((uint32_t)c.H_out);
        p.x_H = c.H;
        p.x_W = c.W;
        p.x_KH = c.KH;
    }
    if (plane) {
        const ConvShape& c = *a.shape;
        p.win_wv = g.win_wv;
        p.win_rows = g.win_rows;
        p.win_wout = c.W_out;
        p.win_kw = c.KW;
        p.win_d = c.d;
        p.win_pad = c.p;
        p.win_cc = c.C_in / 64;
        p.x_H = c.H;
        p.x_W = c.W;
        p.x_KH = c.KH;
        p.pl_u = g.pl_u;
        p.pl_srows = g.pl_u * g.win_rows + (c.KH - 1) * c.d;
        p.pl_n = c.N;
        p.pl_hout = c.H_out;
        p.pl_nacc = g.pl_nacc;
        p.b_stages = g.b_stages;
        p.hp_div = FastDiv((uint32_t)(c.H + 2 * c.p));
    }
    if (g.stages < 2) return CONVGB_ERR_UNSUPPORTED;
    p.partial = a.partial;
    p.y_f32 = a.y_f32;
    p.y_al32 = (reinterpret_cast<uintptr_t>(a.y) & 31u) == 0 ? 1 : 0;
    p.timeout_ns = g_timeout_ns.load();
    p.err = err;
    if ((g.splits > 1 || g.sk) && a.partial == nullptr) return CONVGB_ERR_WORKSPACE;
    return CONVGB_OK;
}

// Launches the GEMM (and, for split-K, the zeroing of the partial sums before
// it and the bias/convert pass after it).
convgb_status launch_gemm(const PreparedGemm& pg, cudaStream_t st)
{
    const IgemmParams& p = pg.p;
    const bool sums = p.splits > 1 || p.sk;  // partial sums in the fp32 buffer
    if (sums &&
        cudaMemsetAsync(p.partial, 0, (size_t)p.M * p.C_out * sizeof(float), st) != cudaSuccess)
        return CONVGB_ERR_CUDA;
    if (launch_igemm(pg.plan.amode, pg.plan.bn, pg.ta, pg.tb, pg.ty, p, st) != cudaSuccess)
        return CONVGB_ERR_CUDA;
    if (sums &&
        launch_finish_split(p.partial, p.bias, p.y, p.M, p.C_out, p.y_f32, st) != cudaSuccess)
        return CONVGB_ERR_CUDA;
    return CONVGB_OK;
}

convgb_status conv_impl(int path, const void* x, const void* w, const void* bias, int N, int C_in,
                        int H, int W, int C_out, int KH, int KW, int s, int p, int d, void* y,
                        int y_dtype, void* ws, size_t ws_bytes, void* stream)
{
    ConvShape c;
    convgb_status st = make_shape(N, C_in, H, W, C_out, KH, KW, s, p, d, &c);
    if (st != CONVGB_OK) return st;
    if (!x || !w || !y) return CONVGB_ERR_INVALID_ARG;
    if (y_dtype != CONVGB_BF16 && y_dtype != CONVGB_F32) return CONVGB_ERR_INVALID_ARG;
    if (path == CONVGB_PATH_AUTO) path = select_path(c);
    if (path != CONVGB_PATH_GATHER && path != CONVGB_PATH_DENSE && path != CONVGB_PATH_STEM &&
        path != CONVGB_PATH_WINDOW && path != CONVGB_PATH_PLANE && path != CONVGB_PATH_IM2WIN &&
        path != CONVGB_PATH_STEMWIN && path != CONVGB_PATH_WINFOLD)
        return CONVGB_ERR_INVALID_ARG;
    if (!path_supports(path, c)) return CONVGB_ERR_UNSUPPORTED;
    WsLayout L = workspace_layout(path, c);
    if (ws_bytes < L.total) return CONVGB_ERR_WORKSPACE;
    if (L.total > 0 && !ws) return CONVGB_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (ws && !aligned16(ws)))
        return CONVGB_ERR_ALIGNMENT;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const GemmPlan plan = plan_gemm(path, c, y_dtype == CONVGB_F32 ? 1 : 0);

    IgemmArgs a;
    a.w = w;
    a.bias = bias;
    a.y = y;
    a.y_f32 = y_dtype == CONVGB_F32 ? 1 : 0;
    a.C_out = C_out;
    a.partial = L.part_bytes ? reinterpret_cast<float*>(wsb + L.part_off) : nullptr;
    int32_t* ibuf = nullptr;
    uint16_t* wpad = nullptr;
    if (path == CONVGB_PATH_DENSE) {
        // 1x1 stride-1: A = x as [N*H*W][C_in]; full-spatial: A = x as [N][H*W*C_in];
        // 1x1 stride s: x read by element-strided boxes.
        a.a_dense = x;
        a.shape = &c;
    } else if (path == CONVGB_PATH_WINDOW || path == CONVGB_PATH_PLANE ||
               path == CONVGB_PATH_STEMWIN || path == CONVGB_PATH_WINFOLD) {
        a.x = static_cast<const uint16_t*>(x);
        a.C_in = C_in;
        a.shape = &c;
    } else if (path == CONVGB_PATH_IM2WIN) {
        // A = the window-order buffer, B = the weights re-packed to its K order
        a.a_dense = wsb + L.win_off;
        wpad = reinterpret_cast<uint16_t*>(wsb + L.wpad_off);
        a.w = wpad;
        a.C_in = C_in;
        a.shape = &c;
    } else {
        ibuf = L.ibuf_bytes ? reinterpret_cast<int32_t*>(wsb + L.ibuf_off) : nullptr;
        a.x = static_cast<const uint16_t*>(x);
        a.ibuf = ibuf;
        a.C_in = C_in;
        a.taps = KH * KW;
        a.HWo = c.H_out * c.W_out;
        a.img_elems = (long long)H * W * C_in;
        a.img_rows = H * W;
        a.x_rows = (long long)N * H * W;
        a.shape = &c;
        if (path == CONVGB_PATH_STEM) {
            // Weights re-packed: narrow window, each kh row's KW*C_in weights
            // padded to a multiple of 8; scalar gather, each tap's channels
            // padded to cp.
            wpad = reinterpret_cast<uint16_t*>(wsb + L.wpad_off);
            a.w = wpad;
            if (plan.amode == kANarrowWin) {
                const NarrowRows nr = narrow_rows(c);
                a.pack_taps = KH;
                a.pack_cin = nr.kwc;
                a.pack_cp = nr.kwcp;
            } else {
                a.cp = stem_cp(c);
                a.k_valid = (long long)a.taps * a.cp;
                a.pack_taps = a.taps;
                a.pack_cin = C_in;
                a.pack_cp = a.cp;
            }
        }
    }
    PreparedGemm pg;
    st = prepare_gemm(plan, a, &pg);
    if (st != CONVGB_OK) return st;
    if (path == CONVGB_PATH_IM2WIN) {
        const int KC = im2win_geom(c).KC;
        if (launch_pack_im2win_weights(static_cast<const uint16_t*>(w), wpad, C_out, KH, KW, C_in,
                                       KC, cs) != cudaSuccess ||
            launch_im2win_padded(c, KC, static_cast<const uint16_t*>(x),
                                 reinterpret_cast<uint16_t*>(wsb + L.win_off), cs) != cudaSuccess)
            return CONVGB_ERR_CUDA;
    } else if (wpad && launch_pack_padded_weights(static_cast<const uint16_t*>(w), wpad, C_out,
                                                  a.pack_taps, a.pack_cin, a.pack_cp,
                                                  (int)plan.K, cs) != cudaSuccess) {
        return CONVGB_ERR_CUDA;
    }
    if (ibuf && launch_build_indirection(c, ibuf, cs) != cudaSuccess) return CONVGB_ERR_CUDA;
    return launch_gemm(pg, cs);
}

}  // namespace

// conv2d_fwd_indirect, and conv2d_fwd_noalloc with build_ibuf = 1: every
// check and the whole plan (tensor maps included) before the first launch;
// then, when asked, the indirection buffer is built into ibuf on the stream,
// and the GEMM follows.
convgb_status conv_indirect(const void* x, const void* w, const void* bias, int N, int C_in, int H,
                            int W, int C_out, int KH, int KW, int stride, int pad, int dilation,
                            int32_t* ibuf, size_t ibuf_bytes, int build_ibuf, void* y,
                            int y_dtype, void* stream)
{
    ConvShape c;
    convgb_status st = make_shape(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, &c);
    if (st != CONVGB_OK) return st;
    if (!x || !w || !y || !ibuf) return CONVGB_ERR_INVALID_ARG;
    if (y_dtype != CONVGB_BF16 && y_dtype != CONVGB_F32) return CONVGB_ERR_INVALID_ARG;
    if (!path_supports(CONVGB_PATH_GATHER, c)) return CONVGB_ERR_UNSUPPORTED;
    if (ibuf_bytes < (size_t)c.H_out * c.W_out * KH * KW * sizeof(int32_t))
        return CONVGB_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        !aligned16(ibuf))
        return CONVGB_ERR_ALIGNMENT;
    // Reusing a caller's buffer leaves no room for split-K partial sums.
    const GemmPlan plan = plan_indirect(c, y_dtype == CONVGB_F32 ? 1 : 0);
    IgemmArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.ibuf = ibuf;
    a.w = w;
    a.bias = bias;
    a.y = y;
    a.y_f32 = y_dtype == CONVGB_F32 ? 1 : 0;
    a.C_out = C_out;
    a.C_in = C_in;
    a.taps = KH * KW;
    a.HWo = c.H_out * c.W_out;
    a.img_elems = (long long)H * W * C_in;
    a.img_rows = H * W;
    a.x_rows = (long long)N * H * W;
    PreparedGemm pg;
    st = prepare_gemm(plan, a, &pg);
    if (st != CONVGB_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (build_ibuf && launch_build_indirection(c, ibuf, cs) != cudaSuccess) return CONVGB_ERR_CUDA;
    return launch_gemm(pg, cs);
}

unsigned* device_error_word()
{
    static unsigned* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned*>(a);
    }
    return addr[dev];
}

int num_sms()
{
    static std::atomic<int> sms[kMaxDevices] = {};
    int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    int v = sms[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
            v = 148;
        sms[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace convgb

using namespace convgb;

extern "C" {

const char* convgb_status_string(int s)
{
    switch (s) {
    case CONVGB_OK: return "ok";
    case CONVGB_ERR_INVALID_ARG: return "invalid argument";
    case CONVGB_ERR_UNSUPPORTED: return "unsupported shape or path";
    case CONVGB_ERR_WORKSPACE: return "workspace or buffer too small";
    case CONVGB_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case CONVGB_ERR_CUDA: return "CUDA runtime or launch failure";
    case CONVGB_ERR_INTERNAL: return "device-side failure (pipeline wait timed out)";
    default: return "unknown status";
    }
}

convgb_status convgb_output_dims(int H, int W, int KH, int KW, int stride, int pad, int dilation,
                                 int* H_out, int* W_out)
{
    if (H < 1 || W < 1 || KH < 1 || KW < 1 || stride < 1 || pad < 0 || dilation < 1)
        return CONVGB_ERR_INVALID_ARG;
    long long ho = out_extent(H, KH, stride, pad, dilation);
    long long wo = out_extent(W, KW, stride, pad, dilation);
    if (ho < 1 || wo < 1) return CONVGB_ERR_INVALID_ARG;
    if (H_out) *H_out = (int)ho;
    if (W_out) *W_out = (int)wo;
    return CONVGB_OK;
}

int convgb_select_path(int N, int C_in, int H, int W, int C_out, int KH, int KW, int stride,
                       int pad, int dilation)
{
    ConvShape c;
    if (make_shape(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, &c) != CONVGB_OK) return -1;
    return select_path(c);
}

size_t convgb_conv2d_fwd_path_workspace_size(int path, int N, int C_in, int H, int W, int C_out,
                                             int KH, int KW, int stride, int pad, int dilation)
{
    ConvShape c;
    if (make_shape(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, &c) != CONVGB_OK) return 0;
    if (path == CONVGB_PATH_AUTO) path = select_path(c);
    if (!path_supports(path, c)) return 0;
    return workspace_layout(path, c).total;
}

size_t convgb_conv2d_fwd_workspace_size(int N, int C_in, int H, int W, int C_out, int KH, int KW,
                                        int stride, int pad, int dilation)
{
    return convgb_conv2d_fwd_path_workspace_size(CONVGB_PATH_AUTO, N, C_in, H, W, C_out, KH, KW,
                                                 stride, pad, dilation);
}

size_t convgb_im2col_bytes(int N, int C_in, int H, int W, int KH, int KW, int stride, int pad,
                           int dilation)
{
    ConvShape c;
    if (make_shape(N, C_in, H, W, 1, KH, KW, stride, pad, dilation, &c) != CONVGB_OK) return 0;
    return (size_t)c.M * (size_t)c.K * 2;
}

convgb_status conv2d_fwd(const void* x, const void* w, const void* bias, int N, int C_in, int H,
                         int W, int C_out, int KH, int KW, int stride, int pad, int dilation,
                         void* y, int y_dtype, void* workspace, size_t workspace_bytes,
                         void* stream)
{
    return conv_impl(CONVGB_PATH_AUTO, x, w, bias, N, C_in, H, W, C_out, KH, KW, stride, pad,
                     dilation, y, y_dtype, workspace, workspace_bytes, stream);
}

convgb_status conv2d_fwd_path(int path, const void* x, const void* w, const void* bias, int N,
                              int C_in, int H, int W, int C_out, int KH, int KW, int stride,
                              int pad, int dilation, void* y, int y_dtype, void* workspace,
                              size_t workspace_bytes, void* stream)
{
    return conv_impl(path, x, w, bias, N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, y,
                     y_dtype, workspace, workspace_bytes, stream);
}

convgb_status conv2d_fwd_indirect(const void* x, const void* w, const void* bias, int N, int C_in,
                                  int H, int W, int C_out, int KH, int KW, int stride, int pad,
                                  int dilation, const int32_t* ibuf, size_t ibuf_bytes, void* y,
                                  int y_dtype, void* stream)
{
    return conv_indirect(x, w, bias, N, C_in, H, W, C_out, KH, KW, stride, pad, dilation,
                         const_cast<int32_t*>(ibuf), ibuf_bytes, 0, y, y_dtype, stream);
}

size_t convgb_indirection_buffer_bytes(int H, int W, int KH, int KW, int stride, int pad,
                                       int dilation)
{
    int ho = 0, wo = 0;
    if (convgb_output_dims(H, W, KH, KW, stride, pad, dilation, &ho, &wo) != CONVGB_OK) return 0;
    return (size_t)ho * wo * KH * KW * sizeof(int32_t);
}

convgb_status build_indirection_buffer(int H, int W, int C_in, int KH, int KW, int stride, int pad,
                                       int dilation, int32_t* ibuf, size_t ibuf_bytes,
                                       void* stream)
{
    ConvShape c;
    convgb_status st = make_shape(1, C_in, H, W, 1, KH, KW, stride, pad, dilation, &c);
    if (st != CONVGB_OK) return st;
    if (!ibuf) return CONVGB_ERR_INVALID_ARG;
    if (!aligned16(ibuf)) return CONVGB_ERR_ALIGNMENT;
    if (ibuf_bytes < (size_t)c.H_out * c.W_out * KH * KW * sizeof(int32_t))
        return CONVGB_ERR_WORKSPACE;
    return launch_build_indirection(c, ibuf, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? CONVGB_OK
               : CONVGB_ERR_CUDA;
}

size_t convgb_im2win_bytes(int N, int C_in, int H, int W, int KH, int KW, int stride, int pad,
                           int dilation)
{
    ConvShape c;
    if (make_shape(N, C_in, H, W, 1, KH, KW, stride, pad, dilation, &c) != CONVGB_OK) return 0;
    size_t w_used = (size_t)(c.W_out - 1) * stride + (size_t)(KW - 1) * dilation + 1;
    return (size_t)N * c.H_out * w_used * KH * C_in * 2;
}

convgb_status im2win_transform(const void* x, int N, int C_in, int H, int W, int KH, int KW,
                               int stride, int pad, int dilation, void* win, size_t win_bytes,
                               void* stream)
{
    ConvShape c;
    convgb_status st = make_shape(N, C_in, H, W, 1, KH, KW, stride, pad, dilation, &c);
    if (st != CONVGB_OK) return st;
    if (!x || !win) return CONVGB_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(win)) return CONVGB_ERR_ALIGNMENT;
    size_t need = convgb_im2win_bytes(N, C_in, H, W, KH, KW, stride, pad, dilation);
    if (win_bytes < need) return CONVGB_ERR_WORKSPACE;
    size_t count = C_in % 8 == 0 ? need / 16 : need / 2;  // loop trips of the kernel
    if (count > (size_t)INT32_MAX) return CONVGB_ERR_UNSUPPORTED;
    return launch_im2win(c, static_cast<const uint16_t*>(x), static_cast<uint16_t*>(win),
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? CONVGB_OK
               : CONVGB_ERR_CUDA;
}

convgb_status convgb_check_device_errors(void* stream, unsigned int* code)
{
    if (code) *code = 0;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess) return CONVGB_ERR_CUDA;
    unsigned* addr = device_error_word();
    if (!addr) return CONVGB_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpy(&v, addr, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return CONVGB_ERR_CUDA;
    if (v == 0) return CONVGB_OK;
    if (cudaMemcpy(addr, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return CONVGB_ERR_CUDA;
    if (code) *code = v;
    return CONVGB_ERR_INTERNAL;
}

void convgb_set_wait_timeout_ns(uint64_t ns)
{
    g_timeout_ns.store(ns ? ns : 1ull);
}

convgb_status convgb_selftest_wait_timeout(uint64_t timeout_ns, void* stream)
{
    unsigned* err = device_error_word();
    if (!err) return CONVGB_ERR_CUDA;
    return launch_selftest_timeout(timeout_ns, err, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? CONVGB_OK
               : CONVGB_ERR_CUDA;
}

convgb_status convgb_plan_info(int path, int N, int C_in, int H, int W, int C_out, int KH, int KW,
                               int stride, int pad, int dilation, int y_dtype, convgb_plan* out)
{
    if (!out) return CONVGB_ERR_INVALID_ARG;
    memset(out, 0, sizeof *out);
    ConvShape c;
    convgb_status st = make_shape(N, C_in, H, W, C_out, KH, KW, stride, pad, dilation, &c);
    if (st != CONVGB_OK) return st;
    if (y_dtype != CONVGB_BF16 && y_dtype != CONVGB_F32) return CONVGB_ERR_INVALID_ARG;
    if (path == CONVGB_PATH_AUTO) path = select_path(c);
    if (!path_supports(path, c)) return CONVGB_ERR_UNSUPPORTED;
    const GemmPlan g = plan_gemm(path, c, y_dtype == CONVGB_F32 ? 1 : 0);
    const bool plane = g.amode == kAPlane || g.amode == kAPlane3 || g.amode == kAPlane3U2;
    const bool rowtiles = is_window(g.amode) ||
                          g.amode == kANarrowWin || g.amode == kAIm2win || g.amode == kAStrided ||
                          is_stemwin(g.amode);
    out->path = path;
    out->a_mode = g.amode;
    out->bn = g.bn;
    out->m_tiles = g.m_tiles;
    out->tile_rows = (plane || is_fold(g.amode)) ? 0 : rowtiles ? g.m_step * c.W_out : 128;
    out->n_tiles = g.n_tiles;
    out->splits = g.splits;
    out->k_blocks = g.num_kb;
    out->stages = g.stages;
    out->weights_resident = g.bres;
    out->cta_pair = g.pair;
    out->tma_store = g.tma_store;
    out->epilogue_tiles = g.tma_store ? g.epi_bufs : 0;
    out->epilogue_c32 = g.epi_c32;
    out->stream_k = g.sk;
    out->segment_outputs = is_fold(g.amode) ? fold_geom(c).G : 0;
    out->segment_rows = is_fold(g.amode) ? fold_geom(c).U : 0;
    return CONVGB_OK;
}

void convgb_set_tuning(int bn, int max_stages, int stream_k)
{
    g_tune_bn.store((bn == 32 || bn == 64 || bn == 128 || bn == 256) ? bn : 0);
    g_tune_stages.store((max_stages >= 2 && max_stages <= 8) ? max_stages : 0);
    g_tune_stream_k.store(stream_k == 1 ? 1 : 0);
}

int convgb_version(void) { return 102; }

}  // extern "C"
