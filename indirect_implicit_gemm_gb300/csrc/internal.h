// internal.h -- declarations shared by the library's translation units.
//
// Host-side shape record, kernel parameter blocks and the launchers each
// kernel file exports to the C-ABI file.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "convgb.h"  // include/ is on the include path
#include "fastdiv.h"

namespace convgb {

// Device error word codes (low byte: what failed; upper bits: role).
enum DeviceErr : unsigned {
    kErrWaitTimeout = 1u,
};

// Role tags stored in bits 8..15 of the error word.
enum Role : unsigned {
    kRoleEpilogue = 1u,
    kRoleGather = 2u,
    kRoleMma = 3u,
    kRoleTma = 4u,
    kRoleSelftest = 5u,
};

// One convolution, with the derived GEMM extents.
struct ConvShape {
    int N, C_in, H, W, C_out, KH, KW, s, p, d;
    int H_out, W_out;
    long long M;   // N * H_out * W_out
    long long K;   // KH * KW * C_in
};

// Parameters of the implicit-GEMM kernel (A gathered or TMA-loaded, B TMA-loaded).
struct IgemmParams {
    const uint16_t* x;       // bf16 [N][H][W][C_in] (gather mode)
    const int32_t* ibuf;     // [H_out*W_out][KH*KW] element offsets or -1 (gather mode)
    const uint16_t* bias;    // bf16 [C_out] or nullptr
    void* y;                 // [M][C_out], bf16 or fp32
    int M;                   // GEMM rows
    int K;                   // GEMM reduction length (elements)
    int C_out;               // GEMM columns
    int C_in;                // channels per tap of x (gather modes)
    int cp;                  // padded channels per tap in K (narrow mode: 4 or a multiple of 8)
    int k_valid;             // taps*cp: K columns that hold data (narrow mode)
    int taps;                // KH*KW (gather modes)
    FastDiv cin_div;         // divides a K index by C_in (gather) or by cp (narrow)
    FastDiv hwo_div;         // divides a row index by H_out*W_out (gather mode)
    long long img_elems;     // H*W*C_in (gather mode)
    int img_rows;            // H*W: pixel rows per image (TMA gather mode)
    int oob_row;             // a row index past the end of x viewed as [N*H*W][C_in]
    int num_kb;              // K blocks per output tile (window mode: KH * C_in/64 stagings)
    int kb_total;            // 64-column blocks of W_row: ceil(K / 64)
    int m_tiles, n_tiles;
    int m_step;              // tile origin step: 128 GEMM rows, or win_rows output rows
    int splits;              // K partitions per output tile (1: no split)
    int sk;                  // 1: stream-K (each CTA a contiguous share of all K blocks;
                             //    partial sums added into `partial`), splits == 1
    int sk_ctas;             // stream-K: CTAs (pairs: clusters) sharing the work
    long long sk_iters;      // stream-K: units * num_kb
    FastDiv split_div;       // divides by splits
    FastDiv ntile_div;       // divides by n_tiles
    int stages;              // shared-memory ring depth (2..8)
    int a_stage_bytes;       // bytes of one A ring slot
    int b_per_stage;         // B K-blocks per ring slot (1; KW in window mode)
    // window mode (stride 1): tile = win_rows output rows of win_wv virtual
    // pixels (W_out real + (KW-1)*d spill); K block kb = (kh, cc)
    int win_wv, win_rows, win_groups, win_wout, win_kw, win_d, win_pad, win_cc;
    // window mode: bytes after the last A slot that its MMAs may still read (an
    // A slot holds the win_rows * win_wv staged rows; the MMAs read 128 + (KW-1)*d
    // rows from it, the ones past the staged rows only for discarded outputs)
    int win_tail;
    FastDiv ho_div;          // divides an output-row index (n*H_out + ho) by H_out
    int x_H, x_W, x_KH;      // window mode: input geometry (L2 prefetch of input rows)
    int st_s;                // strided 1x1 mode: the stride
    // narrow-window mode: staged input rows
    int nw_H, nw_W, nw_KH, nw_s, nw_p, nw_cin;
    int nw_rb;               // bytes per staged row (16-byte multiple)
    int nw_a0;               // byte offset of the row's data inside its staged row
    int nw_kwc, nw_kwcp;     // KW*C_in, and that padded to a multiple of 8
    int nw_slot_bytes;       // bytes of one tile's staged rows
    int nw_slots;            // staged-row slots (2 or 4)
    // staged-window stem (kAStemWin): KC = 64/s values (kh, ci) per input column,
    // sw_khg kernel rows per stage (a group), sw_nkb K blocks read from a stage,
    // the last of them sw_last 16-column steps long; the raw weights [C_out][K]
    // (sw_wbytes bytes at w) are packed into the resident B tiles by the kernel
    const uint16_t* w;
    int sw_kc, sw_khg, sw_nkb, sw_last, sw_kw, sw_wbytes;
    int sw_steps;            // 16-column MMA steps per stage: (sw_nkb - 1) * 4 + sw_last
    // plane mode (stride 1): the batch is one tall padded image of N*(H+2p)
    // virtual rows; a tile is pl_u sub-tiles of win_rows virtual output rows,
    // its A stage for channel block cc holds pl_srows whole padded input rows,
    // and tap (kh, kw) of sub-tile u reads it from row u*win_rows*win_wv +
    // kh*d*win_wv + kw*d on
    int pl_u;                // sub-tiles per tile (1 or 2), each 128 accumulator rows
    int pl_srows;            // staged input rows per A stage: pl_u*win_rows + (KH-1)*d
    int pl_n, pl_hout;       // batch and output height
    int pl_nacc;             // accumulators in tensor memory (each pl_u*BN columns)
    int b_stages;            // streamed weights: B ring slots of one 64-column block
    FastDiv hp_div;          // divides a virtual row index by H + 2p
    // folded window (kAWinFold): a tile is column segment k (fold_g output pixels
    // read through 32 input columns) of output rows 4*hb .. 4*hb + 3 of image n,
    // tile = (n * HB + hb) * spr + k (fold_spr_div divides by the segments of a
    // row, spr; fold_hb_div by the row blocks of an image, HB); MMA width fold_n =
    // KW * C_out, resident weight bytes fold_bbytes, output height fold_hout
    int fold_g, fold_n, fold_bbytes, fold_hout;
    FastDiv fold_spr_div, fold_hb_div;
    int y_al32;              // 1: y starts on a 32-byte boundary (256-bit stores allowed)
    int tma_store;           // 1: epilogue stages 64-column chunks in shared memory and
                             //    stores them with TMA (bf16 y, C_out % 8 == 0, no split)
    int epi_c32;             // TMA-store epilogue: 1 = 32-column chunks (8 KB staging tiles)
    int epi_bufs;            // TMA-store epilogue: staging tiles (2: chunk k+1 is staged
                             //    while chunk k's store still reads its tile)
    int bres;                // 1: all of W's single column tile resident in shared memory
    float* partial;          // splits > 1: fp32 [M][C_out] sums, zeroed before the launch
    int y_f32;               // 1: fp32 output, 0: bf16
    unsigned long long timeout_ns;
    unsigned* err;           // device error word
};

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_build_indirection(const ConvShape& c, int32_t* ibuf, cudaStream_t st);
cudaError_t launch_im2win(const ConvShape& c, const uint16_t* x, uint16_t* win, cudaStream_t st);
cudaError_t launch_pack_padded_weights(const uint16_t* w, uint16_t* wp, int C_out, int taps,
                                       int C_in, int cp, int k_pad, cudaStream_t st);
// im2win path: the padded window-order buffer [N*H_out][W_used][KC] and the
// weights in its K order (kw, kh, ci), [C_out][KW*KC].
cudaError_t launch_im2win_padded(const ConvShape& c, int KC, const uint16_t* x, uint16_t* win,
                                 cudaStream_t st);
cudaError_t launch_pack_im2win_weights(const uint16_t* w, uint16_t* wp, int C_out, int KH, int KW,
                                       int C_in, int KC, cudaStream_t st);

// How the A operand reaches shared memory.
enum AMode : int {
    kADense = 0,   // TMA tiles of a dense [M][K] matrix (1x1 stride-1, full-spatial)
    kAGather = 1,  // cp.async 16-byte pixel chunks through the indirection buffer (C_in % 8 == 0)
    kANarrow = 2,  // scalar loads through the indirection buffer, channels padded to cp (stem)
    kATmaGather = 3,  // TMA tile::gather4 of pixel rows named by the indirection buffer
                      // (C_in % 64 == 0)
    kAWindow = 4,     // stride 1: whole output rows per tile; each input row is staged once
                      // per (kh, 64-channel block) and read by all KW taps at shifted starts
    kANarrowWin = 5,  // small C_in: whole input rows bulk-copied to shared memory per tile,
                      // A built from them; K ordered (kh, kw*C_in) with each kh slice
                      // padded to a multiple of 8
    kAPlane = 6,      // stride 1: tiles of whole padded rows of the stacked batch; each
                      // input row is staged once per (tile, 64-channel block) and read by
                      // all KH*KW taps at shifted starts; weights resident or streamed
                      // one block per ring slot
    kAPlane3 = 7,     // plane mode for 3x3 kernels, one sub-tile: the MMA issue sequence
                      // of a staged block is unrolled at compile time
    kAPlane3U2 = 8,   // plane mode for 3x3 kernels, two sub-tiles per weight block
    kAWindowPair = 9, // window mode on a cluster of two CTAs: one tcgen05.mma.cta_group::2
                      // covers both CTAs' output tiles (256 rows); each CTA holds half of
                      // the weight columns
    kAIm2win = 10,    // A rows read by 3-D TMA boxes from a padded im2win buffer: output
                      // pixel wo of output row g is the contiguous run of KW columns from
                      // column wo*s of row g (rows overlap; tiles of whole output rows)
    kAStrided = 11,   // 1x1 stride-s unpadded layers: A read from x itself by 4-D TMA boxes
                      // with element strides (1, s, s, 1), only the pixels the output
                      // uses; tiles of whole output rows of one image
    kATmaGatherPair = 12,  // TMA gather4 on a cluster of two CTAs (tcgen05.mma.cta_group::2,
                           // 256 rows); each CTA holds half of the weight columns
    kAStemWin = 13,   // three input channels, stride 2 (kAStemWin1, kAStemWin4: stride 1, 4):
                      // per tile, a window-order stage in shared memory whose 128-byte row
                      // r holds input columns s*r-p .. s*r-p+s-1, each as KC = 64/s values
                      // (kh, ci); output pixel wo's K block kb is row wo + kb, so one stage
                      // feeds every K block at shifted starts.  One kernel per stride: each
                      // holds the one stage builder it runs (with the builders of all three
                      // strides in one kernel the 7x7 stride-2 stem ran 100 us, not 65)
    kAStemWin1 = 14,
    kAStemWin4 = 15,
    kAWinFold = 16,   // C_in = 32, stride 1: the KW taps folded into the MMA's columns.  A
                      // tile is one 32-column segment (inside the image row) of four
                      // consecutive output rows, one per TMEM lane quarter; one TMA box
                      // stages its 4 + (KH-1)*d input rows and tap row kh reads them from
                      // kh*d rows on.  A row r is input column c0 + (r % 32) with K = (kh,
                      // ci); B row (kw, co) holds w[co][kh][kw][ci]; the epilogue sums, for
                      // each output pixel, column block kw of the row holding its tap-kw
                      // column (warp shuffles; taps in the padding are left out), so a
                      // segment yields 32 - (KW-1)*d output pixels per row
    kAWinFold3 = 17,  // the folded window for kernels of at most 3 x 3: the same kernel with
                      // its tap loops unrolled to 3 (measured on the 32-channel 3x3 layer at
                      // 150x150: 111.7 us against 126.4 us with loops sized for 7 x 5)
    kAWindowT = 18,   // the window mode's common plan fixed at compile time: KW = 3, resident
                      // weights, TMA-store epilogue in 64-column chunks, no split, no stream-K
                      // (the kernel is smaller: 64-channel 3x3 layer at 112x112 158.9 ->
                      // 145.3 us, 64->128 at 56x56 17.4 -> 16.9 us, in a timing copy)
};
constexpr bool is_window(int amode)
{
    return amode == kAWindow || amode == kAWindowPair || amode == kAWindowT;
}
constexpr bool is_fold(int amode) { return amode == kAWinFold || amode == kAWinFold3; }
// The folded window's limits: kernel width (registers of the epilogue's shuffle
// sum), kernel height (the unrolled MMA sequence), for kAWinFold and for
// kAWinFold3; output rows per tile and bytes of one staged input row segment (32
// columns of 32 channels).
constexpr int kFoldMaxKW = 5;
constexpr int kFoldMaxKH = 7;
constexpr int kFold3MaxK = 3;
constexpr int kFoldRows = 4;
constexpr int kFoldRowBytes = 32 * 64;
constexpr int kFoldBiasBytes = 1024;  // the bias as fp32, after the A stages
// The staged-window stem's A mode for a stride (1, 2 or 4).
constexpr int stemwin_amode(int s) { return s == 1 ? kAStemWin1 : s == 4 ? kAStemWin4 : kAStemWin; }
constexpr bool is_stemwin(int amode)
{
    return amode == kAStemWin || amode == kAStemWin1 || amode == kAStemWin4;
}
// Fewest ring stages the TMA-gather modes run with: their four gather warps
// fill the stages by turns, and each warp's wait on a stage's release must be
// at most one barrier phase ahead of it.
constexpr int kMinGatherTurnStages = 4;
// Dynamic shared memory of one implicit-GEMM CTA, and the deepest ring that fits
// (0 when none does).
int igemm_smem_bytes(int bn, int stages, int bres, int num_kb, int a_stage_bytes,
                     int b_per_stage, int extra_bytes = 0);
int igemm_pick_stages(int bn, int bres, int num_kb, int a_stage_bytes, int b_per_stage,
                      int extra_bytes = 0);
// Rows that window-mode MMAs read from an A ring slot (128 plus the tap spill,
// rounded to 8).
int window_stage_rows(int kw, int d);
// Dynamic shared memory of a folded-window CTA: resident weights of b_bytes
// (a multiple of 1024), `stages` A stages and the fp32 bias.
int fold_smem_bytes(int b_bytes, int stages, int a_stage_bytes);
// Dynamic shared memory of a plane-mode CTA: a_stages A slots, b_blocks weight
// blocks (resident or ring), plus extra bytes.
int plane_smem_bytes(int bn, int a_stages, int a_stage_bytes, int b_blocks, int extra_bytes);
int smem_limit();
cudaError_t launch_igemm(int amode, int bn, const CUtensorMap& tmap_a,
                         const CUtensorMap& tmap_b, const CUtensorMap& tmap_y,
                         const IgemmParams& p, cudaStream_t st);
// Shared memory the TMA-store epilogue adds: one staging tile (128 x 64 bf16)
// and the column tile's bias; a second staging tile when double-buffered.
constexpr int kEpiTileBytes = 16384;
constexpr int kEpiStageBytes = kEpiTileBytes + 1024;
// Narrow staging: 32-column chunks, a 128 x 64-byte tile with 64-byte swizzle.
constexpr int kEpiNarrowTileBytes = 8192;
constexpr int kEpiNarrowStageBytes = kEpiNarrowTileBytes + 1024;
cudaError_t launch_finish_split(const float* partial, const uint16_t* bias, void* y, long long M,
                                int C_out, int y_f32, cudaStream_t st);
cudaError_t launch_selftest_timeout(unsigned long long timeout_ns, unsigned* err,
                                    cudaStream_t st);

// Shared helpers from api.cu.
unsigned* device_error_word();  // address of this device's error word (host-visible pointer)
int num_sms();
// The gather-path convolution with the indirection buffer at `ibuf`: every
// check and the plan first, nothing launched on failure; then, if build_ibuf,
// the buffer is built into ibuf on the stream; then the GEMM (no split K).
convgb_status conv_indirect(const void* x, const void* w, const void* bias, int N, int C_in, int H,
                            int W, int C_out, int KH, int KW, int stride, int pad, int dilation,
                            int32_t* ibuf, size_t ibuf_bytes, int build_ibuf, void* y,
                            int y_dtype, void* stream);

}  // namespace convgb
