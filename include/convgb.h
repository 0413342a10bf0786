/*
 * convgb.h -- C ABI of the GB300 (sm_103a) forward-convolution library.
 *
 * The library computes the forward 2D convolution
 *
 *   Y[n,co,ho,wo] = bias[co] + sum_{ci,kh,kw} X[n,ci,ho*s+kh*d-p, wo*s+kw*d-p] * W[co,ci,kh,kw]
 *
 * ("Unifying Convolutions and GEMM", section 1, the 7-loop convolution; its
 * section 5 adds zero padding and bias; "The Indirect Convolution Algorithm",
 * Abstract, adds dilation) as an implicit GEMM of
 *   M = N*H_out*W_out rows (output pixels), N_gemm = C_out columns,
 *   K = KH*KW*C_in reduction
 * ("Unifying Convolutions and GEMM", sections 2-3: Y_col = X_col * W_row^T),
 * without ever materialising X_col (im2col).  The A operand is gathered
 * through an indirection buffer ("The Indirect Convolution Algorithm",
 * Abstract) straight into shared memory and fed to tcgen05 tensor-core MMA.
 *
 * Conventions for every entry point
 *  - Layouts are channels-last: x is [N][H][W][C_in], w is [C_out][KH][KW][C_in],
 *    y is [N][H_out][W_out][C_out], all dense; bias is [C_out].  Inputs are bf16
 *    (raw 16-bit patterns); y is bf16 or fp32 (fp32 accumulation either way).
 *  - Stride, padding and dilation are symmetric scalars: s >= 1, p >= 0, d >= 1.
 *    H_out = floor((H + 2p - d(KH-1) - 1)/s) + 1, likewise W_out; a shape with
 *    H_out < 1 or W_out < 1 is rejected.
 *  - Pointers named x, w, bias, y, workspace, scratch, win, ibuf are DEVICE pointers
 *    owned by the caller, who must keep them alive until the work queued on
 *    `stream` has finished.  The library allocates no memory per call.
 *    They must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  All work is queued asynchronously on it and on no other stream
 *    (conv2d_fwd_host adds streams of its own, joined to `stream`).
 *  - Every argument, shape, alignment and workspace check happens before the
 *    first launch; a failed check returns an error and queues nothing.
 *    A failed launch returns CONVGB_ERR_CUDA.  Kernels never trap: a device-side
 *    failure (a pipeline wait that timed out) is recorded in a device error word
 *    that convgb_check_device_errors() reads.
 *  - Calls on the same device may run concurrently only on distinct output and
 *    workspace buffers.  Element counts are limited to what the int32 index
 *    arithmetic allows: each of N*H*W*C_in, N*H_out*W_out*C_out and
 *    C_out*KH*KW*C_in must be below 2^31.
 */
#ifndef CONVGB_H
#define CONVGB_H

#include <stddef.h>
#include <stdint.h>

/* Every entry point below is exported from libconvgb.so. */
#if defined(__GNUC__)
#define CONVGB_API __attribute__((visibility("default")))
#else
#define CONVGB_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum convgb_status {
    CONVGB_OK = 0,
    CONVGB_ERR_INVALID_ARG = 1, /* bad shape, null pointer, unknown dtype or path */
    CONVGB_ERR_UNSUPPORTED = 2, /* valid convolution this library does not handle */
    CONVGB_ERR_WORKSPACE = 3,   /* workspace or output buffer smaller than required */
    CONVGB_ERR_ALIGNMENT = 4,   /* a device pointer is not 16-byte aligned */
    CONVGB_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
    CONVGB_ERR_INTERNAL = 6     /* device-side failure (wait timeout) reported by a kernel */
} convgb_status;

typedef enum convgb_dtype {
    CONVGB_BF16 = 0,
    CONVGB_F32 = 1
} convgb_dtype;

/* Kernel family conv2d_fwd_path() may be asked for; conv2d_fwd() picks one. */
typedef enum convgb_path {
    CONVGB_PATH_AUTO = 0,
    CONVGB_PATH_GATHER = 1,   /* implicit GEMM, A gathered through the indirection buffer */
    CONVGB_PATH_DENSE = 2,    /* plain GEMM: 1x1 stride-1 unpadded, or a kernel covering the
                                 whole unpadded image (a dense layer); no workspace */
    CONVGB_PATH_STEM = 3,     /* C_in not a multiple of 8: each tap's channels padded to 4
                                 (C_in <= 4) or to a multiple of 8, scalar gather */
    CONVGB_PATH_WINDOW = 4,   /* stride 1, C_in % 64 == 0, W_out + (KW-1)*d <= 128 and
                                 (KW-1)*d <= 8: tiles of whole output rows; each input row
                                 is staged in shared memory once per (kh, 64-channel block)
                                 by TMA and read by all KW taps ("Im2win", Abstract: the
                                 window order and its continuous accesses, on chip) */
    CONVGB_PATH_PLANE = 5,    /* the window path's shapes: the batch read as one tall image
                                 of padded rows, tiles of whole padded rows; each input row
                                 is staged once per (tile, 64-channel block) and read by all
                                 KH*KW taps; rows and columns of the padding border are
                                 computed and discarded.  No workspace. */
    CONVGB_PATH_IM2WIN = 6,   /* C_in < 16, undilated, W_out <= 128: x re-laid out in window
                                 order ("Im2win", Abstract), each column's (kh, ci) vector
                                 padded to a multiple of 8; every output pixel's A row is then
                                 one contiguous run of KW columns, loaded by TMA.  Workspace:
                                 the re-laid-out input (less than half of im2col, else the
                                 path does not apply) and the re-packed weights. */
    CONVGB_PATH_STEMWIN = 7,  /* C_in = 3, stride 1, 2 or 4, undilated, W_out + ceil(KW/s) - 1
                                 <= 128, at most 16 MMA steps of 16 per stage (KW*KC <= 256,
                                 KC = 64/s), C_in*W*2 and C_out*KH*KW*C_in*2 multiples of 16,
                                 C_out <= 256: the window order of "Im2win" (Abstract) built
                                 in shared memory per output row, with each output pixel's
                                 next s input columns one 128-byte row further on, so the
                                 tensor core reads every K block of the window from the same
                                 rows at shifted starts.  No workspace: nothing goes through
                                 HBM but x, w and y. */
    CONVGB_PATH_WINFOLD = 8   /* C_in = 32, stride 1, W >= 32, C_out a multiple of 32,
                                 KW <= 5, KH <= 7, KW*C_out <= 256, (KW-1)*d <= 24, d <= 8:
                                 the window order of "Im2win" (Abstract) with the KW taps
                                 folded into the tensor core's columns.  Segments of 32
                                 consecutive input columns (inside the row) of an output
                                 row's KH input rows are staged by one TMA box each (rows
                                 outside the image read as zero); one MMA chain over K =
                                 KH*32 gives, per input column, each tap's partial sums for
                                 all C_out (KW*C_out columns), and the epilogue adds, for
                                 each output pixel, tap kw's share from the column it reads
                                 (taps in the padding are left out).  A segment yields
                                 32 - (KW-1)*d output pixels.  No workspace. */
} convgb_path;

/* Short English text for a status code; never NULL. */
CONVGB_API const char* convgb_status_string(int status);

/* Output extent of the convolution (the formula above).  Returns
 * CONVGB_ERR_INVALID_ARG for a bad parameter or an empty output. */
CONVGB_API convgb_status convgb_output_dims(int H, int W, int KH, int KW, int stride, int pad,
                                 int dilation, int* H_out, int* W_out);

/* The path conv2d_fwd() takes for this shape (a CONVGB_PATH_* value), or -1
 * when the shape is invalid or unsupported. */
CONVGB_API int convgb_select_path(int N, int C_in, int H, int W, int C_out, int KH, int KW,
                       int stride, int pad, int dilation);

/* Bytes of workspace conv2d_fwd() needs for this shape on the path it selects,
 * or 0 for an invalid shape.  It holds the indirection buffer (gather and stem
 * paths), the stem path's re-packed weights, and, for layers with too few
 * output tiles to fill the GPU, fp32 partial sums of a split K loop
 * (M*C_out*4 bytes, used only when that is under half the im2col size).
 * 1x1 stride-1 layers need none.  For the benchmark layers the total is a
 * small fraction of convgb_im2col_bytes(); only tiny images with many output
 * channels can exceed it. */
CONVGB_API size_t convgb_conv2d_fwd_workspace_size(int N, int C_in, int H, int W, int C_out, int KH,
                                        int KW, int stride, int pad, int dilation);

/* As above for an explicitly requested path. */
CONVGB_API size_t convgb_conv2d_fwd_path_workspace_size(int path, int N, int C_in, int H, int W,
                                             int C_out, int KH, int KW, int stride,
                                             int pad, int dilation);

/* Bytes an explicit bf16 im2col matrix would take: N*H_out*W_out*C_in*KH*KW*2
 * ("Unifying Convolutions and GEMM", section 2: X_col has (N*H_out*W_out) rows
 * of C_in*KH*KW entries).  The comparator for the workspace claim; 0 if invalid. */
CONVGB_API size_t convgb_im2col_bytes(int N, int C_in, int H, int W, int KH, int KW, int stride,
                           int pad, int dilation);

/*
 * How conv2d_fwd_path() maps a shape onto the implicit-GEMM kernel: the plan
 * it would launch.  (An interface addition of this library for tests,
 * benchmarks and tuning; the pages describe no plan.)  The GEMM of
 * "Unifying Convolutions and GEMM", sections 2-3, is cut into output tiles of
 * `tile_rows` consecutive GEMM rows (output pixels in (n, ho, wo) order) by
 * `bn` columns (output channels).
 */
typedef struct convgb_plan {
    int path;             /* the CONVGB_PATH_* value the call takes */
    int a_mode;           /* how the A operand reaches shared memory (kernel-internal code) */
    int bn;               /* GEMM columns (output channels) per tile */
    int m_tiles;          /* tiles along M */
    int tile_rows;        /* GEMM rows per tile: tile t covers rows [t*tile_rows,
                             (t+1)*tile_rows) of M; 0 when a tile is not one range of M
                             (the plane path, whose tiles hold padding-border pixels) */
    int n_tiles;          /* tiles along C_out */
    int splits;           /* K partitions per tile (1: none; >1: fp32 partial sums) */
    int k_blocks;         /* pipeline stages per tile (one K block each) */
    int stages;           /* shared-memory ring depth */
    int weights_resident; /* 1: the whole weight column tile stays in shared memory */
    int cta_pair;         /* 1: tiles run on pairs of CTAs (tcgen05 cta_group::2) */
    int tma_store;        /* 1: the epilogue stores y through shared memory with TMA */
    int epilogue_tiles;   /* staging tiles of that epilogue (0, 1 or 2) */
    int epilogue_c32;     /* 1: 32-column staging chunks instead of 64 */
    int stream_k;         /* 1: each CTA (pair) takes an equal share of all (tile, K block)
                             steps; tiles split between CTAs meet in fp32 partial sums */
    int segment_outputs;  /* CONVGB_PATH_WINFOLD: output pixels per segment, G (0 on other
                             paths).  Each output row is cut into spr = ceil(W_out / G)
                             segments of G pixels (the last one shorter) and the
                             output rows of an image into HB = ceil(H_out / U) blocks
                             of U = segment_rows; tile t = (n*HB + hb)*spr + k holds
                             segment k of rows U*hb .. U*hb + U - 1 of image n, so
                             tile_rows is 0 */
    int segment_rows;     /* CONVGB_PATH_WINFOLD: output rows per tile, U (4, or 8 for
                             kernels up to 3x3 whose MMA is at most 128 columns wide;
                             0 on other paths) */
} convgb_plan;

/* Fills *plan with what conv2d_fwd_path(path, ...) would launch for this shape
 * and y_dtype; nothing is launched.  Returns the same shape and path errors as
 * conv2d_fwd_path (CONVGB_ERR_INVALID_ARG, CONVGB_ERR_UNSUPPORTED). */
CONVGB_API convgb_status convgb_plan_info(int path, int N, int C_in, int H, int W, int C_out,
                                          int KH, int KW, int stride, int pad, int dilation,
                                          int y_dtype, convgb_plan* plan);

/* Overrides choices of the planner for every later call in this process, for
 * tuning and ablation studies (an interface addition; not from the pages):
 * bn = 32, 64, 128 or 256 forces that tile width (0 = the planner's choice);
 * max_stages = 2..8 caps the shared-memory ring depth of the finished plan
 * (0 = no cap; the TMA-gather modes keep at least four stages);
 * stream_k = 1 lets layers whose units fill less than nine tenths of a wave
 * share out all (tile, K block) steps equally between CTAs, meeting in fp32
 * partial sums (0 = whole units, the default).  Other values mean 0.  Results
 * stay within the parity bounds, only speed changes; a setting may change the
 * workspace size, so query it after this call.  Not synchronised with calls
 * running on other host threads. */
CONVGB_API void convgb_set_tuning(int bn, int max_stages, int stream_k);

/*
 * conv2d_fwd -- forward convolution, y = conv(x, w) + bias.
 *
 * Defined by the formula at the top of this file.  Picks a path with
 * convgb_select_path(): a plain GEMM for 1x1 stride-1 unpadded layers ("The
 * Indirect Convolution Algorithm", Abstract: 1x1 convolutions are directly a
 * GEMM) and for kernels that cover the whole unpadded image ("Unifying
 * Convolutions and GEMM", section 4: such a convolution is a dense layer); a
 * channel-padding stem path when C_in is not a multiple of 8; the window path
 * for the stride-1 layers it covers; the indirection-buffer implicit GEMM for
 * everything else (strided, dilated beyond the window limits, other channel
 * counts).
 *
 *   x         device, bf16 [N][H][W][C_in]
 *   w         device, bf16 [C_out][KH][KW][C_in]
 *   bias      device, bf16 [C_out], or NULL for no bias
 *   y         device, [N][H_out][W_out][C_out] of y_dtype (CONVGB_BF16 rounds
 *             the fp32 accumulator to nearest-even; CONVGB_F32 stores it)
 *   workspace device scratch of at least convgb_conv2d_fwd_workspace_size()
 *             bytes (may be NULL when that is 0); its contents on entry are
 *             ignored and on exit are unspecified
 * Returns CONVGB_OK once the work is queued on `stream`.
 */
CONVGB_API convgb_status conv2d_fwd(const void* x, const void* w, const void* bias, int N, int C_in,
                         int H, int W, int C_out, int KH, int KW, int stride, int pad,
                         int dilation, void* y, int y_dtype, void* workspace,
                         size_t workspace_bytes, void* stream);

/* conv2d_fwd on an explicitly chosen path (a CONVGB_PATH_* value; AUTO behaves
 * like conv2d_fwd).  Returns CONVGB_ERR_UNSUPPORTED when that path cannot
 * compute this shape.  Used to cross-check paths against each other. */
CONVGB_API convgb_status conv2d_fwd_path(int path, const void* x, const void* w, const void* bias,
                              int N, int C_in, int H, int W, int C_out, int KH, int KW,
                              int stride, int pad, int dilation, void* y, int y_dtype,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * conv2d_fwd_indirect -- conv2d_fwd on the gather path with a caller-built
 * indirection buffer, for layers whose geometry repeats across calls: build
 * the buffer once with build_indirection_buffer() (same H, W, C_in, KH, KW,
 * stride, pad, dilation) and pass it here; nothing else is launched.  "The
 * Indirect Convolution Algorithm" (Abstract) builds the buffer once per
 * layer setup in the same way.
 *
 *   ibuf  device, int32 [H_out*W_out][KH*KW] as written by build_indirection_buffer()
 * Requires C_in % 8 == 0 (CONVGB_ERR_UNSUPPORTED otherwise).  Other arguments
 * as conv2d_fwd; no workspace is needed.
 */
CONVGB_API convgb_status conv2d_fwd_indirect(const void* x, const void* w, const void* bias, int N,
                                             int C_in, int H, int W, int C_out, int KH, int KW,
                                             int stride, int pad, int dilation, const int32_t* ibuf,
                                             size_t ibuf_bytes, void* y, int y_dtype, void* stream);

/*
 * conv2d_fwd_noalloc -- conv2d_fwd's gather path for callers that cannot
 * provide a workspace.  (Not from the pages, which have no counterpart: it is
 * an interface convenience of this library.)
 *
 * Who needs it: callers whose device memory is planned and owned by a host
 * framework that offers no allocation hook, and latency-critical loops that
 * must never call cudaMalloc/cudaFree (which can synchronise the device).
 * This call allocates nothing: its scratch (the indirection buffer) lives in
 * a fixed 4 MiB array in the library's device image, which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments, layouts and results as conv2d_fwd (the caller still passes x, w,
 * bias and y).  Requires C_in % 8 == 0 (CONVGB_ERR_UNSUPPORTED otherwise) and
 * H_out*W_out*KH*KW <= 1,048,576 indirection entries (4 MiB); larger shapes
 * return CONVGB_ERR_WORKSPACE before anything is launched.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture.  Every call on a device shares the one array and rewrites all of
 * it that it uses, so nothing needs clearing; calls that may overlap on the
 * GPU (other streams, other host threads) race on it and must be serialised
 * by the caller.
 */
CONVGB_API convgb_status conv2d_fwd_noalloc(const void* x, const void* w, const void* bias, int N,
                                            int C_in, int H, int W, int C_out, int KH, int KW,
                                            int stride, int pad, int dilation, void* y,
                                            int y_dtype, void* stream);

/*
 * conv2d_fwd_host -- conv2d_fwd with x, w and bias read from HOST memory and y
 * written to host memory.  (An interface addition of this library, not from
 * the pages; what it computes is conv2d_fwd's.)
 *
 *   x_host, w_host, bias_host (NULL for no bias), y_host
 *             host memory, layouts and dtypes as conv2d_fwd.  Page-locked
 *             (pinned) buffers let the copies run at full bandwidth and overlap
 *             the computation; pageable ones work, staged by the driver.  They
 *             must stay valid, and y_host unread, until the work queued on
 *             `stream` has finished.  No alignment is required of them.
 *   scratch   DEVICE memory of at least convgb_conv2d_fwd_host_scratch_size()
 *             bytes (same shape arguments, y_dtype, and has_bias = 1 when a
 *             bias is passed), 16-byte aligned, owned by the caller; contents
 *             ignored on entry and unspecified on exit
 *
 * The batch is cut into up to four chunks of whole images.  Three streams of
 * the library (created on first use on each device and kept until the process
 * exits) copy chunk k+1 in, run conv2d_fwd on chunk k and copy chunk k-1 out at
 * the same time; each chunk's input and output sit in one of two slots of the
 * scratch.  The three streams wait for `stream` before the first copy and
 * `stream` waits for them after the last, so the call behaves like work queued
 * on `stream`.  Calls from several host threads on one device queue their work
 * one call at a time.
 *
 * Returns CONVGB_ERR_INVALID_ARG (a NULL pointer, a bad shape or y_dtype),
 * CONVGB_ERR_ALIGNMENT or CONVGB_ERR_WORKSPACE (the scratch) before any CUDA
 * call; otherwise conv2d_fwd's statuses for the chunks' shapes, or
 * CONVGB_ERR_CUDA when a copy, event or stream call fails.  On any failure
 * after the first CUDA call, whatever was queued is still joined to `stream`.
 */
CONVGB_API size_t convgb_conv2d_fwd_host_scratch_size(int N, int C_in, int H, int W, int C_out,
                                                      int KH, int KW, int stride, int pad,
                                                      int dilation, int y_dtype, int has_bias);

CONVGB_API convgb_status conv2d_fwd_host(const void* x_host, const void* w_host,
                                         const void* bias_host, int N, int C_in, int H, int W,
                                         int C_out, int KH, int KW, int stride, int pad,
                                         int dilation, void* y_host, int y_dtype, void* scratch,
                                         size_t scratch_bytes, void* stream);

/* Bytes of the indirection buffer: H_out*W_out*KH*KW*4 (0 if invalid). */
CONVGB_API size_t convgb_indirection_buffer_bytes(int H, int W, int KH, int KW, int stride, int pad,
                                       int dilation);

/*
 * build_indirection_buffer -- the indirection buffer of "The Indirect
 * Convolution Algorithm" (Abstract: the modified GEMM finds its input rows
 * through a buffer that points at pixel rows of the image), as int32 element
 * offsets.
 *
 *   ibuf  device, int32 [H_out*W_out][KH*KW].  Entry (ho*W_out + wo, kh*KW + kw)
 *         holds ((h*W) + w)*C_in with h = ho*s + kh*d - p, w = wo*s + kw*d - p,
 *         the offset of that input pixel's C_in-vector inside one image, or -1
 *         when (h, w) falls in the zero padding.  One buffer serves every image
 *         of a batch (the image offset n*H*W*C_in is added by the consumer).
 *   ibuf_bytes  capacity of ibuf; at least convgb_indirection_buffer_bytes().
 * Requires H*W*C_in < 2^31.
 */
CONVGB_API convgb_status build_indirection_buffer(int H, int W, int C_in, int KH, int KW, int stride,
                                       int pad, int dilation, int32_t* ibuf,
                                       size_t ibuf_bytes, void* stream);

/* Bytes of the im2win buffer: N*H_out*W_used*KH*C_in*2 with
 * W_used = (W_out-1)*s + (KW-1)*d + 1 (0 if invalid). */
CONVGB_API size_t convgb_im2win_bytes(int N, int C_in, int H, int W, int KH, int KW, int stride,
                           int pad, int dilation);

/*
 * im2win_transform -- window-order re-layout of "Im2win: An Efficient
 * Convolution Paradigm on GPU" (Abstract).  The abstract fixes no layout; this
 * library writes
 *
 *   win[n][ho][wc][kh][ci] = x[n][ho*s + kh*d - p][wc - p][ci]   (0 outside the image)
 *
 * for wc in [0, W_used): the KH input rows that output row ho reads are
 * interleaved column by column, so every output pixel's receptive window is
 * one contiguous run of win (stride-1, undilated) and rows are written
 * exactly once.  Bit-exact copy of bf16 values.
 *
 *   x    device, bf16 [N][H][W][C_in]
 *   win  device, bf16, at least convgb_im2win_bytes() bytes
 */
CONVGB_API convgb_status im2win_transform(const void* x, int N, int C_in, int H, int W, int KH, int KW,
                               int stride, int pad, int dilation, void* win,
                               size_t win_bytes, void* stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns CONVGB_OK, CONVGB_ERR_INTERNAL when a kernel
 * recorded a failure since the last call (its raw code in *code when code is
 * not NULL), or CONVGB_ERR_CUDA when the synchronisation itself failed. */
CONVGB_API convgb_status convgb_check_device_errors(void* stream, unsigned int* code);

/* Upper bound, in nanoseconds, on any single pipeline wait inside the kernels
 * (default 4e9).  A wait that runs past it makes the kernel record
 * CONVGB_ERR_INTERNAL, drain its own copies and return instead of hanging.
 * Applies to launches queued after the call, process-wide. */
CONVGB_API void convgb_set_wait_timeout_ns(uint64_t ns);

/* Failure-detection self-test: queues one tiny kernel whose mbarrier wait can
 * never be satisfied, bounded by timeout_ns.  The kernel gives up, records the
 * timeout in the device error word and returns; convgb_check_device_errors()
 * then reports CONVGB_ERR_INTERNAL.  Nothing faults or traps. */
CONVGB_API convgb_status convgb_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/* Library version, major*10000 + minor*100 + patch. */
CONVGB_API int convgb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONVGB_H */
