// igemm.cu -- the tcgen05 implicit-GEMM convolution kernel for sm_103a.
//
// Computes Y_col = X_col * W_row^T + bias ("Unifying Convolutions and GEMM",
// sections 2-3 and 5) without forming X_col: row m of X_col (output pixel
// (n, ho, wo)) and K block kb are gathered on the fly, through the
// indirection buffer of "The Indirect Convolution Algorithm" (Abstract: the
// modified GEMM reads its A rows through pointers to input pixel rows), into a
// 128-byte-swizzled shared-memory tile; W_row tiles arrive by TMA.  The GEMM
// itself runs on the fifth-generation tensor cores: one thread issues
// tcgen05.mma (bf16 x bf16 -> fp32) into accumulators in tensor memory (up to
// four, so the MMAs run ahead of the epilogue), and the epilogue warps read
// them back with tcgen05.ld, add the bias and store channels-last y through a
// staging tile and TMA.  The dense, window, plane, im2win and strided variants
// load A by TMA as well (see AMode).
//
// CTA layout (352 threads, one persistent CTA per SM; launched with
// programmatic stream serialization):
//   warps 0-3  epilogue: TMEM -> registers -> +bias -> bf16/fp32 -> global
//   warps 4-7  A gather (cp.async or TMA gather4 through the indirection
//              buffer), or four more epilogue warps where A comes by TMA
//   warp  8    TMA producer for B (and for A in the TMA-fed variants)
//   warp  9    TMEM allocation and MMA issue (lane 0)
//   warp 10    barrier waits for warp 9, handed over at a named barrier
// Stages cycle through full/empty mbarrier pairs; every wait is bounded in
// time and a timeout makes the whole CTA drain and return with an error code.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace convgb {
namespace {

constexpr int BM = 128;           // GEMM rows per tile (TMEM lanes)
constexpr int BK = 64;            // K elements per stage: one 128-byte swizzle row
constexpr int kEpiWarps = 4;
constexpr int kGatherWarps = 4;
// The MMA warp (9) and its wait warp (10) sit on schedulers 1 and 2, apart
// from the TMA producer (warp 8, scheduler 0).  In plane mode the L2-prefetch
// warp (5) shares scheduler 1 with the MMA warp and backs off between polls.
constexpr int kTmaWarp = kEpiWarps + kGatherWarps;  // 8
constexpr int kMmaWarp = kTmaWarp + 1;              // 9
// Waits on the stage and accumulator barriers for the MMA warp and hands each
// stage over at a named barrier: an mbarrier wait on the MMA-issuing warp
// stalls it until the MMAs already queued have drained (probe: +140 to +240
// cycles per stage at N <= 128), while a named-barrier hand-off costs nothing.
constexpr int kWaitWarp = kMmaWarp + 1;             // 10
constexpr int kThreads = (kWaitWarp + 1) * 32;      // 352
constexpr uint32_t kHandBar = 2;                    // named barrier of the hand-off
constexpr uint32_t kHandThreads = 64;               // the MMA warp and the wait warp
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kRowsPerGatherThread = BM * (BK / 8) / kGatherThreads;  // 8

// Shared-memory plan (all offsets from the start of dynamic shared memory):
//   [0, kHeaderBytes)   mbarriers, TMEM address slot, abort flag
//   then, aligned to 1024 bytes for the 128-byte swizzle:
//   B: `stages` ring buffers of BN x 64 K, or (weights resident) all num_kb
//      K blocks of the single BN-wide column tile, loaded once per CTA
//   A: `stages` ring buffers of 128 x 64 K
// The stage count is chosen on the host from what fits (at most kMaxStages).
constexpr int kMaxStages = 8;
constexpr int kHeaderBytes = 512;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kSmemLimit = 232448;    // opt-in dynamic shared memory per block
constexpr int kMaxAcc = 4;
constexpr int kMaxSlots = 4;  // narrow window: staged-row slots
// Staged-window stem: 16-column MMA steps per stage.  The issue sequence is
// unrolled to this length; measured on the 7x7 stride-2 stem, a 32-step
// sequence ran 111 us against 65 us at 16 (the hot loops of all roles have to
// share the instruction caches).
constexpr int kStemWinMaxSteps = 16;
static_assert((4 * kMaxStages + 2 * kMaxAcc + 3 + 2 * kMaxSlots) * 8 + 8 + 36 + 8 <= kHeaderBytes,
              "header area");

template <int BN>
struct Cfg {
    static constexpr int kBBytes = BN * BK * 2;  // one K block of B
    // Accumulators in TMEM (512 columns): up to four, so the MMAs can run up to
    // three tiles ahead of the epilogue when tiles are short.
    static constexpr int kAcc = (512 / BN) < kMaxAcc ? (512 / BN) : kMaxAcc;
    static constexpr int kTmemCols = kAcc * BN;
    static_assert(kTmemCols >= 32 && kTmemCols <= 512, "TMEM columns");
    static_assert((kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation must be a power of 2");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
};

// Advances a ring position: stage index and the parity of its current fill.
struct Ring {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t stages)
    {
        if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// Shared state every role needs for bounded waits.
struct WaitCtx {
    volatile uint32_t* abort;  // shared flag: some role gave up
    unsigned* err;
    unsigned long long timeout_ns;
};

// Waits for the phase of `bar` with the given parity.  Returns false (and the
// caller must unwind) when the wait exceeds the time limit or another role
// of this CTA has already given up.
// `cluster`: the phase is completed by arrivals from the peer CTA of a pair,
// so the wait acquires at cluster scope.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const WaitCtx& w,
                                         unsigned role, bool cluster = false)
{
    auto test = [&] {
        return cluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const unsigned long long t0 = ptx::globaltimer();
    for (uint32_t spins = 1;; ++spins) {
        if (test()) return true;
        if (*w.abort) return false;
        if ((spins & 31u) == 0 && ptx::globaltimer() - t0 > w.timeout_ns) {
            *w.abort = 1u;
            atomicCAS(w.err, 0u, kErrWaitTimeout | (role << 8));
            return false;
        }
    }
}

// Bounded wait used while unwinding: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           unsigned long long limit_ns)
{
    if (ptx::mbar_try_wait(bar, parity)) return;
    const unsigned long long t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer() - t0 > limit_ns) return;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Stores 32 accumulator columns [co0, co0+32) of row m, adding the bias.
__device__ __forceinline__ void store_chunk(const IgemmParams& p, int m, int co0,
                                            const uint32_t (&r)[32])
{
    float v[32];
    const int ncols = min(32, p.C_out - co0);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    if (p.bias != nullptr) {
        if (ncols == 32 && (p.C_out & 7) == 0) {
            const uint4* b4 = reinterpret_cast<const uint4*>(p.bias + co0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 b = __ldg(b4 + q);
                uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[q * 8 + 2 * e] += bf16_bits_to_float(static_cast<uint16_t>(w[e] & 0xFFFFu));
                    v[q * 8 + 2 * e + 1] += bf16_bits_to_float(static_cast<uint16_t>(w[e] >> 16));
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncols) v[i] += bf16_bits_to_float(__ldg(p.bias + co0 + i));
        }
    }
    const long long row = static_cast<long long>(m) * p.C_out + co0;
    if (p.y_f32) {
        float* out = static_cast<float*>(p.y) + row;
        // 256-bit stores need 32-byte addresses: y itself on a 32-byte boundary
        if (ncols == 32 && (p.C_out & 7) == 0 && p.y_al32) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                ptx::st_global_v8(out + 8 * q, __float_as_uint(v[8 * q]),
                                  __float_as_uint(v[8 * q + 1]), __float_as_uint(v[8 * q + 2]),
                                  __float_as_uint(v[8 * q + 3]), __float_as_uint(v[8 * q + 4]),
                                  __float_as_uint(v[8 * q + 5]), __float_as_uint(v[8 * q + 6]),
                                  __float_as_uint(v[8 * q + 7]));
        } else if (ncols == 32 && (p.C_out & 3) == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(out)[q] =
                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncols) out[i] = v[i];
        }
    } else {
        uint16_t* out = static_cast<uint16_t*>(p.y) + row;
        if (ncols == 32 && (p.C_out & 15) == 0 && p.y_al32) {
            // whole 32-byte sectors: two 256-bit stores
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float* w = v + 16 * h;
                ptx::st_global_v8(out + 16 * h, pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                                  pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]),
                                  pack_bf16x2(w[8], w[9]), pack_bf16x2(w[10], w[11]),
                                  pack_bf16x2(w[12], w[13]), pack_bf16x2(w[14], w[15]));
            }
        } else if (ncols == 32 && (p.C_out & 7) == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                reinterpret_cast<uint4*>(out)[q] =
                    make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]),
                               pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                               pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncols) {
                    __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
                    out[i] = *reinterpret_cast<uint16_t*>(&b);
                }
        }
    }
}

// Work unit `tile` -> output tile origin (first GEMM row, or first output row
// in window mode) and K-block range.  Units are ordered
// (m tile, n tile, K split) with the split fastest, then the n tile, so CTAs
// working at the same time share A rows in L2.
struct Unit {
    int m0, n0, kb0, kb1;
};
// Stream-K: this CTA's (or pair's) share of the flattened (unit, K block)
// iterations, [g0, g1), which starts in unit u0 and ends in unit u1.
struct SkRange {
    long long g0 = 0, g1 = 0;
    int u0 = 0, u1 = -1;
};
// Every role evaluates this once per tile, and on the MMA thread it sits
// between two tiles' MMA groups, so it uses the host-prepared multiply-shift
// dividers (a run-time division, and above all a 64-bit one, costs hundreds of
// cycles there).
// Pair mode: unit `tile` is a pair of consecutive output tiles, the CTA of
// rank r taking tile 2*m + r.
// SK: the kernel is built with stream-K (window modes only: every other mode's
// loops stay as short as before, which matters to the instruction caches).
template <int BN, bool PAIRED, bool SK>
__device__ __forceinline__ Unit unit_of(const IgemmParams& p, int tile, uint32_t rank,
                                        const SkRange& sk)
{
    if (SK && p.sk) {
        // stream-K: the CTA's tile-th segment, unit u0 + tile, cut to [g0, g1)
        const int uu = sk.u0 + tile;
        uint32_t mt = static_cast<uint32_t>(uu), nt = 0;
        if (p.n_tiles > 1) p.ntile_div.divmod(static_cast<uint32_t>(uu), mt, nt);
        Unit u;
        u.m0 = static_cast<int>(PAIRED ? 2u * mt + rank : mt) * p.m_step;
        u.n0 = static_cast<int>(nt) * BN;
        u.kb0 = tile == 0 ? static_cast<int>(sk.g0 - static_cast<long long>(sk.u0) * p.num_kb) : 0;
        u.kb1 = uu == sk.u1 ? static_cast<int>(sk.g1 - static_cast<long long>(sk.u1) * p.num_kb)
                            : p.num_kb;
        return u;
    }
    uint32_t mn = static_cast<uint32_t>(tile), ks = 0;
    if (p.splits > 1) p.split_div.divmod(static_cast<uint32_t>(tile), mn, ks);
    uint32_t mt = mn, nt = 0;
    if (p.n_tiles > 1) p.ntile_div.divmod(mn, mt, nt);
    Unit u;
    u.m0 = static_cast<int>(PAIRED ? 2u * mt + rank : mt) * p.m_step;
    u.n0 = static_cast<int>(nt) * BN;
    u.kb0 = 0;
    u.kb1 = p.num_kb;
    if (p.splits > 1) {
        const uint32_t nkb = static_cast<uint32_t>(p.num_kb);
        u.kb0 = static_cast<int>(p.split_div.div(ks * nkb));
        u.kb1 = static_cast<int>(p.split_div.div((ks + 1u) * nkb));
    }
    return u;
}

// Split-K epilogue: adds 32 fp32 columns of row m into the partial-sum buffer.
__device__ __forceinline__ void reduce_chunk(const IgemmParams& p, int m, int co0,
                                             const uint32_t (&r)[32])
{
    float* out = p.partial + static_cast<long long>(m) * p.C_out + co0;
    const int ncols = min(32, p.C_out - co0);
    if (ncols == 32 && (p.C_out & 3) == 0) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out + 4 * q),
                         "f"(__uint_as_float(r[4 * q])), "f"(__uint_as_float(r[4 * q + 1])),
                         "f"(__uint_as_float(r[4 * q + 2])), "f"(__uint_as_float(r[4 * q + 3]))
                         : "memory");
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < ncols) atomicAdd(out + i, __uint_as_float(r[i]));
    }
}

// One MMA, and a commit to the barrier at `bar` in every CTA that waits on it:
// both CTAs of a pair (multicast), or this CTA.
template <bool PAIRED>
__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t acc)
{
    if (PAIRED)
        ptx::mma_bf16_pair(d, a, b, idesc, acc);
    else
        ptx::mma_bf16(d, a, b, idesc, acc);
}
template <bool PAIRED>
__device__ __forceinline__ void mma_commit_to(uint64_t* bar, bool both = true)
{
    if (PAIRED)
        ptx::mma_commit_pair(bar, both ? 0x3 : 0x1);
    else
        ptx::mma_commit(bar);
}

// ------------------------------------------------------------ staged-window stem
// Three input channels; the stride (a template argument) fixes KC = 64/s values
// per input column and khg = KC / 3 kernel rows per group, so the builders below
// have static register indices.

// Row i of a staged-window stage (128-byte swizzle): the S input columns
// s*r - p .. s*r - p + S - 1 of tile row j (the caller's col_e is the element
// of the first of them inside a staged input row), each as KC values: value
// kl*C + ci of column q is x[h = ho*s - p + kh0 + kl][column][ci], zero where
// kh0 + kl >= KH, where row h lies outside the image (bit kh of hvalid clear),
// and in the KC - khg*C padding values.  Columns outside the image read the
// staged rows' zero borders.
template <int C, int S>
__device__ __forceinline__ void stemwin_row(uint8_t* stage, int i, const uint16_t* rows_j, int rbe,
                                            int col_e, int kh0, int KH, uint32_t hvalid)
{
    constexpr int KC = 64 / S, KHG = KC / C;
    uint32_t v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 0u;
#pragma unroll
    for (int kl = 0; kl < KHG; ++kl) {
        const int kh = kh0 + kl;
        if (kh < KH && ((hvalid >> kh) & 1u)) {
            const uint16_t* src = rows_j + kh * rbe + col_e;
#pragma unroll
            for (int q = 0; q < S; ++q)
#pragma unroll
                for (int ci = 0; ci < C; ++ci) {
                    const int idx = q * KC + kl * C + ci;
                    v[idx >> 1] |= static_cast<uint32_t>(src[q * C + ci]) << (16 * (idx & 1));
                }
        }
    }
#pragma unroll
    for (int q16 = 0; q16 < 8; ++q16)
        *reinterpret_cast<uint4*>(stage + i * 128 + ((q16 ^ (i & 7)) << 4)) =
            make_uint4(v[4 * q16], v[4 * q16 + 1], v[4 * q16 + 2], v[4 * q16 + 3]);
}

// Resident weights of the staged-window stem, from the raw [C_out][KH][KW][C_in]
// weights parked in shared memory: block b = group * nkb + kb holds, for column
// co, K value q*KC + kl*C + ci = w[co][group*khg + kl][kb*S + q][ci] (zero past
// KH, KW and khg), as 128-byte swizzled K-major rows like a TMA-loaded tile.
template <int C, int S>
__device__ __forceinline__ void stemwin_pack(uint8_t* sB, const uint16_t* raw, int bn, int C_out,
                                             int KH, int KW, int nkb, int kbt, int tid, int nthr)
{
    constexpr int KC = 64 / S, KHG = KC / C;
    const int total = kbt * bn * 8;  // 16-byte chunks
    const int rowlen = KH * KW * C;
    for (int e = tid; e < total; e += nthr) {
        const int b = e / (bn * 8);
        const int rem = e - b * bn * 8;
        const int co = rem >> 3, cc = rem & 7;
        const int grp = b / nkb, kb = b - grp * nkb;
        uint32_t v[4] = {0u, 0u, 0u, 0u};
        if (co < C_out) {
            const uint16_t* wr = raw + co * rowlen;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int k = cc * 8 + t;
                const int q = k / KC, r2 = k - q * KC;
                const int kl = r2 / C, ci = r2 - kl * C;
                const int kw = kb * S + q, kh = grp * KHG + kl;
                uint32_t val = 0u;
                if (kl < KHG && kh < KH && kw < KW) val = wr[(kh * KW + kw) * C + ci];
                v[t >> 1] |= val << (16 * (t & 1));
            }
        }
        *reinterpret_cast<uint4*>(sB + b * (bn * 128) + co * 128 + ((cc ^ (co & 7)) << 4)) =
            make_uint4(v[0], v[1], v[2], v[3]);
    }
}

template <int BN, int AMODE>
__global__ void __launch_bounds__(kThreads, 1)
    igemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                 const __grid_constant__ CUtensorMap tmap_b,
                 const __grid_constant__ CUtensorMap tmap_y, const IgemmParams p)
{
    using C = Cfg<BN>;
    // A written by the gather warps (signalled on full_a) or by the TMA warp
    // together with B (signalled on full_b).
    constexpr bool NARROWWIN = AMODE == kANarrowWin;
    constexpr bool STEMWIN = is_stemwin(AMODE);
    constexpr int SW_S = AMODE == kAStemWin1 ? 1 : AMODE == kAStemWin4 ? 4 : 2;  // its stride
    constexpr bool STAGEDROWS = NARROWWIN || STEMWIN;  // input rows bulk-copied per tile
    constexpr bool TMAGATHER = AMODE == kATmaGather || AMODE == kATmaGatherPair;
    constexpr bool GATHER =
        AMODE == kAGather || AMODE == kANarrow || TMAGATHER || NARROWWIN || STEMWIN;
    constexpr bool PAIR = AMODE == kAWindowPair || AMODE == kATmaGatherPair;  // CTA pair
    constexpr bool WINDOW = is_window(AMODE);
    // the window mode's common plan, fixed at compile time (kAWindowT); other
    // modes read it from the parameters
    constexpr bool WT = AMODE == kAWindowT;
    const int tma_store = WT ? 1 : p.tma_store;
    const int epi_c32 = WT ? 0 : p.epi_c32;
    const bool split_k = !WT && p.splits > 1;
    const bool kw3 = WT || p.win_kw == 3;
    const int bres = WT ? 1 : p.bres;
    // B block bytes in this CTA's shared memory (a pair splits B's columns)
    constexpr uint32_t BB = PAIR ? C::kBBytes / 2 : C::kBBytes;
    constexpr bool PLANE = AMODE == kAPlane || AMODE == kAPlane3 || AMODE == kAPlane3U2;
    constexpr bool IM2WIN = AMODE == kAIm2win;
    constexpr bool STRIDED = AMODE == kAStrided;
    constexpr bool FOLD = is_fold(AMODE);
    // the 3x3-sized folded window with 128-column accumulators works in units of
    // two tiles: eight output rows, one box, one hand-off and one commit, the two
    // 4-row halves in a pair of accumulators (one per epilogue warp group)
    constexpr bool FPAIR = AMODE == kAWinFold3 && BN == 128;
    // its tap loops' length (the kernel's code size matters: see kAWinFold3)
    constexpr int FKW = AMODE == kAWinFold3 ? kFold3MaxK : kFoldMaxKW;
    constexpr int FKH = AMODE == kAWinFold3 ? kFold3MaxK : kFoldMaxKH;
    constexpr bool ROWTILES = WINDOW || STAGEDROWS || IM2WIN || STRIDED;  // whole output rows
    // Modes whose gather warps have nothing to gather run the epilogue on eight
    // warps: each thread converts 32 of a 64-column chunk's columns instead of
    // all 64 (the epilogue is latency-bound with one warp per scheduler).
    constexpr bool EPI8 = WINDOW || AMODE == kADense || IM2WIN || STRIDED || FOLD;
    constexpr int kEpiN = EPI8 ? 2 * kEpiThreads : kEpiThreads;
    const uint32_t S = static_cast<uint32_t>(p.stages);
    const uint32_t AST = static_cast<uint32_t>(p.a_stage_bytes);
    extern __shared__ uint8_t smem_raw[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
    uint64_t* full_a = bars;                  // A stage ready
    uint64_t* full_b = bars + kMaxStages;     // B stage ready (tx bytes), count 1
    uint64_t* empty = bars + 2 * kMaxStages;  // MMA done with stage, count 1 (tcgen05.commit)
    uint64_t* empty_b = bars + 3 * kMaxStages;  // plane mode: MMA done with B slot, count 1
    uint64_t* tfull = bars + 4 * kMaxStages;  // accumulator ready, count 1 (tcgen05.commit)
    uint64_t* tempty = tfull + kMaxAcc;       // accumulator drained, count kEpiThreads
    uint64_t* drain = tempty + kMaxAcc;       // MMA unwinding, count 1
    uint64_t* bres_full = drain + 1;          // resident weights loaded (tx bytes), count 1
    uint64_t* stg_full = bres_full + 1;       // narrow window: tile's rows staged (tx bytes)
    uint64_t* stg_empty = stg_full + kMaxSlots;  // narrow window: staged rows consumed
    uint64_t* wpack = stg_empty + kMaxSlots;     // staged-window stem: weights packed, count 1
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wpack + 1);
    uint32_t* abort_flag = tmem_slot + 1;
    // The 128-byte swizzle is a function of shared-memory address bits, so the
    // stage buffers must start on 1024-byte boundaries of the shared window.
    const uint32_t base = ptx::smem_addr(smem_raw) + kHeaderBytes;
    uint8_t* data = smem_raw + kHeaderBytes + ((1024u - (base & 1023u)) & 1023u);
    uint8_t* sB = data;
    const uint32_t SB = PLANE ? static_cast<uint32_t>(p.b_stages) : 1u;  // plane: B ring slots
    const uint32_t b_blocks = bres ? static_cast<uint32_t>(p.kb_total)
                              : PLANE ? SB
                                      : S * static_cast<uint32_t>(p.b_per_stage);
    // Accumulators: plane mode keeps pl_u sub-tiles of BN columns per tile.
    const uint32_t NACC = PLANE ? static_cast<uint32_t>(p.pl_nacc) : static_cast<uint32_t>(C::kAcc);
    const uint32_t ACCW = PLANE ? static_cast<uint32_t>(p.pl_u * BN) : static_cast<uint32_t>(BN);
    constexpr uint32_t kTmemAlloc = PLANE ? 512u : static_cast<uint32_t>(C::kTmemCols);
    // (the folded window's resident weights: KH blocks of KW*C_out 64-byte rows)
    uint8_t* sA = data + (FOLD ? static_cast<uint32_t>(p.fold_bbytes) : b_blocks * BB);
    // narrow window: nw_slots slots of staged input rows; window: the pad that the
    // last A slot's reads past its staged rows fall into
    uint8_t* sStg = sA + S * AST + (WINDOW ? static_cast<uint32_t>(p.win_tail) : 0u);
    const uint32_t NS = STAGEDROWS ? static_cast<uint32_t>(p.nw_slots) : 1u;
    // TMA-store epilogue: a 128 x 64 bf16 staging tile (128-byte swizzle) and the
    // current column tile's bias in fp32.
    uint8_t* sEpi = sStg + (STAGEDROWS ? NS * p.nw_slot_bytes : 0);
    const int epi_tile = epi_c32 ? kEpiNarrowTileBytes : kEpiTileBytes;  // staging tile bytes
    float* sBias = reinterpret_cast<float*>(sEpi + p.epi_bufs * epi_tile);
    // folded window: the bias as fp32 right after the A stages (1 KB)
    float* sBiasF = reinterpret_cast<float*>(sA + S * AST);
    uint32_t* sVote = reinterpret_cast<uint32_t*>(abort_flag + 1);  // up to 8 epilogue-warp votes
    volatile uint32_t* sTilesDone = sVote + 8;  // tiles the epilogue has finished (plane prefetch)
    // wait warp -> MMA warp: 1 if the awaited barrier completed, 0 to unwind; two
    // words used alternately, so a word is rewritten only after the MMA warp has
    // passed the next hand-off and therefore has read it
    volatile uint32_t* sHand = sTilesDone + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Pair mode: both CTAs walk the same sequence of pair units.
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    // Work units: unit t_first, t_first + t_step, ... below total_tiles.  In
    // stream-K mode the CTA (a pair: the cluster) takes the contiguous share
    // [c*W/G, (c+1)*W/G) of the W = units * num_kb (unit, K block) iterations,
    // walked as segments 0, 1, ... of the units it touches; partial sums meet
    // in the fp32 buffer.
    const int cta_idx = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    constexpr bool SKM = WINDOW && !WT;  // stream-K is built into the window kernels only
    SkRange skr;
    if (SKM && p.sk) {
        const long long G = p.sk_ctas, W = p.sk_iters;
        skr.g0 = cta_idx * W / G;
        skr.g1 = (cta_idx + 1) * W / G;
        skr.u0 = static_cast<int>(skr.g0 / p.num_kb);
        skr.u1 = skr.g1 > skr.g0 ? static_cast<int>((skr.g1 - 1) / p.num_kb) : skr.u0 - 1;
    }
    const bool sk_on = SKM && p.sk;
    const int t_first = sk_on ? 0 : cta_idx;
    const int t_step = sk_on ? 1 : PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            // TMA gather: one arrive.expect_tx per stage; thread gathers: every thread arrives.
            ptx::mbar_init(&full_a[s], (TMAGATHER || PLANE) ? 1 : kGatherThreads);
            ptx::mbar_init(&full_b[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (uint32_t s = S; s < SB; ++s) ptx::mbar_init(&full_b[s], 1);
        for (uint32_t s = 0; s < SB; ++s) ptx::mbar_init(&empty_b[s], 1);
        for (uint32_t i = 0; i < NACC; ++i) {
            ptx::mbar_init(&tfull[i], 1);
            // (the folded window: one warp group drains each accumulator)
            ptx::mbar_init(&tempty[i], PAIR ? 2 * kEpiN : FOLD ? kEpiThreads : kEpiN);
        }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(bres_full, 1);
        ptx::mbar_init(wpack, 1);
        for (int i = 0; i < kMaxSlots; ++i) {
            ptx::mbar_init(&stg_full[i], 1);
            ptx::mbar_init(&stg_empty[i], kGatherThreads);
        }
        *sTilesDone = 0u;
        *abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    if (warp == kTmaWarp && lane == 0) {
        if (AMODE == kADense || TMAGATHER || WINDOW || PLANE || IM2WIN || STRIDED || FOLD)
            ptx::prefetch_tensormap(&tmap_a);
        if (!STEMWIN) ptx::prefetch_tensormap(&tmap_b);
    }
    if (warp == kMmaWarp) {
        if (PAIR) {
            ptx::tmem_alloc_pair(tmem_slot, kTmemAlloc);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(tmem_slot, kTmemAlloc);
            ptx::tmem_relinquish();
        }
    }
    if (STAGEDROWS) {
        // Staged rows keep their zero borders for the whole kernel: the bulk
        // copies only ever write row interiors.
        uint4* z = reinterpret_cast<uint4*>(sStg);
        const int n16 = static_cast<int>(NS) * p.nw_slot_bytes / 16;
        for (int i = threadIdx.x; i < n16; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    // a pair's barriers must be initialised before either CTA signals the other's
    if (PAIR)
        ptx::cluster_sync();
    else
        __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Up to here only this CTA's shared memory, TMEM and the kernel parameters
    // were touched.  Launched with programmatic stream serialization, the CTA
    // may have started while the previous kernel on the stream still runs on
    // other SMs: every global read or write below follows that kernel.  The
    // next kernel may begin launching at once; it waits for this one the same
    // way, so only its prologue overlaps this kernel's last tiles.
    ptx::grid_dependency_wait();
    if (threadIdx.x == 0) ptx::grid_launch_dependents();

    const WaitCtx wc{abort_flag, p.err, p.timeout_ns};
    const int total_tiles = sk_on ? skr.u1 - skr.u0 + 1 : p.m_tiles * p.n_tiles * p.splits;

    if (warp < kEpiWarps || (EPI8 && warp < kEpiWarps + kGatherWarps)) {
        // ------------------------------------------------------------ epilogue
        // This thread's accumulator row r = TMEM lane (a warp reaches the lane
        // quarter warp % 4).  Window mode: row r is virtual pixel (wrow, wcol) of
        // the tile's output rows; spill columns (wcol >= W_out) and rows past the
        // tile's output rows are discarded.  With eight warps, warp w takes the
        // 32-column half w / 4 of every 64-column chunk.
        const int quad = warp & 3;
        const int half = EPI8 ? (warp >> 2) : 0;
        const int r = quad * 32 + lane;
        const int et = EPI8 ? static_cast<int>(threadIdx.x) : r;  // index among epilogue threads
        // the accumulator is handed back to the MMA thread, which in a pair sits in CTA 0
        auto release_acc = [&](uint32_t acc) {
            ptx::tc_fence_before();
            if (PAIR && rank != 0) {
                // The peer's epilogue threads meet first and one of them arrives
                // for all: kEpiN separate remote arrivals are serialised across
                // the SM pair (measured: the peer's epilogue took 3.4 us per
                // tile against 2.05 us on CTA 0, and held the pair's exit).
                ptx::named_barrier_sync(1, kEpiN);
                if (et == 0)
                    ptx::mbar_arrive_cluster_count(ptx::mapa(ptx::smem_addr(&tempty[acc]), 0u),
                                                   static_cast<uint32_t>(kEpiN));
            } else {
                ptx::mbar_arrive(&tempty[acc]);
            }
        };
        if (STEMWIN) {
            // The raw weights land in the A stages (bres_full); pack them into the
            // resident B tiles, then release the stages to the gather warps and
            // the weights to the MMA thread (wpack).
            if (wait_bar(bres_full, 0u, wc, kRoleEpilogue))
                stemwin_pack<3, SW_S>(sB, reinterpret_cast<const uint16_t*>(sA), BN, p.C_out,
                                      p.nw_KH, p.sw_kw, p.sw_nkb, p.kb_total, et, kEpiN);
            ptx::fence_proxy_async_smem();
            ptx::named_barrier_sync(1, kEpiN);
            if (et == 0) ptx::mbar_arrive(wpack);
        }
        if (FOLD) {
            // the bias as fp32, once: every tile has the same C_out columns
            for (int i = et; i < p.C_out; i += kEpiN)
                sBiasF[i] = p.bias != nullptr ? bf16_bits_to_float(p.bias[i]) : 0.f;
            ptx::named_barrier_sync(1, kEpiN);
        }
        const int wrow = (ROWTILES || PLANE) ? r / p.win_wv : 0;
        const int wcol = (ROWTILES || PLANE) ? r - wrow * p.win_wv : 0;
        uint32_t lt = 0;
        uint32_t echunk = 0;  // staged chunks so far (double-buffered staging alternates)
        int bias_n0 = -1;
        Ring ar;  // accumulator index and the parity of its current use
        for (int tile = t_first; tile < total_tiles;
             tile += t_step, ++lt, ar.next(FPAIR ? NACC / 2 : NACC)) {
            // folded window: warps 0-3 take the even tiles, 4-7 the odd ones (measured
            // on the 32-channel 3x3 layer at 150x150: 144 -> 124 us against both
            // groups converting half of every tile's channels); in units of two
            // tiles, warp group h takes half h of every unit
            if (FOLD && !FPAIR && (lt & 1u) != static_cast<uint32_t>(half)) continue;
            const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
            const uint32_t acc = FPAIR ? 2u * ar.stage + static_cast<uint32_t>(half) : ar.stage;
            // tcgen05.ld below is warp-collective: the whole warp proceeds or unwinds,
            // and with the TMA store all four warps do (they share named barriers).
            bool ready = __all_sync(0xffffffffu, wait_bar(&tfull[FPAIR ? ar.stage : acc], ar.phase,
                                                          wc, kRoleEpilogue));
            if (tma_store) {
                if (lane == 0) sVote[warp] = ready ? 1u : 0u;
                ptx::named_barrier_sync(1, kEpiN);
                ready = sVote[0] && sVote[1] && sVote[2] && sVote[3] &&
                        (!EPI8 || (sVote[4] && sVote[5] && sVote[6] && sVote[7]));
                ptx::named_barrier_sync(1, kEpiN);
            }
            if (!ready) break;
            ptx::tc_fence_after();
            if (FOLD) {
                // Lane quarter `quad` holds output row ho = 4*hb + quad of the tile:
                // accumulator row r is input column c0 + r, and its column block kw
                // (KW*C_out columns in all) is tap kw's share of the output pixel that
                // reads column c0 + r through tap kw.  The segment owns output pixels
                // k*G .. k*G + G - 1 of the row; lane l computes pixel wo = k*G + l as
                // the sum over the taps whose column wo - p + kw*d lies in the image
                // of block kw of row wo - p + kw*d - c0 (a shuffle; taps outside the
                // image are the zero padding and are left out).  The warp groups 0-3
                // and 4-7 take alternate tiles, each converting all C_out channels.
                uint32_t nhb, k, n, hb;
                p.fold_spr_div.divmod(static_cast<uint32_t>(u.m0), nhb, k);
                p.fold_hb_div.divmod(nhb, n, hb);
                const int ho = (FPAIR ? static_cast<int>(hb) * 2 + half : static_cast<int>(hb)) *
                                   kFoldRows + quad;
                const int wo = static_cast<int>(k) * p.fold_g + lane;
                const bool live = ho < p.fold_hout && lane < p.fold_g && wo < p.win_wout;
                const int c0 = min(max(static_cast<int>(k) * p.fold_g - p.win_pad, 0), p.x_W - 32);
                const int col0 = wo - p.win_pad;  // column of tap 0
                uint32_t taps = 0;                // taps whose column lies in the image
#pragma unroll
                for (int kw = 0; kw < FKW; ++kw) {
                    const int col = col0 + kw * p.win_d;
                    if (kw < p.win_kw && col >= 0 && col < p.x_W) taps |= 1u << kw;
                }
                // a segment that starts at k*G - p lies inside the row with every
                // tap of its pixels (warp-uniform)
                const bool interior = c0 == static_cast<int>(k) * p.fold_g - p.win_pad;
                const long long m =
                    (static_cast<long long>(n) * p.fold_hout + ho) * p.win_wout + wo;
                const int cw = p.C_out;
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * ACCW;
#pragma unroll 1
                for (int c16 = 0; c16 < cw; c16 += 16) {
                    const int co0 = c16;
                    uint32_t v[FKW][16];
#pragma unroll
                    for (int kw = 0; kw < FKW; ++kw)
                        if (kw < p.win_kw)
                            ptx::tmem_ld_32x32b_x16(tb + static_cast<uint32_t>(kw * p.C_out + co0),
                                                    v[kw]);
                    ptx::tmem_ld_wait();
                    if (c16 + 16 >= cw) release_acc(acc);
                    float o[16];
                    if (interior) {
                        // every tap of every pixel in the image, tap kw kw*d rows on
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __uint_as_float(v[0][i]);
#pragma unroll
                        for (int kw = 1; kw < FKW; ++kw)
                            if (kw < p.win_kw) {
                                const int sh = kw * p.win_d;
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    o[i] += __shfl_down_sync(0xffffffffu, __uint_as_float(v[kw][i]), sh);
                            }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = 0.f;
#pragma unroll
                        for (int kw = 0; kw < FKW; ++kw)
                            if (kw < p.win_kw) {
                                // source row, kept in the warp for taps that are left out
                                const int src = (col0 + kw * p.win_d - c0) & 31;
                                const bool use = (taps >> kw) & 1u;
#pragma unroll
                                for (int i = 0; i < 16; ++i) {
                                    const float t =
                                        __shfl_sync(0xffffffffu, __uint_as_float(v[kw][i]), src);
                                    o[i] += use ? t : 0.f;
                                }
                            }
                    }
                    if (!live) continue;
                    {
                        const float4* bs = reinterpret_cast<const float4*>(sBiasF + co0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 bq = bs[q];
                            o[4 * q] += bq.x;
                            o[4 * q + 1] += bq.y;
                            o[4 * q + 2] += bq.z;
                            o[4 * q + 3] += bq.w;
                        }
                    }
                    const long long at = m * p.C_out + co0;
                    if (p.y_f32) {
                        float4* out = reinterpret_cast<float4*>(static_cast<float*>(p.y) + at);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            out[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                    } else {
                        uint16_t* out = static_cast<uint16_t*>(p.y) + at;
                        uint32_t pk[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) pk[q] = pack_bf16x2(o[2 * q], o[2 * q + 1]);
                        if (p.y_al32) {
                            ptx::st_global_v8(out, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
                        } else {
                            reinterpret_cast<uint4*>(out)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            reinterpret_cast<uint4*>(out)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                }
                continue;
            }
            if (tma_store && u.n0 != bias_n0) {  // new column tile: stage its bias
                ptx::named_barrier_sync(1, kEpiN);
                for (int i = et; i < BN; i += kEpiN)
                    sBias[i] = (p.bias != nullptr && u.n0 + i < p.C_out)
                                   ? bf16_bits_to_float(p.bias[u.n0 + i])
                                   : 0.f;
                ptx::named_barrier_sync(1, kEpiN);
                bias_n0 = u.n0;
            }
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * ACCW;
            const int nsub = PLANE ? p.pl_u : 1;
            for (int sub = 0; sub < nsub; ++sub) {
                const bool last_sub = sub + 1 == nsub;
                int m = u.m0 + r;
                if (PLANE) {
                    // virtual row v of the stacked padded batch: image v / (H+2p), row v % (H+2p)
                    const int v = u.m0 + sub * p.win_rows + wrow;
                    uint32_t n, hv;
                    p.hp_div.divmod(static_cast<uint32_t>(v), n, hv);
                    const bool real = wrow < p.win_rows && wcol < p.win_wout &&
                                      static_cast<int>(hv) < p.pl_hout &&
                                      static_cast<int>(n) < p.pl_n;
                    m = real ? (static_cast<int>(n) * p.pl_hout + static_cast<int>(hv)) * p.win_wout +
                                   wcol
                             : p.M;
                } else if (ROWTILES) {
                    const int g = u.m0 + wrow;  // output row n*H_out + ho
                    const bool real = wrow < p.win_rows && wcol < p.win_wout && g < p.win_groups;
                    m = real ? g * p.win_wout + wcol : p.M;
                }
                const uint32_t taddr = tbase + static_cast<uint32_t>(sub * BN);
                const bool live = m < p.M;
                if (EPI8 && tma_store && epi_c32) {
                    // Narrow staging: 32-column chunks in a 128 x 64-byte tile, 64-byte
                    // swizzle (16-byte piece q of staged row s sits at q ^ ((s >> 1) & 3));
                    // warp w converts the 16-column half w / 4 of each chunk.
#pragma unroll 1
                    for (int ch = 0; ch < BN / 32; ++ch) {
                        uint32_t ra[16];
                        ptx::tmem_ld_32x32b_x16(taddr + ch * 32 + half * 16, ra);
                        ptx::tmem_ld_wait();
                        if (last_sub && ch + 1 == BN / 32) release_acc(acc);
                        uint8_t* sE = sEpi + ((p.epi_bufs == 2) ? (echunk & 1u) : 0u) * kEpiNarrowTileBytes;
                        ++echunk;
                        if (et == 0) {
                            if (p.epi_bufs == 2)
                                ptx::bulk_wait_read_1();
                            else
                                ptx::bulk_wait_read_all();
                        }
                        ptx::named_barrier_sync(1, kEpiN);
                        const float4* bs = reinterpret_cast<const float4*>(sBias + ch * 32);
                        const int srow = ROWTILES ? wrow * p.win_wout + wcol : r;
                        const bool keep = !ROWTILES || (wcol < p.win_wout && wrow < p.win_rows);
                        if (keep) {
#pragma unroll
                            for (int qq = 0; qq < 2; ++qq) {
                                const int q = 2 * half + qq;  // 16-byte piece of the row
                                const uint32_t* src = ra + 8 * qq;
                                const float4 b0 = bs[2 * q], b1 = bs[2 * q + 1];
                                uint4 v;
                                v.x = pack_bf16x2(__uint_as_float(src[0]) + b0.x,
                                                  __uint_as_float(src[1]) + b0.y);
                                v.y = pack_bf16x2(__uint_as_float(src[2]) + b0.z,
                                                  __uint_as_float(src[3]) + b0.w);
                                v.z = pack_bf16x2(__uint_as_float(src[4]) + b1.x,
                                                  __uint_as_float(src[5]) + b1.y);
                                v.w = pack_bf16x2(__uint_as_float(src[6]) + b1.z,
                                                  __uint_as_float(src[7]) + b1.w);
                                *reinterpret_cast<uint4*>(sE + srow * 64 +
                                                          ((q ^ ((srow >> 1) & 3)) << 4)) = v;
                            }
                        }
                        ptx::fence_proxy_async_smem();
                        ptx::named_barrier_sync(1, kEpiN);
                        if (et == 0) {
                            const int c0 = u.n0 + ch * 32;
                            if (ROWTILES) {
                                if (u.m0 < p.win_groups)
                                    ptx::tma_store_2d(&tmap_y, sE, c0, u.m0 * p.win_wout);
                            } else {
                                ptx::tma_store_2d(&tmap_y, sE, c0, u.m0);
                            }
                            ptx::bulk_commit_group();
                        }
                    }
                    continue;
                }
                if (tma_store) {
                    // A 64-column chunk goes from registers through the staging tile
                    // to y in four steps: acquire the staging tile (free once the
                    // store that last used it has read it: the previous chunk's, or
                    // with two tiles the one before), pack this thread's row (bias
                    // added, rounded to bf16: 16-byte pieces, 4 with eight warps and
                    // 8 with four; ra, and rb for the second 32 columns with four),
                    // write the pieces, and store the tile.  Row tiles keep only real
                    // output pixels, packed: the tile's output rows are consecutive
                    // rows of y, so one box stores the chunk.  Other tiles keep row r
                    // at r.
                    constexpr int kPieces = EPI8 ? 4 : 8;
                    const int srow = ROWTILES ? wrow * p.win_wout + wcol : r;
                    const bool keep = !ROWTILES || (wcol < p.win_wout && wrow < p.win_rows);
                    auto stage_acquire = [&]() -> uint8_t* {
                        uint8_t* sE = sEpi + ((p.epi_bufs == 2) ? (echunk & 1u) : 0u) * kEpiTileBytes;
                        ++echunk;
                        if (et == 0) {
                            if (p.epi_bufs == 2)
                                ptx::bulk_wait_read_1();
                            else
                                ptx::bulk_wait_read_all();
                        }
                        ptx::named_barrier_sync(1, kEpiN);
                        return sE;
                    };
                    auto pack = [&](int c64, const uint32_t* ra, const uint32_t* rb, uint4* v) {
                        const float4* bs = reinterpret_cast<const float4*>(sBias + c64 * 64);
#pragma unroll
                        for (int qq = 0; qq < kPieces; ++qq) {
                            const int q = (EPI8 ? 4 * half : 0) + qq;  // 16-byte piece of the row
                            const uint32_t* src = (EPI8 || qq < 4) ? ra + 8 * qq : rb + 8 * (qq - 4);
                            const float4 b0 = bs[2 * q], b1 = bs[2 * q + 1];
                            v[qq].x = pack_bf16x2(__uint_as_float(src[0]) + b0.x,
                                                  __uint_as_float(src[1]) + b0.y);
                            v[qq].y = pack_bf16x2(__uint_as_float(src[2]) + b0.z,
                                                  __uint_as_float(src[3]) + b0.w);
                            v[qq].z = pack_bf16x2(__uint_as_float(src[4]) + b1.x,
                                                  __uint_as_float(src[5]) + b1.y);
                            v[qq].w = pack_bf16x2(__uint_as_float(src[6]) + b1.z,
                                                  __uint_as_float(src[7]) + b1.w);
                        }
                    };
                    auto stage_write = [&](uint8_t* sE, const uint4* v) {
                        if (keep) {
#pragma unroll
                            for (int qq = 0; qq < kPieces; ++qq) {
                                const int q = (EPI8 ? 4 * half : 0) + qq;
                                *reinterpret_cast<uint4*>(sE + srow * 128 + ((q ^ (srow & 7)) << 4)) =
                                    v[qq];
                            }
                        }
                    };
                    auto stage_store = [&](uint8_t* sE, int c64) {
                        ptx::fence_proxy_async_smem();
                        ptx::named_barrier_sync(1, kEpiN);
                        if (et == 0) {
                            const int c0 = u.n0 + c64 * 64;
                            if (PLANE) {
                                // one box per real output row of this sub-tile
                                for (int jj = 0; jj < p.win_rows; ++jj) {
                                    uint32_t n, hv;
                                    p.hp_div.divmod(
                                        static_cast<uint32_t>(u.m0 + sub * p.win_rows + jj), n, hv);
                                    if (static_cast<int>(n) >= p.pl_n ||
                                        static_cast<int>(hv) >= p.pl_hout)
                                        continue;
                                    ptx::tma_store_2d(
                                        &tmap_y, sE + jj * p.win_wv * 128, c0,
                                        (static_cast<int>(n) * p.pl_hout + static_cast<int>(hv)) *
                                            p.win_wout);
                                }
                            } else if (ROWTILES) {
                                // win_rows*W_out rows from the tile's first output pixel;
                                // rows past the end of y are not written
                                if (u.m0 < p.win_groups)
                                    ptx::tma_store_2d(&tmap_y, sE, c0, u.m0 * p.win_wout);
                            } else {
                                ptx::tma_store_2d(&tmap_y, sE, c0, u.m0);
                            }
                            ptx::bulk_commit_group();
                        }
                    };
                    if (EPI8 && BN == 128) {
                        // Both chunks' TMEM loads at once: one load latency per tile,
                        // and the accumulator goes back to the MMA thread before the
                        // conversions start.  The second chunk is packed while the
                        // first chunk's store reads the staging tile (measured on the
                        // 64->128 3x3 layer at 56x56: 15.15 -> 14.60 us).
                        uint32_t r0[32], r1[32];
                        ptx::tmem_ld_32x32b_x32(taddr + half * 32, r0);
                        ptx::tmem_ld_32x32b_x32(taddr + 64 + half * 32, r1);
                        ptx::tmem_ld_wait();
                        if (last_sub) release_acc(acc);
                        {
                            uint4 v[kPieces];
                            uint8_t* sE = stage_acquire();
                            pack(0, r0, r0, v);
                            stage_write(sE, v);
                            stage_store(sE, 0);
                        }
                        uint4 v[kPieces];
                        pack(1, r1, r1, v);
                        uint8_t* sE = stage_acquire();
                        stage_write(sE, v);
                        stage_store(sE, 1);
                    } else {
#pragma unroll 1
                        for (int c64 = 0; c64 < BN / 64; ++c64) {
                            uint32_t ra[32], rb[32];
                            if (EPI8) {
                                ptx::tmem_ld_32x32b_x32(taddr + c64 * 64 + half * 32, ra);
                            } else {
                                ptx::tmem_ld_32x32b_x32(taddr + c64 * 64, ra);
                                ptx::tmem_ld_32x32b_x32(taddr + c64 * 64 + 32, rb);
                            }
                            ptx::tmem_ld_wait();
                            if (last_sub && c64 + 1 == BN / 64) release_acc(acc);
                            uint4 v[kPieces];
                            uint8_t* sE = stage_acquire();
                            pack(c64, ra, rb, v);
                            stage_write(sE, v);
                            stage_store(sE, c64);
                        }
                    }
                    continue;
                }
                // Direct stores: two 32-column chunks per TMEM round trip (one per
                // warp half with eight warps); the accumulator is handed back to
                // the MMA warp as soon as its last chunk is in registers.
                if (EPI8) {
                    bool released = false;
#pragma unroll 1
                    for (int ch = half; ch < BN / 32; ch += 2) {
                        uint32_t ra[32];
                        ptx::tmem_ld_32x32b_x32(taddr + ch * 32, ra);
                        ptx::tmem_ld_wait();
                        if (last_sub && ch + 2 >= BN / 32) {
                            release_acc(acc);
                            released = true;
                        }
                        const int co0 = u.n0 + ch * 32;
                        if (live && co0 < p.C_out) {
                            if (split_k || p.sk)
                                reduce_chunk(p, m, co0, ra);
                            else
                                store_chunk(p, m, co0, ra);
                        }
                    }
                    if (last_sub && !released) release_acc(acc);
                } else {
#pragma unroll 1
                    for (int ch = 0; ch < BN / 32; ch += 2) {
                        uint32_t ra[32], rb[32];
                        ptx::tmem_ld_32x32b_x32(taddr + ch * 32, ra);
                        if (ch + 1 < BN / 32) ptx::tmem_ld_32x32b_x32(taddr + (ch + 1) * 32, rb);
                        ptx::tmem_ld_wait();
                        if (last_sub && ch + 2 >= BN / 32) release_acc(acc);
                        const int co0 = u.n0 + ch * 32;
                        if (live && co0 < p.C_out) {
                            if (split_k || p.sk)
                                reduce_chunk(p, m, co0, ra);
                            else
                                store_chunk(p, m, co0, ra);
                        }
                        if (live && ch + 1 < BN / 32 && co0 + 32 < p.C_out) {
                            if (split_k || p.sk)
                                reduce_chunk(p, m, co0 + 32, rb);
                            else
                                store_chunk(p, m, co0 + 32, rb);
                        }
                    }
                }
            }
            if (et == 0) *sTilesDone = lt + 1;
        }
        // Every TMA store has finished before the CTA exits.
        if (tma_store && et == 0) ptx::bulk_wait_all();
    } else if (warp < kEpiWarps + kGatherWarps) {
        // ------------------------------------------------------------ A gather
        if (PLANE && warp == kEpiWarps) {
            // Plane mode: one lane stages, per (tile, channel block cc), the
            // pl_srows padded input rows the tile's taps read: virtual row v0 + j
            // is row (v0 + j) % (H+2p) - p of image (v0 + j) / (H+2p), one box of
            // win_wv pixels x 64 channels starting at column -p.  TMA zero-fills
            // the padding rows and columns; rows past the last image are skipped
            // (they feed only discarded accumulator rows).
            if (lane == 0) {
                const uint32_t row_bytes = static_cast<uint32_t>(p.win_wv) * 128u;
                Ring ring;
                uint32_t issued = 0;
                bool ok = true;
                for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                    const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                    for (int kb = u.kb0; kb < u.kb1; ++kb, ++issued, ring.next(S)) {
                        if (!wait_bar(&empty[ring.stage], ring.phase ^ 1u, wc, kRoleGather)) {
                            ok = false;
                            break;
                        }
                        uint32_t nrows = 0;
                        for (int j = 0; j < p.pl_srows; ++j)
                            nrows += static_cast<int>(
                                         p.hp_div.div(static_cast<uint32_t>(u.m0 + j))) < p.pl_n
                                         ? 1u
                                         : 0u;
                        ptx::mbar_arrive_expect_tx(&full_a[ring.stage], nrows * row_bytes);
                        uint8_t* stage_a = sA + ring.stage * AST;
                        for (int j = 0; j < p.pl_srows; ++j) {
                            uint32_t n, hp;
                            p.hp_div.divmod(static_cast<uint32_t>(u.m0 + j), n, hp);
                            if (static_cast<int>(n) >= p.pl_n) continue;
                            ptx::tma_load_4d(stage_a + j * row_bytes, &tmap_a, &full_a[ring.stage],
                                             kb * BK, -p.win_pad,
                                             static_cast<int>(hp) - p.win_pad, static_cast<int>(n));
                        }
                    }
                }
                // Wait (bounded) for the last loads so none lands after the CTA exits.
                const uint32_t first = issued > S ? issued - S : 0;
                for (uint32_t i = first; i < issued; ++i)
                    drain_wait(&full_a[i % S], (i / S) & 1u, 1000000000ull);
            }
        } else if (PLANE && warp == kEpiWarps + 1) {
            // Pulls the input rows of the CTA's next tiles into L2 with plain
            // prefetches, at most three tiles ahead of the epilogue (advisory
            // pacing: a bounded spin, then prefetch anyway).
            const long long row_elems = static_cast<long long>(p.x_W) * p.C_in;
            const int lines = static_cast<int>((row_elems * 2 + 127) / 128);
            volatile uint32_t* aborted = abort_flag;
            uint32_t lt = 0;
            for (int tile = t_first; tile < total_tiles; tile += t_step, ++lt) {
                // (backs off between polls so the spin takes no issue slots from the
                // epilogue warp on the same scheduler)
                for (uint32_t spin = 0; spin < (1u << 16) && lt > *sTilesDone + 3u && !*aborted;
                     ++spin)
                    __nanosleep(256);
                if (*aborted) break;
                const Unit v = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                if (v.n0 != 0 || v.kb0 != 0) continue;  // one prefetch per row block
                for (int j = 0; j < p.pl_srows; ++j) {
                    uint32_t n, hp;
                    p.hp_div.divmod(static_cast<uint32_t>(v.m0 + j), n, hp);
                    const int h = static_cast<int>(hp) - p.win_pad;
                    if (static_cast<int>(n) >= p.pl_n || h < 0 || h >= p.x_H) continue;
                    const uint8_t* row = reinterpret_cast<const uint8_t*>(
                        p.x + (static_cast<long long>(n) * p.x_H + h) * row_elems);
                    for (int l = lane; l < lines; l += 32) ptx::prefetch_l2_line(row + l * 128);
                }
            }
        } else if (TMAGATHER) {
            // TMA gather4 through the indirection buffer.  The four gather warps
            // take turns: warp gw fills the stages whose sequence number is gw
            // mod 4, so each has four stage-times to look its rows up.  Lane l
            // owns rows 4l..4l+3 of the 128-row tile: it turns each row's
            // (pixel, tap) entry into a row index of x viewed as [N*H*W][C_in]
            // and issues one gather4 of those four 128-byte rows.  On a pair both
            // CTAs' gathers complete on CTA 0's barrier, which CTA 0 arms for both
            // (rows past M gather zeros, so both always deliver a full tile).
            const int gw = warp - kEpiWarps;
            uint32_t it = 0;
            Ring ring;
            bool ok = true;
            for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                int ib4[4];  // first indirection entry of the row's pixel, or -1
                int nb4[4];  // first row of the pixel's image
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int m = u.m0 + 4 * lane + q;
                    ib4[q] = -1;
                    nb4[q] = 0;
                    if (m < p.M) {
                        uint32_t n, pix;
                        p.hwo_div.divmod(static_cast<uint32_t>(m), n, pix);
                        ib4[q] = static_cast<int>(pix) * p.taps;
                        nb4[q] = static_cast<int>(n) * p.img_rows;
                    }
                }
                for (int kb = u.kb0; kb < u.kb1; ++kb, ++it, ring.next(S)) {
                    if (it % kGatherWarps != static_cast<uint32_t>(gw)) continue;
                    uint32_t tap, c0;
                    p.cin_div.divmod(static_cast<uint32_t>(kb * BK), tap, c0);
                    int row[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int off = ib4[q] >= 0 ? __ldg(p.ibuf + ib4[q] + tap) : -1;
                        row[q] = off >= 0 ? nb4[q] + static_cast<int>(
                                                         p.cin_div.div(static_cast<uint32_t>(off)))
                                          : p.oob_row;
                    }
                    const bool ready =
                        wait_bar(&empty[ring.stage], ring.phase ^ 1u, wc, kRoleGather);
                    if (!__all_sync(0xffffffffu, ready)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0 && rank == 0)
                        ptx::mbar_arrive_expect_tx(&full_a[ring.stage],
                                                   kABytes * (PAIR ? 2u : 1u));
                    __syncwarp();
                    if (PAIR)
                        ptx::tma_gather4_pair(sA + ring.stage * AST + lane * 4 * 128, &tmap_a,
                                              ptx::mapa(ptx::smem_addr(&full_a[ring.stage]), 0u),
                                              static_cast<int>(c0), row[0], row[1], row[2],
                                              row[3]);
                    else
                        ptx::tma_gather4(sA + ring.stage * AST + lane * 4 * 128, &tmap_a,
                                         &full_a[ring.stage], static_cast<int>(c0), row[0],
                                         row[1], row[2], row[3]);
                }
            }
            // Wait (bounded) for this warp's last gathers so none lands after exit
            // (a pair's complete on CTA 0's barriers, for both CTAs).
            if (lane == 0 && rank == 0) {
                const uint32_t first = it > S ? it - S : 0;
                for (uint32_t i = first; i < it; ++i)
                    if (i % kGatherWarps == static_cast<uint32_t>(gw))
                        drain_wait(&full_a[i % S], (i / S) & 1u, 1000000000ull);
            }
        } else if (STEMWIN) {
            // Thread t builds stage row t = (tile row j, r) of every group of the
            // tile; rows past the tile's segments keep stale values, which only
            // discarded accumulator rows read.  Nothing is built before the
            // weights are packed: their raw copy sits in the A stages until then.
            const int t = threadIdx.x - kEpiThreads;  // 0..127
            const int j = t / p.win_wv, r = t - j * p.win_wv;
            const int rbe = p.nw_rb / 2;
            const int col_e = (p.nw_a0 - p.nw_p * p.nw_cin * 2) / 2 + p.nw_s * r * p.nw_cin;
            Ring ring;
            uint32_t slot = 0, slot_phase = 0;
            bool ok = wait_bar(wpack, 0u, wc, kRoleGather);
            for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                const int rows = min(p.win_rows, p.win_groups - u.m0);
                const bool live = j < rows;
                uint32_t hvalid = 0u;
                if (live) {
                    uint32_t nn, hh;
                    p.ho_div.divmod(static_cast<uint32_t>(u.m0 + j), nn, hh);
                    const int h0 = static_cast<int>(hh) * p.nw_s - p.nw_p;
                    for (int kh = 0; kh < p.nw_KH; ++kh)
                        if (h0 + kh >= 0 && h0 + kh < p.nw_H) hvalid |= 1u << kh;
                }
                if (!wait_bar(&stg_full[slot], slot_phase, wc, kRoleGather)) {
                    ok = false;
                    break;
                }
                const uint16_t* rows_j = reinterpret_cast<const uint16_t*>(sStg + slot * p.nw_slot_bytes) +
                                         j * p.nw_KH * rbe;
                for (int kb = u.kb0; kb < u.kb1; ++kb, ring.next(S)) {
                    if (!wait_bar(&empty[ring.stage], ring.phase ^ 1u, wc, kRoleGather)) {
                        ok = false;
                        break;
                    }
                    if (live)
                        stemwin_row<3, SW_S>(sA + ring.stage * AST, t, rows_j, rbe, col_e,
                                             kb * p.sw_khg, p.nw_KH, hvalid);
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&full_a[ring.stage]);
                }
                ptx::mbar_arrive(&stg_empty[slot]);
                if (++slot == NS) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
            }
        } else if (NARROWWIN) {
            // Thread t builds A row t: output pixel (tile row j, column wo).  K is
            // (kh, kw*C_in + c) with each kh slice padded to nw_kwcp, so the slice
            // of kh is nw_kwc consecutive elements of the staged input row
            // ho*s - p + kh, starting at pixel wo*s - p.
            const int t = threadIdx.x - kEpiThreads;  // 0..127
            const int j = t / p.win_wv, wo = t - j * p.win_wv;
            const int px_off = wo * p.nw_s * p.nw_cin;  // element offset of the window in its row
            const int lead = p.nw_a0 / 2 - p.nw_p * p.nw_cin;  // element of pixel -p in a row
            Ring ring;
            uint32_t slot = 0, slot_phase = 0;
            bool ok = true;
            for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                const int rows = min(p.win_rows, p.win_groups - u.m0);
                const bool row_live = j < rows;
                int ho = 0;
                if (row_live) {
                    uint32_t nn, hh;
                    p.ho_div.divmod(static_cast<uint32_t>(u.m0 + j), nn, hh);
                    ho = static_cast<int>(hh);
                }
                if (!wait_bar(&stg_full[slot], slot_phase, wc, kRoleGather)) {
                    ok = false;
                    break;
                }
                const uint16_t* stg = reinterpret_cast<const uint16_t*>(sStg + slot * p.nw_slot_bytes);
                int kh = (u.kb0 * BK) / p.nw_kwcp;   // slice of the first chunk
                int o = u.kb0 * BK - kh * p.nw_kwcp;  // offset of the chunk in its slice
                for (int kb = u.kb0; kb < u.kb1; ++kb, ring.next(S)) {
                    if (!wait_bar(&empty[ring.stage], ring.phase ^ 1u, wc, kRoleGather)) {
                        ok = false;
                        break;
                    }
                    uint8_t* stage_a = sA + ring.stage * AST;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t w4[4] = {0u, 0u, 0u, 0u};
                        const int h = ho * p.nw_s - p.nw_p + kh;
                        if (row_live && kh < p.nw_KH && h >= 0 && h < p.nw_H) {
                            const int e = (j * p.nw_KH + kh) * (p.nw_rb / 2) + lead + px_off + o;
                            const uint32_t* wp = reinterpret_cast<const uint32_t*>(stg) + (e >> 1);
                            uint32_t v[5];
#pragma unroll
                            for (int q = 0; q < 5; ++q) v[q] = wp[q];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                w4[q] = (e & 1) ? __funnelshift_r(v[q], v[q + 1], 16) : v[q];
                            // elements past the slice's KW*C_in belong to the next pixels
                            const int valid = p.nw_kwc - o;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                if (2 * q >= valid) w4[q] = 0u;
                                else if (2 * q + 1 >= valid) w4[q] &= 0xFFFFu;
                            }
                        }
                        const int cr = c ^ (t & 7);
                        *reinterpret_cast<uint4*>(stage_a + t * 128 + cr * 16) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        o += 8;
                        if (o >= p.nw_kwcp) {
                            o -= p.nw_kwcp;
                            ++kh;
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&full_a[ring.stage]);
                }
                ptx::mbar_arrive(&stg_empty[slot]);
                if (++slot == NS) {
                    slot = 0;
                    slot_phase ^= 1u;
                }
            }
        } else if (GATHER) {
            // Thread gt owns 16-byte chunk c (8 consecutive K columns) of rows
            // rg, rg+16, ..., rg+112 of every A tile: 8 threads cover one 128-byte row.
            const int gt = threadIdx.x - kEpiThreads;  // 0..127
            const int c = gt & 7;
            const int rg = gt >> 3;
            Ring ring;
            bool ok = true;
            for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                int ib[kRowsPerGatherThread];        // pixel's first ibuf entry, or -1
                long long xb[kRowsPerGatherThread];  // image base (elements)
#pragma unroll
                for (int j = 0; j < kRowsPerGatherThread; ++j) {
                    const int m = u.m0 + rg + 16 * j;
                    ib[j] = -1;
                    xb[j] = 0;
                    if (m < p.M) {
                        uint32_t n, pix;
                        p.hwo_div.divmod(static_cast<uint32_t>(m), n, pix);
                        ib[j] = static_cast<int>(pix) * p.taps;
                        xb[j] = static_cast<long long>(n) * p.img_elems;
                    }
                }
                // Indirection entries of K block `kb` for this thread's rows
                // (16-byte gather), fetched one block ahead of their use.
                int off[kRowsPerGatherThread], nxt[kRowsPerGatherThread];
                uint32_t nxt_ci = 0;
                auto load_offsets = [&](int kb_next) {
                    const int kn = kb_next * BK + c * 8;
                    const bool kval = kb_next < u.kb1 && kn < p.K;
                    uint32_t tap = 0;
                    nxt_ci = 0;
                    if (kval) p.cin_div.divmod(static_cast<uint32_t>(kn), tap, nxt_ci);
#pragma unroll
                    for (int j = 0; j < kRowsPerGatherThread; ++j)
                        nxt[j] = (kval && ib[j] >= 0) ? __ldg(p.ibuf + ib[j] + tap) : -1;
                };
                if (AMODE == kAGather) load_offsets(u.kb0);
                for (int kb = u.kb0; kb < u.kb1; ++kb, ring.next(S)) {
                    if (!wait_bar(&empty[ring.stage], ring.phase ^ 1u, wc, kRoleGather)) {
                        ok = false;
                        break;
                    }
                    const int k = kb * BK + c * 8;
                    uint8_t* stage_a = sA + ring.stage * AST;
                    if (AMODE == kAGather) {
                        // C_in % 8 == 0: the chunk is 8 channels of one tap's pixel.
                        // The indirection entries of this K block were loaded one
                        // block ahead; fetch the next block's now, then copy.  The
                        // thread's arrival on full_a fires when its copies land, so
                        // the thread never waits for them.
                        const uint32_t ci = nxt_ci;
#pragma unroll
                        for (int j = 0; j < kRowsPerGatherThread; ++j) off[j] = nxt[j];
                        load_offsets(kb + 1);
                        const uint32_t dst0 = ptx::smem_addr(stage_a);
#pragma unroll
                        for (int j = 0; j < kRowsPerGatherThread; ++j) {
                            const int r = rg + 16 * j;
                            const uint32_t dst = dst0 + r * 128 + ((c ^ (r & 7)) << 4);
                            const bool live = off[j] >= 0;
                            const uint16_t* src = live ? p.x + xb[j] + off[j] + ci : p.x;
                            ptx::cp_async_16(dst, src, live ? 16u : 0u);
                        }
                        ptx::cp_async_arrive_noinc(&full_a[ring.stage]);
                    } else {
                        // Narrow C_in: K columns are (tap, channel) with channels padded
                        // to cp (4, or a multiple of 8).  cp == 4: the chunk spans taps
                        // t0 and t0+1; otherwise channels [c0, c0+8) of tap t0.
                        const bool two = p.cp == 4;
                        uint32_t t0 = 0, c0 = 0;
                        if (k < p.k_valid) p.cin_div.divmod(static_cast<uint32_t>(k), t0, c0);
                        const bool v0 = k < p.k_valid;
                        const bool v1 = two && (k + 4) < p.k_valid;
#pragma unroll
                        for (int j = 0; j < kRowsPerGatherThread; ++j) {
                            const int o0 = (v0 && ib[j] >= 0) ? __ldg(p.ibuf + ib[j] + t0) : -1;
                            const int o1 =
                                (v1 && ib[j] >= 0) ? __ldg(p.ibuf + ib[j] + t0 + 1) : -1;
                            uint16_t e[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const int o = (two && q >= 4) ? o1 : o0;
                                const int ch = two ? (q & 3) : static_cast<int>(c0) + q;
                                e[q] = (o >= 0 && ch < p.C_in) ? p.x[xb[j] + o + ch] : (uint16_t)0;
                            }
                            const int r = rg + 16 * j;
                            uint4 v;
                            v.x = (uint32_t)e[0] | ((uint32_t)e[1] << 16);
                            v.y = (uint32_t)e[2] | ((uint32_t)e[3] << 16);
                            v.z = (uint32_t)e[4] | ((uint32_t)e[5] << 16);
                            v.w = (uint32_t)e[6] | ((uint32_t)e[7] << 16);
                            *reinterpret_cast<uint4*>(stage_a + r * 128 + ((c ^ (r & 7)) << 4)) = v;
                        }
                        ptx::fence_proxy_async_smem();
                        ptx::mbar_arrive(&full_a[ring.stage]);
                    }
                }
            }
            // No copy may still be landing when the CTA exits.
            if (AMODE == kAGather) ptx::cp_async_wait_all();
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (PLANE && lane == 0) {
            // Per tile and channel block cc: one staged A slot feeds every tap
            // (kh, kw) of every sub-tile; tap (kh, kw) of sub-tile u starts
            // u*win_rows*win_wv + kh*d*win_wv + kw*d rows into the slot.  Streamed
            // weights arrive one (tap, cc) block per B slot.  Descriptors are
            // formed by adding 16-byte-unit offsets to the slot bases (the start
            // address field is the low 14 bits), and nothing on the issue path
            // waits for arithmetic: with N = 128 an MMA lasts 64 cycles and a
            // per-tap index computation between MMA groups would idle the tensor
            // core.  3x3 kernels issue from a compile-time unrolled sequence; other
            // kernels walk the taps with the next tap's offsets formed before the
            // current tap's MMAs are issued.
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
            constexpr int CT = AMODE == kAPlane ? 0 : 9;  // compile-time taps (0: runtime)
            constexpr int CU = AMODE == kAPlane3U2 ? 2 : 1;
            const uint64_t a_desc0 = ptx::sdesc_k_major_sw128(ptx::smem_addr(sA));
            const uint64_t b_desc0 = ptx::sdesc_k_major_sw128(ptx::smem_addr(sB));
            const uint32_t a_slot_step = AST >> 4;
            constexpr uint32_t b_blk_step = BB >> 4;
            const uint32_t sub_step = static_cast<uint32_t>(p.win_rows * p.win_wv * 8);
            const uint32_t row_step = static_cast<uint32_t>(p.win_wv * p.win_d * 8);  // kh + 1
            const uint32_t col_step = static_cast<uint32_t>(p.win_d * 8);             // kw + 1
            uint32_t aoff[CT > 0 ? CT : 1], boff[CT > 0 ? CT : 1];
#pragma unroll
            for (int t = 0; t < CT; ++t) {
                aoff[t] = static_cast<uint32_t>(t / 3) * row_step + static_cast<uint32_t>(t % 3) * col_step;
                boff[t] = static_cast<uint32_t>(t * p.win_cc) * b_blk_step;
            }
            Ring ra, rb;
            uint32_t lt = 0;
            bool ok = !bres || wait_bar(bres_full, 0u, wc, kRoleMma);
            const int taps = p.x_KH * p.win_kw;
            Ring ar;
            for (int tile = t_first; ok && tile < total_tiles;
                 tile += t_step, ++lt, ar.next(NACC)) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                const uint32_t acc = ar.stage;
                if (!wait_bar(&tempty[acc], ar.phase ^ 1u, wc, kRoleMma)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACCW;
                for (int kb = u.kb0; ok && kb < u.kb1; ++kb, ra.next(S)) {
                    const uint64_t ad = a_desc0 + ra.stage * a_slot_step;
                    const uint64_t bres_d = b_desc0 + static_cast<uint32_t>(kb) * b_blk_step;
                    const uint32_t first = kb == u.kb0 ? 0u : 1u;  // accumulate flag of tap 0
                    if (!wait_bar(&full_a[ra.stage], ra.phase, wc, kRoleMma)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (CT > 0) {
#pragma unroll
                        for (int t = 0; t < CT; ++t) {
                            uint64_t bd = bres_d + boff[t];
                            if (!bres) {
                                if (!wait_bar(&full_b[rb.stage], rb.phase, wc, kRoleMma)) {
                                    ok = false;
                                    break;
                                }
                                ptx::tc_fence_after();
                                bd = b_desc0 + rb.stage * b_blk_step;
                            }
#pragma unroll
                            for (int sub = 0; sub < CU; ++sub)
#pragma unroll
                                for (int kk = 0; kk < BK / 16; ++kk)
                                    ptx::mma_bf16(d_tmem + static_cast<uint32_t>(sub * BN),
                                                  ad + aoff[t] + sub * sub_step + 2 * kk,
                                                  bd + 2 * kk, idesc,
                                                  (t != 0 || kk != 0) ? 1u : first);
                            if (!bres) {
                                ptx::mma_commit(&empty_b[rb.stage]);
                                rb.next(SB);
                            }
                        }
                    } else {
                        int kh = 0, kw = 0;
                        uint32_t a_next = 0;
                        uint64_t b_next = bres_d;
                        for (int t = 0; t < taps; ++t) {
                            const uint32_t a_cur = a_next;
                            uint64_t bd = b_next;
                            if (++kw == p.win_kw) {
                                kw = 0;
                                ++kh;
                            }
                            a_next = static_cast<uint32_t>(kh) * row_step +
                                     static_cast<uint32_t>(kw) * col_step;
                            b_next += static_cast<uint64_t>(static_cast<uint32_t>(p.win_cc) *
                                                            b_blk_step);
                            if (!bres) {
                                if (!wait_bar(&full_b[rb.stage], rb.phase, wc, kRoleMma)) {
                                    ok = false;
                                    break;
                                }
                                ptx::tc_fence_after();
                                bd = b_desc0 + rb.stage * b_blk_step;
                            }
                            for (int sub = 0; sub < p.pl_u; ++sub)
#pragma unroll
                                for (int kk = 0; kk < BK / 16; ++kk)
                                    ptx::mma_bf16(d_tmem + static_cast<uint32_t>(sub * BN),
                                                  ad + a_cur + sub * sub_step + 2 * kk,
                                                  bd + 2 * kk, idesc,
                                                  (t != 0 || kk != 0) ? 1u : first);
                            if (!bres) {
                                ptx::mma_commit(&empty_b[rb.stage]);
                                rb.next(SB);
                            }
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(&empty[ra.stage]);
                }
                if (ok) ptx::mma_commit(&tfull[acc]);
            }
            // Make sure no MMA is still reading shared memory or writing TMEM.
            ptx::mma_commit(drain);
            drain_wait(drain, 0, 1000000000ull);
        } else if (!PLANE && rank == 0) {
            // The whole warp walks the units; lane 0 issues.  Every barrier wait
            // is done by the wait warp, which hands each one over at kHandBar
            // with its outcome (the same sequence: weights, then per tile the
            // accumulator and each K block).
            // (in a pair only CTA 0 issues: each MMA covers both CTAs' 128 rows)
            // (the folded window: MMA width KW*C_out, 64-byte rows of 32 channels)
            const uint32_t idesc = FOLD ? ptx::idesc_bf16_f32(BM, p.fold_n)
                                        : ptx::idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
            const uint64_t a_desc0 = FOLD ? ptx::sdesc_k_major_sw64(ptx::smem_addr(sA))
                                          : ptx::sdesc_k_major_sw128(ptx::smem_addr(sA));
            const uint64_t b_desc0 = FOLD ? ptx::sdesc_k_major_sw64(ptx::smem_addr(sB))
                                          : ptx::sdesc_k_major_sw128(ptx::smem_addr(sB));
            const uint32_t a_slot_step = AST >> 4;
            constexpr uint32_t b_blk_step = BB >> 4;
            const uint32_t col_step = static_cast<uint32_t>(p.win_d * 8);  // window: kw + 1
            uint32_t hand = 0;
            auto receive = [&]() -> bool {
                ptx::named_barrier_sync(kHandBar, kHandThreads);
                const bool good = sHand[hand & 1u] != 0u;
                ++hand;
                return good;
            };
            Ring ring;
            bool ok = receive();  // resident weights (or nothing to wait for)
            Ring ar;
            for (int tile = t_first; ok && tile < total_tiles;
                 tile += t_step, ar.next(FPAIR ? C::kAcc / 2 : C::kAcc)) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                const uint32_t acc = ar.stage;
                // accumulator drained by the epilogue (the folded window and the
                // fixed-plan window kernel: handed over with the first stage below)
                if (!FOLD && !WT && !receive()) break;
                ptx::tc_fence_after();
                // (units of two tiles: accumulators 2*acc and 2*acc + 1)
                const uint32_t d_tmem = tmem_base + (FPAIR ? 2u * acc : acc) * BN;
                // window mode: (kh, cc) of the K block, walked instead of divided
                int win_kh = 0, win_cc = 0;
                if (WINDOW && u.kb0 != 0) {  // split K only
                    win_kh = u.kb0 / p.win_cc;
                    win_cc = u.kb0 - win_kh * p.win_cc;
                }
                for (int kb = u.kb0; kb < u.kb1; ++kb, ring.next(S)) {
                    if (!receive()) {  // the stage's A and B have landed
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        // Thread-written A stages (cp.async, st.shared) are read by the
                        // tensor core through the async proxy.
                        if (AMODE == kAGather || AMODE == kANarrow || NARROWWIN || STEMWIN)
                            ptx::fence_proxy_async_smem();
                        ptx::tc_fence_after();
                        // Descriptors as slot bases plus 16-byte-unit offsets: no
                        // division or address arithmetic between MMA groups.
                        const uint64_t ad = a_desc0 + ring.stage * a_slot_step;
                        if (WINDOW) {
                            // One staged (kh, cc) block feeds every kw tap: tap kw reads
                            // the staging rows shifted down by kw*d.
                            const uint64_t bd0 =
                                bres ? b_desc0 + static_cast<uint32_t>(win_kh * p.win_kw * p.win_cc +
                                                                         win_cc) *
                                                       b_blk_step
                                       : b_desc0 + ring.stage * p.b_per_stage * b_blk_step;
                            const uint32_t bstep = bres ? p.win_cc * b_blk_step : b_blk_step;
                            const uint32_t first = kb != u.kb0 ? 1u : 0u;
                            if (kw3) {
#pragma unroll
                                for (int kw = 0; kw < 3; ++kw)
#pragma unroll
                                    for (int kk = 0; kk < BK / 16; ++kk)
                                        mma_issue<PAIR>(d_tmem, ad + kw * col_step + 2 * kk,
                                                      bd0 + kw * bstep + 2 * kk, idesc,
                                                      (kw != 0 || kk != 0) ? 1u : first);
                            } else {
                                for (int kw = 0; kw < p.win_kw; ++kw)
#pragma unroll
                                    for (int kk = 0; kk < BK / 16; ++kk)
                                        mma_issue<PAIR>(d_tmem, ad + kw * col_step + 2 * kk,
                                                      bd0 + kw * bstep + 2 * kk, idesc,
                                                      (kw != 0 || kk != 0) ? 1u : first);
                            }
                        } else if (STEMWIN) {
                            // One stage (kernel-row group kb) feeds its nkb K blocks: K
                            // block j of output pixel (row) i is stage row i + j.  The
                            // sequence is unrolled with compile-time descriptor offsets
                            // (step q: K block q / 4, 16-column step q % 4) so that no
                            // arithmetic sits between the MMAs (an N=64 MMA lasts ~48
                            // cycles, less than a run-time loop's descriptor updates).
                            const uint64_t bd0 =
                                b_desc0 + static_cast<uint32_t>(kb * p.sw_nkb) * b_blk_step;
                            const int nsteps = p.sw_steps;
                            const uint32_t acc0 = kb != u.kb0 ? 1u : 0u;
#pragma unroll
                            for (int q = 0; q < kStemWinMaxSteps; ++q)
                                if (q < nsteps)
                                    mma_issue<PAIR>(d_tmem, ad + 8 * (q >> 2) + 2 * (q & 3),
                                                    bd0 + (q >> 2) * b_blk_step + 2 * (q & 3), idesc,
                                                    q != 0 ? 1u : acc0);
                        } else if (FOLD) {
                            // Tap row kh: the 128 rows from staged row kh*d on (lane
                            // quarter q reads input row 4*hb - p + q + kh*d); weight
                            // block kh is KW*C_out rows (kw, co).  Two 16-channel steps
                            // per kh.
                            const uint32_t a_kh_step =
                                static_cast<uint32_t>(p.win_d * kFoldRowBytes) >> 4;
                            const uint32_t b_kh_step = static_cast<uint32_t>(p.fold_n * 64) >> 4;
#pragma unroll
                            for (int h = 0; h < (FPAIR ? 2 : 1); ++h)
#pragma unroll
                                for (int kh = 0; kh < FKH; ++kh)
                                    if (kh < p.x_KH) {
#pragma unroll
                                        for (int kk = 0; kk < 2; ++kk)
                                            mma_issue<PAIR>(
                                                d_tmem + static_cast<uint32_t>(h * BN),
                                                ad + static_cast<uint32_t>(h * kFoldRows * kFoldRowBytes >> 4) +
                                                    static_cast<uint32_t>(kh) * a_kh_step + 2 * kk,
                                                b_desc0 + static_cast<uint32_t>(kh) * b_kh_step + 2 * kk,
                                                idesc, (kh != 0 || kk != 0) ? 1u : 0u);
                                    }
                        } else {
                            const uint64_t bd =
                                b_desc0 + (bres ? static_cast<uint32_t>(kb) : ring.stage) * b_blk_step;
                            // The last K block may hold fewer than 64 columns: skip the
                            // all-zero 16-column steps.
                            const int ksteps = min(BK / 16, (p.K - kb * BK + 15) / 16);
#pragma unroll
                            for (int kk = 0; kk < BK / 16; ++kk)
                                if (kk < ksteps)
                                    mma_issue<PAIR>(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc,
                                                  (kb != u.kb0 || kk != 0) ? 1u : 0u);
                        }
                        // (the folded window's stages are its accumulators' slots: the
                        // commit to tfull below frees the stage as well)
                        if (!FOLD) mma_commit_to<PAIR>(&empty[ring.stage]);
                    }
                    __syncwarp();
                    if (WINDOW && ++win_cc == p.win_cc) {
                        win_cc = 0;
                        ++win_kh;
                    }
                }
                if (ok && lane == 0) mma_commit_to<PAIR>(&tfull[acc]);
                __syncwarp();
            }
            // Make sure no MMA is still reading shared memory or writing TMEM.
            if (lane == 0) {
                mma_commit_to<PAIR>(drain, false);
                drain_wait(drain, 0, 1000000000ull);
            }
            __syncwarp();
        }
    } else if (warp == kWaitWarp) {
        // ------------------------------------------------------------ barrier waits
        // Mirrors the MMA warp's walk (non-plane modes): lane 0 waits, the warp
        // hands the outcome over; a failed wait is handed over too, and both
        // warps leave their loops at that same hand-off.
        if (!PLANE && rank == 0) {
            uint32_t hand = 0;
            auto waited = [&](uint64_t* bar, uint32_t parity, bool cluster) -> bool {
                uint32_t good = 0u;
                if (lane == 0) good = wait_bar(bar, parity, wc, kRoleMma, cluster) ? 1u : 0u;
                return __shfl_sync(0xffffffffu, good, 0) != 0u;
            };
            auto send = [&](bool good) -> bool {
                if (lane == 0) sHand[hand & 1u] = good ? 1u : 0u;
                ++hand;
                ptx::named_barrier_sync(kHandBar, kHandThreads);
                return good;
            };
            Ring ring;
            // (the staged-window stem's weights are ready once packed: wpack)
            bool ok = send(!bres || waited(STEMWIN ? wpack : bres_full, 0u, false));
            Ring ar;
            for (int tile = t_first; ok && tile < total_tiles;
                 tile += t_step, ar.next(FPAIR ? C::kAcc / 2 : C::kAcc)) {
                const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                // (the folded window: one hand-off per tile, the accumulator and the
                // stage together; in units of two tiles both accumulators.  The
                // fixed-plan window kernel hands the accumulator over with the
                // tile's first K block: each hand-off leaves the MMA thread idle
                // for ~200 cycles, which the tensor core does not hide)
                bool acc_ok = true;
                if (WT)
                    acc_ok = waited(&tempty[ar.stage], ar.phase ^ 1u, PAIR);
                else if (!FOLD && !send(waited(&tempty[ar.stage], ar.phase ^ 1u, PAIR)))
                    break;
                for (int kb = u.kb0; kb < u.kb1; ++kb, ring.next(S)) {
                    bool good = (!WT || kb != u.kb0 || acc_ok) &&
                                (!GATHER || waited(&full_a[ring.stage], ring.phase, false));
                    if (FOLD)
                        good = FPAIR ? waited(&tempty[2 * ar.stage], ar.phase ^ 1u, false) &&
                                           waited(&tempty[2 * ar.stage + 1], ar.phase ^ 1u, false)
                                     : waited(&tempty[ar.stage], ar.phase ^ 1u, false);
                    if (good && (!GATHER || !bres))
                        good = waited(&full_b[ring.stage], ring.phase, false);
                    if (!send(good)) {
                        ok = false;
                        break;
                    }
                }
            }
        }
    } else if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            if (STEMWIN) {
                // raw weights into the A stages, packed there by the epilogue warps
                ptx::mbar_arrive_expect_tx(bres_full, static_cast<uint32_t>(p.sw_wbytes));
                ptx::bulk_copy_g2s(sA, p.w, static_cast<uint32_t>(p.sw_wbytes), bres_full);
            } else if (FOLD) {
                // Weight block kh = rows (kw, co) of w[co][kh][kw][0..31]: one box of
                // C_out rows per (kh, kw) from w viewed as [C_out][KH][KW][32].
                ptx::mbar_arrive_expect_tx(
                    bres_full, static_cast<uint32_t>(p.x_KH * p.fold_n) * 64u);
                for (int kh = 0; kh < p.x_KH; ++kh)
                    for (int kw = 0; kw < p.win_kw; ++kw)
                        ptx::tma_load_4d(sB + (kh * p.fold_n + kw * p.C_out) * 64, &tmap_b, bres_full,
                                         0, kw, kh, 0);
            } else if (bres) {
                // Weights resident: every K block of the one column tile, once (in
                // a pair each CTA holds half of the columns; CTA 0's barrier counts
                // both halves).
                if (rank == 0)
                    ptx::mbar_arrive_expect_tx(bres_full, static_cast<uint32_t>(p.kb_total) * BB *
                                                              (PAIR ? 2u : 1u));
                const uint32_t bres_bar = PAIR ? ptx::mapa(ptx::smem_addr(bres_full), 0u) : 0u;
                // several column tiles: this CTA's (the grid is a multiple of their
                // count, so every unit of the CTA has column tile blockIdx.x % n_tiles)
                const int n0_res =
                    p.n_tiles > 1 ? static_cast<int>(blockIdx.x % static_cast<unsigned>(p.n_tiles)) * BN
                                  : 0;
                for (int kb = 0; kb < p.kb_total; ++kb) {
                    if (PAIR)
                        ptx::tma_load_2d_pair(sB + kb * BB, &tmap_b, bres_bar, kb * BK,
                                              static_cast<int>(rank) * (BN / 2));
                    else
                        ptx::tma_load_2d(sB + kb * BB, &tmap_b, bres_full, kb * BK, n0_res);
                }
                // (the A loads below are issued at once; the weights' arrival is
                // awaited by the MMA thread, and here only before exiting)
            }
            if (STAGEDROWS) {
                // Per tile: every input row its output rows read (KH per output row),
                // copied whole into the tile's staging slot; rows outside the image
                // are skipped (the consumer writes zeros for them).
                const uint32_t row_bytes = static_cast<uint32_t>(p.nw_W * p.nw_cin * 2);
                uint32_t slot = 0, slot_phase = 0, issued = 0;
                for (int tile = t_first; tile < total_tiles; tile += t_step, ++issued) {
                    const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                    if (!wait_bar(&stg_empty[slot], slot_phase ^ 1u, wc, kRoleTma)) break;
                    const int rows = min(p.win_rows, p.win_groups - u.m0);
                    uint32_t copies = 0;
                    for (int jj = 0; jj < rows; ++jj) {
                        uint32_t n, ho;
                        p.ho_div.divmod(static_cast<uint32_t>(u.m0 + jj), n, ho);
                        for (int kh = 0; kh < p.nw_KH; ++kh) {
                            const int h = static_cast<int>(ho) * p.nw_s - p.nw_p + kh;
                            copies += (h >= 0 && h < p.nw_H) ? 1u : 0u;
                        }
                    }
                    ptx::mbar_arrive_expect_tx(&stg_full[slot], copies * row_bytes);
                    uint8_t* slot_base = sStg + slot * p.nw_slot_bytes;
                    for (int jj = 0; jj < rows; ++jj) {
                        uint32_t n, ho;
                        p.ho_div.divmod(static_cast<uint32_t>(u.m0 + jj), n, ho);
                        for (int kh = 0; kh < p.nw_KH; ++kh) {
                            const int h = static_cast<int>(ho) * p.nw_s - p.nw_p + kh;
                            if (h < 0 || h >= p.nw_H) continue;
                            const uint16_t* src =
                                p.x + (static_cast<long long>(n) * p.nw_H + h) * p.nw_W * p.nw_cin;
                            ptx::bulk_copy_g2s(slot_base + (jj * p.nw_KH + kh) * p.nw_rb + p.nw_a0,
                                               src, row_bytes, &stg_full[slot]);
                        }
                    }
                    if (++slot == NS) {
                        slot = 0;
                        slot_phase ^= 1u;
                    }
                }
                // Wait (bounded) for the last copies so none lands after the CTA exits.
                for (uint32_t i = issued > NS ? issued - NS : 0; i < issued; ++i)
                    drain_wait(&stg_full[i % NS], (i / NS) & 1u, 1000000000ull);
            } else if (PLANE) {
                // Streamed weights: block (tap, cc) of the tile's column tile per
                // B slot, in the order the MMA thread consumes them.
                if (!bres) {
                    const int taps = p.x_KH * p.win_kw;
                    Ring rb;
                    uint32_t issued = 0;
                    bool ok = true;
                    for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                        const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                        for (int kb = u.kb0; ok && kb < u.kb1; ++kb)
                            for (int t = 0; t < taps; ++t, ++issued, rb.next(SB)) {
                                if (!wait_bar(&empty_b[rb.stage], rb.phase ^ 1u, wc, kRoleTma)) {
                                    ok = false;
                                    break;
                                }
                                ptx::mbar_arrive_expect_tx(&full_b[rb.stage], BB);
                                ptx::tma_load_2d(sB + rb.stage * BB, &tmap_b,
                                                 &full_b[rb.stage], (t * p.win_cc + kb) * BK, u.n0);
                            }
                    }
                    const uint32_t first = issued > SB ? issued - SB : 0;
                    for (uint32_t i = first; i < issued; ++i)
                        drain_wait(&full_b[i % SB], (i / SB) & 1u, 1000000000ull);
                }
            } else if (WINDOW) {
                // Per (tile, kh, cc): one box of win_wv pixels x 64 channels for each
                // of the tile's output rows (input row ho - p + kh*d, columns -p ..
                // -p + win_wv - 1; TMA zero-fills what lies outside the image), plus
                // the KW weight blocks (kh, 0..KW-1, cc) unless weights are resident.
                const uint32_t row_bytes = static_cast<uint32_t>(p.win_wv) * 128u;
                Ring ring;
                uint32_t issued = 0;
                bool ok = true;
                // A pair: each CTA stages its own tile's rows and its half of the
                // weight columns; all of it completes on CTA 0's barrier, which
                // CTA 0 arms with both CTAs' byte counts.  The peer cannot wait on
                // that barrier, so CTA 0's drain below covers the peer's copies too
                // (neither CTA exits before the final cluster barrier).
                for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                    const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                    const int rows = max(0, min(p.win_rows, p.win_groups - u.m0));
                    int rows_peer = 0;
                    if (PAIR) {
                        const Unit v = unit_of<BN, PAIR, SKM>(p, tile, 1u, skr);
                        rows_peer = max(0, min(p.win_rows, p.win_groups - v.m0));
                    }
                    for (int kb = u.kb0; kb < u.kb1; ++kb, ++issued, ring.next(S)) {
                        if (!wait_bar(&empty[ring.stage], ring.phase ^ 1u, wc, kRoleTma)) {
                            ok = false;
                            break;
                        }
                        const int kh = kb / p.win_cc, cc = kb - kh * p.win_cc;
                        const uint32_t full_cl =
                            PAIR ? ptx::mapa(ptx::smem_addr(&full_b[ring.stage]), 0u) : 0u;
                        if (rank == 0) {
                            const uint32_t tx =
                                static_cast<uint32_t>(rows + rows_peer) * row_bytes +
                                (bres ? 0u
                                        : static_cast<uint32_t>(p.win_kw) * BB * (PAIR ? 2u : 1u));
                            ptx::mbar_arrive_expect_tx(&full_b[ring.stage], tx);
                        }
                        uint8_t* stage_a = sA + ring.stage * AST;
                        for (int j = 0; j < rows; ++j) {
                            uint32_t n, ho;
                            p.ho_div.divmod(static_cast<uint32_t>(u.m0 + j), n, ho);
                            const int h = static_cast<int>(ho) - p.win_pad + kh * p.win_d;
                            if (PAIR)
                                ptx::tma_load_4d_pair(stage_a + j * row_bytes, &tmap_a, full_cl,
                                                      cc * BK, -p.win_pad, h, static_cast<int>(n));
                            else
                                ptx::tma_load_4d(stage_a + j * row_bytes, &tmap_a,
                                                 &full_b[ring.stage], cc * BK, -p.win_pad, h,
                                                 static_cast<int>(n));
                        }
                        if (!bres)
                            for (int kw = 0; kw < p.win_kw; ++kw) {
                                uint8_t* dst = sB + (ring.stage * p.b_per_stage + kw) * BB;
                                const int col = ((kh * p.win_kw + kw) * p.win_cc + cc) * BK;
                                if (PAIR)
                                    ptx::tma_load_2d_pair(dst, &tmap_b, full_cl, col,
                                                          u.n0 + static_cast<int>(rank) * (BN / 2));
                                else
                                    ptx::tma_load_2d(dst, &tmap_b, &full_b[ring.stage], col, u.n0);
                            }
                    }
                }
                const uint32_t first = issued > S ? issued - S : 0;
                if (rank == 0)
                    for (uint32_t i = first; i < issued; ++i)
                        drain_wait(&full_b[i % S], (i / S) & 1u, 1000000000ull);
            } else if (!bres || !GATHER) {
                // im2win, strided 1x1: a box of win_rows output rows x W_out pixels
                // x 64 K
                const uint32_t a_tx =
                    GATHER                ? 0u
                    : (IM2WIN || STRIDED) ? static_cast<uint32_t>(p.win_rows * p.win_wout) * 128u
                    : FOLD                ? AST
                                          : static_cast<uint32_t>(kABytes);
                const uint32_t kTx = (bres ? 0u : static_cast<uint32_t>(BB)) + a_tx;
                Ring ring;
                uint32_t issued = 0;
                bool ok = true;
                for (int tile = t_first; ok && tile < total_tiles; tile += t_step) {
                    const Unit u = unit_of<BN, PAIR, SKM>(p, tile, rank, skr);
                    for (int kb = u.kb0; kb < u.kb1; ++kb, ++issued, ring.next(S)) {
                        // (the folded window: stage s is accumulator slot s, free once
                        // the tile that last used it has completed its MMAs)
                        if (!wait_bar(FOLD ? &tfull[ring.stage] : &empty[ring.stage], ring.phase ^ 1u,
                                      wc, kRoleTma)) {
                            ok = false;
                            break;
                        }
                        if (rank == 0)
                            ptx::mbar_arrive_expect_tx(&full_b[ring.stage],
                                                       kTx * (PAIR ? 2u : 1u));
                        if (FOLD) {
                            // One box: the 32 input columns from c0 of input rows
                            // 4*hb - p .. 4*hb - p + 3 + (KH-1)*d, row after row (2 KB
                            // each).  TMA zero-fills rows outside the image; the columns
                            // all lie inside it.
                            uint32_t nhb, k, n, hb;
                            p.fold_spr_div.divmod(static_cast<uint32_t>(u.m0), nhb, k);
                            p.fold_hb_div.divmod(nhb, n, hb);
                            const int c0 =
                                min(max(static_cast<int>(k) * p.fold_g - p.win_pad, 0), p.x_W - 32);
                            ptx::tma_load_4d(sA + ring.stage * AST, &tmap_a, &full_b[ring.stage], 0,
                                             c0, static_cast<int>(hb) * (FPAIR ? 2 * kFoldRows : kFoldRows) -
                                                     p.win_pad,
                                             static_cast<int>(n));
                        } else if (IM2WIN) {
                            ptx::tma_load_3d(sA + ring.stage * AST, &tmap_a, &full_b[ring.stage],
                                             kb * BK, 0, u.m0);
                        } else if (STRIDED) {
                            // input rows ho*s.. of image n, every s-th pixel and row
                            uint32_t n, ho;
                            p.ho_div.divmod(static_cast<uint32_t>(u.m0), n, ho);
                            ptx::tma_load_4d(sA + ring.stage * AST, &tmap_a, &full_b[ring.stage],
                                             kb * BK, 0, static_cast<int>(ho) * p.st_s,
                                             static_cast<int>(n));
                        } else if (!GATHER)
                            ptx::tma_load_2d(sA + ring.stage * AST, &tmap_a, &full_b[ring.stage],
                                             kb * BK, u.m0);
                        if (!bres) {
                            if (PAIR)  // this CTA's half of the column tile
                                ptx::tma_load_2d_pair(
                                    sB + ring.stage * BB, &tmap_b,
                                    ptx::mapa(ptx::smem_addr(&full_b[ring.stage]), 0u), kb * BK,
                                    u.n0 + static_cast<int>(rank) * (BN / 2));
                            else
                                ptx::tma_load_2d(sB + ring.stage * BB, &tmap_b,
                                                 &full_b[ring.stage], kb * BK, u.n0);
                        }
                    }
                }
                // Wait (bounded) for the last loads so none lands after the CTA exits.
                const uint32_t first = issued > S ? issued - S : 0;
                if (rank == 0)
                    for (uint32_t i = first; i < issued; ++i)
                        drain_wait(&full_b[i % S], (i / S) & 1u, 1000000000ull);
            }
        }
    }

    // The resident weights must have landed before the CTA exits (a pair's
    // land on CTA 0's barrier, for both CTAs).
    if (warp == kTmaWarp && lane == 0 && bres && rank == 0)
        drain_wait(bres_full, 0u, 1000000000ull);
    ptx::tc_fence_before();
    // a pair's CTA 0 reads the peer's shared memory and writes its TMEM: neither
    // CTA leaves before both are done
    if (PAIR)
        ptx::cluster_sync();
    else
        __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        if (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, kTmemAlloc);
        else
            ptx::tmem_dealloc(tmem_base, kTmemAlloc);
    }
}

// A wait nothing will ever satisfy, bounded by the time limit: exercises the
// failure path without faulting or hanging the GPU.
__global__ void selftest_timeout_kernel(unsigned long long timeout_ns, unsigned* err)
{
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx wc{&abort_flag, err, timeout_ns};
        (void)wait_bar(&bar, 0u, wc, kRoleSelftest);
    }
}

// y[m][co] = partial[m][co] + bias[co], rounded to bf16 or stored as fp32.
__global__ void __launch_bounds__(256) finish_split_kernel(const float* __restrict__ partial,
                                                           const uint16_t* __restrict__ bias,
                                                           void* __restrict__ y, long long total,
                                                           int C_out, int y_f32)
{
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += stride) {
        float v = partial[e];
        if (bias != nullptr) v += bf16_bits_to_float(bias[e % C_out]);
        if (y_f32) {
            static_cast<float*>(y)[e] = v;
        } else {
            __nv_bfloat16 b = __float2bfloat16_rn(v);
            static_cast<uint16_t*>(y)[e] = *reinterpret_cast<uint16_t*>(&b);
        }
    }
}

template <int BN, int AMODE>
cudaError_t launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                      const IgemmParams& p, cudaStream_t st)
{
    auto kern = igemm_kernel<BN, AMODE>;
    // Per device (and per instantiation): the shared-memory opt-in, set once,
    // and the pair mode's resident-cluster count for the last size asked.
    constexpr int kDevs = 64;
    static std::mutex mu;
    static bool configured[kDevs] = {};
    static int cluster_smem[kDevs] = {}, cluster_count[kDevs] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!configured[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
            if (e != cudaSuccess) return e;
            configured[dev] = true;
        }
    }
    const int extra = ((AMODE == kANarrowWin || is_stemwin(AMODE)) ? p.nw_slots * p.nw_slot_bytes
                       : is_window(AMODE)                           ? p.win_tail
                                                                    : 0) +
                      (p.tma_store ? (p.epi_c32 ? kEpiNarrowStageBytes + (p.epi_bufs - 1) * kEpiNarrowTileBytes
                                                : kEpiStageBytes + (p.epi_bufs - 1) * kEpiTileBytes)
                                   : 0);
    constexpr bool kPlane = AMODE == kAPlane || AMODE == kAPlane3 || AMODE == kAPlane3U2;
    constexpr bool kPairMode = AMODE == kAWindowPair || AMODE == kATmaGatherPair;
    constexpr bool kFold = is_fold(AMODE);
    constexpr int kFKW = AMODE == kAWinFold3 ? kFold3MaxK : kFoldMaxKW;
    constexpr bool kFPair = AMODE == kAWinFold3 && BN == 128;  // units of two tiles
    constexpr int kFU = kFPair ? 2 * kFoldRows : kFoldRows;     // output rows per unit
    constexpr int kFKH = AMODE == kAWinFold3 ? kFold3MaxK : kFoldMaxKH;
    const int smem =
        kPlane ? plane_smem_bytes(BN, p.stages, p.a_stage_bytes, p.bres ? p.kb_total : p.b_stages,
                                  extra)
        : kFold ? fold_smem_bytes(p.fold_bbytes, p.stages, p.a_stage_bytes)
                : igemm_smem_bytes(kPairMode ? BN / 2 : BN, p.stages, p.bres, p.kb_total,
                                   p.a_stage_bytes, p.b_per_stage, extra);
    if (p.stages < 2 || p.stages > kMaxStages || smem > kSmemLimit) return cudaErrorInvalidValue;
    // gather warps taking turns: at most one phase ahead needs kGatherWarps stages
    static_assert(kMinGatherTurnStages == kGatherWarps, "turn-taking ring depth");
    if ((AMODE == kATmaGather || AMODE == kATmaGatherPair) && p.stages < kMinGatherTurnStages)
        return cudaErrorInvalidValue;
    // 32-column staging exists for the eight-warp epilogue only
    constexpr bool kEpi8 = is_window(AMODE) || AMODE == kADense || AMODE == kAIm2win ||
                           AMODE == kAStrided;
    if (p.epi_c32 && !(kEpi8 && p.tma_store)) return cudaErrorInvalidValue;
    if ((AMODE == kANarrowWin || is_stemwin(AMODE)) && (p.nw_slots < 1 || p.nw_slots > kMaxSlots))
        return cudaErrorInvalidValue;
    if (is_stemwin(AMODE)) {
        // every shared-memory access of the stem's stages and packing stays in bounds:
        // one stage row per gather thread, 128 + nkb - 1 rows per stage, the raw
        // weights inside the A stages, kernel rows in the 32-bit validity mask, and a
        // (C_in, stride) pair the builder is compiled for
        constexpr int kS = AMODE == kAStemWin1 ? 1 : AMODE == kAStemWin4 ? 4 : 2;
        const bool cs_ok = p.nw_cin == 3 && p.nw_s == kS && p.sw_kc == 64 / p.nw_s &&
                           p.sw_khg == p.sw_kc / p.nw_cin;
        if (!cs_ok || !p.bres || p.n_tiles != 1 || p.win_rows * p.win_wv > kGatherThreads ||
            (BM + p.sw_nkb - 1) * 128 > p.a_stage_bytes || p.nw_KH > 31 ||
            p.sw_wbytes > p.stages * p.a_stage_bytes || p.sw_wbytes % 16 != 0 ||
            p.kb_total != p.num_kb * p.sw_nkb || p.sw_last < 1 || p.sw_last > 4 ||
            p.sw_steps != (p.sw_nkb - 1) * 4 + p.sw_last || p.sw_steps > kStemWinMaxSteps)
            return cudaErrorInvalidValue;
    }
    if (is_window(AMODE)) {
        // every MMA read of an A slot (128 + (KW-1)*d rows of 128 bytes from the
        // slot's start) stays inside the ring and its pad, and the staged rows fit
        // a slot; slots and pad keep the staging tile 1024-byte aligned
        if (p.win_tail < 0 || p.win_tail % 1024 != 0 || p.a_stage_bytes % 1024 != 0 ||
            p.win_rows < 1 || p.win_rows * p.win_wv * 128 > p.a_stage_bytes ||
            (BM + (p.win_kw - 1) * p.win_d) * 128 > p.a_stage_bytes + p.win_tail)
            return cudaErrorInvalidValue;
    }
    if (AMODE == kAWindowT &&
        (p.bres != 1 || p.tma_store != 1 || p.epi_c32 != 0 || p.splits != 1 || p.sk ||
         p.win_kw != 3 || p.n_tiles != 1))
        return cudaErrorInvalidValue;  // the plan the kernel is built for
    if (kFold) {
        // the folded window's shared-memory layout, its unrolled loops and its
        // epilogue's register arrays: 32 channels per 64-byte row, KW*C_out MMA
        // columns (a multiple of 16 that fits one BN-column accumulator slot),
        // one K block per tile, weights resident, no split, direct stores
        const bool ok = (BN == 128 || BN == 256) && p.C_in == 32 && p.C_out % 32 == 0 &&
                        p.C_out * 4 <= kFoldBiasBytes &&
                        p.fold_n == p.win_kw * p.C_out && p.fold_n % 16 == 0 && p.fold_n >= 16 &&
                        p.fold_n <= BN && p.win_kw >= 1 && p.win_kw <= kFKW &&
                        p.x_KH >= 1 && p.x_KH <= kFKH && p.win_d >= 1 && p.x_W >= 32 &&
                        p.fold_g == 32 - (p.win_kw - 1) * p.win_d && p.fold_g >= 1 &&
                        p.a_stage_bytes == (kFU + (p.x_KH - 1) * p.win_d) * kFoldRowBytes &&
                        kFU + (p.x_KH - 1) * p.win_d <= 256 && p.num_kb == 1 &&
                        p.fold_bbytes >= p.x_KH * p.fold_n * 64 && p.fold_bbytes % 1024 == 0 &&
                        p.bres == 1 && p.n_tiles == 1 && p.splits == 1 && !p.sk && !p.tma_store &&
                        p.stages == (kFPair ? Cfg<BN>::kAcc / 2 : Cfg<BN>::kAcc) &&
                        p.fold_hout >= 1 && p.m_tiles >= 1 && p.m_step == 1;
        if (!ok) return cudaErrorInvalidValue;
    }
    if (kPlane &&
        ((!p.bres && (p.b_stages < 2 || p.b_stages > kMaxStages)) || p.pl_u < 1 || p.pl_u > 2 ||
         p.pl_nacc < 1 || p.pl_nacc > kMaxAcc || p.pl_nacc * p.pl_u * BN > 512))
        return cudaErrorInvalidValue;
    // the unrolled 3x3 variants fix the taps and the sub-tile count at compile time
    if ((AMODE == kAPlane3 || AMODE == kAPlane3U2) &&
        (p.x_KH != 3 || p.win_kw != 3 || p.pl_u != (AMODE == kAPlane3U2 ? 2 : 1)))
        return cudaErrorInvalidValue;
    const int tiles = p.m_tiles * p.n_tiles * p.splits;  // pair mode: pair units
    IgemmParams q = p;  // this launch's copy: stream-K records its grid in it
    if (p.sk) {
        // stream-K shares out every (unit, K block) iteration: as many CTAs (pairs)
        // as fit, each with at least one iteration; window kernels only, no split,
        // no column-resident weights (a CTA's iterations cross column tiles)
        constexpr bool kWin = AMODE == kAWindow || AMODE == kAWindowPair;
        if (!kWin || p.splits != 1 || (p.bres && p.n_tiles > 1) || p.sk_iters < 1 ||
            p.sk_iters != static_cast<long long>(p.m_tiles) * p.n_tiles * p.num_kb)
            return cudaErrorInvalidValue;
    }
    // Programmatic stream serialization: CTAs may start on SMs the previous
    // kernel has left while its other CTAs finish (the kernel waits for it
    // before touching global memory).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (kPairMode) {
        if (BN < 64) return cudaErrorInvalidValue;
        // Clusters of two CTAs, as many as can be resident at once (two SMs each).
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        int resident = 0;
        {
            std::lock_guard<std::mutex> lock(mu);
            if (cluster_smem[dev] != smem || cluster_count[dev] < 1) {
                int nc = 0;
                cudaLaunchConfig_t occ = cfg;  // the cluster shape alone
                occ.attrs = attr + 1;
                occ.numAttrs = 1;
                occ.gridDim = dim3(static_cast<unsigned>(num_sms() / 2 * 2));
                if (cudaOccupancyMaxActiveClusters(&nc, kern, &occ) != cudaSuccess || nc < 1) {
                    (void)cudaGetLastError();
                    nc = num_sms() / 2;
                }
                cluster_smem[dev] = smem;
                cluster_count[dev] = nc;
            }
            resident = cluster_count[dev];
        }
        int clusters = tiles < resident ? tiles : resident;
        if (p.sk) {
            clusters = p.sk_iters < resident ? static_cast<int>(p.sk_iters) : resident;
            q.sk_ctas = clusters;
        }
        cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters));
        e = cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, q);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    int grid = tiles < num_sms() ? tiles : num_sms();
    if (p.sk) {
        grid = p.sk_iters < num_sms() ? static_cast<int>(p.sk_iters) : num_sms();
        q.sk_ctas = grid;
    }
    // Resident weights with several column tiles: each CTA must see one column
    // tile only, so the grid is a whole multiple of their count.
    if (p.bres && p.n_tiles > 1) {
        if (kPlane || p.splits != 1) return cudaErrorInvalidValue;
        grid = grid >= p.n_tiles ? grid / p.n_tiles * p.n_tiles : p.n_tiles;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, ty, q);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int AMODE>
cudaError_t launch_mode(int bn, const CUtensorMap& ta, const CUtensorMap& tb,
                        const CUtensorMap& ty, const IgemmParams& p, cudaStream_t st)
{
    switch (bn) {
    case 32: return launch_bn<32, AMODE>(ta, tb, ty, p, st);
    case 64: return launch_bn<64, AMODE>(ta, tb, ty, p, st);
    case 128: return launch_bn<128, AMODE>(ta, tb, ty, p, st);
    case 256: return launch_bn<256, AMODE>(ta, tb, ty, p, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int igemm_smem_bytes(int bn, int stages, int bres, int num_kb, int a_stage_bytes,
                     int b_per_stage, int extra_bytes)
{
    const int b_blocks = bres ? num_kb : stages * b_per_stage;
    return kHeaderBytes + 1024 + b_blocks * bn * BK * 2 + stages * a_stage_bytes + extra_bytes;
}

int igemm_pick_stages(int bn, int bres, int num_kb, int a_stage_bytes, int b_per_stage,
                      int extra_bytes)
{
    for (int s = kMaxStages; s >= 2; --s)
        if (igemm_smem_bytes(bn, s, bres, num_kb, a_stage_bytes, b_per_stage, extra_bytes) <=
            kSmemLimit)
            return s;
    return 0;
}

int window_stage_rows(int kw, int d) { return (BM + (kw - 1) * d + 7) / 8 * 8; }

int fold_smem_bytes(int b_bytes, int stages, int a_stage_bytes)
{
    return kHeaderBytes + 1024 + b_bytes + stages * a_stage_bytes + kFoldBiasBytes;
}

int plane_smem_bytes(int bn, int a_stages, int a_stage_bytes, int b_blocks, int extra_bytes)
{
    return kHeaderBytes + 1024 + b_blocks * bn * BK * 2 + a_stages * a_stage_bytes + extra_bytes;
}

int smem_limit() { return kSmemLimit; }

cudaError_t launch_igemm(int amode, int bn, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& ty, const IgemmParams& p, cudaStream_t st)
{
    switch (amode) {
    case kADense: return launch_mode<kADense>(bn, ta, tb, ty, p, st);
    case kAGather: return launch_mode<kAGather>(bn, ta, tb, ty, p, st);
    case kANarrow: return launch_mode<kANarrow>(bn, ta, tb, ty, p, st);
    case kATmaGather: return launch_mode<kATmaGather>(bn, ta, tb, ty, p, st);
    case kAWindow: return launch_mode<kAWindow>(bn, ta, tb, ty, p, st);
    case kAWindowPair: return launch_mode<kAWindowPair>(bn, ta, tb, ty, p, st);
    case kAWindowT: return launch_mode<kAWindowT>(bn, ta, tb, ty, p, st);
    case kAIm2win: return launch_mode<kAIm2win>(bn, ta, tb, ty, p, st);
    case kAStrided: return launch_mode<kAStrided>(bn, ta, tb, ty, p, st);
    case kATmaGatherPair: return launch_mode<kATmaGatherPair>(bn, ta, tb, ty, p, st);
    case kANarrowWin: return launch_mode<kANarrowWin>(bn, ta, tb, ty, p, st);
    case kAPlane: return launch_mode<kAPlane>(bn, ta, tb, ty, p, st);
    case kAPlane3: return launch_mode<kAPlane3>(bn, ta, tb, ty, p, st);
    case kAPlane3U2: return launch_mode<kAPlane3U2>(bn, ta, tb, ty, p, st);
    case kAStemWin: return launch_mode<kAStemWin>(bn, ta, tb, ty, p, st);
    case kAStemWin1: return launch_mode<kAStemWin1>(bn, ta, tb, ty, p, st);
    case kAStemWin4: return launch_mode<kAStemWin4>(bn, ta, tb, ty, p, st);
    // (accumulator slots of 128 or 256 columns: MMA widths up to 128 or 256)
    case kAWinFold:
        return bn == 128   ? launch_bn<128, kAWinFold>(ta, tb, ty, p, st)
               : bn == 256 ? launch_bn<256, kAWinFold>(ta, tb, ty, p, st)
                           : cudaErrorInvalidValue;
    case kAWinFold3:
        return bn == 128   ? launch_bn<128, kAWinFold3>(ta, tb, ty, p, st)
               : bn == 256 ? launch_bn<256, kAWinFold3>(ta, tb, ty, p, st)
                           : cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_finish_split(const float* partial, const uint16_t* bias, void* y, long long M,
                                int C_out, int y_f32, cudaStream_t st)
{
    const long long total = M * C_out;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms()) * 8;
    if (blocks > cap) blocks = cap;
    finish_split_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(partial, bias, y, total, C_out,
                                                                  y_f32);
    return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned long long timeout_ns, unsigned* err, cudaStream_t st)
{
    selftest_timeout_kernel<<<1, 32, 0, st>>>(timeout_ns, err);
    return cudaGetLastError();
}

}  // namespace convgb
