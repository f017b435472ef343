// Block-scaled FP8 GEMM with per-128-K promotion, dense and grouped (MoE).
//
// What it computes ("Six Reasons Deepseek Ai Is A Waste Of Time", paras. 1-3;
// "increased accumulation precision" section of the codingmall FP8 article):
// C[m][n] = sum_g sA[g][m] * sB(n, g) * P_g[m][n], where P_g is the FP8 dot
// product over the g-th 128-element block of K.  The tensor cores produce
// P_g; the CUDA cores scale it and add it into FP32 accumulators
// ("promotion"), once per 128-element K block.
//
// Blackwell design (the pages' Hopper design -- two warpgroups alternating
// WGMMA and promotion -- is prior art; this is its sm_103a counterpart):
//   * producer warp (1 thread): TMA loads of the A tile (128 x 128 B) and
//     B tile (BN x 128 B) into a ring of shared-memory stages (128-byte
//     swizzle), plus, for 1x128-scaled B (weight gradient), bulk copies of
//     both operands' scales of the block into a separate ring of scale slots;
//   * MMA warp (1 thread): 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) per
//     128-K block into one of 512/BN TMEM buffers (128 lanes x BN FP32
//     columns), a fresh accumulation per block; tcgen05.commit releases the
//     smem stage and signals the promotion warps;
//   * BN/128 promotion warpgroups: tcgen05.ld the partial in 16-column
//     chunks (8 for row-scaled B), the next chunk's load in flight while the
//     current one is scaled, release the TMEM buffer once the last chunk has
//     arrived, and accumulate P * (sA * sB) into 128 FP32 registers per thread
//     with packed FP32 FMAs (128x128-block B: each warp prefetches its scales
//     into its own shared-memory ring with cp.async); after the last block,
//     write C.
// The MMA of block i+1 (other TMEM buffer) overlaps the promotion of block i.
// Persistent: one CTA per SM walks tiles blockIdx.x, +gridDim.x, ...; the
// rings carry over from one tile to the next.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "quant.cuh"   // group_scale: the scale rule of the in-kernel quantizer

namespace fp8q {

constexpr int kBM = 128;          // rows of A per tile (TMEM lanes)
constexpr int kBK = 128;          // K per block = scale-group width = one 128-byte swizzle row
constexpr int kScaleSlots = 8;
constexpr int kScaleAhead = 4;    // block-scaled B: scale look-ahead of the promotion warps
constexpr int kScaleRing = 8;     //   ring slots per promotion warp (more than kScaleAhead)
constexpr int kRingSlotFloats = 36;   // 32 row scales + the block scale, padded to 16 bytes
constexpr int kMaxGroups = 512;

// Warp roles, by warpgroup (four consecutive warps, one on each SM
// sub-partition): warpgroup 0 = control (warp 0 = TMA producer, warp kMmaWarp
// = MMA issuer and TMEM owner, the other two idle); warpgroup 1 + h promotes
// the 128-column half h of the tile.  A warp may only read the TMEM lanes
// 32*(warp % 4) .. +31, so promotion warp w takes lane quarter w % 4: each
// thread owns one row of the tile and 128 FP32 accumulators.  For BN = 256
// the control warpgroup gives registers up to the promotion warpgroups
// (setmaxnreg): per sub-partition 56 + 2 * 224 = 504 <= 512 registers a lane.
#ifndef FP8Q_MMA_WARP
#define FP8Q_MMA_WARP 1
#endif
//
// With kQA (activations quantized inside the GEMM), warpgroup 1 is the
// quantizer: thread q converts row q of the A tile of each K block from BF16
// to E4M3 (1x128 scale rule) straight into the operand stage, and the
// promotion warpgroups move up by one.  Registers per lane then split
// 40 (control) + 88 (quantizer) + 2 * 192 (promotion) = 512.
template <int BN, bool kQA = false>
struct GemmShape {
    static constexpr int kHalves = BN / 128;             // 128-column halves of the tile
    static constexpr int kPromoWarps = 4 * kHalves;
    static constexpr int kProducerWarp = 0;
    static constexpr int kMmaWarp = FP8Q_MMA_WARP;
    static constexpr int kFirstQuantWarp = 4;
    static constexpr int kFirstPromoWarp = kQA ? 8 : 4;
    static constexpr int kThreads = 128 * (1 + kHalves + (kQA ? 1 : 0));
    static constexpr bool kRealloc = kHalves > 1;
    static constexpr int kCtrlRegs = kQA ? 40 : 56;
    static constexpr int kQuantRegs = 88;
    static constexpr int kPromoRegs = kQA ? 192 : 224;
    static constexpr int kLaunchRegs = (65536 / kThreads) & ~7;
    static_assert(!kRealloc || 128 * kCtrlRegs + (kQA ? 128 * kQuantRegs : 0) +
                                       128 * kHalves * kPromoRegs <= kThreads * kLaunchRegs,
                  "register split exceeds the launch allocation");
    static_assert(!kQA || kRealloc, "in-kernel quantization needs the 256-column tile");
    // arrivals completing a stage: the producer's (with the TMA byte count),
    // plus one per quantizer warp
    static constexpr int kFullArrivals = 1 + (kQA ? 4 : 0);
    static_assert(kMmaWarp > 0 && kMmaWarp < 4, "MMA warp must be a control warp");
    static constexpr int kStages = BN == 256 ? 3 : 5;
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTbufs = 512 / BN;              // TMEM partial buffers in flight
    static constexpr int kTmemCols = kTbufs * BN;
    // epilogue staging: per promotion warp, two 32-row x 128-byte boxes of C
    // laid out with the 128-byte swizzle the C tensor map uses
    static constexpr int kEpiBoxBytes = 32 * 128;
    static constexpr int kEpiWarpBytes = 2 * kEpiBoxBytes;
    static constexpr int kOffEpi = kStages * kStageBytes;
    static constexpr int kSaBytes = kBM * 4;
    static constexpr int kSbBytes = BN * 4;
    static constexpr int kSlotBytes = kSaBytes + kSbBytes;
    static constexpr int kOffScale = kOffEpi + kPromoWarps * kEpiWarpBytes;
    static constexpr int kOffBars = kOffScale + kScaleSlots * kSlotBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * kScaleSlots + 2 * kTbufs + 1;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kOffSched = kOffMisc + 32;
    static constexpr int kOffGroups = kOffSched + 64;
    static constexpr int kSmemBytes = kOffGroups + 2 * (kMaxGroups + 1) * 4 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kPromoWarps * kScaleRing * kRingSlotFloats * 4 <= kScaleSlots * kSlotBytes,
                  "the promotion warps' scale rings live in the slot area");
    static_assert(kTmemCols <= 512, "TMEM budget");
};

struct GemmArgs {
    const float* sA;        // [K/128][M_total]
    const float* sB;        // block: [G][N/128][K/128]; row: [K/128][N]
    void* C;                // [M_total][N]
    const int* m_offsets;   // grouped: [G+1] device array; dense: nullptr
    int M_total, N, K, G;
    int* status;
    float* ws;              // stream-K partial tiles, or nullptr (whole tiles only)
    int* counters;          // stream-K arrival counters, zero between calls
    const uint16_t* Abf;    // in-kernel quantization: BF16 activations [M_total][K]
    float* sA_out;          // in-kernel quantization: emitted 1x128 scales [K/128][M_total]
                            // (nullptr: none; A8 goes out through the tmA store map)
    int sk_reduce;          // 1: stream-K pieces only write their partials; k_sk_reduce,
                            // launched next, sums them (block-scaled B only); 0: the last
                            // piece of each tile to arrive sums them in this kernel
};

// ------------------------------------------------------------ work schedule
// Output tiles are numbered t = 0 .. tiles-1, each with Kb K blocks.  With a
// workspace, the last (partial) wave -- plus one full wave when the partial
// wave is less than half a wave -- is shared out as "stream-K" work: its tiles' K iterations, laid end to end, are cut into
// sk_ctas equal contiguous ranges, one per CTA; every other tile is done whole
// by CTA t % gridDim.x.  A tile cut between CTAs is finished by whichever of
// them arrives last (per-warp arrival counters): each writes its FP32 partial
// to the workspace and the last sums all of them in K order, so the result
// does not depend on arrival order and no CTA ever waits for another.
struct Sched {
    int tiles, Kb, G;       // G = gridDim.x
    int dp_tiles;           // tiles done whole (a multiple of G)
    int sk_ctas;            // CTAs 0 .. sk_ctas-1 share the stream-K iterations
    long long sk_iters;     // (tiles - dp_tiles) * Kb

    __host__ __device__ void plan(int t_, int kb_, int g_, bool allow_sk) {
        tiles = t_; Kb = kb_; G = g_;
        dp_tiles = tiles; sk_ctas = 0; sk_iters = 0;
        if (!allow_sk || tiles % G == 0) return;
        const int q = tiles / G, r = tiles % G;
        const int dp = q == 0 ? 0 : (2 * r >= G ? q * G : (q - 1) * G);
        const long long S = static_cast<long long>(tiles - dp) * Kb;
        long long g = S / 8;                   // at least 8 K blocks per CTA (so no
                                               // stream-K CTA has an empty range)
        if (g > G) g = G;
        if (g < 1) g = 1;
        const long long sk_max = static_cast<long long>(dp / G) * Kb + (S + g - 1) / g;
        const long long dp_max = static_cast<long long>((tiles + G - 1) / G) * Kb;
        // a cut tile costs its pieces a partial-tile write, an arrival and
        // (for the last) the sum: measured at several microseconds, about 16
        // K blocks of MMA work per CTA
        if (sk_max + 16 >= dp_max) return;
        dp_tiles = dp; sk_ctas = static_cast<int>(g); sk_iters = S;
    }
    __host__ __device__ long long lo(int c) const { return c < sk_ctas ? c * sk_iters / sk_ctas : 0; }
    __host__ __device__ long long hi(int c) const { return c < sk_ctas ? (c + 1) * sk_iters / sk_ctas : 0; }
    // CTA whose stream-K range holds iteration x.
    __host__ __device__ int cta_of(long long x) const {
        return static_cast<int>(((x + 1) * sk_ctas - 1) / sk_iters);
    }
    // Workspace slot of CTA c's piece of stream-K tile `rel`: each CTA has at
    // most two split pieces, the first (slot 2c) and the last (2c + 1) of its
    // range.  Of the CTAs c_lo..c_hi holding pieces of a tile, only c_lo's
    // piece can be the last of its range (its range starts before the tile).
    __host__ __device__ int slot_in_tile(int c, int c_lo, bool clo_started_before) const {
        return 2 * c + ((c == c_lo && clo_started_before) ? 1 : 0);
    }
};

struct Seg {
    int t, kb0, kb1;        // tile and its K-block range [kb0, kb1)
    int rel;                // stream-K tile index (t - dp_tiles) if split, else -1
    int slot;               // workspace slot of this piece (split pieces only)
};

struct SegIter {
    const Sched* sc;
    int c, t_dp;
    long long i, end;
    bool first;             // the next stream-K piece is the first of the range
    __host__ __device__ void start(const Sched* s, int cta) {
        sc = s; c = cta; t_dp = cta; i = s->lo(cta); end = s->hi(cta); first = true;
    }
    __host__ __device__ bool next(Seg& g) {
        if (t_dp < sc->dp_tiles) {
            g.t = t_dp; g.kb0 = 0; g.kb1 = sc->Kb; g.rel = -1;
            t_dp += sc->G;
            return true;
        }
        if (i >= end) return false;
        const int rel = static_cast<int>(i / sc->Kb);
        const int kb0 = static_cast<int>(i % sc->Kb);
        const long long left = end - i;
        const int kb1 = left < sc->Kb - kb0 ? kb0 + static_cast<int>(left) : sc->Kb;
        g.t = sc->dp_tiles + rel; g.kb0 = kb0; g.kb1 = kb1;
        g.rel = (kb0 == 0 && kb1 == sc->Kb) ? -1 : rel;
        g.slot = 2 * c + (first ? 0 : 1);
        first = false;
        i += kb1 - kb0;
        return true;
    }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// acc[j] += (P[2j], P[2j+1]) * scale for the W columns of one TMEM chunk.
// Block-scaled B: one factor f = sA * sB for the whole row segment.
// Row-scaled B (weight gradient): factor fa * sB[n] per column n.
template <bool kRowB, int W>
__device__ __forceinline__ void promote_chunk(float2* acc, const uint32_t (&r)[W], float f,
                                              float fa, const float* sb) {
    if (!kRowB) {
        const float2 ff = make_float2(f, f);
#pragma unroll
        for (int j = 0; j < W / 2; ++j)
            acc[j] = __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])),
                                ff, acc[j]);
    } else {
        const float2 fa2 = make_float2(fa, fa);
        const float4* sb4 = reinterpret_cast<const float4*>(sb);
#pragma unroll
        for (int j4 = 0; j4 < W / 4; ++j4) {
            const float4 q = sb4[j4];
            const float2 f01 = __fmul2_rn(fa2, make_float2(q.x, q.y));
            const float2 f23 = __fmul2_rn(fa2, make_float2(q.z, q.w));
            acc[2 * j4] = __ffma2_rn(
                make_float2(__uint_as_float(r[4 * j4]), __uint_as_float(r[4 * j4 + 1])), f01,
                acc[2 * j4]);
            acc[2 * j4 + 1] = __ffma2_rn(
                make_float2(__uint_as_float(r[4 * j4 + 2]), __uint_as_float(r[4 * j4 + 3])), f23,
                acc[2 * j4 + 1]);
        }
    }
}

// Columns of the partial per tcgen05.ld in the promotion loop (block-scaled
// and row-scaled B).  tcgen05.wait::ld waits for every load the thread has
// in flight, so each wait costs one load latency: wider loads mean fewer
// waits before the TMEM buffer can go back to the MMA warp.
#ifndef FP8Q_PROMO_W
#define FP8Q_PROMO_W 16
#endif
#ifndef FP8Q_PROMO_W_ROW
#define FP8Q_PROMO_W_ROW 8
#endif

// One promotion warp's share of a 128-K block: the thread's 128 columns of
// the TMEM partial, scaled and added into acc.  W < 64: chunks of W columns
// with the next chunk's load in flight while the current one is scaled.
// W = 64: two loads of 64 columns into one register buffer.  The TMEM buffer
// goes back to the MMA warp (one arrive per warp on free_bar) as soon as the
// last load has landed, before that chunk is accumulated.
template <bool kRowB, int W>
__device__ __forceinline__ void promote_block(float2* acc, uint32_t taddr, float f, float fa,
                                              const float* sbc, uint64_t* free_bar, int lane) {
    if constexpr (W == 64) {
        uint32_t r[64];
        tmem_ld_chunk(taddr, r);
        tmem_ld_wait(r);
        promote_chunk<kRowB>(acc, r, f, fa, sbc);
        tmem_ld_chunk(taddr + 64, r);
        tmem_ld_wait(r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(free_bar);
        promote_chunk<kRowB>(acc + 32, r, f, fa, sbc + 64);
    } else {
        constexpr int kC = 128 / W;
        uint32_t r0[W], r1[W];
        tmem_ld_chunk(taddr, r0);
        tmem_ld_wait(r0);
#pragma unroll
        for (int c = 0; c < kC; c += 2) {
            tmem_ld_chunk(taddr + (c + 1) * W, r1);
            promote_chunk<kRowB>(acc + c * (W / 2), r0, f, fa, sbc + c * W);
            tmem_ld_wait(r1);
            if (c + 2 < kC) {
                tmem_ld_chunk(taddr + (c + 2) * W, r0);
            } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(free_bar);
            }
            promote_chunk<kRowB>(acc + (c + 1) * (W / 2), r1, f, fa, sbc + (c + 1) * W);
            if (c + 2 < kC) tmem_ld_wait(r0);
        }
    }
}

// Tile t -> A row of the tile, B row (in the [G*N] view), first column, group.
struct TileCoord {
    int arow, brow, n0, e;
};

template <int BN>
__device__ __forceinline__ TileCoord decode_tile(int t, bool grouped, int N, int G,
                                                 const int* gtile, const int* grow) {
    const int ntn = N / BN;
    TileCoord tc;
    if (!grouped) {
        tc.e = 0;
        tc.arow = (t / ntn) * kBM;
        tc.n0 = (t % ntn) * BN;
        tc.brow = tc.n0;
        return tc;
    }
    int lo = 0, hi = G - 1;          // group e with gtile[e] <= t < gtile[e+1]
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (gtile[mid + 1] <= t) lo = mid + 1; else hi = mid;
    }
    const int local = t - gtile[lo];
    tc.e = lo;
    tc.arow = grow[lo] + (local / ntn) * kBM;
    tc.n0 = (local % ntn) * BN;
    tc.brow = lo * N + tc.n0;
    return tc;
}

// One promotion warp's epilogue: its 32 rows x 128 columns of C, held as one
// row per thread in acc, go out through shared memory and TMA stores.  Each
// round stages two boxes of 32 rows x 128 bytes (64 BF16 or 32 FP32 columns)
// in the warp's own staging area, 16-byte chunk j of row r at chunk position
// j ^ (r % 8) (the 128-byte swizzle, which also spreads the lanes' stores
// over all shared-memory banks), then lane 0 issues the two box stores.
// BF16 output takes one round, FP32 two; before a round overwrites the
// staging area, lane 0 waits until the previous stores have read it.
template <bool kBf16Out>
__device__ __forceinline__ void store_tile_tma(const float2* acc, uint8_t* stg,
                                               const CUtensorMap* tmC, int x0, int y0, int lane) {
    constexpr int kColsPerBox = kBf16Out ? 64 : 32;
    constexpr int kRounds = kBf16Out ? 1 : 2;
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int bx = 0; bx < 2; ++bx) {
            const int box = rd * 2 + bx;
            uint8_t* row = stg + bx * 4096 + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 v;
                if (kBf16Out) {
                    const float2* a = acc + box * 32 + j * 4;
                    v.x = pack_bf16x2(a[0].x, a[0].y);
                    v.y = pack_bf16x2(a[1].x, a[1].y);
                    v.z = pack_bf16x2(a[2].x, a[2].y);
                    v.w = pack_bf16x2(a[3].x, a[3].y);
                } else {
                    const float2* a = acc + box * 16 + j * 2;
                    v = make_uint4(__float_as_uint(a[0].x), __float_as_uint(a[0].y),
                                   __float_as_uint(a[1].x), __float_as_uint(a[1].y));
                }
                *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = v;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmC, stg, x0 + (rd * 2) * kColsPerBox, y0);
            tma_store_2d(tmC, stg + 4096, x0 + (rd * 2 + 1) * kColsPerBox, y0);
            bulk_commit_group();
        }
    }
}

// In-kernel 1x128 quantization of one row of one 128-K block: 128 BF16
// values (v, 16 x 16 bytes) -> 128 E4M3 bytes written into the A tile of an
// operand stage at row `row`, with the same 128-byte swizzle a TMA load of
// the A8 tile would have produced (16-byte chunk j at j ^ (row % 8)).  The
// scale rule is the quantizers': amax is exact (the largest BF16 magnitude,
// found as the largest of the 15-bit magnitude fields, whose order equals the
// order of the finite values), s = amax / 448 and inv = 448 / amax, both
// correctly rounded, the cast is round-to-nearest-even and saturating.
// Returns s.
__device__ __forceinline__ float quant_row_to_stage(const uint4 (&v)[16], uint8_t* tile, int row) {
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        m = __vmaxu2(m, v[i].x & 0x7FFF7FFFu);
        m = __vmaxu2(m, v[i].y & 0x7FFF7FFFu);
        m = __vmaxu2(m, v[i].z & 0x7FFF7FFFu);
        m = __vmaxu2(m, v[i].w & 0x7FFF7FFFu);
    }
    const uint32_t mb = (m & 0xFFFFu) > (m >> 16) ? (m & 0xFFFFu) : (m >> 16);
    float sc, inv;
    group_scale(__uint_as_float(mb << 16), sc, inv);
    uint8_t* base = tile + row * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {          // 16 values per 16-byte chunk
        const uint32_t w[8] = {v[2 * j].x, v[2 * j].y, v[2 * j].z, v[2 * j].w,
                               v[2 * j + 1].x, v[2 * j + 1].y, v[2 * j + 1].z, v[2 * j + 1].w};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint32_t lo = cvt_e4m3x2(__fmul_rn(__uint_as_float(w[2 * h] << 16), inv),
                                           __fmul_rn(__uint_as_float(w[2 * h] & 0xFFFF0000u), inv));
            const uint32_t hi = cvt_e4m3x2(__fmul_rn(__uint_as_float(w[2 * h + 1] << 16), inv),
                                           __fmul_rn(__uint_as_float(w[2 * h + 1] & 0xFFFF0000u), inv));
            o[h] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(base + ((j ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    return sc;
}

template <int BN, bool kRowB, bool kBf16Out, bool kQA = false>
__global__ void __launch_bounds__(GemmShape<BN, kQA>::kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
    using S = GemmShape<BN, kQA>;
    static_assert(!(kQA && kRowB), "in-kernel quantization is for 128x128-block weights");
    constexpr bool kSlots = kRowB || kQA;     // per-block scales go through the slot ring
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBars);
    uint64_t* full = bars;
    uint64_t* empty = full + S::kStages;
    uint64_t* sfull = empty + S::kStages;
    uint64_t* sempty = sfull + kScaleSlots;
    uint64_t* tfull = sempty + kScaleSlots;
    uint64_t* tempty = tfull + S::kTbufs;
    uint64_t* drain = tempty + S::kTbufs;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
    Sched* sched_smem = reinterpret_cast<Sched*>(smem + S::kOffSched);
    int* gtile = reinterpret_cast<int*>(smem + S::kOffGroups);
    int* grow = gtile + (kMaxGroups + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = args.N, Kb = args.K / kBK, ntn = N / BN;
    const bool grouped = args.m_offsets != nullptr;

    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int i = 0; i < S::kStages; ++i) {
            mbar_init(&full[i], S::kFullArrivals);
            mbar_init(&empty[i], 1);
        }
#pragma unroll 1
        for (int i = 0; i < kScaleSlots; ++i) {
            mbar_init(&sfull[i], kQA ? 4 : 1);
            mbar_init(&sempty[i], S::kPromoWarps);
        }
#pragma unroll 1
        for (int i = 0; i < S::kTbufs; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], S::kPromoWarps);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
        int bad = 0, tiles = 0;
        if (grouped) {
            gtile[0] = 0;
#pragma unroll 1
            for (int e = 0; e <= args.G; ++e) {
                const int o = args.m_offsets[e];
                if (o < 0 || (o % kBM) != 0 || o > args.M_total || (e > 0 && o < grow[e - 1])) bad = 1;
                grow[e] = o;
                if (e > 0) {
                    tiles += ((o - grow[e - 1]) / kBM) * ntn;
                    gtile[e] = tiles;
                }
            }
            if (bad) {
                tiles = 0;
                atomicCAS(args.status, kOk, kErrBadGroups);
            }
        } else {
            tiles = (args.M_total / kBM) * ntn;
        }
        misc[1] = static_cast<uint32_t>(tiles);
        sched_smem->plan(tiles, Kb, static_cast<int>(gridDim.x), args.ws != nullptr);
    }
    if (warp == S::kMmaWarp) {
        tmem_alloc(&misc[0], S::kTmemCols);
        tmem_relinquish();
    }
    if (warp == S::kProducerWarp && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmC);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    const Sched& sched = *sched_smem;        // read from shared memory where used

    if (warp < 4) {
        // ----------------------------------------------------- control
        if (S::kRealloc) setmaxnreg_dec<S::kCtrlRegs>();
        if (warp == S::kProducerWarp && lane == 0) {
            // -------------------------------------------------- producer
            uint32_t stage = 0, phase = 0, slot = 0, sphase = 0;
            bool ok = true;
            SegIter si;
            si.start(sched_smem, blockIdx.x);
            Seg sg;
#pragma unroll 1
            while (ok && si.next(sg)) {
                const TileCoord tc = decode_tile<BN>(sg.t, grouped, N, args.G, gtile, grow);
#pragma unroll 1
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, args.status)) { ok = false; break; }
                    uint8_t* sa = smem + stage * S::kStageBytes;
                    if (kQA) {
                        // the quantizer warps write the A tile; TMA brings B
                        mbar_arrive_expect_tx(&full[stage], S::kBBytes);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
                        tma_load_2d(sa, &tmA, &full[stage], kb * kBK, tc.arow);
                    }
                    tma_load_2d(sa + S::kABytes, &tmB, &full[stage], kb * kBK, tc.brow);
                    if (++stage == S::kStages) { stage = 0; phase ^= 1; }

                    if (kRowB) {
                        // weight-gradient form: both operands' 1x128 scales of
                        // this block go through a shared-memory slot
                        if (!mbar_wait(&sempty[slot], sphase ^ 1, args.status)) { ok = false; break; }
                        fence_proxy_async_smem();
                        float* sl = reinterpret_cast<float*>(smem + S::kOffScale + slot * S::kSlotBytes);
                        mbar_arrive_expect_tx(&sfull[slot], S::kSlotBytes);
                        bulk_load(sl, args.sA + static_cast<size_t>(kb) * args.M_total + tc.arow,
                                  S::kSaBytes, &sfull[slot]);
                        bulk_load(sl + kBM, args.sB + static_cast<size_t>(kb) * N + tc.n0,
                                  S::kSbBytes, &sfull[slot]);
                        if (++slot == kScaleSlots) { slot = 0; sphase ^= 1; }
                    }
                }
            }
        } else if (warp == S::kMmaWarp && lane == 0) {
            // ------------------------------------------------------- MMA
            constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, BN);
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true;
            SegIter si;
            si.start(sched_smem, blockIdx.x);
            Seg sg;
#pragma unroll 1
            while (ok && si.next(sg)) {
#pragma unroll 1
                for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                    const uint32_t b = it % S::kTbufs, tph = (it / S::kTbufs) & 1;
                    if (!mbar_wait(&tempty[b], tph ^ 1, args.status)) { ok = false; break; }
                    tc_fence_after();
                    if (!mbar_wait(&full[stage], phase, args.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * S::kStageBytes);
                    const uint64_t ad = sw128_desc(a_addr);
                    const uint64_t bd = sw128_desc(a_addr + S::kABytes);
                    const uint32_t d = tmem_base + b * BN;
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_e4m3(d, ad + 2 * k, bd + 2 * k, kIdesc, k > 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    mma_commit(&tfull[b]);
                    if (++stage == S::kStages) { stage = 0; phase ^= 1; }
                }
            }
            // Every MMA issued above has completed once this barrier flips.
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(drain), 0)) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicCAS(args.status, kOk, kErrTimeout);
                    break;
                }
            }
        }
        __syncwarp();
        tc_fence_before();
        cta_barrier(S::kThreads);
        if (warp == S::kMmaWarp) {
            tc_fence_after();
            tmem_dealloc(tmem_base, S::kTmemCols);
        }
    } else if (kQA && warp < S::kFirstPromoWarp) {
        // ----------------------------------------------------- quantizer
        // Thread q owns row q of every A tile: it loads the row's 128 BF16
        // values of the block (before waiting for the stage, so the loads
        // overlap the wait), quantizes them into the stage, puts the scale in
        // the slot ring for the promotion warps, and -- when the call emits
        // the stored activations and this is the tile of column 0, so that
        // every block is emitted once -- writes the scale to sA_out; lane 0
        // then copies the warp's 32 rows of E4M3 bytes out with a TMA store
        // from the stage (its layout is that of the A8 tensor map).
        setmaxnreg_dec<S::kQuantRegs>();
        const int q = threadIdx.x - S::kFirstQuantWarp * 32;
        const int qw = q >> 5;
        uint32_t stage = 0, phase = 0, slot = 0, sphase = 0;
        bool ok = true;
        SegIter si;
        si.start(sched_smem, blockIdx.x);
        Seg sg;
#pragma unroll 1
        while (ok && si.next(sg)) {
            const TileCoord tc = decode_tile<BN>(sg.t, grouped, N, args.G, gtile, grow);
            const bool emit = args.sA_out != nullptr && tc.n0 == 0;
            const uint16_t* src = args.Abf + static_cast<size_t>(tc.arow + q) * args.K;
#pragma unroll 1
            for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                uint4 v[16];
                const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<size_t>(kb) * kBK);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __ldg(p + i);
                if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1, args.status))) {
                    ok = false;
                    break;
                }
                // Every block commits one bulk group (empty unless it emits),
                // so waiting until kStages - 1 groups are pending means the
                // store of the block that last used this stage has read it.
                if (lane == 0) bulk_wait_read_pending<S::kStages - 1>();
                __syncwarp();
                uint8_t* tile = smem + stage * S::kStageBytes;
                const float sc = quant_row_to_stage(v, tile, q);
                if (emit) args.sA_out[static_cast<size_t>(kb) * args.M_total + tc.arow + q] = sc;
                if (!__all_sync(0xffffffffu, mbar_wait(&sempty[slot], sphase ^ 1, args.status))) {
                    ok = false;
                    break;
                }
                reinterpret_cast<float*>(smem + S::kOffScale + slot * S::kSlotBytes)[q] = sc;
                fence_proxy_async_smem();          // the MMA reads the tile through the async proxy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&full[stage]);
                    mbar_arrive(&sfull[slot]);
                    if (emit) tma_store_2d(&tmA, tile + qw * 4096, kb * kBK, tc.arow + qw * 32);
                    bulk_commit_group();
                }
                if (++stage == S::kStages) { stage = 0; phase ^= 1; }
                if (++slot == kScaleSlots) { slot = 0; sphase ^= 1; }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        tc_fence_before();
        cta_barrier(S::kThreads);
    } else {
        // ----------------------------------------------------- promotion
        if (S::kRealloc) setmaxnreg_inc<S::kPromoRegs>();
        const int half = (warp - S::kFirstPromoWarp) >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;       // TMEM lane = row of the tile
        uint32_t it = 0, slot = 0, sphase = 0;
        bool ok = true;
        float2 acc[64];                            // columns 2j, 2j+1 of this thread's half
        const int pw = warp - S::kFirstPromoWarp;  // promotion warp: one 32 x 128 slice
        SegIter si;
        si.start(sched_smem, blockIdx.x);
        Seg sg;
#pragma unroll 1
        while (ok && si.next(sg)) {
            const TileCoord tc = decode_tile<BN>(sg.t, grouped, N, args.G, gtile, grow);
            // Block-scaled B: this warp's 32 row scales and its half's block
            // scale of each K block come into the warp's own shared-memory ring
            // by cp.async, kScaleAhead blocks ahead, and are read from there.
            // A global load in flight in a promotion warp costs far more than
            // its latency -- the warp's next barrier or TMEM wait waits for it
            // (measured: the forward GEMM ~9% slower with the scales loaded by
            // __ldg several blocks ahead than with none loaded) -- while
            // cp.async writes no register and is waited for per thread.
            const float* sb_blk =
                args.sB + (static_cast<size_t>(tc.e) * (N / 128) + (tc.n0 / 128 + half)) * Kb;
            float* sring = reinterpret_cast<float*>(smem + S::kOffScale) +
                           pw * (kScaleRing * kRingSlotFloats);
            const float* sa_lane = args.sA + tc.arow + quarter * 32 + lane;
            // issue block k's copies (an empty group past the segment's end)
            auto prefetch = [&](int k) {
                if (k < sg.kb1) {
                    float* sl = sring + (k % kScaleRing) * kRingSlotFloats;
                    cp_async_4(sl + lane, sa_lane + static_cast<size_t>(k) * args.M_total);
                    if (lane == 0) cp_async_4(sl + 32, sb_blk + k);
                }
                cp_async_commit();
            };
            float fb_next = 0.0f;
            if (kQA) {
                fb_next = __ldg(sb_blk + sg.kb0);
            } else if (!kRowB) {
                __syncwarp();                          // the last segment's reads are done
#pragma unroll
                for (int q = 0; q < kScaleAhead; ++q) prefetch(sg.kb0 + q);
            }
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = make_float2(0.0f, 0.0f);
#pragma unroll 1
            for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++it) {
                const uint32_t b = it % S::kTbufs, tph = (it / S::kTbufs) & 1;
                float fa, f;
                const float* sbc = reinterpret_cast<const float*>(smem);   // read only if kRowB
                if (kQA) {
                    // the row scale comes from the quantizer warps' slot ring
                    if (!__all_sync(0xffffffffu, mbar_wait(&sfull[slot], sphase, args.status))) {
                        ok = false;
                        break;
                    }
                    fa = reinterpret_cast<const float*>(smem + S::kOffScale + slot * S::kSlotBytes)[row];
                    f = fa * fb_next;
                    if (kb + 1 < sg.kb1) fb_next = __ldg(sb_blk + kb + 1);
                } else if (!kRowB) {
                    cp_async_wait<kScaleAhead - 1>();  // this lane's copies for block kb
                    __syncwarp();                      // and lane 0's block scale
                    const float* sl = sring + (kb % kScaleRing) * kRingSlotFloats;
                    fa = sl[lane];
                    f = fa * sl[32];
                    prefetch(kb + kScaleAhead);        // its slot was last read kScaleRing -
                                                       // kScaleAhead blocks ago
                } else {
                    if (!__all_sync(0xffffffffu, mbar_wait(&sfull[slot], sphase, args.status))) {
                        ok = false;
                        break;
                    }
                    const float* sl =
                        reinterpret_cast<const float*>(smem + S::kOffScale + slot * S::kSlotBytes);
                    fa = sl[row];
                    f = fa;
                    sbc = sl + kBM + half * 128;     // this half's 1x128 B scales
                }
                if (!__all_sync(0xffffffffu, mbar_wait(&tfull[b], tph, args.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * BN + half * 128;
                promote_block<kRowB, (kRowB ? FP8Q_PROMO_W_ROW : FP8Q_PROMO_W)>(
                    acc, taddr, f, fa, sbc, &tempty[b], lane);
                if (kSlots) {
                    // the slot was read with generic loads and is refilled by the
                    // async proxy (a bulk copy): order the reads before that write
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sempty[slot]);
                    if (++slot == kScaleSlots) { slot = 0; sphase ^= 1; }
                }
            }
            if (!ok) break;
            if (sg.rel >= 0) {
                // ------------------------------------- stream-K fix-up (per warp)
                // Partial layout: slot, this warp's slice, column group j (4
                // floats), row -- so a warp's 32 rows of one group are 512
                // contiguous bytes.
                constexpr int kSliceF4 = 32 * 32;          // float4s per 32 x 128 slice
                float4* mine = reinterpret_cast<float4*>(args.ws) +
                               (static_cast<size_t>(sg.slot) * S::kPromoWarps + pw) * kSliceF4 + lane;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    __stcg(mine + j * 32, make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x,
                                                      acc[2 * j + 1].y));
                if (!kRowB && args.sk_reduce) continue;     // k_sk_reduce finishes the tile
                __threadfence();
                __syncwarp();
                // pieces of this tile: one for each CTA c_lo .. c_hi
                const long long tile_start = static_cast<long long>(sg.rel) * Kb;
                const int c_lo = sched.cta_of(tile_start);
                const int c_hi = sched.cta_of(tile_start + Kb - 1);
                const bool clo_before = sched.lo(c_lo) < tile_start;
                int last = 0;
                if (lane == 0) {
                    const int pieces = c_hi - c_lo + 1;
                    int* cnt = args.counters + static_cast<size_t>(sg.rel) * S::kPromoWarps + pw;
                    __threadfence();
                    last = atomicAdd(cnt, 1) == pieces - 1;
                    if (last) {
                        *cnt = 0;                           // ready for the next call
                        __threadfence();
                    }
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (!last) continue;
                // the last piece to arrive sums every piece in K order
#pragma unroll
                for (int j = 0; j < 64; ++j) acc[j] = make_float2(0.0f, 0.0f);
#pragma unroll 1
                for (int c = c_lo; c <= c_hi; ++c) {
                    const float4* src = reinterpret_cast<const float4*>(args.ws) +
                                        (static_cast<size_t>(sched.slot_in_tile(c, c_lo, clo_before)) * S::kPromoWarps + pw) * kSliceF4 + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float4 v = __ldcg(src + j * 32);
                        acc[2 * j].x += v.x;
                        acc[2 * j].y += v.y;
                        acc[2 * j + 1].x += v.z;
                        acc[2 * j + 1].y += v.w;
                    }
                }
            }
            // ------------------------------------------------ epilogue
            store_tile_tma<kBf16Out>(acc, smem + S::kOffEpi + pw * S::kEpiWarpBytes, &tmC,
                                     tc.n0 + half * 128, tc.arow + quarter * 32, lane);
        }
        cp_async_wait<0>();                   // no scale copy still in flight
        if (lane == 0) bulk_wait_all();       // this warp's C stores have landed
        __syncwarp();
        tc_fence_before();
        cta_barrier(S::kThreads);
    }
}

// ------------------------------------------------- stream-K reduction
// The second kernel of a dense GEMM whose schedule cuts every tile (small
// output, long K: no whole-tile wave runs beside the fix-up, so the in-kernel
// sum by one CTA per tile -- ~600 KB of partials through 8 warps -- was half
// the kernel's time).  CTA (rel, pw) sums slice pw (32 rows x 128 columns) of
// stream-K tile rel over its pieces, in K order from zero -- the same
// additions in the same order as the in-kernel fix-up -- and writes it to C.
// A tile that one CTA's range covers whole was written by the GEMM itself.  Warp w takes the 16 columns of float4
// groups 4w .. 4w + 3, lane l row l of the slice; the partial layout is the
// GEMM's (slot, slice, float4 group, row), so each warp's reads are 512
// contiguous bytes per group and every thread has its 20-odd loads in flight
// at once (the in-kernel sum runs one CTA of 8 warps per tile).
template <int BN, bool kBf16Out>
__global__ void __launch_bounds__(256) k_sk_reduce(const float* __restrict__ ws, void* __restrict__ C,
                                                   int N, Sched sc) {
    constexpr int kPromoWarps = 4 * (BN / 128);
    constexpr int kSliceF4 = 32 * 32;
    const int rel = blockIdx.x, pw = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = sc.dp_tiles + rel;
    const int ntn = N / BN;
    const long long tile_start = static_cast<long long>(rel) * sc.Kb;
    const int c_lo = sc.cta_of(tile_start);
    const int c_hi = sc.cta_of(tile_start + sc.Kb - 1);
    if (c_lo == c_hi) return;                       // one piece: written whole
    const bool clo_before = sc.lo(c_lo) < tile_start;
    float4 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int c = c_lo; c <= c_hi; ++c) {
        const float4* src = reinterpret_cast<const float4*>(ws) +
                            (static_cast<size_t>(sc.slot_in_tile(c, c_lo, clo_before)) * kPromoWarps + pw) *
                                kSliceF4 + warp * 4 * 32 + lane;
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldcg(src + i * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[i].x += v[i].x;
            acc[i].y += v[i].y;
            acc[i].z += v[i].z;
            acc[i].w += v[i].w;
        }
    }
    const int half = pw >> 2, quarter = pw & 3;
    const size_t row = static_cast<size_t>(t / ntn) * kBM + quarter * 32 + lane;
    const int col = (t % ntn) * BN + half * 128 + warp * 16;
    if (kBf16Out) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w[2 * i] = pack_bf16x2(acc[i].x, acc[i].y);
            w[2 * i + 1] = pack_bf16x2(acc[i].z, acc[i].w);
        }
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(C) + row * N + col);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(C) + row * N + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = acc[i];
    }
}

}  // namespace fp8q
