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
//     swizzle), plus bulk copies of the block's activation scales (and, for
//     1x128-scaled B, the B scales) into a separate ring of scale slots;
//   * MMA warp (1 thread): 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) per
//     128-K block into one of two TMEM buffers (128 lanes x BN FP32
//     columns), a fresh accumulation per block; tcgen05.commit releases the
//     smem stage and signals the promotion warps;
//   * BN/128 promotion warpgroups: tcgen05.ld the partial in 16-column
//     chunks (8 for row-scaled B), the next chunk's load in flight while the
//     current one is scaled, release the TMEM buffer once the last chunk has
//     arrived, and accumulate P * (sA * sB) into 128 FP32 registers per thread
//     with packed FP32 FMAs; after the last block, write C.
// The MMA of block i+1 (other TMEM buffer) overlaps the promotion of block i.
// Persistent: one CTA per SM walks tiles blockIdx.x, +gridDim.x, ...; the
// rings carry over from one tile to the next.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fp8q {

constexpr int kBM = 128;          // rows of A per tile (TMEM lanes)
constexpr int kBK = 128;          // K per block = scale-group width = one 128-byte swizzle row
constexpr int kScaleSlots = 8;
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
template <int BN>
struct GemmShape {
    static constexpr int kHalves = BN / 128;             // 128-column halves of the tile
    static constexpr int kPromoWarps = 4 * kHalves;
    static constexpr int kProducerWarp = 0;
    static constexpr int kMmaWarp = FP8Q_MMA_WARP;
    static constexpr int kFirstPromoWarp = 4;
    static constexpr int kThreads = 128 * (1 + kHalves);
    static constexpr bool kRealloc = kHalves > 1;
    static constexpr int kCtrlRegs = 56;
    static constexpr int kPromoRegs = 224;
    static_assert(!kRealloc || 128 * kCtrlRegs + 128 * kHalves * kPromoRegs <= kThreads * 168,
                  "register split exceeds the launch allocation");
    static_assert(kMmaWarp > 0 && kMmaWarp < 4, "MMA warp must be a control warp");
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kSaBytes = kBM * 4;
    static constexpr int kSbBytes = BN * 4;
    static constexpr int kSlotBytes = kSaBytes + kSbBytes;
    static constexpr int kOffScale = kStages * kStageBytes;
    static constexpr int kOffBars = kOffScale + kScaleSlots * kSlotBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * kScaleSlots + 5;
    static constexpr int kOffMisc = kOffBars + kNumBars * 8;
    static constexpr int kOffGroups = kOffMisc + 16;
    static constexpr int kSmemBytes = kOffGroups + 2 * (kMaxGroups + 1) * 4 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kTmemCols <= 512, "TMEM budget");
};

struct GemmArgs {
    const float* sA;        // [K/128][M_total]
    const float* sB;        // block: [G][N/128][K/128]; row: [K/128][N]
    void* C;                // [M_total][N]
    const int* m_offsets;   // grouped: [G+1] device array; dense: nullptr
    int M_total, N, K, G;
    int* status;
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

template <int BN, bool kRowB, bool kBf16Out>
__global__ void __launch_bounds__(GemmShape<BN>::kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const GemmArgs args) {
    using S = GemmShape<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBars);
    uint64_t* full = bars;
    uint64_t* empty = full + S::kStages;
    uint64_t* sfull = empty + S::kStages;
    uint64_t* sempty = sfull + kScaleSlots;
    uint64_t* tfull = sempty + kScaleSlots;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
    int* gtile = reinterpret_cast<int*>(smem + S::kOffGroups);
    int* grow = gtile + (kMaxGroups + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = args.N, Kb = args.K / kBK, ntn = N / BN;
    const bool grouped = args.m_offsets != nullptr;

    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int i = 0; i < S::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
#pragma unroll 1
        for (int i = 0; i < kScaleSlots; ++i) {
            mbar_init(&sfull[i], 1);
            mbar_init(&sempty[i], S::kPromoWarps);
        }
        mbar_init(&tfull[0], 1);
        mbar_init(&tfull[1], 1);
        mbar_init(&tempty[0], S::kPromoWarps);
        mbar_init(&tempty[1], S::kPromoWarps);
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
    }
    if (warp == S::kMmaWarp) {
        tmem_alloc(&misc[0], S::kTmemCols);
        tmem_relinquish();
    }
    if (warp == S::kProducerWarp && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    const int num_tiles = static_cast<int>(misc[1]);

    if (warp < S::kFirstPromoWarp) {
        if (S::kRealloc) setmaxnreg_dec<S::kCtrlRegs>();
        if (warp == S::kProducerWarp && lane == 0) {
            // -------------------------------------------------- producer
            uint32_t stage = 0, phase = 0, slot = 0, sphase = 0;
            bool ok = true;
#pragma unroll 1
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
                const TileCoord tc = decode_tile<BN>(t, grouped, N, args.G, gtile, grow);
#pragma unroll 1
                for (int kb = 0; kb < Kb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, args.status)) { ok = false; break; }
                    uint8_t* sa = smem + stage * S::kStageBytes;
                    mbar_arrive_expect_tx(&full[stage], S::kStageBytes);
                    tma_load_2d(sa, &tmA, &full[stage], kb * kBK, tc.arow);
                    tma_load_2d(sa + S::kABytes, &tmB, &full[stage], kb * kBK, tc.brow);
                    if (++stage == S::kStages) { stage = 0; phase ^= 1; }

                    if (kRowB) {
                        // weight-gradient form: both operands' 1x128 scales of
                        // this block go through a shared-memory slot
                        if (!mbar_wait(&sempty[slot], sphase ^ 1, args.status)) { ok = false; break; }
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
#pragma unroll 1
            for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
#pragma unroll 1
                for (int kb = 0; kb < Kb; ++kb, ++it) {
                    const uint32_t b = it & 1, tph = (it >> 1) & 1;
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
    } else {
        // ----------------------------------------------------- promotion
        if (S::kRealloc) setmaxnreg_inc<S::kPromoRegs>();
        const int half = (warp - S::kFirstPromoWarp) >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;       // TMEM lane = row of the tile
        uint32_t it = 0, slot = 0, sphase = 0;
        bool ok = true;
        float2 acc[64];                            // columns 2j, 2j+1 of this thread's half
#pragma unroll 1
        for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
            const TileCoord tc = decode_tile<BN>(t, grouped, N, args.G, gtile, grow);
            // Block-scaled B: this thread's row scale and the 128x128 block scale
            // are read straight from global memory (coalesced), one block ahead.
            const float* sa_row = args.sA + tc.arow + row;
            const float* sb_blk =
                args.sB + (static_cast<size_t>(tc.e) * (N / 128) + (tc.n0 / 128 + half)) * Kb;
            float fa_next = 0.0f, fb_next = 0.0f;
            if (!kRowB) {
                fa_next = __ldg(sa_row);
                fb_next = __ldg(sb_blk);
            }
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = make_float2(0.0f, 0.0f);
#pragma unroll 1
            for (int kb = 0; kb < Kb; ++kb, ++it) {
                const uint32_t b = it & 1, tph = (it >> 1) & 1;
                float fa, f;
                const float* sbc = nullptr;
                if (!kRowB) {
                    fa = fa_next;
                    f = fa_next * fb_next;
                    if (kb + 1 < Kb) {
                        fa_next = __ldg(sa_row + static_cast<size_t>(kb + 1) * args.M_total);
                        fb_next = __ldg(sb_blk + kb + 1);
                    }
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
                if (!kRowB) {
                    // Sixteen-column chunks, the next chunk's load in flight while
                    // the current one is scaled; the TMEM buffer goes back to the
                    // MMA warp as soon as the last chunk has arrived.
                    uint32_t r0[16], r1[16];
                    tmem_ld_chunk(taddr, r0);
                    tmem_ld_wait(r0);
#pragma unroll
                    for (int c = 0; c < 8; c += 2) {
                        tmem_ld_chunk(taddr + (c + 1) * 16, r1);
                        promote_chunk<false>(acc + c * 8, r0, f, fa, nullptr);
                        tmem_ld_wait(r1);
                        if (c + 2 < 8) {
                            tmem_ld_chunk(taddr + (c + 2) * 16, r0);
                        } else {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[b]);
                        }
                        promote_chunk<false>(acc + (c + 1) * 8, r1, f, fa, nullptr);
                        if (c + 2 < 8) tmem_ld_wait(r0);
                    }
                } else {
                    // Eight-column chunks, the next chunk's load in flight while
                    // the current one is scaled.
                    uint32_t r0[8], r1[8];
                    tmem_ld_chunk(taddr, r0);
                    tmem_ld_wait(r0);
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        tmem_ld_chunk(taddr + (c + 1) * 8, r1);
                        promote_chunk<true>(acc + c * 4, r0, f, fa, sbc + c * 8);
                        tmem_ld_wait(r1);
                        if (c + 2 < 16) {
                            tmem_ld_chunk(taddr + (c + 2) * 8, r0);
                        } else {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[b]);
                        }
                        promote_chunk<true>(acc + (c + 1) * 4, r1, f, fa, sbc + (c + 1) * 8);
                        if (c + 2 < 16) tmem_ld_wait(r0);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sempty[slot]);
                    if (++slot == kScaleSlots) { slot = 0; sphase ^= 1; }
                }
            }
            if (!ok) break;
            // ------------------------------------------------ epilogue
            const size_t crow = static_cast<size_t>(tc.arow + row);
            const int ccol = tc.n0 + half * 128;
            if (kBf16Out) {
                __nv_bfloat16* cp = reinterpret_cast<__nv_bfloat16*>(args.C) + crow * N + ccol;
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    uint4 v;
                    v.x = pack_bf16x2(acc[j].x, acc[j].y);
                    v.y = pack_bf16x2(acc[j + 1].x, acc[j + 1].y);
                    v.z = pack_bf16x2(acc[j + 2].x, acc[j + 2].y);
                    v.w = pack_bf16x2(acc[j + 3].x, acc[j + 3].y);
                    *reinterpret_cast<uint4*>(cp + 2 * j) = v;
                }
            } else {
                float* cp = reinterpret_cast<float*>(args.C) + crow * N + ccol;
#pragma unroll
                for (int j = 0; j < 64; j += 2)
                    *reinterpret_cast<float4*>(cp + 2 * j) =
                        make_float4(acc[j].x, acc[j].y, acc[j + 1].x, acc[j + 1].y);
            }
        }
        tc_fence_before();
        cta_barrier(S::kThreads);
    }
}

}  // namespace fp8q
