// Online fine-grained E4M3 quantizers (memory-bound kernels).
//
// Grouping ("Six Reasons Deepseek Ai Is A Waste Of Time", para. 3, and the
// "fine-grained quantization" section of the codingmall FP8/DeepSeek-V3
// article): activations per 1x128 tile (one token, 128 channels), the same
// activations per 128x1 tile for the backward pass, weights per 128x128
// block.  Scaling ("online quantization" section; para. 1 of "Six
// Reasons..."): the group's largest magnitude maps onto 448, the largest
// finite E4M3 value, computed from the data at hand (no history).
//
// Contents: the shared scale rule and cast; k_quant_1x128 (direct loads,
// many short CTAs); k_swiglu_quant_1x128 and k_rmsnorm_quant_1x128 (the cast
// fused into the operator that produces the activation, woojincopolymer
// post, paras. 3-4); k_quant_128x128 and k_quant_128x1 (persistent, TMA
// stage ring); the backward-pass regrouping of stored 1x128 tiles into 128x1
// tiles and the FP8 weight transpose.
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"

namespace fp8q {

constexpr float kE4M3Max = 448.0f;

// s = fl32(amax / 448) is what gets stored; elements are multiplied by
// inv = fl32(448 / amax) before the cast.  amax == 0 stores 1 (the tile is
// all zeros and dequantizes to zeros); an overflowing inverse is clamped.
__device__ __forceinline__ void group_scale(float amax, float& s, float& inv) {
    if (amax == 0.0f) {
        s = 1.0f;
        inv = 1.0f;
        return;
    }
    s = __fdiv_rn(amax, kE4M3Max);
    inv = __fdiv_rn(kE4M3Max, amax);
    if (isinf(inv)) inv = FLT_MAX;
}

// Eight consecutive elements -> FP32, one 16-byte streaming load (BF16) or two (FP32).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float to_f32(__nv_bfloat16 h) { return __bfloat162float(h); }
__device__ __forceinline__ float to_f32(float f) { return f; }

__device__ __forceinline__ float amax8(const float (&v)[8]) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    return a;
}

// Eight values times inv, cast to E4M3, packed little-endian into 8 bytes.
__device__ __forceinline__ uint2 quant8(const float (&v)[8], float inv) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv));
        w[i] = lo;
    }
    uint2 r;
    r.x = w[0] | (w[1] << 16);
    r.y = w[2] | (w[3] << 16);
    return r;
}

// ------------------------------------------------------- streaming skeleton
// The three quantizers share one structure.  A persistent grid (a few CTAs
// per SM) walks its tiles blockIdx.x, +gridDim.x, ...  Thread 0 keeps up to
// kStages tiles in flight, each brought into a shared-memory stage by one TMA
// tensor copy that completes the stage's mbarrier.  Every thread copies its
// part of the tile into registers; one CTA barrier (which also publishes
// partial maxima and agrees on success) then frees the stage, which thread 0
// refills with the tile kStages further on while the current tile is reduced,
// cast and stored from registers.  HBM reads thus stay in flight across tile
// boundaries, with no per-tile launch or ramp.
template <int kStages, int kTileBytes>
struct TileRing {
    static constexpr int kBarOffset = kStages * kTileBytes;
    static constexpr int kSmemBytes = kBarOffset + kStages * 8 + 1024;   // + alignment slack

    uint8_t* base;
    uint64_t* full;

    __device__ void init(uint8_t* smem_raw) {
        base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
        full = reinterpret_cast<uint64_t*>(base + kBarOffset);
        if (threadIdx.x == 0) {
#pragma unroll 1
            for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
            fence_mbar_init();
        }
        __syncthreads();
    }
    __device__ const uint8_t* stage(int i) const { return base + i * kTileBytes; }
    __device__ void load(int i, const CUtensorMap* tm, int32_t x, int32_t y) {
        mbar_arrive_expect_tx(&full[i], kTileBytes);
        tma_load_2d(base + i * kTileBytes, tm, &full[i], x, y);
    }
    // After a failed wait: let the copies this CTA still has in flight land
    // (n_left = tiles issued but not consumed, starting at iteration it).
    __device__ void drain(int it, int n_left) {
#pragma unroll 1
        for (int j = 0; j < n_left; ++j) {
            const int k = it + j;
            mbar_drain(&full[k % kStages], (k / kStages) & 1, 10000000ull);
        }
    }
};

// Eight consecutive elements of a shared-memory tile -> FP32.
__device__ __forceinline__ void lds8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void lds8(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Tiles this CTA walks, and how many of them from iteration `it` on are
// already in flight.
__device__ __forceinline__ int my_tiles(int64_t tiles) {
    return tiles > blockIdx.x ? static_cast<int>((tiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
}

// ------------------------------------------------------------------ 1x128
// Grid (K/128, ceil(M / 64)), 256 threads, plain 16-byte loads straight into
// registers (at this grain, many short CTAs keep more loads in flight than a
// staged pipeline does).  A half-warp (16 lanes x 8 elements) covers one
// 1x128 tile; each thread handles kQ1RowsPerThread rows 16 apart, issuing all
// its loads before reducing.  The warp's 2 * kQ1RowsPerThread tile maxima are
// then gathered onto its first lanes, so one pass of the two correctly
// rounded divisions serves all of them, and the results are shuffled back.
// Scales land at s[g*M + m].
constexpr int kQ1RowsPerThread = 4;
constexpr int kQ1Rows = 16 * kQ1RowsPerThread;

template <typename T>
__global__ void __launch_bounds__(256, 4) k_quant_1x128(const T* __restrict__ x, int64_t M,
                                                        int64_t K, uint8_t* __restrict__ q,
                                                        float* __restrict__ s) {
    constexpr int R = kQ1RowsPerThread;
    const int64_t g = blockIdx.x;
    const int team = threadIdx.x >> 4, tl = threadIdx.x & 15;
    const int lane = threadIdx.x & 31, hw = lane >> 4;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kQ1Rows + team;
    const int64_t col = g * 128 + tl * 8;
    float v[R][8];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int64_t r = r0 + 16 * i;
        if (r < M) {
            load8(x + r * K + col, v[i]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
        }
    }
    // tile maxima: row i of half-warp h ends up on lane 2i + h
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        float a = amax8(v[i]);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const float t = __shfl_sync(0xffffffffu, a, (lane & 1) << 4);
        if ((lane >> 1) == i) mine = t;
    }
    float sc_l, inv_l;
    group_scale(mine, sc_l, inv_l);
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const float inv = __shfl_sync(0xffffffffu, inv_l, 2 * i + hw);
        const float sc = __shfl_sync(0xffffffffu, sc_l, 2 * i + hw);
        const int64_t r = r0 + 16 * i;
        if (r < M) {
            *reinterpret_cast<uint2*>(q + r * K + col) = quant8(v[i], inv);
            if (tl == 0) s[g * M + r] = sc;
        }
    }
}

// ------------------------------------------------- SwiGLU + 1x128 FP8 cast
// The down projection's FP8 input made in one pass (woojincopolymer post,
// para. 3: the FP8 cast fused into the operator that produces the
// activation; para. 4: the SwiGLU output, recomputed from its cached inputs,
// kept as 1x128 FP8 tiles).  h = silu(g) * u = g u / (1 + e^-g) in FP32, then
// the 1x128 rule of k_quant_1x128; h never reaches memory.  Same grid, lane
// layout and lane-parallel scales as k_quant_1x128, with kSwRowsPerThread
// rows per thread.  Gate and up rows are ld elements apart, so ld = 2I reads
// the two halves of one [M][2I] projection output in place.
constexpr int kSwRowsPerThread = 2;
constexpr int kSwRows = 16 * kSwRowsPerThread;

// silu(g) * u in FP32: expf (the accurate one, a few ulp) and IEEE division.
// For g below about -88, e^-g overflows and the result is a zero with the sign
// of -u, as the exact value rounds to.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
    const float e = expf(-g);
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, e)), u);
}

template <typename T>
__global__ void __launch_bounds__(256, 6) k_swiglu_quant_1x128(const T* __restrict__ gate,
                                                               const T* __restrict__ up,
                                                               int64_t M, int64_t I, int64_t ld,
                                                               uint8_t* __restrict__ q,
                                                               float* __restrict__ s) {
    constexpr int R = kSwRowsPerThread;
    const int64_t g = blockIdx.x;
    const int team = threadIdx.x >> 4, tl = threadIdx.x & 15;
    const int lane = threadIdx.x & 31, hw = lane >> 4;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kSwRows + team;
    const int64_t col = g * 128 + tl * 8;
    float v[R][8];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int64_t r = r0 + 16 * i;
        if (r < M) {
            float gv[8], uv[8];
            load8(gate + r * ld + col, gv);
            load8(up + r * ld + col, uv);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[i][j] = swiglu_f32(gv[j], uv[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
        }
    }
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        float a = amax8(v[i]);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const float t = __shfl_sync(0xffffffffu, a, (lane & 1) << 4);
        if ((lane >> 1) == i) mine = t;
    }
    float sc_l, inv_l;
    group_scale(mine, sc_l, inv_l);
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const float inv = __shfl_sync(0xffffffffu, inv_l, 2 * i + hw);
        const float sc = __shfl_sync(0xffffffffu, sc_l, 2 * i + hw);
        const int64_t r = r0 + 16 * i;
        if (r < M) {
            *reinterpret_cast<uint2*>(q + r * I + col) = quant8(v[i], inv);
            if (tl == 0) s[g * M + r] = sc;
        }
    }
}

// ----------------------------------------------- RMSNorm + 1x128 FP8 cast
// Layer normalization fused with the FP8 cast (woojincopolymer post, para.
// 3); DeepSeek-V3's normalization is RMSNorm: y = x w / sqrt(mean(x^2) + eps)
// per row.  A persistent grid of CTAs with K/16 threads each (rounded up to
// whole warps); a CTA walks rows blockIdx.x, +gridDim.x, ..., and each thread
// keeps 16 consecutive elements of its row in registers from the load to the
// store, with the next row's 16 elements already loading while the current
// row is reduced and stored (the weights are re-read per row, from L1).  The row's sum of squares goes through warp
// shuffles and one shared-memory step, r = 1/sqrt(mean + eps) is correctly
// rounded, y = (x r) w, and eight threads (128 elements) form a 1x128 tile
// with the scale rule and cast of k_quant_1x128.  FP32 throughout, so y
// differs from an exact evaluation by the summation's rounding (a few FP32
// ulp of the mean).
constexpr int kRnMaxK = 16384;       // 1024 threads x 16 elements

// Sixteen consecutive elements kept in their storage format until used.
template <typename T>
struct Raw16;

template <>
struct Raw16<__nv_bfloat16> {
    uint4 a, b;
    __device__ void zero() { a = b = make_uint4(0u, 0u, 0u, 0u); }
    __device__ void stream(const __nv_bfloat16* p) {
        a = __ldcs(reinterpret_cast<const uint4*>(p));
        b = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
    }
    __device__ void keep(const __nv_bfloat16* p) {
        a = __ldg(reinterpret_cast<const uint4*>(p));
        b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    }
    __device__ void to_f32(float (&v)[16]) const {
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

template <>
struct Raw16<float> {
    float4 a, b, c, d;
    __device__ void zero() { a = b = c = d = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ void stream(const float* p) {
        const float4* q = reinterpret_cast<const float4*>(p);
        a = __ldcs(q);
        b = __ldcs(q + 1);
        c = __ldcs(q + 2);
        d = __ldcs(q + 3);
    }
    __device__ void keep(const float* p) {
        const float4* q = reinterpret_cast<const float4*>(p);
        a = __ldg(q);
        b = __ldg(q + 1);
        c = __ldg(q + 2);
        d = __ldg(q + 3);
    }
    __device__ void to_f32(float (&v)[16]) const {
        const float4 f[4] = {a, b, c, d};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[4 * i] = f[i].x;
            v[4 * i + 1] = f[i].y;
            v[4 * i + 2] = f[i].z;
            v[4 * i + 3] = f[i].w;
        }
    }
};

template <typename T>
__global__ void __launch_bounds__(1024) k_rmsnorm_quant_1x128(const T* __restrict__ x,
                                                              const T* __restrict__ w, int64_t M,
                                                              int64_t K, float eps,
                                                              uint8_t* __restrict__ q,
                                                              float* __restrict__ s) {
    __shared__ float red[32];
    __shared__ float total;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t k0 = static_cast<int64_t>(t) * 16;
    const bool live = k0 < K;
    Raw16<T> cur, nxt;
    cur.zero();
    nxt.zero();
    int64_t m = blockIdx.x;
    if (live && m < M) cur.stream(x + m * K + k0);
#pragma unroll 1
    for (; m < M; m += gridDim.x) {
        const int64_t mn = m + gridDim.x;
        if (live && mn < M) nxt.stream(x + mn * K + k0);
        float v[16];
        cur.to_f32(v);
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) ss = __fmaf_rn(v[i], v[i], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (warp == 0) {
            float a = lane < nwarps ? red[lane] : 0.0f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) total = a;
        }
        __syncthreads();
        const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(total, static_cast<float>(K)), eps));
        float wv[16];
        {
            Raw16<T> wr;                 // the weights, re-read per row from L1
            wr.zero();
            if (live) wr.keep(w + k0);
            wr.to_f32(wv);
        }
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = __fmul_rn(__fmul_rn(v[i], r), wv[i]);
            a = fmaxf(a, fabsf(v[i]));
        }
        // a 1x128 tile is eight consecutive threads (lanes 8j .. 8j+7 of a warp)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        float sc, inv;
        group_scale(a, sc, inv);
        if (live) {
            float lo[8], hi[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lo[i] = v[i];
                hi[i] = v[8 + i];
            }
            const uint2 p0 = quant8(lo, inv), p1 = quant8(hi, inv);
            *reinterpret_cast<uint4*>(q + m * K + k0) = make_uint4(p0.x, p0.y, p1.x, p1.y);
            if ((t & 7) == 0) s[(k0 / 128) * M + m] = sc;
        }
        cur = nxt;
    }
}

// ---------------------------------------------------------------- 128x128
// Tile = one 128x128 block of w[N][K]; thread (rr, tl) holds rows rr + 16 i
// (i < 8), 8 columns each; block amax via warp shuffles and one shared-memory
// step (double-buffered by iteration parity, so one CTA barrier per tile).
template <typename T>
struct QwCfg {
    static constexpr int kThreads = 256;
    static constexpr int kTileBytes = 128 * 128 * static_cast<int>(sizeof(T));
    static constexpr int kStages = sizeof(T) == 2 ? 3 : 2;
    static constexpr int kCtasPerSm = sizeof(T) == 2 ? 2 : 1;
    using Ring = TileRing<kStages, kTileBytes>;
    static constexpr int kSmemBytes = Ring::kSmemBytes;
};

template <typename T>
__global__ void __launch_bounds__(256, QwCfg<T>::kCtasPerSm)
    k_quant_128x128(const __grid_constant__ CUtensorMap tm, int64_t N, int64_t K,
                    uint8_t* __restrict__ q, float* __restrict__ s, int* status) {
    using C = QwCfg<T>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ float red[2][8];
    typename C::Ring ring;
    ring.init(smem_raw);
    const int64_t Kb = K / 128;
    const int64_t tiles = Kb * (N / 128);
    const int n = my_tiles(tiles);
    const int rr = threadIdx.x >> 4, tl = threadIdx.x & 15, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int j = 0; j < C::kStages && j < n; ++j) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(j) * gridDim.x;
            ring.load(j, &tm, static_cast<int32_t>((t % Kb) * 128), static_cast<int32_t>((t / Kb) * 128));
        }
    }
#pragma unroll 1
    for (int it = 0; it < n; ++it) {
        const int st = it % C::kStages;
        const int64_t t = blockIdx.x + static_cast<int64_t>(it) * gridDim.x;
        const int64_t g = t % Kb, nb = t / Kb;
        float v[8][8];
        const bool got = mbar_wait(&ring.full[st], (it / C::kStages) & 1, status);
        if (got) {
            const T* tile = reinterpret_cast<const T*>(ring.stage(st));
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lds8(tile + (rr + 16 * i) * 128 + tl * 8, v[i]);
                a = fmaxf(a, amax8(v[i]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            if ((threadIdx.x & 31) == 0) red[it & 1][warp] = a;
        }
        if (!__syncthreads_and(got)) {
            if (threadIdx.x == 0) ring.drain(it, min(n - it, C::kStages));
            return;
        }
        if (threadIdx.x == 0 && it + C::kStages < n) {
            const int64_t tn = t + static_cast<int64_t>(C::kStages) * gridDim.x;
            fence_proxy_async_smem();
            ring.load(st, &tm, static_cast<int32_t>((tn % Kb) * 128), static_cast<int32_t>((tn / Kb) * 128));
        }
        float a = red[it & 1][0];
#pragma unroll
        for (int i = 1; i < 8; ++i) a = fmaxf(a, red[it & 1][i]);
        float sc, inv;
        group_scale(a, sc, inv);
        if (threadIdx.x == 0) s[nb * Kb + g] = sc;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint2*>(q + (nb * 128 + rr + 16 * i) * K + g * 128 + tl * 8) =
                quant8(v[i], inv);
    }
}

// ------------------------------------------------------------------ 128x1
// Tile = 128 tokens x 64 channels of x[T][C]; thread (c, tp) reads kTok
// tokens of channel c from shared memory (conflict-free: a warp spans 32
// consecutive channels of one token), the kParts partial maxima of a channel
// meet in shared memory (double-buffered by iteration parity), and the
// thread puts its kTok bytes of qT[c][t0 + kTok tp ..] into a staging tile of
// 64 rows x 128 bytes laid out with the 128-byte swizzle (16-byte chunk j of
// row r at j ^ (r % 8)).  One TMA store per tile writes the staged bytes:
// per-thread stores of 32 bytes to 64 different rows of qT kept the
// load-store unit's queue full (its throttle was the largest stall after the
// loads).  The store of tile it is issued by thread 0 just after the CTA
// barrier of tile it + 1 (which every thread reaches after staging tile it);
// the staging tiles alternate, and before the barrier of tile it thread 0
// waits until the store of tile it - 2, which read the same staging tile,
// has read it.
template <typename T>
struct QtCfg {
    static constexpr int kThreads = 256;
    static constexpr int kParts = kThreads / 64;           // token ranges per channel
    static constexpr int kTok = 128 / kParts;              // tokens per thread
    static constexpr int kTileBytes = 128 * 64 * static_cast<int>(sizeof(T));
    static constexpr int kStages = sizeof(T) == 2 ? 3 : 2;
    static constexpr int kCtasPerSm = sizeof(T) == 2 ? 3 : 2;
    using Ring = TileRing<kStages, kTileBytes>;
    static constexpr int kOutBytes = 64 * 128;              // one staged tile of qT
    static constexpr int kOffOut = (Ring::kBarOffset + kStages * 8 + 1023) / 1024 * 1024;
    static constexpr int kSmemBytes = kOffOut + 2 * kOutBytes + 1024;   // + alignment slack
};

template <typename T>
__global__ void __launch_bounds__(QtCfg<T>::kThreads, QtCfg<T>::kCtasPerSm)
    k_quant_128x1(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmq,
                  int64_t Tn, int64_t C, float* __restrict__ sT, int* status) {
    using Cf = QtCfg<T>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ float red[2][Cf::kParts][64];
    typename Cf::Ring ring;
    ring.init(smem_raw);
    uint8_t* out = ring.base + Cf::kOffOut;        // two staged tiles of qT
    const int64_t CB = C / 64;
    const int64_t tiles = CB * (Tn / 128);
    const int n = my_tiles(tiles);
    const int c = threadIdx.x & 63, tp = threadIdx.x >> 6;
    if (threadIdx.x == 0) {
#pragma unroll 1
        for (int j = 0; j < Cf::kStages && j < n; ++j) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(j) * gridDim.x;
            ring.load(j, &tm, static_cast<int32_t>((t % CB) * 64), static_cast<int32_t>((t / CB) * 128));
        }
    }
    int32_t prev_x = 0, prev_y = 0;                // coordinates of the staged, unstored tile
#pragma unroll 1
    for (int it = 0; it < n; ++it) {
        const int st = it % Cf::kStages;
        const int64_t t = blockIdx.x + static_cast<int64_t>(it) * gridDim.x;
        const int64_t c0 = (t % CB) * 64, tb = t / CB, t0 = tb * 128;
        float v[Cf::kTok];
        const bool got = mbar_wait(&ring.full[st], (it / Cf::kStages) & 1, status);
        if (got) {
            const T* tile = reinterpret_cast<const T*>(ring.stage(st));
            float a = 0.0f;
#pragma unroll
            for (int j = 0; j < Cf::kTok; ++j) {
                v[j] = to_f32(tile[(tp * Cf::kTok + j) * 64 + c]);
                a = fmaxf(a, fabsf(v[j]));
            }
            red[it & 1][tp][c] = a;
        }
        // the staging tile about to be written was last read by the store of
        // tile it - 2: that store must have read it before anyone writes
        if (threadIdx.x == 0) bulk_wait_read_pending<0>();
        if (!__syncthreads_and(got)) {
            if (threadIdx.x == 0) {
                ring.drain(it, min(n - it, Cf::kStages));
                bulk_wait_all();
            }
            return;
        }
        if (threadIdx.x == 0) {
            if (it > 0) {
                tma_store_2d(&tmq, out + ((it - 1) & 1) * Cf::kOutBytes, prev_x, prev_y);
                bulk_commit_group();
            }
            if (it + Cf::kStages < n) {
                const int64_t tn = t + static_cast<int64_t>(Cf::kStages) * gridDim.x;
                fence_proxy_async_smem();
                ring.load(st, &tm, static_cast<int32_t>((tn % CB) * 64), static_cast<int32_t>((tn / CB) * 128));
            }
        }
        prev_x = static_cast<int32_t>(t0);
        prev_y = static_cast<int32_t>(c0);
        float a = red[it & 1][0][c];
#pragma unroll
        for (int p = 1; p < Cf::kParts; ++p) a = fmaxf(a, red[it & 1][p][c]);
        float sc, inv;
        group_scale(a, sc, inv);
        if (tp == 0) sT[tb * C + c0 + c] = sc;
        uint32_t w[Cf::kTok / 4];
#pragma unroll
        for (int i = 0; i < Cf::kTok / 4; ++i) {
            const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[4 * i], inv), __fmul_rn(v[4 * i + 1], inv));
            const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[4 * i + 2], inv), __fmul_rn(v[4 * i + 3], inv));
            w[i] = lo | (hi << 16);
        }
        uint8_t* row = out + (it & 1) * Cf::kOutBytes + c * 128;
#pragma unroll
        for (int i = 0; i < Cf::kTok / 16; ++i) {
            const int chunk = tp * (Cf::kTok / 16) + i;           // 16-byte chunk of the row
            *reinterpret_cast<uint4*>(row + ((chunk ^ (c & 7)) << 4)) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
        fence_proxy_async_smem();                  // staged bytes -> the store's async read
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (n > 0) {
            tma_store_2d(&tmq, out + ((n - 1) & 1) * Cf::kOutBytes, prev_x, prev_y);
            bulk_commit_group();
        }
        bulk_wait_all();
    }
}

// ------------------------------------------------ 1x128 tiles -> 128x1 tiles
// Backward regrouping of the stored forward activations ("Six Reasons...",
// para. 3): q[T][C] with 1x128 scales s[C/128][T] is dequantized -- the E4M3
// decode is exact, times the tile scale in one correctly rounded FP32
// multiplication -- and quantized again per 128 tokens of one channel,
// written transposed (qT[C][T], sT[T/128][C]) like k_quant_128x1.
// Grid (C/64, T/128), 256 threads; a 128-token x 64-channel tile of bytes and
// the 128 token scales of its channel group are staged in shared memory.
__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(h));
}

__global__ void __launch_bounds__(256) k_retile_1x128_to_128x1(const uint8_t* __restrict__ q,
                                                               const float* __restrict__ s,
                                                               int64_t Tn, int64_t C,
                                                               uint8_t* __restrict__ qT,
                                                               float* __restrict__ sT) {
    __shared__ __align__(16) uint8_t tile[128][64];
    __shared__ float tscale[128];
    __shared__ float red[4][64];
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int64_t tb = blockIdx.y, t0 = tb * 128;
    const int64_t g = c0 / 128;                       // 1x128 scale group of these channels
#pragma unroll
    for (int id = threadIdx.x; id < 128 * 4; id += 256) {
        const int row = id >> 2, cc = id & 3;
        reinterpret_cast<uint4*>(&tile[row][0])[cc] =
            __ldcs(reinterpret_cast<const uint4*>(q + (t0 + row) * C + c0) + cc);
    }
    if (threadIdx.x < 128) tscale[threadIdx.x] = s[g * Tn + t0 + threadIdx.x];
    __syncthreads();
    const int c = threadIdx.x & 63, tp = threadIdx.x >> 6;
    float v[32];
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int t = tp * 32 + j;
        v[j] = __fmul_rn(e4m3_to_f32(tile[t][c]), tscale[t]);
        a = fmaxf(a, fabsf(v[j]));
    }
    red[tp][c] = a;
    __syncthreads();
    a = fmaxf(fmaxf(red[0][c], red[1][c]), fmaxf(red[2][c], red[3][c]));
    float sc, inv;
    group_scale(a, sc, inv);
    if (tp == 0) sT[tb * C + c0 + c] = sc;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(v[4 * i], inv), __fmul_rn(v[4 * i + 1], inv));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(v[4 * i + 2], inv), __fmul_rn(v[4 * i + 3], inv));
        w[i] = lo | (hi << 16);
    }
    // The input tile is free (every thread passed the barrier after its last
    // read): stage the 64 channel rows x 128 token bytes there, 16-byte chunk
    // j of row r at j ^ (r % 8), then write whole 128-byte rows of qT (a warp
    // covers four rows) instead of 32 bytes into each of 64 rows per warp.
    uint8_t* stg = &tile[0][0];
#pragma unroll
    for (int i = 0; i < 2; ++i)
        *reinterpret_cast<uint4*>(stg + c * 128 + (((tp * 2 + i) ^ (c & 7)) << 4)) =
            make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    __syncthreads();
#pragma unroll
    for (int id = threadIdx.x; id < 64 * 8; id += 256) {
        const int r = id >> 3, j = id & 7;
        *reinterpret_cast<uint4*>(qT + (c0 + r) * Tn + t0 + j * 16) =
            *reinterpret_cast<const uint4*>(stg + r * 128 + ((j ^ (r & 7)) << 4));
    }
}

// ------------------------------------------------- FP8 weight transpose
// q[N][K] (128x128 block scales s[N/128][K/128]) -> qT[K][N] with
// sT[K/128][N/128]: the transposed weight of the data-gradient GEMM
// dX = dY W, whose blocks and scales are the forward weight's, transposed.
// Grid (K/128, N/128), 256 threads, one 128 x 128 byte block per CTA.
__global__ void __launch_bounds__(256) k_transpose_128x128(const uint8_t* __restrict__ q,
                                                           const float* __restrict__ s, int64_t N,
                                                           int64_t K, uint8_t* __restrict__ qT,
                                                           float* __restrict__ sT) {
    __shared__ __align__(16) uint8_t tile[128][128 + 16];
    const int64_t kb = blockIdx.x, nb = blockIdx.y;
#pragma unroll
    for (int id = threadIdx.x; id < 128 * 8; id += 256) {
        const int row = id >> 3, cc = id & 7;
        *reinterpret_cast<uint4*>(&tile[row][cc * 16]) =
            __ldcs(reinterpret_cast<const uint4*>(q + (nb * 128 + row) * K + kb * 128) + cc);
    }
    if (threadIdx.x == 0) sT[kb * (N / 128) + nb] = s[nb * (K / 128) + kb];
    __syncthreads();
    // output row k (a column of the block) gets 16 consecutive n per task;
    // a warp's lanes take 32 consecutive k of the same n range.  The 16-byte
    // pieces are put back into the tile (row k, stride 144 bytes: a warp's
    // stores spread over all banks) once every thread has read its columns,
    // and leave as whole 128-byte rows of qT (a warp covers four rows).
    uint4 wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int id = threadIdx.x + u * 256;
        const int k = id & 127, n0 = (id >> 7) * 16;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = static_cast<uint32_t>(tile[n0 + 4 * i][k]) |
                   (static_cast<uint32_t>(tile[n0 + 4 * i + 1][k]) << 8) |
                   (static_cast<uint32_t>(tile[n0 + 4 * i + 2][k]) << 16) |
                   (static_cast<uint32_t>(tile[n0 + 4 * i + 3][k]) << 24);
        wv[u] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int id = threadIdx.x + u * 256;
        const int k = id & 127, n0 = (id >> 7) * 16;
        *reinterpret_cast<uint4*>(&tile[k][n0]) = wv[u];
    }
    __syncthreads();
#pragma unroll
    for (int id = threadIdx.x; id < 128 * 8; id += 256) {
        const int k = id >> 3, j = id & 7;
        *reinterpret_cast<uint4*>(qT + (kb * 128 + k) * N + nb * 128 + j * 16) =
            *reinterpret_cast<const uint4*>(&tile[k][j * 16]);
    }
}

}  // namespace fp8q
