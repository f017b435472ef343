// Online fine-grained E4M3 quantizers (memory-bound kernels).
//
// Grouping ("Six Reasons Deepseek Ai Is A Waste Of Time", para. 3, and the
// "fine-grained quantization" section of the codingmall FP8/DeepSeek-V3
// article): activations per 1x128 tile (one token, 128 channels), the same
// activations per 128x1 tile for the backward pass, weights per 128x128
// block.  Scaling ("online quantization" section; para. 1 of "Six
// Reasons..."): the group's largest magnitude maps onto 448, the largest
// finite E4M3 value, computed from the data at hand (no history).
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

// ------------------------------------------------------------------ 1x128
// Grid (K/128, ceil(M / (16 * kRows))), 256 threads.  A half-warp (16 lanes
// x 8 elements) covers one 1x128 tile; each thread handles kRows rows 16
// apart, issuing all kRows loads before reducing.  Scales land at s[g*M + m].
#ifndef FP8Q_Q1_ROWS
#define FP8Q_Q1_ROWS 4
#endif
#ifndef FP8Q_Q1_MINB
#define FP8Q_Q1_MINB 6
#endif
constexpr int kQ1RowsPerThread = FP8Q_Q1_ROWS;
constexpr int kQ1Rows = 16 * kQ1RowsPerThread;

template <typename T>
__global__ void __launch_bounds__(256, FP8Q_Q1_MINB) k_quant_1x128(const T* __restrict__ x, int64_t M,
                                                                  int64_t K, uint8_t* __restrict__ q,
                                                                  float* __restrict__ s) {
    constexpr int R = kQ1RowsPerThread;
    const int64_t g = blockIdx.x;
    const int team = threadIdx.x >> 4, tl = threadIdx.x & 15;
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
#pragma unroll
    for (int i = 0; i < R; ++i) {
        float a = amax8(v[i]);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        float sc, inv;
        group_scale(a, sc, inv);
        const int64_t r = r0 + 16 * i;
        if (r < M) {
            *reinterpret_cast<uint2*>(q + r * K + col) = quant8(v[i], inv);
            if (tl == 0) s[g * M + r] = sc;
        }
    }
}

// ---------------------------------------------------------------- 128x128
// Grid (K/128, N/128), kQwThreads threads, one block per CTA.  Thread (rr, tl)
// holds rows rr + (kQwThreads/16) i of the block, 8 columns each, in
// registers from the load to the store; block amax via warp shuffles and a
// shared-memory step.
#ifndef FP8Q_QW_THREADS
#define FP8Q_QW_THREADS 256
#endif
#ifndef FP8Q_QW_MINB
#define FP8Q_QW_MINB 1
#endif
constexpr int kQwThreads = FP8Q_QW_THREADS;

template <typename T>
__global__ void __launch_bounds__(kQwThreads, FP8Q_QW_MINB) k_quant_128x128(const T* __restrict__ w,
                                                                           int64_t N, int64_t K,
                                                                           uint8_t* __restrict__ q,
                                                                           float* __restrict__ s) {
    constexpr int kWarps = kQwThreads / 32, kStride = kQwThreads / 16, R = 128 / kStride;
    __shared__ float red[kWarps];
    const int64_t g = blockIdx.x, nb = blockIdx.y;
    const int64_t Kb = gridDim.x;
    const int tl = threadIdx.x & 15, rr = threadIdx.x >> 4;
    const int64_t col = g * 128 + tl * 8;
    float v[R][8];
#pragma unroll
    for (int i = 0; i < R; ++i) load8(w + (nb * 128 + rr + kStride * i) * K + col, v[i]);
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < R; ++i) a = fmaxf(a, amax8(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) a = fmaxf(a, red[i]);
    float sc, inv;
    group_scale(a, sc, inv);
    if (threadIdx.x == 0) s[nb * Kb + g] = sc;
#pragma unroll
    for (int i = 0; i < R; ++i)
        *reinterpret_cast<uint2*>(q + (nb * 128 + rr + kStride * i) * K + col) = quant8(v[i], inv);
}

// ------------------------------------------------------------------ 128x1
// Grid (C/64, T/128), 256 threads.  A 128-token x 64-channel tile is staged
// in shared memory with coalesced 16-byte loads; thread (c, tp) then reads
// 32 tokens of channel c (conflict-free: a warp spans 32 consecutive
// channels), the four partial maxima of a channel meet in shared memory, and
// the thread writes its 32 bytes of qT[c][t0 + 32 tp ..] (two 16-byte stores).
template <typename T>
__global__ void __launch_bounds__(256) k_quant_128x1(const T* __restrict__ x, int64_t Tn, int64_t C,
                                                     uint8_t* __restrict__ qT,
                                                     float* __restrict__ sT) {
    __shared__ __align__(16) T tile[128][64];
    __shared__ float red[4][64];
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int64_t tb = blockIdx.y, t0 = tb * 128;
    constexpr int kChunksPerRow = 64 * static_cast<int>(sizeof(T)) / 16;
    constexpr int kChunks = 128 * kChunksPerRow;
#pragma unroll
    for (int id = threadIdx.x; id < kChunks; id += 256) {
        const int row = id / kChunksPerRow, cc = id % kChunksPerRow;
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(x + (t0 + row) * C + c0) + cc);
        reinterpret_cast<uint4*>(&tile[row][0])[cc] = u;
    }
    __syncthreads();
    const int c = threadIdx.x & 63, tp = threadIdx.x >> 6;
    float v[32];
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        v[j] = to_f32(tile[tp * 32 + j][c]);
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
    uint4* dst = reinterpret_cast<uint4*>(qT + (c0 + c) * Tn + t0 + tp * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
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
    uint4* dst = reinterpret_cast<uint4*>(qT + (c0 + c) * Tn + t0 + tp * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
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
    // a warp's lanes take 32 consecutive k of the same n range
#pragma unroll
    for (int id = threadIdx.x; id < 128 * 8; id += 256) {
        const int k = id & 127, n0 = (id >> 7) * 16;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = static_cast<uint32_t>(tile[n0 + 4 * i][k]) |
                   (static_cast<uint32_t>(tile[n0 + 4 * i + 1][k]) << 8) |
                   (static_cast<uint32_t>(tile[n0 + 4 * i + 2][k]) << 16) |
                   (static_cast<uint32_t>(tile[n0 + 4 * i + 3][k]) << 24);
        *reinterpret_cast<uint4*>(qT + (kb * 128 + k) * N + nb * 128 + n0) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace fp8q
