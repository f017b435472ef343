// Expert-parallel MoE data path around the grouped GEMM: FP8 dispatch and
// BF16 combine ("Six Reasons Deepseek Ai Is A Waste Of Time", para. 4: the
// activations are quantized to FP8 before they are dispatched to the
// experts' up projection; the combine stays in BF16).
//
// A rank's tokens, quantized per 1x128 tile, are sent as packed rows: the
// row's E4M3 bytes followed by its H/128 FP32 scales (padded to 16 bytes),
// one row per (token, chosen expert), ordered by expert and, within an
// expert, by (token, slot).  Experts are numbered rank-major (rank d owns
// experts d*E_local .. (d+1)*E_local - 1), so this order is also grouped by
// destination rank.  A receiving rank gets, from each source rank in turn,
// that rank's rows for each of its local experts; it lays them out as the
// grouped GEMM's A operand (each expert's rows contiguous, padded to a
// multiple of 128 with zero rows), runs the grouped GEMM, and sends each
// BF16 result row back in the order it arrived.  The source rank combines a
// token's k results with its gate weights in FP32 and writes BF16.
//
// Kernels: k_ep_route (expert counts and each row's position in the send
// order, deterministic), k_ep_pack, k_ep_unpack, k_ep_zero_pad, k_ep_gather,
// k_ep_combine.  The exchange between ranks (an all-to-all of the packed
// rows and of the BF16 results) is the caller's collective.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fp8q {

constexpr int kEpMaxExperts = 256;
constexpr int kEpRouteThreads = 1024;
constexpr int kErrBadRouting = 7;

// Packed row of the dispatch: H bytes of E4M3, then H/128 FP32 scales,
// padded so that every row starts on a 16-byte boundary.
__host__ __device__ constexpr int64_t ep_row_bytes(int64_t H) {
    return H + ((H / 128) * 4 + 15) / 16 * 16;
}

// One CTA.  Warp w takes a contiguous share of the n = T*k entries (ids, in
// row-major (token, slot) order).  Pass 1: per-warp expert histograms.
// Pass 2: expert totals, their exclusive prefix (the start of each expert's
// rows in the send order), and each warp's start within each expert.
// Pass 3: every warp walks its share in order, 32 entries at a time; lanes
// with the same expert are ranked by lane (match.any + popc), so an entry's
// position is its expert's start + the number of earlier entries of that
// expert.  Any id outside [0, E) records kErrBadRouting and nothing is written.
__global__ void __launch_bounds__(kEpRouteThreads, 1)
    k_ep_route(const int32_t* __restrict__ ids, int64_t n, int E, int32_t* __restrict__ counts,
               int32_t* __restrict__ pos, int* status) {
    __shared__ int hist[kEpRouteThreads / 32][kEpMaxExperts];
    __shared__ int start[kEpMaxExperts];
    __shared__ int bad;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kW = kEpRouteThreads / 32;
    for (int i = threadIdx.x; i < kW * kEpMaxExperts; i += blockDim.x) (&hist[0][0])[i] = 0;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    const int64_t lo = n * warp / kW, hi = n * (warp + 1) / kW;
    for (int64_t i = lo + lane; i < hi; i += 32) {
        const int e = ids[i];
        if (e < 0 || e >= E) bad = 1;
        else atomicAdd(&hist[warp][e], 1);
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) atomicCAS(status, kOk, kErrBadRouting);
        return;
    }
    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        int run = 0;
        for (int w = 0; w < kW; ++w) {
            const int c = hist[w][e];
            hist[w][e] = run;             // this warp's start within expert e
            run += c;
        }
        start[e] = run;                   // total for now
        counts[e] = run;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int e = 0; e < E; ++e) {
            const int c = start[e];
            start[e] = run;
            run += c;
        }
    }
    __syncthreads();
    for (int64_t c0 = lo; c0 < hi; c0 += 32) {
        const int64_t i = c0 + lane;
        const bool live = i < hi;
        const int e = live ? ids[i] : -1 - lane;          // dead lanes match nobody
        const unsigned same = __match_any_sync(0xffffffffu, e);
        if (live) {
            const int rank = __popc(same & ((1u << lane) - 1u));
            pos[i] = start[e] + hist[warp][e] + rank;
        }
        __syncwarp();
        if (live && lane == 31 - __clz(same)) hist[warp][e] += __popc(same);
        __syncwarp();
    }
}

// One warp per (token, slot) entry: token t's E4M3 row and its scales
// (s[g][t], MN-major) go to packed row pos[entry] of `send`.
__global__ void __launch_bounds__(256) k_ep_pack(const uint8_t* __restrict__ q,
                                                 const float* __restrict__ s,
                                                 const int32_t* __restrict__ pos, int64_t T,
                                                 int k, int64_t H, uint8_t* __restrict__ send) {
    const int64_t entry = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (entry >= T * k) return;
    const int64_t t = entry / k;
    const int64_t rb = ep_row_bytes(H);
    uint8_t* dst = send + static_cast<int64_t>(pos[entry]) * rb;
    const uint4* src = reinterpret_cast<const uint4*>(q + t * H);
    for (int64_t c = lane; c < H / 16; c += 32) reinterpret_cast<uint4*>(dst)[c] = __ldg(src + c);
    float* ds = reinterpret_cast<float*>(dst + H);
    for (int64_t g = lane; g < H / 128; g += 32) ds[g] = __ldg(s + g * T + t);
}

// Block b of the receive order (source w, local expert e, b = w*El + e)
// holding packed row i: the largest b with src_off[b] <= i.
__device__ __forceinline__ int ep_block_of(const int64_t* src_off, int nb, int64_t i) {
    int lo = 0, hi = nb - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (src_off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// One warp per received packed row i: its bytes go to row
// dest = dest_base[b] + (i - src_off[b]) of A8 [Mp][H], its scales to
// sA[g][dest] (MN-major, the grouped GEMM's layout).
__global__ void __launch_bounds__(256) k_ep_unpack(const uint8_t* __restrict__ recv, int64_t R,
                                                   int64_t H, const int64_t* __restrict__ src_off,
                                                   const int64_t* __restrict__ dest_base, int nb,
                                                   uint8_t* __restrict__ A8, float* __restrict__ sA,
                                                   int64_t Mp, int* status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= R) return;
    const int b = ep_block_of(src_off, nb, i);
    const int64_t dest = dest_base[b] + (i - src_off[b]);
    if (dest < 0 || dest >= Mp) {                 // inconsistent layout tables: write nothing
        if (lane == 0) atomicCAS(status, kOk, kErrBadRouting);
        return;
    }
    const int64_t rb = ep_row_bytes(H);
    const uint8_t* src = recv + i * rb;
    uint4* dst = reinterpret_cast<uint4*>(A8 + dest * H);
    for (int64_t c = lane; c < H / 16; c += 32) dst[c] = reinterpret_cast<const uint4*>(src)[c];
    const float* ss = reinterpret_cast<const float*>(src + H);
    for (int64_t g = lane; g < H / 128; g += 32) sA[g * Mp + dest] = ss[g];
}

// Zero rows that pad each local expert's rows up to a multiple of 128:
// rows m_offsets[e] + rows_e[e] .. m_offsets[e+1] - 1.  Grid (El, 128 / 8),
// one warp per (expert, padding row).
__global__ void __launch_bounds__(256) k_ep_zero_pad(const int64_t* __restrict__ m_offsets,
                                                     const int64_t* __restrict__ rows_e,
                                                     int64_t H, uint8_t* __restrict__ A8,
                                                     float* __restrict__ sA, int64_t Mp,
                                                     int* status) {
    const int e = blockIdx.x;
    const int r = blockIdx.y * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t row = m_offsets[e] + rows_e[e] + r;
    if (row >= m_offsets[e + 1]) return;
    if (row < 0 || row >= Mp) {
        if (lane == 0) atomicCAS(status, kOk, kErrBadRouting);
        return;
    }
    uint4* dst = reinterpret_cast<uint4*>(A8 + row * H);
    for (int64_t c = lane; c < H / 16; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t g = lane; g < H / 128; g += 32) sA[g * Mp + row] = 0.0f;
}

// One warp per received row i: the grouped GEMM's BF16 result row
// Y[dest(i)] (N columns) goes to row i of `out`, the order the rows arrived in.
__global__ void __launch_bounds__(256) k_ep_gather(const __nv_bfloat16* __restrict__ Y,
                                                   int64_t R, int64_t N,
                                                   const int64_t* __restrict__ src_off,
                                                   const int64_t* __restrict__ dest_base, int nb,
                                                   int64_t Mp, __nv_bfloat16* __restrict__ out,
                                                   int* status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= R) return;
    const int b = ep_block_of(src_off, nb, i);
    const int64_t dest = dest_base[b] + (i - src_off[b]);
    if (dest < 0 || dest >= Mp) {
        if (lane == 0) atomicCAS(status, kOk, kErrBadRouting);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(Y + dest * N);
    uint4* dst = reinterpret_cast<uint4*>(out + i * N);
    for (int64_t c = lane; c < N / 8; c += 32) dst[c] = __ldg(src + c);
}

// out[t][n] = bf16( sum_j w[t][j] * back[pos[t][j]][n] ), the sum in FP32
// over j = 0 .. k-1 in order, rounded once to BF16 (nearest even).  Grid
// (T, ceil(N / 2048)), 256 threads, eight columns (16 bytes) per thread.
__global__ void __launch_bounds__(256) k_ep_combine(const __nv_bfloat16* __restrict__ back,
                                                    const int32_t* __restrict__ pos,
                                                    const float* __restrict__ w, int64_t T,
                                                    int k, int64_t N,
                                                    __nv_bfloat16* __restrict__ out, int* status) {
    const int64_t t = blockIdx.x;
    const int64_t n0 = (static_cast<int64_t>(blockIdx.y) * 256 + threadIdx.x) * 8;
    if (n0 >= N) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
        const float wj = __ldg(w + t * k + j);
        const int64_t row = pos[t * k + j];
        if (row < 0 || row >= T * k) {            // not a position from the route: skip the row
            atomicCAS(status, kOk, kErrBadRouting);
            return;
        }
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(back + row * N + n0));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fmaf_rn(wj, __uint_as_float(u[i] << 16), acc[2 * i]);
            acc[2 * i + 1] = __fmaf_rn(wj, __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
        }
    }
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        op[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(out + t * N + n0) = o;
}

}  // namespace fp8q
