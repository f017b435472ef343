// C ABI of the fp8q library (declared in include/fp8q.h): argument checks,
// TMA descriptor encoding and kernel launches.  No allocation happens here:
// every buffer belongs to the caller.  Library state: a per-device status
// word (a static __device__ variable), cached launch attributes, and
// g_noalloc_scratch, the 40 MiB static device array that fp8q_gemm_noalloc
// uses as its stream-K workspace (one array per device, shared by every call
// of that entry point: calls that overlap on the GPU race).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "ep.cuh"
#include "fp8q.h"
#include "gemm.cuh"
#include "quant.cuh"

namespace fp8q {

__device__ int g_status;   // sticky device-side status, one per device

// Scratch of fp8q_gemm_noalloc: the stream-K workspace kept inside the library
// for callers that cannot allocate device memory.  40 MiB fits the workspace
// of a GPU with up to 159 SMs (37.9 MB on a 148-SM B300).  It is zero when the
// library is loaded and every device that loads the library holds it until
// the process exits.  In host code the name is only a handle: the device
// address comes from cudaGetSymbolAddress (see device_state).
constexpr size_t kNoAllocScratchBytes = size_t(40) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Diagnostic for the bounded waits: one warp waits on an mbarrier that nothing
// arrives on, through the same wait the GEMM pipeline uses, so the wait runs
// out after limit_ns and records kErrTimeout; the kernel then returns.
__global__ void k_selftest_wait(int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const bool done = mbar_wait_for(&bar, 0, status, limit_ns);
    (void)done;
}

// Tensor-pipe throughput probe (a measurement, not part of the method): one
// CTA per SM issues `blocks` x 4 MMAs of 128 x 256 x 32 E4M3 -> FP32 (one
// 128-element K block each) from fixed shared-memory operands into one TMEM
// accumulator, back to back, and waits for them with a bounded wait.  The
// operand bytes are a fixed pseudo-random pattern of finite E4M3 values, so
// the tensor cores see data of realistic bit density, not zeros.
constexpr int kPeakN = 256;
constexpr int kPeakSmem = kBM * kBK + kPeakN * kBK + 1024;

__global__ void __launch_bounds__(128, 1) k_mma_peak(int64_t blocks, int* status) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t done;
    __shared__ uint32_t tbase;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int kBytes = kBM * kBK + kPeakN * kBK;
    for (int i = threadIdx.x; i < kBytes / 4; i += blockDim.x) {
        uint32_t h = static_cast<uint32_t>(i) * 0x9E3779B1u + blockIdx.x * 0x85EBCA6Bu;
        h ^= h >> 15;
        h *= 0x2C1B3C6Du;
        h ^= h >> 12;
        // clearing bit 3 of every byte keeps it off the NaN patterns 0x7F / 0xFF
        reinterpret_cast<uint32_t*>(smem)[i] = h & 0x77777777u;
    }
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(&tbase, kPeakN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, kPeakN);
        const uint32_t a_addr = smem_u32(smem);
        const uint64_t ad = sw128_desc(a_addr);
        const uint64_t bd = sw128_desc(a_addr + kBM * kBK);
#pragma unroll 1
        for (int64_t b = 0; b < blocks; ++b) {
#pragma unroll
            for (int k = 0; k < kBK / 32; ++k)
                mma_e4m3(tbase, ad + 2 * k, bd + 2 * k, kIdesc, (b > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&done);
        if (!mbar_drain(&done, 0, kWaitLimitNs)) atomicCAS(status, kOk, kErrTimeout);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tbase, kPeakN);
    }
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int* status = nullptr;            // device address of g_status on this device
    bool gemm_attr[2][2][2] = {};     // dynamic-smem attribute set, per kernel instance
    bool gemm_qa_attr[2] = {};        // the same for the in-kernel-quantization GEMM
    bool quant_attr[2][2] = {};       // the same for the staged quantizers [kind][bf16 input]
    uint8_t* noalloc_scratch = nullptr;  // device address of g_noalloc_scratch
    bool peak_attr = false;              // dynamic-smem attribute of k_mma_peak set
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// TMA coordinates are 32-bit signed: row and column counts stay below 2^31.
constexpr int64_t kMaxTmaCoord = 0x7fffffff;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_fail() {
    cudaGetLastError();   // clear the sticky runtime error of this thread
    return FP8Q_ERR_CUDA;
}

// Per-device set-up on first use: SM count and the address of g_status.
int device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
    if (dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_fail();
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return cuda_fail();
        d.status = static_cast<int*>(p);
        void* sp = nullptr;
        if (cudaGetSymbolAddress(&sp, g_noalloc_scratch) != cudaSuccess) return cuda_fail();
        d.noalloc_scratch = static_cast<uint8_t*>(sp);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return cuda_fail();
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return FP8Q_OK;
}

// 2-D uint8 tensor [rows][K], K-major, boxes of 128 (K) x box_rows with
// 128-byte swizzle (one box row = one swizzle row).
int encode_kmajor(CUtensorMap* map, const uint8_t* base, int64_t K, int64_t rows, int box_rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// Output C [rows][cols] (FP32 or BF16) for the GEMM epilogue's TMA stores:
// boxes of 32 rows x 128 bytes with the 128-byte swizzle.
int encode_out(CUtensorMap* map, void* base, int out_dtype, int64_t cols, int64_t rows) {
    const bool bf = out_dtype == FP8Q_BF16;
    const cuuint64_t es = bf ? 2 : 4;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = g_encode(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// 2-D tensor [rows][cols] of FP32 or BF16 elements, row-major, boxes of
// box_cols x box_rows copied unswizzled (a box lands in shared memory as
// box_rows rows of box_cols elements); rows past the end read as zeros.
int encode_rows(CUtensorMap* map, const void* base, int in_dtype, int64_t cols, int64_t rows,
                int box_cols, int box_rows) {
    const bool bf = in_dtype == FP8Q_BF16;
    const cuuint64_t es = bf ? 2 : 4;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * es};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = g_encode(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                                2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// Persistent quantizer launch: Cfg::kCtasPerSm CTAs per SM (fewer if there
// are fewer tiles), each walking tiles blockIdx.x, +gridDim.x, ...
template <typename Cfg, typename Kern>
int launch_quant(DeviceState* d, bool& attr, Kern kern, const CUtensorMap& tm, int64_t tiles,
                 int64_t a, int64_t b, uint8_t* q, float* s, cudaStream_t st) {
    constexpr int kSmem = Cfg::kSmemBytes;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
            cudaSuccess)
            return cuda_fail();
        attr = true;
    }
    int64_t grid = static_cast<int64_t>(d->num_sms) * Cfg::kCtasPerSm;
    if (grid > tiles) grid = tiles;
    kern<<<static_cast<unsigned>(grid), Cfg::kThreads, kSmem, st>>>(tm, a, b, q, s, d->status);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : cuda_fail();
}

// Input of a quantizer: BF16 or FP32, tiles of box_cols x box_rows elements.
template <template <typename> class Cfg, template <typename> class Kern>
int quant_common(int kind, const void* x, int in_dtype, int64_t rows, int64_t cols, int box_cols,
                 int box_rows, int64_t tiles, uint8_t* q, float* s, fp8q_stream_t stream) {
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    CUtensorMap tm;
    rc = encode_rows(&tm, x, in_dtype, cols, rows, box_cols, box_rows);
    if (rc != FP8Q_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FP8Q_BF16)
        return launch_quant<Cfg<__nv_bfloat16>>(d, d->quant_attr[kind][1], Kern<__nv_bfloat16>::fn,
                                               tm, tiles, rows, cols, q, s, st);
    return launch_quant<Cfg<float>>(d, d->quant_attr[kind][0], Kern<float>::fn, tm, tiles, rows,
                                    cols, q, s, st);
}

// The 128x1 quantizer: its input map, plus the map of qT [C][T] (uint8) that
// its TMA stores write, boxes of 128 tokens x 64 channels, 128-byte swizzle.
template <typename T>
int launch_quant_128x1(DeviceState* d, bool& attr, const CUtensorMap& tm, const CUtensorMap& tmq,
                       int64_t tiles, int64_t T_, int64_t C, float* sT, cudaStream_t st) {
    using Cfg = QtCfg<T>;
    auto kern = k_quant_128x1<T>;
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::kSmemBytes) != cudaSuccess)
            return cuda_fail();
        attr = true;
    }
    int64_t grid = static_cast<int64_t>(d->num_sms) * Cfg::kCtasPerSm;
    if (grid > tiles) grid = tiles;
    kern<<<static_cast<unsigned>(grid), Cfg::kThreads, Cfg::kSmemBytes, st>>>(tm, tmq, T_, C, sT,
                                                                              d->status);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : cuda_fail();
}
template <typename T> struct KQw { static constexpr auto fn = k_quant_128x128<T>; };

template <int BN, bool kRowB, bool kBf16, bool kQA = false>
int launch_gemm_inst(DeviceState* d, const CUtensorMap& ta, const CUtensorMap& tb,
                     const CUtensorMap& tc, const GemmArgs& args, int tiles_upper, cudaStream_t st) {
    using S = GemmShape<BN, kQA>;
    auto kern = k_gemm<BN, kRowB, kBf16, kQA>;
    bool& attr = kQA ? d->gemm_qa_attr[kBf16] : d->gemm_attr[BN == 256][kRowB][kBf16];
    if (!attr) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kSmemBytes) != cudaSuccess)
            return cuda_fail();
        attr = true;
    }
    int grid = tiles_upper < d->num_sms ? tiles_upper : d->num_sms;
    if (grid < 1) grid = 1;
    kern<<<grid, S::kThreads, S::kSmemBytes, st>>>(ta, tb, tc, args);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : cuda_fail();
}

template <int BN>
int launch_gemm_bn(DeviceState* d, const CUtensorMap& ta, const CUtensorMap& tb,
                   const CUtensorMap& tc, const GemmArgs& args, int tiles_upper, bool row_b,
                   bool bf16, cudaStream_t st) {
    if (row_b)
        return bf16 ? launch_gemm_inst<BN, true, true>(d, ta, tb, tc, args, tiles_upper, st)
                    : launch_gemm_inst<BN, true, false>(d, ta, tb, tc, args, tiles_upper, st);
    return bf16 ? launch_gemm_inst<BN, false, true>(d, ta, tb, tc, args, tiles_upper, st)
                : launch_gemm_inst<BN, false, false>(d, ta, tb, tc, args, tiles_upper, st);
}

// Stream-K workspace: arrival counters (one per promotion warp of each
// stream-K tile; at most 2 * SMs such tiles), then FP32 partial tiles (at most
// two per CTA, one CTA per SM), each a 128 x 256 float block.
constexpr size_t kWsCounterBytes(int sms) {
    return ((static_cast<size_t>(2) * sms * GemmShape<256>::kPromoWarps * sizeof(int) + 255) / 256) * 256;
}
constexpr size_t kWsPartialBytes(int sms) {
    return static_cast<size_t>(2) * sms * (kBM * 256) * sizeof(float);
}

// Everything a GEMM launch needs, made by gemm_plan after every check has
// passed; gemm_launch then only launches.
struct GemmPlan {
    DeviceState* d = nullptr;
    CUtensorMap ta, tb, tc;
    GemmArgs args;
    int BN = 256;
    int tiles_upper = 1;
    bool row_b = false, bf16 = false;
    bool qa = false;                  // A quantized inside the GEMM (BF16 input)
    Sched sk{};                       // dense stream-K: the schedule k_sk_reduce follows
    int sk_tiles = 0;                 //   and its number of cut tiles (0: no reduction)
};

// Checks that need neither a device nor the SM count.
int gemm_check_args(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                    const void* C, int G, int64_t M, int64_t N, int64_t K, int out_dtype,
                    int bscale) {
    if (!A8 || !sA || !B8 || !sB || !C) return FP8Q_ERR_INVALID_ARG;
    if (out_dtype != FP8Q_F32 && out_dtype != FP8Q_BF16) return FP8Q_ERR_INVALID_ARG;
    if (bscale != FP8Q_BSCALE_BLOCK128 && bscale != FP8Q_BSCALE_ROW1x128) return FP8Q_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (M % 128 || N % 128 || K % 128) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (M > (int64_t(1) << 30) || N > (int64_t(1) << 24) || K > (int64_t(1) << 30))
        return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (int64_t(G) * N > (int64_t(1) << 31) - 1) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    // output tiles are counted in 32-bit integers on the device
    if ((M / 128) * (N / 128) > (int64_t(1) << 31) - 1) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(A8, 16) || !aligned(B8, 16) || !aligned(sA, 16) || !aligned(C, 16))
        return FP8Q_ERR_MISALIGNED;
    if (!aligned(sB, bscale == FP8Q_BSCALE_ROW1x128 ? 16 : 4)) return FP8Q_ERR_MISALIGNED;
    return FP8Q_OK;
}

int gemm_plan(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB, void* C,
              const int* m_offsets, int G, int64_t M, int64_t N, int64_t K, int out_dtype,
              int bscale, void* workspace, size_t ws_bytes, GemmPlan& p) {
    int rc = gemm_check_args(A8, sA, B8, sB, C, G, M, N, K, out_dtype, bscale);
    if (rc != FP8Q_OK) return rc;
    if ((rc = device_state(&p.d)) != FP8Q_OK) return rc;
    if (workspace) {
        if (!aligned(workspace, 256)) return FP8Q_ERR_MISALIGNED;
        if (ws_bytes < kWsCounterBytes(p.d->num_sms) + kWsPartialBytes(p.d->num_sms))
            return FP8Q_ERR_INVALID_ARG;
    }
    p.BN = (N % 256 == 0) ? 256 : 128;
    std::memset(&p.ta, 0, sizeof(p.ta));
    std::memset(&p.tb, 0, sizeof(p.tb));
    std::memset(&p.tc, 0, sizeof(p.tc));
    if ((rc = encode_kmajor(&p.ta, A8, K, M, 128)) != FP8Q_OK) return rc;
    if ((rc = encode_kmajor(&p.tb, B8, K, int64_t(G) * N, p.BN)) != FP8Q_OK) return rc;
    if ((rc = encode_out(&p.tc, C, out_dtype, N, M)) != FP8Q_OK) return rc;
    GemmArgs& a = p.args;
    a.sA = sA;
    a.sB = sB;
    a.C = C;
    a.m_offsets = m_offsets;
    a.M_total = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.G = G;
    a.status = p.d->status;
    a.counters = workspace ? static_cast<int*>(workspace) : nullptr;
    a.ws = workspace ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                 kWsCounterBytes(p.d->num_sms))
                     : nullptr;
    const int64_t tiles = (M / 128) * (N / p.BN);
    // with a workspace every SM takes part (stream-K shares out the tail)
    p.tiles_upper = workspace ? p.d->num_sms
                    : tiles > (int64_t(1) << 30) ? (1 << 30) : static_cast<int>(tiles);
    p.row_b = bscale == FP8Q_BSCALE_ROW1x128;
    p.bf16 = out_dtype == FP8Q_BF16;
    a.Abf = nullptr;
    a.sA_out = nullptr;
    // Dense GEMM with a workspace: the host knows the tile count, so it plans
    // the same schedule the kernel will (Sched::plan, same inputs).  When that
    // schedule cuts every tile, a separate reduction kernel sums the pieces
    // across all SMs (measured: the 1024 x 1024 x 16384 GEMM 23% faster than
    // with the in-kernel sum); with whole-tile waves beside the cut tiles the
    // in-kernel sum overlaps them and stays cheaper (a separate reduction made
    // the 7168 x 2048 x 8192 weight-gradient GEMM 5% slower).  Grouped GEMMs
    // (tile count known only on the device) and row-scaled B keep the
    // in-kernel sum.
    a.sk_reduce = 0;
    p.sk_tiles = 0;
    if (workspace && !m_offsets && !p.row_b) {
        const int grid = p.tiles_upper < p.d->num_sms ? p.tiles_upper : p.d->num_sms;
        Sched sc{};
        sc.plan(static_cast<int>(tiles), static_cast<int>(K / kBK), grid, true);
        if (sc.sk_ctas > 0 && sc.dp_tiles == 0) {
            a.sk_reduce = 1;
            p.sk = sc;
            p.sk_tiles = sc.tiles - sc.dp_tiles;
        }
    }
    return FP8Q_OK;
}

// Plan of the GEMM that quantizes its BF16 activations itself
// (fp8q_gemm_quant_a): the same checks and schedule, 256-column tiles,
// 128x128-block weight scales; tmA becomes the store map of the emitted A8
// (boxes of 128 bytes x 32 rows, the quantizer warps' slices).
int gemm_plan_qa(const void* Abf, const uint8_t* B8, const float* sB, void* C, uint8_t* A8_out,
                 float* sA_out, int64_t M, int64_t N, int64_t K, int out_dtype, void* workspace,
                 size_t ws_bytes, GemmPlan& p) {
    if (!Abf) return FP8Q_ERR_INVALID_ARG;
    if ((A8_out == nullptr) != (sA_out == nullptr)) return FP8Q_ERR_INVALID_ARG;
    if (A8_out && !aligned(A8_out, 16)) return FP8Q_ERR_MISALIGNED;
    if (sA_out && !aligned(sA_out, 4)) return FP8Q_ERR_MISALIGNED;
    // the generic checks, with the BF16 input standing in for A8 and sA
    // (both must be 16-byte aligned, which Abf has to be anyway)
    const uint8_t* a8 = static_cast<const uint8_t*>(Abf);
    const float* sa = static_cast<const float*>(Abf);
    int rc = gemm_check_args(a8, sa, B8, sB, C, 1, M, N, K, out_dtype, FP8Q_BSCALE_BLOCK128);
    if (rc != FP8Q_OK) return rc;
    if (N % 256) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    rc = gemm_plan(a8, sa, B8, sB, C, nullptr, 1, M, N, K, out_dtype, FP8Q_BSCALE_BLOCK128,
                   workspace, ws_bytes, p);
    if (rc != FP8Q_OK) return rc;
    std::memset(&p.ta, 0, sizeof(p.ta));
    if (A8_out && (rc = encode_kmajor(&p.ta, A8_out, K, M, 32)) != FP8Q_OK) return rc;
    p.args.sA = nullptr;
    p.args.Abf = static_cast<const uint16_t*>(Abf);
    p.args.sA_out = sA_out;
    p.qa = true;
    return FP8Q_OK;
}

// The stream-K reduction of a dense GEMM (after it, on the same stream).
template <int BN>
int launch_sk_reduce(const GemmPlan& p, cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>(p.sk_tiles), static_cast<unsigned>(4 * (BN / 128)));
    if (p.bf16)
        k_sk_reduce<BN, true><<<grid, 256, 0, st>>>(p.args.ws, p.args.C, p.args.N, p.sk);
    else
        k_sk_reduce<BN, false><<<grid, 256, 0, st>>>(p.args.ws, p.args.C, p.args.N, p.sk);
    return cudaGetLastError() == cudaSuccess ? FP8Q_OK : cuda_fail();
}

int gemm_launch(const GemmPlan& p, cudaStream_t st) {
    int rc;
    if (p.qa)
        rc = p.bf16 ? launch_gemm_inst<256, false, true, true>(p.d, p.ta, p.tb, p.tc, p.args,
                                                               p.tiles_upper, st)
                    : launch_gemm_inst<256, false, false, true>(p.d, p.ta, p.tb, p.tc, p.args,
                                                                p.tiles_upper, st);
    else
        rc = p.BN == 256 ? launch_gemm_bn<256>(p.d, p.ta, p.tb, p.tc, p.args, p.tiles_upper,
                                               p.row_b, p.bf16, st)
                         : launch_gemm_bn<128>(p.d, p.ta, p.tb, p.tc, p.args, p.tiles_upper,
                                               p.row_b, p.bf16, st);
    if (rc != FP8Q_OK || p.sk_tiles == 0) return rc;
    return p.BN == 256 ? launch_sk_reduce<256>(p, st) : launch_sk_reduce<128>(p, st);
}

int gemm_common(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB, void* C,
                const int* m_offsets, int G, int64_t M, int64_t N, int64_t K, int out_dtype,
                int bscale, void* workspace, size_t ws_bytes, cudaStream_t st) {
    GemmPlan p;
    const int rc = gemm_plan(A8, sA, B8, sB, C, m_offsets, G, M, N, K, out_dtype, bscale,
                             workspace, ws_bytes, p);
    return rc != FP8Q_OK ? rc : gemm_launch(p, st);
}

int check_in_dtype(int t) { return (t == FP8Q_F32 || t == FP8Q_BF16) ? FP8Q_OK : FP8Q_ERR_INVALID_ARG; }

int launched() { return cudaGetLastError() == cudaSuccess ? FP8Q_OK : cuda_fail(); }

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" {

int fp8q_quant_act_1x128(const void* x, int in_dtype, int64_t M, int64_t K, uint8_t* q, float* s,
                         fp8q_stream_t stream) {
    if (!x || !q || !s) return FP8Q_ERR_INVALID_ARG;
    if (check_in_dtype(in_dtype) != FP8Q_OK || M <= 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (K % 128) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    const int64_t yblocks = (M + kQ1Rows - 1) / kQ1Rows;
    if (yblocks > 65535 || K / 128 > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(s, 4)) return FP8Q_ERR_MISALIGNED;
    const dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(yblocks));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FP8Q_BF16)
        k_quant_1x128<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), M,
                                                           K, q, s);
    else
        k_quant_1x128<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x), M, K, q, s);
    return launched();
}

int fp8q_swiglu_quant_1x128(const void* gate, const void* up, int in_dtype, int64_t M, int64_t I,
                            int64_t ld, uint8_t* q, float* s, fp8q_stream_t stream) {
    if (!gate || !up || !q || !s) return FP8Q_ERR_INVALID_ARG;
    if (check_in_dtype(in_dtype) != FP8Q_OK || M <= 0 || I <= 0 || ld < I)
        return FP8Q_ERR_INVALID_ARG;
    if (I % 128) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    const int64_t yblocks = (M + kSwRows - 1) / kSwRows;
    if (yblocks > 65535 || I / 128 > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    const int64_t es = in_dtype == FP8Q_BF16 ? 2 : 4;
    if (!aligned(gate, 16) || !aligned(up, 16) || (ld * es) % 16 || !aligned(q, 16) ||
        !aligned(s, 4))
        return FP8Q_ERR_MISALIGNED;
    const dim3 grid(static_cast<unsigned>(I / 128), static_cast<unsigned>(yblocks));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FP8Q_BF16)
        k_swiglu_quant_1x128<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(gate), static_cast<const __nv_bfloat16*>(up), M, I,
            ld, q, s);
    else
        k_swiglu_quant_1x128<float><<<grid, 256, 0, st>>>(static_cast<const float*>(gate),
                                                          static_cast<const float*>(up), M, I, ld,
                                                          q, s);
    return launched();
}

int fp8q_rmsnorm_quant_1x128(const void* x, const void* w, int in_dtype, int64_t M, int64_t K,
                             float eps, uint8_t* q, float* s, fp8q_stream_t stream) {
    if (!x || !w || !q || !s) return FP8Q_ERR_INVALID_ARG;
    if (check_in_dtype(in_dtype) != FP8Q_OK || M <= 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (!(eps > 0.0f) || eps > FLT_MAX) return FP8Q_ERR_INVALID_ARG;
    if (K % 128 || K > kRnMaxK || M > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(q, 16) || !aligned(s, 4))
        return FP8Q_ERR_MISALIGNED;
    DeviceState* d = nullptr;
    const int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    const int threads = static_cast<int>((K / 16 + 31) / 32 * 32);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // persistent: as many CTAs as fit on the GPU at once (at most one per row)
    auto grid_for = [&](const void* kern) -> unsigned {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int64_t g = static_cast<int64_t>(per_sm) * d->num_sms;
        return static_cast<unsigned>(g < M ? g : M);
    };
    if (in_dtype == FP8Q_BF16) {
        auto kern = k_rmsnorm_quant_1x128<__nv_bfloat16>;
        kern<<<grid_for(reinterpret_cast<const void*>(kern)), threads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), M, K, eps,
            q, s);
    } else {
        auto kern = k_rmsnorm_quant_1x128<float>;
        kern<<<grid_for(reinterpret_cast<const void*>(kern)), threads, 0, st>>>(
            static_cast<const float*>(x), static_cast<const float*>(w), M, K, eps, q, s);
    }
    return launched();
}

int fp8q_quant_act_128x1(const void* x, int in_dtype, int64_t T, int64_t C, uint8_t* qT, float* sT,
                         fp8q_stream_t stream) {
    if (!x || !qT || !sT) return FP8Q_ERR_INVALID_ARG;
    if (check_in_dtype(in_dtype) != FP8Q_OK || T <= 0 || C <= 0) return FP8Q_ERR_INVALID_ARG;
    if (T % 128 || C % 64) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (T > kMaxTmaCoord || C > kMaxTmaCoord) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(qT, 16) || !aligned(sT, 4)) return FP8Q_ERR_MISALIGNED;
    const int64_t tiles = (C / 64) * (T / 128);
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    CUtensorMap tm, tmq;
    if ((rc = encode_rows(&tm, x, in_dtype, C, T, 64, 128)) != FP8Q_OK) return rc;
    if ((rc = encode_kmajor(&tmq, qT, T, C, 64)) != FP8Q_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (in_dtype == FP8Q_BF16)
        return launch_quant_128x1<__nv_bfloat16>(d, d->quant_attr[0][1], tm, tmq, tiles, T, C, sT, st);
    return launch_quant_128x1<float>(d, d->quant_attr[0][0], tm, tmq, tiles, T, C, sT, st);
}

int fp8q_quant_w_128x128(const void* w, int in_dtype, int64_t N, int64_t K, uint8_t* q, float* s,
                         fp8q_stream_t stream) {
    if (!w || !q || !s) return FP8Q_ERR_INVALID_ARG;
    if (check_in_dtype(in_dtype) != FP8Q_OK || N <= 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (N % 128 || K % 128) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (N > kMaxTmaCoord || K > kMaxTmaCoord) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w, 16) || !aligned(q, 16) || !aligned(s, 4)) return FP8Q_ERR_MISALIGNED;
    const int64_t tiles = (K / 128) * (N / 128);
    return quant_common<QwCfg, KQw>(1, w, in_dtype, N, K, 128, 128, tiles, q, s, stream);
}

int fp8q_retile_1x128_to_128x1(const uint8_t* q, const float* s, int64_t T, int64_t C,
                               uint8_t* qT, float* sT, fp8q_stream_t stream) {
    if (!q || !s || !qT || !sT) return FP8Q_ERR_INVALID_ARG;
    if (T <= 0 || C <= 0) return FP8Q_ERR_INVALID_ARG;
    if (T % 128 || C % 128) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (T / 128 > 65535 || C / 64 > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(q, 16) || !aligned(qT, 16) || !aligned(s, 4) || !aligned(sT, 4))
        return FP8Q_ERR_MISALIGNED;
    const dim3 grid(static_cast<unsigned>(C / 64), static_cast<unsigned>(T / 128));
    k_retile_1x128_to_128x1<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, s, T, C,
                                                                                       qT, sT);
    return launched();
}

int fp8q_transpose_w_128x128(const uint8_t* q, const float* s, int64_t N, int64_t K, uint8_t* qT,
                             float* sT, fp8q_stream_t stream) {
    if (!q || !s || !qT || !sT) return FP8Q_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0) return FP8Q_ERR_INVALID_ARG;
    if (N % 128 || K % 128) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (N / 128 > 65535 || K / 128 > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(q, 16) || !aligned(qT, 16) || !aligned(s, 4) || !aligned(sT, 4))
        return FP8Q_ERR_MISALIGNED;
    const dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>(N / 128));
    k_transpose_128x128<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q, s, N, K, qT,
                                                                                  sT);
    return launched();
}

int fp8q_gemm(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB, void* C,
              int64_t M, int64_t N, int64_t K, int out_dtype) {
    return gemm_common(A8, sA, B8, sB, C, nullptr, 1, M, N, K, out_dtype, FP8Q_BSCALE_BLOCK128,
                       nullptr, 0, nullptr);
}

int fp8q_gemm_ex(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB, void* C,
                 int64_t M, int64_t N, int64_t K, int out_dtype, int bscale, fp8q_stream_t stream) {
    return gemm_common(A8, sA, B8, sB, C, nullptr, 1, M, N, K, out_dtype, bscale, nullptr, 0,
                       reinterpret_cast<cudaStream_t>(stream));
}

int fp8q_gemm_ws(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB, void* C,
                 int64_t M, int64_t N, int64_t K, int out_dtype, int bscale, void* workspace,
                 size_t workspace_bytes, fp8q_stream_t stream) {
    return gemm_common(A8, sA, B8, sB, C, nullptr, 1, M, N, K, out_dtype, bscale, workspace,
                       workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t fp8q_gemm_workspace_size(void) {
    DeviceState* d = nullptr;
    if (device_state(&d) != FP8Q_OK) return 0;
    return kWsCounterBytes(d->num_sms) + kWsPartialBytes(d->num_sms);
}

int fp8q_gemm_grouped(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                      void* C, const int* m_offsets, int G, int64_t M_total, int64_t N, int64_t K,
                      int out_dtype, fp8q_stream_t stream) {
    if (!m_offsets) return FP8Q_ERR_INVALID_ARG;
    if (G < 1 || G > kMaxGroups) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(m_offsets, 4)) return FP8Q_ERR_MISALIGNED;
    return gemm_common(A8, sA, B8, sB, C, m_offsets, G, M_total, N, K, out_dtype,
                       FP8Q_BSCALE_BLOCK128, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

int fp8q_gemm_quant_a(const void* A, const uint8_t* B8, const float* sB, void* C,
                      uint8_t* A8_out, float* sA_out, int64_t M, int64_t N, int64_t K,
                      int out_dtype, void* workspace, size_t workspace_bytes,
                      fp8q_stream_t stream) {
    GemmPlan p;
    const int rc = gemm_plan_qa(A, B8, sB, C, A8_out, sA_out, M, N, K, out_dtype, workspace,
                                workspace_bytes, p);
    return rc != FP8Q_OK ? rc : gemm_launch(p, reinterpret_cast<cudaStream_t>(stream));
}

int fp8q_gemm_noalloc(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                      void* C, int64_t M, int64_t N, int64_t K, int out_dtype, int bscale,
                      fp8q_stream_t stream) {
    // Every check the workspace GEMM makes (arguments, shape limits, the TMA
    // descriptors) is made before the counter clear below is queued, so that
    // nothing is launched when one of them fails.
    int rc = gemm_check_args(A8, sA, B8, sB, C, 1, M, N, K, out_dtype, bscale);
    if (rc != FP8Q_OK) return rc;
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != FP8Q_OK) return rc;
    const size_t counters = kWsCounterBytes(d->num_sms);
    const size_t need = counters + kWsPartialBytes(d->num_sms);
    if (need > kNoAllocScratchBytes) return FP8Q_ERR_UNSUPPORTED_SHAPE;   // more SMs than it fits
    GemmPlan p;
    if ((rc = gemm_plan(A8, sA, B8, sB, C, nullptr, 1, M, N, K, out_dtype, bscale,
                        d->noalloc_scratch, kNoAllocScratchBytes, p)) != FP8Q_OK)
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the arrival counters must start at zero; a call that failed on the
    // device may have left some set, so clear them every time
    if (cudaMemsetAsync(d->noalloc_scratch, 0, counters, st) != cudaSuccess) return cuda_fail();
    return gemm_launch(p, st);
}

int fp8q_gemm_grouped_ws(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                         void* C, const int* m_offsets, int G, int64_t M_total, int64_t N,
                         int64_t K, int out_dtype, void* workspace, size_t workspace_bytes,
                         fp8q_stream_t stream) {
    if (!m_offsets) return FP8Q_ERR_INVALID_ARG;
    if (G < 1 || G > kMaxGroups) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(m_offsets, 4)) return FP8Q_ERR_MISALIGNED;
    return gemm_common(A8, sA, B8, sB, C, m_offsets, G, M_total, N, K, out_dtype,
                       FP8Q_BSCALE_BLOCK128, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

int64_t fp8q_ep_row_bytes(int64_t H) { return (H > 0 && H % 128 == 0) ? ep_row_bytes(H) : -1; }

int fp8q_ep_route(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* counts,
                  int32_t* pos, fp8q_stream_t stream) {
    if (!counts || (T > 0 && (!topk_ids || !pos))) return FP8Q_ERR_INVALID_ARG;
    if (T < 0 || k < 1 || E < 1) return FP8Q_ERR_INVALID_ARG;
    if (E > kEpMaxExperts || T * k > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(topk_ids, 4) || !aligned(counts, 4) || !aligned(pos, 4)) return FP8Q_ERR_MISALIGNED;
    // T == 0 still launches: the counts are written (all zero)
    DeviceState* d = nullptr;
    const int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    k_ep_route<<<1, kEpRouteThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        topk_ids, T * k, E, counts, pos, d->status);
    return launched();
}

int fp8q_ep_pack(const uint8_t* q, const float* s, const int32_t* pos, int64_t T, int k,
                 int64_t H, uint8_t* send, fp8q_stream_t stream) {
    if (T < 0 || k < 1 || H <= 0) return FP8Q_ERR_INVALID_ARG;
    if (T == 0) return FP8Q_OK;
    if (!q || !s || !pos || !send) return FP8Q_ERR_INVALID_ARG;
    if (H % 128 || T * k > 0x7fffffff) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(q, 16) || !aligned(send, 16) || !aligned(s, 4) || !aligned(pos, 4))
        return FP8Q_ERR_MISALIGNED;
    k_ep_pack<<<static_cast<unsigned>((T * k + 7) / 8), 256, 0,
                reinterpret_cast<cudaStream_t>(stream)>>>(q, s, pos, T, k, H, send);
    return launched();
}

int fp8q_ep_unpack(const uint8_t* recv, int64_t R, int64_t H, const int64_t* src_off,
                   const int64_t* dest_base, int nb, const int64_t* m_offsets,
                   const int64_t* rows_e, int El, uint8_t* A8, float* sA, int64_t Mp,
                   fp8q_stream_t stream) {
    if (!src_off || !dest_base || !m_offsets || !rows_e || !A8 || !sA) return FP8Q_ERR_INVALID_ARG;
    if (R < 0 || H <= 0 || nb < 1 || El < 1 || Mp <= 0 || (R > 0 && !recv))
        return FP8Q_ERR_INVALID_ARG;
    if (H % 128 || Mp % 128 || R > 0x7fffffffLL * 8 || El > 65535) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if ((recv && !aligned(recv, 16)) || !aligned(A8, 16) || !aligned(sA, 4) ||
        !aligned(src_off, 8) || !aligned(dest_base, 8) || !aligned(m_offsets, 8) ||
        !aligned(rows_e, 8))
        return FP8Q_ERR_MISALIGNED;
    DeviceState* d = nullptr;
    const int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (R > 0)
        k_ep_unpack<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
            recv, R, H, src_off, dest_base, nb, A8, sA, Mp, d->status);
    if (cudaGetLastError() != cudaSuccess) return cuda_fail();
    k_ep_zero_pad<<<dim3(static_cast<unsigned>(El), 16), 256, 0, st>>>(m_offsets, rows_e, H, A8,
                                                                        sA, Mp, d->status);
    return launched();
}

int fp8q_ep_gather(const void* Y, int64_t Mp, int64_t R, int64_t N, const int64_t* src_off,
                   const int64_t* dest_base, int nb, void* out, fp8q_stream_t stream) {
    if (R < 0 || N <= 0 || nb < 1 || Mp < 0) return FP8Q_ERR_INVALID_ARG;
    if (R == 0) return FP8Q_OK;
    if (!Y || !src_off || !dest_base || !out) return FP8Q_ERR_INVALID_ARG;
    if (N % 8 || R > 0x7fffffffLL * 8) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(Y, 16) || !aligned(out, 16) || !aligned(src_off, 8) || !aligned(dest_base, 8))
        return FP8Q_ERR_MISALIGNED;
    DeviceState* d = nullptr;
    const int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    k_ep_gather<<<static_cast<unsigned>((R + 7) / 8), 256, 0,
                  reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(Y), R, N, src_off, dest_base, nb, Mp,
        static_cast<__nv_bfloat16*>(out), d->status);
    return launched();
}

int fp8q_ep_combine(const void* back, const int32_t* pos, const float* w, int64_t T, int k,
                    int64_t N, void* out, fp8q_stream_t stream) {
    if (T < 0 || k < 1 || N <= 0) return FP8Q_ERR_INVALID_ARG;
    if (T == 0) return FP8Q_OK;
    if (!pos || !w || !out || !back) return FP8Q_ERR_INVALID_ARG;
    if (N % 8 || T > 0x7fffffff || (N + 2047) / 2048 > 65535) return FP8Q_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(back, 16) || !aligned(out, 16) || !aligned(pos, 4) || !aligned(w, 4))
        return FP8Q_ERR_MISALIGNED;
    DeviceState* d = nullptr;
    const int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>((N + 2047) / 2048));
    k_ep_combine<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16*>(back), pos, w, T, k, N, static_cast<__nv_bfloat16*>(out),
        d->status);
    return launched();
}

int fp8q_get_device_status(fp8q_stream_t stream) {
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return cuda_fail();
    int v = 0;
    if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_fail();
    if (v != FP8Q_OK) {
        const int zero = 0;
        if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return cuda_fail();
    }
    return v;
}

int fp8q_selftest_wait(int64_t limit_ns, fp8q_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > 100000000) return FP8Q_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    k_selftest_wait<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        d->status, static_cast<uint64_t>(limit_ns));
    return launched();
}

int fp8q_bench_mma_peak(int64_t blocks, fp8q_stream_t stream) {
    if (blocks <= 0 || blocks > (int64_t(1) << 20)) return FP8Q_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != FP8Q_OK) return rc;
    if (!d->peak_attr) {
        if (cudaFuncSetAttribute(k_mma_peak, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPeakSmem) != cudaSuccess)
            return cuda_fail();
        d->peak_attr = true;
    }
    k_mma_peak<<<d->num_sms, 128, kPeakSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
        blocks, d->status);
    return launched();
}

int fp8q_num_sms(void) {
    DeviceState* d = nullptr;
    return device_state(&d) == FP8Q_OK ? d->num_sms : -FP8Q_ERR_CUDA;
}

const char* fp8q_status_string(int status) {
    switch (status) {
        case FP8Q_OK: return "ok";
        case FP8Q_ERR_INVALID_ARG: return "invalid argument";
        case FP8Q_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case FP8Q_ERR_MISALIGNED: return "misaligned pointer";
        case FP8Q_ERR_CUDA: return "CUDA error";
        case FP8Q_ERR_TIMEOUT: return "device pipeline wait timed out";
        case FP8Q_ERR_BAD_GROUPS: return "invalid group offsets";
        case FP8Q_ERR_BAD_ROUTING: return "expert id out of range";
        default: return "unknown status";
    }
}

int fp8q_version(void) { return 100; }

}  // extern "C"
