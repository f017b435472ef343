/*
 * fp8q -- fine-grained FP8 (E4M3) quantization and block-scaled FP8 GEMM
 * for NVIDIA B300 (sm_103a).  C ABI.
 *
 * The operations follow DeepSeek-V3's FP8 training recipe as described on the
 * pages:
 *   "Six Reasons Deepseek Ai Is A Waste Of Time" (myomija.com), paras. 1-4;
 *   codingmall.com knowledge-base article on FP8 in DeepSeek-V3 (Greek),
 *     sections "fine-grained quantization", "online quantization",
 *     "increased accumulation precision", "unified E4M3 format";
 *   codingmall.com article on FP8 GEMM in DeepSeek-V3 (Japanese), items 1-8;
 *   woojincopolymer.co.kr board post, paras. 3-4 (the FP8 cast fused into the
 *     operator that produces the activation: RMSNorm, SwiGLU).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All data pointers are DEVICE pointers owned by the caller; the library
 *   never allocates, frees or keeps them (scratch space, where a call can use
 *   it, is a caller-provided workspace argument).  Every call is asynchronous
 *   on the given stream (a cudaStream_t; NULL = the legacy default stream)
 *   and does not synchronize.
 * - Return value: FP8Q_OK or an fp8q_status error code.  Arguments are
 *   checked before anything is launched; on error nothing is launched and
 *   the outputs are untouched.  A failed launch returns FP8Q_ERR_CUDA.
 * - Device-side problems (an inconsistent m_offsets array, a pipeline wait
 *   that exceeded its time limit) are recorded in a sticky device status word
 *   and read with fp8q_get_device_status().  Kernels never trap.
 * - FP8 data is E4M3 (OCP: bias 7, no infinities, 0x7F/0xFF = NaN, largest
 *   finite value 448) stored one byte per element.  The cast is
 *   round-to-nearest-even with saturation to +-448; the sign of zero is kept.
 * - Online scaling ("online quantization" section; para. 1 of "Six
 *   Reasons..."): per group, amax = max |x| over the group;
 *   s = fl32(amax / 448) is stored; each element is cast from
 *   fl32(x * fl32(448 / amax)).  A group with amax == 0 stores s = 1.
 *   448/amax overflowing FP32 is clamped to FLT_MAX.  Dequantized value =
 *   decode(q) * s.  Inputs must be finite.
 * - Row-major, last index contiguous.  Sizes are element counts.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* fp8q_stream_t;

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_INVALID_ARG = 1,      /* null pointer, non-positive size, bad enum */
    FP8Q_ERR_UNSUPPORTED_SHAPE = 2,/* a size this version does not tile (see each call) */
    FP8Q_ERR_MISALIGNED = 3,       /* a pointer is not 16-byte aligned */
    FP8Q_ERR_CUDA = 4,             /* a CUDA runtime/driver call failed */
    FP8Q_ERR_TIMEOUT = 5,          /* device: a pipeline wait exceeded its limit */
    FP8Q_ERR_BAD_GROUPS = 6,       /* device: m_offsets not monotone / not multiples of 128 /
                                      beyond M_total */
    FP8Q_ERR_BAD_ROUTING = 7       /* device: an expert id outside [0, E) */
} fp8q_status;

typedef enum { FP8Q_F32 = 0, FP8Q_BF16 = 1 } fp8q_dtype;

/* How the B operand's scales are grouped (see fp8q_gemm_ex). */
typedef enum {
    FP8Q_BSCALE_BLOCK128 = 0,      /* 128x128 weight blocks: sB[N/128][K/128] */
    FP8Q_BSCALE_ROW1x128 = 1       /* 1x128 tiles of B's rows: sB[K/128][N] */
} fp8q_bscale;

/* ---------------------------------------------------------------- quantize */

/* Activations, one scale per 1x128 tile (per token per 128 channels):
 * "Six Reasons...", para. 3 (grouping item 1); "fine-grained quantization".
 *   x   [M][K]  in_dtype (FP8Q_F32 or FP8Q_BF16), 16-byte aligned
 *   q   [M][K]  uint8 E4M3, 16-byte aligned
 *   s   [K/128][M] float32 (scale of row m, group g at s[g*M + m]), 4-byte aligned
 * Requires M >= 1, K a multiple of 128. */
FP8Q_API int fp8q_quant_act_1x128(const void* x, int in_dtype, int64_t M, int64_t K,
                         uint8_t* q, float* s, fp8q_stream_t stream);

/* Fused SwiGLU + 1x128 FP8 cast: h = silu(gate) * up = gate * up / (1 + e^-gate),
 * computed in FP32 and quantized per 1x128 tile exactly like
 * fp8q_quant_act_1x128, without h being written.  woojincopolymer post,
 * para. 3 (the FP8 cast fused into the operator producing the activation) and
 * para. 4 (the SwiGLU output, recomputed from cached inputs, kept as 1x128
 * FP8 tiles).  h carries FP32 rounding (e^-gate to a few ulp), so results
 * match a correctly rounded evaluation to within a few FP32 ulp of h before
 * the cast, not bit for bit.
 *   gate, up  [M][I] in_dtype, row m at gate + m*ld and up + m*ld (ld >= I
 *             elements; ld = 2I with up = gate + I reads one [M][2I] tensor);
 *             16-byte aligned, ld * element size a multiple of 16
 *   q   [M][I]  uint8 E4M3 (contiguous), 16-byte aligned
 *   s   [I/128][M] float32, 4-byte aligned
 * Requires M >= 1, I a multiple of 128. */
FP8Q_API int fp8q_swiglu_quant_1x128(const void* gate, const void* up, int in_dtype, int64_t M,
                         int64_t I, int64_t ld, uint8_t* q, float* s, fp8q_stream_t stream);

/* Fused RMSNorm + 1x128 FP8 cast: y = x * w / sqrt(mean_k x^2 + eps) per row,
 * computed in FP32 and quantized per 1x128 tile exactly like
 * fp8q_quant_act_1x128, without y being written.  woojincopolymer post,
 * para. 3 (layer normalization fused with the FP8 cast; RMSNorm is
 * DeepSeek-V3's normalization).  The row's sum of squares is an FP32
 * reduction, so results match a correctly rounded evaluation to within a few
 * FP32 ulp of y before the cast, not bit for bit.
 *   x   [M][K]  in_dtype, 16-byte aligned
 *   w   [K]     in_dtype (per-channel weight), 16-byte aligned
 *   eps         > 0 and finite (FP8Q_ERR_INVALID_ARG otherwise)
 *   q   [M][K]  uint8 E4M3, 16-byte aligned
 *   s   [K/128][M] float32, 4-byte aligned
 * Requires M >= 1 (below 2^31), K a multiple of 128 and at most 16384
 * (FP8Q_ERR_UNSUPPORTED_SHAPE otherwise). */
FP8Q_API int fp8q_rmsnorm_quant_1x128(const void* x, const void* w, int in_dtype, int64_t M,
                         int64_t K, float eps, uint8_t* q, float* s, fp8q_stream_t stream);

/* Activations regrouped for the backward pass, one scale per 128x1 tile
 * (128 consecutive tokens of one channel), written transposed so that the
 * result is a K-major GEMM operand whose K runs over tokens:
 * "Six Reasons...", para. 3 (1x128 -> 128x1 conversion in the backward pass).
 *   x   [T][C]  in_dtype, 16-byte aligned
 *   qT  [C][T]  uint8 E4M3, 16-byte aligned
 *   sT  [T/128][C] float32 (scale of channel c, token group tb at sT[tb*C + c])
 * Requires T a multiple of 128, C a multiple of 64, both below 2^31
 * (FP8Q_ERR_UNSUPPORTED_SHAPE otherwise). */
FP8Q_API int fp8q_quant_act_128x1(const void* x, int in_dtype, int64_t T, int64_t C,
                         uint8_t* qT, float* sT, fp8q_stream_t stream);

/* Weights, one scale per 128x128 block (128 output x 128 input channels):
 * "Six Reasons...", para. 3 (grouping item 2); "fine-grained quantization".
 *   w   [N][K]  in_dtype, 16-byte aligned
 *   q   [N][K]  uint8 E4M3, 16-byte aligned
 *   s   [N/128][K/128] float32
 * Requires N and K multiples of 128, both below 2^31
 * (FP8Q_ERR_UNSUPPORTED_SHAPE otherwise). */
FP8Q_API int fp8q_quant_w_128x128(const void* w, int in_dtype, int64_t N, int64_t K,
                         uint8_t* q, float* s, fp8q_stream_t stream);

/* Backward regrouping of stored activations: "Six Reasons...", para. 3
 * (activations converted from 1x128 tiles to 128x1 tiles in the backward
 * pass), starting from the forward pass's stored 1x128 FP8 tiles.  Each element
 * is dequantized (exact E4M3 decode times its tile scale, one FP32 rounding)
 * and quantized again per 128 tokens of one channel, written transposed:
 *   q   [T][C]  uint8 E4M3 (from fp8q_quant_act_1x128), 16-byte aligned
 *   s   [C/128][T] float32
 *   qT  [C][T]  uint8 E4M3, 16-byte aligned; sT [T/128][C] float32
 * (the layout fp8q_quant_act_128x1 writes).  Requires T and C multiples of 128. */
FP8Q_API int fp8q_retile_1x128_to_128x1(const uint8_t* q, const float* s, int64_t T, int64_t C,
                               uint8_t* qT, float* sT, fp8q_stream_t stream);

/* Transposed FP8 weight for the data-gradient GEMM dX = dY W: q[N][K] with
 * 128x128 block scales s[N/128][K/128] -> qT[K][N] with sT[K/128][N/128]
 * (byte-exact; the blocks and their scales are the forward weight's).  Then
 * fp8q_gemm_ex(dY8, sdY, qT, sT, dX, T, K, N, ...) computes dX[T][K].
 * q, qT 16-byte aligned; requires N and K multiples of 128. */
FP8Q_API int fp8q_transpose_w_128x128(const uint8_t* q, const float* s, int64_t N, int64_t K,
                             uint8_t* qT, float* sT, fp8q_stream_t stream);

/* -------------------------------------------------------------------- GEMM */

/* Block-scaled FP8 GEMM  C[M][N] = sum_k (A8[m][k] sA) (B8[n][k] sB), i.e.
 * C = A * B^T with both operands K-major:  "Six Reasons...", paras. 1-2 (FP8
 * inputs, BF16/FP32 outputs, per-group scaling factors along K applied as
 * dequantization on the CUDA cores) and para. 3 / "increased accumulation
 * precision" (tensor-core partials of each 128-element K block are promoted
 * to FP32 registers, scaled, and accumulated in full FP32).
 *   A8  [M][K]  uint8 E4M3, 16-byte aligned     sA [K/128][M] float32, 16-byte aligned
 *   B8  [N][K]  uint8 E4M3, 16-byte aligned     sB [N/128][K/128] float32
 *   C   [M][N]  out_dtype (FP8Q_F32 or FP8Q_BF16, BF16 rounded to nearest even),
 *               16-byte aligned; fully overwritten.
 * Requires M, N, K multiples of 128, M and K at most 2^30, N at most 2^24 and
 * at most 2^31 - 1 output tiles of 128 x 128 (FP8Q_ERR_UNSUPPORTED_SHAPE
 * otherwise).  Runs on the legacy default stream. */
FP8Q_API int fp8q_gemm(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
              void* C, int64_t M, int64_t N, int64_t K, int out_dtype);

/* fp8q_gemm with a stream and a choice of B-scale grouping.
 * bscale = FP8Q_BSCALE_ROW1x128 is the weight-gradient form
 * dW = dY^T X: both operands come from fp8q_quant_act_128x1 (K runs over
 * tokens) and the scale of output (m, n) in K group g is sA[g][m] * sB[g][n];
 * sB is [K/128][N] and must be 16-byte aligned. */
FP8Q_API int fp8q_gemm_ex(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                 void* C, int64_t M, int64_t N, int64_t K, int out_dtype, int bscale,
                 fp8q_stream_t stream);

/* Grouped (MoE) GEMM: "codingmall ... FP8 GEMM" item 8 (dense and MoE
 * support).  Group e owns rows [m_offsets[e], m_offsets[e+1]) of A8 and C and
 * multiplies them by its own weights:
 *   A8  [M_total][K]      sA [K/128][M_total]
 *   B8  [G][N][K]         sB [G][N/128][K/128]
 *   C   [M_total][N]      rows outside every group are not written
 *   m_offsets  DEVICE int32 array of G+1 entries, non-decreasing, each
 *              a multiple of 128, m_offsets[G] <= M_total; checked on the
 *              device (FP8Q_ERR_BAD_GROUPS via fp8q_get_device_status, and
 *              then nothing is written).
 * Requires 1 <= G <= 512, M_total, N, K multiples of 128.  Block scales only. */
FP8Q_API int fp8q_gemm_grouped(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                      void* C, const int* m_offsets, int G, int64_t M_total, int64_t N,
                      int64_t K, int out_dtype, fp8q_stream_t stream);

/* Stream-K workspace.  With a workspace, a GEMM runs on every SM and shares
 * the last partial wave of output tiles (plus one full wave) out by K
 * iterations, so no SM idles at the end; tiles cut between SMs are finished
 * through FP32 partial tiles kept in the workspace.  Results do not depend on
 * the order in which the pieces finish.  When the schedule cuts every tile of
 * a dense GEMM with 128x128-block B scales (few tiles, long K), the call
 * launches a second kernel after the GEMM, on the same stream, that sums the
 * pieces; otherwise the last piece of each cut tile sums them.
 *
 * fp8q_gemm_workspace_size: bytes a workspace must have on the CURRENT device
 * (it depends on the SM count; about 38 MB on a 148-SM B300).  0 on error.
 *
 * The workspace is caller-owned device memory, 256-byte aligned.  Its first
 * 64 * (number of SMs) bytes, rounded up to a multiple of 256, hold arrival
 * counters that must be ZERO before the first call (simplest: cudaMemset the
 * whole workspace once); every call that completes leaves them zero again.
 * After a call that reported a device error, zero them before reusing it.
 * Calls that may run at the same time (different streams) need different
 * workspaces. */
FP8Q_API size_t fp8q_gemm_workspace_size(void);

/* fp8q_gemm_ex with a stream-K workspace (NULL = no workspace: whole tiles
 * only, exactly as fp8q_gemm_ex).  FP8Q_ERR_INVALID_ARG if workspace_bytes is
 * smaller than fp8q_gemm_workspace_size(); FP8Q_ERR_MISALIGNED if the
 * workspace is not 256-byte aligned. */
FP8Q_API int fp8q_gemm_ws(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                 void* C, int64_t M, int64_t N, int64_t K, int out_dtype, int bscale,
                 void* workspace, size_t workspace_bytes, fp8q_stream_t stream);

/* GEMM that quantizes its activations itself: the 1x128 quantization of the
 * BF16 activations happens in the GEMM's producer stage, on the way from
 * global to shared memory, instead of in a separate pass that writes A8 to
 * HBM and reads it back -- woojincopolymer post, para. 4 (the FP8 cast fused
 * with the global-to-shared transfer; the forward activations kept as 1x128
 * FP8 tiles).  The result is that of fp8q_gemm_ws(A8, sA, B8, sB, C, ...)
 * with (A8, sA) = fp8q_quant_act_1x128(A): the quantization follows the same
 * rule bit for bit, and C the same tolerance.
 *   A       [M][K] BF16 activations, 16-byte aligned
 *   B8, sB  [N][K] E4M3 weights with 128x128 block scales [N/128][K/128]
 *   C       [M][N] out_dtype (FP8Q_F32 or FP8Q_BF16), 16-byte aligned
 *   A8_out  [M][K] uint8 (16-byte aligned) and sA_out [K/128][M] float32
 *           (4-byte aligned), or both NULL: when given, the quantized
 *           activations are also written there (the stored forward tiles),
 *           identical to fp8q_quant_act_1x128's output.
 *   workspace, workspace_bytes: the stream-K workspace, as for fp8q_gemm_ws
 *           (NULL: whole tiles only).
 * Requires N a multiple of 256, M and K multiples of 128, and the size
 * limits of fp8q_gemm (FP8Q_ERR_UNSUPPORTED_SHAPE otherwise);
 * FP8Q_ERR_INVALID_ARG if only one of A8_out, sA_out is given. */
FP8Q_API int fp8q_gemm_quant_a(const void* A, const uint8_t* B8, const float* sB, void* C,
                      uint8_t* A8_out, float* sA_out, int64_t M, int64_t N, int64_t K,
                      int out_dtype, void* workspace, size_t workspace_bytes,
                      fp8q_stream_t stream);

/* fp8q_gemm_grouped with a stream-K workspace (same rules as fp8q_gemm_ws). */
FP8Q_API int fp8q_gemm_grouped_ws(const uint8_t* A8, const float* sA, const uint8_t* B8,
                         const float* sB, void* C, const int* m_offsets, int G,
                         int64_t M_total, int64_t N, int64_t K, int out_dtype, void* workspace,
                         size_t workspace_bytes, fp8q_stream_t stream);

/* fp8q_gemm_ws without a caller workspace, for callers that cannot allocate
 * device memory: code that runs inside a framework or plugin whose memory is
 * handed out by someone else (a fixed budget, a caching allocator it cannot
 * reach), or that simply has no allocator of its own.  No counterpart on the
 * pages: this is an engineering convenience of the library, not part of the
 * method.
 *
 * The stream-K workspace lives in a 40 MiB array inside the library, held by
 * every GPU that loads the library until the process exits.  That is enough
 * for a GPU with up to 159 SMs; on a larger GPU the call returns
 * FP8Q_ERR_UNSUPPORTED_SHAPE and launches nothing.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).  It
 * clears the array's arrival counters (an asynchronous memset on `stream`)
 * and then runs exactly as fp8q_gemm_ws.
 *
 * Every call shares the one array per device: calls that may overlap on the
 * GPU (different streams, or host threads, without ordering between them)
 * race and must not be made.  The array's device address is looked up the
 * first time the library is used on a device; make that first call (of any
 * fp8q function) before starting a stream capture. */
FP8Q_API int fp8q_gemm_noalloc(const uint8_t* A8, const float* sA, const uint8_t* B8,
                      const float* sB, void* C, int64_t M, int64_t N, int64_t K, int out_dtype,
                      int bscale, fp8q_stream_t stream);

/* ------------------------------------------ expert-parallel MoE data path */

/* FP8 dispatch and BF16 combine around the grouped GEMM for experts spread
 * over ranks: "Six Reasons...", para. 4 (the activations are quantized to
 * FP8 before they are dispatched to the experts' up projection; the combine
 * stays in BF16).  Experts are numbered rank-major: rank d owns experts
 * d*E_local .. (d+1)*E_local - 1 of E = ranks * E_local.  A rank
 *   1. quantizes its tokens x[T][H] per 1x128 tile (fp8q_quant_act_1x128);
 *   2. fp8q_ep_route: counts per expert and, for every (token, slot), the
 *      row it takes in the send order (expert-major, then token, then slot);
 *   3. fp8q_ep_pack: one packed row per (token, slot) -- the token's H E4M3
 *      bytes, then its H/128 FP32 scales, padded to fp8q_ep_row_bytes(H);
 *   4. sends the rows of each destination's experts to it and receives, from
 *      every source rank in turn, that rank's rows for each local expert
 *      (an all-to-all of packed rows: the caller's collective);
 *   5. fp8q_ep_unpack: received rows -> the grouped GEMM's A8 [Mp][H] and
 *      sA [H/128][Mp], each local expert's rows contiguous and padded with
 *      zero rows to a multiple of 128;
 *   6. fp8q_gemm_grouped_ws with the local experts' weights -> Y [Mp][N] BF16;
 *   7. fp8q_ep_gather: Y's rows back in the order they arrived, and the
 *      reverse all-to-all returns them to their source ranks;
 *   8. fp8q_ep_combine: out[t] = bf16(sum_j w[t][j] * y_tj), FP32 sum.
 * The receive layout tables (per source and local expert: start of its rows
 * in the receive order, src_off[b], and in A8, dest_base[b], b = w*E_local +
 * e; per local expert: m_offsets and rows_e, the real row count) are small
 * and made by the caller from the exchanged counts. */

/* Bytes of one packed dispatch row for hidden size H (a multiple of 128):
 * H + 4*H/128 rounded up to a multiple of 16.  -1 for an invalid H. */
FP8Q_API int64_t fp8q_ep_row_bytes(int64_t H);

/* topk_ids [T][k] int32 (device) -> counts [E] int32 and pos [T][k] int32:
 * pos[t][j] = (rows of experts below e) + (entries of expert e before (t, j)
 * in row-major order), e = topk_ids[t][j]; deterministic.  One CTA.
 * Requires 1 <= E <= 256 and T*k < 2^31; an id outside [0, E) records
 * FP8Q_ERR_BAD_ROUTING in the device status and nothing is written. */
FP8Q_API int fp8q_ep_route(const int32_t* topk_ids, int64_t T, int k, int E, int32_t* counts,
                  int32_t* pos, fp8q_stream_t stream);

/* q [T][H] uint8, s [H/128][T] float32 (fp8q_quant_act_1x128's output),
 * pos [T][k] -> send [T*k][fp8q_ep_row_bytes(H)]: row pos[t][j] gets token
 * t's bytes and scales.  q and send 16-byte aligned; H a multiple of 128. */
FP8Q_API int fp8q_ep_pack(const uint8_t* q, const float* s, const int32_t* pos, int64_t T, int k,
                 int64_t H, uint8_t* send, fp8q_stream_t stream);

/* recv [R][fp8q_ep_row_bytes(H)] -> A8 [Mp][H] uint8 and sA [H/128][Mp]
 * float32: received row i of block b (src_off[b] <= i < src_off[b+1], nb
 * blocks) goes to row dest_base[b] + i - src_off[b]; then the padding rows
 * of each local expert e (m_offsets[e] + rows_e[e] .. m_offsets[e+1] - 1,
 * fewer than 128) are zeroed.  Tables are DEVICE int64 arrays (src_off has
 * nb + 1 entries, m_offsets El + 1).  Mp = m_offsets[El], a multiple of 128. */
FP8Q_API int fp8q_ep_unpack(const uint8_t* recv, int64_t R, int64_t H, const int64_t* src_off,
                   const int64_t* dest_base, int nb, const int64_t* m_offsets,
                   const int64_t* rows_e, int El, uint8_t* A8, float* sA, int64_t Mp,
                   fp8q_stream_t stream);

/* Y [Mp][N] BF16 -> out [R][N] BF16 in the receive order: out[i] =
 * Y[dest_base[b] + i - src_off[b]].  N a multiple of 8, 16-byte aligned.
 * A table entry pointing outside Y's Mp rows records FP8Q_ERR_BAD_ROUTING
 * and that row is skipped (the same holds for fp8q_ep_unpack's rows and
 * fp8q_ep_combine's positions). */
FP8Q_API int fp8q_ep_gather(const void* Y, int64_t Mp, int64_t R, int64_t N, const int64_t* src_off,
                   const int64_t* dest_base, int nb, void* out, fp8q_stream_t stream);

/* back [T*k][N] BF16 (the returned expert results, in the send order), pos
 * [T][k], w [T][k] float32 gate weights -> out [T][N] BF16:
 * out[t][n] = bf16(sum_{j=0..k-1} w[t][j] * back[pos[t][j]][n]), summed in
 * FP32 in slot order, rounded to nearest even.  N a multiple of 8. */
FP8Q_API int fp8q_ep_combine(const void* back, const int32_t* pos, const float* w, int64_t T,
                    int k, int64_t N, void* out, fp8q_stream_t stream);

/* ------------------------------------------------------------------ status */

/* Synchronizes `stream`, returns the sticky device status of the current
 * device (FP8Q_OK if no kernel recorded a problem) and clears it. */
FP8Q_API int fp8q_get_device_status(fp8q_stream_t stream);

/* Diagnostic of the device-side failure detection: launches one warp that
 * waits on a barrier nothing arrives on, through the bounded wait every GEMM
 * pipeline stage uses, with a time limit of limit_ns (1 .. 100,000,000 ns).
 * The wait runs out, FP8Q_ERR_TIMEOUT is recorded in the sticky device
 * status (read it with fp8q_get_device_status), and the kernel returns: the
 * GPU and the CUDA context stay usable.  FP8Q_ERR_INVALID_ARG for a limit out
 * of range.  Not part of the method; used by the library's tests. */
FP8Q_API int fp8q_selftest_wait(int64_t limit_ns, fp8q_stream_t stream);

/* Tensor-pipe throughput probe, a measurement aid (no counterpart on the
 * pages): one CTA per SM issues `blocks` x 4 back-to-back
 * tcgen05.mma.kind::f8f6f4 of shape 128 x 256 x 32 (E4M3 in, FP32 out) from
 * fixed shared-memory operands into TMEM, then waits for them.  The work is
 * fp8q_num_sms() * blocks * 2 * 128 * 256 * 128 flops; timing the launch with
 * CUDA events on `stream` gives the dense FP8 rate the GEMM's roofline is
 * compared with.  1 <= blocks <= 2^20 (FP8Q_ERR_INVALID_ARG otherwise; at
 * 2^20 the launch runs about a quarter of a second).
 * Nothing is read or written in global memory. */
FP8Q_API int fp8q_bench_mma_peak(int64_t blocks, fp8q_stream_t stream);

/* Number of SMs of the current device (negative fp8q_status on error). */
FP8Q_API int fp8q_num_sms(void);

/* Static, human-readable name of a status code. */
FP8Q_API const char* fp8q_status_string(int status);

/* Library version: major*10000 + minor*100 + patch. */
FP8Q_API int fp8q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
