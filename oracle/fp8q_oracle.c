/*
 * fp8q oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the fine-grained FP8
 * path computes: an E4M3 codec, online tile-wise quantization (1x128, 128x1,
 * 128x128), a block-scaled GEMM on dequantized values in FP64, an exact integer
 * cross-check of that GEMM, and an emulator of limited-precision accumulation.
 *
 * Only the test-suite, the package's smoke check and the benchmark's CPU
 * baseline may load this library.  It shares no code, header, table or
 * constant generator with the CUDA library, and the CUDA path never calls it.
 *
 * Sources (web pages on DeepSeek-V3 FP8 training):
 *   [P1] "Six Reasons Deepseek Ai Is A Waste Of Time" (myomija.com board post),
 *        paragraphs 1-4.
 *   [P3] codingmall.com knowledge-base article on FP8 in DeepSeek-V3 (Greek),
 *        sections "fine-grained quantization", "online quantization",
 *        "increased accumulation precision", "unified E4M3 format".
 *   [P4] codingmall.com knowledge-base article on FP8 GEMM in DeepSeek-V3
 *        (Japanese), numbered items 1-8.
 * The E4M3 bit layout itself is not printed on the pages; it is the OCP 8-bit
 * floating-point definition (bias 7, no infinities, S.1111.111 = NaN).
 *
 * Readings taken where the pages are silent:
 *   - max representable E4M3 value = 448; cast = round-to-nearest-even with
 *     saturation to +-448; NaN -> 0x7F; the sign of zero is kept.
 *   - tile scale s = fl32(amax / 448); elements are multiplied by
 *     inv = fl32(448 / amax) and then cast.  amax == 0 -> s = 1, inv = 1.
 *     inv overflowing FP32 (amax below ~1.3e-36) is clamped to FLT_MAX.
 *   - dimensions that are not multiples of 128 form a partial last tile whose
 *     amax runs over the elements that exist.
 *   - 128x128 weight blocks are 128 rows of W[N][K] by 128 columns of K.
 *   - the 128x1 variant groups 128 consecutive tokens of one channel and is
 *     written transposed: qT[C][T], sT[ceil(T/128)][C].
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (no FMA contraction, IEEE single-precision float arithmetic on x86-64 SSE).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define FPO_GROUP 128
#define FPO_E4M3_MAX 448.0f

static int64_t fpo_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* ------------------------------------------------------------------ codec */

/* [P1] para. 1 and [P3] "unified E4M3 format": every tensor is stored as E4M3
 * (4 exponent bits, 3 mantissa bits).  Value of one byte, following the OCP
 * definition: normal  (-1)^s * 2^(e-7) * (1 + m/8)  for e in 1..15
 * (except e=15, m=7 which is NaN); subnormal (-1)^s * 2^-6 * (m/8) for e = 0. */
double fpo_e4m3_decode(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even with saturation, by brute force: the magnitude is
 * compared with the sorted list of all 127 non-negative finite E4M3 values
 * (byte codes 0x00..0x7E, whose decoded values increase with the code).  The
 * bracketing pair [lo, hi] is found by exact comparison; the value goes to
 * the nearer one, and an exact tie (|v| equal to the midpoint, which is exact
 * in double) goes to the even code, i.e. the even mantissa. */
uint8_t fpo_e4m3_encode(float v)
{
    uint8_t sign;
    double a;
    int code;
    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs((double)v);
    if (a >= (double)FPO_E4M3_MAX)          /* saturate, also for +-Inf */
        return (uint8_t)(sign | 0x7E);
    for (code = 0; code < 0x7E; ++code) {
        double lo = fpo_e4m3_decode((uint8_t)code);
        double hi = fpo_e4m3_decode((uint8_t)(code + 1));
        if (a >= lo && a < hi) {
            double mid = 0.5 * (lo + hi);
            int pick;
            if (a < mid)
                pick = code;
            else if (a > mid)
                pick = code + 1;
            else
                pick = (code % 2 == 0) ? code : code + 1;
            return (uint8_t)(sign | pick);
        }
    }
    return (uint8_t)(sign | 0x7E);           /* not reached */
}

void fpo_e4m3_decode_array(const uint8_t* b, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fpo_e4m3_decode(b[i]);
}

void fpo_e4m3_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fpo_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------ tile scale */

/* [P1] para. 1: the largest magnitude of the group is mapped onto the largest
 * representable FP8 value; [P3] "online quantization" and [P4] item 7: the
 * factor is computed from the current tile, with no history of maxima. */
void fpo_tile_scale(float amax, float* s, float* inv)
{
    float iv;
    if (amax == 0.0f) {
        *s = 1.0f;
        *inv = 1.0f;
        return;
    }
    *s = amax / FPO_E4M3_MAX;
    iv = FPO_E4M3_MAX / amax;
    if (isinf(iv))
        iv = FLT_MAX;
    *inv = iv;
}

/* ------------------------------------------------------------- quantizers */

/* [P1] para. 3 ("Figure 7 (a)", item 1) and [P3] "fine-grained quantization":
 * activations are grouped and scaled per token per 128 channels.
 * x[M][K] row-major; q[M][K]; s[Kb][M] with Kb = ceil(K/128). */
void fpo_quant_1x128(const float* x, int64_t M, int64_t K, uint8_t* q, float* s)
{
    int64_t Kb = fpo_ceil_div(K, FPO_GROUP);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < Kb; ++g) {
            int64_t k0 = g * FPO_GROUP;
            int64_t k1 = k0 + FPO_GROUP < K ? k0 + FPO_GROUP : K;
            float amax = 0.0f, sc, inv;
            for (int64_t k = k0; k < k1; ++k) {
                float a = fabsf(x[m * K + k]);
                if (a > amax)
                    amax = a;
            }
            fpo_tile_scale(amax, &sc, &inv);
            s[g * M + m] = sc;
            for (int64_t k = k0; k < k1; ++k) {
                float y = x[m * K + k] * inv;
                q[m * K + k] = fpo_e4m3_encode(y);
            }
        }
    }
}

/* [P1] para. 3: in the backward pass activations are regrouped from 1x128 to
 * 128x1 tiles, i.e. 128 consecutive tokens of one channel share a scale.
 * x[T][C] row-major; output is transposed: qT[C][T], sT[Tb][C], Tb = ceil(T/128). */
void fpo_quant_128x1(const float* x, int64_t T, int64_t C, uint8_t* qT, float* sT)
{
    int64_t Tb = fpo_ceil_div(T, FPO_GROUP);
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t tb = 0; tb < Tb; ++tb) {
            int64_t t0 = tb * FPO_GROUP;
            int64_t t1 = t0 + FPO_GROUP < T ? t0 + FPO_GROUP : T;
            float amax = 0.0f, sc, inv;
            for (int64_t t = t0; t < t1; ++t) {
                float a = fabsf(x[t * C + c]);
                if (a > amax)
                    amax = a;
            }
            fpo_tile_scale(amax, &sc, &inv);
            sT[tb * C + c] = sc;
            for (int64_t t = t0; t < t1; ++t) {
                float y = x[t * C + c] * inv;
                qT[c * T + t] = fpo_e4m3_encode(y);
            }
        }
    }
}

/* [P1] para. 3 (item 2) and [P3] "fine-grained quantization": weights are
 * grouped and scaled per 128 input channels x 128 output channels.
 * w[N][K] row-major; q[N][K]; s[Nb][Kb]. */
void fpo_quant_128x128(const float* w, int64_t N, int64_t K, uint8_t* q, float* s)
{
    int64_t Nb = fpo_ceil_div(N, FPO_GROUP), Kb = fpo_ceil_div(K, FPO_GROUP);
    for (int64_t nb = 0; nb < Nb; ++nb) {
        for (int64_t g = 0; g < Kb; ++g) {
            int64_t n0 = nb * FPO_GROUP, n1 = n0 + FPO_GROUP < N ? n0 + FPO_GROUP : N;
            int64_t k0 = g * FPO_GROUP, k1 = k0 + FPO_GROUP < K ? k0 + FPO_GROUP : K;
            float amax = 0.0f, sc, inv;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float a = fabsf(w[n * K + k]);
                    if (a > amax)
                        amax = a;
                }
            fpo_tile_scale(amax, &sc, &inv);
            s[nb * Kb + g] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k1; ++k) {
                    float y = w[n * K + k] * inv;
                    q[n * K + k] = fpo_e4m3_encode(y);
                }
        }
    }
}

/* [P1] para. 3: in the backward pass the activations are converted from 1x128
 * tiles to 128x1 tiles; with the forward pass's quantized activations stored
 * as 1x128 FP8 tiles ([P2] para. 4), the conversion starts from those tiles.
 * Each stored element is dequantized -- decode(q) * s, the decode exact in
 * float and the product one correctly rounded FP32 multiplication -- and the
 * dequantized tensor is quantized per 128 tokens of one channel exactly as
 * fpo_quant_128x1 does, written transposed.
 * q[T][C], s[ceil(C/128)][T] -> qT[C][T], sT[ceil(T/128)][C]. */
void fpo_retile_1x128_to_128x1(const uint8_t* q, const float* s, int64_t T, int64_t C,
                               uint8_t* qT, float* sT)
{
    float* x = (float*)malloc((size_t)(T * C) * sizeof(float));
    if (!x)
        return;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            float d = (float)fpo_e4m3_decode(q[t * C + c]);
            x[t * C + c] = d * s[(c / FPO_GROUP) * T + t];
        }
    fpo_quant_128x1(x, T, C, qT, sT);
    free(x);
}

/* ---------------------------------------------------- SwiGLU + FP8 cast */

/* [P2] para. 4: the SwiGLU operator's inputs are cached and its output is
 * recomputed in the backward pass; forward activations are stored as 1x128
 * FP8 tiles.  [P2] para. 3: fusing the FP8 cast into the operator that
 * produces the activation.  SwiGLU(g, u) = silu(g) * u with
 * silu(g) = g * sigmoid(g) = g / (1 + e^-g).  Evaluated here in FP64 for each
 * of the n elements of g and u (FP32, widened from BF16 by the caller); the
 * fused quantization is fpo_quant_1x128 applied to the FP64 result rounded
 * once to FP32 (the wrapper does that step). */
void fpo_swiglu_f64(const float* g, const float* u, int64_t n, double* h)
{
    for (int64_t i = 0; i < n; ++i) {
        double gi = (double)g[i];
        h[i] = gi * (double)u[i] / (1.0 + exp(-gi));
    }
}

/* --------------------------------------------------- RMSNorm + FP8 cast */

/* [P2] para. 3: a warp-level cast instruction is proposed so that layer
 * normalization and the FP8 cast can be fused.  DeepSeek-V3's normalization
 * is RMSNorm: y[m][k] = x[m][k] * w[k] / sqrt(mean_k x[m][k]^2 + eps).
 * Evaluated here in FP64 for each row of x[M][K] (FP32, widened from BF16 by
 * the caller), weights w[K]; the fused quantization is fpo_quant_1x128
 * applied to the FP64 result rounded once to FP32 (the wrapper does that). */
void fpo_rmsnorm_f64(const float* x, const float* w, int64_t M, int64_t K, double eps, double* y)
{
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)x[m * K + k];
            ss += v * v;
        }
        double rms = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            y[m * K + k] = (double)x[m * K + k] * (double)w[k] / rms;
    }
}

/* ------------------------------------------------------------------- GEMM */

/* Scale of operand B for output column n and K group g.
 * bmode 0: 128x128 weight blocks, sB[Nb][Kb].
 * bmode 1: B quantized per 1x128 tile in its own rows (the weight-gradient
 *          case, both operands regrouped along tokens), sB[Kb][N]. */
static double fpo_scale_b(const float* sB, int bmode, int64_t N, int64_t Kb, int64_t n, int64_t g)
{
    if (bmode == 0)
        return (double)sB[(n / FPO_GROUP) * Kb + g];
    return (double)sB[g * N + n];
}

/* [P1] paras. 1-2: the GEMM takes FP8 inputs; the per-group factors along the
 * inner dimension K are multiplied in as dequantization; output BF16/FP32.
 * Here every element is dequantized (decode * its group's scale) and
 * C[m][n] = sum_k Ad[m][k] * Bd[n][k] is summed in FP64 in k order.
 * Cabs[m][n] = sum_k |Ad[m][k] * Bd[n][k]| (the tolerance's yardstick).
 * A8[M][K], sA[Kb][M] (entry g*lda_s + m, lda_s = row count of the scale
 * array), B8[N][K].  One output entry: */
static void fpo_entry(const uint8_t* A8, const float* sA, int64_t lda_s, int64_t arow,
                      const uint8_t* B8, const float* sB, int bmode, int64_t N, int64_t n,
                      int64_t K, double* c, double* cabs)
{
    int64_t Kb = fpo_ceil_div(K, FPO_GROUP);
    double acc = 0.0, aacc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        int64_t g = k / FPO_GROUP;
        double a = fpo_e4m3_decode(A8[arow * K + k]) * (double)sA[g * lda_s + arow];
        double b = fpo_e4m3_decode(B8[n * K + k]) * fpo_scale_b(sB, bmode, N, Kb, n, g);
        double p = a * b;
        acc += p;
        aacc += fabs(p);
    }
    *c = acc;
    *cabs = aacc;
}

static int fpo_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Dense GEMM, all entries.  C and Cabs are [M][N]. */
void fpo_gemm_f64(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB, int bmode,
                  int64_t M, int64_t N, int64_t K, double* C, double* Cabs, int nthreads)
{
    int nt = fpo_threads(nthreads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            fpo_entry(A8, sA, M, m, B8, sB, bmode, N, n, K, &C[m * N + n], &Cabs[m * N + n]);
}

/* Dense GEMM, selected entries (mi[i], ni[i]). */
void fpo_gemm_f64_entries(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                          int bmode, int64_t M, int64_t N, int64_t K, const int64_t* mi,
                          const int64_t* ni, int64_t count, double* C, double* Cabs, int nthreads)
{
    int nt = fpo_threads(nthreads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
    for (int64_t i = 0; i < count; ++i)
        fpo_entry(A8, sA, M, mi[i], B8, sB, bmode, N, ni[i], K, &C[i], &Cabs[i]);
}

/* [P4] item 8: dense and MoE (grouped) GEMMs.  Group e owns rows
 * [m_offsets[e], m_offsets[e+1]) of A8[Mtot][K] and C[Mtot][N], and multiplies
 * them by its own weights B8[e][N][K] with block scales sB[e][Nb][Kb].
 * sA is [Kb][Mtot].  Rows outside every group are left untouched. */
void fpo_gemm_grouped_f64(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                          const int64_t* m_offsets, int64_t G, int64_t Mtot, int64_t N, int64_t K,
                          double* C, double* Cabs, int nthreads)
{
    int64_t Nb = fpo_ceil_div(N, FPO_GROUP), Kb = fpo_ceil_div(K, FPO_GROUP);
    int nt = fpo_threads(nthreads);
    (void)nt;
    for (int64_t e = 0; e < G; ++e) {
        const uint8_t* Be = B8 + e * N * K;
        const float* sBe = sB + e * Nb * Kb;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
        for (int64_t m = m_offsets[e]; m < m_offsets[e + 1]; ++m)
            for (int64_t n = 0; n < N; ++n)
                fpo_entry(A8, sA, Mtot, m, Be, sBe, 0, N, n, K, &C[m * N + n], &Cabs[m * N + n]);
    }
}

/* Grouped GEMM, selected entries: rows mi[i] (global row index), columns ni[i]. */
void fpo_gemm_grouped_f64_entries(const uint8_t* A8, const float* sA, const uint8_t* B8,
                                  const float* sB, const int64_t* m_offsets, int64_t G, int64_t Mtot,
                                  int64_t N, int64_t K, const int64_t* mi, const int64_t* ni,
                                  int64_t count, double* C, double* Cabs, int nthreads)
{
    int64_t Nb = fpo_ceil_div(N, FPO_GROUP), Kb = fpo_ceil_div(K, FPO_GROUP);
    int nt = fpo_threads(nthreads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 16) num_threads(nt)
    for (int64_t i = 0; i < count; ++i) {
        int64_t e = -1;
        for (int64_t j = 0; j < G; ++j)
            if (mi[i] >= m_offsets[j] && mi[i] < m_offsets[j + 1])
                e = j;
        if (e < 0) {
            C[i] = NAN;
            Cabs[i] = NAN;
            continue;
        }
        fpo_entry(A8, sA, Mtot, mi[i], B8 + e * N * K, sB + e * Nb * Kb, 0, N, ni[i], K, &C[i],
                  &Cabs[i]);
    }
}

/* ----------------------------------------------------- exact cross-check */

/* Integer value of an E4M3 byte in units of 2^-9 (every finite E4M3 value is
 * an integer multiple of 2^-9), taken straight from the bit fields:
 * subnormal m * 2^-9; normal (8 + m) * 2^(e-1) * 2^-9.  NaN -> 0. */
static int64_t fpo_e4m3_units(uint8_t b)
{
    int e = (b >> 3) & 0xF, m = b & 7;
    int64_t v;
    if (e == 0xF && m == 7)
        return 0;
    v = (e == 0) ? (int64_t)m : ((int64_t)(8 + m) << (e - 1));
    return (b & 0x80) ? -v : v;
}

/* Same result as fpo_gemm_f64 by an independent route: within each K group
 * the FP8 dot product is summed exactly as an int64 count of 2^-18 units,
 * then C = sum_g sA * sB * S_g * 2^-18 in FP64.  [P1] para. 2: the factors are
 * per group along K, so they can be applied once per group. */
void fpo_gemm_exact_int(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                        int bmode, int64_t M, int64_t N, int64_t K, double* C, int nthreads)
{
    int64_t Kb = fpo_ceil_div(K, FPO_GROUP);
    int nt = fpo_threads(nthreads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t g = 0; g < Kb; ++g) {
                int64_t k0 = g * FPO_GROUP, k1 = k0 + FPO_GROUP < K ? k0 + FPO_GROUP : K;
                int64_t S = 0;
                for (int64_t k = k0; k < k1; ++k)
                    S += fpo_e4m3_units(A8[m * K + k]) * fpo_e4m3_units(B8[n * K + k]);
                acc += (double)sA[g * M + m] * fpo_scale_b(sB, bmode, N, Kb, n, g) *
                       ldexp((double)S, -18);
            }
            C[m * N + n] = acc;
        }
    }
}

/* ------------------------------------------- limited-accumulation emulator */

/* Keep `mbits` fraction bits after the leading one, truncating toward zero. */
static double fpo_trunc_bits(double x, int mbits)
{
    int e;
    if (x == 0.0 || !isfinite(x))
        return x;
    e = ilogb(x);
    return ldexp(trunc(ldexp(x, mbits - e)), e - mbits);
}

/* [P1] paras. 2-3 and [P3] "increased accumulation precision": the tensor
 * cores accumulate with a limited bit width; without promotion the error at
 * K = 4096 reaches ~2%, and copying partial sums to FP32 registers at a fixed
 * interval fixes it.  The pages give no model of the hardware, so this is a
 * two-knob stand-in: products (dequantized, FP64) are summed exactly in chunks
 * of `chunk` consecutive k, and each chunk sum is added to an accumulator that
 * is truncated to `mbits` fraction bits after every addition.
 * promote == 0: one such accumulator runs over the first `kmax` elements of K
 *               (no promotion).
 * promote  > 0: the accumulator restarts from zero every `promote` elements of
 *               K and each partial is added to an FP64 total (promotion).
 * Only the first kmax (<= K) elements of K take part.  C is [M][N]. */
void fpo_gemm_trunc_emu(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                        int bmode, int64_t M, int64_t N, int64_t K, int64_t kmax, int chunk,
                        int mbits, int promote, double* C, int nthreads)
{
    int64_t Kb = fpo_ceil_div(K, FPO_GROUP);
    int nt = fpo_threads(nthreads);
    (void)nt;
    if (kmax > K)
        kmax = K;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double total = 0.0, acc = 0.0;
            for (int64_t k0 = 0; k0 < kmax; k0 += chunk) {
                double part = 0.0;
                int64_t k1 = k0 + chunk < kmax ? k0 + chunk : kmax;
                if (promote > 0 && k0 > 0 && k0 % promote == 0) {
                    total += acc;
                    acc = 0.0;
                }
                for (int64_t k = k0; k < k1; ++k) {
                    int64_t g = k / FPO_GROUP;
                    double a = fpo_e4m3_decode(A8[m * K + k]) * (double)sA[g * M + m];
                    double b = fpo_e4m3_decode(B8[n * K + k]) * fpo_scale_b(sB, bmode, N, Kb, n, g);
                    part += a * b;
                }
                acc = fpo_trunc_bits(acc + part, mbits);
            }
            C[m * N + n] = total + acc;
        }
    }
}

/* Reference helper for the FP64 sum over the same first kmax elements. */
void fpo_gemm_f64_prefix(const uint8_t* A8, const float* sA, const uint8_t* B8, const float* sB,
                         int bmode, int64_t M, int64_t N, int64_t K, int64_t kmax, double* C,
                         int nthreads)
{
    int64_t Kb = fpo_ceil_div(K, FPO_GROUP);
    int nt = fpo_threads(nthreads);
    (void)nt;
    if (kmax > K)
        kmax = K;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < kmax; ++k) {
                int64_t g = k / FPO_GROUP;
                double a = fpo_e4m3_decode(A8[m * K + k]) * (double)sA[g * M + m];
                double b = fpo_e4m3_decode(B8[n * K + k]) * fpo_scale_b(sB, bmode, N, Kb, n, g);
                acc += a * b;
            }
            C[m * N + n] = acc;
        }
}

int fpo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
