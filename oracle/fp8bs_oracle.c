/*
 * CPU oracle for the fine-grained FP8 GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this file's library; the product path
 * (the CUDA library and its Python binding) never does, and shares no code,
 * header, table or constant with it.
 *
 * Plain and slow on purpose: one function per step, each step written from
 * its definition, no blocking, no vectorisation, no reordering.
 *
 * Sources followed:
 *  - FP8 grouping: activations in 1x128 tiles (one scale per token per 128
 *    channels), weights in 128x128 blocks (per 128 input x 128 output
 *    channels) -- "personal notes concerning the deepseek core readings"
 *    (why-be.why-be.co.kr), fine-grained quantization paragraph, Figure 7(a).
 *  - Scale: the group's maximum magnitude is mapped onto the largest value
 *    FP8 can represent, and the tensor is quantized online with that factor
 *    -- Q&A post on xn--9g3bo1gtkw0l8ubf92bgle.kr, mixed-precision paragraph
 *    (amax scaling, online quantization).
 *  - The FP8 variant (E4M3), s = amax/448 in FP32 with s = 1 when amax = 0,
 *    and round-to-nearest-even with saturation are fixed by the build's
 *    statement of the problem; the E4M3 encoding is the OCP 8-bit floating
 *    point format (E4M3 "FN": bias 7, no infinity, NaN = S.1111.111).
 *
 * Build: plain C11, no fast-math, no FP contraction, so that every float
 * operation below is one correctly rounded IEEE binary32 operation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* E4M3 codec, from the format definition.                                 */
/* ---------------------------------------------------------------------- */

/* Largest finite E4M3 magnitude: exponent field 15, mantissa 6 -> 1.75*2^8. */
#define FP8O_E4M3_MAX 448.0

/* Value of an E4M3 code. Exponent field e (bias 7) and mantissa m:
 *   e == 0          : subnormal, m * 2^-9
 *   e == 15, m == 7 : NaN
 *   otherwise       : (1 + m/8) * 2^(e-7)                                   */
double fp8o_e4m3_decode(uint8_t code)
{
    int neg = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return neg ? -mag : mag;
}

/* Bit pattern of an exactly representable, non-negative E4M3 magnitude v. */
static uint8_t fp8o_e4m3_pattern(double v)
{
    int ex, e, m;
    if (v == 0.0)
        return 0;
    if (v < ldexp(1.0, -6))                 /* subnormal: v = m * 2^-9 */
        return (uint8_t)(v / ldexp(1.0, -9));
    frexp(v, &ex);                          /* v = f * 2^ex, f in [0.5, 1) */
    e = ex - 1;                             /* v = (1 + m/8) * 2^e */
    m = (int)((v / ldexp(1.0, e) - 1.0) * 8.0);
    return (uint8_t)(((e + 7) << 3) | m);
}

/* Round a finite binary32 y to E4M3: nearest grid value, ties to the even
 * mantissa, then saturate magnitudes above 448 to 448. The sign is kept,
 * so negative values that round to zero give the code of -0 (0x80).
 * The grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3); below 2^-6 the
 * subnormals keep the spacing 2^-9. */
uint8_t fp8o_e4m3_encode(float y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    int ex, e;
    double quantum, n, v;
    if (a == 0.0)
        return sign;
    frexp(a, &ex);
    e = ex - 1;                             /* floor(log2(a)) */
    if (e < -6)
        e = -6;
    quantum = ldexp(1.0, e - 3);
    n = nearbyint(a / quantum);             /* exact division by 2^k; ties to even */
    v = n * quantum;
    if (v > FP8O_E4M3_MAX)
        v = FP8O_E4M3_MAX;                  /* saturate */
    return sign | fp8o_e4m3_pattern(v);
}

/* ---------------------------------------------------------------------- */
/* Quantizers.                                                             */
/* ---------------------------------------------------------------------- */

static float fp8o_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;         /* bf16 is the top half of binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Dequantisation multiplier of one group: s = amax / 448 in binary32
 * (correctly rounded division), or 1 when the group is all zeros. */
float fp8o_group_scale(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
    return amax / 448.0f;
}

/* Power-of-two scale (the scale mode Blackwell's UE8M0 microscaling formats
 * can hold): the smallest s = 2^e, -127 <= e <= 127, with amax / s <= 448,
 * i.e. 2^e >= amax / 448 as real numbers; s = 1 when amax = 0. Found by a
 * plain upward search over e with the exact comparison amax <= 448 * 2^e
 * (both sides exact in binary64). */
float fp8o_group_scale_pow2(float amax)
{
    int e = -127;
    if (amax == 0.0f)
        return 1.0f;
    while (e < 127 && (double)amax > ldexp(448.0, e))
        ++e;
    return ldexpf(1.0f, e);
}

typedef float (*fp8o_scale_fn)(float amax);

/* One element: q = E4M3(x / s), with x / s a correctly rounded binary32
 * division followed by the E4M3 rounding (two roundings, by definition). */
uint8_t fp8o_quantize_value(float x, float s)
{
    float y = x / s;
    return fp8o_e4m3_encode(y);
}

/* Activations, 1x128 tiles: x is bf16 [M, K] with row stride ldx (elements);
 * q is [M, K] with row stride ldq (bytes); scale is [M, K/128] row-major.
 * K must be a multiple of 128. */
static void fp8o_act_tiles(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                           int64_t ldq, float *scale, fp8o_scale_fn group_scale)
{
    int64_t G = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const uint16_t *xg = x + m * ldx + g * 128;
            uint8_t *qg = q + m * ldq + g * 128;
            float amax = 0.0f, s;
            for (int k = 0; k < 128; ++k) {
                float v = fabsf(fp8o_bf16_to_f32(xg[k]));
                if (v > amax)
                    amax = v;
            }
            s = group_scale(amax);
            scale[m * G + g] = s;
            for (int k = 0; k < 128; ++k)
                qg[k] = fp8o_quantize_value(fp8o_bf16_to_f32(xg[k]), s);
        }
    }
}

void fp8o_quantize_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *q, int64_t ldq, float *scale)
{
    fp8o_act_tiles(x, M, K, ldx, q, ldq, scale, fp8o_group_scale);
}

/* The same tiles with power-of-two scales. */
void fp8o_quantize_act_1x128_pow2(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t *q, int64_t ldq, float *scale)
{
    fp8o_act_tiles(x, M, K, ldx, q, ldq, scale, fp8o_group_scale_pow2);
}

/* Weights, 128x128 blocks: w is bf16 [N, K] (output channel x input channel)
 * with row stride ldw; q is [N, K] with row stride ldq; scale is
 * [ceil(N/128), K/128] row-major. The last row block is partial when N is
 * not a multiple of 128; only rows that exist enter its amax. */
static void fp8o_weight_blocks(const uint16_t *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q,
                               int64_t ldq, float *scale, fp8o_scale_fn group_scale)
{
    int64_t G = K / 128;
    int64_t NB = (N + 127) / 128;
    for (int64_t nb = 0; nb < NB; ++nb) {
        int64_t n_end = (nb + 1) * 128 < N ? (nb + 1) * 128 : N;
        for (int64_t g = 0; g < G; ++g) {
            float amax = 0.0f, s;
            for (int64_t n = nb * 128; n < n_end; ++n)
                for (int k = 0; k < 128; ++k) {
                    float v = fabsf(fp8o_bf16_to_f32(w[n * ldw + g * 128 + k]));
                    if (v > amax)
                        amax = v;
                }
            s = group_scale(amax);
            scale[nb * G + g] = s;
            for (int64_t n = nb * 128; n < n_end; ++n)
                for (int k = 0; k < 128; ++k)
                    q[n * ldq + g * 128 + k] =
                        fp8o_quantize_value(fp8o_bf16_to_f32(w[n * ldw + g * 128 + k]), s);
        }
    }
}

void fp8o_quantize_weight_128x128(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                  uint8_t *q, int64_t ldq, float *scale)
{
    fp8o_weight_blocks(w, N, K, ldw, q, ldq, scale, fp8o_group_scale);
}

/* The same blocks with power-of-two scales. */
void fp8o_quantize_weight_128x128_pow2(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                                       uint8_t *q, int64_t ldq, float *scale)
{
    fp8o_weight_blocks(w, N, K, ldw, q, ldq, scale, fp8o_group_scale_pow2);
}

/* Element-wise form used by exhaustive sweeps: codes of x[i] under the
 * scale of amax[i] (power-of-two scales when pow2 != 0). */
void fp8o_quantize_pairs_mode(const uint16_t *amax_bf16, const uint16_t *x_bf16, int64_t n,
                              uint8_t *q, float *scale, int pow2)
{
    for (int64_t i = 0; i < n; ++i) {
        float a = fp8o_bf16_to_f32(amax_bf16[i]);
        float s = pow2 ? fp8o_group_scale_pow2(a) : fp8o_group_scale(a);
        scale[i] = s;
        q[i] = fp8o_quantize_value(fp8o_bf16_to_f32(x_bf16[i]), s);
    }
}

void fp8o_quantize_pairs(const uint16_t *amax_bf16, const uint16_t *x_bf16, int64_t n,
                         uint8_t *q, float *scale)
{
    for (int64_t i = 0; i < n; ++i) {
        float s = fp8o_group_scale(fp8o_bf16_to_f32(amax_bf16[i]));
        scale[i] = s;
        q[i] = fp8o_quantize_value(fp8o_bf16_to_f32(x_bf16[i]), s);
    }
}
