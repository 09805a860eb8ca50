/*
 * rmsq_oracle.c -- CPU oracle for the fused residual-add + RMSNorm + dynamic FP8 / NVFP4 / MXFP4
 * quantisation of a [rows x hidden] activation.
 *
 * TEST INFRASTRUCTURE. This is the plain, slow, obviously correct reference the CUDA path is
 * checked against. Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it; the product path never does. It shares no code, header or table with the CUDA library.
 *
 * Sources (the pages the method is described on):
 *   [rms_norm_fused_fp8]  Modular Mojo API docs, "rms_norm_fused_fp8": the arguments shape, gamma,
 *                         epsilon, weight_offset, scale_ub, scale_output; output float8_e4m3fn with
 *                         a per-row dynamic scale.
 *   [allreduce_fp8]       Modular Mojo API docs, "allreduce_residual_rmsnorm_fp8": residual and
 *                         residual_output (the pre-norm sum), weight_offset as an additive offset
 *                         on gamma, scale_ub as the clamp of the FP8 scale.
 *   [rmsnorm_fp4quant]    FlashInfer "cute_dsl/rmsnorm_fp4quant.py": the constants (E2M1 max 6,
 *                         E4M3 max 448, blocks of 16 / 32), RMSNormFP4QuantKernel phases 2 and 3,
 *                         cvt_f32_to_ue8m0, ue8m0_to_output_scale, cvt_e2m1x8_f32 (nibble order),
 *                         and the swizzled 128x4 scale layout of the rmsnorm_fp4quant docstring.
 *
 * Arithmetic. Every intermediate is computed in double and rounded once to fp32 wherever the
 * method keeps an fp32 value (rstd, w = gamma + offset, y, the FP8 row scale). Formats are encoded
 * by one generic round-to-nearest-even routine (format_round) written from the definition of a
 * binary floating-point format. Parity pins: every function here is pinned by a test that does
 * not re-use this code (torch CPU casts, exhaustive code tables, closed forms, brute force).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* Number formats                                                                              */
/* ------------------------------------------------------------------------------------------ */

/* Round v to nearest, ties to even, in a binary format with `mant_bits` stored mantissa bits
 * and smallest normal exponent `emin` (so subnormals are multiples of 2^(emin - mant_bits)).
 * No overflow handling: the caller saturates or overflows. The quantum of the binade that
 * holds |v| is a power of two, so |v| / quantum is exact and rint() (default rounding mode:
 * to nearest, ties to even) picks the nearest multiple. A carry into the next binade gives
 * that binade's smallest value, which is representable. */
double oracle_format_round(double v, int mant_bits, int emin)
{
    if (v == 0.0 || !isfinite(v)) return v;
    double a = fabs(v);
    int e;
    frexp(a, &e);                 /* a = m * 2^e with m in [0.5, 1): floor(log2 a) = e - 1 */
    int E = e - 1;
    if (E < emin) E = emin;       /* subnormal range: the quantum stops shrinking */
    double quantum = ldexp(1.0, E - mant_bits);
    double r = rint(a / quantum) * quantum;
    return copysign(r, v);
}

/* bf16: 8 significant bits (7 stored), emin -126, largest finite (2 - 2^-7) * 2^127. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Correctly rounded double -> bf16 (IEEE rules: overflow to infinity, NaN stays NaN). */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v)) return 0x7FC0;
    double r = oracle_format_round(v, 7, -126);
    const double bf16_max = ldexp(2.0 - ldexp(1.0, -7), 127);
    if (fabs(r) > bf16_max) r = copysign(INFINITY, v);
    float f = (float)r;           /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* fp16 (IEEE binary16): sign, 5-bit exponent with bias 15, 10 stored mantissa bits. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int ef = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (ef == 0x1F) v = m ? NAN : INFINITY;
    else if (ef == 0) v = ldexp((double)m, -24);              /* m/1024 * 2^-14 */
    else v = ldexp(1.0 + m / 1024.0, ef - 15);
    return sign ? -v : v;
}

uint16_t oracle_double_to_fp16(double v)
{
    if (isnan(v)) return 0x7E00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double r = fabs(oracle_format_round(v, 10, -14));
    if (r > 65504.0) return sign | 0x7C00;                     /* overflow: infinity */
    if (r == 0.0) return sign;
    int e;
    frexp(r, &e);
    int E = e - 1;
    if (E < -14) return sign | (uint16_t)(r / ldexp(1.0, -24)); /* subnormal */
    int m = (int)((r / ldexp(1.0, E) - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)m;
}

/* E4M3 ("float8_e4m3fn"): sign, 4-bit exponent with bias 7, 3 mantissa bits, no infinities,
 * S.1111.111 is NaN, largest finite 448 (0x7E), smallest subnormal 2^-9. */
double oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int ef = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (ef == 0xF && m == 7) v = NAN;
    else if (ef == 0) v = ldexp(m / 8.0, -6);
    else v = ldexp(1.0 + m / 8.0, ef - 7);
    return sign ? -v : v;
}

/* Round to nearest even, saturate finite overflow to +-448 ("satfinite"), NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(double v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double r = fabs(oracle_format_round(v, 3, -6));
    if (r > 448.0 || isinf(v)) r = 448.0;
    if (r == 0.0) return sign;
    int e;
    frexp(r, &e);
    int E = e - 1;
    if (E < -6) return sign | (uint8_t)(r / ldexp(1.0, -9));   /* subnormal: m * 2^-9 */
    int m = (int)((r / ldexp(1.0, E) - 1.0) * 8.0);
    return sign | (uint8_t)((E + 7) << 3) | (uint8_t)m;
}

/* E2M1 (FP4): sign, 2-bit exponent with bias 1, 1 mantissa bit; values 0, .5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_decode(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int ef = (c >> 1) & 3;
    int m = c & 1;
    double v = (ef == 0) ? m * 0.5 : ldexp(1.0 + m / 2.0, ef - 1);
    return sign ? -v : v;
}

/* Round to nearest even, saturate to +-6. Returns the 4-bit code in the low nibble. */
uint8_t oracle_e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0;
    if (isnan(v)) return 0x7;     /* no NaN in E2M1; the oracle never produces one from finite y */
    double r = fabs(oracle_format_round(v, 1, 0));
    if (r > 6.0 || isinf(v)) r = 6.0;
    if (r == 0.0) return sign;
    int e;
    frexp(r, &e);
    int E = e - 1;
    if (E < 0) return sign | 1;                                  /* 0.5, the only subnormal */
    int m = (int)((r / ldexp(1.0, E) - 1.0) * 2.0);
    return sign | (uint8_t)((E + 1) << 1) | (uint8_t)m;
}

/* UE8M0 block scale of an MXFP4 block with max |y| = a ([rmsnorm_fp4quant] cvt_f32_to_ue8m0 and
 * the MXFP4 branch of kernel phase 3): code = ceil(log2(a / 6)) + 127 clamped to [0, 255], and 0
 * when a <= 0. The ceiling is taken exactly: frexp gives a/6 = m * 2^k with m in [0.5, 1), so
 * ceil(log2(a/6)) is k - 1 when m is exactly 0.5 (a power of two) and k otherwise. a/6 in double
 * is a power of two exactly when a = 1.5 * 2^j, since a has at most 24 significant bits. */
int oracle_ue8m0_code(double a)
{
    if (!(a > 0.0)) return 0;
    int k;
    double m = frexp(a / 6.0, &k);
    int e = (m == 0.5) ? k - 1 : k;
    int code = e + 127;
    if (code < 0) code = 0;
    if (code > 255) code = 255;
    return code;
}

/* Row-major or swizzled offset of block scale (row, sf) in a tensor with `num_sf` scales per row.
 * Swizzled: 128x4 tiles laid out [m_tile][k_tile][row % 32][(row % 128) / 32][sf % 4], 512 bytes
 * per tile, k tiles rounded up to whole tiles ([rmsnorm_fp4quant] rmsnorm_fp4quant docstring,
 * is_sf_swizzled_layout). */
int64_t oracle_scale_offset(int64_t row, int64_t sf, int64_t num_sf, int swizzled)
{
    if (!swizzled) return row * num_sf + sf;
    int64_t k_tiles = (num_sf + 3) / 4;
    return (row / 128) * (k_tiles * 512) + (sf / 4) * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4
           + (sf % 4);
}

/* ------------------------------------------------------------------------------------------ */
/* Row math                                                                                    */
/* ------------------------------------------------------------------------------------------ */

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1, ORACLE_F32 = 2 };

static double load_elem(const void* p, int dtype, int64_t i)
{
    switch (dtype) {
    case ORACLE_BF16: return oracle_bf16_to_double(((const uint16_t*)p)[i]);
    case ORACLE_FP16: return oracle_fp16_to_double(((const uint16_t*)p)[i]);
    default: return (double)((const float*)p)[i];
    }
}

/* Round an exact sum to the input dtype and store it. Returns the stored value. */
static double store_elem(void* p, int dtype, int64_t i, double v)
{
    switch (dtype) {
    case ORACLE_BF16: {
        uint16_t b = oracle_double_to_bf16(v);
        if (p) ((uint16_t*)p)[i] = b;
        return oracle_bf16_to_double(b);
    }
    case ORACLE_FP16: {
        uint16_t h = oracle_double_to_fp16(v);
        if (p) ((uint16_t*)p)[i] = h;
        return oracle_fp16_to_double(h);
    }
    default: {
        float f = (float)v;       /* double -> float conversion rounds to nearest even */
        if (p) ((float*)p)[i] = f;
        return (double)f;
    }
    }
}

/* The front half shared by every mode, for one row of `hidden` elements:
 *   s_i  = RN_dtype(x_i + res_i)            residual add, stored as residual_output
 *                                           ([allreduce_fp8] residual / residual_output)
 *   rstd = RN_fp32(1 / sqrt(sum s_i^2 / H + eps))   ([rmsnorm_fp4quant] kernel phase 2)
 *   w_i  = fp32(gamma_i) + fp32(weight_offset), an fp32 add
 *                                           ([allreduce_fp8] weight_offset: offset on gamma)
 *   y_i  = RN_fp32(s_i * rstd * w_i)        ([rmsnorm_fp4quant] kernel phase 3; fp32 products)
 * The norm is taken over the rounded sum s, the value residual_output holds. Sum of two values
 * of a 16-bit float type in double is exact, so one rounding gives the correctly rounded sum. */
static float row_front(const void* x, const void* res, int dtype, const void* gamma, int64_t H,
                       float eps, float weight_offset, void* s_out, float* y)
{
    double ss = 0.0;
    for (int64_t i = 0; i < H; i++) {
        double sum = load_elem(x, dtype, i) + (res ? load_elem(res, dtype, i) : 0.0);
        double s = res ? store_elem(s_out, dtype, i, sum) : sum;
        y[i] = (float)s;          /* hold s until rstd is known; s is exact in fp32 */
        ss += s * s;
    }
    float rstd = (float)(1.0 / sqrt(ss / (double)H + (double)eps));
    for (int64_t i = 0; i < H; i++) {
        float w = (float)load_elem(gamma, dtype, i) + weight_offset;
        y[i] = (float)((double)y[i] * (double)rstd * (double)w);
    }
    return rstd;
}

/* Outputs common to all modes: y and the per-element pre-rounding value (the quantity handed to
 * the final E4M3 / E2M1 rounding) are optional, for the tests' boundary-tolerance rule. */

/* FP8 per-row dynamic quantisation ([rms_norm_fused_fp8], [allreduce_fp8]):
 *   amax = max_i |y_i|;  scale = RN_fp32(min(amax, scale_ub) / 448);  q_i = E4M3(y_i / scale),
 *   with q = 0 on a row whose scale is 0.
 * [rms_norm_fused_fp8] lets the scale be stored as bf16 or fp16 (parameter scales_dtype): the fp32
 * scale is then rounded to that type, and the codes are formed against the stored value so that
 * y ~= dec(q) * stored scale. scale_out receives the stored value widened to fp32. */
int oracle_quant_fp8(const void* input, const void* residual, int dtype, const void* gamma,
                     int64_t rows, int64_t hidden, float eps, float weight_offset, float scale_ub,
                     int scale_dtype, void* residual_output, uint8_t* q, float* scale_out,
                     float* y_out, double* pre_out, float* y_tmp)
{
    size_t esz = dtype == ORACLE_F32 ? 4 : 2;
    for (int64_t r = 0; r < rows; r++) {
        const char* xr = (const char*)input + (size_t)(r * hidden) * esz;
        const char* rr = residual ? (const char*)residual + (size_t)(r * hidden) * esz : NULL;
        char* so = residual_output ? (char*)residual_output + (size_t)(r * hidden) * esz : NULL;
        float* y = y_out ? y_out + r * hidden : y_tmp;
        row_front(xr, rr, dtype, gamma, hidden, eps, weight_offset, so, y);
        float amax = 0.0f;
        for (int64_t i = 0; i < hidden; i++)
            if (fabsf(y[i]) > amax) amax = fabsf(y[i]);
        double clamped = amax < scale_ub ? amax : scale_ub;
        float scale = (float)(clamped / 448.0);
        if (scale_dtype == ORACLE_BF16)
            scale = (float)oracle_bf16_to_double(oracle_double_to_bf16(scale));
        else if (scale_dtype == ORACLE_FP16)
            scale = (float)oracle_fp16_to_double(oracle_double_to_fp16(scale));
        scale_out[r] = scale;
        for (int64_t i = 0; i < hidden; i++) {
            double v = scale > 0.0f ? (double)y[i] / (double)scale : 0.0;
            q[r * hidden + i] = scale > 0.0f ? oracle_e4m3_encode(v) : 0x00;
            if (pre_out) pre_out[r * hidden + i] = v;
        }
    }
    return 0;
}

/* NVFP4 ([rmsnorm_fp4quant] kernel phase 3, E4M3 scale format, block of 16), per block b:
 *   a = max |y_i|;  t = min(gs * a / 6, 448);  s = E4M3(t);
 *   q_i = E2M1(y_i * gs / dec(s)), or 0 for every element when s decodes to 0.
 * gs multiplies into the block scale and into the element factor, so dequant = q * dec(s) / gs.
 * Two E2M1 codes per byte: element 2k in the low nibble, 2k+1 in the high nibble. */
int oracle_quant_nvfp4(const void* input, const void* residual, int dtype, const void* gamma,
                       int64_t rows, int64_t hidden, float eps, float weight_offset, float gs,
                       int swizzled, void* residual_output, uint8_t* out, uint8_t* block_scale,
                       float* y_out, double* pre_out, double* t_out, float* y_tmp)
{
    size_t esz = dtype == ORACLE_F32 ? 4 : 2;
    int64_t nsf = hidden / 16;
    for (int64_t r = 0; r < rows; r++) {
        const char* xr = (const char*)input + (size_t)(r * hidden) * esz;
        const char* rr = residual ? (const char*)residual + (size_t)(r * hidden) * esz : NULL;
        char* so = residual_output ? (char*)residual_output + (size_t)(r * hidden) * esz : NULL;
        float* y = y_out ? y_out + r * hidden : y_tmp;
        row_front(xr, rr, dtype, gamma, hidden, eps, weight_offset, so, y);
        for (int64_t b = 0; b < nsf; b++) {
            double a = 0.0;
            for (int j = 0; j < 16; j++)
                if (fabs((double)y[b * 16 + j]) > a) a = fabs((double)y[b * 16 + j]);
            double t = (double)gs * a / 6.0;
            if (t > 448.0) t = 448.0;
            uint8_t s = oracle_e4m3_encode(t);
            double ds = oracle_e4m3_decode(s);
            block_scale[oracle_scale_offset(r, b, nsf, swizzled)] = s;
            if (t_out) t_out[r * nsf + b] = t;
            for (int j = 0; j < 16; j++) {
                int64_t i = b * 16 + j;
                double v = ds != 0.0 ? (double)y[i] * (double)gs / ds : 0.0;
                uint8_t c = ds != 0.0 ? oracle_e2m1_encode(v) : 0;
                uint8_t* byte = &out[(r * hidden + i) / 2];
                if ((i & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | c);
                else *byte = (uint8_t)((*byte & 0x0F) | (c << 4));
                if (pre_out) pre_out[r * hidden + i] = v;
            }
        }
    }
    return 0;
}

/* MXFP4 ([rmsnorm_fp4quant] kernel phase 3, UE8M0 scale format, block of 32), per block b:
 *   code = oracle_ue8m0_code(max |y_i|);  q_i = E2M1(y_i * 2^(127 - code)), or 0 when code = 0
 *   (ue8m0_to_output_scale maps code 0 to a zero factor). No global scale. */
int oracle_quant_mxfp4(const void* input, const void* residual, int dtype, const void* gamma,
                       int64_t rows, int64_t hidden, float eps, float weight_offset, int swizzled,
                       void* residual_output, uint8_t* out, uint8_t* block_scale, float* y_out,
                       double* pre_out, double* a_out, float* y_tmp)
{
    size_t esz = dtype == ORACLE_F32 ? 4 : 2;
    int64_t nsf = hidden / 32;
    for (int64_t r = 0; r < rows; r++) {
        const char* xr = (const char*)input + (size_t)(r * hidden) * esz;
        const char* rr = residual ? (const char*)residual + (size_t)(r * hidden) * esz : NULL;
        char* so = residual_output ? (char*)residual_output + (size_t)(r * hidden) * esz : NULL;
        float* y = y_out ? y_out + r * hidden : y_tmp;
        row_front(xr, rr, dtype, gamma, hidden, eps, weight_offset, so, y);
        for (int64_t b = 0; b < nsf; b++) {
            double a = 0.0;
            for (int j = 0; j < 32; j++)
                if (fabs((double)y[b * 32 + j]) > a) a = fabs((double)y[b * 32 + j]);
            int code = oracle_ue8m0_code(a);
            block_scale[oracle_scale_offset(r, b, nsf, swizzled)] = (uint8_t)code;
            if (a_out) a_out[r * nsf + b] = a;
            for (int j = 0; j < 32; j++) {
                int64_t i = b * 32 + j;
                double v = code != 0 ? ldexp((double)y[i], 127 - code) : 0.0;
                uint8_t c = code != 0 ? oracle_e2m1_encode(v) : 0;
                uint8_t* byte = &out[(r * hidden + i) / 2];
                if ((i & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | c);
                else *byte = (uint8_t)((*byte & 0x0F) | (c << 4));
                if (pre_out) pre_out[r * hidden + i] = v;
            }
        }
    }
    return 0;
}

/* y only (no quantisation), for the global-amax pre-pass pins and for gs = 448 * 6 / amax(y). */
int oracle_rmsnorm(const void* input, const void* residual, int dtype, const void* gamma,
                   int64_t rows, int64_t hidden, float eps, float weight_offset,
                   void* residual_output, float* y_out, float* rstd_out)
{
    size_t esz = dtype == ORACLE_F32 ? 4 : 2;
    for (int64_t r = 0; r < rows; r++) {
        const char* xr = (const char*)input + (size_t)(r * hidden) * esz;
        const char* rr = residual ? (const char*)residual + (size_t)(r * hidden) * esz : NULL;
        char* so = residual_output ? (char*)residual_output + (size_t)(r * hidden) * esz : NULL;
        float rstd = row_front(xr, rr, dtype, gamma, hidden, eps, weight_offset, so,
                               y_out + r * hidden);
        if (rstd_out) rstd_out[r] = rstd;
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Array forms of the encoders, so the tests can sweep many values in one call.               */
/* ------------------------------------------------------------------------------------------ */

void oracle_e4m3_encode_f64_array(const double* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e4m3_encode_f32_array(const float* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode((double)v[i]);
}

void oracle_e2m1_encode_f64_array(const double* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e2m1_encode(v[i]);
}

void oracle_e2m1_encode_f32_array(const float* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e2m1_encode((double)v[i]);
}

void oracle_bf16_round_array(const double* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_double_to_bf16(v[i]);
}

void oracle_fp16_round_array(const double* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_double_to_fp16(v[i]);
}

void oracle_ue8m0_code_array(const double* a, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)oracle_ue8m0_code(a[i]);
}
