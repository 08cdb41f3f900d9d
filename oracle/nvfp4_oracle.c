/*
 * NVFP4 paged KV cache -- CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct statement of what the
 * GPU library computes. Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the product path never does, and it shares no code, header, table or
 * constant generator with the CUDA sources.
 *
 * Sources (web pages; cited by title and section):
 *   [LMSYS]  "Accelerating Long-Context and Agentic Inference with NVFP4 KV Cache" (LMSYS blog):
 *            introduction + Figure 1 (format), "NVFP4 KV Implementation in SGLang" (three paths),
 *            "NVFP4 KV Decode Attention Kernel Implementation" + Figure 3 (decode kernel).
 *   [TRTLLM] "KV Cache Compression in TensorRT LLM" (NVIDIA tech blog):
 *            "NVFP4 Cold-Page Compression" > Introduction + Figure 6 (page layouts),
 *            "How It Works in TensorRT LLM" (encode/decode fused with the copy),
 *            "Evaluation" > Accuracy + Figure 15 (round trips do not accumulate error).
 *
 * Arithmetic convention. Every step the format defines in FP32 is evaluated as an fp64
 * operation followed by an explicit round to fp32 (round_to_format with 24 bits). For a single
 * +, -, x or / of two fp32 operands that equals the IEEE fp32 operation, because 53 >= 2*24+2
 * makes the double rounding innocuous. Roundings to E2M1 / E4M3 / BF16 / FP16 are done on the
 * exact value with round-half-to-even, by scaling to an integer significand and calling
 * nearbyint() (the default rounding mode is round-to-nearest-even).
 *
 * Readings of points the pages leave open (each one stated again where it is used):
 *   R1 block axis: a block is 16 consecutive elements along head_dim of one token.
 *   R2 byte packing, two forms (a pool uses one):
 *      dim pairs   (packing 0): data[page][head][token][head_dim/2], byte j holds head dims 2j
 *                  (low nibble) and 2j+1 (high nibble) of one token; scales[page][head][token][D/16].
 *      token pairs (packing 1): data[page][head][token/2][head_dim], byte d holds head dim d of
 *                  tokens 2p (low nibble) and 2p+1 (high nibble); scales[page][head][token/2][D/16][2],
 *                  the scales of a block for tokens 2p and 2p+1 side by side.
 *      Both hold the same codes and scales; only the byte order inside a page differs.
 *   R3 page layout (HND): every (page, head) owns one contiguous run of T tokens.
 *   R4 scale pick: s = E4M3_rne_satfinite(fp32(amax_block / fp32(6 g))).
 *   R5 element code: c = E2M1_rne_satfinite(fp32(x * r)), r = fp32(1 / fp32(s g)) or 0 if s g == 0;
 *      the sign is kept, so a negative value that rounds to zero is code 0x8.
 *   R6 decode: v = e2m1(c) * e4m3(s) (exact), then fp32(v * g), then the output rounding.
 *   R7 global scale: g = fp32(amax_tensor / 2688) (2688 = 448 * 6); g = 1 if that is 0.
 *   R8 FP8 output: E4M3_rne_satfinite(fp32(v * fp32(g / out_scale))), sign kept.
 *   R10 two-component (2FP4) encoding of the RoPE part of K in a cold page: c1 = the encoding
 *      of x (R4, R5); with v1 = e2m1(c1) * e4m3(s1), the residual r = fp32(x - fp32(v1 g)) is
 *      encoded the same way with the same g into c2; decode = fp32(fp32(v1 g) + fp32(v2 g)),
 *      then the 16-bit rounding.
 *   R9 FP8 workspace copy of a chunk (extend path): E4M3_rne_satfinite(fp32(x * m)),
 *      m = fp32(1 / ws_scale), sign kept; pages keep the plain [page][head][token][dim] order.
 *
 * Build: plain C99, no SIMD intrinsics, -ffp-contract=off (no fused multiply-add), optional
 * OpenMP over independent pages / (sequence, head) pairs.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes shared with the Python wrapper of this oracle (not with the GPU library) */
enum { ORC_BF16 = 0, ORC_FP16 = 1, ORC_FP8_E4M3 = 2 };

/* ------------------------------------------------------------------------------------------ */
/* Rounding to a binary floating-point format                                                 */
/* ------------------------------------------------------------------------------------------ */

/*
 * Round the real number y (held exactly in a double) to the nearest member of a binary format
 * with p significand bits (hidden bit included) and smallest normal exponent emin; numbers
 * below 2^emin are subnormal with the fixed quantum 2^(emin - p + 1). Ties go to the even
 * significand. There is no upper bound here; callers saturate or overflow as the format says.
 */
static double round_to_format(double y, int p, int emin)
{
    if (y == 0.0 || !isfinite(y))
        return y;
    int e2;
    (void)frexp(fabs(y), &e2);      /* |y| = f * 2^e2 with f in [0.5, 1) */
    int lead = e2 - 1;              /* exponent of the leading bit        */
    if (lead < emin)
        lead = emin;
    int shift = p - 1 - lead;       /* quantum is 2^-shift                */
    double q = ldexp(y, shift);     /* exact: only the exponent changes   */
    double r = nearbyint(q);        /* round half to even                 */
    return ldexp(r, -shift);
}

/* IEEE binary32: 24 bits, emin -126, overflow to infinity. */
static double fp32(double y)
{
    double r = round_to_format(y, 24, -126);
    if (fabs(r) > 3.4028234663852886e38)
        r = copysign(INFINITY, r);
    return r;
}

/* bfloat16: 8 bits, emin -126, largest finite (2 - 2^-7) * 2^127, overflow to infinity. */
static double bf16_round(double y)
{
    double r = round_to_format(y, 8, -126);
    if (fabs(r) > 3.3895313892515355e38)
        r = copysign(INFINITY, r);
    return r;
}

/* IEEE binary16: 11 bits, emin -14, largest finite 65504, overflow to infinity. */
static double fp16_round(double y)
{
    double r = round_to_format(y, 11, -14);
    if (fabs(r) > 65504.0)
        r = copysign(INFINITY, r);
    return r;
}

/* ------------------------------------------------------------------------------------------ */
/* E2M1 (FP4): sign, 2 exponent bits (bias 1), 1 mantissa bit, no inf / NaN.                   */
/* [LMSYS intro, Figure 1]: the values are 4-bit E2M1. Magnitudes by code 0..7:                */
/* 0, 0.5, 1, 1.5, 2, 3, 4, 6.                                                                 */
/* ------------------------------------------------------------------------------------------ */

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

static double e2m1_value(int code)
{
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* RNE to E2M1 (p = 2, emin = 0), saturating at 6; the sign bit follows the sign of y. */
static int e2m1_encode(double y)
{
    int sign = signbit(y) ? 8 : 0;
    double m = round_to_format(fabs(y), 2, 0);
    if (m > 6.0)
        m = 6.0;
    for (int k = 0; k < 8; ++k)
        if (E2M1_MAG[k] == m)
            return sign | k;
    return -1; /* unreachable for finite y */
}

/* ------------------------------------------------------------------------------------------ */
/* E4M3 ("fn" variant): bias 7, no inf, NaN = S.1111.111, largest finite 448,                  */
/* smallest normal 2^-6, subnormal step 2^-9. [LMSYS intro]: each block has an FP8 scale.      */
/* ------------------------------------------------------------------------------------------ */

static double e4m3_value(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* RNE to E4M3 (p = 4, emin = -6), saturating at 448 ("satfinite"); sign follows y. */
static uint8_t e4m3_encode(double y)
{
    int sign = signbit(y) ? 0x80 : 0;
    double m = round_to_format(fabs(y), 4, -6);
    if (m > 448.0)
        m = 448.0;
    if (m == 0.0)
        return (uint8_t)sign;
    int e2;
    double f = frexp(m, &e2); /* m = f * 2^e2, f in [0.5,1) */
    int lead = e2 - 1;
    if (lead < -6) /* subnormal: m = k * 2^-9, k in 1..7 */
        return (uint8_t)(sign | (int)ldexp(m, 9));
    int mant = (int)ldexp(2.0 * f - 1.0, 3); /* (m / 2^lead - 1) * 8 */
    return (uint8_t)(sign | ((lead + 7) << 3) | mant);
}

/* ------------------------------------------------------------------------------------------ */
/* 16-bit float bit patterns <-> values                                                        */
/* ------------------------------------------------------------------------------------------ */

static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static uint16_t bf16_bits(double v) /* v must already be a bfloat16 value */
{
    float f = (float)v; /* exact */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double fp16_value(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

static uint16_t fp16_bits(double v) /* v must already be a binary16 value */
{
    uint16_t s = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(s | 0x7C00);
    if (a == 0.0)
        return s;
    int e2;
    double f = frexp(a, &e2);
    int lead = e2 - 1;
    if (lead < -14)
        return (uint16_t)(s | (int)ldexp(a, 24));
    int mant = (int)ldexp(2.0 * f - 1.0, 10);
    return (uint16_t)(s | ((lead + 15) << 10) | mant);
}

/* One source element as the exact fp32 value the encoder starts from (step 1 of encode). */
static double load_src(int dtype, const void* src, size_t idx, double src_scale)
{
    switch (dtype) {
    case ORC_BF16:
        return bf16_value(((const uint16_t*)src)[idx]);
    case ORC_FP16:
        return fp16_value(((const uint16_t*)src)[idx]);
    default: /* FP8 E4M3 input: x = fp32(e4m3 * src_scale) */
        return fp32(e4m3_value(((const uint8_t*)src)[idx]) * src_scale);
    }
}

/* Byte index of element (page p, head h, token t, head dim d) in a packed-code pool, and which
   nibble holds it (R2). */
static size_t code_index(int packing, size_t p, int h, int t, int d, int H, int T, int D, int* hi)
{
    if (packing == 1) {
        *hi = t & 1;
        return (((size_t)p * H + h) * (size_t)(T / 2) + (size_t)(t / 2)) * (size_t)D + (size_t)d;
    }
    *hi = d & 1;
    return (((size_t)p * H + h) * (size_t)T + (size_t)t) * (size_t)(D / 2) + (size_t)(d / 2);
}

/* Byte index of the scale of block b (head dims 16b..16b+15) of token t (R2). */
static size_t scale_index(int packing, size_t p, int h, int t, int b, int H, int T, int NB)
{
    if (packing == 1)
        return ((((size_t)p * H + h) * (size_t)(T / 2) + (size_t)(t / 2)) * (size_t)NB + (size_t)b) * 2 +
               (size_t)(t & 1);
    return (((size_t)p * H + h) * (size_t)T + (size_t)t) * (size_t)NB + (size_t)b;
}

static int get_code(const uint8_t* data, size_t idx, int hi)
{
    return hi ? (data[idx] >> 4) : (data[idx] & 15);
}

static void put_code(uint8_t* data, size_t idx, int hi, int code)
{
    data[idx] = hi ? (uint8_t)((data[idx] & 0x0F) | (code << 4)) : (uint8_t)((data[idx] & 0xF0) | code);
}

/* ------------------------------------------------------------------------------------------ */
/* Exported scalar conversions (used by the tests to pin the roundings and by the exhaustive  */
/* fp32 sweeps).                                                                               */
/* ------------------------------------------------------------------------------------------ */

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

double orc_round_to_format(double y, int p, int emin) { return round_to_format(y, p, emin); }
double orc_fp32(double y) { return fp32(y); }
double orc_bf16_round(double y) { return bf16_round(y); }
double orc_fp16_round(double y) { return fp16_round(y); }
double orc_e2m1_value(int code) { return e2m1_value(code); }
int orc_e2m1_encode(double y) { return e2m1_encode(y); }
double orc_e4m3_value(int b) { return e4m3_value((uint8_t)b); }
int orc_e4m3_encode(double y) { return e4m3_encode(y); }
double orc_bf16_value(int h) { return bf16_value((uint16_t)h); }
int orc_bf16_bits(double v) { return bf16_bits(v); }
double orc_fp16_value(int h) { return fp16_value((uint16_t)h); }
int orc_fp16_bits(double v) { return fp16_bits(v); }

/* E2M1 codes of n fp32 inputs (finite), one code per output byte. */
void orc_e2m1_encode_f32(const float* x, size_t n, uint8_t* out)
{
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; ++i)
        out[i] = (uint8_t)e2m1_encode((double)x[i]);
}

/* E4M3 (satfinite) codes of n fp32 inputs (finite). */
void orc_e4m3_encode_f32(const float* x, size_t n, uint8_t* out)
{
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < (long long)n; ++i)
        out[i] = e4m3_encode((double)x[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* Global (tensor) scale. R7.                                                                  */
/* [LMSYS intro]: one more scale, FP32, per tensor; [LMSYS "Limitations"]: the                 */
/* experiments used 1.0, and calibration may reduce overflow / underflow. The calibrated       */
/* rule maps the tensor maximum to the top of both grids: amax / (448 * 6).                    */
/* ------------------------------------------------------------------------------------------ */

/* max |x| over every slot of the listed pages (page ids NULL = 0..num_pages-1). */
double orc_tensor_amax(int H, int D, int T, int src_dtype, const void* src,
                       const int32_t* src_page_ids, int num_pages, double src_scale)
{
    size_t page_elems = (size_t)H * T * D;
    double amax = 0.0;
    src_scale = fp32(src_scale); /* the source scale is an FP32 scalar */
#pragma omp parallel for reduction(max : amax) schedule(static)
    for (int i = 0; i < num_pages; ++i) {
        size_t sp = (size_t)(src_page_ids ? src_page_ids[i] : i);
        for (size_t e = 0; e < page_elems; ++e) {
            double a = fabs(load_src(src_dtype, src, sp * page_elems + e, src_scale));
            if (a > amax)
                amax = a;
        }
    }
    return amax;
}

double orc_global_scale_from_amax(double amax)
{
    double g = fp32(amax / 2688.0); /* amax is an fp32 value; one fp32 division */
    return (g == 0.0) ? 1.0 : g;
}

/* ------------------------------------------------------------------------------------------ */
/* Encode one block of 16 values (steps A2..A4). R4, R5.                                       */
/* ------------------------------------------------------------------------------------------ */

static void encode_block(const double* x, double g, int* c, uint8_t* scale_out)
{
    double d = fp32(6.0 * g);                 /* fp32(6 g)                                */
    double a = 0.0;                           /* block amax (exact)                       */
    for (int i = 0; i < 16; ++i)
        if (fabs(x[i]) > a)
            a = fabs(x[i]);
    uint8_t s_code = e4m3_encode(fp32(a / d)); /* scale pick, RNE + satfinite              */
    double s = e4m3_value(s_code);
    double sg = fp32(s * g);
    double r = (sg == 0.0) ? 0.0 : fp32(1.0 / sg);
    for (int i = 0; i < 16; ++i)
        c[i] = e2m1_encode(fp32(x[i] * r));
    *scale_out = s_code;
}

/*
 * Quantize pages (K or V of one layer) to NVFP4.
 * [TRTLLM "How It Works", the paragraph on the fused encode and decode]: a batch of pages goes
 * through one encoder; [LMSYS Path 1 / Path 2]: the current K/V is quantized and written into
 * the NVFP4 cache. Layout R3; src pages are [page][H][T][D] in src_dtype.
 */
void orc_quantize_pages(int H, int D, int T, int packing, int src_dtype, const void* src,
                        const int32_t* src_page_ids, double src_scale, double g,
                        uint8_t* dst_data, uint8_t* dst_scales, const int32_t* dst_page_ids,
                        int num_pages)
{
    int NB = D / 16;
    size_t page_elems = (size_t)H * T * D;
    src_scale = fp32(src_scale); /* FP32 scalars (tensor scale, source scale) */
    g = fp32(g);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < num_pages; ++i) {
        size_t sp = (size_t)(src_page_ids ? src_page_ids[i] : i);
        size_t dp = (size_t)(dst_page_ids ? dst_page_ids[i] : i);
        for (int h = 0; h < H; ++h)
            for (int t = 0; t < T; ++t)
                for (int b = 0; b < NB; ++b) {
                    double x[16];
                    int c[16];
                    size_t row = ((size_t)h * T + t); /* token row within the page */
                    for (int k = 0; k < 16; ++k)
                        x[k] = load_src(src_dtype, src, sp * page_elems + row * D + b * 16 + k,
                                        src_scale);
                    uint8_t sc;
                    encode_block(x, g, c, &sc);
                    for (int k = 0; k < 16; ++k) {
                        int hi;
                        size_t idx = code_index(packing, dp, h, t, b * 16 + k, H, T, D, &hi);
                        put_code(dst_data, idx, hi, c[k]);
                    }
                    dst_scales[scale_index(packing, dp, h, t, b, H, T, NB)] = sc;
                }
    }
}

/*
 * FP8 workspace copy of source pages (BF16, FP16, or FP8 read as x = fp32(e4m3 * src_scale)).
 * R9. [LMSYS Path 2]: the current chunk's K/V are copied into the FP8 workspace that the
 * extend attention reads (and, separately, written to the NVFP4 cache: orc_quantize_pages).
 */
void orc_cast_fp8_pages(int H, int D, int T, int src_dtype, const void* src,
                        const int32_t* src_page_ids, double src_scale, double ws_scale,
                        uint8_t* dst, const int32_t* dst_page_ids, int num_pages)
{
    size_t page_elems = (size_t)H * T * D;
    double m = fp32(1.0 / fp32(ws_scale)); /* FP32 scalar and its FP32 reciprocal */
    double ss = fp32(src_scale);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < num_pages; ++i) {
        size_t sp = (size_t)(src_page_ids ? src_page_ids[i] : i);
        size_t dp = (size_t)(dst_page_ids ? dst_page_ids[i] : i);
        for (size_t e = 0; e < page_elems; ++e) {
            double x = load_src(src_dtype, src, sp * page_elems + e, ss);
            dst[dp * page_elems + e] = e4m3_encode(fp32(x * m));
        }
    }
}

/*
 * Two-component encoding of n_blocks blocks of 16 consecutive 16-bit source values. R10.
 * [TRTLLM "The RoPE part of K"]: the RoPE part can be stored as two FP4 components, the
 * second holding the first one's rounding error. Codes are packed two per byte, value 2j of a
 * block in the low nibble of byte j (8 bytes per block); one scale byte per block.
 */
void orc_encode_2fp4_blocks(int n_blocks, int src_dtype, const void* src, double g,
                            uint8_t* codes1, uint8_t* scales1, uint8_t* codes2, uint8_t* scales2)
{
    g = fp32(g);
    for (int blk = 0; blk < n_blocks; ++blk) {
        double x[16], r[16];
        int c1[16], c2[16];
        uint8_t s1, s2;
        for (int k = 0; k < 16; ++k)
            x[k] = load_src(src_dtype, src, (size_t)blk * 16 + k, 1.0);
        encode_block(x, g, c1, &s1);
        for (int k = 0; k < 16; ++k) {
            double v1 = e2m1_value(c1[k]) * e4m3_value(s1); /* exact */
            r[k] = fp32(x[k] - fp32(v1 * g));
        }
        encode_block(r, g, c2, &s2);
        for (int j = 0; j < 8; ++j) {
            codes1[(size_t)blk * 8 + j] = (uint8_t)(c1[2 * j] | (c1[2 * j + 1] << 4));
            codes2[(size_t)blk * 8 + j] = (uint8_t)(c2[2 * j] | (c2[2 * j + 1] << 4));
        }
        scales1[blk] = s1;
        scales2[blk] = s2;
    }
}

/* Decode of the two-component blocks into 16-bit bit patterns (ORC_BF16 / ORC_FP16). R10. */
void orc_decode_2fp4_blocks(int n_blocks, const uint8_t* codes1, const uint8_t* scales1,
                            const uint8_t* codes2, const uint8_t* scales2, double g,
                            int out_dtype, uint16_t* out)
{
    g = fp32(g);
    for (int blk = 0; blk < n_blocks; ++blk)
        for (int k = 0; k < 16; ++k) {
            uint8_t b1 = codes1[(size_t)blk * 8 + k / 2], b2 = codes2[(size_t)blk * 8 + k / 2];
            int c1 = (k & 1) ? (b1 >> 4) : (b1 & 15), c2 = (k & 1) ? (b2 >> 4) : (b2 & 15);
            double v1 = e2m1_value(c1) * e4m3_value(scales1[blk]);
            double v2 = e2m1_value(c2) * e4m3_value(scales2[blk]);
            double y = fp32(fp32(v1 * g) + fp32(v2 * g));
            out[(size_t)blk * 16 + k] = (out_dtype == ORC_BF16) ? bf16_bits(bf16_round(y))
                                                                  : fp16_bits(fp16_round(y));
        }
}

/*
 * Dequantize pages. R6, R8.
 * [TRTLLM "How It Works"]: on the way back the decoder dequantizes into the GPU pool (BF16/FP16);
 * [LMSYS Path 2]: the cached prefix is gathered, dequantized and written into an FP8 workspace.
 * out_dtype: ORC_BF16 / ORC_FP16 (uint16 bit patterns) or ORC_FP8_E4M3 (bytes).
 */
void orc_dequantize_pages(int H, int D, int T, int packing, const uint8_t* src_data,
                          const uint8_t* src_scales, const int32_t* src_page_ids, double g,
                          int out_dtype, void* dst, const int32_t* dst_page_ids, double out_scale,
                          int num_pages)
{
    int NB = D / 16;
    size_t page_elems = (size_t)H * T * D;
    g = fp32(g); /* FP32 scalars (tensor scale, FP8 output scale) */
    out_scale = fp32(out_scale);
    double m = fp32(g / out_scale); /* FP8 output multiplier (R8) */
#pragma omp parallel for schedule(static)
    for (int i = 0; i < num_pages; ++i) {
        size_t sp = (size_t)(src_page_ids ? src_page_ids[i] : i);
        size_t dp = (size_t)(dst_page_ids ? dst_page_ids[i] : i);
        for (int h = 0; h < H; ++h)
            for (int t = 0; t < T; ++t)
                for (int d = 0; d < D; ++d) {
                    int hi;
                    size_t idx = code_index(packing, sp, h, t, d, H, T, D, &hi);
                    double s = e4m3_value(src_scales[scale_index(packing, sp, h, t, d / 16, H, T, NB)]);
                    double v = e2m1_value(get_code(src_data, idx, hi)) * s; /* exact */
                    size_t o = dp * page_elems + ((size_t)h * T + t) * D + d;
                    if (out_dtype == ORC_BF16)
                        ((uint16_t*)dst)[o] = bf16_bits(bf16_round(fp32(v * g)));
                    else if (out_dtype == ORC_FP16)
                        ((uint16_t*)dst)[o] = fp16_bits(fp16_round(fp32(v * g)));
                    else
                        ((uint8_t*)dst)[o] = e4m3_encode(fp32(v * m));
                }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Paged GQA decode attention over NVFP4 K/V, exact in fp64 (steps A7..A10 by definition).    */
/* [LMSYS Path 3]: decode reads NVFP4 K/V directly from the cache; [LMSYS decode kernel,       */
/* Figure 3]: BF16 queries, K/V dequantized from packed tiles and E4M3 block scales, global    */
/* K/V scales applied through the attention scaling. Attention itself is the plain definition: */
/* out = sum_t softmax(z)_t v_t,  z_t = sm_scale * q . k_t,  lse = log sum_t exp(z_t).          */
/* Token t of sequence b lives in page page_table[b][t / T], slot t % T. Query head qh reads   */
/* KV head qh / (Hq / H). An empty sequence gives out = 0 and lse = -inf. `want` (optional,    */
/* [B][Hq]) selects the pairs to compute so that large cases can be sampled.                    */
/* ------------------------------------------------------------------------------------------ */

static double dequant_elem(int packing, const uint8_t* data, const uint8_t* scales, size_t page,
                           int h, int t, int d, int H, int T, int D)
{
    int hi;
    size_t idx = code_index(packing, page, h, t, d, H, T, D, &hi);
    return e2m1_value(get_code(data, idx, hi)) *
           e4m3_value(scales[scale_index(packing, page, h, t, d / 16, H, T, D / 16)]);
}

void orc_paged_decode_attention(int B, int Hq, int H, int D, int T, int k_packing,
                                int v_packing, const uint16_t* q_bf16,
                                const uint8_t* k_data, const uint8_t* k_scales, double g_k,
                                const uint8_t* v_data, const uint8_t* v_scales, double g_v,
                                const int32_t* page_table, int max_pages_per_seq,
                                const int32_t* seq_lens, double sm_scale, const uint8_t* want,
                                double* out, double* lse)
{
    int G = Hq / H;
    g_k = fp32(g_k); /* FP32 scalars of the call: tensor scales and softmax scale */
    g_v = fp32(g_v);
    sm_scale = fp32(sm_scale);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int qh = 0; qh < Hq; ++qh) {
            if (want && !want[(size_t)b * Hq + qh])
                continue; /* (sequence, head) pair not requested: left untouched */
            int h = qh / G;
            int L = seq_lens[b];
            double* o = out + ((size_t)b * Hq + qh) * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            if (L <= 0) {
                if (lse)
                    lse[(size_t)b * Hq + qh] = -INFINITY;
                continue;
            }
            const uint16_t* qv = q_bf16 + ((size_t)b * Hq + qh) * D;
            /* first pass: the maximum score (scores are recomputed in the second pass) */
            double zmax = -INFINITY;
            for (int t = 0; t < L; ++t) {
                size_t page = (size_t)page_table[(size_t)b * max_pages_per_seq + t / T];
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qv[d]) *
                           (dequant_elem(k_packing, k_data, k_scales, page, h, t % T, d, H, T, D) * g_k);
                double zt = sm_scale * dot;
                if (zt > zmax)
                    zmax = zt;
            }
            /* second pass: weights, normaliser and weighted sum of values */
            double l = 0.0;
            for (int t = 0; t < L; ++t) {
                size_t page = (size_t)page_table[(size_t)b * max_pages_per_seq + t / T];
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qv[d]) *
                           (dequant_elem(k_packing, k_data, k_scales, page, h, t % T, d, H, T, D) * g_k);
                double w = exp(sm_scale * dot - zmax);
                l += w;
                for (int d = 0; d < D; ++d)
                    o[d] += w * (dequant_elem(v_packing, v_data, v_scales, page, h, t % T, d, H, T, D) * g_v);
            }
            for (int d = 0; d < D; ++d)
                o[d] /= l;
            if (lse)
                lse[(size_t)b * Hq + qh] = zmax + log(l);
        }
}

/*
 * The same attention over unquantized BF16 K/V pages ([page][H][T][D] bit patterns). Used only
 * to report the quantization error of NVFP4 attention against BF16 attention.
 */
void orc_paged_decode_attention_bf16(int B, int Hq, int H, int D, int T, const uint16_t* q_bf16,
                                     const uint16_t* k_bf16, const uint16_t* v_bf16,
                                     const int32_t* page_table, int max_pages_per_seq,
                                     const int32_t* seq_lens, double sm_scale, double* out)
{
    int G = Hq / H;
    sm_scale = fp32(sm_scale);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int qh = 0; qh < Hq; ++qh) {
            int h = qh / G;
            int L = seq_lens[b];
            double* o = out + ((size_t)b * Hq + qh) * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            if (L <= 0)
                continue;
            const uint16_t* qv = q_bf16 + ((size_t)b * Hq + qh) * D;
            double zmax = -INFINITY;
            for (int t = 0; t < L; ++t) {
                size_t row = ((size_t)page_table[(size_t)b * max_pages_per_seq + t / T] * H + h) * T + t % T;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qv[d]) * bf16_value(k_bf16[row * D + d]);
                if (sm_scale * dot > zmax)
                    zmax = sm_scale * dot;
            }
            double l = 0.0;
            for (int t = 0; t < L; ++t) {
                size_t row = ((size_t)page_table[(size_t)b * max_pages_per_seq + t / T] * H + h) * T + t % T;
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += bf16_value(qv[d]) * bf16_value(k_bf16[row * D + d]);
                double w = exp(sm_scale * dot - zmax);
                l += w;
                for (int d = 0; d < D; ++d)
                    o[d] += w * bf16_value(v_bf16[row * D + d]);
            }
            for (int d = 0; d < D; ++d)
                o[d] /= l;
        }
}
