/*
 * qm_oracle.c -- the oracle: a plain, slow CPU restatement of the packed
 * weight formats and of the products over them, computed in float64.
 *
 * TEST INFRASTRUCTURE ONLY. Its users are the tests, the smoke check and the
 * CPU-baseline leg of the benchmark. The CUDA library never includes, links
 * or calls it, and it shares no header, helper, table or constant with the
 * library: every decoder and rounding helper below is written here, from the
 * format definitions.
 *
 * Sources (page title -- section):
 *   [MLX]  "GPTQModel wiki: MLX Apple Silicon" -- "Concepts: method, checkpoint,
 *          runtime, and tensor layout" (affine value = code*scale + bias) and
 *          "Packed layouts and exact transcoding" (continuous little-endian
 *          code stream per uint32 row, lowest index in the lowest bits).
 *   [NXQ]  "Nx_quant (raven-ml.dev API docs)" -- "Weights" (type t: Mxfp4,
 *          Q8_0 layouts; e2m1/e8m0 rules), "Products" (dequant, apply,
 *          apply_experts, take).
 *   [TGP]  "Quantized inference in tinygpt's HFModel" -- "Problem" (uint32
 *          words, companion .scales/.biases, bf16 scales).
 *
 * Conventions shared with the Python wrapper (oracle/__init__.py) only:
 *   format: 0 = MLX affine, 1 = GGUF Q8_0, 2 = MXFP4 (scales apart),
 *           3 = MXFP4 in GGUF's blocks, 4 = GGUF Q4_K, 5 = GGUF Q6_K
 *   dtype : 0 = float32, 1 = bfloat16, 2 = float16
 *   An index array is int32 when its `ids64` flag is 0, int64 otherwise.
 *
 * Readings taken where the pages leave a step open:
 *   - an affine value is ONE float32 rounding of code*scale + bias (IEEE
 *     fusedMultiplyAdd, fmaf), as [NXQ] "Products/dequant" says every value
 *     of a weight is a float32 value;
 *   - scales/biases of an affine weight are row-major [rows, k/group_size],
 *     group g covering inputs [g*gs, (g+1)*gs);
 *   - e2m1: bit 3 is the sign, bits 2..0 index the magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6} in that order;
 *   - a position outside [0, len) -- negative included -- is out of range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Scalar decoders (IEEE-754 binary16, bfloat16, OCP e2m1 / e8m0)      */
/* ------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double or_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0x1F)
        mag = (f == 0) ? INFINITY : NAN;
    else if (e == 0)
        mag = ldexp((double)f, -24);              /* subnormal: f * 2^-24 */
    else
        mag = ldexp((double)(1024 + f), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of a binary32. */
double or_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double mag;
    if (e == 0xFF)
        mag = (f == 0) ? INFINITY : NAN;
    else if (e == 0)
        mag = ldexp((double)f, -133);             /* subnormal: f * 2^-126 / 128 */
    else
        mag = ldexp((double)(128 + f), e - 134);  /* (1 + f/128) * 2^(e-127) */
    return sign ? -mag : mag;
}

/* e2m1 magnitudes in code order, [NXQ] "Weights": 0, .5, 1, 1.5, 2, 3, 4, 6. */
static const double OR_E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double or_e2m1_to_f64(int code)
{
    double m = OR_E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;                   /* sign 1, magnitude 0 -> -0. */
}

/* e8m0: 2^(s-127); the byte 255 is NaN ([NXQ] "Weights"). */
double or_e8m0_to_f64(int s)
{
    if (s == 255)
        return NAN;
    return ldexp(1.0, s - 127);
}

/* ------------------------------------------------------------------ */
/* Rounding helpers: round-to-nearest, ties to even, from the values   */
/* ------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* Round a float32 to bfloat16. The two candidates are the bfloat16 numbers
 * that bracket f (truncation toward zero, and the next one away from zero);
 * the nearer wins and a tie goes to the one with an even last bit. */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
    if (isnan(f))
        return (uint16_t)(sign | 0x7FC0);
    if (isinf(f))
        return (uint16_t)(sign | 0x7F80);
    uint16_t lo = (uint16_t)((u >> 16) & 0x7FFF);   /* |f| truncated */
    uint16_t hi = (uint16_t)(lo + 1);               /* next magnitude (may be inf) */
    double a = fabs((double)f);
    double vlo = or_bf16_to_f64(lo);
    /* above the largest finite bfloat16 the next candidate is 2^128, whose
     * encoding is infinity */
    double vhi = (lo == 0x7F7F) ? ldexp(1.0, 128) : or_bf16_to_f64(hi);
    uint16_t r;
    if (a - vlo < vhi - a)
        r = lo;
    else if (a - vlo > vhi - a)
        r = hi;
    else
        r = (lo & 1) ? hi : lo;
    return (uint16_t)(sign | r);
}

/* Round a float32 to binary16 (subnormals kept, overflow to infinity). */
uint16_t or_f32_to_f16(float f)
{
    uint16_t sign = (f32_bits(f) >> 16) & 0x8000;
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00);
    double a = fabs((double)f);
    if (isinf(f))
        return (uint16_t)(sign | 0x7C00);
    /* quantum of the binade a falls in (the subnormal quantum below 2^-14) */
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    int q_exp = (a < ldexp(1.0, -14)) ? -24 : (e - 1) - 10;
    double r = ldexp(a, -q_exp);  /* a in units of the quantum, exact */
    double fl = floor(r);
    double diff = r - fl;
    double n;
    if (diff > 0.5)
        n = fl + 1.0;
    else if (diff < 0.5)
        n = fl;
    else
        n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = ldexp(n, q_exp);   /* the rounded magnitude, exact */
    if (v > 65504.0)
        return (uint16_t)(sign | 0x7C00);
    if (v < ldexp(1.0, -14))      /* subnormal (or zero): v = n * 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(v, 24));
    frexp(v, &e);
    int be = (e - 1) + 15;                             /* biased exponent */
    uint16_t frac = (uint16_t)(ldexp(v, -(e - 1)) * 1024.0 - 1024.0);
    return (uint16_t)(sign | (be << 10) | frac);
}

static double or_scale_to_f64(const void* p, int64_t i, int sdt)
{
    uint16_t h = ((const uint16_t*)p)[i];
    return (sdt == 2) ? or_f16_to_f64(h) : or_bf16_to_f64(h);
}

/* ------------------------------------------------------------------ */
/* Unpacking and the float32 value of one row                          */
/* ------------------------------------------------------------------ */

/* MLX affine code i of one row: bits [i*b, i*b + b) of the row's words read
 * as one little-endian bit stream, bit t being bit (t mod 32) of word t/32
 * ([MLX] "Packed layouts and exact transcoding"). */
uint32_t or_affine_code(const uint32_t* row_words, int bits, int64_t i)
{
    uint32_t c = 0;
    for (int t = 0; t < bits; ++t) {
        int64_t pos = i * bits + t;
        uint32_t bit = (row_words[pos / 32] >> (pos % 32)) & 1u;
        c |= bit << t;
    }
    return c;
}

/* MXFP4 code i of one row: byte i/2, low nibble for even i, high for odd
 * ([NXQ] "Weights", Mxfp4.codes). */
int or_mxfp4_code(const uint8_t* row_bytes, int64_t i)
{
    uint8_t b = row_bytes[i / 2];
    return (i % 2 == 0) ? (b & 0xF) : (b >> 4);
}

/* MXFP4 in GGUF's blocks ([NXQ] "Weights", Mxfp4_blocks.blocks): 17 bytes per
 * 32 values, the e8m0 scale byte first, then 16 bytes; byte j holds value j
 * of the block in its low nibble and value j + 16 in its high nibble. */
static int or_mxfp4_block_code(const uint8_t* block, int t)
{
    uint8_t b = block[1 + (t % 16)];
    return (t < 16) ? (b & 0xF) : (b >> 4);
}

/* Q8_0 block layout ([NXQ] "Weights", Q8_0.blocks): 34 bytes per 32 values,
 * a little-endian float16 d, then 32 int8 quants. */
static double or_q8_0_d(const uint8_t* block)
{
    uint16_t h = (uint16_t)(block[0] | (block[1] << 8));
    return or_f16_to_f64(h);
}

static int or_q8_0_q(const uint8_t* block, int t)
{
    return (int)(int8_t)block[2 + t];
}

/* GGUF Q4_K ([NXQ] "Weights", Q4_K): 144 bytes per 256 values -- float16 d,
 * float16 dmin, 12 bytes holding eight 6-bit scales and eight 6-bit mins (one
 * each per sub-block of 32 values), then 128 bytes of 4-bit quants. The page
 * gives the fields and their order and defers the arrangement inside them to
 * ggml's block_q4_K; that arrangement, restated:
 *   - the 12 bytes as bytes b0..b11: sub-blocks 0..3 take their scale from the
 *     low 6 bits of b0..b3 and their min from the low 6 bits of b4..b7;
 *     sub-blocks 4..7 take the low 4 bits of their scale from the low nibble
 *     of b8..b11 and of their min from its high nibble, and the top 2 bits of
 *     their scale from the top 2 bits of b0..b3, of their min from the top 2
 *     bits of b4..b7;
 *   - the quants in four runs of 32 bytes, run c serving values 64c .. 64c+63:
 *     its byte l holds value 64c + l in the low nibble (sub-block 2c) and
 *     value 64c + 32 + l in the high nibble (sub-block 2c + 1).
 * Value = d * sc * q - dmin * m ([NXQ]), computed as ggml's float32 dequant
 * computes it, products left to right: every product is exact in float32 and
 * the value rounds once, at the subtraction ([NXQ] "Products", dequant). */
static void or_q4_k_sub(const uint8_t* blk, int j, int* sc, int* m)
{
    const uint8_t* b = blk + 4;                 /* the 12 scale/min bytes */
    if (j < 4) {
        *sc = b[j] & 0x3F;
        *m = b[4 + j] & 0x3F;
    } else {
        *sc = (b[8 + (j - 4)] & 0x0F) | ((b[j - 4] >> 6) << 4);
        *m = (b[8 + (j - 4)] >> 4) | ((b[j] >> 6) << 4);
    }
}

static float or_q4_k_value(const uint8_t* blk, int i)
{
    double d = or_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = or_f16_to_f64((uint16_t)(blk[2] | (blk[3] << 8)));
    int c = i / 64, r = i % 64;
    int j = 2 * c + (r >= 32);                  /* sub-block */
    uint8_t byte = blk[16 + 32 * c + (r % 32)];
    int q = (r < 32) ? (byte & 0x0F) : (byte >> 4);
    int sc, m;
    or_q4_k_sub(blk, j, &sc, &m);
    /* d * sc * q and dmin * m are exact in float64 and their difference too
     * (at most 50 bits apart): the cast is the one rounding */
    return (float)(d * sc * q - dmin * m);
}

/* GGUF Q6_K ([NXQ] "Weights", Q6_K): 210 bytes per 256 values -- 128 bytes of
 * the quants' low 4 bits (ql), 64 bytes of their high 2 bits (qh), sixteen
 * int8 scales (one per sub-block of 16 values), then float16 d. The
 * arrangement inside the fields (ggml's block_q6_K), restated: the block is two
 * halves of 128 values, half h using ql[64h .. 64h+63], qh[32h .. 32h+31] and
 * scales[8h .. 8h+7]; within a half, value 32t + l (t = 0..3, l = 0..31) has
 * its low 4 bits in ql[64h + l + 32(t mod 2)] (the low nibble for t < 2, the
 * high one for t >= 2), its high 2 bits in bits 2t, 2t+1 of qh[32h + l], and
 * the scale scales[8h + 2t + l/16]. Value = d * sc * (q - 32) ([NXQ]), exact
 * in float32. */
static float or_q6_k_value(const uint8_t* blk, int i)
{
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    const int8_t* scales = (const int8_t*)(blk + 192);
    double d = or_f16_to_f64((uint16_t)(blk[208] | (blk[209] << 8)));
    int h = i / 128, r = i % 128, t = r / 32, l = r % 32;
    uint8_t lo_byte = ql[64 * h + l + 32 * (t % 2)];
    int lo = (t < 2) ? (lo_byte & 0x0F) : (lo_byte >> 4);
    int hi = (qh[32 * h + l] >> (2 * t)) & 3;
    int q = lo | (hi << 4);
    int sc = scales[8 * h + 2 * t + l / 16];
    return (float)(d * sc * (q - 32));
}

/* Float32 values of row r (of `rows`) of a weight, k of them, into v[k]. */
void or_row_values(int fmt, int bits, int gs, int sdt, int64_t k,
                   const void* codes, const void* scales, const void* biases,
                   int64_t r, float* v)
{
    if (fmt == 0) {                                   /* MLX affine */
        int64_t words = k * bits / 32;
        const uint32_t* rw = (const uint32_t*)codes + r * words;
        int64_t ng = k / gs;
        for (int64_t i = 0; i < k; ++i) {
            uint32_t c = or_affine_code(rw, bits, i);
            float s = (float)or_scale_to_f64(scales, r * ng + i / gs, sdt);
            float b = (float)or_scale_to_f64(biases, r * ng + i / gs, sdt);
            v[i] = fmaf((float)c, s, b);              /* one rounding */
        }
    } else if (fmt == 1) {                            /* GGUF Q8_0 */
        const uint8_t* rb = (const uint8_t*)codes + r * (k / 32) * 34;
        for (int64_t i = 0; i < k; ++i) {
            const uint8_t* blk = rb + (i / 32) * 34;
            v[i] = (float)(or_q8_0_d(blk) * (double)or_q8_0_q(blk, (int)(i % 32)));
        }
    } else if (fmt == 4) {                            /* GGUF Q4_K */
        const uint8_t* rb = (const uint8_t*)codes + r * (k / 256) * 144;
        for (int64_t i = 0; i < k; ++i)
            v[i] = or_q4_k_value(rb + (i / 256) * 144, (int)(i % 256));
    } else if (fmt == 5) {                            /* GGUF Q6_K */
        const uint8_t* rb = (const uint8_t*)codes + r * (k / 256) * 210;
        for (int64_t i = 0; i < k; ++i)
            v[i] = or_q6_k_value(rb + (i / 256) * 210, (int)(i % 256));
    } else if (fmt == 3) {                            /* MXFP4 in GGUF's blocks */
        const uint8_t* rb = (const uint8_t*)codes + r * (k / 32) * 17;
        for (int64_t i = 0; i < k; ++i) {
            const uint8_t* blk = rb + (i / 32) * 17;
            double x = or_e2m1_to_f64(or_mxfp4_block_code(blk, (int)(i % 32))) * or_e8m0_to_f64(blk[0]);
            v[i] = (float)x;                          /* exact, or +-inf past float32 */
        }
    } else {                                          /* MXFP4, scales apart */
        const uint8_t* rc = (const uint8_t*)codes + r * (k / 2);
        const uint8_t* rs = (const uint8_t*)scales + r * (k / 32);
        for (int64_t i = 0; i < k; ++i) {
            double x = or_e2m1_to_f64(or_mxfp4_code(rc, i)) * or_e8m0_to_f64(rs[i / 32]);
            v[i] = (float)x;                          /* exact, or +-inf past float32 */
        }
    }
}

/* ------------------------------------------------------------------ */
/* dequant: every value rounded once to the output dtype               */
/* ([NXQ] "Products", dequant)                                         */
/* ------------------------------------------------------------------ */

static void or_store(void* out, int64_t idx, int dt, float v)
{
    if (dt == 0)
        ((float*)out)[idx] = v;
    else if (dt == 1)
        ((uint16_t*)out)[idx] = or_f32_to_bf16(v);
    else
        ((uint16_t*)out)[idx] = or_f32_to_f16(v);
}

/* ------------------------------------------------------------------ */
/* quantize_q8_0: float32 rows to Q8_0 blocks ([NXQ] "Weights",        */
/* val quantize_q8_0)                                                   */
/* ------------------------------------------------------------------ */

/* x [rows, k] float32 -> blocks [rows, k/32*34]. Per block of 32 values:
 * a NaN anywhere gives a NaN scale and quants 0; else an infinity gives the
 * scale +inf and quants 0; else d = amax / 127 at float32, stored at float16
 * rounded to nearest, and quant j = round(v_j * (1 / d)) with halves away from
 * zero, the reciprocal and products at float32 and 1/d = 0 where d is 0; a
 * product that is not finite (1/d past float32's range) has the quant 0. */
void or_quantize_q8_0(const float* x, int64_t rows, int64_t k, uint8_t* blocks)
{
    int64_t nb = k / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const float* v = x + r * k + b * 32;
            uint8_t* out = blocks + (r * nb + b) * 34;
            int has_nan = 0, has_inf = 0;
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                if (isnan(v[j]))
                    has_nan = 1;
                else if (isinf(v[j]))
                    has_inf = 1;
                else if (fabsf(v[j]) > amax)
                    amax = fabsf(v[j]);
            }
            uint16_t h;
            int8_t q[32];
            if (has_nan || has_inf) {
                h = has_nan ? 0x7E00 : 0x7C00;
                for (int j = 0; j < 32; ++j) q[j] = 0;
            } else {
                float d = amax / 127.0f;
                float id = (d != 0.0f) ? 1.0f / d : 0.0f;
                h = or_f32_to_f16(d);
                for (int j = 0; j < 32; ++j) {
                    float p = v[j] * id;
                    q[j] = isfinite(p) ? (int8_t)roundf(p) : 0;
                }
            }
            out[0] = (uint8_t)(h & 0xFF);          /* little-endian float16 */
            out[1] = (uint8_t)(h >> 8);
            for (int j = 0; j < 32; ++j) out[2 + j] = (uint8_t)q[j];
        }
}

/* rows = product of the leading axes times n; out is [rows, k] of dtype dt. */
void or_dequant(int fmt, int bits, int gs, int sdt, int64_t rows, int64_t k,
                const void* codes, const void* scales, const void* biases,
                int dt, void* out)
{
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)k);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            or_row_values(fmt, bits, gs, sdt, k, codes, scales, biases, r, v);
            for (int64_t i = 0; i < k; ++i)
                or_store(out, r * k + i, dt, v[i]);
        }
        free(v);
    }
}

/* ------------------------------------------------------------------ */
/* apply: y[m, j] = sum_i x[m, i] * w[j, i], float64, i ascending      */
/* ([NXQ] "Products", apply). The result is left unrounded: the final  */
/* rounding to x's dtype is the comparison's business.                 */
/* ------------------------------------------------------------------ */

static double or_load(const void* p, int64_t idx, int dt)
{
    if (dt == 0)
        return (double)((const float*)p)[idx];
    if (dt == 1)
        return or_bf16_to_f64(((const uint16_t*)p)[idx]);
    return or_f16_to_f64(((const uint16_t*)p)[idx]);
}

/* x is [M, k] of dtype xdt; y is [M, rows] float64. */
void or_apply(int fmt, int bits, int gs, int sdt, int64_t rows, int64_t k,
              const void* codes, const void* scales, const void* biases,
              const void* x, int xdt, int64_t M, double* y)
{
    double* xd = (double*)malloc(sizeof(double) * (size_t)(M * k + 1));
    for (int64_t t = 0; t < M * k; ++t)
        xd[t] = or_load(x, t, xdt);
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)k);
#pragma omp for schedule(dynamic, 16)
        for (int64_t j = 0; j < rows; ++j) {
            or_row_values(fmt, bits, gs, sdt, k, codes, scales, biases, j, v);
            for (int64_t m = 0; m < M; ++m) {
                double acc = 0.0;
                for (int64_t i = 0; i < k; ++i)
                    acc += xd[m * k + i] * (double)v[i];
                y[m * rows + j] = acc;
            }
        }
        free(v);
    }
    free(xd);
}

/* Selected entries of the same product: out[e] = y[m_idx[e], j_idx[e]].
 * Used where the full product is too large for the oracle. */
void or_apply_entries(int fmt, int bits, int gs, int sdt, int64_t rows, int64_t k,
                      const void* codes, const void* scales, const void* biases,
                      const void* x, int xdt, int64_t n_entries,
                      const int64_t* m_idx, const int64_t* j_idx, double* out)
{
    (void)rows;
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)k);
#pragma omp for schedule(dynamic, 4)
        for (int64_t e = 0; e < n_entries; ++e) {
            or_row_values(fmt, bits, gs, sdt, k, codes, scales, biases, j_idx[e], v);
            double acc = 0.0;
            for (int64_t i = 0; i < k; ++i)
                acc += or_load(x, m_idx[e] * k + i, xdt) * (double)v[i];
            out[e] = acc;
        }
        free(v);
    }
}

/* ------------------------------------------------------------------ */
/* take: gather along an axis of each packed part, no decoding         */
/* ([NXQ] "Products", take). A part is viewed as [outer, len, inner]    */
/* bytes around the gathered axis; out is [outer, n_ids, inner].        */
/* A position outside [0, len) gathers zero bytes.                      */
/* ------------------------------------------------------------------ */

static int64_t or_id(const void* ids, int ids64, int64_t p)
{
    return ids64 ? ((const int64_t*)ids)[p] : (int64_t)((const int32_t*)ids)[p];
}

void or_take_part(const void* src, int64_t outer, int64_t len, int64_t inner_bytes,
                  const void* ids, int ids64, int64_t n_ids, void* dst)
{
    const uint8_t* s = (const uint8_t*)src;
    uint8_t* d = (uint8_t*)dst;
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t p = 0; p < n_ids; ++p) {
            int64_t id = or_id(ids, ids64, p);
            uint8_t* dp = d + (o * n_ids + p) * inner_bytes;
            if (id >= 0 && id < len)
                memcpy(dp, s + (o * len + id) * inner_bytes, (size_t)inner_bytes);
            else
                memset(dp, 0, (size_t)inner_bytes);
        }
}

/* ------------------------------------------------------------------ */
/* Routing: a stable sort of the flattened positions by expert id      */
/* ([NXQ] "Products", apply_experts: positions in range are summed in  */
/* one contraction, each with the matrix its id names).                */
/* counts[e] = positions naming e; offsets[e] = sum of counts before e */
/* (offsets[E] = positions in range); perm lists the in-range positions */
/* by ascending expert, ties by ascending position. Returns the number  */
/* of positions out of range.                                           */
/* ------------------------------------------------------------------ */

int64_t or_route(const void* ids, int ids64, int64_t P, int64_t E,
                 int64_t* counts, int64_t* offsets, int64_t* perm)
{
    int64_t c = 0;
    for (int64_t e = 0; e < E; ++e) {
        offsets[e] = c;
        counts[e] = 0;
        for (int64_t p = 0; p < P; ++p)
            if (or_id(ids, ids64, p) == e) {
                perm[c++] = p;
                counts[e]++;
            }
    }
    offsets[E] = c;
    return P - c;
}

/* ------------------------------------------------------------------ */
/* apply_experts ([NXQ] "Products", apply_experts): at each position p */
/* of ids [T, topk], the product of expert ids[p]'s matrix [n, k] with  */
/* p's row of x, or zeros where ids[p] is not in [0, E). x has x_rows   */
/* rows: T (one row per token, broadcast over its topk positions) or    */
/* T*topk (one row per position). y is [T*topk, n] float64.             */
/* ------------------------------------------------------------------ */

static int64_t or_x_row(int64_t p, int64_t topk, int64_t x_rows, int64_t T)
{
    return (x_rows == T) ? p / topk : p;
}

void or_apply_experts(int fmt, int bits, int gs, int sdt, int64_t E, int64_t n, int64_t k,
                      const void* codes, const void* scales, const void* biases,
                      const void* ids, int ids64, int64_t T, int64_t topk,
                      const void* x, int64_t x_rows, int xdt, double* y)
{
    int64_t P = T * topk;
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)k);
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < P; ++p) {
            int64_t id = or_id(ids, ids64, p);
            if (id < 0 || id >= E) {
                for (int64_t j = 0; j < n; ++j)
                    y[p * n + j] = 0.0;
                continue;
            }
            int64_t xr = or_x_row(p, topk, x_rows, T);
            for (int64_t j = 0; j < n; ++j) {
                or_row_values(fmt, bits, gs, sdt, k, codes, scales, biases, id * n + j, v);
                double acc = 0.0;
                for (int64_t i = 0; i < k; ++i)
                    acc += or_load(x, xr * k + i, xdt) * (double)v[i];
                y[p * n + j] = acc;
            }
        }
        free(v);
    }
}

/* Selected entries of apply_experts: out[e] = y[p_idx[e], j_idx[e]]. */
void or_apply_experts_entries(int fmt, int bits, int gs, int sdt, int64_t E, int64_t n, int64_t k,
                              const void* codes, const void* scales, const void* biases,
                              const void* ids, int ids64, int64_t T, int64_t topk,
                              const void* x, int64_t x_rows, int xdt,
                              int64_t n_entries, const int64_t* p_idx, const int64_t* j_idx,
                              double* out)
{
#pragma omp parallel
    {
        float* v = (float*)malloc(sizeof(float) * (size_t)k);
#pragma omp for schedule(dynamic, 4)
        for (int64_t e = 0; e < n_entries; ++e) {
            int64_t p = p_idx[e];
            int64_t id = or_id(ids, ids64, p);
            if (id < 0 || id >= E) {
                out[e] = 0.0;
                continue;
            }
            int64_t xr = or_x_row(p, topk, x_rows, T);
            or_row_values(fmt, bits, gs, sdt, k, codes, scales, biases, id * n + j_idx[e], v);
            double acc = 0.0;
            for (int64_t i = 0; i < k; ++i)
                acc += or_load(x, xr * k + i, xdt) * (double)v[i];
            out[e] = acc;
        }
        free(v);
    }
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Vector forms of the scalar helpers above, for exhaustive checks.
 * or_round_array: float32 -> dtype dt (0 f32 copy, 1 bf16, 2 f16).
 * or_decode_array: 16-bit patterns of dtype dt (1 bf16, 2 f16) -> float64. */
void or_round_array(const float* in, int64_t count, int dt, void* out)
{
    for (int64_t i = 0; i < count; ++i)
        or_store(out, i, dt, in[i]);
}

void or_decode_array(const uint16_t* in, int64_t count, int dt, double* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = (dt == 1) ? or_bf16_to_f64(in[i]) : or_f16_to_f64(in[i]);
}
