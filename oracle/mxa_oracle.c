/*
 * mxa_oracle.c -- plain, slow CPU oracle for MXFP8 block-scaled attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Sources (page titles, sections):
 *   [FA4]    "Flash Attention 4 + MXFP8 on Blackwell" (aixai.ru write-up):
 *            "Что такое MXFP8", "Квантование dS без транспонирования".
 *   [FLAMIA] "FLAMIA 阅读笔记" (reading notes on FLAMIA):
 *            sec. 2 "前置知识" (attention, softmax gradient, online softmax,
 *            the two hardware formats), sec. 3 (token blocks, Hadamard),
 *            sec. 4 "E4M3 为什么常常不受尺度翻倍影响" (scale rule
 *            e = ceil(log2(a/448))), sec. 6 (packed documents, visible pairs).
 *
 * Everything here is written from the format and the equations, in fp64,
 * without tiling, fusion or reordering:
 *   - E4M3 (OCP "fn" variant): bias 7, normals (1+m/8)*2^(E-7), subnormals
 *     m*2^-9, 0x7F/0xFF NaN, max finite 448, no infinity.  Encoding picks the
 *     nearest representable value (ties to the even code), saturating to 448.
 *   - UE8M0: byte b is the power of two 2^(b-127).
 *   - Scale exponent: the smallest integer e with amax / 2^e <= 448
 *     ([FLAMIA] sec. 4, the saturation bound); an all-zero group takes e = 0.
 *   - Attention: S = alpha Q K^T, P = softmax over the visible keys,
 *     O = P V, LSE = m + ln l ([FLAMIA] sec. 2).
 *   - Backward: dV = P^T G, E = G V^T, D = G.O, U = P (E - D),
 *     dQ = alpha U K, dK = alpha U^T Q ([FLAMIA] sec. 2).
 *   - Algorithm 1 ([FLAMIA] sec. 5): the same direct attention with the
 *     roundings its steps name (orc_attn_fwd_alg1, orc_attn_bwd_alg1).
 *
 * Unpinned: none.  orc_dq_row_boost states a reading (the bound a library
 * documents for its per-row FP16 dQ boost; the pages give only the shape of
 * the choice), pinned by checking that the bound holds.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Formats                                                                   */
/* ------------------------------------------------------------------------ */

/* bf16 bit pattern -> double (exact: bf16 is the top half of an fp32). */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* E4M3 decode, from the field definition. */
double orc_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int E = (c >> 3) & 0xF;
    int M = c & 7;
    double v;
    if (E == 15 && M == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)M, -9);
    else
        v = ldexp(1.0 + M / 8.0, E - 7);
    return s ? -v : v;
}

/* E4M3 encode: nearest of the 127 non-negative finite values (0x00..0x7E),
 * ties to the even code (= even mantissa), saturating to 448; the sign bit is
 * kept, so a negative value that rounds to zero gives 0x80. */
uint8_t orc_e4m3_encode(double y)
{
    if (isnan(y))
        return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    if (a >= 448.0)
        return sign | 0x7E;
    int best = 0;
    double best_err = a; /* distance to code 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

/* Element-wise encode of n values (used by the exhaustive codec checks). */
void orc_e4m3_encode_array(const double* y, int64_t n, uint8_t* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(y[i]);
}

/* UE8M0 byte <-> power of two. */
double orc_ue8m0_decode(uint8_t b)
{
    if (b == 0xFF)
        return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* Scale exponent of a group with max magnitude amax: the smallest integer e
 * such that amax / 2^e <= 448.  All-zero groups take e = 0 (the agreed finite
 * scale).  The result is clamped to the UE8M0 range [-127, 127]. */
int orc_mx_exponent(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int e = ilogb(amax) - 10; /* certainly too small: amax/2^e >= 2^10 > 448 */
    while (amax > ldexp(448.0, e))
        ++e;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* ------------------------------------------------------------------------ */
/* Document geometry                                                         */
/* ------------------------------------------------------------------------ */

/* cu_seqlens == NULL means one document covering all T tokens. */
static void doc_range(const int32_t* cu, int ndocs, int64_t T, int b, int64_t* s, int64_t* e)
{
    if (!cu) {
        *s = 0;
        *e = T;
        (void)ndocs;
        (void)b;
        return;
    }
    *s = cu[b];
    *e = cu[b + 1];
}

static int num_docs_eff(const int32_t* cu, int ndocs) { return cu ? ndocs : 1; }

/* Number of 32-token groups of a document of n tokens, counted from its start. */
static int64_t nblk32(int64_t n) { return (n + 31) / 32; }

/* Offset of document b's first 32-token group in the concatenated group list. */
int64_t orc_block_offset(const int32_t* cu, int ndocs, int64_t T, int b)
{
    int64_t off = 0;
    for (int i = 0; i < b; ++i) {
        int64_t s, e;
        doc_range(cu, ndocs, T, i, &s, &e);
        off += nblk32(e - s);
    }
    return off;
}

int64_t orc_total_blocks(const int32_t* cu, int ndocs, int64_t T)
{
    return orc_block_offset(cu, ndocs, T, num_docs_eff(cu, ndocs));
}

/* Visible (query, key) pairs of causal documents: sum n (n + 1) / 2
 * ([FLAMIA] sec. 6). */
int64_t orc_visible_pairs(const int32_t* cu, int ndocs, int64_t T)
{
    int64_t c = 0;
    for (int b = 0; b < num_docs_eff(cu, ndocs); ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        c += (e - s) * (e - s + 1) / 2;
    }
    return c;
}

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                */
/* ------------------------------------------------------------------------ */

/* Row view: one scale per (token, head, 32 consecutive channels).
 * x: bf16 bits [T, H, d]; codes: [T, H, d]; scales: UE8M0 bytes [T, H, d/32]. */
void orc_quant_row(const uint16_t* x, int64_t T, int H, int d, uint8_t* codes, uint8_t* scales)
{
    int G = d / 32;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h)
            for (int g = 0; g < G; ++g) {
                const uint16_t* xs = x + (t * H + h) * d + g * 32;
                double amax = 0.0;
                for (int i = 0; i < 32; ++i) {
                    double v = fabs(orc_bf16_to_double(xs[i]));
                    if (v > amax)
                        amax = v;
                }
                int e = orc_mx_exponent(amax);
                for (int i = 0; i < 32; ++i)
                    codes[(t * H + h) * d + g * 32 + i] = orc_e4m3_encode(ldexp(orc_bf16_to_double(xs[i]), -e));
                scales[(t * H + h) * G + g] = (uint8_t)(e + 127);
            }
}

/* Per-key view ([FLAMIA] sec. 4, moving the scale across the boundary: each
 * key of a diagonal tile carries its own power-of-two scale): one scale per
 * (token, head) over all d channels, by the same rule as every MX group.
 * codes [T, H, d]; scales: logical [T, H]. */
void orc_quant_key(const uint16_t* x, int64_t T, int H, int d, uint8_t* codes, uint8_t* scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            const uint16_t* xs = x + (t * H + h) * d;
            double amax = 0.0;
            for (int i = 0; i < d; ++i) {
                double v = fabs(orc_bf16_to_double(xs[i]));
                if (v > amax)
                    amax = v;
            }
            int e = orc_mx_exponent(amax);
            for (int i = 0; i < d; ++i)
                codes[(t * H + h) * d + i] = orc_e4m3_encode(ldexp(orc_bf16_to_double(xs[i]), -e));
            scales[t * H + h] = (uint8_t)(e + 127);
        }
}

/* Token view: one scale per (document, 32 consecutive tokens counted from the
 * document start, head, channel); the last group of a document may be short
 * and no group crosses a document boundary.
 * scales: logical [H, d, NB] with NB = sum over docs of ceil(n/32), document
 * b's groups starting at orc_block_offset(b). */
void orc_quant_tok(const uint16_t* x, int64_t T, int H, int d, const int32_t* cu, int ndocs,
                   uint8_t* codes, uint8_t* scales)
{
    int nd = num_docs_eff(cu, ndocs);
    int64_t NB = orc_total_blocks(cu, ndocs, T);
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t boff = orc_block_offset(cu, ndocs, T, b);
        int64_t nbk = nblk32(e - s);
#pragma omp parallel for schedule(static)
        for (int64_t kb = 0; kb < nbk; ++kb) {
            int64_t t0 = s + kb * 32, t1 = t0 + 32 < e ? t0 + 32 : e;
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < d; ++c) {
                    double amax = 0.0;
                    for (int64_t t = t0; t < t1; ++t) {
                        double v = fabs(orc_bf16_to_double(x[(t * H + h) * d + c]));
                        if (v > amax)
                            amax = v;
                    }
                    int ex = orc_mx_exponent(amax);
                    for (int64_t t = t0; t < t1; ++t)
                        codes[(t * H + h) * d + c] = orc_e4m3_encode(ldexp(orc_bf16_to_double(x[(t * H + h) * d + c]), -ex));
                    scales[((int64_t)h * d + c) * NB + boff + kb] = (uint8_t)(ex + 127);
                }
        }
    }
}

/* Normalized 128-point Hadamard rotation of one vector, in IEEE fp32, in the
 * Sylvester order: for h = 1, 2, 4, ..., 64, every pair (i, i + h) inside a
 * block of 2h becomes (a + b, a - b); the result is multiplied by the fp32
 * value of 128^(-1/2).  ([FLAMIA] sec. 3, "旋转为什么有时适得其反": the
 * rotation H with H H^T = I leaves Q K^T unchanged.)  The fp32 sequence is the
 * reading taken because the codes computed from it must match bit for bit. */
void orc_hadamard128_f32(const float* in, float* out)
{
    float v[128];
    for (int i = 0; i < 128; ++i)
        v[i] = in[i];
    for (int h = 1; h < 128; h *= 2)
        for (int i = 0; i < 128; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
    const float r = (float)0.08838834764831845; /* fp32 nearest to 128^-1/2 */
    for (int i = 0; i < 128; ++i)
        out[i] = v[i] * r;
}

/* Token-block view ([FLAMIA] sec. 3, "让同一份码跨两个方向使用"): one
 * exponent per (document, 32 consecutive tokens from the document start,
 * head) shared by all d channels; the same codes serve both contraction axes.
 * With hadamard != 0 (d == 128) every (token, head) vector is first rotated
 * (orc_hadamard128_f32) and the block statistics are taken on the rotated
 * fp32 values.  scales: logical [H, NB]. */
void orc_quant_tokblock(const uint16_t* x, int64_t T, int H, int d, const int32_t* cu, int ndocs,
                        int hadamard, uint8_t* codes, uint8_t* scales)
{
    int nd = num_docs_eff(cu, ndocs);
    int64_t NB = orc_total_blocks(cu, ndocs, T);
    float* y = (float*)malloc(sizeof(float) * (size_t)T * H * d);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            float in[128];
            const uint16_t* xs = x + (t * H + h) * d;
            float* ys = y + (t * H + h) * d;
            if (hadamard) {
                for (int i = 0; i < 128; ++i)
                    in[i] = (float)orc_bf16_to_double(xs[i]);
                orc_hadamard128_f32(in, ys);
            } else {
                for (int i = 0; i < d; ++i)
                    ys[i] = (float)orc_bf16_to_double(xs[i]);
            }
        }
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t boff = orc_block_offset(cu, ndocs, T, b);
        int64_t nbk = nblk32(e - s);
#pragma omp parallel for schedule(static)
        for (int64_t kb = 0; kb < nbk; ++kb) {
            int64_t t0 = s + kb * 32, t1 = t0 + 32 < e ? t0 + 32 : e;
            for (int h = 0; h < H; ++h) {
                double amax = 0.0;
                for (int64_t t = t0; t < t1; ++t)
                    for (int c = 0; c < d; ++c) {
                        double v = fabs((double)y[(t * H + h) * d + c]);
                        if (v > amax)
                            amax = v;
                    }
                int ex = orc_mx_exponent(amax);
                for (int64_t t = t0; t < t1; ++t)
                    for (int c = 0; c < d; ++c)
                        codes[(t * H + h) * d + c] = orc_e4m3_encode(ldexp((double)y[(t * H + h) * d + c], -ex));
                scales[(int64_t)h * NB + boff + kb] = (uint8_t)(ex + 127);
            }
        }
    }
    free(y);
}

/* ------------------------------------------------------------------------ */
/* RMSNorm feeding the quantizers (fused producer)                           */
/* ------------------------------------------------------------------------ */

/* RMSNorm of every (token, head) vector of x (bf16 bits [T, H, d]) in IEEE
 * fp32 ([FA4 write-up], "Fused RMSNorm+Quantize": the normalization runs as
 * the prologue of the quantizer that reads the data anyway).  The fp32
 * sequence is the reading taken so that the codes computed from y match bit
 * for bit:
 *   s_k = sum of x_c * x_c over channels 16k .. 16k + 15, in channel order;
 *   s = the d/16 partial sums added pairwise: (s0 + s1), (s2 + s3), ... then
 *       the pairs of those, and so on;
 *   r = 1 / sqrt(s / d + eps) (correctly rounded sqrt and division), 0 when
 *       s / d + eps is 0;
 *   y_c = (x_c * r) * w_c (w == NULL: w_c = 1).
 * y: fp32 [T, H, d]. */
void orc_rmsnorm_f32(const uint16_t* x, int64_t T, int H, int d, const float* w, float eps, float* y)
{
    int nk = d / 16;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T * H; ++r) {
        const uint16_t* xs = x + r * d;
        float part[8];
        for (int k = 0; k < nk; ++k) {
            float acc = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float v = (float)orc_bf16_to_double(xs[16 * k + i]);
                float sq = v * v;
                acc = acc + sq;
            }
            part[k] = acc;
        }
        for (int span = 1; span < nk; span *= 2)
            for (int k = 0; k + span < nk; k += 2 * span)
                part[k] = part[k] + part[k + span];
        float ms = part[0] / (float)d;
        float den = ms + eps;
        float rr = den == 0.0f ? 0.0f : 1.0f / sqrtf(den);
        for (int c = 0; c < d; ++c) {
            float v = (float)orc_bf16_to_double(xs[c]);
            float t = v * rr;
            y[r * d + c] = w ? t * w[c] : t;
        }
    }
}

/* The quantizers of fp32 input (the RMSNorm output): the same rules as
 * orc_quant_row, orc_quant_tok and orc_quant_tokblock, reading fp32 values. */
void orc_quant_row_f32(const float* x, int64_t T, int H, int d, uint8_t* codes, uint8_t* scales)
{
    int G = d / 32;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h)
            for (int g = 0; g < G; ++g) {
                const float* xs = x + (t * H + h) * d + g * 32;
                double amax = 0.0;
                for (int i = 0; i < 32; ++i) {
                    double v = fabs((double)xs[i]);
                    if (v > amax)
                        amax = v;
                }
                int e = orc_mx_exponent(amax);
                for (int i = 0; i < 32; ++i)
                    codes[(t * H + h) * d + g * 32 + i] = orc_e4m3_encode(ldexp((double)xs[i], -e));
                scales[(t * H + h) * G + g] = (uint8_t)(e + 127);
            }
}

void orc_quant_tok_f32(const float* x, int64_t T, int H, int d, const int32_t* cu, int ndocs, uint8_t* codes,
                       uint8_t* scales)
{
    int nd = num_docs_eff(cu, ndocs);
    int64_t NB = orc_total_blocks(cu, ndocs, T);
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t boff = orc_block_offset(cu, ndocs, T, b);
        int64_t nbk = nblk32(e - s);
#pragma omp parallel for schedule(static)
        for (int64_t kb = 0; kb < nbk; ++kb) {
            int64_t t0 = s + kb * 32, t1 = t0 + 32 < e ? t0 + 32 : e;
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < d; ++c) {
                    double amax = 0.0;
                    for (int64_t t = t0; t < t1; ++t) {
                        double v = fabs((double)x[(t * H + h) * d + c]);
                        if (v > amax)
                            amax = v;
                    }
                    int ex = orc_mx_exponent(amax);
                    for (int64_t t = t0; t < t1; ++t)
                        codes[(t * H + h) * d + c] = orc_e4m3_encode(ldexp((double)x[(t * H + h) * d + c], -ex));
                    scales[((int64_t)h * d + c) * NB + boff + kb] = (uint8_t)(ex + 127);
                }
        }
    }
}

void orc_quant_tokblock_f32(const float* x, int64_t T, int H, int d, const int32_t* cu, int ndocs, int hadamard,
                            uint8_t* codes, uint8_t* scales)
{
    int nd = num_docs_eff(cu, ndocs);
    int64_t NB = orc_total_blocks(cu, ndocs, T);
    float* y = (float*)malloc(sizeof(float) * (size_t)T * H * d);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T * H; ++r) {
        if (hadamard)
            orc_hadamard128_f32(x + r * d, y + r * d);
        else
            for (int i = 0; i < d; ++i)
                y[r * d + i] = x[r * d + i];
    }
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t boff = orc_block_offset(cu, ndocs, T, b);
        int64_t nbk = nblk32(e - s);
#pragma omp parallel for schedule(static)
        for (int64_t kb = 0; kb < nbk; ++kb) {
            int64_t t0 = s + kb * 32, t1 = t0 + 32 < e ? t0 + 32 : e;
            for (int h = 0; h < H; ++h) {
                double amax = 0.0;
                for (int64_t t = t0; t < t1; ++t)
                    for (int c = 0; c < d; ++c) {
                        double v = fabs((double)y[(t * H + h) * d + c]);
                        if (v > amax)
                            amax = v;
                    }
                int ex = orc_mx_exponent(amax);
                for (int64_t t = t0; t < t1; ++t)
                    for (int c = 0; c < d; ++c)
                        codes[(t * H + h) * d + c] = orc_e4m3_encode(ldexp((double)y[(t * H + h) * d + c], -ex));
                scales[(int64_t)h * NB + boff + kb] = (uint8_t)(ex + 127);
            }
        }
    }
    free(y);
}

/* ------------------------------------------------------------------------ */
/* Dequantization (exact in fp64): value = decode(code) * 2^(byte - 127)      */
/* ------------------------------------------------------------------------ */

void orc_dequant_row(const uint8_t* codes, const uint8_t* scales, int64_t T, int H, int d, double* out)
{
    int G = d / 32;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < d; ++c)
                out[(t * H + h) * d + c] = orc_e4m3_decode(codes[(t * H + h) * d + c]) *
                                           orc_ue8m0_decode(scales[(t * H + h) * G + c / 32]);
}

void orc_dequant_tok(const uint8_t* codes, const uint8_t* scales, int64_t T, int H, int d,
                     const int32_t* cu, int ndocs, double* out)
{
    int64_t NB = orc_total_blocks(cu, ndocs, T);
    for (int b = 0; b < num_docs_eff(cu, ndocs); ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t boff = orc_block_offset(cu, ndocs, T, b);
#pragma omp parallel for schedule(static)
        for (int64_t t = s; t < e; ++t)
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < d; ++c)
                    out[(t * H + h) * d + c] = orc_e4m3_decode(codes[(t * H + h) * d + c]) *
                                               orc_ue8m0_decode(scales[((int64_t)h * d + c) * NB + boff + (t - s) / 32]);
    }
}

void orc_dequant_tokblock(const uint8_t* codes, const uint8_t* scales, int64_t T, int H, int d,
                          const int32_t* cu, int ndocs, double* out)
{
    int64_t NB = orc_total_blocks(cu, ndocs, T);
    for (int b = 0; b < num_docs_eff(cu, ndocs); ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t boff = orc_block_offset(cu, ndocs, T, b);
#pragma omp parallel for schedule(static)
        for (int64_t t = s; t < e; ++t)
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < d; ++c)
                    out[(t * H + h) * d + c] = orc_e4m3_decode(codes[(t * H + h) * d + c]) *
                                               orc_ue8m0_decode(scales[(int64_t)h * NB + boff + (t - s) / 32]);
    }
}

/* ------------------------------------------------------------------------ */
/* Direct attention (no tiling)                                              */
/* ------------------------------------------------------------------------ */

static double dot(const double* a, const double* b, int d)
{
    double s = 0.0;
    for (int k = 0; k < d; ++k)
        s += a[k] * b[k];
    return s;
}

/* Forward of one query row: the visible keys are [s, i] when causal, else
 * [s, e).  Writes O_i (d values) and returns LSE_i = m + ln l.  Uses the
 * direct softmax, S_ij = alpha Q_i . K_j, P_ij = exp(S_ij - m) / l. */
static double fwd_row(const double* Q, const double* K, const double* V, int Hq, int Hkv, int d,
                      int64_t s, int64_t e, int causal, double alpha, int64_t i, int h, double* o,
                      double* Srow)
{
    int hk = h / (Hq / Hkv);
    int64_t jend = causal ? i + 1 : e;
    const double* q = Q + (i * Hq + h) * d;
    double m = -INFINITY;
    for (int64_t j = s; j < jend; ++j) {
        Srow[j - s] = alpha * dot(q, K + (j * Hkv + hk) * d, d);
        if (Srow[j - s] > m)
            m = Srow[j - s];
    }
    double l = 0.0;
    for (int k = 0; k < d; ++k)
        o[k] = 0.0;
    for (int64_t j = s; j < jend; ++j) {
        double p = exp(Srow[j - s] - m);
        l += p;
        const double* v = V + (j * Hkv + hk) * d;
        for (int k = 0; k < d; ++k)
            o[k] += p * v[k];
    }
    for (int k = 0; k < d; ++k)
        o[k] /= l;
    return m + log(l);
}

static int doc_of(const int32_t* cu, int ndocs, int64_t t)
{
    if (!cu)
        return 0;
    int b = 0;
    while (b + 1 < ndocs && cu[b + 1] <= t)
        ++b;
    return b;
}

/* Attention forward over dequantized operands.
 * Q [T, Hq, d] (score view), K [T, Hkv, d] (score view), V [T, Hkv, d]
 * (the view the P V product uses); O [T, Hq, d]; LSE [Hq, T].
 * sel == NULL: every query row; else nsel (token, head) pairs.  Rows not
 * computed are left untouched. */
void orc_attn_fwd(const double* Q, const double* K, const double* V, int64_t T, int Hq, int Hkv, int d,
                  const int32_t* cu, int ndocs, int causal, double alpha, const int32_t* sel, int64_t nsel,
                  double* O, double* LSE)
{
    int64_t n = sel ? nsel : T * Hq;
    int64_t maxlen = 0;
    for (int b = 0; b < num_docs_eff(cu, ndocs); ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        if (e - s > maxlen)
            maxlen = e - s;
    }
#pragma omp parallel
    {
        double* Srow = (double*)malloc(sizeof(double) * (size_t)(maxlen + 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n; ++r) {
            int64_t i = sel ? sel[2 * r] : r / Hq;
            int h = sel ? sel[2 * r + 1] : (int)(r % Hq);
            int b = doc_of(cu, ndocs, i);
            int64_t s, e;
            doc_range(cu, ndocs, T, b, &s, &e);
            LSE[(int64_t)h * T + i] = fwd_row(Q, K, V, Hq, Hkv, d, s, e, causal, alpha, i, h, O + (i * Hq + h) * d, Srow);
        }
        free(Srow);
    }
}

/* Causal attention forward with the per-key fold on the diagonal tile
 * ([FLAMIA] sec. 4): P_ij (s_j v_j) = (P_ij s_j) v_j, so the value row of key
 * j is its per-key view Vkey_j (decoded: s_j times its codes) when j lies in
 * the same 128-token tile of the document as query i -- the tile whose
 * 32-token scale groups would straddle i -- and its token view Vtok_j for
 * the fully visible tiles before it.  The softmax is the direct one of
 * orc_attn_fwd.  Q, K [T, H*, d] score views; Vtok, Vkey [T, Hkv, d] decoded;
 * O [T, Hq, d]; LSE [Hq, T]. */
void orc_attn_fwd_fold(const double* Q, const double* K, const double* Vtok, const double* Vkey, int64_t T,
                       int Hq, int Hkv, int d, const int32_t* cu, int ndocs, double alpha, double* O, double* LSE)
{
    int nd = num_docs_eff(cu, ndocs);
    int grp = Hq / Hkv;
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t n = e - s;
        if (n <= 0)
            continue;
#pragma omp parallel
        {
            double* Srow = (double*)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 8) collapse(2)
            for (int h = 0; h < Hq; ++h)
                for (int64_t i = s; i < e; ++i) {
                    int hk = h / grp;
                    const double* q = Q + (i * Hq + h) * d;
                    double m = -INFINITY;
                    for (int64_t j = s; j <= i; ++j) {
                        Srow[j - s] = alpha * dot(q, K + (j * Hkv + hk) * d, d);
                        if (Srow[j - s] > m)
                            m = Srow[j - s];
                    }
                    double* o = O + (i * Hq + h) * d;
                    for (int k = 0; k < d; ++k)
                        o[k] = 0.0;
                    double l = 0.0;
                    int64_t diag0 = s + ((i - s) / 128) * 128; /* first key of i's tile */
                    for (int64_t j = s; j <= i; ++j) {
                        double p = exp(Srow[j - s] - m);
                        l += p;
                        const double* v = (j >= diag0 ? Vkey : Vtok) + (j * Hkv + hk) * d;
                        for (int k = 0; k < d; ++k)
                            o[k] += p * v[k];
                    }
                    for (int k = 0; k < d; ++k)
                        o[k] /= l;
                    LSE[(int64_t)h * T + i] = m + log(l);
                }
            free(Srow);
        }
    }
}

/* Attention backward over dequantized operands, direct (no tiling).
 * Inputs (all [T, H*, d] fp64):
 *   Qs, Ks : score views (rebuild S, exactly as the forward);
 *   Vo     : the V view the forward's P V used (rebuilds O);
 *   Vr, Gr : views for E = G V^T and D = G . O (the same G in both);
 *   Qt, Kt, Gt : views for dK = alpha U^T Q, dQ = alpha U K, dV = P^T G.
 * Outputs dQ [T, Hq, d], dK [T, Hkv, d], dV [T, Hkv, d]; also O [T, Hq, d],
 * LSE [Hq, T] and D [Hq, T] of the computed rows.
 * units == NULL: all (document, kv-head) units; else nunits (doc, kv-head)
 * pairs.  dK/dV of a kv-head sum over the Hq/Hkv query heads of its group.
 * Pass 1 (per query row) builds LSE, O, D and dQ; pass 2 (per key row)
 * rebuilds P and U from LSE and D and sums dK and dV. */
void orc_attn_bwd(const double* Qs, const double* Ks, const double* Vo, const double* Vr, const double* Gr,
                  const double* Qt, const double* Kt, const double* Gt, int64_t T, int Hq, int Hkv, int d,
                  const int32_t* cu, int ndocs, int causal, double alpha, const int32_t* units, int nunits,
                  double* dQ, double* dK, double* dV, double* O, double* LSE, double* D)
{
    int nd = num_docs_eff(cu, ndocs);
    int nu = units ? nunits : nd * Hkv;
    int grp = Hq / Hkv;
    for (int u = 0; u < nu; ++u) {
        int b = units ? units[2 * u] : u / Hkv;
        int hk = units ? units[2 * u + 1] : u % Hkv;
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t n = e - s;
        if (n <= 0)
            continue;
        /* pass 1: rows */
#pragma omp parallel
        {
            double* Srow = (double*)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 8) collapse(2)
            for (int hh = 0; hh < grp; ++hh)
                for (int64_t i = s; i < e; ++i) {
                    int h = hk * grp + hh;
                    double* o = O + (i * Hq + h) * d;
                    double lse = fwd_row(Qs, Ks, Vo, Hq, Hkv, d, s, e, causal, alpha, i, h, o, Srow);
                    LSE[(int64_t)h * T + i] = lse;
                    const double* g = Gr + (i * Hq + h) * d;
                    double Di = dot(g, o, d);
                    D[(int64_t)h * T + i] = Di;
                    double* dq = dQ + (i * Hq + h) * d;
                    for (int k = 0; k < d; ++k)
                        dq[k] = 0.0;
                    int64_t jend = causal ? i + 1 : e;
                    for (int64_t j = s; j < jend; ++j) {
                        double P = exp(Srow[j - s] - lse);
                        double E = dot(g, Vr + (j * Hkv + hk) * d, d);
                        double U = P * (E - Di);
                        const double* kt = Kt + (j * Hkv + hk) * d;
                        for (int k = 0; k < d; ++k)
                            dq[k] += alpha * U * kt[k];
                    }
                }
            free(Srow);
        }
        /* pass 2: key columns */
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t j = s; j < e; ++j) {
            double* dk = dK + (j * Hkv + hk) * d;
            double* dv = dV + (j * Hkv + hk) * d;
            for (int k = 0; k < d; ++k) {
                dk[k] = 0.0;
                dv[k] = 0.0;
            }
            const double* kj = Ks + (j * Hkv + hk) * d;
            const double* vj = Vr + (j * Hkv + hk) * d;
            for (int hh = 0; hh < grp; ++hh) {
                int h = hk * grp + hh;
                int64_t ibeg = causal ? j : s;
                for (int64_t i = ibeg; i < e; ++i) {
                    double S = alpha * dot(Qs + (i * Hq + h) * d, kj, d);
                    double P = exp(S - LSE[(int64_t)h * T + i]);
                    const double* g = Gr + (i * Hq + h) * d;
                    double E = dot(g, vj, d);
                    double U = P * (E - D[(int64_t)h * T + i]);
                    const double* gt = Gt + (i * Hq + h) * d;
                    const double* qt = Qt + (i * Hq + h) * d;
                    for (int k = 0; k < d; ++k) {
                        dv[k] += P * gt[k];
                        dk[k] += alpha * U * qt[k];
                    }
                }
            }
        }
    }
}

/* Causal backward with the per-key fold on the diagonal tile ([FLAMIA] sec. 4:
 * the K factor of dQ moves into dS, the "K fold", as the V factor of the
 * forward moves into P).  The same direct backward as orc_attn_bwd, except
 * that on query i's own 128-token tile of its document (keys
 * [s + 128 floor((i - s) / 128), i]) O_i takes each key's per-key value row
 * Vkey_j (the folded forward) and dQ_i takes each key's per-key row Kkey_j;
 * the tiles before it use Vo and Kt.  D = G . O uses that O.  Inputs as
 * orc_attn_bwd plus Vkey, Kkey [T, Hkv, d] (decoded per-key views); every
 * (document, kv head) unit. */
void orc_attn_bwd_fold(const double* Qs, const double* Ks, const double* Vo, const double* Vr, const double* Gr,
                       const double* Qt, const double* Kt, const double* Gt, const double* Vkey, const double* Kkey,
                       int64_t T, int Hq, int Hkv, int d, const int32_t* cu, int ndocs, double alpha, double* dQ,
                       double* dK, double* dV, double* O, double* LSE, double* D)
{
    int nd = num_docs_eff(cu, ndocs);
    int grp = Hq / Hkv;
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        int64_t n = e - s;
        if (n <= 0)
            continue;
        for (int hk = 0; hk < Hkv; ++hk) {
            /* pass 1: rows */
#pragma omp parallel
            {
                double* Srow = (double*)malloc(sizeof(double) * (size_t)n);
#pragma omp for schedule(dynamic, 8) collapse(2)
                for (int hh = 0; hh < grp; ++hh)
                    for (int64_t i = s; i < e; ++i) {
                        int h = hk * grp + hh;
                        int64_t diag0 = s + ((i - s) / 128) * 128;
                        const double* q = Qs + (i * Hq + h) * d;
                        double m = -INFINITY;
                        for (int64_t j = s; j <= i; ++j) {
                            Srow[j - s] = alpha * dot(q, Ks + (j * Hkv + hk) * d, d);
                            if (Srow[j - s] > m)
                                m = Srow[j - s];
                        }
                        double* o = O + (i * Hq + h) * d;
                        for (int k = 0; k < d; ++k)
                            o[k] = 0.0;
                        double l = 0.0;
                        for (int64_t j = s; j <= i; ++j) {
                            double p = exp(Srow[j - s] - m);
                            l += p;
                            const double* v = (j >= diag0 ? Vkey : Vo) + (j * Hkv + hk) * d;
                            for (int k = 0; k < d; ++k)
                                o[k] += p * v[k];
                        }
                        for (int k = 0; k < d; ++k)
                            o[k] /= l;
                        double lse = m + log(l);
                        LSE[(int64_t)h * T + i] = lse;
                        const double* g = Gr + (i * Hq + h) * d;
                        double Di = dot(g, o, d);
                        D[(int64_t)h * T + i] = Di;
                        double* dq = dQ + (i * Hq + h) * d;
                        for (int k = 0; k < d; ++k)
                            dq[k] = 0.0;
                        for (int64_t j = s; j <= i; ++j) {
                            double P = exp(Srow[j - s] - lse);
                            double E = dot(g, Vr + (j * Hkv + hk) * d, d);
                            double U = P * (E - Di);
                            const double* kt = (j >= diag0 ? Kkey : Kt) + (j * Hkv + hk) * d;
                            for (int k = 0; k < d; ++k)
                                dq[k] += alpha * U * kt[k];
                        }
                    }
                free(Srow);
            }
            /* pass 2: key columns, as orc_attn_bwd */
#pragma omp parallel for schedule(dynamic, 8)
            for (int64_t j = s; j < e; ++j) {
                double* dk = dK + (j * Hkv + hk) * d;
                double* dv = dV + (j * Hkv + hk) * d;
                for (int k = 0; k < d; ++k) {
                    dk[k] = 0.0;
                    dv[k] = 0.0;
                }
                const double* kj = Ks + (j * Hkv + hk) * d;
                const double* vj = Vr + (j * Hkv + hk) * d;
                for (int hh = 0; hh < grp; ++hh) {
                    int h = hk * grp + hh;
                    for (int64_t i = j; i < e; ++i) {
                        double S = alpha * dot(Qs + (i * Hq + h) * d, kj, d);
                        double P = exp(S - LSE[(int64_t)h * T + i]);
                        const double* g = Gr + (i * Hq + h) * d;
                        double E = dot(g, vj, d);
                        double U = P * (E - D[(int64_t)h * T + i]);
                        const double* gt = Gt + (i * Hq + h) * d;
                        const double* qt = Qt + (i * Hq + h) * d;
                        for (int k = 0; k < d; ++k) {
                            dv[k] += P * gt[k];
                            dk[k] += alpha * U * qt[k];
                        }
                    }
                }
            }
        }
    }
}

/* Cross-attention (query and key/value documents of different lengths, no
 * mask): the queries of document b, rows [cu_q[b], cu_q[b+1]) of Q, attend
 * to that document's keys and values, rows [cu_k[b], cu_k[b+1]) of K and V.
 * The arithmetic is the direct softmax of orc_attn_fwd with the key range
 * taken from the key side.  Q [Tq, Hq, d]; K, V [Tk, Hkv, d]; O [Tq, Hq, d];
 * LSE [Hq, Tq].  Both offset arrays are required. */
void orc_attn_fwd_x(const double* Q, const double* K, const double* V, int64_t Tq, int64_t Tk, int Hq, int Hkv,
                    int d, const int32_t* cu_q, const int32_t* cu_k, int ndocs, double alpha, double* O,
                    double* LSE)
{
    int64_t maxk = 0;
    for (int b = 0; b < ndocs; ++b)
        if (cu_k[b + 1] - cu_k[b] > maxk)
            maxk = cu_k[b + 1] - cu_k[b];
    (void)Tk;
#pragma omp parallel
    {
        double* Srow = (double*)malloc(sizeof(double) * (size_t)(maxk + 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < Tq * Hq; ++r) {
            int64_t i = r / Hq;
            int h = (int)(r % Hq);
            int b = 0;
            while (b + 1 < ndocs && cu_q[b + 1] <= i)
                ++b;
            LSE[(int64_t)h * Tq + i] =
                fwd_row(Q, K, V, Hq, Hkv, d, cu_k[b], cu_k[b + 1], 0, alpha, i, h, O + (i * Hq + h) * d, Srow);
        }
        free(Srow);
    }
}

/* Cross-attention backward, direct: orc_attn_bwd's two passes with the query
 * rows of document b from the query side and its key rows from the key side
 * (no mask).  Views as in orc_attn_bwd; Ks, Vo, Vr, Kt have Tk rows, the rest
 * Tq.  dQ [Tq, Hq, d]; dK, dV [Tk, Hkv, d]; O [Tq, Hq, d]; LSE, D [Hq, Tq]. */
void orc_attn_bwd_x(const double* Qs, const double* Ks, const double* Vo, const double* Vr, const double* Gr,
                    const double* Qt, const double* Kt, const double* Gt, int64_t Tq, int64_t Tk, int Hq, int Hkv,
                    int d, const int32_t* cu_q, const int32_t* cu_k, int ndocs, double alpha, double* dQ, double* dK,
                    double* dV, double* O, double* LSE, double* D)
{
    int grp = Hq / Hkv;
    (void)Tk;
    for (int b = 0; b < ndocs; ++b) {
        int64_t sq = cu_q[b], eq = cu_q[b + 1], sk = cu_k[b], ek = cu_k[b + 1];
        for (int hk = 0; hk < Hkv; ++hk) {
            /* pass 1: query rows */
#pragma omp parallel
            {
                double* Srow = (double*)malloc(sizeof(double) * (size_t)(ek - sk + 1));
#pragma omp for schedule(dynamic, 8) collapse(2)
                for (int hh = 0; hh < grp; ++hh)
                    for (int64_t i = sq; i < eq; ++i) {
                        int h = hk * grp + hh;
                        double* o = O + (i * Hq + h) * d;
                        double lse = fwd_row(Qs, Ks, Vo, Hq, Hkv, d, sk, ek, 0, alpha, i, h, o, Srow);
                        LSE[(int64_t)h * Tq + i] = lse;
                        const double* g = Gr + (i * Hq + h) * d;
                        double Di = dot(g, o, d);
                        D[(int64_t)h * Tq + i] = Di;
                        double* dq = dQ + (i * Hq + h) * d;
                        for (int k = 0; k < d; ++k)
                            dq[k] = 0.0;
                        for (int64_t j = sk; j < ek; ++j) {
                            double P = exp(Srow[j - sk] - lse);
                            double E = dot(g, Vr + (j * Hkv + hk) * d, d);
                            double U = P * (E - Di);
                            const double* kt = Kt + (j * Hkv + hk) * d;
                            for (int k = 0; k < d; ++k)
                                dq[k] += alpha * U * kt[k];
                        }
                    }
                free(Srow);
            }
            /* pass 2: key rows */
#pragma omp parallel for schedule(dynamic, 8)
            for (int64_t j = sk; j < ek; ++j) {
                double* dk = dK + (j * Hkv + hk) * d;
                double* dv = dV + (j * Hkv + hk) * d;
                for (int k = 0; k < d; ++k) {
                    dk[k] = 0.0;
                    dv[k] = 0.0;
                }
                const double* kj = Ks + (j * Hkv + hk) * d;
                const double* vj = Vr + (j * Hkv + hk) * d;
                for (int hh = 0; hh < grp; ++hh) {
                    int h = hk * grp + hh;
                    for (int64_t i = sq; i < eq; ++i) {
                        double S = alpha * dot(Qs + (i * Hq + h) * d, kj, d);
                        double P = exp(S - LSE[(int64_t)h * Tq + i]);
                        const double* g = Gr + (i * Hq + h) * d;
                        double E = dot(g, vj, d);
                        double U = P * (E - D[(int64_t)h * Tq + i]);
                        const double* gt = Gt + (i * Hq + h) * d;
                        const double* qt = Qt + (i * Hq + h) * d;
                        for (int k = 0; k < d; ++k) {
                            dv[k] += P * gt[k];
                            dk[k] += alpha * U * qt[k];
                        }
                    }
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FP16 dQ reduction with a per-row boost                                    */
/* ------------------------------------------------------------------------ */

/* ceil(log2 x) of a positive finite value, exactly: x = f 2^e, f in [0.5, 1). */
static int cl2d(double x)
{
    int e;
    double f = frexp(x, &e);
    return f == 0.5 ? e - 1 : e;
}

#define ORC_CL2_NONE (-2000) /* cl2 of an all-zero vector */

/* cl2(max_c |x_c|) of one d-vector, or ORC_CL2_NONE. */
static int cl2_maxabs(const double* x, int d)
{
    double m = 0.0;
    for (int c = 0; c < d; ++c)
        if (fabs(x[c]) > m)
            m = fabs(x[c]);
    return m > 0.0 ? cl2d(m) : ORC_CL2_NONE;
}

/* The power-of-two boost 2^beta of every query row of the FP16 dQ reduction
 * in its strict form ([FLAMIA] sec. 4, "最后一条通道在累加器里": dQ partial
 * sums boosted by a power of two, the strict option taking each row's own G
 * norm with the maxima of V and K over the visible keys only).  The pages
 * give the shape of the choice, b_i = 2^floor(log2(h / a_i)) for a bound a_i
 * of the row's magnitude and a target h.  READING, not a page value: this
 * restates the bound the library documents for its MXA_DQ_FP16_ROW mode, so
 * comparing the library's exponents with these compares it with its own
 * stated specification; the pins only check that the bound holds:
 *   a_i = 2^(4 + cl2(alpha) + log2(d) + s(n_i) + g_i + V_i + K_i), h = 2^15,
 *   g_i = cl2(max_c |G_ic|), V_i = max_{j visible} cl2(max_c |V_jc|),
 *   K_i = max_{j visible} cl2(max_c |K_jc|), n_i = visible keys,
 *   s(n) = 1 + max(0, cl2(n) - 14), cl2(1) = 0,
 *   beta_i = clamp(15 - log2(a_i), -100, 100).
 * Gr [T, Hq, d], Vr and Kr [T, Hkv, d]: the decoded ROW views (fp64).
 * alpha: the fp32 softmax scale.  beta: [Hq, T]. */
void orc_dq_row_boost(const double* Gr, const double* Vr, const double* Kr, int64_t T, int Hq, int Hkv, int d,
                      const int32_t* cu, int ndocs, int causal, float alpha, int32_t* beta)
{
    int nd = num_docs_eff(cu, ndocs);
    int grp = Hq / Hkv;
    int log2d = 0;
    while ((1 << log2d) < d)
        ++log2d;
    int ca = cl2d((double)alpha);
    for (int b = 0; b < nd; ++b) {
        int64_t s, e;
        doc_range(cu, ndocs, T, b, &s, &e);
        if (e <= s)
            continue;
        int* ve = (int*)malloc(sizeof(int) * (size_t)(e - s));
        int* ke = (int*)malloc(sizeof(int) * (size_t)(e - s));
        for (int hk = 0; hk < Hkv; ++hk) {
            for (int64_t j = s; j < e; ++j) {
                ve[j - s] = cl2_maxabs(Vr + (j * Hkv + hk) * d, d);
                ke[j - s] = cl2_maxabs(Kr + (j * Hkv + hk) * d, d);
            }
            for (int h = hk * grp; h < (hk + 1) * grp; ++h) {
                for (int64_t i = s; i < e; ++i) {
                    int64_t jend = causal ? i + 1 : e;
                    int Vi = ORC_CL2_NONE, Ki = ORC_CL2_NONE;
                    for (int64_t j = s; j < jend; ++j) {
                        if (ve[j - s] > Vi)
                            Vi = ve[j - s];
                        if (ke[j - s] > Ki)
                            Ki = ke[j - s];
                    }
                    int64_t n = jend - s;
                    int ln = n <= 1 ? 0 : cl2d((double)n);
                    int sp = 1 + (ln > 14 ? ln - 14 : 0);
                    int g = cl2_maxabs(Gr + (i * Hq + h) * d, d);
                    int bt = 15 - (4 + ca + log2d + sp + g + Vi + Ki);
                    beta[(int64_t)h * T + i] = bt < -100 ? -100 : (bt > 100 ? 100 : bt);
                }
            }
        }
        free(ve);
        free(ke);
    }
}

/* ------------------------------------------------------------------------ */
/* Algorithm 1: the low-precision forward and the matching backward recompute */
/* ------------------------------------------------------------------------ */

/* [FLAMIA] sec. 5, Algorithm 1 ("低精度前向与一致的反向重算"), with the
 * roundings its steps name.  Each can be switched off, so that the result
 * falls back to the direct fp64 attention above:
 *   ORC_RND_P  - step 07: the forward's weights are quantized, E4M3(2^c p)
 *                with c = 4 and the constant scale 2^-4 ("概率上限由两个参数
 *                共同决定": (c, tau) = (4, 4)); O is normalised by the sum of
 *                the quantized weights;
 *   ORC_RND_O  - step 08: O is saved in bf16 (the D of step 09 reads it);
 *   ORC_RND_P8 - step 15: dV's probability operand is E4M3(2^8 P) 2^-8
 *                (the 2^8 boost of the backward, same passage);
 *   ORC_RND_DS - step 14: U = P (E - D) is quantized per 32 x 32 block of
 *                the tile by the MX rule ([FA4] "Квантование dS без
 *                транспонирования": one exponent per 32 x 32 block, both axes
 *                counted from the document start, before alpha);
 *   ORC_RND_LSE - step 08: the row LSE is saved in fp32 and step 12 rebuilds
 *                P from that saved value.  At a row whose scores span
 *                thousands of nats one fp32 ulp of the LSE is 1e-4, which
 *                moves every P of the row by that factor; lse_ulps moves the
 *                saved value by that many fp32 ulps, spanning the results an
 *                fp32 LSE admits.
 * Step 07's reference maximum follows the online statistics of steps 04-06
 * ("概率上限由两个参数共同决定": the reference may stay up to tau = 4 behind the
 * true maximum, in base-2 coordinates x = S log2(e)).  The keys of a row are
 * walked in key tiles of ref_tile keys counted from the key document's start;
 * with t_max the largest x of a tile's visible keys, the reference is
 *   m = ceil(t_max) at the first tile, and m = ceil(t_max) again at any later
 *   tile whose t_max exceeds m + 4 (else m stays);
 * and every key of a tile takes the weight p = 2^(x - m) against the m in
 * force after its tile's update.  Readings (the pages leave these open): the
 * reference lies on the integer grid, so a raise rescales the earlier sums by
 * an exact power of two and the E4M3 weights of the normal range equal those
 * of any other integer reference ([FLAMIA] sec. 4, scale doubling) -- only
 * weights below 2^-10 of the reference (E4M3 subnormals after the 2^4 boost)
 * depend on the schedule; the integer decision is taken in IEEE fp32 from
 * the fp32-rounded raw score q.k times the fp32 product alpha * log2(e), as a
 * kernel holding fp32 scores takes it; ref_tile = 0 means one tile holding
 * every visible key (m = ceil(max x) of the row).
 * The E4M3 code of each forward weight is likewise decided in fp32, the
 * precision in which an fp32 score holds it: the boosted weight is
 * 2^(x32) with x32 = fma32(fl32(q.k), fl32(alpha log2 e), 4 - m), its exact
 * power of two rounded to fp32, then to E4M3 (at scores of 10^4 an fp32
 * score fixes a weight only to about 4e-5, so a weight near a tie between
 * two codes is decided by that rounding). */
#define ORC_RND_P 1
#define ORC_RND_O 2
#define ORC_RND_P8 4
#define ORC_RND_DS 8
#define ORC_RND_LSE 16 /* step 08: LSE saved in fp32; the backward rebuilds P from it */

#define ORC_LOG2E 1.4426950408889634074

/* Nearest E4M3 value to y as fp64 (ties to the even code, saturating to 448,
 * sign kept): the value orc_e4m3_decode(orc_e4m3_encode(y)) by a binary search
 * over the ascending finite codes 0x00..0x7E instead of a scan. */
double orc_e4m3_round(double y)
{
    if (isnan(y))
        return y;
    double a = fabs(y);
    if (a >= 448.0)
        return copysign(448.0, y);
    int lo = 0, hi = 0x7E; /* invariant: decode(lo) <= a < decode(hi + 1) */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (orc_e4m3_decode((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    double v0 = orc_e4m3_decode((uint8_t)lo), v1 = orc_e4m3_decode((uint8_t)(lo + 1));
    double r;
    if (a - v0 < v1 - a)
        r = v0;
    else if (a - v0 > v1 - a)
        r = v1;
    else
        r = (lo & 1) ? v1 : v0;
    return copysign(r, y);
}

void orc_e4m3_round_array(const double* y, int64_t n, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_round(y[i]);
}

/* Nearest bf16 value of x (8 significant bits, ties to even), as fp64. */
double orc_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    frexp(x, &e); /* |x| = f 2^e, f in [0.5, 1) */
    if (e < -125)
        e = -125; /* bf16 subnormals: fixed spacing 2^-133 */
    return ldexp(rint(ldexp(x, 8 - e)), e - 8);
}

void orc_round_bf16_array(const double* x, int64_t n, double* out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_round_bf16(x[i]);
}

/* MX rule on a group of values: y -> E4M3(y / 2^e) 2^e with e the group's
 * scale exponent (orc_mx_exponent of its largest magnitude). */
static void mx_round_group(double* y, int64_t n, int64_t stride)
{
    double amax = 0.0;
    for (int64_t k = 0; k < n; ++k)
        if (fabs(y[k * stride]) > amax)
            amax = fabs(y[k * stride]);
    int e = orc_mx_exponent(amax);
    for (int64_t k = 0; k < n; ++k)
        y[k * stride] = ldexp(orc_e4m3_round(ldexp(y[k * stride], -e)), e);
}

/* Steps 05-08 for one query row over the visible keys [ks, kend) of kv head
 * hk (ks = the key document's first token).  Writes O_i (d values) and
 * returns LSE_i = m + ln sum_j exp(S_j - m) (the unquantized sum).
 *   S_j = alpha q . K_j;  p_j = 2^(S_j log2 e - mu_j) with mu_j the reference
 *   in force at key j's tile (the schedule above, ref_tile keys per tile);
 *   keys j < diag0: weight w_j = E4M3(2^4 p_j) 2^-4 (ORC_RND_P) or p_j, and
 *     value row V_j;
 *   keys j >= diag0 (the per-key fold of [FLAMIA] sec. 4 on the query's own
 *     128-token tile; Vkey_j = codes_j 2^e_j with e_j = vkey_sf_j - 127):
 *     y_j = 2^4 p_j 2^e_j, quantized per 32 keys (counted from ks) by the MX
 *     rule (ORC_RND_P), multiplies the codes: weight y_j 2^-4 2^-e_j on the
 *     value row Vkey_j;
 *   O_i = sum_j w_j row_j / sum_j w_j, rounded to bf16 (ORC_RND_O).
 * diag0 >= kend: no fold.  Srow, y, mu, raw: scratch of kend - ks values. */
static double fwd_row_alg1(const double* q, const double* K, const double* V, const double* Vkey,
                           const uint8_t* vkey_sf, int Hkv, int hk, int d, int64_t ks, int64_t kend, int64_t diag0,
                           double alpha, int rnd, int64_t ref_tile, double* o, double* Srow, double* y, double* mu,
                           double* raw)
{
    double m = -INFINITY;
    for (int64_t j = ks; j < kend; ++j) {
        raw[j - ks] = dot(q, K + (j * Hkv + hk) * d, d); /* the score q . k before alpha */
        Srow[j - ks] = alpha * raw[j - ks];
        if (Srow[j - ks] > m)
            m = Srow[j - ks];
    }
    double l = 0.0;
    for (int64_t j = ks; j < kend; ++j)
        l += exp(Srow[j - ks] - m);
    double lse = m + log(l);
    /* the reference in force at each key's tile */
    const float sl2 = (float)alpha * 1.4426950408889634f;
    {
        int64_t tile = ref_tile > 0 ? ref_tile : (kend - ks > 0 ? kend - ks : 1);
        float mref = -INFINITY;
        for (int64_t t0 = ks; t0 < kend; t0 += tile) {
            int64_t t1 = t0 + tile < kend ? t0 + tile : kend;
            float tmax = -INFINITY;
            for (int64_t j = t0; j < t1; ++j)
                if ((float)raw[j - ks] > tmax)
                    tmax = (float)raw[j - ks];
            float ts = tmax * sl2;
            if (t0 == ks || ts > mref + 4.0f)
                mref = ceilf(ts);
            for (int64_t j = t0; j < t1; ++j)
                mu[j - ks] = (double)mref;
        }
    }
    /* each weight joins the sums in the frame of the last reference: the
     * sums are rescaled by 2^(m_old - m_new) whenever the reference rises */
    const double mlast = kend > ks ? mu[kend - 1 - ks] : 0.0;
    for (int k = 0; k < d; ++k)
        o[k] = 0.0;
    double W = 0.0;
    int64_t f0 = diag0 < kend ? diag0 : kend;
    for (int64_t j = ks; j < f0; ++j) {
        double w;
        if (rnd & ORC_RND_P) {
            float x32 = fmaf((float)raw[j - ks], sl2, 4.0f - (float)mu[j - ks]);
            w = orc_e4m3_round((double)(float)exp2((double)x32)) / 16.0;
        } else {
            w = exp2(Srow[j - ks] * ORC_LOG2E - mu[j - ks]);
        }
        w = ldexp(w, (int)(mu[j - ks] - mlast));
        const double* v = V + (j * Hkv + hk) * d;
        for (int k = 0; k < d; ++k)
            o[k] += w * v[k];
        W += w;
    }
    if (f0 < kend) {
        for (int64_t j = f0; j < kend; ++j) {
            int ej = (int)vkey_sf[j * Hkv + hk] - 127;
            double p16;
            if (rnd & ORC_RND_P) {
                float x32 = fmaf((float)raw[j - ks], sl2, 4.0f - (float)mu[j - ks]);
                p16 = (double)(float)exp2((double)x32);
            } else {
                p16 = 16.0 * exp2(Srow[j - ks] * ORC_LOG2E - mu[j - ks]);
            }
            y[j - ks] = ldexp(p16, ej + (int)(mu[j - ks] - mlast));
        }
        if (rnd & ORC_RND_P)
            for (int64_t g0 = f0; g0 < kend; g0 += 32) /* f0 - ks is a multiple of 128 */
                mx_round_group(y + (g0 - ks), (kend - g0 < 32 ? kend - g0 : 32), 1);
        for (int64_t j = f0; j < kend; ++j) {
            int ej = (int)vkey_sf[j * Hkv + hk] - 127;
            double wc = y[j - ks] / 16.0; /* the weight on the codes */
            const double* v = Vkey + (j * Hkv + hk) * d;
            for (int k = 0; k < d; ++k)
                o[k] += wc * ldexp(v[k], -ej);
            W += ldexp(wc, -ej);
        }
    }
    for (int k = 0; k < d; ++k) {
        o[k] /= W;
        if (rnd & ORC_RND_O)
            o[k] = orc_round_bf16(o[k]);
    }
    return lse;
}

/* The LSE as step 08 saves it: rounded to fp32, then moved by k fp32 ulps. */
static double saved_lse(double lse, int k)
{
    float f = (float)lse;
    for (; k > 0; --k)
        f = nextafterf(f, INFINITY);
    for (; k < 0; ++k)
        f = nextafterf(f, -INFINITY);
    return (double)f;
}

/* Key side of document b: [*ks, *ke) on the key rows (cu_k == NULL: the
 * query side's documents). */
static void key_range(const int32_t* cu_q, const int32_t* cu_k, int ndocs, int64_t Tq, int64_t Tk, int b,
                      int64_t* ks, int64_t* ke)
{
    if (cu_k)
        doc_range(cu_k, ndocs, Tk, b, ks, ke);
    else
        doc_range(cu_q, ndocs, Tq, b, ks, ke);
}

/* Algorithm 1's forward (steps 04-08) in fp64, direct: every query row i of
 * document b attends to the keys [ks, ks + (i - s) + 1) when causal, else to
 * all keys of the document's key side.  Q [Tq, Hq, d] and K [Tk, Hkv, d]
 * score views; V [Tk, Hkv, d] the view of the P V product; Vkey, vkey_sf
 * (decoded per-key view of V and its UE8M0 bytes [Tk, Hkv], causal
 * self-attention only) or NULL: the per-key fold on each query's own
 * 128-token tile.  cu_q == NULL: one document of Tq tokens; cu_k == NULL: the
 * key documents are the query documents (self-attention).  rnd: ORC_RND_P |
 * ORC_RND_O for Algorithm 1, 0 for the direct softmax.  ref_tile: the key
 * tile of the reference schedule (0: one tile).  sel == NULL: every row, else
 * nsel (token, head) pairs.  O [Tq, Hq, d]; LSE [Hq, Tq]. */
void orc_attn_fwd_alg1(const double* Q, const double* K, const double* V, const double* Vkey,
                       const uint8_t* vkey_sf, int64_t Tq, int64_t Tk, int Hq, int Hkv, int d, const int32_t* cu_q,
                       const int32_t* cu_k, int ndocs, int causal, double alpha, int rnd, int64_t ref_tile,
                       const int32_t* sel, int64_t nsel, double* O, double* LSE)
{
    int nd = num_docs_eff(cu_q, ndocs);
    int grp = Hq / Hkv;
    int64_t maxk = 0;
    for (int b = 0; b < nd; ++b) {
        int64_t ks, ke;
        key_range(cu_q, cu_k, ndocs, Tq, Tk, b, &ks, &ke);
        if (ke - ks > maxk)
            maxk = ke - ks;
    }
    int64_t n = sel ? nsel : Tq * Hq;
#pragma omp parallel
    {
        double* Srow = (double*)malloc(sizeof(double) * (size_t)(maxk + 1));
        double* y = (double*)malloc(sizeof(double) * (size_t)(maxk + 1));
        double* mu = (double*)malloc(sizeof(double) * (size_t)(maxk + 1));
        double* raw = (double*)malloc(sizeof(double) * (size_t)(maxk + 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < n; ++r) {
            int64_t i = sel ? sel[2 * r] : r / Hq;
            int h = sel ? sel[2 * r + 1] : (int)(r % Hq);
            int b = doc_of(cu_q, ndocs, i);
            int64_t s, e, ks, ke;
            doc_range(cu_q, ndocs, Tq, b, &s, &e);
            key_range(cu_q, cu_k, ndocs, Tq, Tk, b, &ks, &ke);
            int64_t kend = causal ? ks + (i - s) + 1 : ke;
            int64_t diag0 = Vkey ? ks + ((i - s) / 128) * 128 : kend;
            LSE[(int64_t)h * Tq + i] = fwd_row_alg1(Q + (i * Hq + h) * d, K, V, Vkey, vkey_sf, Hkv, h / grp, d, ks,
                                                    kend, diag0, alpha, rnd, ref_tile, O + (i * Hq + h) * d, Srow, y,
                                                    mu, raw);
        }
        free(Srow);
        free(y);
        free(mu);
        free(raw);
    }
}

/* Algorithm 1's backward (steps 09-16 without the FP16 accumulator, which
 * the tolerance covers) in fp64, direct, per (document, kv head) unit:
 *   O_i, LSE_i from the forward above (the same views and roundings);
 *   D_i = Gr_i . O_i                                        (step 09)
 *   P_ij = exp(S_ij - LSE_i); E_ij = Gr_i . Vr_j              (steps 11-13)
 *   U_ij = P_ij (E_ij - D_i); U~ = U quantized per 32 x 32 block, queries and
 *     keys counted from their document starts (ORC_RND_DS)     (step 14)
 *   dV_j = sum_i E4M3(2^8 P_ij) 2^-8 Gt_i (ORC_RND_P8), dK_j = alpha sum_i
 *     U~_ij Qt_i, dQ_i = alpha sum_j U~_ij Kt_j, dK and dV summed over the
 *     query heads of the kv group                              (step 15)
 * Views as orc_attn_bwd (Qs, Ks, Vo, Vr, Gr, Qt, Kt, Gt), plus:
 *   Vkey, vkey_sf: the forward's per-key fold (as orc_attn_fwd_alg1);
 *   Kkey, kkey_sf: the strict dQ operand ([FLAMIA] sec. 4: per-query dS
 *     scales and the K fold): dQ_i takes U quantized per (query i, 32 keys)
 *     instead of per block, and on query i's own 128-token tile the folded
 *     values U_ij 2^ek_j times the per-key codes Kkey_j 2^-ek_j; dK keeps
 *     the block quantization.
 * cu_q == NULL: one document; cu_k == NULL: self-attention (Tk = Tq).
 * lse_ulps: with ORC_RND_LSE, the saved fp32 LSE moved by that many ulps.
 * units == NULL: every (document, kv head); else nunits pairs.  Outputs
 * dQ [Tq, Hq, d], dK and dV [Tk, Hkv, d], O [Tq, Hq, d], LSE (as saved) and
 * D [Hq, Tq] of the units' rows. */
void orc_attn_bwd_alg1(const double* Qs, const double* Ks, const double* Vo, const double* Vr, const double* Gr,
                       const double* Qt, const double* Kt, const double* Gt, const double* Vkey,
                       const uint8_t* vkey_sf, const double* Kkey, const uint8_t* kkey_sf, int64_t Tq, int64_t Tk,
                       int Hq, int Hkv, int d, const int32_t* cu_q, const int32_t* cu_k, int ndocs, int causal,
                       double alpha, int rnd, int64_t ref_tile, int lse_ulps, const int32_t* units, int nunits,
                       double* dQ, double* dK, double* dV, double* O, double* LSE, double* D)
{
    int nd = num_docs_eff(cu_q, ndocs);
    int nu = units ? nunits : nd * Hkv;
    int grp = Hq / Hkv;
    for (int u = 0; u < nu; ++u) {
        int b = units ? units[2 * u] : u / Hkv;
        int hk = units ? units[2 * u + 1] : u % Hkv;
        int64_t s, e, ks, ke;
        doc_range(cu_q, ndocs, Tq, b, &s, &e);
        key_range(cu_q, cu_k, ndocs, Tq, Tk, b, &ks, &ke);
        int64_t nq = e - s, nk = ke - ks;
        for (int64_t j = ks; j < ke; ++j)
            for (int k = 0; k < d; ++k) {
                dK[(j * Hkv + hk) * d + k] = 0.0;
                dV[(j * Hkv + hk) * d + k] = 0.0;
            }
        if (nq <= 0 || nk <= 0)
            continue;
        double* Ub = (double*)malloc(sizeof(double) * (size_t)nq * (size_t)nk); /* U~ of one query head */
        for (int hh = 0; hh < grp; ++hh) {
            int h = hk * grp + hh;
            /* rows, 32 at a time (one block row of U) */
#pragma omp parallel
            {
                double* Srow = (double*)malloc(sizeof(double) * (size_t)nk);
                double* y = (double*)malloc(sizeof(double) * (size_t)nk);
                double* mu = (double*)malloc(sizeof(double) * (size_t)nk);
                double* raw = (double*)malloc(sizeof(double) * (size_t)nk);
#pragma omp for schedule(dynamic, 1)
                for (int64_t qb = 0; qb < nq; qb += 32) {
                    int64_t qn = nq - qb < 32 ? nq - qb : 32;
                    for (int64_t r = 0; r < qn; ++r) {
                        int64_t i = s + qb + r;
                        int64_t kend = causal ? ks + (i - s) + 1 : ke;
                        int64_t diag0 = Vkey ? ks + ((i - s) / 128) * 128 : kend;
                        double* o = O + (i * Hq + h) * d;
                        double lse = fwd_row_alg1(Qs + (i * Hq + h) * d, Ks, Vo, Vkey, vkey_sf, Hkv, hk, d, ks, kend,
                                                  diag0, alpha, rnd, ref_tile, o, Srow, y, mu, raw);
                        if (rnd & ORC_RND_LSE)
                            lse = saved_lse(lse, lse_ulps);
                        LSE[(int64_t)h * Tq + i] = lse;
                        const double* g = Gr + (i * Hq + h) * d;
                        double Di = dot(g, o, d);
                        D[(int64_t)h * Tq + i] = Di;
                        double* urow = Ub + (qb + r) * nk;
                        for (int64_t j = ks; j < ke; ++j) {
                            if (j < kend) {
                                double P = exp(Srow[j - ks] - lse);
                                double E = dot(g, Vr + (j * Hkv + hk) * d, d);
                                urow[j - ks] = P * (E - Di);
                            } else {
                                urow[j - ks] = 0.0;
                            }
                        }
                        /* strict dQ operand: per (query, 32 keys) from the unquantized U */
                        if (Kkey) {
                            int64_t kd0 = ks + ((i - s) / 128) * 128;
                            for (int64_t j = ks; j < kend; ++j)
                                y[j - ks] = j >= kd0 ? ldexp(urow[j - ks], (int)kkey_sf[j * Hkv + hk] - 127)
                                                     : urow[j - ks];
                            if (rnd & ORC_RND_DS)
                                for (int64_t g0 = ks; g0 < kend; g0 += 32)
                                    mx_round_group(y + (g0 - ks), (kend - g0 < 32 ? kend - g0 : 32), 1);
                            double* dq = dQ + (i * Hq + h) * d;
                            for (int k = 0; k < d; ++k)
                                dq[k] = 0.0;
                            for (int64_t j = ks; j < kend; ++j) {
                                if (j >= kd0) {
                                    int ek = (int)kkey_sf[j * Hkv + hk] - 127;
                                    const double* kr = Kkey + (j * Hkv + hk) * d;
                                    for (int k = 0; k < d; ++k)
                                        dq[k] += alpha * y[j - ks] * ldexp(kr[k], -ek);
                                } else {
                                    const double* kr = Kt + (j * Hkv + hk) * d;
                                    for (int k = 0; k < d; ++k)
                                        dq[k] += alpha * y[j - ks] * kr[k];
                                }
                            }
                        }
                    }
                    /* step 14: the 32 x 32 blocks of this block row */
                    if (rnd & ORC_RND_DS)
                        for (int64_t kb = 0; kb < nk; kb += 32) {
                            int64_t kn = nk - kb < 32 ? nk - kb : 32;
                            double amax = 0.0;
                            for (int64_t r = 0; r < qn; ++r)
                                for (int64_t c = 0; c < kn; ++c) {
                                    double a = fabs(Ub[(qb + r) * nk + kb + c]);
                                    if (a > amax)
                                        amax = a;
                                }
                            int ex = orc_mx_exponent(amax);
                            for (int64_t r = 0; r < qn; ++r)
                                for (int64_t c = 0; c < kn; ++c) {
                                    double* x = Ub + (qb + r) * nk + kb + c;
                                    *x = ldexp(orc_e4m3_round(ldexp(*x, -ex)), ex);
                                }
                        }
                    if (!Kkey)
                        for (int64_t r = 0; r < qn; ++r) {
                            int64_t i = s + qb + r;
                            double* dq = dQ + (i * Hq + h) * d;
                            for (int k = 0; k < d; ++k)
                                dq[k] = 0.0;
                            for (int64_t j = ks; j < ke; ++j) {
                                double uq = Ub[(qb + r) * nk + (j - ks)];
                                if (uq == 0.0)
                                    continue;
                                const double* kr = Kt + (j * Hkv + hk) * d;
                                for (int k = 0; k < d; ++k)
                                    dq[k] += alpha * uq * kr[k];
                            }
                        }
                }
                free(Srow);
                free(y);
                free(mu);
                free(raw);
            }
            /* key rows: dV and dK of this query head */
#pragma omp parallel for schedule(dynamic, 8)
            for (int64_t j = ks; j < ke; ++j) {
                double* dk = dK + (j * Hkv + hk) * d;
                double* dv = dV + (j * Hkv + hk) * d;
                const double* kj = Ks + (j * Hkv + hk) * d;
                int64_t ibeg = causal ? s + (j - ks) : s;
                for (int64_t i = ibeg; i < e; ++i) {
                    double S = alpha * dot(Qs + (i * Hq + h) * d, kj, d);
                    double P = exp(S - LSE[(int64_t)h * Tq + i]);
                    double P8 = (rnd & ORC_RND_P8) ? orc_e4m3_round(256.0 * P) / 256.0 : P;
                    double uq = Ub[(i - s) * nk + (j - ks)];
                    const double* gt = Gt + (i * Hq + h) * d;
                    const double* qt = Qt + (i * Hq + h) * d;
                    for (int k = 0; k < d; ++k) {
                        dv[k] += P8 * gt[k];
                        dk[k] += alpha * uq * qt[k];
                    }
                }
            }
        }
        free(Ub);
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
