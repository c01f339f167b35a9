/*
 * fp4_oracle.c -- CPU oracle for the FP4 block-scaled quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded restatement
 * of what the pages define. Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header, table or constant generator with the CUDA library.
 *
 * Sources, cited by page title and section:
 *   [NV] "Pretraining Large Language Models with NVFP4" (arXiv 2509.25149):
 *        section A3 (background: E2M1 value set, MXFP4/NVFP4 scales, tensor-core
 *        semantics), sections 4.2-4.4 (RHT, 2D scaling, stochastic rounding),
 *        App. B.1-B.4 (quantisation), App. C (Hadamard transform).
 *   [UE] arXiv 2609.02846 summary page ("UE5M3 block scales"): method-details
 *        bullets and the English abstract (UE5M3 scales, held amax refreshed
 *        every 50 steps, target T, SR on backward gradients only).
 *   [PX] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
 *        SC'11 -- the Philox4x32-10 counter-based generator.
 *
 * Arithmetic: every quantiser step is one IEEE binary32 operation rounded to
 * nearest-even (the file is built with -ffp-contract=off, so nothing is fused);
 * the GEMM sums run in binary64. Where the pages are silent the reading taken is
 * marked "Reading:" and listed in the design notes.
 *
 * Parity status: every function here is pinned by a CPU test against values the
 * pages print, closed forms, library routines or brute force -- except the
 * scale-layout permutation (orc_swizzle_scales), whose pins are a bijection test
 * and the GPU GEMM parity, and Philox against an independent library
 * implementation (Triton's), not a published known-answer table.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_SHAPE 2
#define ORC_ERR_STATE 3

/* scale formats */
#define ORC_FMT_E4M3 0  /* NVFP4 block scale */
#define ORC_FMT_UE5M3 1 /* UE5M3 block scale ([UE]) */
#define ORC_FMT_UE8M0 2 /* MXFP4 block scale ([NV] A3) */

/* block shapes */
#define ORC_BLOCK_1x16 0
#define ORC_BLOCK_16x16 1
#define ORC_BLOCK_1x32 2

int orc_version(void) { return 1; }

/* ------------------------------------------------------------------------- */
/* Number formats                                                             */
/* ------------------------------------------------------------------------- */

/* BF16 is the upper half of an IEEE binary32 pattern, so widening is exact. */
float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* [NV] A3: an E2M1 element has one sign, two exponent and one mantissa bit and
 * encodes +-0, 0.5, 1, 1.5, 2, 3, 4, 6. Code = sign*8 + magnitude index. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint8_t code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Generic unsigned minifloat with `ebits` exponent bits, `mbits` mantissa bits,
 * exponent bias `bias` and subnormals at exponent field 0.
 *
 * Round x >= 0 to the nearest representable value with ties to the value whose
 * last mantissa bit is 0 (round-to-nearest-even), then saturate to `maxval`
 * ("satfinite"). The rounding is the textbook one: pick the quantum q of the
 * binade that holds x (the subnormal quantum below the smallest normal), scale
 * x by 1/q (exact: q is a power of two), round to an integer with rint() in the
 * default ties-to-even mode, and scale back. */
double orc_minifloat_round(double x, int ebits, int mbits, int bias, double maxval) {
    (void)ebits;
    if (!(x > 0.0)) return 0.0;
    if (x >= maxval) return maxval;
    double min_normal = ldexp(1.0, 1 - bias);
    double q;
    if (x < min_normal) {
        q = ldexp(1.0, 1 - bias - mbits);
    } else {
        int e;
        frexp(x, &e); /* x = f * 2^e, f in [0.5, 1) -> binade [2^(e-1), 2^e) */
        q = ldexp(1.0, (e - 1) - mbits);
    }
    double r = rint(x / q) * q;
    return r > maxval ? maxval : r;
}

/* Encode a representable unsigned minifloat value into its code bits. */
static uint8_t minifloat_code(double v, int mbits, int bias) {
    if (v == 0.0) return 0;
    double min_normal = ldexp(1.0, 1 - bias);
    if (v < min_normal) {
        double m = v / ldexp(1.0, 1 - bias - mbits);
        return (uint8_t)m; /* exponent field 0 */
    }
    int e;
    double f = frexp(v, &e); /* v = f*2^e, f in [0.5,1) -> v = (2f) * 2^(e-1) */
    int efield = (e - 1) + bias;
    int mant = (int)((2.0 * f - 1.0) * (double)(1 << mbits));
    return (uint8_t)((efield << mbits) | mant);
}

static double minifloat_value(uint8_t code, int mbits, int bias) {
    int efield = code >> mbits;
    int mant = code & ((1 << mbits) - 1);
    if (efield == 0) return ldexp((double)mant, 1 - bias - mbits);
    return ldexp(1.0 + (double)mant / (double)(1 << mbits), efield - bias);
}

/* Scale formats.
 *   E4M3 ([NV] App. B.1: largest magnitude 448): OCP FP8 E4M3 -- bias 7,
 *     subnormals, 0x7F is NaN, so the largest finite code 0x7E = 448. The scale
 *     is non-negative, so the sign bit is always 0.
 *   UE5M3 ([UE]): unsigned, 5 exponent bits, 3 mantissa bits. Reading: bias 15,
 *     subnormals at exponent field 0, no infinities, 0xFF is NaN, so the largest
 *     finite code is 0xFE = 1.75 * 2^16 = 114688 and the smallest subnormal 2^-17.
 *   UE8M0 ([NV] A3): 2^(code-127), code 0..254, 0xFF NaN. */
#define UE5M3_MAX 114688.0

double orc_scale_max(int fmt) {
    if (fmt == ORC_FMT_E4M3) return 448.0;
    if (fmt == ORC_FMT_UE5M3) return UE5M3_MAX;
    return ldexp(1.0, 127);
}

double orc_scale_decode(int fmt, uint8_t code) {
    if (fmt == ORC_FMT_E4M3) return minifloat_value(code & 0x7F, 3, 7);
    if (fmt == ORC_FMT_UE5M3) return minifloat_value(code, 3, 15);
    return ldexp(1.0, (int)code - 127);
}

/* RNE + satfinite encode of a non-negative FP32 scale s (E4M3 or UE5M3). */
uint8_t orc_scale_encode(int fmt, float s) {
    double v;
    if (fmt == ORC_FMT_E4M3) {
        v = orc_minifloat_round((double)s, 4, 3, 7, 448.0);
        return minifloat_code(v, 3, 7);
    }
    v = orc_minifloat_round((double)s, 5, 3, 15, UE5M3_MAX);
    return minifloat_code(v, 3, 15);
}

/* E2M1 with round-to-nearest-even and saturation at +-6 ([NV] App. B.3, the
 * conversion Q(.); A3 "saturate"). Reading: the code's sign bit is the input's
 * sign bit, so -0 and negative values that round to zero give code 0x8. */
uint8_t orc_e2m1_rne(float v) {
    double a = fabs((double)v);
    double r = orc_minifloat_round(a, 2, 1, 1, 6.0);
    uint8_t mag = minifloat_code(r, 1, 1);
    return (uint8_t)((signbit(v) ? 8 : 0) | mag);
}

/* Stochastic rounding ([NV] 4.4): round |v| to one of its two neighbouring E2M1
 * magnitudes lo <= |v| < hi, choosing hi with probability proportional to the
 * distance from lo. Reading of the random-bit contract: the one of the native
 * FP4 stochastic-rounding conversion that [NV] A3 ("hardware support") says
 * Blackwell provides -- each element draws a uniform 16-bit integer R and rounds
 * up iff R + floor(frac * 2^16) >= 2^16, where frac = (|v| - lo) / (hi - lo).
 * frac is exact in FP32 (Sterbenz lemma: hi <= 2 lo whenever lo > 0, and hi - lo
 * is a power of two), and so are frac * 2^16 and its floor, so
 * P(up) = floor(frac * 2^16) / 2^16, within 2^-16 of frac (never above it).
 * |v| >= 6 saturates to 6; the code's sign bit is v's. */
uint8_t orc_e2m1_sr(float v, uint32_t r16) {
    float a = fabsf(v);
    uint8_t sign = signbit(v) ? 8 : 0;
    if (a >= 6.0f) return (uint8_t)(sign | 7);
    int lo = 0;
    while (lo < 7 && E2M1_MAG[lo + 1] <= (double)a) lo++;
    float flo = (float)E2M1_MAG[lo];
    float fhi = (float)E2M1_MAG[lo + 1];
    float frac = (a - flo) / (fhi - flo);
    uint32_t fh = (uint32_t)floorf(frac * 65536.0f);
    int up = (r16 & 0xFFFFu) + fh >= 65536u;
    return (uint8_t)(sign | (lo + up));
}

/* MXFP4 scale ([NV] A3 and App. B.4): the decode scale amax_B/6 rounded UP to
 * the next power of two. Reading of the exact rule: e is the smallest integer
 * with 6 * 2^e >= amax_B, found here by plain search; the caller clamps it to
 * the UE8M0 range [-127, 127]. amax_B == 0 gives -127. */
int orc_ue8m0_exponent(float amax_b) {
    if (!(amax_b > 0.0f)) return -127;
    int e = -160;
    while (ldexp(6.0, e) < (double)amax_b) e++;
    return e;
}

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 ([PX]): 10 rounds of the multiply-xor bijection on a 4x32-bit  */
/* counter, with the 2x32-bit key advanced by the Weyl constants each round.   */
/* ------------------------------------------------------------------------- */

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; round++) {
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Reading of the stochastic-rounding bits: one Philox(key = seed, counter =
 * (lo32(e>>3), hi32(e>>3), tensor_id, lo32(step))) call serves the eight
 * elements e>>3 of the quantized operand (e its row-major linear index). Each
 * 32-bit word serves two of them: word 2 ((e>>2) & 1) + (e & 1), so a quad of
 * elements 4q .. 4q+3 takes two words, one for its even and one for its odd
 * elements. Within the word, the element with (e>>1) & 1 == 0 takes bytes 2
 * (high) and 0 (low), the other bytes 3 (high) and 1 (low) -- the two 16-bit
 * draws the native conversion reads from one random operand. Returns R. */
uint32_t orc_sr_bits(uint64_t seed, uint32_t tensor_id, uint64_t step, uint64_t e) {
    uint32_t ctr[4] = {(uint32_t)(e >> 3), (uint32_t)(e >> 35), tensor_id, (uint32_t)step};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    uint32_t word = w[2 * ((e >> 2) & 1) + (e & 1)];
    if (((e >> 1) & 1) == 0) return (((word >> 16) & 0xFFu) << 8) | (word & 0xFFu);
    return ((word >> 24) << 8) | ((word >> 8) & 0xFFu);
}

/* ------------------------------------------------------------------------- */
/* Random Hadamard transform ([NV] 4.2 and App. C)                             */
/* ------------------------------------------------------------------------- */

/* [NV] 4.2: one random diagonal sign vector D_r, shared by every layer for the
 * whole run. Reading: bit i of word 0 of Philox(key = seed,
 * counter = (0, 0, 0xFFFFFFFF, 0xFFFFFFFF)) set means d_i = -1. */
uint32_t orc_rht_sign_word(uint64_t seed) {
    uint32_t ctr[4] = {0u, 0u, 0xFFFFFFFFu, 0xFFFFFFFFu};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    return w[0] & 0xFFFFu;
}

/* [NV] App. C: v' = H_r v with H_r = D_r H_16 and H_16 the normalised Sylvester
 * Hadamard matrix H_N = (1/sqrt 2) H_2 (x) H_{N/2}. Reading of the FP32 order:
 * the unnormalised transform is formed by butterfly stages of half-width 1, 2,
 * 4, 8 -- each pair (i, i+h) with (i & h) == 0 becomes (a + b, a - b) -- then
 * every element is multiplied by 1/4 = (1/sqrt 2)^4, then element i by d_i. */
void orc_rht16(float v[16], uint32_t sign_word) {
    for (int h = 1; h < 16; h <<= 1) {
        for (int i = 0; i < 16; i++) {
            if (i & h) continue;
            float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    for (int i = 0; i < 16; i++) {
        v[i] = v[i] * 0.25f;
        if ((sign_word >> i) & 1u) v[i] = -v[i];
    }
}

/* ------------------------------------------------------------------------- */
/* Quantiser                                                                  */
/* ------------------------------------------------------------------------- */

/* The quantized operand is a matrix A' of R' x C' values whose columns run along
 * the GEMM dot-product dimension ([NV] 4.3: scaling is applied along the dot
 * dimension). Rowwise: A' = X. Colwise: A' = X^T (the backward-pass operand). */
typedef struct {
    const uint16_t* in;
    int64_t rows, cols; /* input X, row-major BF16 */
    int colwise;
} operand_t;

static float operand_at(const operand_t* op, int64_t r, int64_t c) {
    if (op->colwise) return orc_bf16_to_f32(op->in[c * op->cols + r]);
    return orc_bf16_to_f32(op->in[r * op->cols + c]);
}

/* Load the 16 consecutive dot-dimension values of operand row r starting at
 * column c0, applying the RHT when requested (the RHT tile is the 1x16 block). */
static void load16(const operand_t* op, int64_t r, int64_t c0, int rht, uint32_t signs, float v[16]) {
    for (int i = 0; i < 16; i++) v[i] = operand_at(op, r, c0 + i);
    if (rht) orc_rht16(v, signs);
}

/* [NV] App. B.1: amax_X = max |x_i| over the whole tensor; with the RHT the
 * amax is taken in the rotated space ([NV] App. C: the scale is computed on H X). */
float orc_tensor_amax(const uint16_t* in, int64_t rows, int64_t cols, int colwise, int rht, uint64_t seed) {
    operand_t op = {in, rows, cols, colwise};
    int64_t R = colwise ? cols : rows, C = colwise ? rows : cols;
    uint32_t signs = orc_rht_sign_word(seed);
    float amax = 0.0f;
    for (int64_t r = 0; r < R; r++) {
        for (int64_t c0 = 0; c0 < C; c0 += 16) {
            float v[16];
            load16(&op, r, c0, rht, signs, v);
            for (int i = 0; i < 16; i++) {
                float a = fabsf(v[i]);
                if (a > amax) amax = a;
            }
        }
    }
    return amax;
}

/* [NV] App. B.1-B.2: s_enc,G maps the largest local decode scale
 * max_B s_dec,L,B = amax_X / 6 onto the scale format's target T, i.e.
 * s_enc,G = 6 T / amax_X (T = 448, the E4M3 maximum, for NVFP4; [UE]: T = 448 by
 * default or 2048 for UE5M3 scales with a held amax). Reading for edge cases:
 * amax == 0 gives 1; a non-finite quotient gives FLT_MAX. */
float orc_global_encode_scale(float amax, float target_T) {
    if (amax == 0.0f) return 1.0f;
    float six_t = 6.0f * target_T;
    float s = six_t / amax;
    if (!isfinite(s)) s = 3.40282346638528859812e+38f;
    return s;
}

/* Quantize input X (rows x cols, row-major BF16) into the operand A'.
 *
 * Outputs cover operand rows [op_r0, op_r1):
 *   codes  : (op_r1-op_r0) x C'/2 bytes, element 2i in the low nibble of byte i
 *            (Reading: the tensor-core packing order), row-major;
 *   scales : (op_r1-op_r0) x C'/bs bytes, plain row-major, one per 1 x bs block
 *            (a 16x16 block's scale is repeated for each of its 16 rows, [NV] 4.3);
 *   *s_dec_out = s_dec,G (1.0 for MXFP4); *amax_out = the amax the scale used.
 *   counters[0..3] += elem_sat, elem_underflow, scale_sat, scale_underflow.
 *     Reading: elem_sat counts |v| > 6 before rounding; elem_underflow counts
 *     x != 0 whose code magnitude is 0; scale_sat counts blocks whose scale
 *     exceeds the format maximum before encoding; scale_underflow counts blocks
 *     with amax_B > 0 and an encoded scale of 0 (MXFP4: an exponent clamped up
 *     to -127). Each element / block is counted once.
 *
 * Tensor scale: MXFP4 has none ([NV] A3). Otherwise current scaling uses the
 * amax of this tensor; held scaling ([UE]: the amax is refreshed every
 * `refresh_every` steps and held in between) refreshes when
 * step % refresh_every == 0 or when the held state is not valid yet, and
 * otherwise uses the held amax.
 *
 * per_row ([NV] B.1: the global scale may span a smaller granularity, such as
 * a row, to save the extra memory pass). Reading: each operand row r gets its
 * own s_enc,G(r) = 6 * T / amax_r with amax_r = max |x| over that row -- B.1's
 * formula with the tensor replaced by the row -- and s_dec,G(r) = 1 / s_enc,G(r)
 * goes to s_dec_rows[r - op_r0]; *s_dec_out and *amax_out are set to 0. Current
 * scaling of a plain (no RHT) rowwise 1 x 16 operand only; held must be 0. */
int orc_quantize(int scale_fmt, int block, int sr, int colwise, int rht,
                 uint64_t seed, uint32_t tensor_id, uint64_t step,
                 int held, float target_T, uint32_t refresh_every,
                 float* st_amax, int32_t* st_valid, uint64_t* st_last,
                 const uint16_t* in, int64_t rows, int64_t cols,
                 int64_t op_r0, int64_t op_r1,
                 uint8_t* codes, uint8_t* scales, float* s_dec_out, float* amax_out,
                 uint64_t counters[4], int per_row, float* s_dec_rows) {
    int64_t R = colwise ? cols : rows, C = colwise ? rows : cols;
    int bs = (block == ORC_BLOCK_1x32) ? 32 : 16;
    int two_d = (block == ORC_BLOCK_16x16);
    if (scale_fmt < 0 || scale_fmt > 2 || block < 0 || block > 2) return ORC_ERR_ARG;
    if ((scale_fmt == ORC_FMT_UE8M0) != (block == ORC_BLOCK_1x32)) return ORC_ERR_ARG;
    if (rht && block != ORC_BLOCK_1x16) return ORC_ERR_ARG;
    if (R < 0 || C < 0 || C % bs != 0) return ORC_ERR_SHAPE;
    if (two_d && R % 16 != 0) return ORC_ERR_SHAPE;
    if (op_r0 < 0 || op_r1 > R || op_r0 > op_r1) return ORC_ERR_SHAPE;
    if (two_d && op_r0 % 16 != 0) return ORC_ERR_SHAPE;
    if (per_row && (held || colwise || rht || block != ORC_BLOCK_1x16 || scale_fmt == ORC_FMT_UE8M0 ||
                    s_dec_rows == NULL))
        return ORC_ERR_ARG;

    operand_t op = {in, rows, cols, colwise};
    uint32_t signs = orc_rht_sign_word(seed);

    /* Tensor-level scale (B.1), current or held. */
    float s_enc_g = 1.0f, s_dec_g = 1.0f, amax_used = 0.0f;
    if (scale_fmt != ORC_FMT_UE8M0 && !per_row) {
        if (held) {
            if (refresh_every == 0) return ORC_ERR_ARG;
            if (step % refresh_every == 0 || !*st_valid) {
                amax_used = orc_tensor_amax(in, rows, cols, colwise, rht, seed);
                *st_amax = amax_used;
                *st_valid = 1;
                *st_last = step;
            } else {
                amax_used = *st_amax;
            }
        } else {
            amax_used = orc_tensor_amax(in, rows, cols, colwise, rht, seed);
        }
        s_enc_g = orc_global_encode_scale(amax_used, target_T);
        s_dec_g = 1.0f / s_enc_g;
    }
    *s_dec_out = per_row ? 0.0f : s_dec_g;
    *amax_out = amax_used;

    int64_t nb = C / bs;
    float fmt_max = (float)orc_scale_max(scale_fmt);
    for (int64_t r = op_r0; r < op_r1; r++) {
        if (per_row) {
            /* B.1 over one row: the row's amax, its encode and decode scales */
            float amax_r = 0.0f;
            for (int64_t c = 0; c < C; c++) {
                float a = fabsf(operand_at(&op, r, c));
                if (a > amax_r) amax_r = a;
            }
            s_enc_g = orc_global_encode_scale(amax_r, target_T);
            s_dec_g = 1.0f / s_enc_g;
            s_dec_rows[r - op_r0] = s_dec_g;
        }
        for (int64_t b = 0; b < nb; b++) {
            int64_t c0 = b * bs;
            float v[32];
            /* the block's own values (post-RHT when requested) */
            if (bs == 32) {
                for (int i = 0; i < 32; i++) v[i] = operand_at(&op, r, c0 + i);
            } else {
                load16(&op, r, c0, rht, signs, v);
            }
            /* block amax: over the 1 x bs block, or the whole 16 x 16 tile */
            float amax_b = 0.0f;
            if (two_d) {
                int64_t rt0 = (r / 16) * 16;
                for (int64_t rr = rt0; rr < rt0 + 16; rr++)
                    for (int i = 0; i < 16; i++) {
                        float a = fabsf(operand_at(&op, rr, c0 + i));
                        if (a > amax_b) amax_b = a;
                    }
            } else {
                for (int i = 0; i < bs; i++) {
                    float a = fabsf(v[i]);
                    if (a > amax_b) amax_b = a;
                }
            }
            int count_block = !two_d || (r % 16 == 0);

            uint8_t scode;
            float s_enc_l = 0.0f; /* 0 marks a zero scale: no division happens */
            if (scale_fmt == ORC_FMT_UE8M0) {
                /* B.4: power-of-two decode scale rounded up; value scaled by 2^-e. */
                int e = orc_ue8m0_exponent(amax_b);
                if (e > 127) { e = 127; if (count_block) counters[2]++; }
                if (e < -127) { e = -127; if (count_block && amax_b > 0.0f) counters[3]++; }
                scode = (uint8_t)(e + 127);
                s_enc_l = ldexpf(1.0f, -e);
            } else {
                /* B.2: s_dec,L,B = amax_B / 6, multiplied by s_enc,G, rounded
                 * (RNE, satfinite) into the scale format. */
                float s_dec_l = amax_b / 6.0f;
                float s = s_dec_l * s_enc_g;
                if (s > fmt_max && count_block) counters[2]++;
                scode = orc_scale_encode(scale_fmt, s);
                if (scode == 0) {
                    if (amax_b > 0.0f && count_block) counters[3]++;
                } else {
                    /* B.2: s_enc,L,B = 1 / (fp32(s_hat) * s_dec,G) */
                    float s_hat = (float)orc_scale_decode(scale_fmt, scode);
                    float denom = s_hat * s_dec_g;
                    s_enc_l = 1.0f / denom;
                }
            }
            scales[(r - op_r0) * nb + b] = scode;

            for (int i = 0; i < bs; i++) {
                float x = v[i];
                int64_t c = c0 + i;
                uint8_t code;
                if (s_enc_l == 0.0f) {
                    code = signbit(x) ? 8 : 0;
                } else {
                    /* B.3: x_hat = Q(x * s_enc,L,B) */
                    float val = x * s_enc_l;
                    if (fabsf(val) > 6.0f) counters[0]++;
                    if (sr) {
                        uint64_t e = (uint64_t)r * (uint64_t)C + (uint64_t)c;
                        code = orc_e2m1_sr(val, orc_sr_bits(seed, tensor_id, step, e));
                    } else {
                        code = orc_e2m1_rne(val);
                    }
                }
                if (x != 0.0f && (code & 7) == 0) counters[1]++;
                uint8_t* byte = &codes[(r - op_r0) * (C / 2) + c / 2];
                if (c % 2 == 0) *byte = (uint8_t)((*byte & 0xF0) | code);
                else *byte = (uint8_t)((*byte & 0x0F) | (code << 4));
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Dequantize ([NV] A3: decoded back to the original range with the scales;   */
/* App. B.3: the local and global decode scales are stored with the codes).   */
/* x~ = RN(RN(e2m1 * s_hat) * s_dec,G) in FP32; the first product is exact.    */
/* ------------------------------------------------------------------------- */
void orc_dequantize(int scale_fmt, int bs, int64_t R, int64_t C,
                    const uint8_t* codes, const uint8_t* scales, float s_dec_g, const float* s_dec_rows,
                    float* out) {
    int64_t nb = C / bs;
    for (int64_t r = 0; r < R; r++)
        for (int64_t c = 0; c < C; c++) {
            uint8_t byte = codes[r * (C / 2) + c / 2];
            uint8_t code = (c % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            float e = (float)orc_e2m1_value(code);
            float s = (float)orc_scale_decode(scale_fmt, scales[r * nb + c / bs]);
            float t = e * s;
            out[r * C + c] = t * (s_dec_rows != NULL ? s_dec_rows[r] : s_dec_g);
        }
}

/* ------------------------------------------------------------------------- */
/* Block-scaled GEMM ([NV] App. B.3 "Tensor Core processing" and A3 hardware   */
/* support: each 16/32-element partial dot product is multiplied by both block */
/* decode scales, accumulated in high precision, and the two global decode     */
/* scales are applied to the final output).                                   */
/*                                                                            */
/*   C[m,n] = s_dec,G,A * s_dec,G,B * sum_k (e2m1(a_mk) s_A) (e2m1(b_nk) s_B)  */
/*   (s_dec,G,A[m] per row of A when a_sdec_rows != NULL: [NV] B.1's finer     */
/*   granularity; a row's decode scale is constant along the dot dimension)    */
/*   S[m,n] = |s_dec,G,A * s_dec,G,B| * sum_k |(e2m1(a_mk) s_A)(e2m1(b_nk) s_B)| */
/*                                                                            */
/* in binary64: every factor is exact in binary32 and every product exact in  */
/* binary64. A and B are both K-major: A is M x K, B is N x K, codes packed two */
/* per byte, plain scales M x K/bs and N x K/bs.                              */
/* If ms == NULL the full M x N output is written row-major; otherwise only   */
/* the npairs outputs (ms[i], ns[i]).                                          */
/* ------------------------------------------------------------------------- */
static double dq(int scale_fmt, int bs, int64_t K, const uint8_t* codes, const uint8_t* scales, int64_t r, int64_t k) {
    uint8_t byte = codes[r * (K / 2) + k / 2];
    uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    return orc_e2m1_value(code) * orc_scale_decode(scale_fmt, scales[r * (K / bs) + k / bs]);
}

static void gemm_one(int scale_fmt, int bs, int64_t K,
                     const uint8_t* a_codes, const uint8_t* a_scales, float a_sdec,
                     const uint8_t* b_codes, const uint8_t* b_scales, float b_sdec,
                     int64_t m, int64_t n, double* c_out, double* s_out) {
    double sum = 0.0, sabs = 0.0;
    for (int64_t k = 0; k < K; k++) {
        double p = dq(scale_fmt, bs, K, a_codes, a_scales, m, k) * dq(scale_fmt, bs, K, b_codes, b_scales, n, k);
        sum += p;
        sabs += fabs(p);
    }
    double alpha = (double)a_sdec * (double)b_sdec;
    *c_out = alpha * sum;
    *s_out = fabs(alpha) * sabs;
}

void orc_gemm(int scale_fmt, int bs, int64_t M, int64_t N, int64_t K,
              const uint8_t* a_codes, const uint8_t* a_scales, float a_sdec, const float* a_sdec_rows,
              const uint8_t* b_codes, const uint8_t* b_scales, float b_sdec,
              const int64_t* ms, const int64_t* ns, int64_t npairs,
              double* c_ref, double* s_abs) {
    if (ms == NULL) {
        for (int64_t m = 0; m < M; m++)
            for (int64_t n = 0; n < N; n++)
                gemm_one(scale_fmt, bs, K, a_codes, a_scales, a_sdec_rows != NULL ? a_sdec_rows[m] : a_sdec,
                         b_codes, b_scales, b_sdec, m, n, &c_ref[m * N + n], &s_abs[m * N + n]);
    } else {
        for (int64_t i = 0; i < npairs; i++)
            gemm_one(scale_fmt, bs, K, a_codes, a_scales, a_sdec_rows != NULL ? a_sdec_rows[ms[i]] : a_sdec,
                     b_codes, b_scales, b_sdec, ms[i], ns[i], &c_ref[i], &s_abs[i]);
    }
}

/* ------------------------------------------------------------------------- */
/* Tensor-core scale-factor layout. The pages say only that the tensor cores   */
/* read one 8-bit scale per 16/32-element block ([NV] A3). The byte order is   */
/* the one the PTX ISA's tcgen05 block-scaling section gives for a scale       */
/* matrix copied into tensor memory with 32 lanes x 128 bits replicated to the */
/* four lane quadrants: within a chunk of 128 rows x 4 consecutive blocks      */
/* (512 bytes), row r and block j sit at byte 16*(r % 32) + 4*(r / 32) + j.   */
/* Reading: chunks are stored row-tile major, the K chunks of one 128-row tile */
/* contiguous: chunk (rt, kt) starts at byte 512 * (rt * NB/4 + kt).           */
/* ------------------------------------------------------------------------- */
int orc_swizzle_scales(int64_t R, int64_t NB, const uint8_t* plain, uint8_t* out) {
    if (R % 128 != 0 || NB % 4 != 0) return ORC_ERR_SHAPE;
    for (int64_t r = 0; r < R; r++)
        for (int64_t j = 0; j < NB; j++) {
            int64_t rt = r / 128, kt = j / 4, rr = r % 128, jj = j % 4;
            int64_t off = 512 * (rt * (NB / 4) + kt) + 16 * (rr % 32) + 4 * (rr / 32) + jj;
            out[off] = plain[r * NB + j];
        }
    return ORC_OK;
}
