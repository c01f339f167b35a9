// fp4_device.cuh -- device-side number formats, counter-based RNG and the
// 16-point Hadamard transform used by the quantizer kernels (sm_103a).
//
// Every quantizer step is one IEEE binary32 operation rounded to nearest-even;
// the __f*_rn intrinsics below keep the compiler from fusing or reordering
// them, so the GPU reproduces the published step order bit for bit.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp4bs {

// Device status codes (same numbers as fp4_status_t).
constexpr int kStatusOk = 0;
constexpr int kStatusState = 5;
constexpr int kStatusTimeout = 7;

__device__ __forceinline__ void record_status(int* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// BF16 halves of a 32-bit word widened to FP32 (BF16 is the top half of an
// FP32 pattern, so the widening is exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Unpack 16 BF16 values held in two 128-bit words.
__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float v[16]) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
}

// ---------------------------------------------------------------------------
// E2M1 ("Pretraining LLMs with NVFP4", section A3): magnitudes
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}, code = sign * 8 + magnitude index.
//
// Stochastic rounding (section 4.4; section A3, hardware support: Blackwell
// converts to FP4 with stochastic rounding natively). Element x rounds |x| in
// [lo, hi) up iff R + floor(frac * 2^16) >= 2^16 for its 16-bit draw R, where
// frac = (|x| - lo) / (hi - lo); |x| >= 6 saturates; the code keeps x's sign.
// That is the decision of cvt.rs.satfinite.e2m1x4.f32. Of its four sources the
// 4th (lowest result nibble) takes R from bytes 2 (high) and 0 (low) of the
// random operand and the 2nd (third nibble) from bytes 3 and 1 (measured on
// GB300 over 10^7 probed element/draw pairs, no mismatch); the other two read
// bit-reversed copies of the same bits and are fed zeros here. So one 32-bit
// random word serves two elements as it stands. Returns x_lo's code in nibble 0
// and x_hi's in nibble 2 (nibbles 1 and 3 zero).
__device__ __forceinline__ uint32_t e2m1_sr_pair_hw(float x_lo, float x_hi, uint32_t rbits) {
    uint16_t d;
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(d)
        : "f"(0.0f), "f"(x_hi), "f"(0.0f), "f"(x_lo), "r"(rbits));
    return d;
}

// Sixteen SR codes (element i in nibble i of lo / hi) from the eight words of
// the block's two Philox calls (sr_block_bits): quad q = 4q .. 4q + 3 draws its
// even elements (4q, 4q + 2) from word 2 (q & 1) of r[q >> 1] and its odd ones
// (4q + 1, 4q + 3) from word 2 (q & 1) + 1, so the odd pair's conversion lands
// one nibble up and one add interleaves the two into the quad's 16 bits.
__device__ __forceinline__ void e2m1_sr_x16(const float x[16], const uint4 r[2], uint32_t& lo, uint32_t& hi) {
    uint32_t qd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t we = (q & 1) ? r[q >> 1].z : r[q >> 1].x;
        const uint32_t wo = (q & 1) ? r[q >> 1].w : r[q >> 1].y;
        qd[q] = e2m1_sr_pair_hw(x[4 * q], x[4 * q + 2], we) + 16u * e2m1_sr_pair_hw(x[4 * q + 1], x[4 * q + 3], wo);
    }
    lo = __byte_perm(qd[0], qd[1], 0x5410u);
    hi = __byte_perm(qd[2], qd[3], 0x5410u);
}

// Eight FP32 values -> eight E2M1 codes (element i in nibble i) with the
// hardware conversion cvt.rn.satfinite.e2m1x2.f32, which rounds to nearest-even,
// saturates at +-6 and keeps the sign of values that round to zero (its first
// source goes to the upper nibble).
__device__ __forceinline__ uint32_t e2m1_rne_x8(const float* v) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// Number of zero-magnitude codes among the 8 nibbles of a code word.
__device__ __forceinline__ uint32_t zero_mag_count8(uint32_t w) {
    const uint32_t t = w & 0x77777777u;
    return 8u - (uint32_t)__popc((t | (t >> 1) | (t >> 2)) & 0x11111111u);
}


// ---------------------------------------------------------------------------
// Block-scale formats with a 3-bit mantissa, encoded round-to-nearest-even and
// saturating ("satfinite"): E4M3 (bias 7, largest finite code 0x7E = 448) and
// UE5M3 (bias 15, largest finite code 0xFE = 114688, 0xFF reserved). The input
// is a non-negative FP32 scale. Normal range: round the FP32 mantissa to 3 bits
// (add half an ulp minus one plus the kept LSB, then truncate) and rebias the
// exponent; subnormal range: scale by the reciprocal subnormal quantum (a power
// of two, exact) and round to an integer.
template <int BIAS, uint32_t MAXCODE>
__device__ __forceinline__ uint32_t scale_encode_m3(float s, float maxval) {
    if (!(s > 0.0f)) return 0u;
    if (s >= maxval) return MAXCODE;
    const float min_normal = __uint_as_float((uint32_t)(127 + 1 - BIAS) << 23);
    if (s < min_normal) {
        const float inv_quantum = __uint_as_float((uint32_t)(127 + BIAS + 2) << 23);
        return (uint32_t)__float2int_rn(__fmul_rn(s, inv_quantum));
    }
    const uint32_t b = __float_as_uint(s);
    const uint32_t r = b + 0x7FFFFu + ((b >> 20) & 1u);
    const uint32_t code = ((((r >> 23) & 0xFFu) - 127u + (uint32_t)BIAS) << 3) | ((r >> 20) & 7u);
    return code < MAXCODE ? code : MAXCODE;
}

template <int BIAS>
__device__ __forceinline__ float scale_decode_m3(uint32_t code) {
    const uint32_t e = (code >> 3) & 0x1Fu, m = code & 7u;
    if (e == 0u) return __fmul_rn((float)m, __uint_as_float((uint32_t)(127 + 1 - BIAS - 3) << 23));
    return __uint_as_float(((e - (uint32_t)BIAS + 127u) << 23) | (m << 20));
}

constexpr int kFmtE4M3 = 0;
constexpr int kFmtUE5M3 = 1;
constexpr int kFmtUE8M0 = 2;

template <int FMT>
struct ScaleFmt;
// E4M3 through the hardware conversions: cvt.rn.satfinite.e4m3x2.f32 rounds to
// nearest-even (subnormals included) and saturates at 448; every E4M3 value is
// an FP16 value, so the decode through f16x2 is exact.
__device__ __forceinline__ uint32_t e4m3_encode_hw(float s) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(s));
    return (uint32_t)d & 0xFFu;
}
__device__ __forceinline__ float e4m3_decode_hw(uint32_t code) {
    uint32_t h2;
    const uint16_t c2 = (uint16_t)(code | (code << 8));  // same code in both lanes
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(h2));
    return f;
}

template <>
struct ScaleFmt<kFmtE4M3> {
    static constexpr float kMax = 448.0f;
    static constexpr uint32_t kMaxCode = 0x7Eu;
    __device__ static __forceinline__ uint32_t encode(float s) { return e4m3_encode_hw(s); }
    __device__ static __forceinline__ float decode(uint32_t c) { return e4m3_decode_hw(c & 0x7Fu); }
};
template <>
struct ScaleFmt<kFmtUE5M3> {
    static constexpr float kMax = 114688.0f;
    static constexpr uint32_t kMaxCode = 0xFEu;
    __device__ static __forceinline__ uint32_t encode(float s) { return scale_encode_m3<15, 0xFEu>(s, kMax); }
    __device__ static __forceinline__ float decode(uint32_t c) { return scale_decode_m3<15>(c); }
};

// MXFP4 scale (section A3, App. B.4): amax_B / 6 rounded up to a power of two.
// Returns the smallest e with 6 * 2^e >= amax (before clamping to [-127, 127]):
// with amax = 1.f * 2^E, 6 * 2^e = 1.5 * 2^(e+2), so e = E - 2 when 1.f <= 1.5
// and E - 1 otherwise. Subnormal amax gives -128 (below the range, clamped up).
__device__ __forceinline__ int ue8m0_exponent(float amax) {
    if (!(amax > 0.0f)) return -127;
    const uint32_t b = __float_as_uint(amax);
    const int E = (int)((b >> 23) & 0xFFu);
    if (E == 0) return -128;
    return (b & 0x7FFFFFu) <= 0x400000u ? E - 127 - 2 : E - 127 - 1;
}

// 2^k as an FP32 value for k in [-149, 127] (exact, subnormal below -126).
__device__ __forceinline__ float exp2_exact(int k) {
    if (k >= -126) return __uint_as_float((uint32_t)(k + 127) << 23);
    return __uint_as_float(1u << (k + 149));
}

// RN(a / 6) in binary32 by division with a precomputed reciprocal and one
// correction step (Markstein's residual correction, IBM J. Res. Dev. 34(1),
// 1990; Muller et al., "Handbook of Floating-Point Arithmetic", on division by
// a constant): q0 = RN(a * y) with y = RN(1/6), the residual r = a - 6 q0 is
// exact in one fused multiply-add, and q1 = RN(q0 + r * y). A GPU test checks
// it bit for bit against the correctly rounded quotient over whole binades
// (normal binades all behave alike, being exact scalings of one another, as
// long as no step leaves the normal range). Below 2^-120 the residual nears
// the subnormal range, and an infinite or NaN a would make r = inf - inf: both
// take the IEEE division instead.
__device__ __forceinline__ float div6_rn(float a) {
    if (!(a >= 0x1p-120f && a <= 0x1.fffffep127f)) return __fdiv_rn(a, 6.0f);
    const float y = 0x1.555556p-3f;
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-6.0f, q0, a);
    return __fmaf_rn(r, y, q0);
}

// Max |x| of 16 BF16 values held as 8 words, and whether any of them is +-0,
// with the packed BF16 magnitude max/min (max/min.xorsign.abs.bf16x2: the
// magnitude of the result is max/min(|a|, |b|); its sign is discarded here).
__device__ __forceinline__ float amax_bf16x16(const uint32_t w[8], bool& any_zero) {
    uint32_t mx = w[0], mn = w[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(mx) : "r"(w[i]));
        asm("min.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(mn) : "r"(w[i]));
    }
    mx &= 0x7FFF7FFFu;
    mn &= 0x7FFF7FFFu;
    any_zero = (mn & 0xFFFFu) == 0u || (mn >> 16) == 0u;
    return __uint_as_float(max(mx & 0xFFFFu, mx >> 16) << 16);
}

// Max |v| of 16 FP32 values, and whether any of them is +-0.
__device__ __forceinline__ float amax_f32x16(const float v[16], bool& any_zero) {
    float mx = 0.0f, mn = fabsf(v[0]);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        mx = fmaxf(mx, fabsf(v[i]));
        mn = fminf(mn, fabsf(v[i]));
    }
    any_zero = mn == 0.0f;
    return mx;
}

// Number of zero-magnitude codes among the 16 nibbles of two code words: a
// magnitude m <= 7 plus 7 reaches bit 3 of its nibble iff m != 0 (no carry
// leaves the nibble).
__device__ __forceinline__ uint32_t zero_mag_count16(uint32_t lo, uint32_t hi) {
    const uint32_t na = ((lo & 0x77777777u) + 0x77777777u) & 0x88888888u;
    const uint32_t nb = ((hi & 0x77777777u) + 0x77777777u) & 0x88888888u;
    return 16u - (uint32_t)__popc(na | (nb >> 1));
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of the multiply-xor bijection on a 4 x 32-bit counter with
// the 2 x 32-bit key bumped by the Weyl constants between rounds.
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u, kPhiloxW1 = 0xBB67AE85u;  // Weyl key increments

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        // one 32 x 32 -> 64-bit multiply gives both halves of each product
        unsigned long long p0, p1;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(0xD2511F53u));
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(0xCD9E8D57u));
        const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Random bits for stochastic rounding: one Philox(counter = (lo32(e >> 3),
// hi32(e >> 3), tensor_id, lo32(step)), key = seed) call serves the eight
// operand elements e >> 3 (e the row-major linear index of the quantized
// operand); its words are laid out for e2m1_sr_x16. sr_block_bits returns the
// two calls c0, c0 + 1 of one 16-element block (c0 = e0 >> 3 of its first
// element, even, so both counters share hi32(c0)). Their first round multiplies
// the same third counter word (tensor_id) and their second round the same first
// word, so those two products are formed once per block; every other step is
// the plain round.
__device__ __forceinline__ void sr_block_bits(uint64_t c0, uint32_t tensor_id, uint32_t step_lo,
                                              const uint32_t (&rk)[20], uint4 r[2]) {
    unsigned long long p;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(tensor_id), "r"(0xCD9E8D57u));
    const uint32_t x1 = (uint32_t)(p >> 32) ^ (uint32_t)(c0 >> 32) ^ rk[0];  // word 0 after the first Philox round
    const uint32_t y1k = (uint32_t)p ^ rk[2];                                // word 1 after it, with the next key folded in
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(x1), "r"(0xD2511F53u));
    const uint32_t z2k = (uint32_t)(p >> 32) ^ rk[3], w2 = (uint32_t)p;    // second-round parts from word 0
    const uint32_t sk = step_lo ^ rk[1];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        unsigned long long p0, p1;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"((uint32_t)c0 + (uint32_t)i), "r"(0xD2511F53u));
        const uint32_t z1 = (uint32_t)(p0 >> 32) ^ sk, w1 = (uint32_t)p0;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(z1), "r"(0xCD9E8D57u));
        uint4 c = make_uint4((uint32_t)(p1 >> 32) ^ y1k, (uint32_t)p1, z2k ^ w1, w2);
#pragma unroll
        for (int round = 2; round < 10; ++round) {
            asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(0xD2511F53u));
            asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(0xCD9E8D57u));
            c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk[2 * round], (uint32_t)p1,
                           (uint32_t)(p0 >> 32) ^ c.w ^ rk[2 * round + 1], (uint32_t)p0);
        }
        r[i] = c;
    }
}

// ---------------------------------------------------------------------------
// Packed FP32 pairs: two independent lanes per 64-bit register, each operation
// one IEEE binary32 round-to-nearest-even per lane (add/sub/mul.rn.f32x2).
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f2 r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Number of the N values with |x| > 6 before rounding, i.e. that saturate to
// +-6. RN(|x| * 2^100 - 6 * 2^100) from one fused multiply-add carries the sign
// of |x| - 6 (zero only for |x| == 6) and, when positive, is at least
// ulp(6) * 2^100 > 1 (+inf if it overflows), so clamped to [0, 1] it is
// exactly 1 for a saturating value and 0 otherwise; N such terms sum exactly in
// FP32. One FMA-pipe instruction per value and a packed adder tree, in place of
// a compare and an integer add per value.
template <int N>
__device__ __forceinline__ uint32_t e2m1_saturating_count(const float* x) {
    static_assert(N == 16 || N == 32, "16 or 32 values");
    f2 a[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i)
        a[i] = f2_pack(__saturatef(__fmaf_rn(fabsf(x[2 * i]), 0x1p100f, -0x1.8p102f)),
                       __saturatef(__fmaf_rn(fabsf(x[2 * i + 1]), 0x1p100f, -0x1.8p102f)));
#pragma unroll
    for (int w = N / 4; w >= 1; w /= 2)
#pragma unroll
        for (int i = 0; i < w; ++i) a[i] = f2_add(a[i], a[i + w]);
    float lo, hi;
    f2_unpack(a[0], lo, hi);
    return (uint32_t)__fadd_rn(lo, hi);
}

// x[i] = RN(v[i] * m) for 16 values, two per instruction.
__device__ __forceinline__ void scale16(const float v[16], float m, float x[16]) {
    const f2 mm = f2_pack(m, m);
#pragma unroll
    for (int i = 0; i < 16; i += 2) f2_unpack(f2_mul(f2_pack(v[i], v[i + 1]), mm), x[i], x[i + 1]);
}

// Unnormalised, unsigned 16-point Walsh-Hadamard butterfly in Sylvester order
// (the H_16 part of the RHT, App. C) on two independent vectors held in the two
// lanes of v[16]: stages of half-width 1, 2, 4, 8, each a[i] + a[i+h] and
// a[i] - a[i+h] rounded to nearest, exactly the per-lane steps of rht16.
__device__ __forceinline__ void wht16x2(f2 v[16]) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            const f2 a = v[i], b = v[i + h];
            v[i] = f2_add(a, b);
            v[i + h] = f2_sub(a, b);
        }
    }
}

// Sign nibble masks of the RHT sign vector: bit 3 of nibble i (i < 8) of lo, and
// of nibble i - 8 of hi, is bit i of signs.
__device__ __forceinline__ void rht_sign_masks(uint32_t signs, uint32_t& lo, uint32_t& hi) {
    lo = 0u;
    hi = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        lo |= ((signs >> i) & 1u) << (4 * i + 3);
        hi |= ((signs >> (i + 8)) & 1u) << (4 * i + 3);
    }
}

// Sign vector of the random Hadamard transform (section 4.2: one vector shared
// by every layer for the whole run): bit i of word 0 of Philox(counter =
// (0, 0, 0xFFFFFFFF, 0xFFFFFFFF), key = seed); a set bit negates row i.
__device__ __forceinline__ uint32_t rht_sign_word(uint32_t key0, uint32_t key1) {
    return philox4x32_10(make_uint4(0u, 0u, 0xFFFFFFFFu, 0xFFFFFFFFu), key0, key1).x & 0xFFFFu;
}

// ---------------------------------------------------------------------------
// Tensor scale ("Pretraining LLMs with NVFP4", App. B.1-B.2): s_enc,G maps the
// largest block decode scale amax / 6 onto the target T: s_enc,G = 6 T / amax.
// amax == 0 gives 1; a non-finite quotient gives FLT_MAX. s_dec,G = 1 / s_enc,G.
__device__ __forceinline__ float global_encode_scale(float amax, float target_T) {
    if (amax == 0.0f) return 1.0f;
    float s = __fdiv_rn(__fmul_rn(6.0f, target_T), amax);
    if (!(fabsf(s) <= 3.40282346638528859812e+38f)) s = 3.40282346638528859812e+38f;
    return s;
}

// Byte offset of the scale of operand row r, block j in the tensor-core
// scale-factor layout: 512-byte chunks of 128 rows x 4 blocks, chunk (rt, kt)
// at 512 * (rt * nblk / 4 + kt), row r / block j of a chunk at
// 16 * (r % 32) + 4 * ((r % 128) / 32) + (j % 4).
__device__ __forceinline__ int64_t tc_scale_offset(int64_t r, int64_t j, int64_t nblk) {
    return 512 * ((r >> 7) * (nblk >> 2) + (j >> 2)) + 16 * (r & 31) + 4 * ((r & 127) >> 5) + (j & 3);
}

}  // namespace fp4bs
