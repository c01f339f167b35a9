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
// Round-to-nearest-even with saturation at 6 (App. B.3), as a sum of threshold
// tests: each midpoint between neighbours rounds toward the even index, so the
// tests at 0.25, 1.25, 2.5 and 5 are strict and those at 0.75, 1.75, 3.5 are
// inclusive. The sign bit of the code is the sign bit of v.
__device__ __forceinline__ uint32_t e2m1_rne(float v) {
    const float a = fabsf(v);
    const uint32_t m = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                       (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                       (uint32_t)(a > 5.0f);
    return m | ((__float_as_uint(v) >> 28) & 8u);
}

// Stochastic rounding (section 4.4) with a 16-bit uniform r16: |v| in
// [lo, hi) rounds up iff r16 < frac * 2^16, frac = (|v| - lo) / (hi - lo).
// The test is done exactly on the bit pattern of |v| = 2^e (1 + m):
//   |v| in [1, 6): lo is |v| truncated to one mantissa bit (code 2 + 2e + that
//     bit), hi - lo = 2^(e-1), so frac * 2^16 = (low 22 mantissa bits) / 2^6;
//   |v| in [0.5, 1): lo = 0.5 (code 1), frac * 2^16 = (23 mantissa bits) / 2^7;
//   |v| < 0.5: lo = 0 (code 0), frac * 2^16 = |v| * 2^17 (an exact scaling).
// |v| >= 6 saturates to 6.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t r16) {
    const uint32_t b = __float_as_uint(v);
    const uint32_t sign = (b >> 28) & 8u;
    const uint32_t a = b & 0x7FFFFFFFu;
    if (a >= 0x40C00000u) return 7u | sign;
    uint32_t code, up;
    if (a >= 0x3F800000u) {
        code = 2u + 2u * ((a >> 23) - 127u) + ((a >> 22) & 1u);
        up = (r16 << 6) < (a & 0x3FFFFFu) ? 1u : 0u;
    } else if (a >= 0x3F000000u) {
        code = 1u;
        up = (r16 << 7) < (a & 0x7FFFFFu) ? 1u : 0u;
    } else {
        code = 0u;
        up = (float)r16 < __fmul_rn(__uint_as_float(a), 131072.0f) ? 1u : 0u;
    }
    return (code + up) | sign;
}

// Eight FP32 values -> eight E2M1 codes (element i in nibble i) with the
// hardware conversion cvt.rn.satfinite.e2m1x2.f32, which rounds to nearest-even
// and saturates at +-6 (its first source goes to the upper nibble). The sign
// bits of the inputs are OR-ed in afterwards so that values rounding to zero
// keep their sign whatever the instruction does with negative zero.
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
    uint32_t signs = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) signs |= (__float_as_uint(v[i]) >> (28 - 4 * i)) & (8u << (4 * i));
    return out | signs;
}

// Number of zero-magnitude codes among the 8 nibbles of a code word.
__device__ __forceinline__ uint32_t zero_mag_count8(uint32_t w) {
    const uint32_t t = w & 0x77777777u;
    return 8u - (uint32_t)__popc((t | (t >> 1) | (t >> 2)) & 0x11111111u);
}

// Count of values that saturate (|v| > 6 before rounding).
__device__ __forceinline__ uint32_t e2m1_saturates(float v) { return fabsf(v) > 6.0f ? 1u : 0u; }

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
template <>
struct ScaleFmt<kFmtE4M3> {
    static constexpr float kMax = 448.0f;
    __device__ static __forceinline__ uint32_t encode(float s) { return scale_encode_m3<7, 0x7Eu>(s, kMax); }
    __device__ static __forceinline__ float decode(uint32_t c) { return scale_decode_m3<7>(c & 0x7Fu); }
};
template <>
struct ScaleFmt<kFmtUE5M3> {
    static constexpr float kMax = 114688.0f;
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

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of the multiply-xor bijection on a 4 x 32-bit counter with
// the 2 x 32-bit key bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Random bits for stochastic rounding: operand element e (row-major linear
// index of the quantized operand) uses 16-bit half (e & 1) of word
// ((e >> 1) & 3) of Philox(counter = (lo32(e >> 3), hi32(e >> 3), tensor_id,
// lo32(step)), key = seed). One call covers 8 consecutive elements; this
// returns the four words for the group g = e >> 3.
__device__ __forceinline__ uint4 sr_group_bits(uint64_t g, uint32_t tensor_id, uint32_t step_lo,
                                               uint32_t key0, uint32_t key1) {
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), tensor_id, step_lo), key0, key1);
}

__device__ __forceinline__ uint32_t sr_half(const uint4& w, int i) {  // element i of the group, 0..7
    const uint32_t word = (i >> 1) == 0 ? w.x : (i >> 1) == 1 ? w.y : (i >> 1) == 2 ? w.z : w.w;
    return (i & 1) ? (word >> 16) : (word & 0xFFFFu);
}

// Sign vector of the random Hadamard transform (section 4.2: one vector shared
// by every layer for the whole run): bit i of word 0 of Philox(counter =
// (0, 0, 0xFFFFFFFF, 0xFFFFFFFF), key = seed); a set bit negates row i.
__device__ __forceinline__ uint32_t rht_sign_word(uint32_t key0, uint32_t key1) {
    return philox4x32_10(make_uint4(0u, 0u, 0xFFFFFFFFu, 0xFFFFFFFFu), key0, key1).x & 0xFFFFu;
}

// v <- D_r * (H_16 / 4) * v ("Pretraining LLMs with NVFP4", App. C): butterfly
// stages of half-width 1, 2, 4, 8 producing the Sylvester-ordered transform,
// then the (1/sqrt 2)^4 = 1/4 normalisation, then the sign of row i.
__device__ __forceinline__ void rht16(float v[16], uint32_t signs) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            const float a = v[i], b = v[i + h];
            v[i] = __fadd_rn(a, b);
            v[i + h] = __fsub_rn(a, b);
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float q = __fmul_rn(v[i], 0.25f);
        v[i] = __uint_as_float(__float_as_uint(q) ^ (((signs >> i) & 1u) << 31));
    }
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
