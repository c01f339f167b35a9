// quantize.cu -- memory-bound quantizer kernels for sm_103a.
//
// Implements the quantization of "Pretraining Large Language Models with NVFP4"
// (arXiv 2509.25149): tensor amax and tensor scale (App. B.1), block scale
// (App. B.2), E2M1 conversion with RNE or stochastic rounding (App. B.3,
// section 4.4), the 16-point random Hadamard transform on Wgrad operands
// (section 4.2, App. C), 2D 16x16 weight scaling (section 4.3) and MXFP4 1x32
// power-of-two scales (section A3, App. B.4); plus the UE5M3 block scales and
// held-amax tensor scaling of the UE5M3 pretraining paper (arXiv 2609.02846).
//
// Data movement: coalesced 128-bit (rowwise) or 64-bit (colwise) BF16 loads;
// each thread owns whole 16-element blocks (rowwise: 16 consecutive elements;
// colwise: 16 tokens of 4 channels), so block amax, scale and rounding stay in
// registers. RNE conversion uses the hardware E2M1 convert (two values per
// instruction); event counts use bit tricks on the packed codes. Codes are
// stored as packed 64-bit nibble words; groups of four lanes whose scales are
// adjacent in the tensor-core layout merge them into one 32-bit store. Every
// kernel is a grid-stride loop over a grid of a few CTAs per SM.
#include <cstdint>

#include <cuda_bf16.h>

#include "fp4_device.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace fp4bs {

namespace {

constexpr int kThreads = 256;

struct QParams {
    const uint16_t* in;
    int64_t rows, cols;
    int64_t ld;  // input row stride in elements (>= cols, a multiple of 8)
    uint8_t* codes;
    uint8_t* scales;
    float* s_dec;
    uint8_t* codes_t;
    uint8_t* scales_t;
    float* s_dec_t;
    fp4_amax_state_t* state;
    uint64_t* counters;
    const float* partials;
    int npartials;
    int held, refresh;
    int given;    // the tensor amax is the state's (computed ahead by fp4_tensor_amax): no pass, no refresh
    int count_t;  // 16x16 with two outputs: the counters follow the transposed output
    float target_T;
    uint32_t tensor_id, step_lo, key0, key1;
    uint32_t round_key[20];  // Philox key of round r: (key0 + r W0, key1 + r W1), W the Weyl constants
    uint64_t step;
    int* status;
};

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// Input offset of unit u of a row-major rows x cols input cut into units of
// `unit` elements (per_row = cols / unit of them per row) when its rows lie ld
// elements apart: unit * u for a dense input (ld == cols, the common case, no
// division), else row * ld + column.
__device__ __forceinline__ int64_t strided_off(int64_t u, int unit, int64_t per_row, int64_t cols, int64_t ld) {
    if (ld == cols) return (int64_t)unit * u;
    return (u / per_row) * ld + (int64_t)unit * (u % per_row);
}

// Block-wide max of a non-negative float (all threads of the CTA call it).
__device__ float cta_max(float v) {
    __shared__ float red[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    __syncthreads();
    return m;
}

// Tensor scale of this call (App. B.1; held amax per the UE5M3 paper), computed
// redundantly by every CTA from the amax partials or the held state. CTA 0
// publishes s_dec,G and, on refresh steps, the new held state. Returns false
// (uniformly over the CTA) when a given amax is not valid (the status word then
// holds FP4_ERR_STATE and nothing is written).
__device__ bool cta_tensor_scale(const QParams& q, float& s_enc, float& s_dec) {
    __shared__ float s_amax;
    __shared__ int s_valid;
    // held scaling refreshes on refresh steps and whenever the held state is
    // not valid yet (the amax pass then ran; see the amax kernels' skip rule)
    if (threadIdx.x == 0) {
        s_valid = (q.held && !q.refresh) ? q.state->valid : 0;
        s_amax = s_valid ? q.state->amax_held : 0.0f;
    }
    __syncthreads();
    if (q.given && s_valid == 0) {
        if (threadIdx.x == 0) record_status(q.status, kStatusState);
        return false;
    }
    const bool use_held = s_valid != 0;
    if (!use_held) {
        float m = 0.0f;
        for (int i = threadIdx.x; i < q.npartials; i += blockDim.x) m = fmaxf(m, q.partials[i]);
        m = cta_max(m);
        if (threadIdx.x == 0) s_amax = m;
        __syncthreads();
    }
    const float amax = s_amax;
    s_enc = global_encode_scale(amax, q.target_T);
    s_dec = __fdiv_rn(1.0f, s_enc);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (q.s_dec) *q.s_dec = s_dec;
        if (q.s_dec_t) *q.s_dec_t = s_dec;
        if (q.held && !use_held) {
            q.state->amax_held = amax;
            q.state->valid = 1;
            q.state->last_refresh_step = q.step;
        }
    }
    return true;
}

// Sum the four per-thread event counts over the warp and add them to the
// caller's 64-bit counters.
__device__ __forceinline__ void flush_counters(uint64_t* counters, uint32_t c0, uint32_t c1, uint32_t c2,
                                               uint32_t c3) {
    if (counters == nullptr) return;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        c0 += __shfl_xor_sync(0xFFFFFFFFu, c0, o);
        c1 += __shfl_xor_sync(0xFFFFFFFFu, c1, o);
        c2 += __shfl_xor_sync(0xFFFFFFFFu, c2, o);
        c3 += __shfl_xor_sync(0xFFFFFFFFu, c3, o);
    }
    if ((threadIdx.x & 31) == 0) {
        if (c0) atomicAdd((unsigned long long*)&counters[0], (unsigned long long)c0);
        if (c1) atomicAdd((unsigned long long*)&counters[1], (unsigned long long)c1);
        if (c2) atomicAdd((unsigned long long*)&counters[2], (unsigned long long)c2);
        if (c3) atomicAdd((unsigned long long*)&counters[3], (unsigned long long)c3);
    }
}

struct Counts {
    uint32_t esat = 0, eunder = 0, ssat = 0, sunder = 0;
};

// (row, col) of tile t in a row-major grid with `cols` tiles per row. at()
// divides once; advance() adds another cursor's offset with one carry (both
// columns are below `cols`), so a grid-stride loop over tiles, whose threads
// each convert only a few dozen elements per tile, needs no 64-bit division.
struct TileCursor {
    int64_t row, col;
    __device__ __forceinline__ static TileCursor at(int64_t t, int64_t cols) { return TileCursor{t / cols, t % cols}; }
    __device__ __forceinline__ void advance(const TileCursor& d, int64_t cols) {
        row += d.row;
        col += d.col;
        if (col >= cols) {
            col -= cols;
            ++row;
        }
    }
};

// Sign bits of eight values placed at bit 3 of nibble i (the code's sign).
__device__ __forceinline__ uint32_t sign_nibbles8(const float* v) {
    uint32_t s = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) s |= (__float_as_uint(v[i]) >> (28 - 4 * i)) & (8u << (4 * i));
    return s;
}

// Local encode scale per block-scale code (App. B.2-B.3), one table per
// operand and CTA: s_enc,L(c) = RN(1 / RN(decode(c) * s_dec,G)) depends only on
// the code c once the tensor scale is known. Unused codes hold 0.
template <int FMT>
__device__ __forceinline__ void fill_enc_table(float* tab, float s_dec) {
    using F = ScaleFmt<FMT>;
    for (int c = threadIdx.x; c < 256; c += blockDim.x)
        tab[c] = (c == 0 || (uint32_t)c > F::kMaxCode) ? 0.0f : __frcp_rn(__fmul_rn(F::decode((uint32_t)c), s_dec));
}

// Quantize one 1x16 block (App. B.2-B.3): scale in the block format (RNE,
// satfinite), local encode scale, E2M1 codes packed into two 32-bit words
// (element i in nibble i). The block's values are w_i = sign_i * pre * v[i]:
// plain blocks (RHT false) take v as is; RHT blocks pass the raw Hadamard
// butterfly in v with pre = 1/4 and the sign vector as nibble masks (bit 3 of
// nibble i), so the normalisation and the signs fold into the element scale
// and the code sign bits. Folding is exact: pre * v[i] is exact, and so is
// pre * s_enc,L unless s_enc,L < 2^-124, where the two products are taken
// apart. vmax is max |v[i]|, any_zero whether some v[i] is +-0; enc_tab holds
// s_enc,L per scale code (fill_enc_table). `c0` = (index of element 0) / 8, the
// first of the block's two SR counters. DIRECT: no table; s_enc,L is formed
// from `s_dec` for this block alone (the expression fill_enc_table uses).
// Event counts: scale saturation and underflow; element saturation, counted
// per element only when the scaled block max exceeds 6 (rounding is monotone,
// so otherwise no element can); element underflow = zero-magnitude codes minus
// zero inputs.
template <int FMT, bool SR, bool RHT, bool DIRECT = false>
__device__ __forceinline__ uint32_t quantize_block16(const float v[16], float vmax, bool any_zero,
                                                     const float* enc_tab, float s_enc, uint64_t c0, const QParams& q,
                                                     uint32_t smask_lo, uint32_t smask_hi, uint32_t& lo, uint32_t& hi,
                                                     Counts& cnt, float s_dec = 0.0f) {
    using F = ScaleFmt<FMT>;
    const float amax_b = RHT ? __fmul_rn(vmax, 0.25f) : vmax;
    const float s = __fmul_rn(div6_rn(amax_b), s_enc);
    const uint32_t sc = F::encode(s);
    cnt.ssat += s > F::kMax ? 1u : 0u;
    uint32_t nzero = 0u;
    if (any_zero) {
#pragma unroll
        for (int i = 0; i < 16; ++i) nzero += v[i] == 0.0f ? 1u : 0u;
    }
    if (sc == 0u) {
        cnt.sunder += amax_b > 0.0f ? 1u : 0u;
        cnt.eunder += 16u - nzero;
        lo = sign_nibbles8(v) ^ smask_lo;
        hi = sign_nibbles8(v + 8) ^ smask_hi;
        return 0u;
    }
    const float enc_l = DIRECT ? __frcp_rn(__fmul_rn(F::decode(sc), s_dec)) : enc_tab[sc];
    float x[16];
    float xmax;
    if (!RHT || enc_l >= 0x1p-124f) {
        const float m = RHT ? __fmul_rn(enc_l, 0.25f) : enc_l;
        scale16(v, m, x);
        xmax = __fmul_rn(vmax, m);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = __fmul_rn(__fmul_rn(v[i], 0.25f), enc_l);
        xmax = __fmul_rn(amax_b, enc_l);
    }
    if (xmax > 6.0f) cnt.esat += e2m1_saturating_count<16>(x);
    if (SR) {
        uint4 r[2];
        sr_block_bits(c0, q.tensor_id, q.step_lo, q.round_key, r);
        e2m1_sr_x16(x, r, lo, hi);
    } else {
        lo = e2m1_rne_x8(x);
        hi = e2m1_rne_x8(x + 8);
    }
    if (RHT) {
        lo ^= smask_lo;
        hi ^= smask_hi;
    }
    cnt.eunder += zero_mag_count16(lo, hi) - nzero;
    return sc;
}

// ----------------------------------------------------------------------------
// K1: tensor amax partials (App. B.1: one extra pass over the tensor).

// Plain amax over all elements: max of |bf16| as 16-bit integers (BF16 bit
// patterns of non-negative values order like their values). Each thread issues
// eight 16-byte loads before reducing them, so a resident CTA keeps 32 KB of
// reads in flight.
constexpr int kAmaxVec = 8;

// Held scaling on a non-refresh step: the pass is only needed while the held
// state is not valid yet; with a valid state every CTA returns at once.
__device__ __forceinline__ bool amax_pass_skipped(const fp4_amax_state_t* a, const fp4_amax_state_t* b) {
    return a != nullptr && a->valid != 0 && (b == nullptr || b->valid != 0);
}

__global__ void __launch_bounds__(kThreads, 4) amax_plain_kernel(const uint4* __restrict__ in, int64_t n_vec,
                                                                 int64_t row_vec, int64_t ld_vec,
                                                                 float* __restrict__ partials,
                                                                 const fp4_amax_state_t* skip_if_valid) {
    pdl_begin();
    if (amax_pass_skipped(skip_if_valid, nullptr)) return;
    uint32_t m = 0u;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kAmaxVec - 1) * stride < n_vec; i += kAmaxVec * stride) {
        uint4 v[kAmaxVec];
#pragma unroll
        for (int k = 0; k < kAmaxVec; ++k) v[k] = __ldg(in + strided_off(i + k * stride, 1, row_vec, row_vec, ld_vec));
#pragma unroll
        for (int k = 0; k < kAmaxVec; ++k)
            m = __vmaxu2(m, __vmaxu2(__vmaxu2(v[k].x & 0x7FFF7FFFu, v[k].y & 0x7FFF7FFFu),
                                     __vmaxu2(v[k].z & 0x7FFF7FFFu, v[k].w & 0x7FFF7FFFu)));
    }
    for (; i < n_vec; i += stride) {
        const uint4 a = __ldg(in + strided_off(i, 1, row_vec, row_vec, ld_vec));
        m = __vmaxu2(m, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                 __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
    }
    const uint32_t mm = max(m & 0xFFFFu, m >> 16);
    const float f = cta_max(__uint_as_float(mm << 16));
    if (threadIdx.x == 0) partials[blockIdx.x] = f;
}

// amax in the rotated space (App. C): each thread transforms 16 tokens of 4
// channels (sixteen 64-bit loads, two channels per packed butterfly) and keeps
// the max magnitude. The RHT's signs do not change magnitudes and its 1/4 is an
// exact scaling, so the max is taken over the raw butterfly and scaled once.
__global__ void __launch_bounds__(kThreads) amax_rht_cols_kernel(const uint16_t* __restrict__ in, int64_t T,
                                                                 int64_t C, int64_t ld, float* __restrict__ partials,
                                                                 const fp4_amax_state_t* skip_if_valid) {
    pdl_begin();
    if (amax_pass_skipped(skip_if_valid, nullptr)) return;
    const int64_t ug = C / 4, uj = T / 16, units = ug * uj;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float m = 0.0f;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int64_t g = u % ug, j = u / ug;
        uint2 x[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) x[t] = __ldg(reinterpret_cast<const uint2*>(in + (16 * j + t) * ld + 4 * g));
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            f2 pv[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const uint32_t w = pr ? x[t].y : x[t].x;
                pv[t] = f2_pack(bf16_lo(w), bf16_hi(w));
            }
            wht16x2(pv);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                float a, b;
                f2_unpack(pv[t], a, b);
                m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
            }
        }
    }
    m = cta_max(__fmul_rn(m, 0.25f));
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// ----------------------------------------------------------------------------
// K2: rowwise 1x16 quantizer (activations X for Fprop, gradients dY for Dgrad).
// Flat block index b covers rows x cols/16; block b's elements are the 16
// consecutive inputs at 16 b, its codes the 8 bytes at 8 b. A warp takes 64
// consecutive blocks per step (lane l: blocks base + l and base + 32 + l), with
// all four 16-byte loads issued before either block is converted.
template <int FMT, bool SR, bool TCL>
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(QParams q) {
    pdl_begin();
    __shared__ float enc_tab[256];
    float s_enc, s_dec;
    if (!cta_tensor_scale(q, s_enc, s_dec)) return;
    fill_enc_table<FMT>(enc_tab, s_dec);
    __syncthreads();
    const int64_t nb_row = q.cols / 16;
    const int64_t nblk = q.rows * nb_row;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    Counts cnt;
    for (int64_t base = warp * 64; base < nblk; base += nwarps * 64) {
        uint4 in[2][2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t b = base + 32 * u + lane;
            if (b < nblk) {
                const int64_t o = strided_off(b, 16, nb_row, q.cols, q.ld);
                in[u][0] = ldg16(q.in + o);
                in[u][1] = ldg16(q.in + o + 8);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t b = base + 32 * u + lane;
            const bool active = b < nblk;
            uint32_t sc = 0u;
            if (active) {
                const uint4 a = in[u][0], c = in[u][1];
                const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
                bool any_zero;
                const float vmax = amax_bf16x16(w, any_zero);
                float v[16];
                unpack16(a, c, v);
                uint32_t lo, hi;
                sc = quantize_block16<FMT, SR, false>(v, vmax, any_zero, enc_tab, s_enc, (uint64_t)(2 * b), q, 0u, 0u,
                                                      lo, hi, cnt);
                *reinterpret_cast<uint2*>(q.codes + 8 * b) = make_uint2(lo, hi);
            }
            if (TCL) {
                // lanes 4k..4k+3 hold the four adjacent scale bytes of one row
                uint32_t w = sc << (8 * (lane & 3));
                w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);
                w |= __shfl_xor_sync(0xFFFFFFFFu, w, 2);
                if (active && (lane & 3) == 0) {
                    const int64_t r = b / nb_row, j = b % nb_row;
                    *reinterpret_cast<uint32_t*>(q.scales + tc_scale_offset(r, j, nb_row)) = w;
                }
            } else if (active) {
                q.scales[b] = (uint8_t)sc;
            }
        }
    }
    flush_counters(q.counters, cnt.esat, cnt.eunder, cnt.ssat, cnt.sunder);
}

// ----------------------------------------------------------------------------
// K2r: rowwise 1x16 quantizer with one tensor scale per operand row (App. B.1:
// the global scale at the granularity of a row, so that current scaling needs
// no separate amax pass). A warp owns whole rows: it takes the row's amax
// (max |bf16| as 16-bit integers, eight 16-byte loads in flight per lane),
// forms s_enc,G(r) and s_dec,G(r) exactly as the tensor-wide scale is formed,
// then converts the row's blocks as the rowwise kernel does, re-reading the row
// from cache (one pass over memory). With no table per row, each block forms
// its s_enc,L directly.
template <int FMT, bool SR, bool TCL>
__global__ void __launch_bounds__(kThreads) quantize_rows_rowscale_kernel(QParams q) {
    pdl_begin();
    const int64_t nb_row = q.cols / 16, n_vec = q.cols / 8;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    Counts cnt;
    for (int64_t r = warp; r < q.rows; r += nwarps) {
        const uint4* row = reinterpret_cast<const uint4*>(q.in + r * q.ld);
        uint32_t m = 0u;
        int64_t i = lane;
        for (; i + 32 * (kAmaxVec - 1) < n_vec; i += 32 * kAmaxVec) {
            uint4 v[kAmaxVec];
#pragma unroll
            for (int k = 0; k < kAmaxVec; ++k) v[k] = __ldg(row + i + 32 * k);
#pragma unroll
            for (int k = 0; k < kAmaxVec; ++k)
                m = __vmaxu2(m, __vmaxu2(__vmaxu2(v[k].x & 0x7FFF7FFFu, v[k].y & 0x7FFF7FFFu),
                                         __vmaxu2(v[k].z & 0x7FFF7FFFu, v[k].w & 0x7FFF7FFFu)));
        }
        for (; i < n_vec; i += 32) {
            const uint4 a = __ldg(row + i);
            m = __vmaxu2(m, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                     __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
        }
        m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float amax = __uint_as_float(m << 16);
        const float s_enc = global_encode_scale(amax, q.target_T);
        const float s_dec = __fdiv_rn(1.0f, s_enc);
        if (lane == 0) q.s_dec[r] = s_dec;
        for (int64_t base = 0; base < nb_row; base += 64) {
            uint4 in[2][2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t j = base + 32 * u + lane;
                if (j < nb_row) {
                    in[u][0] = ldg16(q.in + r * q.ld + 16 * j);
                    in[u][1] = ldg16(q.in + r * q.ld + 16 * j + 8);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t j = base + 32 * u + lane;
                const int64_t b = r * nb_row + j;  // flat block index
                const bool active = j < nb_row;
                uint32_t sc = 0u;
                if (active) {
                    const uint4 a = in[u][0], c = in[u][1];
                    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
                    bool any_zero;
                    const float vmax = amax_bf16x16(w, any_zero);
                    float v[16];
                    unpack16(a, c, v);
                    uint32_t lo, hi;
                    sc = quantize_block16<FMT, SR, false, true>(v, vmax, any_zero, nullptr, s_enc, (uint64_t)(2 * b), q,
                                                                0u, 0u, lo, hi, cnt, s_dec);
                    *reinterpret_cast<uint2*>(q.codes + 8 * b) = make_uint2(lo, hi);
                }
                if (TCL) {
                    // lanes 4k..4k+3 hold the four adjacent scale bytes of this row
                    uint32_t w = sc << (8 * (lane & 3));
                    w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);
                    w |= __shfl_xor_sync(0xFFFFFFFFu, w, 2);
                    if (active && (lane & 3) == 0)
                        *reinterpret_cast<uint32_t*>(q.scales + tc_scale_offset(r, j, nb_row)) = w;
                } else if (active) {
                    q.scales[b] = (uint8_t)sc;
                }
            }
        }
    }
    flush_counters(q.counters, cnt.esat, cnt.eunder, cnt.ssat, cnt.sunder);
}

// ----------------------------------------------------------------------------
// K3: colwise 1x16 quantizer with optional fused RHT16 (Wgrad operands X^T and
// dY^T, section 4.2-4.3). The operand is the input's transpose: operand row c
// (a channel) holds tokens along the dot dimension. Each thread owns 16 tokens
// of 4 channels (sixteen 64-bit loads); a warp covers 4 token tiles x 8 channel
// groups (64 tokens x 32 channels), lane = 4 * channel_group + tile, so the
// four lanes of a channel write 32 contiguous code bytes and four adjacent
// scale bytes.
template <int FMT, bool SR, bool RHT, bool TCL>
__global__ void __launch_bounds__(kThreads, 2) quantize_cols_kernel(QParams q) {
    pdl_begin();
    __shared__ float enc_tab[256];
    float s_enc, s_dec;
    if (!cta_tensor_scale(q, s_enc, s_dec)) return;
    fill_enc_table<FMT>(enc_tab, s_dec);
    __syncthreads();
    const int64_t T = q.rows, C = q.cols;
    const int64_t ug = C / 4, uj = T / 16;
    const int64_t wg_count = (ug + 7) / 8, wj_count = (uj + 3) / 4;
    const int64_t wunits = wg_count * wj_count;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint32_t signs = RHT ? rht_sign_word(q.key0, q.key1) : 0u;
    uint32_t smask_lo = 0u, smask_hi = 0u;
    if (RHT) rht_sign_masks(signs, smask_lo, smask_hi);
    Counts cnt;
    for (int64_t wu = warp; wu < wunits; wu += nwarps) {
        const int64_t g = (wu % wg_count) * 8 + (lane >> 2);
        const int64_t j = (wu / wg_count) * 4 + (lane & 3);
        const bool active = g < ug && j < uj;
        uint2 x[16];
#pragma unroll
        for (int t = 0; t < 16; ++t)
            x[t] = active ? __ldg(reinterpret_cast<const uint2*>(q.in + (16 * j + t) * q.ld + 4 * g)) : make_uint2(0, 0);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
            // channels 4g + 2pr (low lane) and 4g + 2pr + 1 (high lane)
            f2 pv[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const uint32_t w = pr ? x[t].y : x[t].x;
                pv[t] = f2_pack(bf16_lo(w), bf16_hi(w));
            }
            if (RHT) wht16x2(pv);
#pragma unroll
            for (int ln = 0; ln < 2; ++ln) {
                float v[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float a, b;
                    f2_unpack(pv[t], a, b);
                    v[t] = ln ? b : a;
                }
                const int64_t c = 4 * g + 2 * pr + ln;
                uint32_t lo = 0u, hi = 0u, sc = 0u;
                if (active) {
                    bool any_zero;
                    const float vmax = amax_f32x16(v, any_zero);
                    sc = quantize_block16<FMT, SR, RHT>(v, vmax, any_zero, enc_tab, s_enc,
                                                        (uint64_t)((c * T + 16 * j) >> 3), q, smask_lo, smask_hi, lo,
                                                        hi, cnt);
                    *reinterpret_cast<uint2*>(q.codes + c * (T / 2) + 8 * j) = make_uint2(lo, hi);
                }
                if (TCL) {
                    uint32_t w = sc << (8 * (lane & 3));
                    w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);
                    w |= __shfl_xor_sync(0xFFFFFFFFu, w, 2);
                    if (active && (lane & 3) == 0)
                        *reinterpret_cast<uint32_t*>(q.scales + tc_scale_offset(c, j, uj)) = w;
                } else if (active) {
                    q.scales[c * uj + j] = (uint8_t)sc;
                }
            }
        }
    }
    flush_counters(q.counters, cnt.esat, cnt.eunder, cnt.ssat, cnt.sunder);
}

// ----------------------------------------------------------------------------
// K4: 2D 16x16 weight quantizer (section 4.3). A half-warp owns one 16x16 tile
// of W [N x K]: lane i loads row i, the tile amax is a 16-lane shuffle max, and
// each lane converts its row. The transposed operand W^T [K x N] reuses the same
// codes: lane i gathers column i from the other lanes' packed rows, so
// quantize(W)^T == quantize(W^T) holds by construction. Either output may be
// omitted (null codes pointer).
template <int FMT, bool TCL_W, bool TCL_WT>
__global__ void __launch_bounds__(kThreads) quantize_2d_kernel(QParams q) {
    pdl_begin();
    float s_enc, s_dec;
    if (!cta_tensor_scale(q, s_enc, s_dec)) return;
    using F = ScaleFmt<FMT>;
    const int64_t N = q.rows, K = q.cols, tn_count = N / 16, tk_count = K / 16;
    const int64_t tiles = tn_count * tk_count;
    const int lane = threadIdx.x & 31, i = lane & 15;
    const int64_t hw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
    const int64_t nhw = ((int64_t)gridDim.x * blockDim.x) >> 4;
    Counts cnt;
    // loop bound rounded to whole warps so every shuffle has its full warp
    for (int64_t base = hw & ~(int64_t)1; base < tiles; base += nhw) {
        const int64_t t = base + (lane >> 4);
        const bool active = t < tiles;
        const int64_t tk = active ? t % tk_count : 0, tn = active ? t / tk_count : 0;
        const int64_t n = 16 * tn + i, k0 = 16 * tk;
        float v[16];
        if (active) {
            const uint4 a = ldg16(q.in + n * q.ld + k0), c = ldg16(q.in + n * q.ld + k0 + 8);
            unpack16(a, c, v);
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.0f;
        }
        float amax_t = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) amax_t = fmaxf(amax_t, fabsf(v[e]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax_t = fmaxf(amax_t, __shfl_xor_sync(0xFFFFFFFFu, amax_t, o));
        const float s = __fmul_rn(__fdiv_rn(amax_t, 6.0f), s_enc);
        const uint32_t sc = F::encode(s);
        const bool count_tile = active && i == 0;
        if (count_tile) {
            cnt.ssat += s > F::kMax ? 1u : 0u;
            cnt.sunder += (sc == 0u && amax_t > 0.0f) ? 1u : 0u;
        }
        uint32_t lo = 0u, hi = 0u;
        uint32_t nzero = 0u;
#pragma unroll
        for (int e = 0; e < 16; ++e) nzero += (__float_as_uint(v[e]) << 1) == 0u ? 1u : 0u;
        if (sc == 0u) {
            lo = sign_nibbles8(v);
            hi = sign_nibbles8(v + 8);
            if (active) cnt.eunder += 16u - nzero;
        } else {
            const float s_enc_l = __frcp_rn(__fmul_rn(F::decode(sc), s_dec));
            float x[16];
            scale16(v, s_enc_l, x);
            lo = e2m1_rne_x8(x);
            hi = e2m1_rne_x8(x + 8);
            if (active) {
                if (__fmul_rn(amax_t, s_enc_l) > 6.0f) cnt.esat += e2m1_saturating_count<16>(x);
                cnt.eunder += zero_mag_count8(lo) + zero_mag_count8(hi) - nzero;
            }
        }
        if (q.codes != nullptr && active) {
            *reinterpret_cast<uint2*>(q.codes + n * (K / 2) + k0 / 2) = make_uint2(lo, hi);
            q.scales[TCL_W ? tc_scale_offset(n, tk, tk_count) : n * tk_count + tk] = (uint8_t)sc;
        }
        if (q.codes_t != nullptr) {
            // column i of the tile: nibble i of every row rr
            uint32_t tlo = 0u, thi = 0u;
            const int src_base = lane & 16;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const uint32_t wlo = __shfl_sync(0xFFFFFFFFu, lo, src_base + rr);
                const uint32_t whi = __shfl_sync(0xFFFFFFFFu, hi, src_base + rr);
                const uint32_t nib = (i < 8 ? (wlo >> (4 * i)) : (whi >> (4 * (i - 8)))) & 0xFu;
                if (rr < 8) tlo |= nib << (4 * rr);
                else thi |= nib << (4 * (rr - 8));
            }
            if (active) {
                const int64_t kr = k0 + i;
                *reinterpret_cast<uint2*>(q.codes_t + kr * (N / 2) + 8 * tn) = make_uint2(tlo, thi);
                q.scales_t[TCL_WT ? tc_scale_offset(kr, tn, tn_count) : kr * tn_count + tn] = (uint8_t)sc;
            }
        }
    }
    flush_counters(q.counters, cnt.esat, cnt.eunder, cnt.ssat, cnt.sunder);
}

// K4b: the same 2D quantizer for N % 64 == 0 and K % 128 == 0, fed by TMA. A CTA
// walks 64 x 128 tiles of W (kept kTileStages deep in a shared ring, each tile
// two 64 x 64 boxes with the 128-byte swizzle); a group of 8 lanes owns one
// 16 x 16 block: lane l converts rows l and l + 8 of W (the block amax is a
// 3-step shuffle max over the group) and columns 2l and 2l + 1 as rows of W^T,
// converting the same values with the same scale, so quantize(W)^T ==
// quantize(W^T) holds by construction. Counters follow W.
constexpr int kTileStages = 3;
constexpr int k2dTileBytes = 64 * 128 * 2;
constexpr int k2dSmemBytes = kTileStages * k2dTileBytes + 1024;

// Byte offset of element (r, c) of a staged 64 x 128 BF16 tile: half c / 64,
// 128-byte row r, 16-byte chunk ((c % 64) / 8) XOR (r % 8).
__device__ __forceinline__ uint32_t tile2d_offset(int r, int c) {
    return (uint32_t)((c >> 6) * 8192 + r * 128 + (((((c & 63) >> 3) ^ (r & 7))) << 4) + ((c & 7) << 1));
}

template <int FMT, bool SR, bool TCL_W, bool TCL_WT>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_2d_tile_kernel(const __grid_constant__ CUtensorMap tmap_w, QParams q) {
    pdl_begin();
    extern __shared__ uint8_t tile2d_smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tile2d_smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ float tab[256];
    __shared__ __align__(8) uint64_t full_bar[kTileStages];
    float s_enc, s_dec;
    if (!cta_tensor_scale(q, s_enc, s_dec)) return;
    fill_enc_table<FMT>(tab, s_dec);
    if (threadIdx.x == 0) {
        for (int k = 0; k < kTileStages; ++k) tc::mbar_init(tc::smem_u32(&full_bar[k]), 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    using F = ScaleFmt<FMT>;
    const int64_t N = q.rows, K = q.cols, tiles_k = K / 128, ntiles = (N / 64) * tiles_k;
    const int64_t tk_count = K / 16, tn_count = N / 16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, l = lane & 7;
    const int bn = warp >> 1, bk = 4 * (warp & 1) + (lane >> 3);  // this group's block in the tile
    auto issue = [&](int64_t t, int s) {
        const int64_t n0 = (t / tiles_k) * 64, k0 = (t % tiles_k) * 128;
        const uint32_t bar = tc::smem_u32(&full_bar[s]);
        tc::mbar_arrive_expect_tx(bar, k2dTileBytes);
        tc::tma_load_2d(tc::smem_u32(ring + s * k2dTileBytes), &tmap_w, (int32_t)k0, (int32_t)n0, bar);
        tc::tma_load_2d(tc::smem_u32(ring + s * k2dTileBytes + 8192), &tmap_w, (int32_t)(k0 + 64), (int32_t)n0, bar);
    };
    if (tid == 0) {
        tc::prefetch_tmap(&tmap_w);
        for (int k = 0; k < kTileStages; ++k) {
            const int64_t tk = blockIdx.x + (int64_t)k * gridDim.x;
            if (tk < ntiles) issue(tk, k);
        }
    }
    Counts cnt;
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = (int)(it % kTileStages);
        const bool ok = tc::mbar_wait(tc::smem_u32(&full_bar[s]), (it / kTileStages) & 1u, q.status);
        const uint8_t* tile = ring + s * k2dTileBytes;
        const int64_t n0 = (t / tiles_k) * 64, k0 = (t % tiles_k) * 128;
        // ---- W rows 16 bn + l and 16 bn + l + 8 of the block
        uint32_t w[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 16 * bn + l + 8 * h;
            const uint4 a = *reinterpret_cast<const uint4*>(tile + tile2d_offset(r, 16 * bk));
            const uint4 c = *reinterpret_cast<const uint4*>(tile + tile2d_offset(r, 16 * bk + 8));
            w[h][0] = a.x; w[h][1] = a.y; w[h][2] = a.z; w[h][3] = a.w;
            w[h][4] = c.x; w[h][5] = c.y; w[h][6] = c.z; w[h][7] = c.w;
        }
        bool z0, z1;
        float amax = fmaxf(amax_bf16x16(w[0], z0), amax_bf16x16(w[1], z1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
        float v[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[h][2 * i] = bf16_lo(w[h][i]);
                v[h][2 * i + 1] = bf16_hi(w[h][i]);
            }
        uint32_t nzero = 0u;  // zeros among this lane's 32 values of W
        if (z0 || z1) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 16; ++i) nzero += v[h][i] == 0.0f ? 1u : 0u;
        }
        const float sval = __fmul_rn(div6_rn(amax), s_enc);
        const uint32_t sc = F::encode(sval);
        if (l == 0) {
            cnt.ssat += sval > F::kMax ? 1u : 0u;
            cnt.sunder += (sc == 0u && amax > 0.0f) ? 1u : 0u;
        }
        const float enc_l = tab[sc];
        uint32_t cw[2][2];
        if (sc == 0u) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                cw[h][0] = sign_nibbles8(v[h]);
                cw[h][1] = sign_nibbles8(v[h] + 8);
            }
            if (!q.count_t) cnt.eunder += 32u - nzero;
        } else {
            float x[2][16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                scale16(v[h], enc_l, x[h]);
                if (SR) {
                    // W element (n, k) has index n K + k
                    const int64_t e0 = (n0 + 16 * bn + l + 8 * h) * K + k0 + 16 * bk;
                    uint4 r[2];
                    sr_block_bits((uint64_t)(e0 >> 3), q.tensor_id, q.step_lo, q.round_key, r);
                    e2m1_sr_x16(x[h], r, cw[h][0], cw[h][1]);
                } else {
                    cw[h][0] = e2m1_rne_x8(x[h]);
                    cw[h][1] = e2m1_rne_x8(x[h] + 8);
                }
            }
            if (__fmul_rn(amax, enc_l) > 6.0f)
                cnt.esat += e2m1_saturating_count<16>(x[0]) + e2m1_saturating_count<16>(x[1]);
            if (!q.count_t)
                cnt.eunder += zero_mag_count16(cw[0][0], cw[0][1]) + zero_mag_count16(cw[1][0], cw[1][1]) - nzero;
        }
        if (q.codes != nullptr) {
            const int64_t jb = (k0 >> 4) + bk;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t n = n0 + 16 * bn + l + 8 * h;
                *reinterpret_cast<uint2*>(q.codes + n * (K / 2) + (k0 + 16 * bk) / 2) = make_uint2(cw[h][0], cw[h][1]);
                q.scales[TCL_W ? tc_scale_offset(n, jb, tk_count) : n * tk_count + jb] = (uint8_t)sc;
            }
        }
        // ---- W^T rows k = 16 bk + 2 l and + 1: columns of the block, 16 values along n
        if (q.codes_t != nullptr) {
            float c0[16], c1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t ww = *reinterpret_cast<const uint32_t*>(tile + tile2d_offset(16 * bn + i, 16 * bk + 2 * l));
                c0[i] = bf16_lo(ww);
                c1[i] = bf16_hi(ww);
            }
            uint32_t tw[2][2];
            if (sc == 0u) {
                tw[0][0] = sign_nibbles8(c0);
                tw[0][1] = sign_nibbles8(c0 + 8);
                tw[1][0] = sign_nibbles8(c1);
                tw[1][1] = sign_nibbles8(c1 + 8);
                if (q.count_t) cnt.eunder += 32u - nzero;  // the same values, transposed
            } else {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float x[16];
                    scale16(hh ? c1 : c0, enc_l, x);
                    if (SR) {
                        // W^T element (k, n) has index k N + n
                        const int64_t e0 = (k0 + 16 * bk + 2 * l + hh) * N + n0 + 16 * bn;
                        uint4 r[2];
                        sr_block_bits((uint64_t)(e0 >> 3), q.tensor_id, q.step_lo, q.round_key, r);
                        e2m1_sr_x16(x, r, tw[hh][0], tw[hh][1]);
                    } else {
                        tw[hh][0] = e2m1_rne_x8(x);
                        tw[hh][1] = e2m1_rne_x8(x + 8);
                    }
                }
                if (q.count_t)
                    cnt.eunder += zero_mag_count16(tw[0][0], tw[0][1]) + zero_mag_count16(tw[1][0], tw[1][1]) - nzero;
            }
            const int64_t jb = (n0 >> 4) + bn;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t k = k0 + 16 * bk + 2 * l + h;
                *reinterpret_cast<uint2*>(q.codes_t + k * (N / 2) + (n0 + 16 * bn) / 2) = make_uint2(tw[h][0], tw[h][1]);
                q.scales_t[TCL_WT ? tc_scale_offset(k, jb, tn_count) : k * tn_count + jb] = (uint8_t)sc;
            }
        }
        if (!__syncthreads_and(ok)) break;
        if (tid == 0) {
            const int64_t tn = t + (int64_t)kTileStages * gridDim.x;
            if (tn < ntiles) issue(tn, s);
        }
    }
    flush_counters(q.counters, cnt.esat, cnt.eunder, cnt.ssat, cnt.sunder);
}

// ----------------------------------------------------------------------------
// K5: MXFP4 1x32 rowwise quantizer (section A3, App. B.4): UE8M0 scale = the
// power of two that rounds amax_B / 6 up, value scaled by 2^-e exactly, RNE.
template <bool TCL>
__global__ void __launch_bounds__(kThreads) quantize_mx_rows_kernel(QParams q) {
    pdl_begin();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (q.s_dec) *q.s_dec = 1.0f;
    }
    const int64_t nb_row = q.cols / 32, nblk = q.rows * nb_row;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    Counts cnt;
    for (int64_t base = warp * 32; base < nblk; base += nwarps * 32) {
        const int64_t b = base + lane;
        const bool active = b < nblk;
        uint32_t sc = 0u;
        if (active) {
            float v[32];
            const int64_t o = strided_off(b, 32, nb_row, q.cols, q.ld);
            unpack16(ldg16(q.in + o), ldg16(q.in + o + 8), v);
            unpack16(ldg16(q.in + o + 16), ldg16(q.in + o + 24), v + 16);
            float amax_b = 0.0f;
#pragma unroll
            for (int e = 0; e < 32; ++e) amax_b = fmaxf(amax_b, fabsf(v[e]));
            int ex = ue8m0_exponent(amax_b);
            if (ex > 127) {
                ex = 127;
                cnt.ssat++;
            }
            if (ex < -127) {
                ex = -127;
                if (amax_b > 0.0f) cnt.sunder++;
            }
            sc = (uint32_t)(ex + 127);
            const float inv = exp2_exact(-ex);
            float x[32];
            uint32_t nzero = 0u;
            scale16(v, inv, x);
            scale16(v + 16, inv, x + 16);
#pragma unroll
            for (int e = 0; e < 32; ++e) nzero += (__float_as_uint(v[e]) << 1) == 0u ? 1u : 0u;
            if (__fmul_rn(amax_b, inv) > 6.0f) cnt.esat += e2m1_saturating_count<32>(x);
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = e2m1_rne_x8(x + 8 * k);
            cnt.eunder += zero_mag_count8(w[0]) + zero_mag_count8(w[1]) + zero_mag_count8(w[2]) +
                          zero_mag_count8(w[3]) - nzero;
            *reinterpret_cast<uint4*>(q.codes + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (TCL) {
            uint32_t w = sc << (8 * (lane & 3));
            w |= __shfl_xor_sync(0xFFFFFFFFu, w, 1);
            w |= __shfl_xor_sync(0xFFFFFFFFu, w, 2);
            if (active && (lane & 3) == 0) {
                const int64_t r = b / nb_row, j = b % nb_row;
                *reinterpret_cast<uint32_t*>(q.scales + tc_scale_offset(r, j, nb_row)) = w;
            }
        } else if (active) {
            q.scales[b] = (uint8_t)sc;
        }
    }
    flush_counters(q.counters, cnt.esat, cnt.eunder, cnt.ssat, cnt.sunder);
}

// ----------------------------------------------------------------------------
// K6: dequantize (section A3: decode back to the original range; App. B.3):
// x = RN(RN(e2m1 * s_hat) * s_dec,G) in FP32, stored as BF16 (RNE) or FP32.
template <int FMT, int BS, bool TCL, bool OUT32>
__global__ void __launch_bounds__(kThreads) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                              const uint8_t* __restrict__ scales,
                                                              const float* __restrict__ s_dec_p, int s_dec_rows,
                                                              int64_t rows, int64_t cols, void* __restrict__ out) {
    pdl_begin();
    const float s_dec0 = s_dec_rows ? 0.0f : *s_dec_p;
    const int64_t nb_row = cols / BS, nblk = rows * nb_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += stride) {
        const int64_t r = b / nb_row, j = b % nb_row;
        const float s_dec = s_dec_rows ? s_dec_p[r] : s_dec0;
        const uint32_t sc = scales[TCL ? tc_scale_offset(r, j, nb_row) : b];
        float s_hat;
        if constexpr (FMT == kFmtUE8M0) s_hat = exp2_exact((int)sc - 127);
        else s_hat = ScaleFmt<FMT>::decode(sc);
        uint32_t w[BS / 8];
#pragma unroll
        for (int k = 0; k < BS / 8; ++k) w[k] = reinterpret_cast<const uint32_t*>(codes + (BS / 2) * b)[k];
#pragma unroll
        for (int e = 0; e < BS; e += 8) {
            float o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t code = (w[e >> 3] >> (4 * k)) & 0xFu;
                const uint32_t m = code & 7u;
                const float mag = m <= 4u ? 0.5f * (float)m : (m == 5u ? 3.0f : (m == 6u ? 4.0f : 6.0f));
                const float val = (code & 8u) ? -mag : mag;
                o[k] = __fmul_rn(__fmul_rn(val, s_hat), s_dec);
            }
            if (OUT32) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + BS * b + e);
                dst[0] = make_float4(o[0], o[1], o[2], o[3]);
                dst[1] = make_float4(o[4], o[5], o[6], o[7]);
            } else {
                uint32_t p[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
                    p[k] = *reinterpret_cast<const uint32_t*>(&h);
                }
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + BS * b + e) = make_uint4(p[0], p[1], p[2], p[3]);
            }
        }
    }
}

// ----------------------------------------------------------------------------
// K7: dual quantizer. One BF16 input X [T x C] yields both operands a linear
// layer takes from it -- X rowwise (1x16 blocks along C, Fprop / Dgrad) and X^T
// colwise (1x16 blocks along T, optional RHT16, Wgrad) -- from one read of X.
// Each output is bit-identical to what its own quantize call would produce
// (its own tensor scale, rounding mode, tensor id and counters).

// Both amaxes from one read: plain max|x| for the rowwise operand and, with the
// RHT, max|H x| over 16-token tiles for the colwise one. Each thread owns 16
// tokens x 4 channels.
template <bool RHT>
__global__ void __launch_bounds__(kThreads) amax_dual_kernel(const uint16_t* __restrict__ in, int64_t T, int64_t C,
                                                             int64_t ld, float* __restrict__ partials_row,
                                                             float* __restrict__ partials_col,
                                                             const fp4_amax_state_t* skip_row,
                                                             const fp4_amax_state_t* skip_col) {
    pdl_begin();
    if (amax_pass_skipped(skip_row, skip_col)) return;
    const int64_t ug = C / 4, uj = T / 16, units = ug * uj;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    uint32_t mr = 0u;
    float mc = 0.0f;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int64_t g = u % ug, j = u / ug;
        uint2 x[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) x[t] = __ldg(reinterpret_cast<const uint2*>(in + (16 * j + t) * ld + 4 * g));
#pragma unroll
        for (int t = 0; t < 16; ++t) mr = __vmaxu2(mr, __vmaxu2(x[t].x & 0x7FFF7FFFu, x[t].y & 0x7FFF7FFFu));
        if (RHT) {
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                f2 pv[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const uint32_t w = pr ? x[t].y : x[t].x;
                    pv[t] = f2_pack(bf16_lo(w), bf16_hi(w));
                }
                wht16x2(pv);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float a, b;
                    f2_unpack(pv[t], a, b);
                    mc = fmaxf(mc, fmaxf(fabsf(a), fabsf(b)));
                }
            }
        }
    }
    const float fr = cta_max(__uint_as_float(max(mr & 0xFFFFu, mr >> 16) << 16));
    const float fc = RHT ? cta_max(__fmul_rn(mc, 0.25f)) : fr;
    if (threadIdx.x == 0) {
        partials_row[blockIdx.x] = fr;
        partials_col[blockIdx.x] = fc;
    }
}

constexpr int kDualTT = 64;    // tokens per tile
constexpr int kDualTC = 128;   // channels per tile

constexpr int kDualStages = 3;                       // tiles in flight per CTA
constexpr int kDualTileBytes = kDualTT * kDualTC * 2;  // 16 KB of BF16
constexpr int kDualSmemBytes = kDualStages * kDualTileBytes + 1024;

// The conversion pass. A CTA walks 64-token x 128-channel tiles of X; one
// thread keeps kDualStages tiles in flight with TMA loads into a shared-memory
// ring (an mbarrier per stage), and all threads convert the current tile: two
// rowwise blocks each (16 consecutive channels of one token, two 128-bit shared
// loads) and one colwise pair (16 tokens of two adjacent channels, sixteen
// 32-bit shared loads, so a warp reads 32 consecutive channel pairs of one token
// row per load and never conflicts on a bank). T % 128 == 0, C % 128 == 0.
template <int FMT, bool SR_ROW, bool SR_COL, bool RHT>
__global__ void __launch_bounds__(kThreads, 2)
    quantize_dual_kernel(const __grid_constant__ CUtensorMap tmap_x, QParams qr, QParams qc) {
    pdl_begin();
    extern __shared__ uint8_t dual_smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dual_smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ float tab_r[256], tab_c[256];
    __shared__ __align__(8) uint64_t full_bar[kDualStages];
    float se_r, sd_r, se_c, sd_c;
    if (!cta_tensor_scale(qr, se_r, sd_r)) return;
    __syncthreads();
    if (!cta_tensor_scale(qc, se_c, sd_c)) return;
    fill_enc_table<FMT>(tab_r, sd_r);
    fill_enc_table<FMT>(tab_c, sd_c);
    if (threadIdx.x == 0) {
        for (int k = 0; k < kDualStages; ++k) tc::mbar_init(tc::smem_u32(&full_bar[k]), 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    const int64_t T = qr.rows, C = qr.cols;
    const int64_t tiles_c = C / kDualTC, ntiles = (T / kDualTT) * tiles_c;
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t signs = RHT ? rht_sign_word(qc.key0, qc.key1) : 0u;
    uint32_t smask_lo = 0u, smask_hi = 0u;
    if (RHT) rht_sign_masks(signs, smask_lo, smask_hi);
    const int64_t nb_row = C / 16, nb_col = T / 16;
    // Per-thread parts of the output offsets (the tile's parts are added per tile;
    // t0 is a multiple of 64 and c0 of 128, so tile and thread parts separate).
    // Rowwise blocks (r, b) and (r + 32, b); tensor-core scale offset of row
    // t0 + r, block c0/16 + b = tile part + 512 (b / 4) + 16 (r % 32) + 4 (r / 32) + b % 4.
    const int r_row = tid >> 3, b_row = tid & 7;
    const int64_t code_row_thr = 8 * (int64_t)r_row * nb_row + 8 * b_row;  // + 256 nb_row for r + 32
    const uint32_t sc_row_thr = 512u * (b_row >> 2) + 16u * (r_row & 31) + (b_row & 3);
    // Colwise pair: channels c0 + 2 cp + ch, token block t0/16 + jb.
    const int cp = tid & 63, jb = tid >> 6;
    Counts cr, cc;
    auto issue = [&](TileCursor at, int s) {
        const uint32_t bar = tc::smem_u32(&full_bar[s]);
        tc::mbar_arrive_expect_tx(bar, kDualTileBytes);
        tc::tma_load_2d(tc::smem_u32(ring + s * kDualTileBytes), &tmap_x, (int32_t)(at.col * kDualTC),
                        (int32_t)(at.row * kDualTT), bar);
    };
    if (tid == 0) {
        tc::prefetch_tmap(&tmap_x);
        for (int k = 0; k < kDualStages; ++k) {
            const int64_t tk = blockIdx.x + (int64_t)k * gridDim.x;
            if (tk < ntiles) issue(TileCursor::at(tk, tiles_c), k);
        }
    }
    // this tile's and the refill tile's coordinates, advanced without a division
    TileCursor cur = TileCursor::at(blockIdx.x, tiles_c);
    TileCursor ahead = TileCursor::at(blockIdx.x + (int64_t)kDualStages * gridDim.x, tiles_c);
    const TileCursor step = TileCursor::at(gridDim.x, tiles_c);
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = (int)(it % kDualStages);
        const bool ok = tc::mbar_wait(tc::smem_u32(&full_bar[s]), (it / kDualStages) & 1u, qr.status);
        const uint16_t* tile = reinterpret_cast<const uint16_t*>(ring + s * kDualTileBytes);
        const int64_t t0 = cur.row * kDualTT, c0 = cur.col * kDualTC;
        // rowwise: blocks (r, b) and (r + 32, b) of the tile's 64 x 8 blocks
        const int64_t code_row_tile = 8 * t0 * nb_row + (c0 >> 1);
        const int64_t sc_row_tile = 512 * ((t0 >> 7) * (nb_row >> 2) + (c0 >> 6)) + ((t0 & 64) >> 3);
        // kept rolled: with stochastic rounding the unrolled body's code size
        // costs more in instruction fetch than the loop saves (measured)
#pragma unroll 1
        for (int i = 0; i < 2; ++i) {
            const int r = r_row + 32 * i;
            const uint4 a = *reinterpret_cast<const uint4*>(&tile[r * kDualTC + 16 * b_row]);
            const uint4 c = *reinterpret_cast<const uint4*>(&tile[r * kDualTC + 16 * b_row + 8]);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
            bool any_zero;
            const float vmax = amax_bf16x16(w, any_zero);
            float v[16];
            unpack16(a, c, v);
            const int64_t code_off = code_row_tile + code_row_thr + 256 * i * nb_row;  // = 8 * block index
            uint32_t lo, hi;
            const uint32_t sc = quantize_block16<FMT, SR_ROW, false>(v, vmax, any_zero, tab_r, se_r,
                                                                     (uint64_t)(code_off >> 2), qr, 0u, 0u, lo, hi, cr);
            *reinterpret_cast<uint2*>(qr.codes + code_off) = make_uint2(lo, hi);
            uint32_t ww = sc << (8 * (lane & 3));
            ww |= __shfl_xor_sync(0xFFFFFFFFu, ww, 1);
            ww |= __shfl_xor_sync(0xFFFFFFFFu, ww, 2);
            if ((lane & 3) == 0)
                *reinterpret_cast<uint32_t*>(qr.scales + sc_row_tile + sc_row_thr + 4u * i) = ww;
        }
        // colwise: channel pair cp, token block jb
        {
            f2 pv[16];
#pragma unroll
            for (int tt = 0; tt < 16; ++tt) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[(16 * jb + tt) * kDualTC + 2 * cp]);
                pv[tt] = f2_pack(bf16_lo(w), bf16_hi(w));
            }
            if (RHT) wht16x2(pv);
            const int64_t code_col_tile = c0 * (T >> 1) + (t0 >> 1) + 8 * jb;
            const int64_t sc_col_tile = 512 * ((c0 >> 7) * (nb_col >> 2) + (t0 >> 6)) + jb;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                float v[16];
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) {
                    float a, b;
                    f2_unpack(pv[tt], a, b);
                    v[tt] = ch ? b : a;
                }
                bool any_zero;
                const float vmax = amax_f32x16(v, any_zero);
                const int cc_local = 2 * cp + ch;  // channel within the tile
                const int64_t code_off = code_col_tile + (int64_t)cc_local * (T >> 1);  // = 8 * block index
                uint32_t lo, hi;
                const uint32_t sc = quantize_block16<FMT, SR_COL, RHT>(v, vmax, any_zero, tab_c, se_c,
                                                                       (uint64_t)(code_off >> 2), qc, smask_lo,
                                                                       smask_hi, lo, hi, cc);
                *reinterpret_cast<uint2*>(qc.codes + code_off) = make_uint2(lo, hi);
                qc.scales[sc_col_tile + 16 * (cc_local & 31) + 4 * (cc_local >> 5)] = (uint8_t)sc;
            }
        }
        // every thread is done reading stage s (and every wait succeeded):
        // refill it with the tile kDualStages steps ahead
        if (!__syncthreads_and(ok)) break;
        if (tid == 0) {
            const int64_t tn = t + (int64_t)kDualStages * gridDim.x;
            if (tn < ntiles) issue(ahead, s);
        }
        cur.advance(step, tiles_c);
        ahead.advance(step, tiles_c);
    }
    flush_counters(qr.counters, cr.esat, cr.eunder, cr.ssat, cr.sunder);
    flush_counters(qc.counters, cc.esat, cc.eunder, cc.ssat, cc.sunder);
}

// Tensor amax ahead of quantization (fp4_tensor_amax): the plain amax and/or
// the post-RHT colwise amax of a T x C tensor (T % 64 == 0, C % 128 == 0), one
// read, in 128-thread CTAs with one 16 KB TMA tile ring each (49 KB of shared
// memory, few registers), two CTAs per SM. Sized so a CTA fits on an SM beside
// two conversion-pass CTAs of the dual quantizer: run on a second stream, the
// amax of one tensor overlaps the (issue-bound) conversion of another.
constexpr int kAmaxTileThreads = 128;
template <bool PLAIN, bool RHT>
__global__ void __launch_bounds__(kAmaxTileThreads)
    amax_tile_kernel(const __grid_constant__ CUtensorMap tmap_x, int64_t T, int64_t C, float* __restrict__ part_plain,
                     float* __restrict__ part_rht, int* status) {
    pdl_begin();
    extern __shared__ uint8_t amax_smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(amax_smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[kDualStages];
    __shared__ float red[2][kAmaxTileThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid == 0) {
        for (int k = 0; k < kDualStages; ++k) tc::mbar_init(tc::smem_u32(&full_bar[k]), 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    const int64_t tiles_c = C / kDualTC, ntiles = (T / kDualTT) * tiles_c;
    auto issue = [&](TileCursor at, int s) {
        const uint32_t bar = tc::smem_u32(&full_bar[s]);
        tc::mbar_arrive_expect_tx(bar, kDualTileBytes);
        tc::tma_load_2d(tc::smem_u32(ring + s * kDualTileBytes), &tmap_x, (int32_t)(at.col * kDualTC),
                        (int32_t)(at.row * kDualTT), bar);
    };
    if (tid == 0) {
        tc::prefetch_tmap(&tmap_x);
        for (int k = 0; k < kDualStages; ++k) {
            const int64_t tk = blockIdx.x + (int64_t)k * gridDim.x;
            if (tk < ntiles) issue(TileCursor::at(tk, tiles_c), k);
        }
    }
    // the refill tile's coordinates, advanced without a division
    TileCursor ahead = TileCursor::at(blockIdx.x + (int64_t)kDualStages * gridDim.x, tiles_c);
    const TileCursor step = TileCursor::at(gridDim.x, tiles_c);
    uint32_t mp = 0u;   // max |x| as BF16 bit pairs
    float mr = 0.0f;    // max |RHT x| (times 4: the 1/4 is applied once at the end)
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = (int)(it % kDualStages);
        const bool ok = tc::mbar_wait(tc::smem_u32(&full_bar[s]), (it / kDualStages) & 1u, status);
        const uint8_t* tile = ring + s * kDualTileBytes;
        if (PLAIN) {
            // 64 x 128 BF16 = 1024 16-byte chunks, eight per thread
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 a = *reinterpret_cast<const uint4*>(tile + 16 * (tid + kAmaxTileThreads * i));
                mp = __vmaxu2(mp, __vmaxu2(__vmaxu2(a.x & 0x7FFF7FFFu, a.y & 0x7FFF7FFFu),
                                           __vmaxu2(a.z & 0x7FFF7FFFu, a.w & 0x7FFF7FFFu)));
            }
        }
        if (RHT) {
            // 4 token blocks x 64 channel pairs; a thread takes two of them
#pragma unroll 1
            for (int u = 0; u < 2; ++u) {
                const int unit = tid + kAmaxTileThreads * u, cp = unit & 63, jb = unit >> 6;
                f2 pv[16];
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + (16 * jb + tt) * (kDualTC * 2) + 4 * cp);
                    pv[tt] = f2_pack(bf16_lo(w), bf16_hi(w));
                }
                wht16x2(pv);
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) {
                    float a, b;
                    f2_unpack(pv[tt], a, b);
                    mr = fmaxf(mr, fmaxf(fabsf(a), fabsf(b)));
                }
            }
        }
        if (!__syncthreads_and(ok)) break;
        if (tid == 0) {
            const int64_t tn = t + (int64_t)kDualStages * gridDim.x;
            if (tn < ntiles) issue(ahead, s);
        }
        ahead.advance(step, tiles_c);
    }
    float vp = __uint_as_float(max(mp & 0xFFFFu, mp >> 16) << 16), vr = __fmul_rn(mr, 0.25f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        vp = fmaxf(vp, __shfl_xor_sync(0xFFFFFFFFu, vp, o));
        vr = fmaxf(vr, __shfl_xor_sync(0xFFFFFFFFu, vr, o));
    }
    if (lane == 0) {
        red[0][tid >> 5] = vp;
        red[1][tid >> 5] = vr;
    }
    __syncthreads();
    if (tid == 0) {
        float a = 0.0f, b = 0.0f;
#pragma unroll
        for (int w = 0; w < kAmaxTileThreads / 32; ++w) {
            a = fmaxf(a, red[0][w]);
            b = fmaxf(b, red[1][w]);
        }
        if (PLAIN) part_plain[blockIdx.x] = a;
        if (RHT) part_rht[blockIdx.x] = b;
    }
}

// Reduce amax partials into tensor-amax records (one CTA); a null record is skipped.
__global__ void __launch_bounds__(kThreads) amax_finalize_kernel(const float* __restrict__ part_a, fp4_amax_state_t* st_a,
                                                                 const float* __restrict__ part_b, fp4_amax_state_t* st_b,
                                                                 int n, uint64_t step) {
    pdl_begin();
    float a = 0.0f, b = 0.0f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (st_a) a = fmaxf(a, part_a[i]);
        if (st_b) b = fmaxf(b, part_b[i]);
    }
    a = cta_max(a);
    b = cta_max(b);
    if (threadIdx.x == 0) {
        if (st_a) {
            st_a->amax_held = a;
            st_a->valid = 1;
            st_a->last_refresh_step = step;
        }
        if (st_b) {
            st_b->amax_held = b;
            st_b->valid = 1;
            st_b->last_refresh_step = step;
        }
    }
}

int grid_for(int64_t threads_wanted, int per_sm) {
    const int64_t want = (threads_wanted + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    int64_t g = want < cap ? want : cap;
    return (int)(g < 1 ? 1 : g);
}

template <int FMT>
cudaError_t launch_fmt(const QuantJob& j, const QParams& q, cudaStream_t st) {
    const bool tcl = j.layout == FP4_LAYOUT_TCGEN05;
    if (j.block == FP4_BLOCK_16x16) {
        const int64_t tiles = (j.rows / 16) * (j.cols / 16);
        const int grid = grid_for(tiles * 16, 8);
        // the kernel's primary output is W (rowwise); for COLWISE the operand is
        // W^T, which the kernel writes through its transposed output
        QParams p = q;
        p.count_t = j.colwise;  // the counters follow the requested operand
        int lw, lwt;
        if (j.colwise) {
            p.codes = j.codes_t;
            p.scales = j.scales_t;
            p.s_dec = j.s_dec_t;
            p.codes_t = j.codes;
            p.scales_t = j.scales;
            p.s_dec_t = j.s_dec;
            lw = j.layout_t;
            lwt = j.layout;
        } else {
            lw = j.layout;
            lwt = j.layout_t;
        }
        const bool a = lw == FP4_LAYOUT_TCGEN05, b = lwt == FP4_LAYOUT_TCGEN05;
        CUtensorMap tmap_w;
        if (j.rows % 64 == 0 && j.cols % 128 == 0 && make_tmap_bf16_2d(&tmap_w, j.in, j.rows, j.cols, 64, 64, true, j.ld)) {
            const int64_t ntiles = (j.rows / 64) * (j.cols / 128);
            const int64_t cap = (int64_t)num_sms() * 2;
            const int g2 = (int)(ntiles < cap ? ntiles : cap);
#define FP4_2D_TILE(TA, TB)                                                                                          \
    do {                                                                                                            \
        auto kern = j.sr ? quantize_2d_tile_kernel<FMT, true, TA, TB> : quantize_2d_tile_kernel<FMT, false, TA, TB>;  \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, k2dSmemBytes);      \
        if (e != cudaSuccess) return e;                                                                             \
        (void)launch_pdl(kern, g2, kThreads, k2dSmemBytes, st, tmap_w, p);                                                        \
    } while (0)
            if (a && b) FP4_2D_TILE(true, true);
            else if (a) FP4_2D_TILE(true, false);
            else if (b) FP4_2D_TILE(false, true);
            else FP4_2D_TILE(false, false);
#undef FP4_2D_TILE
            return cudaGetLastError();
        }
        if (j.sr) return cudaErrorNotSupported;  // the half-warp kernel rounds to nearest only
        if (a && b) (void)launch_pdl(quantize_2d_kernel<FMT, true, true>, grid, kThreads, 0, st, p);
        else if (a) (void)launch_pdl(quantize_2d_kernel<FMT, true, false>, grid, kThreads, 0, st, p);
        else if (b) (void)launch_pdl(quantize_2d_kernel<FMT, false, true>, grid, kThreads, 0, st, p);
        else (void)launch_pdl(quantize_2d_kernel<FMT, false, false>, grid, kThreads, 0, st, p);
        return cudaGetLastError();
    }
    if (!j.colwise) {
        const int grid = grid_for(j.rows * (j.cols / 16), 8);
        if (j.sr) {
            if (tcl) (void)launch_pdl(quantize_rows_kernel<FMT, true, true>, grid, kThreads, 0, st, q);
            else (void)launch_pdl(quantize_rows_kernel<FMT, true, false>, grid, kThreads, 0, st, q);
        } else {
            if (tcl) (void)launch_pdl(quantize_rows_kernel<FMT, false, true>, grid, kThreads, 0, st, q);
            else (void)launch_pdl(quantize_rows_kernel<FMT, false, false>, grid, kThreads, 0, st, q);
        }
        return cudaGetLastError();
    }
    const int64_t wunits = ((j.cols / 4 + 7) / 8) * ((j.rows / 16 + 3) / 4);
    const int grid = grid_for(wunits * 32, 8);
#define FP4_COLS(SR, RHT, TCL) launch_pdl(quantize_cols_kernel<FMT, SR, RHT, TCL>, grid, kThreads, 0, st, q)
    if (j.sr) {
        if (j.rht) { if (tcl) FP4_COLS(true, true, true); else FP4_COLS(true, true, false); }
        else { if (tcl) FP4_COLS(true, false, true); else FP4_COLS(true, false, false); }
    } else {
        if (j.rht) { if (tcl) FP4_COLS(false, true, true); else FP4_COLS(false, true, false); }
        else { if (tcl) FP4_COLS(false, false, true); else FP4_COLS(false, false, false); }
    }
#undef FP4_COLS
    return cudaGetLastError();
}

int amax_grid(const QuantJob& j) {
    if (j.rht) {
        const int64_t units = (j.cols / 4) * (j.rows / 16);
        int g = grid_for(units, 8);
        return g < kMaxAmaxPartials ? g : kMaxAmaxPartials;
    }
    const int64_t nvec = j.rows * j.cols / 8;
    int g = grid_for((nvec + kAmaxVec - 1) / kAmaxVec, 4);
    return g < kMaxAmaxPartials ? g : kMaxAmaxPartials;
}

QParams make_params(const QuantJob& j) {
    QParams q{};
    q.in = j.in;
    q.rows = j.rows;
    q.cols = j.cols;
    q.ld = j.ld;
    q.codes = j.codes;
    q.scales = j.scales;
    q.s_dec = j.s_dec;
    q.codes_t = j.codes_t;
    q.scales_t = j.scales_t;
    q.s_dec_t = j.s_dec_t;
    q.state = j.state;
    q.given = j.given;
    q.counters = j.counters;
    q.partials = j.partials;
    q.held = j.held;
    q.refresh = j.refresh;
    q.target_T = j.target_T;
    q.tensor_id = j.tensor_id;
    q.step = j.step;
    q.step_lo = (uint32_t)j.step;
    q.key0 = (uint32_t)j.seed;
    q.key1 = (uint32_t)(j.seed >> 32);
    for (int r = 0; r < 10; ++r) {
        q.round_key[2 * r] = q.key0 + (uint32_t)r * kPhiloxW0;
        q.round_key[2 * r + 1] = q.key1 + (uint32_t)r * kPhiloxW1;
    }
    q.status = j.status;
    return q;
}

}  // namespace

int amax_partials_needed(const QuantJob& j) {
    if (j.scale_fmt == kFmtUE8M0 || j.given || j.per_row) return 0;
    if (j.rows == 0 || j.cols == 0) return 0;
    return amax_grid(j);  // held non-refresh steps too: the state may not be valid yet
}

cudaError_t launch_quantize(const QuantJob& j, cudaStream_t st) {
    QParams q = make_params(j);
    if (j.rows == 0 || j.cols == 0) return cudaSuccess;

    if (j.scale_fmt == kFmtUE8M0) {
        const int grid = grid_for(j.rows * (j.cols / 32), 8);
        if (j.layout == FP4_LAYOUT_TCGEN05) (void)launch_pdl(quantize_mx_rows_kernel<true>, grid, kThreads, 0, st, q);
        else (void)launch_pdl(quantize_mx_rows_kernel<false>, grid, kThreads, 0, st, q);
        return cudaGetLastError();
    }
    if (j.per_row) {
        // one warp per operand row (E4M3, rowwise 1x16: checked by the caller)
        const int grid = grid_for(j.rows * 32, 8);
        const bool tcl = j.layout == FP4_LAYOUT_TCGEN05;
#define FP4_ROWSCALE(SR, TCL) launch_pdl(quantize_rows_rowscale_kernel<kFmtE4M3, SR, TCL>, grid, kThreads, 0, st, q)
        if (j.sr) { if (tcl) FP4_ROWSCALE(true, true); else FP4_ROWSCALE(true, false); }
        else { if (tcl) FP4_ROWSCALE(false, true); else FP4_ROWSCALE(false, false); }
#undef FP4_ROWSCALE
        return cudaGetLastError();
    }
    // pass 1 (current scaling, or a held-amax refresh step): amax partials
    const int np = amax_partials_needed(j);
    q.npartials = np;
    if (np > 0) {
        const fp4_amax_state_t* skip = (j.held && !j.refresh) ? j.state : nullptr;
        if (j.rht)
            (void)launch_pdl(amax_rht_cols_kernel, np, kThreads, 0, st, j.in, j.rows, j.cols, j.ld, j.partials, skip);
        else
            (void)launch_pdl(amax_plain_kernel, np, kThreads, 0, st, reinterpret_cast<const uint4*>(j.in),
                             j.rows * j.cols / 8, j.cols / 8, j.ld / 8, j.partials, skip);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // pass 2: scale and convert
    if (j.scale_fmt == kFmtE4M3) return launch_fmt<kFmtE4M3>(j, q, st);
    return launch_fmt<kFmtUE5M3>(j, q, st);
}

namespace {
__global__ void div6_selftest_kernel(const float* __restrict__ in, float* __restrict__ out, int64_t n) {
    pdl_begin();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = div6_rn(in[i]);
}
}  // namespace

cudaError_t launch_div6_selftest(const float* in, float* out, int64_t n, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    (void)launch_pdl(div6_selftest_kernel, grid_for(n, 4), kThreads, 0, st, in, out, n);
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const DequantJob& j, cudaStream_t st) {
    if (j.rows == 0 || j.cols == 0) return cudaSuccess;
    const int grid = grid_for(j.rows * (j.cols / j.block_k), 8);
    const bool tcl = j.layout == FP4_LAYOUT_TCGEN05;
#define FP4_DQ(FMT, BS)                                                                                           \
    do {                                                                                                          \
        if (tcl) {                                                                                                \
            if (j.out_fp32) (void)launch_pdl(dequantize_kernel<FMT, BS, true, true>, grid, kThreads, 0, st, j.codes, j.scales, j.s_dec, j.s_dec_rows, j.rows, j.cols, j.out); \
            else (void)launch_pdl(dequantize_kernel<FMT, BS, true, false>, grid, kThreads, 0, st, j.codes, j.scales, j.s_dec, j.s_dec_rows, j.rows, j.cols, j.out); \
        } else {                                                                                                  \
            if (j.out_fp32) (void)launch_pdl(dequantize_kernel<FMT, BS, false, true>, grid, kThreads, 0, st, j.codes, j.scales, j.s_dec, j.s_dec_rows, j.rows, j.cols, j.out); \
            else (void)launch_pdl(dequantize_kernel<FMT, BS, false, false>, grid, kThreads, 0, st, j.codes, j.scales, j.s_dec, j.s_dec_rows, j.rows, j.cols, j.out); \
        }                                                                                                         \
    } while (0)
    if (j.scale_fmt == kFmtE4M3) FP4_DQ(kFmtE4M3, 16);
    else if (j.scale_fmt == kFmtUE5M3) FP4_DQ(kFmtUE5M3, 16);
    else FP4_DQ(kFmtUE8M0, 32);
#undef FP4_DQ
    return cudaGetLastError();
}

int dual_amax_grid(const QuantJob& jc) {
    const int64_t units = (jc.rows / 16) * (jc.cols / 4);  // input T x C: 16 tokens x 4 channels per thread
    int g = grid_for(units, 8);
    return g < kMaxAmaxPartials ? g : kMaxAmaxPartials;
}

cudaError_t launch_tensor_amax(const uint16_t* in, int64_t T, int64_t C, int64_t ld, fp4_amax_state_t* st_plain,
                               fp4_amax_state_t* st_col, bool rht, uint64_t step, float* partials, int* status,
                               cudaStream_t st) {
    if (T == 0 || C == 0) {
        // an empty tensor has amax 0
        (void)launch_pdl(amax_finalize_kernel, 1, kThreads, 0, st, partials, st_plain, partials + kMaxAmaxPartials,
                         st_col, 0, step);
        return cudaGetLastError();
    }
    float* part_plain = partials;
    float* part_col = partials + kMaxAmaxPartials;
    const bool plain = st_plain != nullptr || (st_col != nullptr && !rht);
    const bool post_rht = st_col != nullptr && rht;
    int np;
    CUtensorMap tmap_x;
    if (T % kDualTT == 0 && C % kDualTC == 0 && make_tmap_bf16_2d(&tmap_x, in, T, C, kDualTT, kDualTC, false, ld)) {
        // two CTAs per SM when the pass runs alone; beside a conversion pass one fits
        // and the other follows
        const int64_t ntiles = (T / kDualTT) * (C / kDualTC), cap = 2 * (int64_t)num_sms();
        np = (int)(ntiles < cap ? ntiles : cap);
        const int smem = kDualStages * kDualTileBytes + 1024;
#define FP4_AMAX_TILE(P, R)                                                                                     \
    do {                                                                                                        \
        auto kern = amax_tile_kernel<P, R>;                                                                     \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);          \
        if (e != cudaSuccess) return e;                                                                         \
        (void)launch_pdl(kern, np, kAmaxTileThreads, smem, st, tmap_x, T, C, part_plain, part_col, status);     \
    } while (0)
        if (plain && post_rht) FP4_AMAX_TILE(true, true);
        else if (plain) FP4_AMAX_TILE(true, false);
        else FP4_AMAX_TILE(false, true);
#undef FP4_AMAX_TILE
    } else {
        // other shapes: the quantizer's own amax passes
        QuantJob j{};
        j.rows = T;
        j.cols = C;
        j.ld = ld;
        j.colwise = post_rht;
        j.rht = post_rht;
        np = amax_grid(j);
        if (plain)
            (void)launch_pdl(amax_plain_kernel, np, kThreads, 0, st, reinterpret_cast<const uint4*>(in), T * C / 8,
                             C / 8, ld / 8, part_plain, (const fp4_amax_state_t*)nullptr);
        if (post_rht)
            (void)launch_pdl(amax_rht_cols_kernel, np, kThreads, 0, st, in, T, C, ld, part_col,
                             (const fp4_amax_state_t*)nullptr);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // a colwise record without RHT takes the plain amax
    (void)launch_pdl(amax_finalize_kernel, 1, kThreads, 0, st, part_plain, st_plain,
                     post_rht ? part_col : part_plain, st_col, np, step);
    return cudaGetLastError();
}

cudaError_t launch_quantize_dual(const QuantJob& jr, const QuantJob& jc, cudaStream_t st) {
    if (jr.rows == 0 || jr.cols == 0) return cudaSuccess;
    QParams qr = make_params(jr), qc = make_params(jc);
    if (!jr.given) {
        // held non-refresh steps: the pass runs only while a held state is not valid yet
        const bool held_step = jr.held && !jr.refresh;
        const fp4_amax_state_t* skip_r = held_step ? jr.state : nullptr;
        const fp4_amax_state_t* skip_c = held_step ? jc.state : nullptr;
        const int np = dual_amax_grid(jc);
        qr.npartials = qc.npartials = np;
        if (jc.rht)
            (void)launch_pdl(amax_dual_kernel<true>, np, kThreads, 0, st, jr.in, jr.rows, jr.cols, jr.ld, jr.partials, jc.partials, skip_r,
                                                             skip_c);
        else
            (void)launch_pdl(amax_dual_kernel<false>, np, kThreads, 0, st, jr.in, jr.rows, jr.cols, jr.ld, jr.partials, jc.partials, skip_r,
                                                              skip_c);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int64_t ntiles = (jr.rows / kDualTT) * (jr.cols / kDualTC);
    const int64_t cap = (int64_t)num_sms() * 2;
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    CUtensorMap tmap_x;
    if (!make_tmap_bf16_2d(&tmap_x, jr.in, jr.rows, jr.cols, kDualTT, kDualTC, false, jr.ld)) return cudaErrorInvalidValue;
#define FP4_DUAL(FMT, SR, RHT)                                                                                   \
    do {                                                                                                         \
        auto kern = quantize_dual_kernel<FMT, SR, SR, RHT>;                                                      \
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDualSmemBytes); \
        if (e != cudaSuccess) return e;                                                                          \
        (void)launch_pdl(kern, grid, kThreads, kDualSmemBytes, st, tmap_x, qr, qc);                                            \
    } while (0)
    if (jr.scale_fmt == kFmtE4M3) {
        if (jr.sr) { if (jc.rht) FP4_DUAL(kFmtE4M3, true, true); else FP4_DUAL(kFmtE4M3, true, false); }
        else { if (jc.rht) FP4_DUAL(kFmtE4M3, false, true); else FP4_DUAL(kFmtE4M3, false, false); }
    } else {
        if (jr.sr) { if (jc.rht) FP4_DUAL(kFmtUE5M3, true, true); else FP4_DUAL(kFmtUE5M3, true, false); }
        else { if (jc.rht) FP4_DUAL(kFmtUE5M3, false, true); else FP4_DUAL(kFmtUE5M3, false, false); }
    }
#undef FP4_DUAL
    return cudaGetLastError();
}

}  // namespace fp4bs
