// gemm_ue5m3.cu -- software-emulated UE5M3 block-scaled GEMM on sm_103a.
//
// The UE5M3 pretraining paper (arXiv 2609.02846, abstract and limitations)
// runs its UE5M3-scaled FP4 GEMMs in software emulation because no tensor core
// reads UE5M3 block scales. The product it needs is the same block-scaled sum
// as NVFP4 ("Pretraining LLMs with NVFP4", App. B.3):
//     D[m,n] = s_dec,G,A * s_dec,G,B * sum_k (a_mk s_A)(b_nk s_B).
// Each decoded operand value a * s (an E2M1 value times a UE5M3 scale) has at
// most 6 significant bits and an exponent inside the BF16 range, so it is EXACT
// in BF16; a BF16 x BF16 tensor-core MMA with FP32 accumulation then computes
// the same products the native path would.
//
// Design (one persistent CTA per SM, 128 x 128 output tiles, 704 threads):
//   warp 0      : TMA producer -- raw FP4 code tiles (K = 256) and scale chunks;
//   warps 2-17  : decode -- per K = 64 slice, each thread expands one 16-byte
//                 raw chunk (32 values) of one operand row into BF16 with
//                 byte-permute table lookups, multiplies by the block scale
//                 (packed BF16 multiply, exact) and writes the 128-byte-swizzled
//                 K-major layout the tensor core reads. Sixteen warps keep four
//                 per scheduler: measured on GB300, four decode warps (one per
//                 scheduler) left the MMA waiting for decoded data 66 % of the time;
//   warp 1      : one lane issues tcgen05.mma kind::f16 (K = 16) on each decoded
//                 slice and commits it back to the decoders;
//   warps 18-21 : epilogue -- each raw stage (K = 256) is one accumulator chunk in
//                 one of two tensor-memory buffers; the epilogue adds the chunk
//                 to a running FP32 sum kept in a third tensor-memory region
//                 (tcgen05.ld both, add with round-to-nearest, tcgen05.st), so no
//                 accumulator lives in registers, and at the last chunk of a tile
//                 stores alpha * (sum + chunk).
// After a rebias pass (fp4_gemm_ws) this kernel computes only the output tiles
// whose rows did not fit, usually one 128-row tile-row (where the native
// kernel ran 128 x 256 tiles, a flagged B row tile takes the other half of its
// pair along: the native kernel skipped both): a warp lists the
// flagged A and B row tiles in shared memory, the flagged tiles are numbered
// from those lists and dealt out one per CTA, and when they are fewer than the
// CTAs, each tile's K is split into S contiguous parts (S = CTAs / tiles, at
// most one part per 256-value stage). Each part leaves its FP32 sums in the
// workspace; per 32-row quarter of the tile, the epilogue warp that finishes
// last (a counter per quarter) adds the S parts in order p = 0 .. S-1, which
// fixes the result whatever the CTAs' timing, and writes the output.
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tcgen05.cuh"

namespace fp4bs {

namespace {

struct EmuParams {
    const uint8_t* a_scales;
    const uint8_t* b_scales;
    const float* a_sdec;
    const float* b_sdec;
    void* d;
    int64_t M, N, K;
    int accumulate;
    int* status;
    const uint8_t* rb_flags;  // nullable: after a rebias pass, compute only the flagged tiles (none set: return)
    int64_t rb_nflags;
    int use_list;             // number the flagged tiles from shared-memory lists (else scan every tile)
    int rb_pair;              // 2: the native kernel skipped 128 x 256 tiles, so a flagged B tile takes its pair along
    uint32_t* split_cnt;      // nullable: 4 counters per split tile, zero on entry, left zero
    float* split_buf;         // FP32 partial tiles, split_cap of them
    int64_t split_cap;
};

struct EmuCfg {
    static constexpr int BM = 128, BN = 128, BK = 256;
    static constexpr int DEC_WARPS = 16, FIRST_DEC_WARP = 2, EPI_WARPS = 4, FIRST_EPI_WARP = 18;
    static constexpr int RAW_STAGES = 3, DEC_STAGES = 3;
    static constexpr int RAW_A = BM * 128, RAW_B = BN * 128;     // FP4 codes, 128 B per row
    static constexpr int RAW_SFA = BM * 16, RAW_SFB = BN * 16;   // 16 scale blocks per row
    static constexpr uint32_t RAW_TX = RAW_A + RAW_B + RAW_SFA + RAW_SFB;
    static constexpr int DEC_A = BM * 128, DEC_B = BN * 128;     // BF16, K = 64 -> 128 B per row
    static constexpr int OFF_RAW_A = 0;
    static constexpr int OFF_RAW_B = OFF_RAW_A + RAW_STAGES * RAW_A;
    static constexpr int OFF_DEC_A = OFF_RAW_B + RAW_STAGES * RAW_B;
    static constexpr int OFF_DEC_B = OFF_DEC_A + DEC_STAGES * DEC_A;
    static constexpr int OFF_SFA = OFF_DEC_B + DEC_STAGES * DEC_B;
    static constexpr int OFF_SFB = OFF_SFA + RAW_STAGES * RAW_SFA;
    static constexpr int OFF_BAR = OFF_SFB + RAW_STAGES * RAW_SFB;
    static constexpr int NUM_BARS = 2 * RAW_STAGES + 2 * DEC_STAGES + 4 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    // lists of flagged A row tiles, unflagged A row tiles and flagged B row
    // tiles (16-bit tile indices), and their counts
    static constexpr int LIST_CAP = 4096;
    static constexpr int OFF_LIST = OFF_MISC + 32;
    static constexpr int SMEM_BYTES = OFF_LIST + 2 * LIST_CAP + 1024;
    static constexpr int THREADS = 32 * (FIRST_EPI_WARP + EPI_WARPS);
    static constexpr int TMEM_COLS = 512;  // two 128-column chunk accumulators + the running sum
    static constexpr int SUM_COL = 2 * BN;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Eight E2M1 codes (one 32-bit word, element i in nibble i) -> eight BF16
// values times the block scale. The E2M1 magnitudes {0,.5,1,1.5,2,3,4,6} have
// BF16 patterns 0x0000, 0x3F00, 0x3F80, 0x3FC0, 0x4000, 0x4040, 0x4080, 0x40C0:
// their high and low bytes are looked up with byte permutes indexed by the
// 3-bit magnitude codes, the code's sign bit goes to bit 15, and the packed
// BF16 multiply by the scale is exact (at most 6 significant bits).
__device__ __forceinline__ uint4 decode8(uint32_t w, __nv_bfloat162 scale2) {
    constexpr uint32_t HI_0123 = 0x3F3F3F00u, HI_4567 = 0x40404040u;
    constexpr uint32_t LO_0123 = 0xC0800000u, LO_4567 = 0xC0804000u;
    const uint32_t sel_a = w & 0x7777u, sel_b = (w >> 16) & 0x7777u;
    uint32_t hi_a = __byte_perm(HI_0123, HI_4567, sel_a), lo_a = __byte_perm(LO_0123, LO_4567, sel_a);
    uint32_t hi_b = __byte_perm(HI_0123, HI_4567, sel_b), lo_b = __byte_perm(LO_0123, LO_4567, sel_b);
    const uint32_t u = w & 0x88888888u;
    const uint32_t even = u << 4, odd = u;  // bit 7 of byte k: sign of element 2k / 2k+1
    hi_a |= __byte_perm(even, odd, 0x5140) & 0x80808080u;
    hi_b |= __byte_perm(even, odd, 0x7362) & 0x80808080u;
    uint32_t p[4] = {__byte_perm(lo_a, hi_a, 0x5140), __byte_perm(lo_a, hi_a, 0x7362),
                     __byte_perm(lo_b, hi_b, 0x5140), __byte_perm(lo_b, hi_b, 0x7362)};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&p[k]);
        v = __hmul2(v, scale2);
        p[k] = *reinterpret_cast<uint32_t*>(&v);
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

__device__ __forceinline__ __nv_bfloat162 ue5m3_bf16x2(uint32_t code) {
    const __nv_bfloat16 h = __float2bfloat16_rn(scale_decode_m3<15>(code));
    return __nv_bfloat162(h, h);
}

// Decode half h (one 16-byte raw chunk, 32 values) of an operand row's K = 64
// slice kk into the swizzled BF16 row of the decoded tile.
__device__ __forceinline__ void decode_half(const uint8_t* raw, const uint8_t* sf, uint8_t* dec, int r, int kk,
                                            int h) {
    const int sw = r & 7;
    {
        const int cr = 2 * kk + h;  // raw 16-byte chunk: values 32 cr .. 32 cr + 31 of the 256
        const uint4 codes = *reinterpret_cast<const uint4*>(raw + r * 128 + ((cr ^ sw) << 4));
        const uint16_t s2 =
            *reinterpret_cast<const uint16_t*>(sf + 512 * (cr >> 1) + 16 * (r & 31) + 4 * ((r >> 5) & 3) + 2 * (cr & 1));
        const __nv_bfloat162 s_lo = ue5m3_bf16x2(s2 & 0xFFu), s_hi = ue5m3_bf16x2(s2 >> 8);
        const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int oc = 4 * h + k;  // output 16-byte chunk (8 BF16 values) of the 128-byte row
            *reinterpret_cast<uint4*>(dec + r * 128 + ((oc ^ sw) << 4)) = decode8(w[k], k < 2 ? s_lo : s_hi);
        }
    }
}

// One unit of work: output tile (mb, nb), stages [kb0, kb1) of its K, and
// with split > 1 the partial tile it leaves (slot, part).
struct EmuItem {
    int64_t mb, nb;
    int kb0, kb1;
    int64_t tile_item;
    int part;
};

// The work of a launch. Without a rebias pass: every tile, all of K. After
// one: with lists, the flagged tiles numbered as all tiles of the flagged A
// row tiles (A-list order, B fastest) then the flagged B row tiles of the
// other A row tiles, each split into `split` parts; without lists (shapes too
// large for them), every tile scanned and the unflagged ones skipped.
struct EmuWork {
    int64_t num_m, num_n, count;
    int num_k, split;
    int64_t fa, fb;
    const uint16_t* l_fa;
    const uint16_t* l_nfa;
    const uint16_t* l_fb;
    const uint8_t* flags;
    int pair;

    template <bool LISTED>
    __device__ bool item(int64_t j, EmuItem& it) const {
        if (LISTED) {
            const int64_t i = j / split;
            it.part = (int)(j % split);
            it.tile_item = i;
            if (i < fa * num_n) {
                it.mb = l_fa[i / num_n];
                it.nb = i % num_n;
            } else {
                const int64_t i2 = i - fa * num_n;
                it.mb = l_nfa[i2 / fb];
                it.nb = l_fb[i2 % fb];
            }
            it.kb0 = (int)((int64_t)it.part * num_k / split);
            it.kb1 = (int)((int64_t)(it.part + 1) * num_k / split);
            return true;
        }
        it.mb = j % num_m;
        it.nb = j / num_m;
        it.kb0 = 0;
        it.kb1 = num_k;
        it.tile_item = j;
        it.part = 0;
        return flags == nullptr || rb_tile_flagged(flags, num_m, it.mb, it.nb / pair, pair);
    }
};

// LISTED: the rebias fallback with flagged-tile lists and K split (else the
// plain tile loop, skipping unflagged tiles when rb_flags is set).
template <bool OUT32, bool LISTED>
__global__ void __launch_bounds__(EmuCfg::THREADS, 1)
    gemm_ue5m3_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                      const EmuParams p) {
    using C = EmuCfg;
    // after a rebias pass: the native kernel took every output tile when no
    // row was flagged (uniform across the grid); otherwise this kernel computes
    // the flagged tiles only (every role skips the same others)
    if (p.rb_flags != nullptr) {
        pdl_wait();
        if (!rb_any_flag(p.rb_flags, p.rb_nflags)) return;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sb = tc::smem_u32(smem);
    auto bar = [&](int i) { return sb + C::OFF_BAR + 8u * i; };
    auto raw_full = [&](int s) { return bar(s); };
    auto raw_empty = [&](int s) { return bar(C::RAW_STAGES + s); };
    auto dec_full = [&](int s) { return bar(2 * C::RAW_STAGES + s); };
    auto dec_empty = [&](int s) { return bar(2 * C::RAW_STAGES + C::DEC_STAGES + s); };
    auto accf = [&](int a) { return bar(2 * C::RAW_STAGES + 2 * C::DEC_STAGES + a); };
    auto acce = [&](int a) { return bar(2 * C::RAW_STAGES + 2 * C::DEC_STAGES + 2 + a); };
    const uint32_t drain = bar(2 * C::RAW_STAGES + 2 * C::DEC_STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);

    const int64_t num_m = p.M / C::BM, num_n = p.N / C::BN, tiles = num_m * num_n;
    const int num_k = (int)(p.K / C::BK);
    const int64_t chunks_k = p.K / 64;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::RAW_STAGES; ++s) {
            tc::mbar_init(raw_full(s), 1);
            tc::mbar_init(raw_empty(s), C::DEC_WARPS);
        }
        for (int s = 0; s < C::DEC_STAGES; ++s) {
            tc::mbar_init(dec_full(s), C::DEC_WARPS);
            tc::mbar_init(dec_empty(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            tc::mbar_init(accf(a), 1);
            tc::mbar_init(acce(a), C::EPI_WARPS);
        }
        tc::mbar_init(drain, 1);
        tc::mbar_init_fence();
        tc::prefetch_tmap(&tmap_a);
        tc::prefetch_tmap(&tmap_b);
    }
    if (p.rb_flags == nullptr) pdl_wait();
    pdl_trigger();
    if (warp == 1) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    uint16_t* lists = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST);
    int* counts = reinterpret_cast<int*>(smem + C::OFF_MISC + 16);  // flagged A, flagged B row tiles
    if (LISTED && warp == C::FIRST_DEC_WARP) {
        // lists[0 .. fa): flagged A row tiles; lists[num_m .. 2 num_m - fa):
        // the others; lists[2 num_m ..): flagged B row tiles (ascending)
        int fa = 0, nfa = 0, fbn = 0;
        for (int64_t base = 0; base < num_m; base += 32) {
            const int64_t mb = base + lane;
            const bool in = mb < num_m, f = in && p.rb_flags[mb] != 0;
            const uint32_t bf = __ballot_sync(0xFFFFFFFFu, f), bn = __ballot_sync(0xFFFFFFFFu, in && !f);
            const uint32_t below = (1u << lane) - 1u;
            if (f) lists[fa + __popc(bf & below)] = (uint16_t)mb;
            if (in && !f) lists[num_m + nfa + __popc(bn & below)] = (uint16_t)mb;
            fa += __popc(bf);
            nfa += __popc(bn);
        }
        for (int64_t base = 0; base < num_n; base += 32) {
            const int64_t nb = base + lane;
            const bool f = nb < num_n && (p.rb_flags[num_m + nb] != 0 ||
                                          (p.rb_pair == 2 && p.rb_flags[num_m + (nb ^ 1)] != 0));
            const uint32_t bf = __ballot_sync(0xFFFFFFFFu, f);
            if (f) lists[2 * num_m + fbn + __popc(bf & ((1u << lane) - 1u))] = (uint16_t)nb;
            fbn += __popc(bf);
        }
        if (lane == 0) {
            counts[0] = fa;
            counts[1] = fbn;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    EmuWork wk;
    wk.num_m = num_m;
    wk.num_n = num_n;
    wk.num_k = num_k;
    wk.flags = p.rb_flags;
    wk.pair = p.rb_pair;
    wk.split = 1;
    wk.count = tiles;
    wk.fa = wk.fb = 0;
    wk.l_fa = lists;
    wk.l_nfa = lists + num_m;
    wk.l_fb = lists + 2 * num_m;
    if (LISTED) {
        wk.fa = counts[0];
        wk.fb = counts[1];
        const int64_t f = wk.fa * num_n + (num_m - wk.fa) * wk.fb;  // >= 1: some flag is set
        int64_t split = 1;
        if (p.split_buf != nullptr && f < gridDim.x) {
            split = gridDim.x / f;
            if (split > num_k) split = num_k;
            if (split * f > p.split_cap) split = p.split_cap / f;
            if (split < 1) split = 1;
        }
        wk.split = (int)split;
        wk.count = f * split;
    }

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int64_t j = blockIdx.x; j < wk.count && ok; j += gridDim.x) {
                EmuItem w;
                if (!wk.template item<LISTED>(j, w)) continue;
                const int64_t mb = w.mb, nb = w.nb;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const int s = (int)(it % C::RAW_STAGES);
                    const uint32_t ph = (it / C::RAW_STAGES) & 1u;
                    if (!tc::mbar_wait(raw_empty(s), ph ^ 1u, p.status)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(raw_full(s), C::RAW_TX);
                    tc::tma_load_2d(sb + C::OFF_RAW_A + s * C::RAW_A, &tmap_a, kb * 128, (int32_t)(mb * C::BM),
                                    raw_full(s));
                    tc::tma_load_2d(sb + C::OFF_RAW_B + s * C::RAW_B, &tmap_b, kb * 128, (int32_t)(nb * C::BN),
                                    raw_full(s));
                    tc::bulk_load(sb + C::OFF_SFA + s * C::RAW_SFA, p.a_scales + 512 * (mb * chunks_k + 4 * kb),
                                  C::RAW_SFA, raw_full(s));
                    tc::bulk_load(sb + C::OFF_SFB + s * C::RAW_SFB, p.b_scales + 512 * (nb * chunks_k + 4 * kb),
                                  C::RAW_SFB, raw_full(s));
                }
            }
        }
    } else if (warp >= C::FIRST_DEC_WARP && warp < C::FIRST_DEC_WARP + C::DEC_WARPS) {
        // ------------------------------------------------------------ decoders
        const int t = threadIdx.x - 32 * C::FIRST_DEC_WARP;  // 0 .. 511
        const int op = t >> 8, h = (t >> 7) & 1, r = t & 127;  // operand (A/B), raw chunk half, row
        uint32_t it_raw = 0, it_dec = 0;
        bool ok = true;
        for (int64_t j = blockIdx.x; j < wk.count && ok; j += gridDim.x) {
            EmuItem w;
            if (!wk.template item<LISTED>(j, w)) continue;
            for (int kb = w.kb0; kb < w.kb1 && ok; ++kb, ++it_raw) {
                const int rs = (int)(it_raw % C::RAW_STAGES);
                if (!tc::mbar_wait(raw_full(rs), (it_raw / C::RAW_STAGES) & 1u, p.status)) {
                    ok = false;
                    break;
                }
                const uint8_t* raw = op ? smem + C::OFF_RAW_B + rs * C::RAW_B : smem + C::OFF_RAW_A + rs * C::RAW_A;
                const uint8_t* sf = op ? smem + C::OFF_SFB + rs * C::RAW_SFB : smem + C::OFF_SFA + rs * C::RAW_SFA;
                for (int kk = 0; kk < 4; ++kk, ++it_dec) {
                    const int ds = (int)(it_dec % C::DEC_STAGES);
                    if (!tc::mbar_wait(dec_empty(ds), ((it_dec / C::DEC_STAGES) & 1u) ^ 1u, p.status)) {
                        ok = false;
                        break;
                    }
                    decode_half(raw, sf, op ? smem + C::OFF_DEC_B + ds * C::DEC_B : smem + C::OFF_DEC_A + ds * C::DEC_A,
                                r, kk, h);
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(dec_full(ds));
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(raw_empty(rs));
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = tc::idesc_bf16(C::BM, C::BN);
            uint32_t it_dec = 0, chunk = 0;
            bool ok = true;
            for (int64_t j = blockIdx.x; j < wk.count && ok; j += gridDim.x) {
                EmuItem w;
                if (!wk.template item<LISTED>(j, w)) continue;
                for (int kb = w.kb0; kb < w.kb1 && ok; ++kb, ++chunk) {
                    // one raw stage = one accumulator chunk
                    const int buf = (int)(chunk & 1u);
                    if (!tc::mbar_wait(acce(buf), ((chunk >> 1) & 1u) ^ 1u, p.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t d_tmem = tmem + (uint32_t)(buf * C::BN);
                    for (int kk = 0; kk < 4; ++kk, ++it_dec) {
                        const int ds = (int)(it_dec % C::DEC_STAGES);
                        if (!tc::mbar_wait(dec_full(ds), (it_dec / C::DEC_STAGES) & 1u, p.status)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t a_s = sb + C::OFF_DEC_A + ds * C::DEC_A;
                        const uint32_t b_s = sb + C::OFF_DEC_B + ds * C::DEC_B;
#pragma unroll
                        for (int k16 = 0; k16 < 4; ++k16)
                            tc::mma_bf16(d_tmem, tc::kmajor_sw128_desc(a_s + 32 * k16),
                                         tc::kmajor_sw128_desc(b_s + 32 * k16), IDESC, (kk | k16) != 0 ? 1u : 0u);
                        tc::commit(dec_empty(ds));
                    }
                    if (ok) tc::commit(accf(buf));
                }
            }
            tc::commit(drain);
            tc::mbar_wait(drain, 0, p.status);
        }
    } else if (warp >= C::FIRST_EPI_WARP) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // the TMEM lane quadrant this warp may access
        const float alpha = __fmul_rn(*p.a_sdec, *p.b_sdec);
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t chunk = 0;
        bool ok = true;
        // alpha * the 32 sums of row m, columns n0 .. n0 + 31, to the output
        auto write_out = [&](const uint32_t (&rs)[32], int64_t m, int64_t n0) {
            if (OUT32) {
                float* dst = static_cast<float*>(p.d) + m * p.N + n0;
#pragma unroll
                for (int v = 0; v < 32; v += 4) {
                    float4 o = make_float4(__fmul_rn(__uint_as_float(rs[v]), alpha),
                                           __fmul_rn(__uint_as_float(rs[v + 1]), alpha),
                                           __fmul_rn(__uint_as_float(rs[v + 2]), alpha),
                                           __fmul_rn(__uint_as_float(rs[v + 3]), alpha));
                    if (p.accumulate) {
                        const float4 old = *reinterpret_cast<const float4*>(dst + v);
                        o.x = __fadd_rn(o.x, old.x);
                        o.y = __fadd_rn(o.y, old.y);
                        o.z = __fadd_rn(o.z, old.z);
                        o.w = __fadd_rn(o.w, old.w);
                    }
                    *reinterpret_cast<float4*>(dst + v) = o;
                }
            } else {
                uint16_t* dst = static_cast<uint16_t*>(p.d) + m * p.N + n0;
#pragma unroll
                for (int v = 0; v < 32; v += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const __nv_bfloat162 hh =
                            __floats2bfloat162_rn(__fmul_rn(__uint_as_float(rs[v + 2 * k]), alpha),
                                                  __fmul_rn(__uint_as_float(rs[v + 2 * k + 1]), alpha));
                        w[k] = *reinterpret_cast<const uint32_t*>(&hh);
                    }
                    *reinterpret_cast<uint4*>(dst + v) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        };
        const bool split = LISTED && wk.split > 1;
        for (int64_t j = blockIdx.x; j < wk.count && ok; j += gridDim.x) {
            EmuItem w;
            if (!wk.template item<LISTED>(j, w)) continue;
            const int64_t mb = w.mb, nb = w.nb;
            const int64_t m = mb * C::BM + q * 32 + lane;
            // this part's FP32 sums of row m of the tile (split only)
            float* part_row = split ? p.split_buf + ((size_t)j * C::BM + (size_t)(q * 32 + lane)) * C::BN : nullptr;
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++chunk) {
                const int buf = (int)(chunk & 1u);
                if (!tc::mbar_wait(accf(buf), (chunk >> 1) & 1u, p.status)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const bool first = kb == w.kb0, last = kb == w.kb1 - 1;
#pragma unroll 1
                for (int c = 0; c < C::BN; c += 32) {
                    uint32_t rc[32], rs[32];
                    tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)(buf * C::BN + c), rc);
                    if (!first) tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)(C::SUM_COL + c), rs);
                    tc::tmem_ld_wait();
                    if (first) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) rs[i] = rc[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float a0, a1;
                            f2_unpack(f2_add(f2_pack(__uint_as_float(rs[i]), __uint_as_float(rs[i + 1])),
                                             f2_pack(__uint_as_float(rc[i]), __uint_as_float(rc[i + 1]))),
                                      a0, a1);
                            rs[i] = __float_as_uint(a0);
                            rs[i + 1] = __float_as_uint(a1);
                        }
                    }
                    if (!last) {
                        tc::tmem_st_32x32b_x32(lane_base + (uint32_t)(C::SUM_COL + c), rs);
                        continue;
                    }
                    if (split) {
#pragma unroll
                        for (int v = 0; v < 32; v += 4)
                            __stcg(reinterpret_cast<uint4*>(part_row + c + v),
                                   make_uint4(rs[v], rs[v + 1], rs[v + 2], rs[v + 3]));
                        continue;
                    }
                    // last chunk of the tile: alpha * sum to the output row m, columns nb * BN + c ..
                    write_out(rs, m, nb * C::BN + c);
                }
                // the running sum is written before this warp's next loads of it
                if (!last) tc::tmem_st_wait();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(acce(buf));
            }
            if (!ok || !split) continue;
            // split: this warp's 32 rows of part w.part are in the workspace;
            // the warp that counts the last part of this quarter adds the parts
            // in order p = 0 .. split - 1 and writes the output rows
            __threadfence();
            __syncwarp();
            uint32_t prev = 0;
            if (lane == 0) prev = atomicAdd(p.split_cnt + 4 * w.tile_item + q, 1u);
            prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
            if (prev != (uint32_t)(wk.split - 1)) continue;
            __threadfence();
            const float* row0 =
                p.split_buf + ((size_t)(w.tile_item * wk.split) * C::BM + (size_t)(q * 32 + lane)) * C::BN;
#pragma unroll 1
            for (int c = 0; c < C::BN; c += 32) {
                uint32_t rs[32];
#pragma unroll
                for (int v = 0; v < 32; v += 4) {
                    const uint4 u = __ldcg(reinterpret_cast<const uint4*>(row0 + c + v));
                    rs[v] = u.x;
                    rs[v + 1] = u.y;
                    rs[v + 2] = u.z;
                    rs[v + 3] = u.w;
                }
                for (int pp = 1; pp < wk.split; ++pp) {
                    const float* row = row0 + (size_t)pp * C::BM * C::BN;
#pragma unroll
                    for (int v = 0; v < 32; v += 4) {
                        const float4 u = __ldcg(reinterpret_cast<const float4*>(row + c + v));
                        rs[v] = __float_as_uint(__fadd_rn(__uint_as_float(rs[v]), u.x));
                        rs[v + 1] = __float_as_uint(__fadd_rn(__uint_as_float(rs[v + 1]), u.y));
                        rs[v + 2] = __float_as_uint(__fadd_rn(__uint_as_float(rs[v + 2]), u.z));
                        rs[v + 3] = __float_as_uint(__fadd_rn(__uint_as_float(rs[v + 3]), u.w));
                    }
                }
                write_out(rs, m, nb * C::BN + c);
            }
            if (lane == 0) p.split_cnt[4 * w.tile_item + q] = 0u;  // zero again for the next call
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <bool OUT32>
cudaError_t run_emu(const GemmJob& j, cudaStream_t st) {
    CUtensorMap ta, tb;
    if (!make_tmap_u8_sw128(&ta, j.a_codes, j.M, j.K / 2, EmuCfg::BM)) return cudaErrorInvalidValue;
    if (!make_tmap_u8_sw128(&tb, j.b_codes, j.N, j.K / 2, EmuCfg::BN)) return cudaErrorInvalidValue;
    const int64_t num_m = j.M / EmuCfg::BM, num_n = j.N / EmuCfg::BN;
    const bool rb = j.rb_emulated && j.rb_flags != nullptr;
    // the flagged-tile lists hold 2 num_m + num_n 16-bit entries
    const int use_list = rb && 2 * num_m + num_n <= EmuCfg::LIST_CAP && num_m < 65536 && num_n < 65536;
    EmuParams p{j.a_scales, j.b_scales, j.a_sdec, j.b_sdec, j.d, j.M, j.N, j.K, j.accumulate, j.status,
                rb ? j.rb_flags : nullptr, j.rb_nflags, use_list, j.N % 256 == 0 ? 2 : 1,
                use_list ? j.split_cnt : nullptr,
                use_list ? j.split_buf : nullptr, use_list ? j.split_cap : 0};
    auto kern = use_list ? gemm_ue5m3_kernel<OUT32, true> : gemm_ue5m3_kernel<OUT32, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, EmuCfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (j.M / EmuCfg::BM) * (j.N / EmuCfg::BN);
    const int grid = (int)(tiles < num_sms() ? tiles : num_sms());
    (void)launch_pdl(kern, grid, EmuCfg::THREADS, EmuCfg::SMEM_BYTES, st, ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_ue5m3(const GemmJob& j, cudaStream_t st) {
    if (j.out_fp32) return run_emu<true>(j, st);
    return run_emu<false>(j, st);
}

}  // namespace fp4bs
