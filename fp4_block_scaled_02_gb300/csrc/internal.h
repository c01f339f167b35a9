// internal.h -- host-side interface between the C-ABI layer (api.cu) and the
// kernel translation units (quantize.cu, gemm_nvfp4.cu, gemm_ue5m3.cu).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fp4bs.h"

namespace fp4bs {

// Programmatic dependent launch. Every kernel of the library is launched with
// launch_pdl, so the stream may start it while the kernel before it is still
// finishing; the kernel calls pdl_wait() before its first access to global
// memory (and before it allocates tensor memory), which returns once the
// previous grid has completed and its writes are visible, and then pdl_trigger()
// so the next kernel can be scheduled onto SMs as they free up. Only on-chip
// setup (shared memory, mbarrier init, tensor-map prefetch) may precede the wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
    pdl_wait();
    pdl_trigger();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// One quantizer launch, after validation. Operand shape is rows x cols of the
// INPUT; `colwise` makes the operand its transpose.
struct QuantJob {
    int scale_fmt;      // kFmtE4M3 / kFmtUE5M3 / kFmtUE8M0
    int block;          // FP4_BLOCK_*
    int sr;             // stochastic rounding
    int colwise;
    int rht;
    int held;           // held-amax tensor scale (also set for a given amax)
    int refresh;        // held: this step refreshes the amax
    int given;          // the amax is the state's, computed ahead (FP4_TSCALE_GIVEN)
    int per_row;        // one tensor scale per operand row (FP4_TSCALE_ROW), s_dec[rows]
    float target_T;
    uint32_t tensor_id;
    uint64_t seed;
    uint64_t step;
    const uint16_t* in;
    int64_t rows, cols;
    int64_t ld;         // input row stride in elements (>= cols, a multiple of 8)
    // primary output (the operand) and, for 16x16, the optional transposed one
    uint8_t* codes;
    uint8_t* scales;
    float* s_dec;
    int layout;         // FP4_LAYOUT_*
    uint8_t* codes_t;
    uint8_t* scales_t;
    float* s_dec_t;
    int layout_t;
    fp4_amax_state_t* state;
    uint64_t* counters;  // nullable
    float* partials;     // amax-pass workspace
    int* status;         // device status word
};

// Largest number of amax partials (one per CTA of the amax pass).
constexpr int kMaxAmaxPartials = 2048;

int num_sms();
cudaError_t launch_quantize(const QuantJob& job, cudaStream_t stream);
// Rowwise (jr) and colwise (jc) quantization of the same input in one pass
// (T % 128 == 0, C % 128 == 0, tensor-core scale layout, same format, rounding
// and tensor-scale mode; each job's partials hold kMaxAmaxPartials floats).
cudaError_t launch_quantize_dual(const QuantJob& jr, const QuantJob& jc, cudaStream_t stream);
// Number of amax partials the amax pass of `job` writes (0: no amax pass).
int amax_partials_needed(const QuantJob& job);
// Tensor amax records ahead of quantization: the plain amax of the T x C BF16
// tensor into st_plain and/or the post-RHT colwise amax (rht) or the plain one
// (!rht) into st_col; null records are skipped. partials: 2 * kMaxAmaxPartials
// floats. status: the device status word (bounded waits).
cudaError_t launch_tensor_amax(const uint16_t* in, int64_t T, int64_t C, int64_t ld, fp4_amax_state_t* st_plain,
                               fp4_amax_state_t* st_col, bool rht, uint64_t step, float* partials, int* status,
                               cudaStream_t stream);

struct DequantJob {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* s_dec;
    int s_dec_rows;     // s_dec holds one float per row
    int64_t rows, cols;
    int scale_fmt, block_k, layout;
    void* out;
    int out_fp32;
};
cudaError_t launch_dequantize(const DequantJob& job, cudaStream_t stream);

// Block-scaled GEMM D = alpha * A * B^T over K-major quantized operands.
struct GemmJob {
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    const float* a_sdec;
    int a_sdec_rows;    // a_sdec holds one float per row of A
    const uint8_t* b_codes;
    const uint8_t* b_scales;
    const float* b_sdec;
    int64_t M, N, K;
    int scale_fmt;
    void* d;
    int out_fp32;
    int accumulate;
    int* status;
    // UE5M3 operands rebiased onto E4M3 scales (launch_rebias_ue5m3): the scale
    // pointers above hold the E4M3 bytes and a_off / b_off the per-row power-of-
    // two offsets. rb_flags[0 .. rb_nflags) are the rebias pass's per-tile
    // "does not fit" bytes: the rebiased kernel returns at once if any is set,
    // the emulated kernel (rb_emulated) if none is.
    const int8_t* a_off;
    const int8_t* b_off;
    const uint8_t* rb_flags;
    int64_t rb_nflags;
    int rb_emulated;
    // emulated fallback after a rebias pass: workspace for splitting the
    // flagged tiles' K (4 counters per split tile, zero on entry; split_cap
    // FP32 128 x 128 partial tiles); null: no split
    uint32_t* split_cnt;
    float* split_buf;
    int64_t split_cap;
};
// Split tiles of the emulated fallback (bounds the counters and partial
// tiles the workspace holds; at least the SM count).
constexpr int64_t kEmuSplitMaxTiles = 256;
cudaError_t launch_gemm_nvfp4(const GemmJob& job, cudaStream_t stream);
cudaError_t launch_gemm_ue5m3(const GemmJob& job, cudaStream_t stream);
// Rewrite the UE5M3 block scales of A (M rows) and B (N rows), tensor-core
// layout with K / 16 scales per row, as E4M3 scales times a per-row power of
// two: s = e4m3_out * 2^off[row] exactly. flags[t] (one byte per 128-row tile,
// A's tiles first, M / 128 + N / 128 in all) is set to 1 if a row of tile t
// has scales spanning more binades than E4M3 holds, else to 0.
// It also zeroes n_clear words at `clear` (the emulated fallback's split counters).
cudaError_t launch_rebias_ue5m3(const uint8_t* a_scales, int64_t M, const uint8_t* b_scales, int64_t N, int64_t K,
                                uint8_t* a_out, uint8_t* b_out, int8_t* a_off, int8_t* b_off, uint8_t* flags,
                                uint32_t* clear, int64_t n_clear, cudaStream_t stream);
// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// completes; after limit_ns the wait records FP4_ERR_DEVICE_TIMEOUT in *status
// and the kernel returns.
cudaError_t launch_wait_selftest(uint64_t limit_ns, int* status, cudaStream_t stream);
// out[i] = the quantizer's RN(in[i] / 6) for i < n (diagnostic).
cudaError_t launch_div6_selftest(const float* in, float* out, int64_t n, cudaStream_t stream);
// Rebiased UE5M3 products: whether output tile (mb, nb) -- 128 rows of A, and
// b_tiles_per_tile 128-row tiles of B -- holds a row that did not fit one E4M3
// offset (flags: one byte per 128-row tile, A's tiles first). Such tiles are
// computed by the emulated kernel, all others by the native one.
__device__ __forceinline__ bool rb_tile_flagged(const uint8_t* flags, int64_t a_tiles, int64_t mb, int64_t nb,
                                                int b_tiles_per_tile) {
    bool bad = flags[mb] != 0;
    for (int h = 0; h < b_tiles_per_tile; ++h) bad |= flags[a_tiles + nb * b_tiles_per_tile + h] != 0;
    return bad;
}

// Any of the n bytes at f nonzero (every thread of the calling warp gets the answer).
__device__ __forceinline__ bool rb_any_flag(const uint8_t* f, int64_t n) {
    bool any = false;
    for (int64_t i = threadIdx.x & 31; i < n; i += 32) any |= f[i] != 0;
    return __any_sync(0xFFFFFFFFu, any) != 0;
}

// 2-D byte-matrix TMA descriptor with 128-byte rows per box row and 128-byte
// swizzling (defined in gemm_nvfp4.cu).
bool make_tmap_u8_sw128(CUtensorMap* map, const void* base, int64_t rows, int64_t row_bytes, int box_rows);
// 2-D BF16 matrix tensor map with box_rows x box_cols tiles, unswizzled or with
// the 128-byte swizzle; rows lie ld elements apart (ld = 0: cols) (defined in
// gemm_nvfp4.cu).
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows, int box_cols,
                       bool swizzle128 = false, int64_t ld = 0);

}  // namespace fp4bs
