/*
 * fp4bs.h -- C ABI of the GB300 FP4 block-scaled quantized linear library
 * (libfp4bs.so, sm_103a).
 *
 * The library implements the data-parallel hot path of FP4 pretraining as
 * "Pretraining Large Language Models with NVFP4" (arXiv 2509.25149) and the
 * UE5M3 block-scale paper summarised at arXiv 2609.02846 describe it:
 *   - a quantizer: tensor amax -> FP32 tensor scale (App. B.1; or a held amax
 *     refreshed every N steps, or one scale per operand row, the finer
 *     granularity B.1 suggests), per-block scale (App. B.2) in E4M3, UE5M3 or
 *     UE8M0, E2M1 conversion with round-to-nearest-even or stochastic rounding
 *     (App. B.3, section 4.4), optional 16x16 random Hadamard transform on the
 *     Wgrad operands (section 4.2, App. C), 2D 16x16 weight scaling (4.3);
 *   - the three block-scaled FP4 GEMMs of a linear layer (section 4.1, Fig. 5:
 *     Fprop, Dgrad, Wgrad) on tcgen05 tensor cores (App. B.3) for NVFP4 and
 *     MXFP4 operands (section A3), and for UE5M3 scales, which no tensor core
 *     reads, a software-emulated path and an exact rebias onto E4M3 scales
 *     that runs on the native MMA (fp4_gemm_ws).
 *
 * Conventions for every entry point:
 *   - Ownership: the caller allocates and frees every buffer (inputs, codes,
 *     scales, tensor scales, counters, held-amax state, workspace, outputs).
 *     The library never allocates device memory. Pointers are DEVICE pointers
 *     unless stated otherwise and must be 16-byte aligned.
 *   - Execution: work is enqueued on the given CUDA stream (a cudaStream_t
 *     passed as void*; NULL = legacy default stream) and the call returns before
 *     it completes. Argument checks run synchronously on the host first: a call
 *     that fails them returns an error and enqueues nothing.
 *   - Device-side errors (a bounded wait that timed out, a given amax record
 *     that is not valid) are recorded in a per-device status word read by
 *     fp4_device_status().
 *   - Kernels are launched with programmatic dependent launch: each may start
 *     while the previous kernel on the stream finishes, and waits for it
 *     (griddepcontrol.wait) before touching global memory, so stream order
 *     holds for all data.
 *   - Shapes: an operand is `rows x cols` with `cols` the dot-product dimension
 *     (K-major). BF16 inputs are row-major with their rows `ld` elements apart
 *     (ld >= cols and a multiple of 8, so every row starts 16-byte aligned; ld
 *     is not checked for empty inputs): a column slice of a wider buffer is
 *     quantized in place.
 */
#ifndef FP4BS_H
#define FP4BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP4_OK = 0,
    FP4_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, inconsistent options */
    FP4_ERR_UNSUPPORTED = 2,   /* valid but not implemented combination */
    FP4_ERR_SHAPE = 3,         /* dimension not a multiple the path needs */
    FP4_ERR_ALIGNMENT = 4,     /* pointer not 16-byte aligned */
    FP4_ERR_STATE = 5,         /* a given amax record (FP4_TSCALE_GIVEN) was not valid (device status) */
    FP4_ERR_CUDA = 6,          /* a CUDA runtime call failed */
    FP4_ERR_DEVICE_TIMEOUT = 7,/* a bounded device-side wait gave up */
    FP4_ERR_WORKSPACE = 8      /* workspace missing or too small */
} fp4_status_t;

/* Block-scale formats.
 *   E4M3  : NVFP4 (App. B.1-B.2): OCP E4M3, max 448, one FP32 tensor scale.
 *   UE5M3 : unsigned E5M3, bias 15, max 114688 (0xFE; 0xFF reserved), with a
 *           current or held tensor scale (UE5M3 page, method details).
 *   UE8M0 : MXFP4 (section A3): power of two 2^(code-127), no tensor scale. */
typedef enum { FP4_SCALE_E4M3 = 0, FP4_SCALE_UE5M3 = 1, FP4_SCALE_UE8M0 = 2 } fp4_scale_fmt_t;

/* Block shapes: 1x16 along the dot dimension (activations, gradients),
 * 16x16 (weights, section 4.3), 1x32 (MXFP4, section A3). */
typedef enum { FP4_BLOCK_1x16 = 0, FP4_BLOCK_16x16 = 1, FP4_BLOCK_1x32 = 2 } fp4_block_t;

typedef enum { FP4_ROUND_RNE = 0, FP4_ROUND_SR = 1 } fp4_round_t;

/* Tensor scale: per-call amax (App. B.1: CURRENT), held amax refreshed when
 * step % refresh_every == 0 or when the held state is not valid yet (UE5M3
 * page: refresh every 50 steps; other steps use the held amax: HELD), or the
 * amax a previous fp4_tensor_amax call left in the state record (GIVEN: the
 * same bytes as CURRENT without the call's own amax pass). ROW: current
 * scaling per operand row, the finer granularity App. B.1 suggests to save the
 * extra memory pass: row r of the operand gets s_enc,G(r) = 6 T / amax_r from
 * its own amax, computed in the same single pass that converts it, and
 * s_dec,G(r) goes to s_dec_global[r]. ROW needs E4M3 scales, 1x16 blocks,
 * ROWWISE without RHT, an output with sdec_per_row set (s_dec_global holding
 * rows floats) and no workspace; fp4_quantize_dual does not take it. */
typedef enum {
    FP4_TSCALE_CURRENT = 0,
    FP4_TSCALE_HELD = 1,
    FP4_TSCALE_GIVEN = 2,
    FP4_TSCALE_ROW = 3
} fp4_tscale_t;

/* ROWWISE: the operand is the input itself (blocks run along its columns).
 * COLWISE: the operand is the input's transpose (blocks run along the input's
 * rows); this is how Wgrad consumes X and dY (section 4.3). */
typedef enum { FP4_ORIENT_ROWWISE = 0, FP4_ORIENT_COLWISE = 1 } fp4_orient_t;

/* Scale storage. PLAIN: row-major rows x (cols / block) bytes. TCGEN05: the
 * tensor-core scale-factor layout; rows must be a multiple of 128 and
 * cols / block a multiple of 4. Chunk (rt, kt) of 128 rows x 4 blocks is
 * 512 bytes at offset 512 * (rt * (cols/block/4) + kt); row r, block j of a
 * chunk is at byte 16 * (r % 32) + 4 * ((r % 128) / 32) + (j % 4). */
typedef enum { FP4_LAYOUT_PLAIN = 0, FP4_LAYOUT_TCGEN05 = 1 } fp4_scale_layout_t;

/* Quantizer options (all fields read by fp4_quantize). */
typedef struct {
    int32_t scale_fmt;       /* fp4_scale_fmt_t */
    int32_t block;           /* fp4_block_t; UE8M0 <=> 1x32 */
    int32_t round;           /* fp4_round_t; SR for gradients only (section 4.4) */
    int32_t orient;          /* fp4_orient_t */
    int32_t rht;             /* nonzero: 16-point RHT along the block dimension;
                                COLWISE 1x16 only (section 4.2: Wgrad inputs) */
    int32_t tscale;          /* fp4_tscale_t (ignored for UE8M0) */
    float target_T;          /* scale target: 448 for E4M3; 448 or 2048 for UE5M3 */
    uint32_t refresh_every;  /* held mode refresh period (50) */
    uint32_t tensor_id;      /* keys the SR random stream; 0xFFFFFFFF is reserved */
    int32_t scale_layout;    /* fp4_scale_layout_t for the outputs */
    int32_t emit_transpose;  /* 16x16 only: also write the transposed operand */
    int32_t reserved;        /* must be 0 */
    uint64_t seed;           /* RNG seed: SR bits and the RHT sign vector */
    uint64_t step;           /* training step: SR stream and held-amax refresh */
} fp4_quant_params_t;

/* A quantized operand: rows x cols E2M1 codes, K-major, element 2i of a row in
 * the low nibble of byte i; block scales; and the FP32 decode tensor scale
 * s_dec,G (App. B.1; 1.0 for UE8M0), one for the tensor or one per row. */
typedef struct {
    uint8_t* codes;          /* rows * cols / 2 bytes */
    uint8_t* scales;         /* rows * cols / block_k bytes */
    float* s_dec_global;     /* one float, or rows floats with sdec_per_row */
    int64_t rows;
    int64_t cols;            /* dot-product dimension */
    int32_t scale_fmt;       /* fp4_scale_fmt_t */
    int32_t block_k;         /* 16 or 32: scale block length along cols */
    int32_t scale_layout;    /* fp4_scale_layout_t */
    int32_t sdec_per_row;    /* 0: one s_dec,G; 1: s_dec_global[r] per row
                                (FP4_TSCALE_ROW outputs; E4M3 only) */
} fp4_tensor_t;

/* Held-amax record of one tensor (device memory, 16 bytes, zero-initialised by
 * the caller before first use). */
typedef struct {
    float amax_held;
    int32_t valid;
    uint64_t last_refresh_step;
} fp4_amax_state_t;

/* Sizes of the codes and scales buffers fp4_quantize writes for an input of
 * rows x cols (for COLWISE the operand is cols x rows). Host only.
 * fp4_quantized_bytes is the same call under its other name. */
fp4_status_t fp4_quantized_sizes(const fp4_quant_params_t* p, int64_t rows, int64_t cols,
                                 size_t* codes_bytes, size_t* scales_bytes);
fp4_status_t fp4_quantized_bytes(const fp4_quant_params_t* p, int64_t rows, int64_t cols,
                                 size_t* codes_bytes, size_t* scales_bytes);

/* Device workspace bytes fp4_quantize needs (the per-CTA amax partials of the
 * amax pass); 0 when no amax pass runs (UE8M0, FP4_TSCALE_GIVEN, FP4_TSCALE_ROW).
 * Host only. */
size_t fp4_workspace_bytes(const fp4_quant_params_t* p, int64_t rows, int64_t cols);

/* Quantize a row-major BF16 input `in_bf16` (rows x cols, rows ld elements
 * apart) into `out` ("Pretraining LLMs with NVFP4", App. B.1-B.3; sections
 * 4.2-4.4). ld < cols or not a multiple of 8: FP4_ERR_SHAPE.
 *   out      : operand descriptor (rows/cols = operand shape, i.e. transposed
 *              for COLWISE); codes, scales and s_dec_global are written.
 *   out_t    : 16x16 with emit_transpose: the transposed operand (cols x rows)
 *              with the same codes and scales transposed (section 4.3); else NULL.
 *   state    : held-amax record (FP4_TSCALE_HELD), else NULL. Refresh steps, and
 *              steps that find it not valid yet, compute the amax and write it;
 *              other steps use it (their amax pass returns at once). With
 *              FP4_TSCALE_GIVEN: the record fp4_tensor_amax wrote, read and not
 *              changed (no amax pass, ws may be NULL); a record that is not
 *              valid when the kernel runs writes nothing and leaves
 *              FP4_ERR_STATE in the device status word.
 *   counters : NULL or 4 device uint64: elem_sat, elem_underflow, scale_sat,
 *              scale_underflow; the call ADDS its counts (the caller zeroes).
 *   ws       : device workspace of fp4_workspace_bytes() bytes (any content).
 * Shapes: block dimension a multiple of the block length; 16x16 needs both
 * dimensions multiples of 16; TCGEN05 layout needs operand rows % 128 == 0 and
 * operand cols % (4 * block) == 0. rows == 0 or cols == 0 is a no-op. */
fp4_status_t fp4_quantize(const fp4_quant_params_t* p, const void* in_bf16, int64_t rows, int64_t cols, int64_t ld,
                          const fp4_tensor_t* out, const fp4_tensor_t* out_t, fp4_amax_state_t* state,
                          uint64_t* counters, void* ws, size_t ws_bytes, void* stream);

/* Rowwise and colwise quantization of ONE input in a single pass: the two
 * operands a linear layer takes from X (or dY) -- `out_row` (rows x cols,
 * blocks along cols, for Fprop/Dgrad) and `out_col` (cols x rows, blocks along
 * rows, optional RHT, for Wgrad). Each output, its tensor scale, held state and
 * counters are bit-identical to a separate fp4_quantize call with p_row /
 * p_col ("Pretraining LLMs with NVFP4", App. B; sections 4.2-4.4); the input is
 * read once per pass instead of twice. Requirements: p_row ROWWISE and p_col
 * COLWISE, both 1x16, same scale format (E4M3 or UE5M3), rounding mode,
 * tensor-scale mode and step, TCGEN05 scale layout; rows and cols multiples
 * of 128; ws at least 2 * fp4_workspace_bytes() bytes. */
fp4_status_t fp4_quantize_dual(const fp4_quant_params_t* p_row, const fp4_quant_params_t* p_col, const void* in_bf16,
                               int64_t rows, int64_t cols, int64_t ld, const fp4_tensor_t* out_row,
                               const fp4_tensor_t* out_col,
                               fp4_amax_state_t* state_row, fp4_amax_state_t* state_col, uint64_t* counters_row,
                               uint64_t* counters_col, void* ws, size_t ws_bytes, void* stream);

/* fp4_quantize without a workspace argument, for callers that cannot
 * allocate device memory at all (for example a plug-in inside another
 * framework's engine that owns the memory budget, or a latency-critical loop
 * that must never reach an allocator). The papers have no counterpart: this is
 * a library convenience. The amax partials go to a library-owned 8 KB device
 * array (2048 floats, held by every GPU that loads the library until exit)
 * instead of a caller workspace; calls needing more partials than it holds
 * are rejected with FP4_ERR_WORKSPACE (no shape does: the amax pass caps its
 * partials at 2048). The first call on each device that runs an amax pass
 * (current scaling or held amax) looks up the array's device address, so make
 * it before any stream capture; calls with no amax pass (UE8M0, given amax,
 * per-row scales) never use the array. All calls share the array: calls that
 * overlap on the GPU race on it. Everything else is as for fp4_quantize, and
 * no device memory is allocated or freed. */
fp4_status_t fp4_quantize_noalloc(const fp4_quant_params_t* p, const void* in_bf16, int64_t rows, int64_t cols,
                                  int64_t ld, const fp4_tensor_t* out, const fp4_tensor_t* out_t,
                                  fp4_amax_state_t* state, uint64_t* counters, void* stream);

/* Tensor amax ahead of quantization (App. B.1: the amax that current scaling
 * takes in its first memory pass), as a separate call so that it can run on
 * another stream while other work proceeds. Computes the amax of the operand
 * that p describes (max |x|, or max |RHT x| along tokens for a colwise operand
 * with rht) and writes *out = {amax, valid = 1, last_refresh_step = p->step}
 * when the stream reaches it. A later fp4_quantize with tscale
 * FP4_TSCALE_GIVEN and state = out then quantizes exactly as FP4_TSCALE_CURRENT
 * would (same s_enc,G), without its own amax pass. Only p's scale_fmt (E4M3 or
 * UE5M3), block, orient, rht and step are read; shapes follow the quantize call
 * with the same parameters. in: device BF16, 16-byte aligned. ws: device,
 * 16-byte aligned, at least 2 * 2048 * 4 bytes, not shared with calls in flight.
 * For T % 64 == 0 and C % 128 == 0 the pass runs in 128-thread CTAs (two per
 * SM; one fits beside the dual quantizer's conversion pass); other shapes use
 * the quantizer's own amax kernels. fp4_tensor_amax_dual writes the rowwise
 * operand's amax (out_row) and the colwise one's (out_col, post-RHT when
 * p_col->rht) from one read. */
fp4_status_t fp4_tensor_amax(const fp4_quant_params_t* p, const void* in_bf16, int64_t rows, int64_t cols, int64_t ld,
                             fp4_amax_state_t* out, void* ws, size_t ws_bytes, void* stream);
fp4_status_t fp4_tensor_amax_dual(const fp4_quant_params_t* p_row, const fp4_quant_params_t* p_col, const void* in_bf16,
                                  int64_t rows, int64_t cols, int64_t ld, fp4_amax_state_t* out_row,
                                  fp4_amax_state_t* out_col, void* ws, size_t ws_bytes, void* stream);

/* Decode an operand back to real values, x = e2m1 * s_hat * s_dec,G computed as
 * RN(RN(e2m1 * s_hat) * s_dec,G) in FP32 (section A3; App. B.3), written as
 * rows x cols BF16 (out_fp32 == 0) or FP32; with sdec_per_row, row r takes
 * s_dec_global[r]. */
fp4_status_t fp4_dequantize(const fp4_tensor_t* t, void* out, int out_fp32, void* stream);

/* Block-scaled GEMM D[M x N] = s_dec,G,A * s_dec,G,B * sum_k (a_mk s_A)(b_nk s_B)
 * with FP32 accumulation ("Pretraining LLMs with NVFP4", App. B.3; A3 hardware
 * support). A is M x K, B is N x K, both quantized, K-major, TCGEN05 scale
 * layout, same scale format. A may carry one s_dec,G per row (sdec_per_row,
 * E4M3 only: output row m is scaled by s_dec,G,A[m] * s_dec,G,B); B may not
 * (FP4_ERR_UNSUPPORTED). E4M3 (block 16) runs natively (tcgen05
 * kind::mxf4nvf4); UE8M0 (MXFP4, block 32, section A3) runs natively too
 * (tcgen05 kind::mxf4) with alpha = 1: MXFP4 has no tensor scale, so its
 * s_dec_global is not read; UE5M3 (block 16) runs the software-emulated path
 * (operands decoded to BF16 in shared memory, tcgen05 kind::f16). Mixed scale
 * formats are FP4_ERR_UNSUPPORTED. M and N must be multiples of 128
 * and K of 256. Output row-major M x N: BF16 (out_fp32 == 0) or FP32; with
 * accumulate != 0 (FP32 only) D is added to the existing output. */
fp4_status_t fp4_gemm(const fp4_tensor_t* a, const fp4_tensor_t* b, void* d, int out_fp32,
                      int accumulate, void* stream);

/* fp4_gemm with a caller workspace, which gives UE5M3 operands the exact fast
 * path (no tensor core reads UE5M3 scales, "UE5M3 block scales" abstract; the
 * rebias is this library's design): a first kernel rewrites every row's UE5M3
 * block scales as E4M3 scales times one power of two per row,
 * s = e4m3 * 2^o_row exactly, the native kind::mxf4nvf4 GEMM runs on the E4M3
 * scales and multiplies output (m, n) by 2^(o_m + o_n) before alpha, which
 * gives the same sum as the UE5M3-scaled products. A row whose nonzero scales
 * span more than E4M3's 15 binades cannot be rebiased: the output tiles its
 * 128-row tile touches are computed by the emulated kernel, all others by the
 * native one; the split is made on the device (no host synchronisation), and
 * the emulated kernel returns at once when no row was flagged. When the
 * flagged output tiles are fewer than the SMs, the emulated kernel splits
 * their K across the idle SMs and adds the FP32 parts in a fixed order (the
 * result does not depend on timing). ws: device, 16-byte aligned, at least
 * fp4_gemm_workspace_bytes(a, b) bytes (about (M + N) * K / 16, plus up to
 * 16 MB of FP32 partial tiles for that split), owned by the caller,
 * overwritten, not to be shared by calls in flight at the same time.
 * Too small or NULL: FP4_ERR_WORKSPACE. Other scale formats ignore ws and run
 * exactly as fp4_gemm. After the stream has run the call, byte t of ws
 * (t < M / 128 + N / 128, A's 128-row tiles first) is 1 if tile t held a row
 * that did not fit and 0 otherwise: all zero means the native kernel computed
 * every output. */
size_t fp4_gemm_workspace_bytes(const fp4_tensor_t* a, const fp4_tensor_t* b);
fp4_status_t fp4_gemm_ws(const fp4_tensor_t* a, const fp4_tensor_t* b, void* d, int out_fp32, int accumulate,
                         void* ws, size_t ws_bytes, void* stream);

/* The three GEMMs of a linear layer Y = X W^T (section 4.1, Fig. 5):
 *   Fprop: Y[T x N]  = X[T x K]   . W[N x K]^T     (x rowwise, w 16x16), BF16 out
 *   Dgrad: dX[T x K] = dY[T x N]  . Wt[K x N]^T    (dy rowwise, wt = W^T operand), BF16 out
 *   Wgrad: dW[N x K] = dYt[N x T] . Xt[K x T]^T    (colwise + RHT operands), FP32 out
 *          (weight gradients stay FP32, section 4.1); accumulate adds into dW. */
fp4_status_t fp4_linear_fprop(const fp4_tensor_t* x, const fp4_tensor_t* w, void* y_bf16, void* stream);
fp4_status_t fp4_linear_dgrad(const fp4_tensor_t* dy, const fp4_tensor_t* wt, void* dx_bf16, void* stream);
fp4_status_t fp4_linear_wgrad(const fp4_tensor_t* dyt, const fp4_tensor_t* xt, float* dw_fp32,
                              int accumulate, void* stream);

/* Diagnostic: exercises the path every kernel's bounded waits take on a stall.
 * One thread of a one-block kernel waits on an mbarrier that nothing completes;
 * after limit_us microseconds (1 .. 2,000,000) the wait gives up, records
 * FP4_ERR_DEVICE_TIMEOUT in the device status word and the kernel returns,
 * leaving the context usable. fp4_device_status() then reports the timeout. */
fp4_status_t fp4_selftest_wait_timeout(uint32_t limit_us, void* stream);

/* Diagnostic: out[i] = RN(in[i] / 6) in binary32 as the quantizer forms it
 * (the RN(amax_B / 6) of the block-scale step, App. B.2), for n device floats
 * (16-byte aligned, no overlap), so that the step can be checked against the
 * correctly rounded quotient. n < 0: FP4_ERR_SHAPE. */
fp4_status_t fp4_selftest_div6(const float* in, float* out, int64_t n, void* stream);

/* Synchronise `stream`, then return and clear the current device's status word
 * (FP4_OK when no device-side error was recorded). fp4_last_device_status is
 * the same call under its other name. */
fp4_status_t fp4_device_status(void* stream);
fp4_status_t fp4_last_device_status(void* stream);

/* The same status word without synchronising: when `stream` reaches this call,
 * the status word (an fp4_status_t value) is written to *dst and the word is
 * cleared, in stream order. dst: 4-byte aligned device memory, or host memory
 * the device can write (pinned); read it after the stream has passed the call
 * (an event, or a later synchronisation). Returns FP4_ERR_INVALID_ARG for a
 * null or misaligned dst; otherwise the launch status. */
fp4_status_t fp4_device_status_record(int32_t* dst, void* stream);

/* Static description of a status code. */
const char* fp4_status_string(fp4_status_t s);

/* Library ABI version (incremented on incompatible changes). */
int fp4_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FP4BS_H */
