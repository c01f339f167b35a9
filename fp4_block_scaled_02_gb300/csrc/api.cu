// api.cu -- the extern "C" entry points of libfp4bs.so: synchronous argument
// checks, then kernel launches on the caller's stream. No entry point
// allocates device memory.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "fp4_device.cuh"
#ifndef FP4BS_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

#include "internal.h"

namespace fp4bs {

// Per-device status word: bounded waits that time out record a code here
// (first error wins).
__device__ int g_device_status;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int* g_status_ptr[kMaxDevices];

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fp4_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? FP4_OK : FP4_ERR_CUDA; }

}  // namespace

int num_sms() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

int* device_status_ptr() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_status_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

}  // namespace fp4bs

namespace fp4bs {
namespace {

// Stream-ordered status read: when the stream reaches it, move the status word
// (and its reset to 0) into *dst.
__global__ void status_record_kernel(int* status, int32_t* dst) {
    pdl_begin();
    *dst = atomicExch(status, 0);
}

}  // namespace
}  // namespace fp4bs

using namespace fp4bs;

namespace {

int block_len(int block) { return block == FP4_BLOCK_1x32 ? 32 : 16; }

// Row stride of a BF16 input: at least its width and a multiple of 8 elements,
// so that every row starts 16-byte aligned like the base pointer.
bool ld_ok(int64_t rows, int64_t cols, int64_t ld) {
    if (rows == 0 || cols == 0) return true;
    return ld >= cols && ld % 8 == 0;
}

// Argument checks shared by the quantizer entry points (everything but the
// workspace). Fills `job` on success.
fp4_status_t check_quantize_args(const fp4_quant_params_t* p, const void* in, int64_t rows, int64_t cols, int64_t ld,
                                 const fp4_tensor_t* out, const fp4_tensor_t* out_t, fp4_amax_state_t* state,
                                 uint64_t* counters, QuantJob& job) {
    if (p == nullptr || out == nullptr) return FP4_ERR_INVALID_ARG;
    if (p->reserved != 0) return FP4_ERR_INVALID_ARG;
    if (p->scale_fmt < 0 || p->scale_fmt > 2 || p->block < 0 || p->block > 2) return FP4_ERR_INVALID_ARG;
    if (p->round < 0 || p->round > 1 || p->orient < 0 || p->orient > 1) return FP4_ERR_INVALID_ARG;
    if (p->tscale < 0 || p->tscale > 3 || p->scale_layout < 0 || p->scale_layout > 1) return FP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return FP4_ERR_SHAPE;
    if (!ld_ok(rows, cols, ld)) return FP4_ERR_SHAPE;
    if (p->tensor_id == 0xFFFFFFFFu) return FP4_ERR_INVALID_ARG;
    const bool mx = p->scale_fmt == FP4_SCALE_UE8M0;
    if (mx != (p->block == FP4_BLOCK_1x32)) return FP4_ERR_INVALID_ARG;
    if (p->rht && (p->block != FP4_BLOCK_1x16 || p->orient != FP4_ORIENT_COLWISE)) return FP4_ERR_INVALID_ARG;
    if (mx && (p->round != FP4_ROUND_RNE || p->orient != FP4_ORIENT_ROWWISE)) return FP4_ERR_UNSUPPORTED;
    // 16x16 with SR runs only on the TMA tile path: whole 64 x 128 input tiles
    if (p->block == FP4_BLOCK_16x16 && p->round != FP4_ROUND_RNE && (rows % 64 != 0 || cols % 128 != 0))
        return FP4_ERR_UNSUPPORTED;
    if (p->emit_transpose && p->block != FP4_BLOCK_16x16) return FP4_ERR_INVALID_ARG;
    if (p->emit_transpose && out_t == nullptr) return FP4_ERR_INVALID_ARG;
    const bool held = !mx && p->tscale == FP4_TSCALE_HELD;
    const bool given = !mx && p->tscale == FP4_TSCALE_GIVEN;
    // per-row current scaling: E4M3, plain rowwise 1x16 only, into a per-row s_dec
    const bool per_row = !mx && p->tscale == FP4_TSCALE_ROW;
    if (out->sdec_per_row != (per_row ? 1 : 0)) return FP4_ERR_INVALID_ARG;
    if (per_row && (p->scale_fmt != FP4_SCALE_E4M3 || p->block != FP4_BLOCK_1x16 ||
                    p->orient != FP4_ORIENT_ROWWISE || p->rht || p->emit_transpose))
        return FP4_ERR_UNSUPPORTED;
    if (held && (state == nullptr || p->refresh_every == 0)) return FP4_ERR_INVALID_ARG;
    if (given && state == nullptr) return FP4_ERR_INVALID_ARG;
    if (!mx && !(p->target_T > 0.0f && p->target_T <= 3.0e38f)) return FP4_ERR_INVALID_ARG;

    const int bs = block_len(p->block);
    const bool colwise = p->orient == FP4_ORIENT_COLWISE;
    const int64_t R = colwise ? cols : rows, C = colwise ? rows : cols;
    if (out->rows != R || out->cols != C) return FP4_ERR_SHAPE;
    if (out->scale_fmt != p->scale_fmt || out->block_k != bs || out->scale_layout != p->scale_layout)
        return FP4_ERR_INVALID_ARG;
    if (C % bs != 0) return FP4_ERR_SHAPE;
    if (p->block == FP4_BLOCK_16x16 && (R % 16 != 0)) return FP4_ERR_SHAPE;
    if (colwise && p->block == FP4_BLOCK_1x16 && (cols % 8 != 0)) return FP4_ERR_SHAPE;
    if (p->scale_layout == FP4_LAYOUT_TCGEN05 && (R % 128 != 0 || (C / bs) % 4 != 0)) return FP4_ERR_SHAPE;
    if (p->emit_transpose) {
        if (out_t->sdec_per_row != 0) return FP4_ERR_INVALID_ARG;
        if (out_t->rows != C || out_t->cols != R) return FP4_ERR_SHAPE;
        if (out_t->scale_fmt != p->scale_fmt || out_t->block_k != 16) return FP4_ERR_INVALID_ARG;
        if (out_t->scale_layout == FP4_LAYOUT_TCGEN05 && (C % 128 != 0 || (R / 16) % 4 != 0)) return FP4_ERR_SHAPE;
    }
    const bool empty = rows == 0 || cols == 0;
    if (!empty) {
        if (in == nullptr || out->codes == nullptr || out->scales == nullptr) return FP4_ERR_INVALID_ARG;
        if (!aligned16(in) || !aligned16(out->codes)) return FP4_ERR_ALIGNMENT;
        if (p->scale_layout == FP4_LAYOUT_TCGEN05 && !aligned16(out->scales)) return FP4_ERR_ALIGNMENT;
        if (p->emit_transpose) {
            if (out_t->codes == nullptr || out_t->scales == nullptr) return FP4_ERR_INVALID_ARG;
            if (!aligned16(out_t->codes)) return FP4_ERR_ALIGNMENT;
        }
    }
    if (!mx && out->s_dec_global == nullptr) return FP4_ERR_INVALID_ARG;

    job = QuantJob{};
    job.scale_fmt = p->scale_fmt;
    job.block = p->block;
    job.sr = p->round == FP4_ROUND_SR;
    job.colwise = colwise;
    job.rht = p->rht != 0;
    job.held = held || given;
    job.refresh = given ? 0 : held ? (p->step % p->refresh_every == 0) : 1;
    job.given = given;
    job.per_row = per_row;
    job.target_T = p->target_T;
    job.tensor_id = p->tensor_id;
    job.seed = p->seed;
    job.step = p->step;
    job.in = static_cast<const uint16_t*>(in);
    job.rows = rows;
    job.cols = cols;
    job.ld = ld;
    job.codes = out->codes;
    job.scales = out->scales;
    job.s_dec = out->s_dec_global;
    job.layout = out->scale_layout;
    if (p->emit_transpose) {
        job.codes_t = out_t->codes;
        job.scales_t = out_t->scales;
        job.s_dec_t = out_t->s_dec_global;
        job.layout_t = out_t->scale_layout;
    }
    job.state = state;
    job.counters = counters;
    return FP4_OK;
}

// The amax pass's partials go to ws: enough room for every partial it writes,
// 16-byte aligned (nothing is checked or used when the call runs no amax pass).
fp4_status_t attach_workspace(QuantJob& job, void* ws, size_t ws_bytes) {
    const int np = amax_partials_needed(job);
    if (np == 0) return FP4_OK;
    if (ws == nullptr || ws_bytes < (size_t)np * sizeof(float)) return FP4_ERR_WORKSPACE;
    if (!aligned16(ws)) return FP4_ERR_ALIGNMENT;
    job.partials = static_cast<float*>(ws);
    return FP4_OK;
}

fp4_status_t check_quantize(const fp4_quant_params_t* p, const void* in, int64_t rows, int64_t cols, int64_t ld,
                            const fp4_tensor_t* out, const fp4_tensor_t* out_t, fp4_amax_state_t* state,
                            uint64_t* counters, void* ws, size_t ws_bytes, QuantJob& job) {
    fp4_status_t s = check_quantize_args(p, in, rows, cols, ld, out, out_t, state, counters, job);
    if (s != FP4_OK) return s;
    return attach_workspace(job, ws, ws_bytes);
}

fp4_status_t check_operand(const fp4_tensor_t* t) {
    if (t == nullptr || t->codes == nullptr || t->scales == nullptr || t->s_dec_global == nullptr)
        return FP4_ERR_INVALID_ARG;
    if (t->sdec_per_row != 0 && (t->sdec_per_row != 1 || t->scale_fmt != FP4_SCALE_E4M3))
        return FP4_ERR_INVALID_ARG;
    if (!aligned16(t->codes) || !aligned16(t->scales)) return FP4_ERR_ALIGNMENT;
    return FP4_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Allocation-free quantize.
//
// Some callers cannot allocate device memory at all: a plug-in running inside
// another framework's engine, whose memory budget is owned and pre-planned by
// that engine, or a latency-critical loop that must never reach an allocator.
// fp4_quantize needs a caller-provided workspace for the amax partials of its
// first pass; fp4_quantize_noalloc instead uses the library's own file-scope
// scratch array below. Its size is the largest number of partials the amax
// pass ever writes (kNoAllocScratchFloats floats = 8 KB), and every GPU that
// loads this library keeps that array until the process exits.
//
// The array's host-side name is only a stand-in for the device symbol, so its
// device address is looked up once per device (cudaGetSymbolAddress, with the
// device current) by the first call on that device that runs an amax pass
// (current scaling, or a held-amax call); make that first call before any
// stream capture begins. Calls that run no amax pass (UE8M0, a given amax, per-
// row scales) never touch the array. Every call shares the one array and it
// keeps the last call's contents; nothing in it needs to start at zero,
// because the amax pass writes every partial the conversion pass reads. Calls
// whose work overlaps on the GPU (different streams, no ordering between
// them) race on the array.
namespace {

constexpr int kNoAllocScratchFloats = kMaxAmaxPartials;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];
float* g_noalloc_ptr[kMaxDevices];

float* noalloc_scratch_ptr() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        float* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = ptr;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

namespace {

fp4_status_t prepare_gemm(const fp4_tensor_t* a, const fp4_tensor_t* b, void* d, int out_fp32, int accumulate,
                          GemmJob& j) {
    fp4_status_t s = check_operand(a);
    if (s != FP4_OK) return s;
    s = check_operand(b);
    if (s != FP4_OK) return s;
    if (d == nullptr) return FP4_ERR_INVALID_ARG;
    if (!aligned16(d)) return FP4_ERR_ALIGNMENT;
    if (accumulate && !out_fp32) return FP4_ERR_INVALID_ARG;
    const int bs = a->scale_fmt == FP4_SCALE_UE8M0 ? 32 : 16;
    if (a->scale_fmt != b->scale_fmt || a->block_k != bs || b->block_k != bs) return FP4_ERR_UNSUPPORTED;
    if (a->scale_layout != FP4_LAYOUT_TCGEN05 || b->scale_layout != FP4_LAYOUT_TCGEN05) return FP4_ERR_UNSUPPORTED;
    if (b->sdec_per_row) return FP4_ERR_UNSUPPORTED;  // per-row decode scales on A only
    if (a->cols != b->cols) return FP4_ERR_SHAPE;
    if (a->rows % 128 != 0 || b->rows % 128 != 0 || a->cols % 256 != 0 || a->cols <= 0 || a->rows <= 0 ||
        b->rows <= 0)
        return FP4_ERR_SHAPE;
    j = GemmJob{};
    j.a_codes = a->codes;
    j.a_scales = a->scales;
    j.a_sdec = a->s_dec_global;
    j.a_sdec_rows = a->sdec_per_row != 0;
    j.b_codes = b->codes;
    j.b_scales = b->scales;
    j.b_sdec = b->s_dec_global;
    j.M = a->rows;
    j.N = b->rows;
    j.K = a->cols;
    j.scale_fmt = a->scale_fmt;
    j.d = d;
    j.out_fp32 = out_fp32 != 0;
    j.accumulate = accumulate != 0;
    j.status = device_status_ptr();
    if (j.status == nullptr) return FP4_ERR_CUDA;
    return FP4_OK;
}

// UE5M3 rebias workspace: per-tile "does not fit" bytes, per-row offsets of A
// and B, rebiased scales of A and B (each part 16-byte aligned).
struct RebiasLayout {
    size_t off_a, off_b, sc_a, sc_b, cnt, split, total;
    int64_t split_tiles;
};
// fp4_gemm_ws's workspace: flags, per-row offsets, rebiased scales, then for
// the emulated fallback 4 counters per split tile and the FP32 partial tiles
// (at most one per tile and 256-value stage, and kEmuSplitMaxTiles).
RebiasLayout rebias_layout(int64_t M, int64_t N, int64_t K) {
    auto up16 = [](size_t x) { return (x + 15) & ~size_t(15); };
    RebiasLayout l{};
    l.off_a = up16((size_t)(M / 128 + N / 128));
    l.off_b = l.off_a + up16((size_t)M);
    l.sc_a = l.off_b + up16((size_t)N);
    l.sc_b = l.sc_a + up16((size_t)(M * (K / 16)));
    l.cnt = l.sc_b + up16((size_t)(N * (K / 16)));
    const int64_t work = (M / 128) * (N / 128) * (K / 256);
    l.split_tiles = work < kEmuSplitMaxTiles ? work : kEmuSplitMaxTiles;
    l.split = l.cnt + up16((size_t)(4 * kEmuSplitMaxTiles) * sizeof(uint32_t));
    l.total = l.split + (size_t)l.split_tiles * 128 * 128 * sizeof(float);
    return l;
}

}  // namespace

namespace {

// Shape rules of a tensor amax: those of the quantize call with the same
// parameters (its blocks must tile the tensor).
fp4_status_t check_amax_params(const fp4_quant_params_t* p, int64_t rows, int64_t cols) {
    if (p == nullptr) return FP4_ERR_INVALID_ARG;
    if (p->scale_fmt < 0 || p->scale_fmt > 1) return FP4_ERR_INVALID_ARG;  // MXFP4 has no tensor amax
    if (p->block < 0 || p->block > 1 || p->orient < 0 || p->orient > 1) return FP4_ERR_INVALID_ARG;
    if (p->rht && (p->block != FP4_BLOCK_1x16 || p->orient != FP4_ORIENT_COLWISE)) return FP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0) return FP4_ERR_SHAPE;
    const bool colwise = p->orient == FP4_ORIENT_COLWISE;
    const int64_t R = colwise ? cols : rows, C = colwise ? rows : cols;
    if (C % 16 != 0) return FP4_ERR_SHAPE;
    if (p->block == FP4_BLOCK_16x16 && R % 16 != 0) return FP4_ERR_SHAPE;
    if (colwise && cols % 8 != 0) return FP4_ERR_SHAPE;
    return FP4_OK;
}

}  // namespace

namespace {

// An NVTX range around each launching entry point, so profilers show the C-ABI
// calls on their timelines (no cost without a profiler attached; compile with
// FP4BS_NO_NVTX to leave them out).
struct NvtxRange {
    explicit NvtxRange(const char* name) {
#ifndef FP4BS_NO_NVTX
        nvtxRangePushA(name);
#else
        (void)name;
#endif
    }
    ~NvtxRange() {
#ifndef FP4BS_NO_NVTX
        nvtxRangePop();
#endif
    }
};

}  // namespace

extern "C" {

int fp4_abi_version(void) { return 3; }

const char* fp4_status_string(fp4_status_t s) {
    switch (s) {
        case FP4_OK: return "ok";
        case FP4_ERR_INVALID_ARG: return "invalid argument";
        case FP4_ERR_UNSUPPORTED: return "unsupported combination";
        case FP4_ERR_SHAPE: return "unsupported shape";
        case FP4_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case FP4_ERR_STATE: return "given amax record not valid";
        case FP4_ERR_CUDA: return "CUDA runtime error";
        case FP4_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case FP4_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

fp4_status_t fp4_quantized_sizes(const fp4_quant_params_t* p, int64_t rows, int64_t cols, size_t* codes_bytes,
                                 size_t* scales_bytes) {
    if (p == nullptr || codes_bytes == nullptr || scales_bytes == nullptr) return FP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || p->block < 0 || p->block > 2) return FP4_ERR_INVALID_ARG;
    const int bs = block_len(p->block);
    const int64_t R = p->orient == FP4_ORIENT_COLWISE ? cols : rows;
    const int64_t C = p->orient == FP4_ORIENT_COLWISE ? rows : cols;
    if (C % bs != 0) return FP4_ERR_SHAPE;
    *codes_bytes = (size_t)(R * C / 2);
    *scales_bytes = (size_t)(R * (C / bs));
    return FP4_OK;
}

size_t fp4_workspace_bytes(const fp4_quant_params_t* p, int64_t rows, int64_t cols) {
    (void)rows;
    (void)cols;
    if (p == nullptr || p->scale_fmt == FP4_SCALE_UE8M0 || p->tscale == FP4_TSCALE_GIVEN ||
        p->tscale == FP4_TSCALE_ROW)
        return 0;
    return (size_t)kMaxAmaxPartials * sizeof(float);
}

fp4_status_t fp4_quantize(const fp4_quant_params_t* p, const void* in_bf16, int64_t rows, int64_t cols, int64_t ld,
                          const fp4_tensor_t* out, const fp4_tensor_t* out_t, fp4_amax_state_t* state,
                          uint64_t* counters, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("fp4_quantize");
    QuantJob job;
    fp4_status_t s = check_quantize(p, in_bf16, rows, cols, ld, out, out_t, state, counters, ws, ws_bytes, job);
    if (s != FP4_OK) return s;
    if (rows == 0 || cols == 0) return FP4_OK;
    job.status = device_status_ptr();
    if (job.status == nullptr) return FP4_ERR_CUDA;
    return from_cuda(launch_quantize(job, static_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_quantize_noalloc(const fp4_quant_params_t* p, const void* in_bf16, int64_t rows, int64_t cols,
                                  int64_t ld, const fp4_tensor_t* out, const fp4_tensor_t* out_t,
                                  fp4_amax_state_t* state, uint64_t* counters, void* stream) {
    NvtxRange nvtx_range("fp4_quantize_noalloc");
    QuantJob job;
    fp4_status_t s = check_quantize_args(p, in_bf16, rows, cols, ld, out, out_t, state, counters, job);
    if (s != FP4_OK) return s;
    // the scratch is offered as a workspace of its fixed size, looked up only
    // when the call runs an amax pass: a call that would need more partials
    // than it holds is rejected with FP4_ERR_WORKSPACE before anything is launched
    const int np = amax_partials_needed(job);
    if (np > kNoAllocScratchFloats) return FP4_ERR_WORKSPACE;
    if (np > 0) {
        float* scratch = noalloc_scratch_ptr();
        if (scratch == nullptr) return FP4_ERR_CUDA;
        s = attach_workspace(job, scratch, sizeof(float) * kNoAllocScratchFloats);
        if (s != FP4_OK) return s;
    }
    if (rows == 0 || cols == 0) return FP4_OK;
    job.status = device_status_ptr();
    if (job.status == nullptr) return FP4_ERR_CUDA;
    return from_cuda(launch_quantize(job, static_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_quantize_dual(const fp4_quant_params_t* p_row, const fp4_quant_params_t* p_col, const void* in_bf16,
                               int64_t rows, int64_t cols, int64_t ld, const fp4_tensor_t* out_row,
                               const fp4_tensor_t* out_col,
                               fp4_amax_state_t* state_row, fp4_amax_state_t* state_col, uint64_t* counters_row,
                               uint64_t* counters_col, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("fp4_quantize_dual");
    if (p_row == nullptr || p_col == nullptr) return FP4_ERR_INVALID_ARG;
    if (p_row->orient != FP4_ORIENT_ROWWISE || p_col->orient != FP4_ORIENT_COLWISE) return FP4_ERR_INVALID_ARG;
    if (p_row->block != FP4_BLOCK_1x16 || p_col->block != FP4_BLOCK_1x16) return FP4_ERR_UNSUPPORTED;
    if (p_row->scale_fmt != p_col->scale_fmt || p_row->scale_fmt == FP4_SCALE_UE8M0) return FP4_ERR_UNSUPPORTED;
    if (p_row->round != p_col->round || p_row->tscale != p_col->tscale) return FP4_ERR_UNSUPPORTED;
    if (p_row->tscale == FP4_TSCALE_ROW) return FP4_ERR_UNSUPPORTED;  // a colwise row is a whole column
    if (p_row->tscale == FP4_TSCALE_HELD && p_row->refresh_every != p_col->refresh_every) return FP4_ERR_UNSUPPORTED;
    if (p_row->step != p_col->step) return FP4_ERR_UNSUPPORTED;
    if (p_row->scale_layout != FP4_LAYOUT_TCGEN05 || p_col->scale_layout != FP4_LAYOUT_TCGEN05)
        return FP4_ERR_UNSUPPORTED;
    if (rows % 128 != 0 || cols % 128 != 0) return FP4_ERR_SHAPE;
    const size_t half = (size_t)kMaxAmaxPartials * sizeof(float);
    const bool given = p_row->tscale == FP4_TSCALE_GIVEN;  // no amax pass: no workspace needed
    if (!given && (ws == nullptr || ws_bytes < 2 * half)) return FP4_ERR_WORKSPACE;
    QuantJob jr, jc;
    fp4_status_t s =
        check_quantize(p_row, in_bf16, rows, cols, ld, out_row, nullptr, state_row, counters_row, ws, half, jr);
    if (s != FP4_OK) return s;
    s = check_quantize(p_col, in_bf16, rows, cols, ld, out_col, nullptr, state_col, counters_col,
                       given ? nullptr : static_cast<char*>(ws) + half, half, jc);
    if (s != FP4_OK) return s;
    if (rows == 0 || cols == 0) return FP4_OK;
    jr.status = jc.status = device_status_ptr();
    if (jr.status == nullptr) return FP4_ERR_CUDA;
    return from_cuda(launch_quantize_dual(jr, jc, static_cast<cudaStream_t>(stream)));
}


fp4_status_t fp4_tensor_amax(const fp4_quant_params_t* p, const void* in_bf16, int64_t rows, int64_t cols, int64_t ld,
                             fp4_amax_state_t* out, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("fp4_tensor_amax");
    fp4_status_t s = check_amax_params(p, rows, cols);
    if (s != FP4_OK) return s;
    if (!ld_ok(rows, cols, ld)) return FP4_ERR_SHAPE;
    if (out == nullptr || (rows > 0 && cols > 0 && in_bf16 == nullptr)) return FP4_ERR_INVALID_ARG;
    if (ws == nullptr || ws_bytes < 2 * (size_t)kMaxAmaxPartials * sizeof(float)) return FP4_ERR_WORKSPACE;
    if (!aligned16(ws) || !aligned16(in_bf16)) return FP4_ERR_ALIGNMENT;
    int* status = device_status_ptr();
    if (status == nullptr) return FP4_ERR_CUDA;
    const bool rht = p->rht != 0;
    return from_cuda(launch_tensor_amax(static_cast<const uint16_t*>(in_bf16), rows, cols, ld, rht ? nullptr : out,
                                        rht ? out : nullptr, rht, p->step, static_cast<float*>(ws), status,
                                        static_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_tensor_amax_dual(const fp4_quant_params_t* p_row, const fp4_quant_params_t* p_col, const void* in_bf16,
                                  int64_t rows, int64_t cols, int64_t ld, fp4_amax_state_t* out_row,
                                  fp4_amax_state_t* out_col, void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("fp4_tensor_amax_dual");
    fp4_status_t s = check_amax_params(p_row, rows, cols);
    if (s != FP4_OK) return s;
    if (!ld_ok(rows, cols, ld)) return FP4_ERR_SHAPE;
    s = check_amax_params(p_col, rows, cols);
    if (s != FP4_OK) return s;
    if (p_row->orient != FP4_ORIENT_ROWWISE || p_col->orient != FP4_ORIENT_COLWISE) return FP4_ERR_INVALID_ARG;
    if (p_row->step != p_col->step) return FP4_ERR_UNSUPPORTED;
    if (out_row == nullptr || out_col == nullptr || (rows > 0 && cols > 0 && in_bf16 == nullptr))
        return FP4_ERR_INVALID_ARG;
    if (ws == nullptr || ws_bytes < 2 * (size_t)kMaxAmaxPartials * sizeof(float)) return FP4_ERR_WORKSPACE;
    if (!aligned16(ws) || !aligned16(in_bf16)) return FP4_ERR_ALIGNMENT;
    int* status = device_status_ptr();
    if (status == nullptr) return FP4_ERR_CUDA;
    return from_cuda(launch_tensor_amax(static_cast<const uint16_t*>(in_bf16), rows, cols, ld, out_row, out_col,
                                        p_col->rht != 0, p_row->step, static_cast<float*>(ws), status,
                                        static_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_dequantize(const fp4_tensor_t* t, void* out, int out_fp32, void* stream) {
    NvtxRange nvtx_range("fp4_dequantize");
    if (t == nullptr || out == nullptr) return FP4_ERR_INVALID_ARG;
    if (t->rows == 0 || t->cols == 0) return FP4_OK;
    fp4_status_t s = check_operand(t);
    if (s != FP4_OK && s != FP4_ERR_ALIGNMENT) return s;
    if (!aligned16(t->codes) || !aligned16(out)) return FP4_ERR_ALIGNMENT;
    if (t->scale_fmt < 0 || t->scale_fmt > 2) return FP4_ERR_INVALID_ARG;
    const int bs = t->scale_fmt == FP4_SCALE_UE8M0 ? 32 : 16;
    if (t->block_k != bs || t->rows < 0 || t->cols % bs != 0) return FP4_ERR_SHAPE;
    if (t->scale_layout == FP4_LAYOUT_TCGEN05 && (t->rows % 128 != 0 || (t->cols / bs) % 4 != 0))
        return FP4_ERR_SHAPE;
    DequantJob j{t->codes, t->scales, t->s_dec_global, t->sdec_per_row != 0, t->rows, t->cols, t->scale_fmt, bs,
                 t->scale_layout, out, out_fp32 != 0};
    return from_cuda(launch_dequantize(j, static_cast<cudaStream_t>(stream)));
}


fp4_status_t fp4_gemm(const fp4_tensor_t* a, const fp4_tensor_t* b, void* d, int out_fp32, int accumulate,
                      void* stream) {
    NvtxRange nvtx_range("fp4_gemm");
    GemmJob j;
    fp4_status_t s = prepare_gemm(a, b, d, out_fp32, accumulate, j);
    if (s != FP4_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (a->scale_fmt != FP4_SCALE_UE5M3) return from_cuda(launch_gemm_nvfp4(j, st));  // NVFP4 and MXFP4
    return from_cuda(launch_gemm_ue5m3(j, st));
}

size_t fp4_gemm_workspace_bytes(const fp4_tensor_t* a, const fp4_tensor_t* b) {
    if (a == nullptr || b == nullptr || a->scale_fmt != FP4_SCALE_UE5M3 || a->rows < 0 || b->rows < 0 ||
        a->cols < 0)
        return 0;
    return rebias_layout(a->rows, b->rows, a->cols).total;
}

fp4_status_t fp4_gemm_ws(const fp4_tensor_t* a, const fp4_tensor_t* b, void* d, int out_fp32, int accumulate,
                         void* ws, size_t ws_bytes, void* stream) {
    NvtxRange nvtx_range("fp4_gemm_ws");
    GemmJob j;
    fp4_status_t s = prepare_gemm(a, b, d, out_fp32, accumulate, j);
    if (s != FP4_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (a->scale_fmt != FP4_SCALE_UE5M3) return from_cuda(launch_gemm_nvfp4(j, st));
    const RebiasLayout l = rebias_layout(j.M, j.N, j.K);
    if (ws == nullptr || ws_bytes < l.total) return FP4_ERR_WORKSPACE;
    if (!aligned16(ws)) return FP4_ERR_ALIGNMENT;
    uint8_t* w = static_cast<uint8_t*>(ws);
    uint8_t* flags = w;
    int8_t* a_off = reinterpret_cast<int8_t*>(w + l.off_a);
    int8_t* b_off = reinterpret_cast<int8_t*>(w + l.off_b);
    uint8_t* a_sc = w + l.sc_a;
    uint8_t* b_sc = w + l.sc_b;
    uint32_t* split_cnt = reinterpret_cast<uint32_t*>(w + l.cnt);
    cudaError_t e = launch_rebias_ue5m3(j.a_scales, j.M, j.b_scales, j.N, j.K, a_sc, b_sc, a_off, b_off, flags,
                                        split_cnt, 4 * kEmuSplitMaxTiles, st);
    if (e != cudaSuccess) return from_cuda(e);
    // native MMA on the rebiased scales, unless a row did not fit; then the
    // emulated kernel (which reads the UE5M3 scales) runs instead
    GemmJob jn = j;
    jn.a_scales = a_sc;
    jn.b_scales = b_sc;
    jn.a_off = a_off;
    jn.b_off = b_off;
    jn.rb_flags = flags;
    jn.rb_nflags = j.M / 128 + j.N / 128;
    e = launch_gemm_nvfp4(jn, st);
    if (e != cudaSuccess) return from_cuda(e);
    GemmJob je = j;
    je.rb_flags = flags;
    je.rb_nflags = jn.rb_nflags;
    je.rb_emulated = 1;
    je.split_cnt = split_cnt;
    je.split_buf = reinterpret_cast<float*>(w + l.split);
    je.split_cap = l.split_tiles;
    return from_cuda(launch_gemm_ue5m3(je, st));
}

fp4_status_t fp4_linear_fprop(const fp4_tensor_t* x, const fp4_tensor_t* w, void* y_bf16, void* stream) {
    return fp4_gemm(x, w, y_bf16, 0, 0, stream);
}

fp4_status_t fp4_linear_dgrad(const fp4_tensor_t* dy, const fp4_tensor_t* wt, void* dx_bf16, void* stream) {
    return fp4_gemm(dy, wt, dx_bf16, 0, 0, stream);
}

fp4_status_t fp4_linear_wgrad(const fp4_tensor_t* dyt, const fp4_tensor_t* xt, float* dw_fp32, int accumulate,
                              void* stream) {
    return fp4_gemm(dyt, xt, dw_fp32, 1, accumulate, stream);
}

fp4_status_t fp4_selftest_wait_timeout(uint32_t limit_us, void* stream) {
    if (limit_us == 0 || limit_us > 2000000u) return FP4_ERR_INVALID_ARG;
    int* status = device_status_ptr();
    if (status == nullptr) return FP4_ERR_CUDA;
    return from_cuda(launch_wait_selftest((uint64_t)limit_us * 1000ull, status, static_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_selftest_div6(const float* in, float* out, int64_t n, void* stream) {
    if (n < 0) return FP4_ERR_SHAPE;
    if (n > 0 && (in == nullptr || out == nullptr)) return FP4_ERR_INVALID_ARG;
    if (n > 0 && (!aligned16(in) || !aligned16(out))) return FP4_ERR_ALIGNMENT;
    return from_cuda(launch_div6_selftest(in, out, n, static_cast<cudaStream_t>(stream)));
}

fp4_status_t fp4_device_status_record(int32_t* dst, void* stream) {
    if (dst == nullptr || (reinterpret_cast<uintptr_t>(dst) & 3u) != 0) return FP4_ERR_INVALID_ARG;
    int* p = device_status_ptr();
    if (p == nullptr) return FP4_ERR_CUDA;
    (void)launch_pdl(status_record_kernel, 1, 1, 0, static_cast<cudaStream_t>(stream), p, dst);
    return from_cuda(cudaGetLastError());
}

fp4_status_t fp4_last_device_status(void* stream) { return fp4_device_status(stream); }

fp4_status_t fp4_quantized_bytes(const fp4_quant_params_t* p, int64_t rows, int64_t cols, size_t* codes_bytes,
                                 size_t* scales_bytes) {
    return fp4_quantized_sizes(p, rows, cols, codes_bytes, scales_bytes);
}

fp4_status_t fp4_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FP4_ERR_CUDA;
    int* p = device_status_ptr();
    if (p == nullptr) return FP4_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FP4_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FP4_ERR_CUDA;
    }
    return static_cast<fp4_status_t>(v);
}

}  // extern "C"
