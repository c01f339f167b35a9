"""fp4_quantize_noalloc, the quantize entry point for callers that cannot
allocate device memory (a plug-in inside another engine that owns the whole
memory budget, or a latency-critical loop that must never reach an allocator):
it keeps the amax partials in a library-owned device array instead of a
caller workspace. Its outputs must equal fp4_quantize's bit for bit (the
quantizer tests' tolerance), on consecutive calls that share that array.

The file name sorts last so that a failure here comes after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

fb = pytest.importorskip("fp4_block_scaled_02_gb300")
from gpu_common import to_gpu_bf16  # noqa: E402
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, random_bf16  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    fb._lib.load()


def _noalloc(cfg, x, out, state=None, counters=None):
    L = fb._lib.load()
    p = cfg.params()
    d = out.desc()
    st = L.fp4_quantize_noalloc(ctypes.byref(p), ctypes.c_void_p(x.data_ptr()), x.shape[0], x.shape[1],
                                fb.row_stride(x), ctypes.byref(d), None,
                                ctypes.c_void_p(state.buf.data_ptr()) if state is not None else None,
                                ctypes.c_void_p(counters.data_ptr()) if counters is not None else None,
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    fb._lib.check(st, "fp4_quantize_noalloc")


def _run_both(cfg, bits, state_a=None, state_b=None):
    x = to_gpu_bf16(bits)
    rows, cols = bits.shape
    R, C = (cols, rows) if cfg.orient == fb.FP4_ORIENT_COLWISE else (rows, cols)
    ref, got = fb.QTensor.empty(R, C, cfg.scale_fmt), fb.QTensor.empty(R, C, cfg.scale_fmt)
    got.codes.fill_(0xAA)
    got.scales.fill_(0xAA)
    c_ref = torch.zeros(4, dtype=torch.int64, device="cuda")
    c_got = torch.zeros(4, dtype=torch.int64, device="cuda")
    ws = torch.empty(fb.fp4_workspace_bytes(cfg, rows, cols) // 4 + 4, dtype=torch.float32, device="cuda")
    fb.fp4_quantize(cfg, x, ref, state=state_a, counters=c_ref, ws=ws)
    _noalloc(cfg, x, got, state=state_b, counters=c_got)
    assert fb.fp4_device_status() == 0
    assert torch.equal(ref.codes, got.codes)
    assert torch.equal(ref.scales, got.scales)
    assert ref.s_dec[0:1].view(torch.int32).item() == got.s_dec[0:1].view(torch.int32).item()
    assert torch.equal(c_ref, c_got)


def test_noalloc_matches_workspace_quantize_on_consecutive_calls():
    # call 1: a large tensor with a large amax (many partials); call 2: a smaller
    # tensor with a smaller amax, so stale partials of call 1 would show if read
    big = f32_to_bf16_bits(bf16_bits_to_f32(random_bf16(71, (4096, 2048), "student_t4")) * np.float32(40.0))
    _run_both(fb.QuantConfig(round=fb.FP4_ROUND_SR, seed=9, tensor_id=3, step=5), big)
    small = random_bf16(72, (512, 768), "normal")
    _run_both(fb.QuantConfig(orient=fb.FP4_ORIENT_COLWISE, rht=True, seed=1, tensor_id=1), small)


def test_noalloc_held_amax_refresh_and_reuse():
    sa, sb = fb.AmaxState(), fb.AmaxState()
    base = random_bf16(73, (1024, 1024), "log_normal_1e-4_2")
    for step, factor in [(0, 1.0), (1, 100.0), (50, 0.01)]:
        bits = f32_to_bf16_bits(bf16_bits_to_f32(base) * np.float32(factor))
        cfg = fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE5M3, tscale=fb.FP4_TSCALE_HELD, target_T=2048.0,
                             round=fb.FP4_ROUND_SR, step=step, seed=2, tensor_id=4)
        _run_both(cfg, bits, sa, sb)
        assert torch.equal(sa.buf, sb.buf)
