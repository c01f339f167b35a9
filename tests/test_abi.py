"""The C-ABI library loads and exports every entry point include/fp4bs.h
declares; host-side argument checks work without a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp4_block_scaled_02_gb300 import build, _lib
    build.build()
    return _lib.load()


def _declared():
    with open(os.path.join(ROOT, "include", "fp4bs.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(fp4_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "fp4_quantize" in names and "fp4_linear_wgrad" in names and len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    from fp4_block_scaled_02_gb300 import _lib
    assert sorted(_lib.EXPORTED) == names


def test_status_strings_and_version(lib):
    assert lib.fp4_abi_version() == 3
    for s in range(9):
        assert lib.fp4_status_string(s)
    assert lib.fp4_status_string(0) == b"ok"


def test_sizes_and_workspace_without_gpu(lib):
    from fp4_block_scaled_02_gb300 import _lib as L
    p = L.fp4_quant_params_t(0, 0, 0, 0, 0, 0, 448.0, 50, 0, 1, 0, 0, 0, 0)
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.fp4_quantized_sizes(ctypes.byref(p), 256, 512, ctypes.byref(c), ctypes.byref(s)) == 0
    assert (c.value, s.value) == (256 * 256, 256 * 32)
    p.orient = L.FP4_ORIENT_COLWISE
    assert lib.fp4_quantized_sizes(ctypes.byref(p), 256, 512, ctypes.byref(c), ctypes.byref(s)) == 0
    assert (c.value, s.value) == (512 * 128, 512 * 16)
    assert lib.fp4_quantized_sizes(ctypes.byref(p), 250, 512, ctypes.byref(c), ctypes.byref(s)) == L.FP4_ERR_SHAPE
    assert lib.fp4_workspace_bytes(ctypes.byref(p), 256, 512) >= 4
    p.scale_fmt = L.FP4_SCALE_UE8M0
    assert lib.fp4_workspace_bytes(ctypes.byref(p), 256, 512) == 0


def test_selftest_rejects_bad_limits_without_launching(lib):
    from fp4_block_scaled_02_gb300 import _lib as L
    assert lib.fp4_selftest_wait_timeout(0, None) == L.FP4_ERR_INVALID_ARG
    assert lib.fp4_selftest_wait_timeout(2000001, None) == L.FP4_ERR_INVALID_ARG


def test_argument_checks_return_before_any_launch(lib):
    from fp4_block_scaled_02_gb300 import _lib as L
    p = L.fp4_quant_params_t(0, 0, 0, 0, 0, 0, 448.0, 50, 0, 1, 0, 0, 0, 0)
    t = L.fp4_tensor_t(16, 16, 16, 128, 64, 0, 16, 1, 0)
    assert lib.fp4_quantize(None, None, 0, 0, 0, None, None, None, None, None, 0, None) == L.FP4_ERR_INVALID_ARG
    p.rht = 1   # RHT only with colwise 1x16
    assert lib.fp4_quantize(ctypes.byref(p), ctypes.c_void_p(16), 128, 64, 64, ctypes.byref(t), None, None, None,
                            None, 0, None) == L.FP4_ERR_INVALID_ARG
    p.rht = 0
    p.tensor_id = 0xFFFFFFFF  # reserved
    assert lib.fp4_quantize(ctypes.byref(p), ctypes.c_void_p(16), 128, 64, 64, ctypes.byref(t), None, None, None,
                            None, 0, None) == L.FP4_ERR_INVALID_ARG
    p.tensor_id = 0
    assert lib.fp4_quantize(ctypes.byref(p), ctypes.c_void_p(8), 128, 64, 64, ctypes.byref(t), None, None, None,
                            ctypes.c_void_p(16), 8192, None) == L.FP4_ERR_ALIGNMENT
    a = L.fp4_tensor_t(16, 16, 16, 100, 256, 0, 16, 1, 0)
    b = L.fp4_tensor_t(16, 16, 16, 128, 256, 0, 16, 1, 0)
    assert lib.fp4_gemm(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(16), 1, 0, None) == L.FP4_ERR_SHAPE
    a.rows = 128
    a.scale_fmt = L.FP4_SCALE_UE8M0
    assert lib.fp4_gemm(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(16), 1, 0, None) == L.FP4_ERR_UNSUPPORTED


def test_per_row_scale_argument_rules_without_gpu(lib):
    # FP4_TSCALE_ROW (App. B.1's per-row global scale): rowwise E4M3 1x16 into an
    # output flagged sdec_per_row, no workspace; everything else refused before
    # any launch
    from fp4_block_scaled_02_gb300 import _lib as L
    p = L.fp4_quant_params_t(0, 0, 0, 0, 0, L.FP4_TSCALE_ROW, 448.0, 50, 0, 1, 0, 0, 0, 0)
    assert lib.fp4_workspace_bytes(ctypes.byref(p), 256, 512) == 0
    flat = L.fp4_tensor_t(16, 16, 16, 128, 64, 0, 16, 1, 0)
    rows = L.fp4_tensor_t(16, 16, 16, 128, 64, 0, 16, 1, 1)

    def q(params, out, r=128, c=64):
        return lib.fp4_quantize(ctypes.byref(params), ctypes.c_void_p(16), r, c, c, ctypes.byref(out), None, None,
                                None, None, 0, None)
    assert q(p, flat) == L.FP4_ERR_INVALID_ARG            # ROW needs a per-row s_dec output
    cur = L.fp4_quant_params_t(0, 0, 0, 0, 0, L.FP4_TSCALE_CURRENT, 448.0, 50, 0, 1, 0, 0, 0, 0)
    assert q(cur, rows) == L.FP4_ERR_INVALID_ARG          # and only ROW writes one
    p.orient = L.FP4_ORIENT_COLWISE
    colrows = L.fp4_tensor_t(16, 16, 16, 64, 128, 0, 16, 1, 1)
    assert q(p, colrows) == L.FP4_ERR_UNSUPPORTED         # a colwise row spans the whole tensor
    p.orient = L.FP4_ORIENT_ROWWISE
    p.scale_fmt = rows.scale_fmt = L.FP4_SCALE_UE5M3
    assert q(p, rows) == L.FP4_ERR_UNSUPPORTED            # E4M3 only
    p.tscale = 4
    assert q(p, rows) == L.FP4_ERR_INVALID_ARG            # no such mode
    # GEMM: per-row decode scales on A only, E4M3 only
    a = L.fp4_tensor_t(16, 16, 16, 128, 256, 0, 16, 1, 1)
    b = L.fp4_tensor_t(16, 16, 16, 128, 256, 0, 16, 1, 1)
    assert lib.fp4_gemm(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(16), 1, 0, None) == L.FP4_ERR_UNSUPPORTED
    b.sdec_per_row = 2
    assert lib.fp4_gemm(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(16), 1, 0, None) == L.FP4_ERR_INVALID_ARG
    b.sdec_per_row = 0
    a.scale_fmt = b.scale_fmt = L.FP4_SCALE_UE5M3
    assert lib.fp4_gemm(ctypes.byref(a), ctypes.byref(b), ctypes.c_void_p(16), 1, 0, None) == L.FP4_ERR_INVALID_ARG


def test_row_stride_rules_without_gpu(lib):
    # the input's rows lie ld elements apart: ld >= cols and a multiple of 8
    # (each row starts 16-byte aligned); every entry point that reads an input
    # checks it before anything else touches the device
    from fp4_block_scaled_02_gb300 import _lib as L
    p = L.fp4_quant_params_t(0, 0, 0, 0, 0, 0, 448.0, 50, 0, 1, 0, 0, 0, 0)
    pc = L.fp4_quant_params_t(0, 0, 0, L.FP4_ORIENT_COLWISE, 1, 0, 448.0, 50, 1, 1, 0, 0, 0, 0)
    t = L.fp4_tensor_t(16, 16, 16, 128, 128, 0, 16, 1, 0)
    x, ws = ctypes.c_void_p(16), ctypes.c_void_p(16)
    for ld in (127, 120, 132):  # narrower than the input, narrower and unaligned, not a multiple of 8
        assert lib.fp4_quantize(ctypes.byref(p), x, 128, 128, ld, ctypes.byref(t), None, None, None, ws, 1 << 16,
                                None) == L.FP4_ERR_SHAPE, ld
        assert lib.fp4_quantize_noalloc(ctypes.byref(p), x, 128, 128, ld, ctypes.byref(t), None, None, None,
                                        None) == L.FP4_ERR_SHAPE, ld
        assert lib.fp4_quantize_dual(ctypes.byref(p), ctypes.byref(pc), x, 128, 128, ld, ctypes.byref(t),
                                     ctypes.byref(t), None, None, None, None, ws, 1 << 16,
                                     None) == L.FP4_ERR_SHAPE, ld
        assert lib.fp4_tensor_amax(ctypes.byref(p), x, 128, 128, ld, ctypes.c_void_p(16), ws, 1 << 16,
                                   None) == L.FP4_ERR_SHAPE, ld
        assert lib.fp4_tensor_amax_dual(ctypes.byref(p), ctypes.byref(pc), x, 128, 128, ld, ctypes.c_void_p(16),
                                        ctypes.c_void_p(32), ws, 1 << 16, None) == L.FP4_ERR_SHAPE, ld
    # an empty input needs no stride
    assert lib.fp4_quantize(ctypes.byref(p), x, 0, 128, 0, ctypes.byref(L.fp4_tensor_t(16, 16, 16, 0, 128, 0, 16, 1, 0)),
                            None, None, None, None, 0, None) == L.FP4_OK


def test_noalloc_argument_errors_come_before_the_scratch_lookup(lib):
    # an invalid call is refused by its argument checks alone: no CUDA call is
    # made (without a GPU a device lookup would report FP4_ERR_CUDA instead)
    from fp4_block_scaled_02_gb300 import _lib as L
    p = L.fp4_quant_params_t(0, 0, 0, 0, 1, 0, 448.0, 50, 0, 1, 0, 0, 0, 0)  # RHT on a rowwise operand
    t = L.fp4_tensor_t(16, 16, 16, 128, 64, 0, 16, 1, 0)
    assert lib.fp4_quantize_noalloc(ctypes.byref(p), ctypes.c_void_p(16), 128, 64, 64, ctypes.byref(t), None, None,
                                    None, None) == L.FP4_ERR_INVALID_ARG
    p.rht = 0
    assert lib.fp4_quantize_noalloc(ctypes.byref(p), ctypes.c_void_p(8), 128, 64, 64, ctypes.byref(t), None, None,
                                    None, None) == L.FP4_ERR_ALIGNMENT


def test_status_record_and_aliases_without_gpu(lib):
    from fp4_block_scaled_02_gb300 import _lib as L
    assert lib.fp4_device_status_record(None, None) == L.FP4_ERR_INVALID_ARG
    assert lib.fp4_device_status_record(ctypes.c_void_p(18), None) == L.FP4_ERR_INVALID_ARG  # not 4-byte aligned
    p = L.fp4_quant_params_t(0, 0, 0, 0, 0, 0, 448.0, 50, 0, 1, 0, 0, 0, 0)
    c1, s1, c2, s2 = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.fp4_quantized_bytes(ctypes.byref(p), 256, 512, ctypes.byref(c1), ctypes.byref(s1)) == 0
    assert lib.fp4_quantized_sizes(ctypes.byref(p), 256, 512, ctypes.byref(c2), ctypes.byref(s2)) == 0
    assert (c1.value, s1.value) == (c2.value, s2.value)
