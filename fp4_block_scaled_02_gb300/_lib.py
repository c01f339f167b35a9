"""ctypes binding of libfp4bs.so (include/fp4bs.h).

Argument marshalling only: every step of the quantizer and the GEMMs runs in
the CUDA library. PyTorch provides device memory and streams. If the library
is missing the calls raise; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(HERE, "_build", "libfp4bs.so")

# fp4_status_t
FP4_OK = 0
FP4_ERR_INVALID_ARG = 1
FP4_ERR_UNSUPPORTED = 2
FP4_ERR_SHAPE = 3
FP4_ERR_ALIGNMENT = 4
FP4_ERR_STATE = 5
FP4_ERR_CUDA = 6
FP4_ERR_DEVICE_TIMEOUT = 7
FP4_ERR_WORKSPACE = 8

# enums
FP4_SCALE_E4M3, FP4_SCALE_UE5M3, FP4_SCALE_UE8M0 = 0, 1, 2
FP4_BLOCK_1x16, FP4_BLOCK_16x16, FP4_BLOCK_1x32 = 0, 1, 2
FP4_ROUND_RNE, FP4_ROUND_SR = 0, 1
FP4_TSCALE_CURRENT, FP4_TSCALE_HELD, FP4_TSCALE_GIVEN, FP4_TSCALE_ROW = 0, 1, 2, 3
FP4_ORIENT_ROWWISE, FP4_ORIENT_COLWISE = 0, 1
FP4_LAYOUT_PLAIN, FP4_LAYOUT_TCGEN05 = 0, 1

EXPORTED = ["fp4_quantized_sizes", "fp4_workspace_bytes", "fp4_quantize", "fp4_dequantize", "fp4_gemm",
            "fp4_linear_fprop", "fp4_linear_dgrad", "fp4_linear_wgrad", "fp4_device_status",
            "fp4_status_string", "fp4_abi_version", "fp4_quantize_noalloc", "fp4_quantize_dual",
            "fp4_gemm_workspace_bytes", "fp4_gemm_ws", "fp4_tensor_amax", "fp4_tensor_amax_dual",
            "fp4_selftest_wait_timeout", "fp4_selftest_div6", "fp4_device_status_record", "fp4_last_device_status",
            "fp4_quantized_bytes"]


class fp4_quant_params_t(ctypes.Structure):
    _fields_ = [("scale_fmt", ctypes.c_int32), ("block", ctypes.c_int32), ("round", ctypes.c_int32),
                ("orient", ctypes.c_int32), ("rht", ctypes.c_int32), ("tscale", ctypes.c_int32),
                ("target_T", ctypes.c_float), ("refresh_every", ctypes.c_uint32),
                ("tensor_id", ctypes.c_uint32), ("scale_layout", ctypes.c_int32),
                ("emit_transpose", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("seed", ctypes.c_uint64), ("step", ctypes.c_uint64)]


class fp4_tensor_t(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("s_dec_global", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("scale_fmt", ctypes.c_int32),
                ("block_k", ctypes.c_int32), ("scale_layout", ctypes.c_int32),
                ("sdec_per_row", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


class Fp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.fp4_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load the library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(SO_PATH):
                raise RuntimeError(f"libfp4bs.so is not built ({SO_PATH}); run __graft_entry__.build() "
                                   "or python fp4_block_scaled_02_gb300/build.py")
            L = ctypes.CDLL(SO_PATH)
            P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            QP = ctypes.POINTER(fp4_quant_params_t)
            TP = ctypes.POINTER(fp4_tensor_t)
            L.fp4_quantized_sizes.argtypes = [QP, i64, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            L.fp4_quantized_sizes.restype = i32
            L.fp4_quantized_bytes.argtypes = [QP, i64, i64, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            L.fp4_quantized_bytes.restype = i32
            L.fp4_workspace_bytes.argtypes = [QP, i64, i64]
            L.fp4_workspace_bytes.restype = sz
            L.fp4_quantize.argtypes = [QP, P, i64, i64, i64, TP, TP, P, P, P, sz, P]
            L.fp4_quantize.restype = i32
            L.fp4_quantize_dual.argtypes = [QP, QP, P, i64, i64, i64, TP, TP, P, P, P, P, P, sz, P]
            L.fp4_quantize_dual.restype = i32
            L.fp4_quantize_noalloc.argtypes = [QP, P, i64, i64, i64, TP, TP, P, P, P]
            L.fp4_quantize_noalloc.restype = i32
            L.fp4_tensor_amax.argtypes = [QP, P, i64, i64, i64, P, P, sz, P]
            L.fp4_tensor_amax.restype = i32
            L.fp4_tensor_amax_dual.argtypes = [QP, QP, P, i64, i64, i64, P, P, P, sz, P]
            L.fp4_tensor_amax_dual.restype = i32
            L.fp4_dequantize.argtypes = [TP, P, i32, P]
            L.fp4_dequantize.restype = i32
            L.fp4_gemm.argtypes = [TP, TP, P, i32, i32, P]
            L.fp4_gemm.restype = i32
            L.fp4_gemm_workspace_bytes.argtypes = [TP, TP]
            L.fp4_gemm_workspace_bytes.restype = sz
            L.fp4_gemm_ws.argtypes = [TP, TP, P, i32, i32, P, sz, P]
            L.fp4_gemm_ws.restype = i32
            L.fp4_linear_fprop.argtypes = [TP, TP, P, P]
            L.fp4_linear_fprop.restype = i32
            L.fp4_linear_dgrad.argtypes = [TP, TP, P, P]
            L.fp4_linear_dgrad.restype = i32
            L.fp4_linear_wgrad.argtypes = [TP, TP, P, i32, P]
            L.fp4_linear_wgrad.restype = i32
            L.fp4_selftest_wait_timeout.argtypes = [ctypes.c_uint32, P]
            L.fp4_selftest_wait_timeout.restype = i32
            L.fp4_selftest_div6.argtypes = [P, P, i64, P]
            L.fp4_selftest_div6.restype = i32
            L.fp4_device_status.argtypes = [P]
            L.fp4_device_status.restype = i32
            L.fp4_last_device_status.argtypes = [P]
            L.fp4_last_device_status.restype = i32
            L.fp4_device_status_record.argtypes = [P, P]
            L.fp4_device_status_record.restype = i32
            L.fp4_status_string.argtypes = [i32]
            L.fp4_status_string.restype = ctypes.c_char_p
            L.fp4_abi_version.argtypes = []
            L.fp4_abi_version.restype = i32
            _lib = L
    return _lib


def check(status: int, where: str) -> None:
    if status != FP4_OK:
        raise Fp4Error(status, where)
