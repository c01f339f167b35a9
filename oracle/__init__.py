"""CPU oracle for the FP4 block-scaled quantized linear layer.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``fp4_block_scaled_02_gb300``) never imports it, and
this package imports nothing from the product: the two share only the seeded
input generators, which hold none of the method's arithmetic.

The arithmetic lives in ``fp4_oracle.c`` (plain C, binary32 step by step as
"Pretraining Large Language Models with NVFP4", App. B, defines it; binary64 for
the GEMM sums). This module compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# scale formats / block shapes (must match fp4_oracle.c)
FMT_E4M3, FMT_UE5M3, FMT_UE8M0 = 0, 1, 2
BLOCK_1x16, BLOCK_16x16, BLOCK_1x32 = 0, 1, 2
OK, ERR_ARG, ERR_SHAPE, ERR_STATE = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            i64, u64, u32, i32, f32 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_int, ctypes.c_float)
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f32.restype = f32
            L.orc_e2m1_value.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_value.restype = ctypes.c_double
            L.orc_minifloat_round.argtypes = [ctypes.c_double, i32, i32, i32, ctypes.c_double]
            L.orc_minifloat_round.restype = ctypes.c_double
            L.orc_scale_decode.argtypes = [i32, ctypes.c_uint8]
            L.orc_scale_decode.restype = ctypes.c_double
            L.orc_scale_encode.argtypes = [i32, f32]
            L.orc_scale_encode.restype = ctypes.c_uint8
            L.orc_scale_max.argtypes = [i32]
            L.orc_scale_max.restype = ctypes.c_double
            L.orc_e2m1_rne.argtypes = [f32]
            L.orc_e2m1_rne.restype = ctypes.c_uint8
            L.orc_e2m1_sr.argtypes = [f32, u32]
            L.orc_e2m1_sr.restype = ctypes.c_uint8
            L.orc_ue8m0_exponent.argtypes = [f32]
            L.orc_ue8m0_exponent.restype = i32
            L.orc_philox4x32_10.argtypes = [P, P, P]
            L.orc_philox4x32_10.restype = None
            L.orc_sr_bits.argtypes = [u64, u32, u64, u64]
            L.orc_sr_bits.restype = u32
            L.orc_rht_sign_word.argtypes = [u64]
            L.orc_rht_sign_word.restype = u32
            L.orc_rht16.argtypes = [P, u32]
            L.orc_rht16.restype = None
            L.orc_tensor_amax.argtypes = [P, i64, i64, i32, i32, u64]
            L.orc_tensor_amax.restype = f32
            L.orc_global_encode_scale.argtypes = [f32, f32]
            L.orc_global_encode_scale.restype = f32
            L.orc_quantize.argtypes = [i32, i32, i32, i32, i32, u64, u32, u64, i32, f32, u32,
                                       P, P, P, P, i64, i64, i64, i64, P, P, P, P, P, i32, P]
            L.orc_quantize.restype = i32
            L.orc_dequantize.argtypes = [i32, i32, i64, i64, P, P, f32, P, P]
            L.orc_dequantize.restype = None
            L.orc_gemm.argtypes = [i32, i32, i64, i64, i64, P, P, f32, P, P, P, f32, P, P, i64, P, P]
            L.orc_gemm.restype = None
            L.orc_swizzle_scales.argtypes = [i64, i64, P, P]
            L.orc_swizzle_scales.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__({ERR_ARG: "invalid argument", ERR_SHAPE: "bad shape",
                          ERR_STATE: "held-amax state error (reserved)"}.get(code, str(code)))
        self.code = code


# --------------------------------------------------------------------------- formats
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e2m1_rne(v: float) -> int:
    return lib().orc_e2m1_rne(v)


def e2m1_sr(v: float, r: int) -> int:
    return lib().orc_e2m1_sr(v, r)


def scale_encode(fmt: int, s: float) -> int:
    return lib().orc_scale_encode(fmt, s)


def scale_decode(fmt: int, code: int) -> float:
    return lib().orc_scale_decode(fmt, code)


def scale_max(fmt: int) -> float:
    return lib().orc_scale_max(fmt)


def minifloat_round(x: float, ebits: int, mbits: int, bias: int, maxval: float) -> float:
    return lib().orc_minifloat_round(x, ebits, mbits, bias, maxval)


def ue8m0_exponent(amax: float) -> int:
    return lib().orc_ue8m0_exponent(amax)


def global_encode_scale(amax: float, target_T: float) -> float:
    return lib().orc_global_encode_scale(amax, target_T)


# --------------------------------------------------------------------------- RNG, RHT
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_bits(seed: int, tensor_id: int, step: int, e: int) -> int:
    return lib().orc_sr_bits(seed, tensor_id, step, e)


def rht_sign_word(seed: int) -> int:
    return lib().orc_rht_sign_word(seed)


def rht16(v, seed: int) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(16)).copy()
    lib().orc_rht16(_p(a), rht_sign_word(seed))
    return a


# --------------------------------------------------------------------------- quantizer
class HeldState:
    """Held-amax record of one tensor ([UE] periodic tensor scaling)."""

    def __init__(self):
        self.amax = np.zeros(1, dtype=np.float32)
        self.valid = np.zeros(1, dtype=np.int32)
        self.last = np.zeros(1, dtype=np.uint64)

    def copy(self) -> "HeldState":
        s = HeldState()
        s.amax[:] = self.amax
        s.valid[:] = self.valid
        s.last[:] = self.last
        return s


def tensor_amax(x_bits: np.ndarray, colwise: bool = False, rht: bool = False, seed: int = 0) -> float:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, C = x.shape
    return lib().orc_tensor_amax(_p(x), R, C, int(colwise), int(rht), seed)


def quantize(x_bits: np.ndarray, *, scale_fmt: int = FMT_E4M3, block: int = BLOCK_1x16,
             sr: bool = False, colwise: bool = False, rht: bool = False, seed: int = 0,
             tensor_id: int = 0, step: int = 0, held: bool = False, target_T: float = 448.0,
             refresh_every: int = 50, state: HeldState | None = None,
             op_rows: tuple[int, int] | None = None, per_row: bool = False) -> dict:
    """Quantize a row-major BF16 bit array ``x_bits`` (rows x cols, uint16).

    Returns codes (R' x C'/2 uint8), plain scales (R' x C'/bs uint8), s_dec (float),
    amax (float) and counters (uint64[4]) for operand rows ``op_rows`` (default all).
    With ``per_row`` each operand row has its own tensor scale ([NV] B.1's finer
    granularity): ``s_dec_rows`` (float32 per returned row) holds them and s_dec is 0.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    R, C = (cols, rows) if colwise else (rows, cols)
    bs = 32 if block == BLOCK_1x32 else 16
    r0, r1 = op_rows if op_rows is not None else (0, R)
    codes = np.zeros((r1 - r0, C // 2), dtype=np.uint8)
    scales = np.zeros((r1 - r0, C // bs), dtype=np.uint8)
    sdec = np.zeros(1, dtype=np.float32)
    amax = np.zeros(1, dtype=np.float32)
    counters = np.zeros(4, dtype=np.uint64)
    sdec_rows = np.zeros(r1 - r0, dtype=np.float32)
    st = state if state is not None else HeldState()
    rc = lib().orc_quantize(scale_fmt, block, int(sr), int(colwise), int(rht), seed, tensor_id, step,
                            int(held), target_T, refresh_every, _p(st.amax), _p(st.valid), _p(st.last),
                            _p(x), rows, cols, r0, r1, _p(codes), _p(scales), _p(sdec), _p(amax),
                            _p(counters), int(per_row), _p(sdec_rows) if per_row else None)
    if rc != OK:
        raise OracleError(rc)
    out = {"codes": codes, "scales": scales, "s_dec": float(sdec[0]), "amax": float(amax[0]),
           "counters": counters}
    if per_row:
        out["s_dec_rows"] = sdec_rows
    return out


def _sdec_arg(s_dec, n: int):
    """A tensor decode scale (float) or one per row (array of n floats)."""
    if np.ndim(s_dec) == 0:
        return float(s_dec), None
    rows = np.ascontiguousarray(s_dec, dtype=np.float32)
    assert rows.shape == (n,)
    return 0.0, rows


def dequantize(codes: np.ndarray, scales: np.ndarray, s_dec, scale_fmt: int = FMT_E4M3,
               bs: int = 16) -> np.ndarray:
    """s_dec: the tensor decode scale, or an array with one per row."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    R, C = c.shape[0], c.shape[1] * 2
    out = np.zeros((R, C), dtype=np.float32)
    sd, rows = _sdec_arg(s_dec, R)
    lib().orc_dequantize(scale_fmt, bs, R, C, _p(c), _p(s), sd, _p(rows) if rows is not None else None, _p(out))
    return out


def gemm(a_codes, a_scales, a_sdec, b_codes, b_scales, b_sdec, *, scale_fmt: int = FMT_E4M3,
         bs: int = 16, pairs: tuple[np.ndarray, np.ndarray] | None = None):
    """FP64 block-scaled GEMM C = A B^T of two K-major quantized operands.

    Returns (C_ref, S) where S = |alpha| sum |a b| is the error-bound scale. With
    ``pairs=(ms, ns)`` only those outputs are computed (1-D arrays). ``a_sdec``
    may be an array with one decode scale per row of A."""
    ac = np.ascontiguousarray(a_codes, dtype=np.uint8)
    asc = np.ascontiguousarray(a_scales, dtype=np.uint8)
    bc = np.ascontiguousarray(b_codes, dtype=np.uint8)
    bsc = np.ascontiguousarray(b_scales, dtype=np.uint8)
    M, K = ac.shape[0], ac.shape[1] * 2
    N = bc.shape[0]
    assert bc.shape[1] * 2 == K
    sa, rows = _sdec_arg(a_sdec, M)
    sa_rows = _p(rows) if rows is not None else None
    if pairs is None:
        c = np.zeros((M, N), dtype=np.float64)
        s = np.zeros((M, N), dtype=np.float64)
        lib().orc_gemm(scale_fmt, bs, M, N, K, _p(ac), _p(asc), sa, sa_rows, _p(bc), _p(bsc), b_sdec,
                       None, None, 0, _p(c), _p(s))
    else:
        ms = np.ascontiguousarray(pairs[0], dtype=np.int64)
        ns = np.ascontiguousarray(pairs[1], dtype=np.int64)
        c = np.zeros(ms.shape[0], dtype=np.float64)
        s = np.zeros(ms.shape[0], dtype=np.float64)
        lib().orc_gemm(scale_fmt, bs, M, N, K, _p(ac), _p(asc), sa, sa_rows, _p(bc), _p(bsc), b_sdec,
                       _p(ms), _p(ns), ms.shape[0], _p(c), _p(s))
    return c, s


def swizzle_scales(plain: np.ndarray) -> np.ndarray:
    """Plain R x NB scales -> the tensor-core chunk layout (flat uint8, R*NB bytes)."""
    p = np.ascontiguousarray(plain, dtype=np.uint8)
    R, NB = p.shape
    out = np.zeros(R * NB, dtype=np.uint8)
    rc = lib().orc_swizzle_scales(R, NB, _p(p), _p(out))
    if rc != OK:
        raise OracleError(rc)
    return out
