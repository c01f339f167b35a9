"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import fp4_block_scaled_02_gb300 as fb
import oracle

FMT_TO_ORACLE = {fb.FP4_SCALE_E4M3: oracle.FMT_E4M3, fb.FP4_SCALE_UE5M3: oracle.FMT_UE5M3,
                 fb.FP4_SCALE_UE8M0: oracle.FMT_UE8M0}
BLOCK_TO_ORACLE = {fb.FP4_BLOCK_1x16: oracle.BLOCK_1x16, fb.FP4_BLOCK_16x16: oracle.BLOCK_16x16,
                   fb.FP4_BLOCK_1x32: oracle.BLOCK_1x32}


def to_gpu_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


def new_ws():
    return torch.zeros(4096, dtype=torch.float32, device="cuda")


def gpu_quantize(cfg: fb.QuantConfig, bits: np.ndarray, state=None, with_transpose=False):
    rows, cols = bits.shape
    colwise = cfg.orient == fb.FP4_ORIENT_COLWISE
    R, C = (cols, rows) if colwise else (rows, cols)
    out = fb.QTensor.empty(R, C, cfg.scale_fmt, cfg.layout)
    out.codes.fill_(0xAA)
    out.scales.fill_(0xAA)
    out_t = None
    if with_transpose:
        out_t = fb.QTensor.empty(C, R, cfg.scale_fmt, cfg.layout)
    counters = torch.zeros(4, dtype=torch.int64, device="cuda")
    fb.fp4_quantize(cfg, to_gpu_bf16(bits), out, out_t, state=state, counters=counters, ws=new_ws())
    torch.cuda.synchronize()
    return out, out_t, counters


def oracle_quantize(cfg: fb.QuantConfig, bits: np.ndarray, state=None, colwise=None):
    return oracle.quantize(
        bits, scale_fmt=FMT_TO_ORACLE[cfg.scale_fmt], block=BLOCK_TO_ORACLE[cfg.block],
        sr=cfg.round == fb.FP4_ROUND_SR,
        colwise=(cfg.orient == fb.FP4_ORIENT_COLWISE) if colwise is None else colwise,
        rht=cfg.rht, seed=cfg.seed, tensor_id=cfg.tensor_id, step=cfg.step,
        held=cfg.tscale == fb.FP4_TSCALE_HELD, target_T=cfg.target_T, refresh_every=cfg.refresh_every,
        state=state)


def expected_scale_bytes(plain: np.ndarray, layout: int) -> np.ndarray:
    if layout == fb.FP4_LAYOUT_TCGEN05:
        return oracle.swizzle_scales(plain)
    return plain.reshape(-1)


def assert_quant_equal(gpu: fb.QTensor, ref: dict, layout: int, counters=None, check_sdec=True):
    codes = gpu.codes.cpu().numpy()
    assert np.array_equal(codes, ref["codes"]), _first_diff(codes, ref["codes"])
    sc = gpu.scales.cpu().numpy()
    want = expected_scale_bytes(ref["scales"], layout)
    assert np.array_equal(sc, want), _first_diff(sc, want)
    if check_sdec:
        got = gpu.s_dec[0:1].cpu().numpy().view(np.uint32)[0]
        exp = np.array([ref["s_dec"]], dtype=np.float32).view(np.uint32)[0]
        assert got == exp, (hex(got), hex(exp))
    if counters is not None:
        assert counters.cpu().numpy().astype(np.uint64).tolist() == ref["counters"].tolist()


def _first_diff(a, b):
    a, b = np.asarray(a).reshape(-1), np.asarray(b).reshape(-1)
    if a.shape != b.shape:
        return f"shape {a.shape} vs {b.shape}"
    idx = np.flatnonzero(a != b)
    return f"{idx.size} diffs, first at {idx[:8].tolist()}: {a[idx[:8]].tolist()} vs {b[idx[:8]].tolist()}"


def upload_operand(ref: dict, rows: int, cols: int, scale_fmt=fb.FP4_SCALE_E4M3) -> fb.QTensor:
    """An oracle-quantized operand copied to the device in the tensor-core layout."""
    t = fb.QTensor.empty(rows, cols, scale_fmt, fb.FP4_LAYOUT_TCGEN05)
    t.codes.copy_(torch.from_numpy(ref["codes"]))
    t.scales.copy_(torch.from_numpy(oracle.swizzle_scales(ref["scales"])))
    t.s_dec[0] = ref["s_dec"]
    return t


def gemm_bound_ok(c_gpu: np.ndarray, c_ref: np.ndarray, s: np.ndarray, bf16: bool):
    """|C - C_ref| <= 2^-20 S for FP32 outputs. A BF16 output is the FP32 result
    rounded to nearest with 8 significant bits, an error of at most half an ulp,
    i.e. 2^-8 of the value's magnitude: |C - C_ref| <= 2^-20 S + 2^-8 (|C_ref| + 2^-20 S)."""
    c = c_gpu.astype(np.float64)
    tol = 2.0 ** -20 * s
    if bf16:
        tol = tol + 2.0 ** -8 * (np.abs(c_ref) + 2.0 ** -20 * s)
    err = np.abs(c - c_ref)
    ok = err <= tol
    ok |= (s == 0) & (c == 0)
    return ok, err, tol
