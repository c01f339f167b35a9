"""GPU parity of per-row tensor scaling (FP4_TSCALE_ROW: "Pretraining Large
Language Models with NVFP4", App. B.1, the global scale at the granularity of a
row) against the oracle: bit-exact codes, scale bytes, per-row s_dec and
counters from the one-pass quantizer; dequantize with per-row s_dec; the GEMM
with one decode scale per row of A within the 2^-20 bound; rejected
combinations.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

fb = pytest.importorskip("fp4_block_scaled_02_gb300")
from gpu_common import expected_scale_bytes, gemm_bound_ok, to_gpu_bf16, upload_operand  # noqa: E402
import oracle  # noqa: E402
from workloads import random_bf16  # noqa: E402

TC, PLAIN = fb.FP4_LAYOUT_TCGEN05, fb.FP4_LAYOUT_PLAIN


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    fb._lib.load()


def _rows_with_spread(seed, shape, dist):
    """Rows whose amaxes spread over many binades (row r scaled by 2^(r % 29 - 14)),
    plus an all-zero row and a row of one nonzero value."""
    bits = random_bf16(seed, shape, dist)
    x = (torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float()).numpy()
    x *= np.exp2((np.arange(shape[0]) % 29 - 14).astype(np.float32))[:, None]
    x[1] = 0.0
    x[2] = 0.0
    x[2, 7] = -3.0e-5
    return torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)


def _quantize_rows(cfg, bits):
    R, C = bits.shape
    out = fb.QTensor.empty(R, C, layout=cfg.layout, per_row=True)
    out.codes.fill_(0xAA)
    out.scales.fill_(0xAA)
    cnt = torch.zeros(4, dtype=torch.int64, device="cuda")
    fb.fp4_quantize(cfg, to_gpu_bf16(bits), out, counters=cnt)
    assert fb.fp4_device_status() == 0
    return out, cnt


CASES = [
    # (shape, dist, round, layout, seed, tensor_id, step)
    ((256, 768), "student_t4", fb.FP4_ROUND_RNE, TC, 0, 0, 0),
    ((384, 512), "log_normal_1e-4_2", fb.FP4_ROUND_SR, TC, 5, 3, 17),
    ((37, 80), "normal_outliers", fb.FP4_ROUND_RNE, PLAIN, 0, 0, 0),
    ((129, 2064), "log_uniform_1e-6_1e-2", fb.FP4_ROUND_SR, PLAIN, 9, 7, 3),  # rows longer than 1024
    ((128, 16), "normal", fb.FP4_ROUND_RNE, PLAIN, 0, 0, 0),                   # one block per row
]


@pytest.mark.parametrize("case", CASES)
def test_rowscale_quantize_matches_oracle(case):
    shape, dist, rnd, layout, seed, tid, step = case
    bits = _rows_with_spread(41, shape, dist)
    cfg = fb.QuantConfig(round=rnd, layout=layout, seed=seed, tensor_id=tid, step=step, tscale=fb.FP4_TSCALE_ROW)
    out, cnt = _quantize_rows(cfg, bits)
    ref = oracle.quantize(bits, sr=rnd == fb.FP4_ROUND_SR, seed=seed, tensor_id=tid, step=step, per_row=True)
    codes = out.codes.cpu().numpy()
    assert np.array_equal(codes, ref["codes"])
    assert np.array_equal(out.scales.cpu().numpy(), expected_scale_bytes(ref["scales"], layout))
    sd = out.s_dec[:shape[0]].cpu().numpy()
    assert np.array_equal(sd.view(np.uint32), ref["s_dec_rows"].view(np.uint32))
    assert cnt.cpu().numpy().astype(np.uint64).tolist() == ref["counters"].tolist()


def test_rowscale_dequantize_per_row():
    bits = _rows_with_spread(42, (256, 512), "normal")
    cfg = fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW)
    out, _ = _quantize_rows(cfg, bits)
    ref = oracle.quantize(bits, per_row=True)
    want = oracle.dequantize(ref["codes"], ref["scales"], ref["s_dec_rows"])
    got = torch.empty((256, 512), dtype=torch.float32, device="cuda")
    fb.fp4_dequantize(out, got)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("M,N,K,out32", [(256, 384, 512, False), (384, 256, 1024, True), (1280, 1152, 768, False)])
def test_gemm_per_row_a_scale(M, N, K, out32):
    bits = _rows_with_spread(43, (M, K), "student_t4")
    a, _ = _quantize_rows(fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW), bits)
    ra = oracle.quantize(bits, per_row=True)
    rb = oracle.quantize(random_bf16(44, (N, K), "weight"))
    b = upload_operand(rb, N, K)
    d = torch.empty((M, N), dtype=torch.float32 if out32 else torch.bfloat16, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec_rows"], rb["codes"], rb["scales"], rb["s_dec"])
    ok, err, tol = gemm_bound_ok(d.float().cpu().numpy(), c_ref, s, bf16=not out32)
    assert ok.all(), f"{(~ok).sum()} outside the bound"
    # the linear-layer entry point (Fprop: x rowwise per row, w tensor-wide) is the same GEMM
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fb.fp4_linear_fprop(a, b, y)
    torch.cuda.synchronize()
    if not out32:
        assert torch.equal(y, d)


def test_rowscale_rejections():
    x = to_gpu_bf16(random_bf16(45, (128, 256), "normal"))
    row = fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW)
    per_row = fb.QTensor.empty(128, 256, per_row=True)
    plain = fb.QTensor.empty(128, 256)
    # the output must carry per-row s_dec, and only ROW writes one
    with pytest.raises(fb.Fp4Error):
        fb.fp4_quantize(row, x, plain)
    with pytest.raises(fb.Fp4Error):
        fb.fp4_quantize(fb.QuantConfig(), x, per_row, ws=torch.zeros(4096, dtype=torch.float32, device="cuda"))
    # rowwise E4M3 1x16 without RHT only
    for cfg, out in ((fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW, orient=fb.FP4_ORIENT_COLWISE),
                      fb.QTensor.empty(256, 128, per_row=True)),
                     (fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW, scale_fmt=fb.FP4_SCALE_UE5M3),
                      fb.QTensor.empty(128, 256, fb.FP4_SCALE_UE5M3, per_row=True))):
        with pytest.raises(fb.Fp4Error):
            fb.fp4_quantize(cfg, x, out)
    # per-row decode scales on B are not supported
    fb.fp4_quantize(row, x, per_row)
    d = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")
    b_rows = fb.QTensor.empty(128, 256, per_row=True)
    fb.fp4_quantize(row, x, b_rows)
    with pytest.raises(fb.Fp4Error):
        fb.fp4_gemm(per_row, b_rows, d)
    # the one-read dual quantizer does not take it
    ws = torch.zeros(8192, dtype=torch.float32, device="cuda")
    with pytest.raises(fb.Fp4Error):
        fb.fp4_quantize_dual(row, fb.QuantConfig(tscale=fb.FP4_TSCALE_ROW, orient=fb.FP4_ORIENT_COLWISE), x,
                             per_row, fb.QTensor.empty(256, 128), ws=ws)
    assert fb.fp4_device_status() == 0
