"""GPU parity of the block-scaled GEMMs against the oracle's FP64 GEMM.

Acceptance per output element: |C - C_ref| <= 2^-20 * S with
S = |alpha| sum_k |a_k b_k| (FP32 outputs), plus half a BF16 ulp of C_ref for
BF16 outputs. Operands are quantized by the oracle and uploaded, so the GEMM is
checked on its own; the end-to-end tests quantize on the GPU, check those bytes
against the oracle, then run the three GEMMs of a linear layer.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

fb = pytest.importorskip("fp4_block_scaled_02_gb300")
from gpu_common import (assert_quant_equal, gemm_bound_ok, oracle_quantize,  # noqa: E402
                        to_gpu_bf16, upload_operand)
import oracle  # noqa: E402
from workloads import WORKLOADS, linear_inputs, random_bf16  # noqa: E402

UE = fb.FP4_SCALE_UE5M3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    fb._lib.load()


def _operand(seed, rows, cols, dist, fmt=fb.FP4_SCALE_E4M3, **kw):
    bits = random_bf16(seed, (rows, cols), dist)
    cfg = fb.QuantConfig(scale_fmt=fmt, **kw)
    ref = oracle_quantize(cfg, bits)
    return ref, upload_operand(ref, rows, cols, fmt)


def _check(c_gpu, c_ref, s, bf16):
    ok, err, tol = gemm_bound_ok(c_gpu, c_ref, s, bf16)
    if not ok.all():
        i = np.flatnonzero(~ok.reshape(-1))[:5]
        raise AssertionError(f"{(~ok).sum()} of {ok.size} outside bound; first {i.tolist()}: "
                             f"gpu {c_gpu.reshape(-1)[i]}, ref {c_ref.reshape(-1)[i]}, tol {tol.reshape(-1)[i]}")


# N % 256 == 0 runs 128 x 256 tiles, other N 128 x 128 tiles; K = 1280 and 2560
# end in a partial accumulator chunk
SHAPES = [(128, 128, 256), (256, 384, 512), (384, 256, 1024), (1280, 1152, 768), (640, 1024, 1280),
          (512, 768, 2560)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out32", [False, True])
def test_gemm_nvfp4_full_output(M, N, K, out32):
    ra, a = _operand(31, M, K, "student_t4")
    rb, b = _operand(32, N, K, "weight")
    d = torch.empty((M, N), dtype=torch.float32 if out32 else torch.bfloat16, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"])
    _check(d.float().cpu().numpy(), c_ref, s, bf16=not out32)


@pytest.mark.parametrize("M,N,K", [(4096, 2048, 512), (2048, 2176, 1280)])
def test_gemm_nvfp4_persistent_wrap_sampled(M, N, K):
    # more output tiles than SMs (256 tiles of 128 x 256; 272 of 128 x 128): each
    # CTA loops over several tiles and accumulator chunks
    ra, a = _operand(33, M, K, "normal")
    rb, b = _operand(34, N, K, "log_normal_1e-4_2")
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, M, 4000), rng.integers(0, N, 4000)
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                           pairs=(ms, ns))
    _check(d.cpu().numpy()[ms, ns], c_ref, s, bf16=False)


MX = fb.FP4_SCALE_UE8M0


# MXFP4 ("Pretraining Large Language Models with NVFP4", A3): UE8M0 scales per
# 32 values, tcgen05 kind::mxf4; N % 256 selects the tile width as for NVFP4 and
# K = 2304 ends in a partial accumulator chunk
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (384, 256, 1024), (640, 1024, 2304),
                                   (512, 768, 2560)])
@pytest.mark.parametrize("out32", [False, True])
def test_gemm_mxfp4_full_output(M, N, K, out32):
    ra, a = _operand(41, M, K, "student_t4", fmt=MX, block=fb.FP4_BLOCK_1x32)
    rb, b = _operand(42, N, K, "log_normal_1e-4_2", fmt=MX, block=fb.FP4_BLOCK_1x32)
    # MXFP4 has no tensor scale: whatever the s_dec words hold is not read
    a.s_dec.fill_(7.0)
    b.s_dec.fill_(-3.0)
    d = torch.empty((M, N), dtype=torch.float32 if out32 else torch.bfloat16, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], 1.0, rb["codes"], rb["scales"], 1.0,
                           scale_fmt=oracle.FMT_UE8M0, bs=32)
    _check(d.float().cpu().numpy(), c_ref, s, bf16=not out32)


def test_gemm_mxfp4_persistent_wrap_sampled():
    M, N, K = 4096, 2048, 768
    ra, a = _operand(43, M, K, "normal", fmt=MX, block=fb.FP4_BLOCK_1x32)
    rb, b = _operand(44, N, K, "weight", fmt=MX, block=fb.FP4_BLOCK_1x32)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    rng = np.random.default_rng(1)
    ms, ns = rng.integers(0, M, 4000), rng.integers(0, N, 4000)
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], 1.0, rb["codes"], rb["scales"], 1.0,
                           scale_fmt=oracle.FMT_UE8M0, bs=32, pairs=(ms, ns))
    _check(d.cpu().numpy()[ms, ns], c_ref, s, bf16=False)


def test_gemm_mixed_scale_formats_are_rejected():
    _, a = _operand(45, 128, 256, "normal")
    _, b = _operand(46, 128, 256, "normal", fmt=MX, block=fb.FP4_BLOCK_1x32)
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_gemm(a, b, torch.empty((128, 128), dtype=torch.float32, device="cuda"))
    assert e.value.status == fb._lib.FP4_ERR_UNSUPPORTED


def test_gemm_accumulate_fp32():
    M, N, K = 256, 256, 512
    ra, a = _operand(35, M, K, "normal")
    rb, b = _operand(36, N, K, "normal")
    base = torch.randn((M, N), dtype=torch.float32, device="cuda",
                       generator=torch.Generator("cuda").manual_seed(0))
    d = base.clone()
    fb.fp4_linear_wgrad(a, b, d, accumulate=True)
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"])
    got = d.cpu().numpy().astype(np.float64) - base.cpu().numpy().astype(np.float64)
    tol = 2.0 ** -20 * s + 2.0 ** -23 * np.abs(d.cpu().numpy())
    assert np.all(np.abs(got - c_ref) <= tol)


def test_gemm_zero_operand_gives_zero():
    M, N, K = 128, 128, 256
    ra, a = _operand(37, M, K, "normal")
    a.codes.zero_()
    rb, b = _operand(38, N, K, "normal")
    d = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert torch.count_nonzero(d).item() == 0


@pytest.mark.parametrize("K", [2048, 8192, 8448, 21504])
def test_gemm_all_positive_products_within_bound(K):
    """All-positive products are the worst case for an accumulator that loses
    low bits as it adds: the losses never cancel. With every code positive and
    block scales near 1, each output's partial sums grow monotonically over K,
    and the FP32 result must still lie within 2^-20 * sum |a b| of the exact sum
    (App. B.3: FP32 accumulation of the block-scaled products). K runs up to
    21504, the longest dot product of the workloads (the 8B down-projection's
    Fprop and its up-projection's Dgrad); K = 8448 = 33 * 256 ends in a partial
    accumulator chunk of one stage."""
    M, N = 256, 256
    rng = np.random.default_rng(K)

    def positive_operand(rows):
        c = rng.integers(1, 8, size=(rows, K), dtype=np.uint8)  # E2M1 magnitudes 0.5 .. 6
        codes = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
        scales = rng.integers(0x34, 0x3C, size=(rows, K // 16), dtype=np.uint8)  # E4M3 0.625 .. 1.75
        return {"codes": codes, "scales": scales, "s_dec": 1.0}

    ra, rb = positive_operand(M), positive_operand(N)
    a, b = upload_operand(ra, M, K), upload_operand(rb, N, K)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], 1.0, rb["codes"], rb["scales"], 1.0)
    assert np.all(c_ref > 0)
    _check(d.cpu().numpy(), c_ref, s, bf16=False)


def test_gemm_shape_validation():
    _, a = _operand(39, 128, 256, "normal")
    _, b = _operand(40, 128, 256, "normal")
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_gemm(a, b, torch.empty((128, 128), dtype=torch.bfloat16, device="cuda"), accumulate=True)
    assert e.value.status == fb._lib.FP4_ERR_INVALID_ARG
    a.rows = 100
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_gemm(a, b, torch.empty((128, 128), dtype=torch.float32, device="cuda"))
    assert e.value.status == fb._lib.FP4_ERR_SHAPE


def _linear_end_to_end(w, which=0, fmt=fb.FP4_SCALE_E4M3, rht=True, sample=None):
    """Quantize X, W, dY on the GPU per the recipe (checked bit-exact against the
    oracle), run Fprop, Dgrad and Wgrad, and compare each with the oracle GEMM."""
    inp = linear_inputs(w, which)
    lin = w.linears[which]
    T, K, N = lin.tokens, lin.k_in, lin.n_out
    L = fb.Fp4Linear(T, K, N, scale_fmt=fmt, rht=rht, seed=w.rht_seed)
    x, wt, dy = to_gpu_bf16(inp["x"]), to_gpu_bf16(inp["w"]), to_gpu_bf16(inp["dy"])
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    L.step(x, wt, dy, y, dx, dw)
    assert fb.fp4_device_status() == 0
    b = L.bufs
    cfgs = {
        "x": (L._cfg(0, 0), inp["x"]),
        "w": (L._cfg(2, 0, block=fb.FP4_BLOCK_16x16), inp["w"]),
        "wt": (L._cfg(2, 0, block=fb.FP4_BLOCK_16x16, orient=fb.FP4_ORIENT_COLWISE), inp["w"]),
        "dy": (L._cfg(3, 0, round=fb.FP4_ROUND_SR), inp["dy"]),
        "xt": (L._cfg(1, 0, orient=fb.FP4_ORIENT_COLWISE, rht=rht), inp["x"]),
        "dyt": (L._cfg(4, 0, orient=fb.FP4_ORIENT_COLWISE, rht=rht, round=fb.FP4_ROUND_SR), inp["dy"]),
    }
    refs = {}
    for k, (cfg, bits) in cfgs.items():
        refs[k] = oracle_quantize(cfg, bits)
        assert_quant_equal(b[k], refs[k], fb.FP4_LAYOUT_TCGEN05)
    # one counter row per tensor id: X, X^T, W (both orientations, each element
    # once), dY, dY^T
    counters = L.counters.cpu().numpy()
    for row, key in enumerate(("x", "xt", "w", "dy", "dyt")):
        assert counters[row].tolist() == refs[key]["counters"].tolist(), key
    for out, (ka, kb), bf16 in [(y, ("x", "w"), True), (dx, ("dy", "wt"), True), (dw, ("dyt", "xt"), False)]:
        ra, rb = refs[ka], refs[kb]
        if sample is None:
            c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"])
            _check(out.float().cpu().numpy(), c_ref, s, bf16)
        else:
            rng = np.random.default_rng(1)
            ms = rng.integers(0, out.shape[0], sample)
            ns = rng.integers(0, out.shape[1], sample)
            c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                                   pairs=(ms, ns))
            _check(out.float().cpu().numpy()[ms, ns], c_ref, s, bf16)


def test_tiny_linear_end_to_end():
    _linear_end_to_end(WORKLOADS["tiny"])


@pytest.mark.parametrize("which", [0, 1])
def test_1p2b_linear_end_to_end_sampled(which):
    _linear_end_to_end(WORKLOADS["1.2b"], which, sample=3000)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (1280, 1152, 768)])
@pytest.mark.parametrize("out32", [False, True])
def test_gemm_ue5m3_emulated_full_output(M, N, K, out32):
    ra, a = _operand(41, M, K, "log_normal_1e-4_2", fmt=UE, target_T=2048.0)
    rb, b = _operand(42, N, K, "student_t4", fmt=UE, target_T=448.0)
    d = torch.empty((M, N), dtype=torch.float32 if out32 else torch.bfloat16, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                           scale_fmt=oracle.FMT_UE5M3)
    _check(d.float().cpu().numpy(), c_ref, s, bf16=not out32)


def _ws_for(a, b):
    return torch.zeros(fb.fp4_gemm_workspace_bytes(a, b), dtype=torch.uint8, device="cuda")


def _took_native(ws, a, b) -> bool:
    """The rebias pass leaves one zero byte per 128-row tile at the start of the
    workspace when every row of the tile fit."""
    return int(ws[: a.rows // 128 + b.rows // 128].sum().item()) == 0


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (1280, 1152, 768), (512, 1024, 2304),
                                   (512, 1024, 2048)])
@pytest.mark.parametrize("out32", [False, True])
def test_gemm_ue5m3_rebiased_native_full_output(M, N, K, out32):
    """UE5M3 operands on the native MMA after the per-row rebias onto E4M3."""
    ra, a = _operand(41, M, K, "log_normal_1e-4_2", fmt=UE, target_T=2048.0)
    rb, b = _operand(42, N, K, "student_t4", fmt=UE, target_T=448.0)
    d = torch.empty((M, N), dtype=torch.float32 if out32 else torch.bfloat16, device="cuda")
    ws = _ws_for(a, b)
    fb.fp4_gemm(a, b, d, ws=ws)
    assert fb.fp4_device_status() == 0
    assert _took_native(ws, a, b)
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                           scale_fmt=oracle.FMT_UE5M3)
    _check(d.float().cpu().numpy(), c_ref, s, bf16=not out32)


def _set_row(scales, r, codes):
    scales[r, :] = np.resize(np.array(codes, dtype=np.uint8), scales.shape[1])


def test_gemm_ue5m3_rebias_edges_and_fallback():
    """Rows at the edge of what one E4M3 offset covers: the largest scale with
    mantissa 7 (placed at E4M3 exponent 7) and the smallest 13 binades below;
    mantissa <= 6 (exponent 8) with the smallest 14 binades below; UE5M3
    subnormal scales. All fit and run natively. One more binade in a single row
    sends the output tiles of its 128-row tile to the emulated kernel while the
    native kernel computes the rest; then one more row of B does the same for
    its tile column (the emulated kernel numbers both kinds of flagged tiles and
    splits their K over the idle SMs). Every output gives the oracle's sums."""
    M, N, K = 256, 256, 512
    ra, _ = _operand(45, M, K, "normal", fmt=UE)
    rb, _ = _operand(46, N, K, "weight", fmt=UE)
    sa, sb = ra["scales"].copy(), rb["scales"].copy()
    _set_row(sa, 0, [0xA7, 0x38, 0x60, 0x80, 0x00])   # E 5 (f 7) .. -8
    _set_row(sa, 130, [0xA6, 0x30, 0x99])              # E 5 (f 6) .. -9
    _set_row(sb, 7, [0x50, 0x01, 0x03, 0x07, 0x0F])    # E -5 .. -17 (subnormals)
    _set_row(sb, 255, [0x00])                          # all-zero row
    for fallback in (False, True, "a_and_b"):
        if fallback:
            _set_row(sa, 9, [0xA7, 0x30])              # 14 binades under a mantissa-7 maximum
        if fallback == "a_and_b":
            _set_row(sb, 200, [0xA7, 0x30])            # and in B's second 128-row tile
        ra2, rb2 = dict(ra, scales=sa), dict(rb, scales=sb)
        a, b = upload_operand(ra2, M, K, UE), upload_operand(rb2, N, K, UE)
        for out32 in (False, True):
            d = torch.empty((M, N), dtype=torch.float32 if out32 else torch.bfloat16, device="cuda")
            ws = _ws_for(a, b)
            fb.fp4_gemm(a, b, d, ws=ws)
            assert fb.fp4_device_status() == 0
            assert _took_native(ws, a, b) == (fallback is False)
            c_ref, s = oracle.gemm(ra2["codes"], sa, ra2["s_dec"], rb2["codes"], sb, rb2["s_dec"],
                                   scale_fmt=oracle.FMT_UE5M3)
            _check(d.float().cpu().numpy(), c_ref, s, bf16=not out32)


def test_gemm_ue5m3_fallback_more_tiles_than_sms_on_narrow_tiles():
    """A B row that does not fit, with N % 256 != 0 (the native kernel runs
    128 x 128 tiles, so only that tile column falls back) and 160 A row tiles:
    160 flagged output tiles, more than the SMs, so the emulated kernel deals
    them out from its lists without splitting K. Whole 128-row tiles (the
    first, a middle one and the last; output rows are independent) give the
    oracle's sums."""
    M, N, K = 160 * 128, 384, 256
    ra, a = _operand(61, M, K, "normal", fmt=UE)
    rb, _ = _operand(62, N, K, "weight", fmt=UE)
    sb = rb["scales"].copy()
    _set_row(sb, 140, [0xA7, 0x30])  # 14 binades under a mantissa-7 maximum, B's tile 1
    rb2 = dict(rb, scales=sb)
    b = upload_operand(rb2, N, K, UE)
    d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = _ws_for(a, b)
    fb.fp4_gemm(a, b, d, ws=ws)
    assert fb.fp4_device_status() == 0
    flags = ws[: M // 128 + N // 128].cpu().numpy()
    assert flags[: M // 128].sum() == 0 and flags[M // 128:].tolist() == [0, 1, 0]
    out = d.float().cpu().numpy()
    for t in (0, 79, 159):
        r = slice(128 * t, 128 * (t + 1))
        c_ref, s = oracle.gemm(ra["codes"][r], ra["scales"][r], ra["s_dec"], rb2["codes"], sb, rb2["s_dec"],
                               scale_fmt=oracle.FMT_UE5M3)
        _check(out[r], c_ref, s, bf16=True)


def test_gemm_ue5m3_workspace_checks():
    _, a = _operand(47, 128, 256, "normal", fmt=UE)
    _, b = _operand(48, 128, 256, "normal", fmt=UE)
    need = fb.fp4_gemm_workspace_bytes(a, b)
    assert need >= 2 * 128 * 256 // 16
    d = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_gemm(a, b, d, ws=torch.empty(need - 16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == fb._lib.FP4_ERR_WORKSPACE
    _, c = _operand(49, 128, 256, "normal")
    assert fb.fp4_gemm_workspace_bytes(c, c) == 0  # NVFP4 needs none


@pytest.mark.parametrize("native", [False, True])
def test_gemm_ue5m3_wide_scale_range_sampled(native):
    # scales spread over many binades: a x10^3 drift against a held amax
    # saturates some blocks and drives others toward the UE5M3 subnormals
    M, N, K = 1024, 1024, 1024
    from workloads import bf16_bits_to_f32, f32_to_bf16_bits
    bits = random_bf16(43, (M, K), "log_normal_1e-4_2")
    cfg = fb.QuantConfig(scale_fmt=UE, tscale=fb.FP4_TSCALE_HELD, target_T=2048.0)
    st = oracle.HeldState()
    oracle_quantize(cfg, bits, state=st)
    cfg.step = 1
    drift = f32_to_bf16_bits(bf16_bits_to_f32(bits) * np.float32(1e3))
    ra = oracle_quantize(cfg, drift, state=st)
    assert ra["counters"][2] > 0
    a = upload_operand(ra, M, K, UE)
    rb, b = _operand(44, N, K, "weight", fmt=UE)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d, ws=_ws_for(a, b) if native else None)
    assert fb.fp4_device_status() == 0
    rng = np.random.default_rng(2)
    ms, ns = rng.integers(0, M, 3000), rng.integers(0, N, 3000)
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                           scale_fmt=oracle.FMT_UE5M3, pairs=(ms, ns))
    _check(d.cpu().numpy()[ms, ns], c_ref, s, bf16=False)


@pytest.mark.parametrize("T_target,native", [(448.0, False), (2048.0, False), (448.0, True), (2048.0, True)])
def test_ue5m3_periodic_scaling_sweep_steps(T_target, native):
    """Sweep workload (4096 -> 4096, T = 8192): held amax refreshed every 50 steps,
    UE5M3 scales, SR on gradients, no RHT, emulated or rebiased native GEMMs. Steps 0, 49, 50, 99
    run in order on the GPU and the oracle; quantized bytes, counters and held
    state match exactly and sampled GEMM outputs meet the bound."""
    from workloads import sweep_dy
    w = WORKLOADS["ue5m3_sweep"]
    lin = w.linears[0]
    inp = linear_inputs(w, 0)
    T, K, N = lin.tokens, lin.k_in, lin.n_out
    L = fb.Fp4Linear(T, K, N, scale_fmt=UE, rht=False, held=True, target_T=T_target, seed=w.sr_seed,
                     ue5m3_native=native)
    x, wt = to_gpu_bf16(inp["x"]), to_gpu_bf16(inp["w"])
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    states = {k: oracle.HeldState() for k in ("x", "w", "wt", "dy", "xt", "dyt")}
    rng = np.random.default_rng(3)
    for step in (0, 49, 50, 99):
        dyb = sweep_dy(inp["dy"], step, w.steps)
        L.counters.zero_()
        L.step(x, wt, to_gpu_bf16(dyb), y, dx, dw, step=step)
        assert fb.fp4_device_status() == 0
        cfgs = {
            "x": (L._cfg(0, step), inp["x"], 0),
            "w": (L._cfg(2, step, block=fb.FP4_BLOCK_16x16), inp["w"], 2),
            # W^T shares W's quantize call, held amax and counter row
            "wt": (L._cfg(2, step, block=fb.FP4_BLOCK_16x16, orient=fb.FP4_ORIENT_COLWISE), inp["w"], None),
            "dy": (L._cfg(3, step, round=fb.FP4_ROUND_SR), dyb, 3),
            "xt": (L._cfg(1, step, orient=fb.FP4_ORIENT_COLWISE), inp["x"], 1),
            "dyt": (L._cfg(4, step, orient=fb.FP4_ORIENT_COLWISE, round=fb.FP4_ROUND_SR), dyb, 4),
        }
        refs = {}
        for k, (cfg, bits, ci) in cfgs.items():
            refs[k] = oracle_quantize(cfg, bits, state=states[k])
            assert_quant_equal(L.bufs[k], refs[k], fb.FP4_LAYOUT_TCGEN05)
            if ci is None:
                continue
            assert L.counters[ci].cpu().numpy().tolist() == refs[k]["counters"].tolist(), (step, k)
            gst = L.states[ci]
            assert np.float32(gst.amax) == states[k].amax[0] and gst.last_refresh_step == int(states[k].last[0])
        ms, ns = rng.integers(0, T, 1500), rng.integers(0, N, 1500)
        for out, (ka, kb), bf16 in [(y, ("x", "w"), True), (dx, ("dy", "wt"), True), (dw, ("dyt", "xt"), False)]:
            ra, rb = refs[ka], refs[kb]
            mm = ms % out.shape[0]
            nn = ns % out.shape[1]
            c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                                   scale_fmt=oracle.FMT_UE5M3, pairs=(mm, nn))
            _check(out.float().cpu().numpy()[mm, nn], c_ref, s, bf16)


def _banded_linear(w, which, band=128, samples=1000):
    """Full-size linear of a large workload: the GPU runs the whole recipe; the
    oracle quantizes three bands of `band` operand rows of every operand -- the
    first, the last and one at random (the tensor amax still covers the whole
    tensor) -- whose bytes must match the GPU's exactly, and GEMM outputs sampled
    where the bands cross must meet the bound: in the first output tile, in the
    last one (past the first persistent wave of tiles) and in a random one."""
    inp = linear_inputs(w, which)
    lin = w.linears[which]
    T, K, N = lin.tokens, lin.k_in, lin.n_out
    L = fb.Fp4Linear(T, K, N, rht=True, seed=w.rht_seed)
    x, wt, dy = to_gpu_bf16(inp["x"]), to_gpu_bf16(inp["w"]), to_gpu_bf16(inp["dy"])
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    L.step(x, wt, dy, y, dx, dw)
    assert fb.fp4_device_status() == 0
    rng = np.random.default_rng(5)
    cfgs = {
        "x": (L._cfg(0, 0), inp["x"], T),
        "w": (L._cfg(2, 0, block=fb.FP4_BLOCK_16x16), inp["w"], N),
        "wt": (L._cfg(2, 0, block=fb.FP4_BLOCK_16x16, orient=fb.FP4_ORIENT_COLWISE), inp["w"], K),
        "dy": (L._cfg(3, 0, round=fb.FP4_ROUND_SR), inp["dy"], T),
        "xt": (L._cfg(1, 0, orient=fb.FP4_ORIENT_COLWISE, rht=True), inp["x"], K),
        "dyt": (L._cfg(4, 0, orient=fb.FP4_ORIENT_COLWISE, rht=True, round=fb.FP4_ROUND_SR), inp["dy"], N),
    }
    refs, r0s = {}, {}
    for k, (cfg, bits, R) in cfgs.items():
        r0s[k] = [0, R - band, int(rng.integers(1, R // band - 1)) * band]
        refs[k] = []
        q = L.bufs[k]
        nb = q.cols // 16
        for r0 in r0s[k]:
            ref = oracle.quantize(bits, scale_fmt=oracle.FMT_E4M3,
                                  block=oracle.BLOCK_16x16 if cfg.block == fb.FP4_BLOCK_16x16 else oracle.BLOCK_1x16,
                                  sr=cfg.round == fb.FP4_ROUND_SR, colwise=cfg.orient == fb.FP4_ORIENT_COLWISE,
                                  rht=cfg.rht, seed=cfg.seed, tensor_id=cfg.tensor_id, step=0,
                                  op_rows=(r0, r0 + band))
            refs[k].append(ref)
            assert np.array_equal(q.codes[r0:r0 + band].cpu().numpy(), ref["codes"]), (k, r0)
            # scales of the band: the band is one 128-row tile of the tensor-core layout
            got = q.scales.view(-1, nb * 128)[r0 // 128].cpu().numpy()
            assert np.array_equal(got, oracle.swizzle_scales(ref["scales"])), (k, r0)
            assert np.float32(q.s_dec[0].item()) == np.float32(ref["s_dec"]), k
    for out, (ka, kb), bf16 in [(y, ("x", "w"), True), (dx, ("dy", "wt"), True), (dw, ("dyt", "xt"), False)]:
        host = out.float().cpu().numpy()
        for i in range(3):  # first tile, last tile, a random tile
            ra, rb = refs[ka][i], refs[kb][i]
            ms = rng.integers(0, band, samples)
            ns = rng.integers(0, band, samples)
            c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"],
                                   pairs=(ms, ns))
            _check(host[r0s[ka][i] + ms, r0s[kb][i] + ns], c_ref, s, bf16)


@pytest.mark.parametrize("which", [0, 1])
def test_8b_linear_full_size_banded(which):
    _banded_linear(WORKLOADS["8b"], which)


@pytest.mark.parametrize("which", [0, 1])
def test_12b_linear_full_size_banded(which):
    _banded_linear(WORKLOADS["12b"], which)


def test_8b_mxfp4_side_by_side_counters():
    """The 8B workload's activations and gradients through the MXFP4 1x32
    quantizer next to NVFP4: full-tensor event counters equal the oracle's."""
    w = WORKLOADS["8b"]
    inp = linear_inputs(w, 0)
    for key in ("x", "dy"):
        bits = inp[key]
        for cfg in (fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE8M0, block=fb.FP4_BLOCK_1x32),
                    fb.QuantConfig()):
            out = fb.QTensor.empty(bits.shape[0], bits.shape[1], cfg.scale_fmt)
            cnt = torch.zeros(4, dtype=torch.int64, device="cuda")
            fb.fp4_quantize(cfg, to_gpu_bf16(bits), out, counters=cnt,
                            ws=torch.empty(4096, dtype=torch.float32, device="cuda"))
            ref = oracle_quantize(cfg, bits)
            assert cnt.cpu().numpy().tolist() == ref["counters"].tolist(), (key, cfg.scale_fmt)
            assert np.array_equal(out.codes.cpu().numpy(), ref["codes"])


def test_8b_mxfp4_fprop_full_size_sampled():
    """The 8B up-projection (T = 8192, 4096 -> 21504) with X and W through the
    MXFP4 1x32 quantizer on the GPU (bytes equal to the oracle's) and the
    kind::mxf4 GEMM: sampled outputs of Y = X W^T within the bound."""
    w = WORKLOADS["8b"]
    inp = linear_inputs(w, 0)
    cfg = fb.QuantConfig(scale_fmt=MX, block=fb.FP4_BLOCK_1x32)
    ops, refs = [], []
    for key in ("x", "w"):
        bits = inp[key]
        out = fb.QTensor.empty(bits.shape[0], bits.shape[1], MX)
        fb.fp4_quantize(cfg, to_gpu_bf16(bits), out, ws=torch.empty(4096, dtype=torch.float32, device="cuda"))
        ref = oracle_quantize(cfg, bits)
        assert np.array_equal(out.codes.cpu().numpy(), ref["codes"]), key
        assert np.array_equal(out.scales.cpu().numpy(), oracle.swizzle_scales(ref["scales"])), key
        ops.append(out)
        refs.append(ref)
    T, N = inp["x"].shape[0], inp["w"].shape[0]
    y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    fb.fp4_linear_fprop(ops[0], ops[1], y)
    assert fb.fp4_device_status() == 0
    rng = np.random.default_rng(2)
    ms, ns = rng.integers(0, T, 3000), rng.integers(0, N, 3000)
    c_ref, s = oracle.gemm(refs[0]["codes"], refs[0]["scales"], 1.0, refs[1]["codes"], refs[1]["scales"], 1.0,
                           scale_fmt=oracle.FMT_UE8M0, bs=32, pairs=(ms, ns))
    _check(y.float().cpu().numpy()[ms, ns], c_ref, s, bf16=True)


def test_step_from_host_equals_the_device_step():
    """Fp4Linear.step_host (pinned host in, pinned host out, copies on their own
    streams) gives the outputs of Fp4Linear.step on device copies of the inputs,
    also when two layers' calls interleave over several steps."""
    T, K, N = 512, 256, 512
    rng_in = [(random_bf16(60 + 3 * i, (T, K), "student_t4"), random_bf16(61 + 3 * i, (N, K), "weight"),
               random_bf16(62 + 3 * i, (T, N), "log_normal_1e-4_2")) for i in range(2)]
    layers = [fb.Fp4Linear(T, K, N, rht=True, seed=1, layer=i) for i in range(2)]
    host_in = [[torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory() for b in bits] for bits in rng_in]
    host_out = [[torch.empty((T, N), dtype=torch.bfloat16).pin_memory(), torch.empty((T, K), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((N, K), dtype=torch.float32).pin_memory()] for _ in range(2)]
    for _ in range(3):
        for L, hi, ho in zip(layers, host_in, host_out):
            L.step_host(*hi, *ho)
    torch.cuda.synchronize()
    assert fb.fp4_device_status() == 0
    for i, (hi, ho) in enumerate(zip(host_in, host_out)):
        L = fb.Fp4Linear(T, K, N, rht=True, seed=1, layer=i)
        y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        dx = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
        L.step(*(t.cuda() for t in hi), y, dx, dw)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), ho[0]) and torch.equal(dx.cpu(), ho[1]) and torch.equal(dw.cpu(), ho[2])


def test_held_amax_checkpoint_resume_is_byte_identical():
    """UE5M3 held-amax recipe: a run interrupted after step 30, its layer state
    saved, restored into a new layer and continued to step 55 (past the refresh
    at 50) leaves the same bytes and outputs as the uninterrupted run."""
    from workloads import sweep_dy
    T, K, N = 512, 256, 512
    xb, wb = random_bf16(70, (T, K), "student_t4"), random_bf16(71, (N, K), "weight")
    dyb = random_bf16(72, (T, N), "log_normal_1e-4_2")
    x, w = to_gpu_bf16(xb), to_gpu_bf16(wb)
    mk = lambda: fb.Fp4Linear(T, K, N, scale_fmt=UE, rht=False, held=True, target_T=2048.0, seed=5)
    outs = lambda: (torch.empty((T, N), dtype=torch.bfloat16, device="cuda"),
                    torch.empty((T, K), dtype=torch.bfloat16, device="cuda"),
                    torch.empty((N, K), dtype=torch.float32, device="cuda"))
    steps = list(range(0, 56, 5)) + [50, 55]
    steps = sorted(set(steps))
    a, oa = mk(), outs()
    for s in steps:
        a.step(x, w, to_gpu_bf16(sweep_dy(dyb, s, 100)), *oa, step=s)
    b, ob = mk(), outs()
    for s in [t for t in steps if t <= 30]:
        b.step(x, w, to_gpu_bf16(sweep_dy(dyb, s, 100)), *ob, step=s)
    saved = b.state_dict()
    del b
    c, oc = mk(), outs()
    c.load_state_dict(saved)
    for s in [t for t in steps if t > 30]:
        c.step(x, w, to_gpu_bf16(sweep_dy(dyb, s, 100)), *oc, step=s)
    torch.cuda.synchronize()
    assert fb.fp4_device_status() == 0
    for k in a.bufs:
        assert torch.equal(a.bufs[k].codes, c.bufs[k].codes), k
        assert torch.equal(a.bufs[k].scales, c.bufs[k].scales), k
    for u, v in zip(oa, oc):
        assert torch.equal(u, v)
    for sa, sc in zip(a.states, c.states):
        assert torch.equal(sa.buf, sc.buf)


def test_bounded_wait_times_out_and_the_context_stays_usable():
    """A kernel waiting on an mbarrier that nothing completes gives up after the
    limit, records FP4_ERR_DEVICE_TIMEOUT, and later work runs normally."""
    fb.fp4_selftest_wait_timeout(50000)  # 50 ms
    assert fb.fp4_device_status() == fb._lib.FP4_ERR_DEVICE_TIMEOUT
    assert fb.fp4_device_status() == 0   # read and cleared
    ra, a = _operand(73, 128, 256, "normal")
    rb, b = _operand(74, 128, 256, "normal")
    d = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d)
    assert fb.fp4_device_status() == 0
    c_ref, s = oracle.gemm(ra["codes"], ra["scales"], ra["s_dec"], rb["codes"], rb["scales"], rb["s_dec"])
    _check(d.cpu().numpy(), c_ref, s, bf16=False)


@pytest.mark.parametrize("fmt", [fb.FP4_SCALE_E4M3, MX, UE])
def test_gemm_is_deterministic(fmt):
    """Two launches of the same product give the same bits (no atomics, fixed
    accumulation order), for NVFP4, MXFP4 and rebiased UE5M3 alike."""
    M, N, K = 2048, 2176, 1280
    kw = dict(block=fb.FP4_BLOCK_1x32) if fmt == MX else {}
    _, a = _operand(75, M, K, "normal", fmt=fmt, **kw)
    _, b = _operand(76, N, K, "student_t4", fmt=fmt, **kw)
    ws = _ws_for(a, b) if fmt == UE else None
    d1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    d2 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fb.fp4_gemm(a, b, d1, ws=ws)
    fb.fp4_gemm(a, b, d2, ws=ws)
    assert fb.fp4_device_status() == 0
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))
