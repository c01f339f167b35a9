"""GPU parity of the quantizer kernels against the CPU oracle, through the C ABI.

Bit-exact on codes, scale bytes (plain and tensor-core layouts), the FP32
decode tensor scale, the four event counters and the held-amax state. Sizes
span several tiles; plain-layout cases have ragged shapes.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

fb = pytest.importorskip("fp4_block_scaled_02_gb300")
from gpu_common import (assert_quant_equal, gpu_quantize, new_ws, oracle_quantize,  # noqa: E402
                        to_gpu_bf16)
import oracle  # noqa: E402
from workloads import bf16_bits_to_f32, f32_to_bf16_bits, random_bf16  # noqa: E402

TC, PLAIN = fb.FP4_LAYOUT_TCGEN05, fb.FP4_LAYOUT_PLAIN


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    fb._lib.load()


ROWWISE_CASES = [
    # (shape, dist, round, layout, seed, tensor_id, step)
    ((384, 512), "student_t4", fb.FP4_ROUND_RNE, TC, 0, 0, 0),
    ((256, 768), "log_normal_1e-4_2", fb.FP4_ROUND_SR, TC, 5, 3, 17),
    ((128, 64), "normal_outliers", fb.FP4_ROUND_RNE, TC, 0, 0, 0),
    ((37, 80), "normal", fb.FP4_ROUND_RNE, PLAIN, 0, 0, 0),
    ((129, 48), "log_uniform_1e-6_1e-2", fb.FP4_ROUND_SR, PLAIN, 9, 7, 3),
]


@pytest.mark.parametrize("case", ROWWISE_CASES)
def test_rowwise_1x16(case):
    shape, dist, rnd, layout, seed, tid, step = case
    bits = random_bf16(11, shape, dist)
    cfg = fb.QuantConfig(round=rnd, layout=layout, seed=seed, tensor_id=tid, step=step)
    out, _, cnt = gpu_quantize(cfg, bits)
    assert_quant_equal(out, oracle_quantize(cfg, bits), layout, cnt)


COLWISE_CASES = [
    # (input shape (tokens, channels), dist, round, rht, layout, seed)
    ((512, 256), "student_t4", fb.FP4_ROUND_RNE, False, TC, 0),
    ((512, 256), "normal_outliers", fb.FP4_ROUND_RNE, True, TC, 0),
    ((256, 384), "log_normal_1e-4_2", fb.FP4_ROUND_SR, True, TC, 1),
    ((192, 128), "log_uniform_1e-6_1e-2", fb.FP4_ROUND_SR, False, TC, 3),
    ((48, 24), "normal", fb.FP4_ROUND_RNE, True, PLAIN, 0),
    ((80, 40), "log_normal_1e-4_2", fb.FP4_ROUND_SR, True, PLAIN, 2),
]


@pytest.mark.parametrize("case", COLWISE_CASES)
def test_colwise_1x16_with_rht(case):
    shape, dist, rnd, rht, layout, seed = case
    bits = random_bf16(12, shape, dist)
    cfg = fb.QuantConfig(round=rnd, rht=rht, orient=fb.FP4_ORIENT_COLWISE, layout=layout, seed=seed,
                         tensor_id=4, step=2)
    out, _, cnt = gpu_quantize(cfg, bits)
    assert_quant_equal(out, oracle_quantize(cfg, bits), layout, cnt)


# N % 64 == 0 and K % 128 == 0 run the TMA-fed tile kernel, other shapes the
# half-warp-per-block kernel
@pytest.mark.parametrize("shape,layout", [((384, 256), TC), ((256, 512), TC), ((128, 256), PLAIN), ((48, 80), PLAIN),
                                          ((256, 144), PLAIN)])
@pytest.mark.parametrize("orient", [fb.FP4_ORIENT_ROWWISE, fb.FP4_ORIENT_COLWISE])
def test_weights_2d_both_orientations(shape, layout, orient):
    bits = random_bf16(13, shape, "weight")
    cfg = fb.QuantConfig(block=fb.FP4_BLOCK_16x16, layout=layout, emit_transpose=True, orient=orient)
    out, out_t, cnt = gpu_quantize(cfg, bits, with_transpose=True)
    ref = oracle_quantize(cfg, bits)
    ref_t = oracle_quantize(cfg, bits, colwise=orient == fb.FP4_ORIENT_ROWWISE)
    assert_quant_equal(out, ref, layout, cnt)
    assert_quant_equal(out_t, ref_t, layout)
    # quantize(W)^T == quantize(W^T): the two outputs hold the same nibbles
    a = out.codes.cpu().numpy()
    b = out_t.codes.cpu().numpy()
    ua = np.stack([a & 0xF, a >> 4], axis=-1).reshape(a.shape[0], -1)
    ub = np.stack([b & 0xF, b >> 4], axis=-1).reshape(b.shape[0], -1)
    assert np.array_equal(ua.T, ub)


def test_weights_2d_zero_tiny_and_huge_blocks():
    """Whole 16 x 16 blocks of zeros (scale code 0), blocks of tiny values whose
    E4M3 scale underflows, and one huge block saturating the other blocks'
    scales to 448 through a large tensor amax, on the tile kernel's shapes."""
    rng = np.random.default_rng(21)
    x = rng.normal(0.0, 0.02, (256, 512)).astype(np.float32)
    x[0:16, 0:16] = 0.0
    x[16:32, 32:48] = 0.0
    x[32:48, 16:32] *= 1e-30
    x[64:80, 128:144] *= 1e4
    bits = f32_to_bf16_bits(x)
    for layout in (TC, PLAIN):
        cfg = fb.QuantConfig(block=fb.FP4_BLOCK_16x16, layout=layout, emit_transpose=True)
        out, out_t, cnt = gpu_quantize(cfg, bits, with_transpose=True)
        assert_quant_equal(out, oracle_quantize(cfg, bits), layout, cnt)
        assert_quant_equal(out_t, oracle_quantize(cfg, bits, colwise=True), layout)


# 2D scaling of gradients with SR (16x16 blocks on a gradient operand, in both
# orientations): runs on the tile kernel's shapes; every element draws the word
# of its own index in the operand it lands in, so the two outputs round apart
@pytest.mark.parametrize("shape,layout,fmt", [((256, 512), TC, fb.FP4_SCALE_E4M3), ((192, 384), PLAIN, fb.FP4_SCALE_E4M3),
                                              ((128, 256), TC, fb.FP4_SCALE_UE5M3)])
@pytest.mark.parametrize("orient", [fb.FP4_ORIENT_ROWWISE, fb.FP4_ORIENT_COLWISE])
def test_2d_blocks_with_stochastic_rounding(shape, layout, fmt, orient):
    bits = random_bf16(24, shape, "log_normal_1e-4_2")
    cfg = fb.QuantConfig(block=fb.FP4_BLOCK_16x16, scale_fmt=fmt, round=fb.FP4_ROUND_SR, layout=layout,
                         emit_transpose=True, orient=orient, seed=6, tensor_id=9, step=41)
    out, out_t, cnt = gpu_quantize(cfg, bits, with_transpose=True)
    assert_quant_equal(out, oracle_quantize(cfg, bits), layout, cnt)
    assert_quant_equal(out_t, oracle_quantize(cfg, bits, colwise=orient == fb.FP4_ORIENT_ROWWISE), layout)
    # the scales are shared; the codes of the two outputs are independent draws
    a = out.codes.cpu().numpy()
    b = out_t.codes.cpu().numpy()
    ua = np.stack([a & 0xF, a >> 4], axis=-1).reshape(a.shape[0], -1)
    ub = np.stack([b & 0xF, b >> 4], axis=-1).reshape(b.shape[0], -1)
    assert not np.array_equal(ua.T, ub)


def test_2d_stochastic_rounding_needs_whole_tiles():
    """16x16 with SR runs only where the input is whole 64 x 128 tiles."""
    for shape in ((48, 256), (128, 80)):
        x = to_gpu_bf16(random_bf16(25, shape, "normal"))
        out = fb.QTensor.empty(*shape, layout=PLAIN)
        cfg = fb.QuantConfig(block=fb.FP4_BLOCK_16x16, round=fb.FP4_ROUND_SR, layout=PLAIN)
        with pytest.raises(fb.Fp4Error) as e:
            fb.fp4_quantize(cfg, x, out, ws=new_ws())
        assert e.value.status == fb._lib.FP4_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,layout", [((256, 512), TC), ((384, 128), TC), ((10, 64), PLAIN), ((3, 96), PLAIN)])
def test_mxfp4_1x32(shape, layout):
    bits = random_bf16(14, shape, "student_t4")
    cfg = fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE8M0, block=fb.FP4_BLOCK_1x32, layout=layout)
    out, _, cnt = gpu_quantize(cfg, bits)
    ref = oracle_quantize(cfg, bits)
    assert_quant_equal(out, ref, layout, cnt)
    assert int(cnt[0]) == 0


def test_ue5m3_current_and_held_amax():
    base = random_bf16(15, (256, 512), "log_normal_1e-4_2")
    state = fb.AmaxState()
    ostate = oracle.HeldState()
    for step, factor in [(0, 1.0), (1, 30.0), (49, 1e-3), (50, 1e3), (51, 1.0)]:
        bits = f32_to_bf16_bits(bf16_bits_to_f32(base) * np.float32(factor))
        cfg = fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE5M3, tscale=fb.FP4_TSCALE_HELD, target_T=2048.0,
                             round=fb.FP4_ROUND_SR, step=step, seed=4, tensor_id=3)
        out, _, cnt = gpu_quantize(cfg, bits, state=state)
        ref = oracle_quantize(cfg, bits, state=ostate)
        assert_quant_equal(out, ref, TC, cnt)
        assert state.valid == 1 and state.last_refresh_step == int(ostate.last[0])
        assert np.float32(state.amax) == ostate.amax[0]
    cfg = fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE5M3, target_T=448.0)
    out, _, cnt = gpu_quantize(cfg, base)
    assert_quant_equal(out, oracle_quantize(cfg, base), TC, cnt)


def test_held_state_not_valid_refreshes_on_a_non_refresh_step():
    # the held amax refreshes on step % 50 == 0 and also whenever the state is
    # not valid yet; afterwards non-refresh steps hold it
    assert fb.fp4_device_status() == 0
    bits = random_bf16(16, (128, 64), "normal")
    state, ostate = fb.AmaxState(), oracle.HeldState()
    for step, factor in [(7, 1.0), (8, 100.0)]:
        x = f32_to_bf16_bits(bf16_bits_to_f32(bits) * np.float32(factor))
        cfg = fb.QuantConfig(scale_fmt=fb.FP4_SCALE_UE5M3, tscale=fb.FP4_TSCALE_HELD, target_T=2048.0, step=step)
        out, _, cnt = gpu_quantize(cfg, x, state=state)
        ref = oracle_quantize(cfg, x, state=ostate)
        assert_quant_equal(out, ref, TC, cnt)
        assert state.valid == 1 and state.last_refresh_step == 7 == int(ostate.last[0])
    assert fb.fp4_device_status() == 0


def test_current_scaling_nvfp4_large_values_and_zero_tensor():
    bits = np.zeros((128, 64), dtype=np.uint16)
    cfg = fb.QuantConfig()
    out, _, cnt = gpu_quantize(cfg, bits)
    assert_quant_equal(out, oracle_quantize(cfg, bits), TC, cnt)
    big = random_bf16(17, (128, 128), "normal")
    big = f32_to_bf16_bits(bf16_bits_to_f32(big) * np.float32(1e30))
    out, _, cnt = gpu_quantize(cfg, big)
    assert_quant_equal(out, oracle_quantize(cfg, big), TC, cnt)


def test_empty_input_is_a_no_op():
    cfg = fb.QuantConfig(layout=PLAIN)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    out = fb.QTensor.empty(0, 64, layout=PLAIN)
    fb.fp4_quantize(cfg, x, out, ws=new_ws())
    torch.cuda.synchronize()


@pytest.mark.parametrize("fmt,block,shape", [(fb.FP4_SCALE_E4M3, fb.FP4_BLOCK_1x16, (256, 256)),
                                             (fb.FP4_SCALE_UE5M3, fb.FP4_BLOCK_1x16, (128, 512)),
                                             (fb.FP4_SCALE_UE8M0, fb.FP4_BLOCK_1x32, (128, 256))])
@pytest.mark.parametrize("layout", [TC, PLAIN])
def test_dequantize(fmt, block, shape, layout):
    bits = random_bf16(18, shape, "student_t4")
    cfg = fb.QuantConfig(scale_fmt=fmt, block=block, layout=layout)
    out, _, _ = gpu_quantize(cfg, bits)
    ref = oracle_quantize(cfg, bits)
    bs = 32 if fmt == fb.FP4_SCALE_UE8M0 else 16
    want = oracle.dequantize(ref["codes"], ref["scales"], ref["s_dec"], {0: 0, 1: 1, 2: 2}[fmt], bs)
    y32 = torch.empty(shape, dtype=torch.float32, device="cuda")
    fb.fp4_dequantize(out, y32)
    y16 = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    fb.fp4_dequantize(out, y16)
    torch.cuda.synchronize()
    assert np.array_equal(y32.cpu().numpy().view(np.uint32), want.view(np.uint32))
    assert torch.equal(y16.cpu(), torch.from_numpy(want).to(torch.bfloat16))


def test_quantize_is_deterministic():
    bits = random_bf16(19, (256, 512), "log_normal_1e-4_2")
    cfg = fb.QuantConfig(round=fb.FP4_ROUND_SR, rht=True, orient=fb.FP4_ORIENT_COLWISE, seed=3)
    a, _, ca = gpu_quantize(cfg, bits)
    b, _, cb = gpu_quantize(cfg, bits)
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales) and torch.equal(ca, cb)


def test_validation_errors_launch_nothing():
    x = to_gpu_bf16(random_bf16(20, (128, 64), "normal"))
    out = fb.QTensor.empty(128, 64)
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_quantize(fb.QuantConfig(), x, out, ws=None)            # current scaling needs workspace
    assert e.value.status == fb._lib.FP4_ERR_WORKSPACE
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_quantize(fb.QuantConfig(rht=True), x, out, ws=new_ws())  # RHT needs colwise
    assert e.value.status == fb._lib.FP4_ERR_INVALID_ARG
    bad = fb.QTensor.empty(128, 48)
    with pytest.raises(fb.Fp4Error) as e:
        fb.fp4_quantize(fb.QuantConfig(), to_gpu_bf16(random_bf16(21, (128, 48), "normal")), bad, ws=new_ws())
    assert e.value.status == fb._lib.FP4_ERR_SHAPE                      # 48/16 = 3 blocks: not a multiple of 4


def test_e2m1_conversion_exhaustive_over_bf16_magnitudes():
    """Every BF16 value in [-6, 6] (both zeros and every tie point included)
    reaches the E2M1 conversion unscaled: one block holds 2688 = 6 * 448, so
    s_enc,G = 1, and every other block's first element is 6, so its E4M3
    scale is exactly 1 and v = x. Codes must equal the oracle's."""
    pos = np.arange(0, 0x40C1, dtype=np.uint16)                  # +0 .. +6.0
    vals = np.concatenate([pos, pos | 0x8000])                   # and their negatives (incl. -0)
    per_block = 15
    nblk = -(-vals.size // per_block)
    body = np.zeros(nblk * per_block, dtype=np.uint16)
    body[:vals.size] = vals
    blocks = body.reshape(nblk, per_block)
    six = np.full((nblk, 1), 0x40C0, dtype=np.uint16)            # 6.0
    bits = np.concatenate([six, blocks], axis=1)
    head = np.zeros((1, 16), dtype=np.uint16)
    head[0, 0] = f32_to_bf16_bits(np.array([2688.0], np.float32))[0]
    bits = np.ascontiguousarray(np.concatenate([head, bits], axis=0))
    # RNE once; SR with four different draws per value (steps 0..3)
    for rnd, step in [(fb.FP4_ROUND_RNE, 0)] + [(fb.FP4_ROUND_SR, k) for k in range(4)]:
        cfg = fb.QuantConfig(layout=PLAIN, round=rnd, seed=5, tensor_id=2, step=step)
        out, _, cnt = gpu_quantize(cfg, bits)
        ref = oracle_quantize(cfg, bits)
        assert ref["s_dec"] == 1.0
        assert_quant_equal(out, ref, PLAIN, cnt)


def test_e4m3_block_scale_ties_and_neighbours():
    """Block amaxes 6 * m for every midpoint m between neighbouring E4M3 values
    up to 448 (subnormals included) and the BF16 neighbours of 6 * m, with
    s_enc,G = 1 (one block holds 2688 = 6 * 448): s = RN(amax / 6) = m exactly,
    so every tie of the block-scale encode (App. B.2, RNE) is exercised, in
    both the rowwise and the colwise kernels."""
    e4 = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mids = (e4[:-1] + e4[1:]) / 2
    amax = f32_to_bf16_bits((6.0 * mids).astype(np.float32))
    assert np.array_equal(bf16_bits_to_f32(amax).astype(np.float64), 6.0 * mids)   # exact in BF16
    amax = np.concatenate([amax, amax + 1, amax - 1])
    amax = amax[(amax > 0) & (bf16_bits_to_f32(amax) <= 2688.0)]
    rng = np.random.default_rng(4)
    rows = np.zeros((amax.size + 1, 16), dtype=np.float32)
    rows[0, 0] = 2688.0
    a = bf16_bits_to_f32(amax)
    rows[1:, 0] = a
    rows[1:, 1:] = a[:, None] * rng.uniform(-1.0, 1.0, (amax.size, 15))
    nrow = -(-rows.shape[0] // 16) * 16                            # whole 16-row tiles for the colwise case
    rows = np.concatenate([rows, np.zeros((nrow - rows.shape[0], 16), np.float32)])
    bits = f32_to_bf16_bits(rows)
    for orient in (fb.FP4_ORIENT_ROWWISE, fb.FP4_ORIENT_COLWISE):
        src = bits if orient == fb.FP4_ORIENT_ROWWISE else np.ascontiguousarray(bits.T)
        cfg = fb.QuantConfig(layout=PLAIN, orient=orient)
        out, _, cnt = gpu_quantize(cfg, src)
        ref = oracle_quantize(cfg, src)
        assert ref["s_dec"] == 1.0
        assert_quant_equal(out, ref, PLAIN, cnt)


DUAL_CASES = [
    # (input shape, dist, scale fmt, round, rht, held, target_T)
    ((256, 384), "student_t4", fb.FP4_SCALE_E4M3, fb.FP4_ROUND_RNE, True, False, 448.0),
    ((384, 256), "log_normal_1e-4_2", fb.FP4_SCALE_E4M3, fb.FP4_ROUND_SR, True, False, 448.0),
    ((256, 256), "normal_outliers", fb.FP4_SCALE_E4M3, fb.FP4_ROUND_RNE, False, False, 448.0),
    ((512, 640), "log_normal_1e-4_2", fb.FP4_SCALE_UE5M3, fb.FP4_ROUND_SR, False, True, 2048.0),
]


@pytest.mark.parametrize("case", DUAL_CASES)
def test_dual_quantize_equals_two_separate_calls_and_oracle(case):
    shape, dist, fmt, rnd, rht, held, T = case
    base = random_bf16(22, shape, dist)
    tsc = fb.FP4_TSCALE_HELD if held else fb.FP4_TSCALE_CURRENT
    states = [fb.AmaxState() for _ in range(4)]
    ostates = [oracle.HeldState(), oracle.HeldState()]
    for step, factor in ([(0, 1.0), (1, 50.0), (50, 0.02)] if held else [(3, 1.0)]):
        bits = f32_to_bf16_bits(bf16_bits_to_f32(base) * np.float32(factor))
        x = to_gpu_bf16(bits)
        cr = fb.QuantConfig(scale_fmt=fmt, round=rnd, tscale=tsc, target_T=T, seed=7, tensor_id=3, step=step)
        cc = fb.QuantConfig(scale_fmt=fmt, round=rnd, tscale=tsc, target_T=T, seed=7, tensor_id=4, step=step,
                            orient=fb.FP4_ORIENT_COLWISE, rht=rht)
        R, C = shape
        dr, dc = fb.QTensor.empty(R, C, fmt), fb.QTensor.empty(C, R, fmt)
        sr_, sc_ = fb.QTensor.empty(R, C, fmt), fb.QTensor.empty(C, R, fmt)
        cnt = torch.zeros((4, 4), dtype=torch.int64, device="cuda")
        ws = torch.zeros(8192, dtype=torch.float32, device="cuda")
        fb.fp4_quantize_dual(cr, cc, x, dr, dc, states[0], states[1], cnt[0], cnt[1], ws=ws)
        fb.fp4_quantize(cr, x, sr_, state=states[2], counters=cnt[2], ws=new_ws())
        fb.fp4_quantize(cc, x, sc_, state=states[3], counters=cnt[3], ws=new_ws())
        assert fb.fp4_device_status() == 0
        for a, b in ((dr, sr_), (dc, sc_)):
            assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
            assert a.s_dec[0:1].view(torch.int32).item() == b.s_dec[0:1].view(torch.int32).item()
        assert torch.equal(cnt[0], cnt[2]) and torch.equal(cnt[1], cnt[3])
        assert torch.equal(states[0].buf, states[2].buf) and torch.equal(states[1].buf, states[3].buf)
        assert_quant_equal(dr, oracle_quantize(cr, bits, state=ostates[0] if held else None), TC, cnt[0])
        assert_quant_equal(dc, oracle_quantize(cc, bits, state=ostates[1] if held else None), TC, cnt[1])


# Tensor amax ahead of quantization (fp4_tensor_amax) and the given-amax mode:
# the amax equals the oracle's tensor amax of the same operand, and quantizing
# with it reproduces current scaling byte for byte. Tile shapes (T % 64,
# C % 128) take the 128-thread tile pass, the others the quantizer's own kernels.
AMAX_SHAPES = [(256, 512), (192, 384), (48, 80), (128, 208)]


@pytest.mark.parametrize("shape", AMAX_SHAPES)
def test_tensor_amax_matches_the_oracle(shape):
    bits = random_bf16(26, shape, "log_normal_1e-4_2")
    x = to_gpu_bf16(bits)
    ws = torch.zeros(fb.AMAX_WS_BYTES // 4, dtype=torch.float32, device="cuda")
    R, C = shape
    cases = [(fb.QuantConfig(step=5), False, False)]
    if R % 16 == 0 and C % 8 == 0:
        cases += [(fb.QuantConfig(orient=fb.FP4_ORIENT_COLWISE, rht=True, seed=3, step=5), True, True),
                  (fb.QuantConfig(orient=fb.FP4_ORIENT_COLWISE, step=5), True, False)]
    if R % 16 == 0 and C % 16 == 0:
        cases += [(fb.QuantConfig(block=fb.FP4_BLOCK_16x16, step=5), False, False)]
    for cfg, colwise, rht in cases:
        st = fb.AmaxState()
        fb.fp4_tensor_amax(cfg, x, st, ws)
        assert fb.fp4_device_status() == 0
        ref = oracle.tensor_amax(bits, colwise=colwise, rht=rht, seed=cfg.seed)
        assert np.float32(st.amax) == np.float32(ref), (cfg, st.amax, ref)
        assert st.valid == 1 and st.last_refresh_step == 5
    if R % 16 == 0 and C % 16 == 0:
        sr_, sc_ = fb.AmaxState(), fb.AmaxState()
        fb.fp4_tensor_amax_dual(fb.QuantConfig(step=2), fb.QuantConfig(orient=fb.FP4_ORIENT_COLWISE, rht=True,
                                                                       seed=3, step=2), x, sr_, sc_, ws)
        assert fb.fp4_device_status() == 0
        assert np.float32(sr_.amax) == np.float32(oracle.tensor_amax(bits))
        assert np.float32(sc_.amax) == np.float32(oracle.tensor_amax(bits, colwise=True, rht=True, seed=3))


GIVEN_CASES = [
    # (shape, fmt, round, target_T)
    ((256, 512), fb.FP4_SCALE_E4M3, fb.FP4_ROUND_SR, 448.0),
    ((384, 256), fb.FP4_SCALE_UE5M3, fb.FP4_ROUND_RNE, 2048.0),
]


@pytest.mark.parametrize("case", GIVEN_CASES)
def test_given_amax_equals_current_scaling(case):
    shape, fmt, rnd, T = case
    bits = random_bf16(27, shape, "student_t4")
    x = to_gpu_bf16(bits)
    R, C = shape
    ws = torch.zeros(fb.AMAX_WS_BYTES // 4, dtype=torch.float32, device="cuda")
    kw = dict(scale_fmt=fmt, round=rnd, target_T=T, seed=4, step=9)
    cr = fb.QuantConfig(tensor_id=3, **kw)
    cc = fb.QuantConfig(tensor_id=4, orient=fb.FP4_ORIENT_COLWISE, rht=True, **kw)
    cw = fb.QuantConfig(tensor_id=2, block=fb.FP4_BLOCK_16x16, emit_transpose=True, scale_fmt=fmt, target_T=T)
    giv = dict(tscale=fb.FP4_TSCALE_GIVEN)
    # dual: current vs given
    a_r, a_c, g_r, g_c = (fb.QTensor.empty(R, C, fmt), fb.QTensor.empty(C, R, fmt),
                          fb.QTensor.empty(R, C, fmt), fb.QTensor.empty(C, R, fmt))
    cnt = torch.zeros((4, 4), dtype=torch.int64, device="cuda")
    fb.fp4_quantize_dual(cr, cc, x, a_r, a_c, None, None, cnt[0], cnt[1], ws=torch.zeros(8192, device="cuda"))
    st_r, st_c = fb.AmaxState(), fb.AmaxState()
    fb.fp4_tensor_amax_dual(cr, cc, x, st_r, st_c, ws)
    fb.fp4_quantize_dual(fb.QuantConfig(tensor_id=3, **kw, **giv),
                         fb.QuantConfig(tensor_id=4, orient=fb.FP4_ORIENT_COLWISE, rht=True, **kw, **giv),
                         x, g_r, g_c, st_r, st_c, cnt[2], cnt[3])
    assert fb.fp4_device_status() == 0
    for a, g in ((a_r, g_r), (a_c, g_c)):
        assert torch.equal(a.codes, g.codes) and torch.equal(a.scales, g.scales)
        assert a.s_dec[0:1].view(torch.int32).item() == g.s_dec[0:1].view(torch.int32).item()
    assert torch.equal(cnt[0], cnt[2]) and torch.equal(cnt[1], cnt[3])
    assert st_r.valid == 1 and st_c.valid == 1  # read, not changed
    # 16x16 with both outputs: current vs given
    w1, w1t, w2, w2t = (fb.QTensor.empty(R, C, fmt), fb.QTensor.empty(C, R, fmt),
                        fb.QTensor.empty(R, C, fmt), fb.QTensor.empty(C, R, fmt))
    fb.fp4_quantize(cw, x, w1, w1t, ws=new_ws())
    st_w = fb.AmaxState()
    fb.fp4_tensor_amax(cw, x, st_w, ws)
    cwg = fb.QuantConfig(tensor_id=2, block=fb.FP4_BLOCK_16x16, emit_transpose=True, scale_fmt=fmt, target_T=T, **giv)
    fb.fp4_quantize(cwg, x, w2, w2t, state=st_w)
    assert fb.fp4_device_status() == 0
    for a, g in ((w1, w2), (w1t, w2t)):
        assert torch.equal(a.codes, g.codes) and torch.equal(a.scales, g.scales)
    assert_quant_equal(g_r, oracle_quantize(cr, bits), TC, cnt[2])


def test_given_amax_not_valid_leaves_a_state_error():
    x = to_gpu_bf16(random_bf16(28, (256, 256), "normal"))
    out = fb.QTensor.empty(256, 256)
    out.codes.fill_(0xAA)
    st = fb.AmaxState()  # zeroed: not valid
    fb.fp4_quantize(fb.QuantConfig(tscale=fb.FP4_TSCALE_GIVEN), x, out, state=st)
    assert fb.fp4_device_status() == fb._lib.FP4_ERR_STATE
    assert int((out.codes != 0xAA).sum().item()) == 0  # nothing written
    assert fb.fp4_device_status() == 0  # the status word was cleared by the read


def test_linear_with_amax_on_a_side_stream_equals_the_plain_schedule():
    """Fp4Linear computing W's and dY's amaxes on a second stream (given-amax
    quantization) leaves the same quantized operands, counters and outputs."""
    T, K, N = 512, 256, 512
    xb = random_bf16(29, (T, K), "student_t4")
    wb = random_bf16(30, (N, K), "weight")
    dyb = random_bf16(31, (T, N), "log_normal_1e-4_2")
    x, w, dy = to_gpu_bf16(xb), to_gpu_bf16(wb), to_gpu_bf16(dyb)
    outs = []
    for overlap in (False, True):
        L = fb.Fp4Linear(T, K, N, rht=True, seed=2, overlap_amax=overlap)
        assert (L.side is not None) == overlap
        y = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        dx = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
        for step in (0, 1):
            L.counters.zero_()
            L.step(x, w, dy, y, dx, dw, step=step)
        torch.cuda.synchronize()
        assert fb.fp4_device_status() == 0
        outs.append((L, y, dx, dw))
    (a, ya, dxa, dwa), (b, yb, dxb, dwb) = outs
    for k in a.bufs:
        assert torch.equal(a.bufs[k].codes, b.bufs[k].codes), k
        assert torch.equal(a.bufs[k].scales, b.bufs[k].scales), k
        assert torch.equal(a.bufs[k].s_dec[:1], b.bufs[k].s_dec[:1]), k  # element 0 is the tensor scale
    assert torch.equal(a.counters, b.counters)
    assert torch.equal(ya, yb) and torch.equal(dxa, dxb) and torch.equal(dwa, dwb)


# Strided inputs: the operand is a column slice of a wider BF16 buffer (rows ld
# elements apart), quantized in place. Each case must give exactly the bytes,
# tensor scale and counters the oracle gives for the dense copy of the slice.
STRIDED_CASES = [
    # (name, rows, cols, col offset, buffer width, config)
    ("rowwise_sr_tc", 256, 384, 64, 640, dict(round=fb.FP4_ROUND_SR, seed=3, tensor_id=3, step=7)),
    ("rowwise_rne_plain", 40, 96, 8, 200, dict(layout=PLAIN)),
    ("colwise_rht_sr", 256, 128, 128, 520, dict(orient=fb.FP4_ORIENT_COLWISE, rht=True, round=fb.FP4_ROUND_SR,
                                                seed=1, tensor_id=4)),
    ("2d_tma_tiles", 256, 256, 16, 1000, dict(block=fb.FP4_BLOCK_16x16)),
    ("2d_plain_kernel", 48, 80, 24, 136, dict(block=fb.FP4_BLOCK_16x16, layout=PLAIN)),
    ("mxfp4", 128, 256, 32, 512, dict(scale_fmt=fb.FP4_SCALE_UE8M0, block=fb.FP4_BLOCK_1x32)),
    ("ue5m3_held", 128, 512, 256, 1024, dict(scale_fmt=fb.FP4_SCALE_UE5M3, tscale=fb.FP4_TSCALE_HELD,
                                             target_T=2048.0, round=fb.FP4_ROUND_SR, tensor_id=3)),
]


@pytest.mark.parametrize("case", STRIDED_CASES, ids=[c[0] for c in STRIDED_CASES])
def test_strided_column_slice_matches_the_dense_copy(case):
    name, R, C, c0, width, kw = case
    buf = random_bf16(500 + len(name), (R, width), "student_t4")
    dense = np.ascontiguousarray(buf[:, c0:c0 + C])
    x = to_gpu_bf16(buf)[:, c0:c0 + C]
    assert x.stride(0) == width and not x.is_contiguous()
    cfg = fb.QuantConfig(**kw)
    colwise = cfg.orient == fb.FP4_ORIENT_COLWISE
    OR, OC = (C, R) if colwise else (R, C)
    out = fb.QTensor.empty(OR, OC, cfg.scale_fmt, cfg.layout)
    state = fb.AmaxState() if cfg.tscale == fb.FP4_TSCALE_HELD else None
    ref_state = oracle.HeldState() if state is not None else None
    counters = torch.zeros(4, dtype=torch.int64, device="cuda")
    fb.fp4_quantize(cfg, x, out, state=state, counters=counters, ws=new_ws())
    assert fb.fp4_device_status() == 0
    ref = oracle_quantize(cfg, dense, state=ref_state)
    assert_quant_equal(out, ref, cfg.layout, counters=counters, check_sdec=cfg.scale_fmt != fb.FP4_SCALE_UE8M0)


def test_strided_dual_and_tensor_amax_match_the_dense_copy():
    """The one-read rowwise + colwise call, its tensor amax ahead (TMA tile pass)
    and the given-amax conversion, on a column slice: the same bytes as the
    dense copy through the oracle."""
    T, C, c0, width = 256, 384, 128, 768
    buf = random_bf16(520, (T, width), "log_normal_1e-4_2")
    dense = np.ascontiguousarray(buf[:, c0:c0 + C])
    x = to_gpu_bf16(buf)[:, c0:c0 + C]
    cr = fb.QuantConfig(round=fb.FP4_ROUND_SR, seed=2, tensor_id=3)
    cc = fb.QuantConfig(round=fb.FP4_ROUND_SR, orient=fb.FP4_ORIENT_COLWISE, rht=True, seed=2, tensor_id=4)
    ref_r, ref_c = oracle_quantize(cr, dense), oracle_quantize(cc, dense)
    o_r, o_c = fb.QTensor.empty(T, C), fb.QTensor.empty(C, T)
    k_r, k_c = torch.zeros(4, dtype=torch.int64, device="cuda"), torch.zeros(4, dtype=torch.int64, device="cuda")
    fb.fp4_quantize_dual(cr, cc, x, o_r, o_c, counters_row=k_r, counters_col=k_c,
                         ws=torch.zeros(fb.AMAX_WS_BYTES // 4, dtype=torch.float32, device="cuda"))
    assert fb.fp4_device_status() == 0
    assert_quant_equal(o_r, ref_r, TC, counters=k_r)
    assert_quant_equal(o_c, ref_c, TC, counters=k_c)
    s_r, s_c = fb.AmaxState(), fb.AmaxState()
    fb.fp4_tensor_amax_dual(cr, cc, x, s_r, s_c, torch.zeros(fb.AMAX_WS_BYTES // 4, dtype=torch.float32,
                                                               device="cuda"))
    assert np.float32(s_r.amax) == np.float32(ref_r["amax"]) and np.float32(s_c.amax) == np.float32(ref_c["amax"])
    g_r, g_c = fb.QTensor.empty(T, C), fb.QTensor.empty(C, T)
    giv = dict(tscale=fb.FP4_TSCALE_GIVEN)
    fb.fp4_quantize_dual(fb.QuantConfig(round=fb.FP4_ROUND_SR, seed=2, tensor_id=3, **giv),
                         fb.QuantConfig(round=fb.FP4_ROUND_SR, orient=fb.FP4_ORIENT_COLWISE, rht=True, seed=2,
                                        tensor_id=4, **giv), x, g_r, g_c, s_r, s_c)
    assert fb.fp4_device_status() == 0
    assert_quant_equal(g_r, ref_r, TC)
    assert_quant_equal(g_c, ref_c, TC)


def test_device_status_record_is_stream_ordered():
    """fp4_device_status_record writes the status word in stream order without
    synchronising: a bounded wait that times out (the self-test) shows up in the
    record that follows it, and the record after that reads 0 again."""
    rec = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    fb.fp4_device_status_record(rec[0:1])
    fb.fp4_selftest_wait_timeout(2000)
    fb.fp4_device_status_record(rec[1:2])
    torch.cuda.synchronize()
    assert rec.cpu().tolist() == [fb._lib.FP4_OK, fb._lib.FP4_ERR_DEVICE_TIMEOUT]
    assert fb.fp4_device_status() == 0  # the record cleared the word


def test_div6_is_correctly_rounded_over_whole_binades():
    """The quantizer's RN(amax_B / 6) (App. B.2's decode-scale step, one multiply
    and two fused multiply-adds) equals the correctly rounded binary32 quotient
    (numpy's IEEE division) for every float of the binades [1, 2), [2^-120,
    2^-119) (the lowest it takes) and [2^127, 2^128) (the highest), of the
    binade [2^-122, 2^-121) and of a sample of subnormals, where the IEEE
    division takes over, and at 0, FLT_MAX and infinity."""
    import ctypes
    L = fb._lib.load()
    mant = np.arange(1 << 23, dtype=np.uint32)
    parts = [((e + 127) << 23) | mant for e in (0, -120, 127, -122)]
    parts.append(np.random.default_rng(0).integers(1, 1 << 23, 1 << 16, dtype=np.uint32))  # subnormals
    parts.append(np.array([0, 0x7F7FFFFF, 0x7F800000], dtype=np.uint32))
    bits = np.concatenate(parts)
    a = bits.view(np.float32)
    want = (a / np.float32(6.0)).astype(np.float32)
    x = torch.from_numpy(a.copy()).cuda()
    y = torch.empty_like(x)
    st = L.fp4_selftest_div6(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.numel(),
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    fb._lib.check(st, "fp4_selftest_div6")
    got = y.cpu().numpy()
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, f"{bad.size} mismatches, first inputs {a[bad[:4]].tolist()}"
