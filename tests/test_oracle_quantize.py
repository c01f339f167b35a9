"""Pins for the oracle's quantizer ("Pretraining Large Language Models with NVFP4",
App. B.1-B.3, sections 4.3-4.4; the UE5M3 page's periodic tensor scaling).

Checks use closed forms the pages state (the tensor amax maps to the scale
target; every block amax maps to +-6 up to scale rounding), the transpose
invariance of 2D weight scaling, SR unbiasedness over 10^6 draws, and counts
recomputed here in float64 from the inputs.
"""
import numpy as np
import pytest
import torch

from workloads import bf16_bits_to_f32, f32_to_bf16_bits, random_bf16


def unpack(codes):
    lo = codes & 0xF
    hi = codes >> 4
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def code_values(codes):
    u = unpack(codes)
    return np.where(u & 8, -1.0, 1.0) * E2M1[u & 7]


def e4m3_decode(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


def ue5m3_decode(b):
    b = b.astype(np.int64)
    e, m = b >> 3, b & 7
    return np.where(e == 0, m / 8 * 2.0 ** -14, (1 + m / 8) * 2.0 ** (e - 15))


def test_tensor_amax_block_gets_scale_target(orc):
    # B.1/B.2: s_enc,G maps max_B s_dec,L,B = amax_X / 6 onto 448, so the block
    # holding amax_X gets the largest E4M3 scale, 448 (code 0x7E)
    for seed in range(5):
        x = random_bf16(seed, (64, 256), "student_t4")
        q = orc.quantize(x)
        xf = np.abs(bf16_bits_to_f32(x)).reshape(64, 16, 16).max(axis=2)
        r, b = np.unravel_index(np.argmax(xf), xf.shape)
        assert q["scales"][r, b] == 0x7E
        assert q["amax"] == np.abs(bf16_bits_to_f32(x)).max()
        assert q["s_dec"] == np.float32(1.0) / np.float32(np.float32(2688.0) / np.float32(q["amax"]))


@pytest.mark.parametrize("T", [448.0, 2048.0])
def test_held_amax_block_gets_target_T(orc, T):
    x = random_bf16(9, (32, 128), "student_t4")
    q = orc.quantize(x, scale_fmt=orc.FMT_UE5M3, held=True, target_T=T, step=0)
    xf = np.abs(bf16_bits_to_f32(x)).reshape(32, 8, 16).max(axis=2)
    r, b = np.unravel_index(np.argmax(xf), xf.shape)
    assert ue5m3_decode(q["scales"][r:r + 1, b])[0] == T


def test_block_amax_maps_to_six(orc):
    # A3 / B.2: each block's amax is scaled onto the FP4 maximum 6; with a 3-bit
    # scale mantissa the scaled amax lies within 6 (1 +- 2^-4)
    x = random_bf16(3, (128, 512), "student_t4")
    q = orc.quantize(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    amax_b = np.abs(xf).reshape(128, 32, 16).max(axis=2)
    s_hat = e4m3_decode(q["scales"])
    normal = s_hat >= 2.0 ** -6
    scaled = amax_b / (s_hat * q["s_dec"])
    assert normal.sum() > 1000
    assert np.all(np.abs(scaled[normal] - 6.0) <= 6.0 * 2.0 ** -4 * (1 + 1e-6))


def _check_rne_codes(q, xf, bs, s_hat):
    """Each code is the E2M1 value nearest x * s_enc,L (ties excepted)."""
    v = xf / np.repeat(s_hat * q["s_dec"], bs, axis=1)
    got = code_values(q["codes"])
    a = np.minimum(np.abs(v), 6.0)
    dist = np.abs(a[..., None] - E2M1[None, None, :])
    best = E2M1[np.argmin(dist, axis=-1)]
    second = np.sort(dist, axis=-1)
    near_tie = (second[..., 1] - second[..., 0]) <= 1e-5 * np.maximum(a, 1e-30)
    ok = (np.abs(got) == best) | near_tie
    return ok


def test_rne_codes_are_nearest_values(orc):
    x = random_bf16(4, (64, 256), "normal_outliers")
    q = orc.quantize(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    s_hat = e4m3_decode(q["scales"])
    ok = _check_rne_codes(q, xf, 16, s_hat)
    assert ok.all()
    sign_ok = (np.signbit(xf) == (unpack(q["codes"]) >= 8))
    assert sign_ok.all()


def test_two_d_scaling_is_transpose_invariant(orc):
    # 4.3: 16x16 weight blocks give one quantized representation for W and W^T
    w = random_bf16(5, (64, 128), "weight")
    wt = np.ascontiguousarray(w.T)
    qa = orc.quantize(w, block=orc.BLOCK_16x16)
    qb = orc.quantize(wt, block=orc.BLOCK_16x16)
    assert np.array_equal(unpack(qa["codes"]).T, unpack(qb["codes"]))
    ta = qa["scales"][::16, :]           # one scale per 16x16 tile
    tb = qb["scales"][::16, :]
    assert np.array_equal(ta.T, tb)
    # every row of a tile carries the tile's scale
    assert np.array_equal(qa["scales"], np.repeat(ta, 16, axis=0))
    # colwise quantization of W is quantization of the materialised W^T
    qc = orc.quantize(w, block=orc.BLOCK_16x16, colwise=True)
    assert np.array_equal(qc["codes"], qb["codes"]) and np.array_equal(qc["scales"], qb["scales"])
    assert qa["s_dec"] == qb["s_dec"]


def test_colwise_is_quantization_of_transpose(orc):
    x = random_bf16(6, (64, 96), "student_t4")
    qa = orc.quantize(x, colwise=True, sr=True, seed=3, tensor_id=4, step=2)
    qb = orc.quantize(np.ascontiguousarray(x.T), sr=True, seed=3, tensor_id=4, step=2)
    for k in ("codes", "scales"):
        assert np.array_equal(qa[k], qb[k])


def test_rht_quantize_uses_rotated_values(orc):
    x = random_bf16(7, (64, 32), "normal_outliers")
    q = orc.quantize(x, colwise=True, rht=True, seed=1)
    xt = bf16_bits_to_f32(np.ascontiguousarray(x.T))
    rot = np.stack([np.concatenate([orc.rht16(row[i:i + 16], 1) for i in range(0, 64, 16)])
                    for row in xt])
    assert q["amax"] == np.abs(rot).max()
    deq = orc.dequantize(q["codes"], q["scales"], q["s_dec"])
    # dequantized values approximate the rotated operand, not the raw one
    err_rot = np.abs(deq - rot).mean()
    err_raw = np.abs(deq - xt).mean()
    assert err_rot < 0.25 * err_raw


def test_counters_recount(orc):
    # elem_underflow and scale_underflow recounted exactly; elem_sat and scale_sat
    # bracketed by float64 recounts with a small margin around the thresholds
    x = random_bf16(8, (128, 256), "log_normal_1e-4_2")
    xs = f32_to_bf16_bits(bf16_bits_to_f32(x) * np.float32(1e3))
    for held, T, scale_dec in [(False, 448.0, e4m3_decode), (True, 2048.0, ue5m3_decode)]:
        fmt = orc.FMT_UE5M3 if held else orc.FMT_E4M3
        st = orc.HeldState()
        orc.quantize(x, scale_fmt=fmt, held=held, target_T=T, state=st, step=0)
        q = orc.quantize(xs, scale_fmt=fmt, held=held, target_T=T, state=st, step=1 if held else 0)
        xf = bf16_bits_to_f32(xs).astype(np.float64)
        c = q["counters"].astype(np.int64)
        mags = unpack(q["codes"]) & 7
        assert c[1] == np.sum((xf != 0) & (mags == 0))
        amax_b = np.abs(xf).reshape(128, 16, 16).max(axis=2)
        assert c[3] == np.sum((amax_b > 0) & (q["scales"] == 0))
        s_enc = 1.0 / q["s_dec"]
        s = amax_b / 6.0 * s_enc
        smax = 448.0 if not held else 114688.0
        assert np.sum(s > smax * (1 + 1e-6)) <= c[2] <= np.sum(s > smax * (1 - 1e-6))
        s_hat = scale_dec(q["scales"])
        with np.errstate(divide="ignore", invalid="ignore"):
            v = np.abs(xf) / np.repeat(s_hat * q["s_dec"], 16, axis=1)
        v = np.where(np.repeat(s_hat, 16, axis=1) > 0, v, 0)
        assert np.sum(v > 6 * (1 + 1e-6)) <= c[0] <= np.sum(v > 6 * (1 - 1e-6))
        if held:
            assert c[0] > 0 and c[2] > 0   # the x1000 drift saturates against the held amax


def test_held_amax_refresh_rule(orc):
    x0 = random_bf16(10, (32, 64), "student_t4")
    x1 = f32_to_bf16_bits(bf16_bits_to_f32(x0) * np.float32(3.0))
    st = orc.HeldState()
    kw = dict(scale_fmt=orc.FMT_UE5M3, held=True, target_T=2048.0, refresh_every=50, sr=True, seed=2)
    # a state that is not valid yet refreshes on any step, like step 0 would
    st7 = orc.HeldState()
    q7 = orc.quantize(x0, step=7, state=st7, **kw)
    cur7 = orc.quantize(x0, step=7, scale_fmt=orc.FMT_UE5M3, target_T=2048.0, sr=True, seed=2)
    assert q7["s_dec"] == cur7["s_dec"] and np.array_equal(q7["codes"], cur7["codes"])
    assert st7.valid[0] == 1 and st7.last[0] == 7
    q0 = orc.quantize(x0, step=0, state=st, **kw)
    cur = orc.quantize(x0, step=0, scale_fmt=orc.FMT_UE5M3, target_T=2048.0, sr=True, seed=2)
    assert np.array_equal(q0["codes"], cur["codes"]) and q0["s_dec"] == cur["s_dec"]
    q49 = orc.quantize(x1, step=49, state=st, **kw)
    assert q49["s_dec"] == q0["s_dec"] and q49["amax"] == q0["amax"]
    q50 = orc.quantize(x1, step=50, state=st, **kw)
    cur50 = orc.quantize(x1, step=50, scale_fmt=orc.FMT_UE5M3, target_T=2048.0, sr=True, seed=2)
    assert q50["s_dec"] == cur50["s_dec"] != q0["s_dec"]
    assert np.array_equal(q50["codes"], cur50["codes"])
    assert st.last[0] == 50 and st.valid[0] == 1


def test_sr_is_unbiased_over_a_million_draws(orc):
    # 4.4: rounding up with probability proportional to the distance from the
    # lower neighbour makes the expected code value equal to the input.
    # Construction: one block holds 2688 so s_enc,G = 1; every other block has
    # amax 6, so its scale is 1 and v = x exactly.
    rows = 66667
    for v in [0.3046875, 1.2265625, 2.71875, 4.5625, 5.5]:
        blk = np.full((rows, 16), v, dtype=np.float32)
        blk[:, 0] = 6.0
        blk[0, 0] = 2688.0
        bits = f32_to_bf16_bits(blk)
        q = orc.quantize(bits, sr=True, seed=123, tensor_id=3, step=1)
        assert q["s_dec"] == 1.0
        vals = code_values(q["codes"])[1:, 1:]
        assert np.all(e4m3_decode(q["scales"][1:]) == 1.0)
        n = vals.size
        lo = E2M1[E2M1 <= v].max()
        hi = E2M1[E2M1 > v].min()
        assert set(np.unique(vals)) <= {lo, hi}
        bound = 5 * (hi - lo) / (2 * np.sqrt(n)) + (hi - lo) * 2.0 ** -16
        assert abs(vals.mean() - v) <= bound, (v, vals.mean())
    # RNE path draws nothing
    q1 = orc.quantize(bits, sr=False, seed=1)
    q2 = orc.quantize(bits, sr=False, seed=2)
    assert np.array_equal(q1["codes"], q2["codes"])


def test_degenerate_blocks(orc):
    x = np.zeros((16, 64), dtype=np.uint16)
    x[1, 3] = 0x8000                               # -0.0
    x[2, 16:32] = f32_to_bf16_bits(np.full(16, 1e-30, np.float32))
    x[3, 32] = f32_to_bf16_bits(np.array([5.0], np.float32))[0]
    q = orc.quantize(x)
    assert q["scales"][0, 0] == 0
    u = unpack(q["codes"])
    assert u[1, 3] == 8 and u[0, 0] == 0
    # 1e-30 next to amax 5: its block scale underflows to zero
    assert q["scales"][2, 1] == 0 and q["counters"][3] == 1 and q["counters"][1] == 16
    zero = orc.quantize(np.zeros((16, 32), dtype=np.uint16))
    assert zero["s_dec"] == 1.0 and not zero["codes"].any() and not zero["counters"].any()
    empty = orc.quantize(np.zeros((0, 32), dtype=np.uint16))
    assert empty["codes"].shape == (0, 16)


def test_mxfp4_never_saturates_elements(orc):
    x = random_bf16(12, (64, 256), "student_t4")
    q = orc.quantize(x, scale_fmt=orc.FMT_UE8M0, block=orc.BLOCK_1x32)
    assert q["counters"][0] == 0 and q["s_dec"] == 1.0
    xf = np.abs(bf16_bits_to_f32(x)).reshape(64, 8, 32).max(axis=2)
    e = q["scales"].astype(np.int64) - 127
    assert np.all(6.0 * 2.0 ** e >= xf) and np.all(6.0 * 2.0 ** (e - 1) < xf)


def test_dequantize_closed_form(orc):
    x = random_bf16(13, (32, 64), "normal")
    q = orc.quantize(x)
    deq = orc.dequantize(q["codes"], q["scales"], q["s_dec"])
    want = (code_values(q["codes"]) * np.repeat(e4m3_decode(q["scales"]), 16, axis=1)).astype(np.float32)
    want = want * np.float32(q["s_dec"])
    assert np.array_equal(deq, want)


def test_argument_validation(orc):
    x = random_bf16(14, (16, 48), "normal")
    with pytest.raises(orc.OracleError):
        orc.quantize(x[:, :40])                                  # cols not a multiple of 16
    with pytest.raises(orc.OracleError):
        orc.quantize(x, scale_fmt=orc.FMT_UE8M0)                 # MX needs 1x32
    with pytest.raises(orc.OracleError):
        orc.quantize(x, rht=True, block=orc.BLOCK_16x16)


def test_per_row_tensor_scale_is_each_rows_own_current_scale(orc):
    # B.1's finer granularity, reading: each operand row is scaled as if it were
    # the whole tensor. Row by row, the per-row mode must give the bytes that
    # current tensor scaling gives the one-row tensor x[r:r+1] (RNE), and the
    # row's s_dec must be that call's s_dec.
    rng_rows = [random_bf16(31, (1, 96), d) for d in ("normal", "student_t4", "log_normal_1e-4_2")]
    x = np.concatenate(rng_rows + [np.zeros((1, 96), np.uint16)], axis=0)  # last row all +0
    q = orc.quantize(x, per_row=True)
    assert q["s_dec"] == 0.0 and q["s_dec_rows"].shape == (4,)
    total = np.zeros(4, dtype=np.uint64)
    for r in range(x.shape[0]):
        one = orc.quantize(x[r:r + 1])
        assert np.array_equal(q["codes"][r], one["codes"][0]), r
        assert np.array_equal(q["scales"][r], one["scales"][0]), r
        assert np.float32(q["s_dec_rows"][r]) == np.float32(one["s_dec"]), r
        total += one["counters"]
    assert np.array_equal(q["counters"], total)
    # a zero row: s_enc,G = 1 (B.1 has no amax to divide by), every code +0
    assert q["s_dec_rows"][3] == 1.0 and not q["codes"][3].any()
    # the row holding amax_r gets block scale T = 448 (B.1: amax_r maps to 6 * 448)
    for r in range(3):
        vals = np.abs(bf16_bits_to_f32(x[r]))
        blk = int(np.argmax(vals)) // 16
        assert e4m3_decode(q["scales"][r:r + 1, blk:blk + 1])[0, 0] == 448.0


def test_per_row_equals_tensor_scale_when_rows_share_their_amax(orc):
    # every row holds the same amax (one planted 8.0 per row), so each row's
    # scale equals the tensor's: the per-row mode must reproduce current tensor
    # scaling bit for bit, SR draws included (they index the whole operand)
    x = random_bf16(32, (48, 64), "normal")
    v = np.abs(bf16_bits_to_f32(x))
    assert v.max() < 8.0
    x[:, 5] = f32_to_bf16_bits(np.full(48, 8.0, np.float32))
    for sr in (False, True):
        a = orc.quantize(x, per_row=True, sr=sr, seed=9, tensor_id=2, step=4)
        b = orc.quantize(x, sr=sr, seed=9, tensor_id=2, step=4)
        assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["scales"], b["scales"])
        assert np.all(a["s_dec_rows"] == np.float32(b["s_dec"]))
        assert np.array_equal(a["counters"], b["counters"])
    # operand-row windows see the same rows
    w = orc.quantize(x, per_row=True, op_rows=(16, 32))
    full = orc.quantize(x, per_row=True)
    assert np.array_equal(w["codes"], full["codes"][16:32])
    assert np.array_equal(w["s_dec_rows"], full["s_dec_rows"][16:32])


def test_per_row_rejects_what_it_does_not_define(orc):
    x = random_bf16(33, (32, 64), "normal")
    for kw in (dict(colwise=True), dict(colwise=True, rht=True), dict(held=True),
               dict(block=orc.BLOCK_16x16), dict(scale_fmt=orc.FMT_UE8M0, block=orc.BLOCK_1x32)):
        with pytest.raises(orc.OracleError):
            orc.quantize(x, per_row=True, **kw)
