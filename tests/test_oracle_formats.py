"""Pins for the oracle's number formats (CPU only).

Each check compares the oracle with something other than itself: the value set
and limits the pages print (tests/golden), PyTorch's float8_e4m3fn conversion,
or a brute-force nearest-value search written here from the format definition.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_values(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(line)
    return vals


def _read_kv(name):
    return dict(line.split() for line in _read_values(name))


E2M1_SET = [float(v) for v in _read_values("e2m1_value_set.txt")]
LIMITS = _read_kv("format_limits.txt")


def test_e2m1_decode_matches_page_value_set(orc):
    assert len(E2M1_SET) == 8
    for code in range(8):
        assert orc.e2m1_value(code) == E2M1_SET[code]
        assert orc.e2m1_value(code | 8) == -E2M1_SET[code]
    assert max(E2M1_SET) == float(LIMITS["e2m1_max"])


def _brute_e2m1(x: float) -> int:
    """Nearest E2M1 magnitude, ties to the even code, saturating at 6."""
    a = abs(x)
    sign = 8 if math.copysign(1.0, x) < 0 else 0
    if a >= E2M1_SET[-1]:
        return sign | 7
    best, best_d = None, None
    for idx, m in enumerate(E2M1_SET):
        d = abs(a - m)
        if best is None or d < best_d or (d == best_d and idx % 2 == 0):
            best, best_d = idx, d
    return sign | best


def test_e2m1_rne_exhaustive_over_bf16(orc):
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    L = orc.lib()
    bad = []
    for b, v in zip(bits[finite], vals[finite]):
        got = L.orc_e2m1_rne(float(v))
        want = _brute_e2m1(float(v))
        if got != want:
            bad.append((hex(int(b)), float(v), got, want))
            if len(bad) > 10:
                break
    assert not bad, bad


def test_e2m1_rne_ties_go_to_even_code(orc):
    # midpoints between neighbouring magnitudes, and the expected even-code winner
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        assert orc.e2m1_value(orc.e2m1_rne(v)) == want
        assert orc.e2m1_value(orc.e2m1_rne(-v)) == -want
    assert orc.e2m1_rne(-0.0) == 8
    assert orc.e2m1_rne(-0.1) == 8
    assert orc.e2m1_rne(1e30) == 7


def test_e2m1_sr_thresholds_worked_by_hand(orc):
    # 4.4 stochastic rounding, reading: up iff R + floor(frac * 2^16) >= 2^16 for
    # the element's 16-bit draw R (the native FP4 SR conversion's contract). Each
    # case: value, lower code, and the first R that rounds UP (every R below it
    # rounds down), worked out by hand from frac; None = no draw rounds up.
    cases = [
        (1.25, 2, 1 << 15),                   # lo 1, hi 1.5: frac 1/2 -> 32768 -> R >= 32768
        (0.75, 1, 1 << 15),                   # lo 0.5, hi 1: frac 1/2
        (0.3046875, 0, 65536 - 39936),        # lo 0, hi 0.5: frac 0.609375 -> 39936
        (5.5, 6, 65536 - 49152),              # lo 4, hi 6: frac 3/4 -> 49152
        (1.0 + 2.0 ** -17 + 2.0 ** -21, 2, 65535),  # frac 2^-16 + 2^-20 -> floor 1
        (1.0 + 3 * 2.0 ** -17, 2, 65533),     # frac 3 * 2^-16 -> 3
        (2.0 ** -17, 0, 65535),               # frac 2^-16 -> 1: only R = 0xFFFF rounds up
        (2.0 ** -20, 0, None),                # frac 2^-19 -> floor 0: never up
    ]
    for v, lo_code, first_up in cases:
        for sgn in (1.0, -1.0):
            sign = 8 if sgn < 0 else 0
            assert orc.e2m1_sr(sgn * v, 0) == sign | lo_code, v
            if first_up is None:
                assert orc.e2m1_sr(sgn * v, 0xFFFF) == sign | lo_code, v
                continue
            assert orc.e2m1_sr(sgn * v, first_up - 1) == sign | lo_code, (v, first_up)
            assert orc.e2m1_sr(sgn * v, first_up) == sign | (lo_code + 1), (v, first_up)
            assert orc.e2m1_sr(sgn * v, 0xFFFF) == sign | (lo_code + 1), v
    # on the grid nothing rounds up, whatever the draw
    for v, code in ((1.0, 2), (3.0, 5), (0.0, 0), (0.5, 1)):
        assert orc.e2m1_sr(v, 0xFFFF) == code
    assert orc.e2m1_sr(-0.0, 0xFFFF) == 8
    assert orc.e2m1_sr(6.0, 0) == 7 and orc.e2m1_sr(-7.0, 0) == 15 and orc.e2m1_sr(1e30, 0) == 7


def test_e2m1_sr_probability_by_enumerating_every_draw(orc):
    # 4.4: rounding up with probability proportional to the distance from the lower
    # neighbour. Over all 2^16 draws exactly floor(frac * 2^16) must round up, for
    # fractions that 16 bits hold exactly and for ones they truncate (1/3, 1/7, ...).
    from fractions import Fraction
    cases = [(1.25, 1.0, 1.5), (0.3046875, 0.0, 0.5), (5.5, 4.0, 6.0),
             (1.0 + 1.0 / 6.0, 1.0, 1.5), (2.0 + 1.0 / 7.0, 2.0, 3.0), (0.5 + 1.0 / 3.0 / 2.0, 0.5, 1.0),
             (4.0 + 2.0 ** -15, 4.0, 6.0), (2.0 ** -18, 0.0, 0.5)]
    for v, lo, hi in cases:
        v32 = float(np.float32(v))
        frac = (Fraction(v32) - Fraction(lo)) / (Fraction(hi) - Fraction(lo))
        want = int(frac * 65536)  # floor
        lo_code = E2M1_SET.index(lo)  # the page's value set, in code order
        codes = np.array([orc.e2m1_sr(v32, r) for r in range(65536)])
        assert set(np.unique(codes)) <= {lo_code, lo_code + 1}
        assert int(np.sum(codes == lo_code + 1)) == want, (v, want)
        # the draws that round up are the top ones: R >= 2^16 - floor(frac * 2^16)
        assert np.all(codes[65536 - want:] == lo_code + 1) and np.all(codes[:65536 - want] == lo_code)


def _brute_nearest(s: float, table: list[float]) -> int:
    """Index of the nearest table value, ties to the even index, saturating."""
    if s >= table[-1]:
        return len(table) - 1
    best, best_d = 0, None
    for i, t in enumerate(table):
        d = abs(s - t)
        if best_d is None or d < best_d or (d == best_d and i % 2 == 0):
            best, best_d = i, d
    return best


def _e4m3_table():
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().tolist()


def test_e4m3_decode_matches_torch(orc):
    table = _e4m3_table()
    for code, v in enumerate(table):
        assert orc.scale_decode(orc.FMT_E4M3, code) == v
    assert table[-1] == float(LIMITS["e4m3_max"])


def _probe_values(table, rng, n_random):
    vals = list(table)
    for a, b in zip(table[:-1], table[1:]):
        mid = (a + b) / 2
        vals += [mid, np.nextafter(np.float32(mid), np.float32(0)).item(),
                 np.nextafter(np.float32(mid), np.float32(1e9)).item()]
    vals += list(rng.uniform(0, table[-1] * 1.1, size=n_random))
    vals += list(np.exp(rng.uniform(np.log(1e-8), np.log(table[-1]), size=n_random)))
    return [float(np.float32(v)) for v in vals]


def test_e4m3_encode_matches_torch_and_brute_force(orc):
    table = _e4m3_table()
    rng = np.random.default_rng(1)
    vals = _probe_values(table, rng, 3000)
    tv = torch.tensor(vals, dtype=torch.float32)
    in_range = tv <= 448.0
    torch_rt = tv[in_range].to(torch.float8_e4m3fn).float().tolist()
    ours_in = [orc.scale_decode(orc.FMT_E4M3, orc.scale_encode(orc.FMT_E4M3, v))
               for v, ok in zip(vals, in_range.tolist()) if ok]
    assert ours_in == torch_rt
    for v in vals:
        assert orc.scale_encode(orc.FMT_E4M3, v) == _brute_nearest(v, table)
    assert orc.scale_encode(orc.FMT_E4M3, 1e6) == 0x7E
    assert orc.scale_encode(orc.FMT_E4M3, 2.0 ** -10) == 0      # half the smallest subnormal: tie to 0
    assert orc.scale_encode(orc.FMT_E4M3, 2.0 ** -10 * 1.0001) == 1


def _ue5m3_table():
    # Reading (the pages name UE5M3 but give no encoding): unsigned, 5 exponent bits
    # with bias 15, 3 mantissa bits, subnormals at exponent 0, 0xFF reserved.
    t = []
    for code in range(0xFF):
        e, m = code >> 3, code & 7
        t.append(m / 8 * 2.0 ** -14 if e == 0 else (1 + m / 8) * 2.0 ** (e - 15))
    return t


def test_ue5m3_encode_brute_force(orc):
    table = _ue5m3_table()
    assert table == sorted(table) and len(set(table)) == 255
    for code, v in enumerate(table):
        assert orc.scale_decode(orc.FMT_UE5M3, code) == v
    assert table[-1] == orc.scale_max(orc.FMT_UE5M3) == 114688.0
    assert table[1] == 2.0 ** -17
    rng = np.random.default_rng(2)
    vals = _probe_values(table, rng, 3000)
    for v in vals:
        assert orc.scale_encode(orc.FMT_UE5M3, v) == _brute_nearest(v, table)
    # 448 and 2048, the targets T of the periodic-scaling recipe, are exact
    assert orc.scale_decode(orc.FMT_UE5M3, orc.scale_encode(orc.FMT_UE5M3, 448.0)) == 448.0
    assert orc.scale_decode(orc.FMT_UE5M3, orc.scale_encode(orc.FMT_UE5M3, 2048.0)) == 2048.0


def test_ue8m0_range_matches_page(orc):
    lo, hi = int(LIMITS["ue8m0_min_exp"]), int(LIMITS["ue8m0_max_exp"])
    assert orc.scale_decode(orc.FMT_UE8M0, 0) == 2.0 ** lo
    assert orc.scale_decode(orc.FMT_UE8M0, 254) == 2.0 ** hi
    for code in range(255):
        assert orc.scale_decode(orc.FMT_UE8M0, code) == 2.0 ** (code - 127)


def test_ue8m0_round_up_is_smallest_covering_power(orc):
    rng = np.random.default_rng(3)
    vals = list(np.exp(rng.uniform(np.log(1e-30), np.log(1e30), size=2000)).astype(np.float32))
    vals += [6.0 * 2.0 ** k for k in range(-20, 20)]
    for a in vals:
        a = float(np.float32(a))
        e = orc.ue8m0_exponent(a)
        assert 6.0 * 2.0 ** e >= a
        assert 6.0 * 2.0 ** (e - 1) < a


def test_mxfp4_worked_example_appendix_b4(orc):
    ex = _read_kv("mxfp4_worked_example.txt")
    eps = 2.0 ** -6   # 3 + eps must be exact in BF16 (8 significant bits)
    amax = 3.0 + eps
    e = orc.ue8m0_exponent(amax)
    assert 2.0 ** e == float(ex["decode_scale"])
    # the block through the full quantizer: amax element -> 3, nothing reaches 4 or 6
    from workloads import f32_to_bf16_bits
    vals = np.linspace(-amax, amax, 32).astype(np.float32)
    vals[0] = amax
    bits = f32_to_bf16_bits(vals.reshape(1, 32))
    q = orc.quantize(bits, scale_fmt=orc.FMT_UE8M0, block=orc.BLOCK_1x32)
    assert q["scales"][0, 0] == 127
    deq = orc.dequantize(q["codes"], q["scales"], 1.0, orc.FMT_UE8M0, 32)
    assert np.max(np.abs(deq)) == float(ex["max_code_value"])
    assert not np.any(np.isin(np.abs(deq), [4.0, 6.0]))
    assert round(math.log2(3 / 0.5), 2) == float(ex["binades_used"])
    assert round(math.log2(6 / 0.5), 2) == float(ex["binades_full"])
    assert int(LIMITS["mxfp4_block"]) == 32 and int(LIMITS["nvfp4_block"]) == 16
