"""Pins for the oracle's block-scaled GEMM ("Pretraining Large Language Models
with NVFP4", App. B.3 and section A3: per-block partial dot products times both
block decode scales, accumulated, then times both global decode scales).

Checks: exact rational arithmetic (Python Fractions) on small shapes, numpy's
float64 matmul of independently dequantized operands, and an exhaustive table of
all 16 x 16 code pairs.
"""
from fractions import Fraction

import numpy as np
import torch

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _val(code):
    return (-1 if code & 8 else 1) * E2M1[code & 7]


def _rand_operand(rng, rows, K, scale_lo=0x20, scale_hi=0x60):
    codes = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi, size=(rows, K // 16), dtype=np.uint8)
    return codes, scales


def _e4m3(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


def _dequant64(codes, scales):
    lo, hi = codes & 0xF, codes >> 4
    u = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    u[:, 0::2], u[:, 1::2] = lo, hi
    v = np.vectorize(_val, otypes=[np.float64])(u)
    return v * np.repeat(_e4m3(scales), 16, axis=1)


def test_gemm_exact_rational(orc):
    rng = np.random.default_rng(21)
    M, N, K = 8, 8, 64
    ac, asc = _rand_operand(rng, M, K)
    bc, bsc = _rand_operand(rng, N, K)
    sa, sb = np.float32(0.0123), np.float32(3.7)
    c, s = orc.gemm(ac, asc, float(sa), bc, bsc, float(sb))
    A, B = _dequant64(ac, asc), _dequant64(bc, bsc)
    alpha = Fraction(float(sa)) * Fraction(float(sb))
    for m in range(M):
        for n in range(N):
            exact = alpha * sum(Fraction(A[m, k]) * Fraction(B[n, k]) for k in range(K))
            sabs = abs(alpha) * sum(abs(Fraction(A[m, k]) * Fraction(B[n, k])) for k in range(K))
            assert abs(Fraction(c[m, n]) - exact) <= Fraction(2) ** -45 * sabs
            assert abs(Fraction(s[m, n]) - sabs) <= Fraction(2) ** -45 * sabs


def test_gemm_matches_numpy_on_dequantized_operands(orc):
    rng = np.random.default_rng(22)
    M, N, K = 64, 64, 64
    ac, asc = _rand_operand(rng, M, K)
    bc, bsc = _rand_operand(rng, N, K)
    c, s = orc.gemm(ac, asc, 0.5, bc, bsc, 0.25)
    A, B = _dequant64(ac, asc), _dequant64(bc, bsc)
    ref = 0.125 * (A @ B.T)
    sref = 0.125 * (np.abs(A) @ np.abs(B).T)
    assert np.all(np.abs(c - ref) <= 1e-12 * sref + 1e-300)
    assert np.allclose(s, sref, rtol=1e-12)
    # sampled outputs equal the full ones
    ms, ns = rng.integers(0, M, 50), rng.integers(0, N, 50)
    cs, ss = orc.gemm(ac, asc, 0.5, bc, bsc, 0.25, pairs=(ms, ns))
    assert np.array_equal(cs, c[ms, ns]) and np.array_equal(ss, s[ms, ns])


def test_gemm_exhaustive_code_pairs(orc):
    # row i of A holds code i in every position, row j of B code j: C[i, j] = K v_i v_j s_a s_b
    K = 32
    ac = np.array([[i | (i << 4)] * (K // 2) for i in range(16)], dtype=np.uint8)
    bc = ac.copy()
    asc = np.full((16, K // 16), 0x38, dtype=np.uint8)   # E4M3 1.0
    bsc = np.full((16, K // 16), 0x40, dtype=np.uint8)   # E4M3 2.0
    c, s = orc.gemm(ac, asc, 1.0, bc, bsc, 1.0)
    for i in range(16):
        for j in range(16):
            assert c[i, j] == K * _val(i) * _val(j) * 1.0 * 2.0
            assert s[i, j] == abs(c[i, j])


def test_gemm_mxfp4_block32_exact_rational(orc):
    # MXFP4 ("Pretraining Large Language Models with NVFP4", A3): UE8M0 block
    # scales are powers of two 2^(code - 127), one per 32 values; no tensor scale
    rng = np.random.default_rng(23)
    M, N, K = 6, 5, 96
    ac = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    bc = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    asc = rng.integers(100, 150, size=(M, K // 32), dtype=np.uint8)
    bsc = rng.integers(110, 140, size=(N, K // 32), dtype=np.uint8)
    c, s = orc.gemm(ac, asc, 1.0, bc, bsc, 1.0, scale_fmt=orc.FMT_UE8M0, bs=32)

    def val(codes, scales, r, k):
        byte = int(codes[r, k // 2])
        code = byte & 0xF if k % 2 == 0 else byte >> 4
        return Fraction(_val(code)) * Fraction(2) ** (int(scales[r, k // 32]) - 127)

    for m in range(M):
        for n in range(N):
            terms = [val(ac, asc, m, k) * val(bc, bsc, n, k) for k in range(K)]
            exact, sabs = sum(terms), sum(abs(t) for t in terms)
            assert abs(Fraction(c[m, n]) - exact) <= Fraction(2) ** -45 * sabs
            assert Fraction(s[m, n]) == sabs or abs(Fraction(s[m, n]) - sabs) <= Fraction(2) ** -45 * sabs


def test_gemm_zero_bound_means_zero(orc):
    ac = np.zeros((4, 16), dtype=np.uint8)
    c, s = orc.gemm(ac, np.zeros((4, 2), np.uint8), 1.0, ac, np.zeros((4, 2), np.uint8), 1.0)
    assert not c.any() and not s.any()


def test_scale_layout_is_a_bijection(orc):
    R, NB = 256, 12
    idx = np.arange(R * NB, dtype=np.int64).reshape(R, NB)
    lo = orc.swizzle_scales((idx & 0xFF).astype(np.uint8)).astype(np.int64)
    hi = orc.swizzle_scales((idx >> 8).astype(np.uint8)).astype(np.int64)
    perm = lo | (hi << 8)
    assert np.array_equal(np.sort(perm), np.arange(R * NB))


def test_scale_layout_positions(orc):
    # 128 rows x 4 blocks per 512-byte chunk: row r, block j at 16 (r % 32) + 4 (r // 32) + j;
    # chunks of one 128-row tile are contiguous along K
    R, NB = 256, 8
    for (r, j, off) in [(0, 0, 0), (0, 1, 1), (1, 0, 16), (32, 0, 4), (127, 3, 511),
                        (0, 4, 512), (128, 0, 1024), (129, 5, 1024 + 512 + 16 + 1)]:
        plain = np.zeros((R, NB), dtype=np.uint8)
        plain[r, j] = 1
        assert np.flatnonzero(orc.swizzle_scales(plain)).tolist() == [off]


def test_gemm_per_row_a_scale_exact_rational(orc):
    # A's decode scale per row (B.1's finer granularity): C[m, n] = sa[m] sb sum_k a b
    rng = np.random.default_rng(23)
    M, N, K = 6, 5, 64
    ac, asc = _rand_operand(rng, M, K)
    bc, bsc = _rand_operand(rng, N, K)
    sa = np.array([0.0123, 1.0, 2.0 ** -20, 7.25, 0.5, 3.0e4], dtype=np.float32)
    sb = np.float32(0.375)
    c, s = orc.gemm(ac, asc, sa, bc, bsc, float(sb))
    A, B = _dequant64(ac, asc), _dequant64(bc, bsc)
    for m in range(M):
        alpha = Fraction(float(sa[m])) * Fraction(float(sb))
        for n in range(N):
            exact = alpha * sum(Fraction(A[m, k]) * Fraction(B[n, k]) for k in range(K))
            sabs = abs(alpha) * sum(abs(Fraction(A[m, k]) * Fraction(B[n, k])) for k in range(K))
            assert abs(Fraction(c[m, n]) - exact) <= Fraction(2) ** -45 * sabs
            assert abs(Fraction(s[m, n]) - sabs) <= Fraction(2) ** -45 * sabs
    ms, ns = np.array([5, 0, 3]), np.array([1, 4, 0])
    cs, ss = orc.gemm(ac, asc, sa, bc, bsc, float(sb), pairs=(ms, ns))
    assert np.array_equal(cs, c[ms, ns]) and np.array_equal(ss, s[ms, ns])
