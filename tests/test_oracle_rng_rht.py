"""Pins for the oracle's Philox4x32-10 generator and the 16x16 random Hadamard
transform ("Pretraining Large Language Models with NVFP4", section 4.2, App. C).

Philox is checked against Triton's independent implementation (its CPU
interpreter); the Hadamard transform against the Kronecker recursion the page
states, against scipy's Sylvester Hadamard matrix, and by orthogonality.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import scipy.linalg

TRITON_PROBE = r'''
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl
@triton.jit
def k(seed, c0p, c1p, c2p, c3p, o0, o1, o2, o3, n, BLOCK: tl.constexpr):
    i = tl.arange(0, BLOCK)
    m = i < n
    c0 = tl.load(c0p + i, mask=m); c1 = tl.load(c1p + i, mask=m)
    c2 = tl.load(c2p + i, mask=m); c3 = tl.load(c3p + i, mask=m)
    a, b, c, d = tl.random.philox(seed, c0, c1, c2, c3)
    tl.store(o0 + i, a, mask=m); tl.store(o1 + i, b, mask=m)
    tl.store(o2 + i, c, mask=m); tl.store(o3 + i, d, mask=m)
cases = json.loads(sys.stdin.read())
out = []
for seed, ctrs in cases:
    cs = [torch.tensor([c[j] for c in ctrs], dtype=torch.uint32) for j in range(4)]
    os_ = [torch.empty(len(ctrs), dtype=torch.uint32) for _ in range(4)]
    k[(1,)](seed, *cs, *os_, len(ctrs), BLOCK=64)
    out.append([[int(os_[j][i]) & 0xFFFFFFFF for j in range(4)] for i in range(len(ctrs))])
print(json.dumps(out))
'''


def test_philox_matches_triton(orc):
    pytest.importorskip("triton")
    import json
    rng = np.random.default_rng(7)
    cases = []
    seeds = [0, 1, 0xFFFFFFFF, 0x123456789ABCDEF0, int(rng.integers(0, 2**63))]
    for seed in seeds:
        ctrs = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64).tolist()
        ctrs[0] = [0, 0, 0, 0]
        ctrs[1] = [0, 0, 0xFFFFFFFF, 0xFFFFFFFF]
        cases.append([seed, ctrs])
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", TRITON_PROBE], input=json.dumps(cases),
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    want = json.loads(res.stdout.strip().splitlines()[-1])
    for (seed, ctrs), w in zip(cases, want):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for ctr, ww in zip(ctrs, w):
            assert orc.philox4x32_10(ctr, key).tolist() == ww


def test_sr_bits_index_contract(orc):
    # one Philox block per 8 elements (counter e >> 3); word 2 ((e >> 2) & 1) +
    # (e & 1); the element with (e >> 1) & 1 == 0 takes bytes 2:0 of the word,
    # the other bytes 3:1 (high byte first)
    seed, tid, step = 0xDEADBEEF12345, 3, 77
    for e in [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 1 << 33, (1 << 40) + 5, (1 << 40) + 14]:
        w = orc.philox4x32_10([(e >> 3) & 0xFFFFFFFF, (e >> 35) & 0xFFFFFFFF, tid, step & 0xFFFFFFFF],
                              [seed & 0xFFFFFFFF, seed >> 32])
        b = int(w[2 * ((e >> 2) & 1) + (e & 1)]).to_bytes(4, "little")
        want = b[2] * 256 + b[0] if (e >> 1) & 1 == 0 else b[3] * 256 + b[1]
        assert orc.sr_bits(seed, tid, step, e) == want
    # the eight elements of one block use all 256 bits once
    got = sorted(orc.sr_bits(seed, tid, step, e) for e in range(8))
    w = orc.philox4x32_10([0, 0, tid, step], [seed & 0xFFFFFFFF, seed >> 32])
    halves = []
    for x in w.tolist():
        b = x.to_bytes(4, "little")
        halves += [b[2] * 256 + b[0], b[3] * 256 + b[1]]
    assert got == sorted(halves)


def _kron_hadamard(n):
    # App. C: H_N = H_2 (x) H_{N/2} with +-1 entries (normalisation applied separately)
    if n == 1:
        return np.ones((1, 1))
    h2 = np.array([[1.0, 1.0], [1.0, -1.0]])
    return np.kron(h2, _kron_hadamard(n // 2))


def test_hadamard16_orthogonality():
    h = _kron_hadamard(16)
    assert np.array_equal(h @ h.T, 16 * np.eye(16))
    assert np.array_equal(h, scipy.linalg.hadamard(16))


def _signs(orc, seed):
    w = orc.rht_sign_word(seed)
    return np.array([-1.0 if (w >> i) & 1 else 1.0 for i in range(16)])


def test_rht16_is_signed_normalised_hadamard(orc):
    h = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(11)
    for seed in [0, 1, 12345]:
        d = _signs(orc, seed)
        for _ in range(200):
            v = rng.standard_normal(16).astype(np.float32) * np.float32(10 ** rng.uniform(-4, 4))
            want = d * (h @ v.astype(np.float64)) / 4.0
            got = orc.rht16(v, seed).astype(np.float64)
            tol = 16 * 2.0 ** -24 * np.sum(np.abs(v)) / 4.0
            assert np.all(np.abs(got - want) <= tol)


def test_rht16_sign_applied_after_hadamard(orc):
    # H_r = D_r H: the unit vector e_j maps to column j of H with row i negated when d_i = -1
    h = scipy.linalg.hadamard(16)
    for seed in [0, 1, 99]:
        d = _signs(orc, seed)
        assert not np.all(d == 1) and not np.all(d == -1)
        for j in range(16):
            e = np.zeros(16, dtype=np.float32)
            e[j] = 1.0
            assert np.array_equal(orc.rht16(e, seed), (d * h[:, j] / 4.0).astype(np.float32))


def test_rht16_preserves_dot_products(orc):
    rng = np.random.default_rng(5)
    for _ in range(100):
        a = rng.standard_normal(16).astype(np.float32)
        b = rng.standard_normal(16).astype(np.float32)
        ra, rb = orc.rht16(a, 0).astype(np.float64), orc.rht16(b, 0).astype(np.float64)
        # orthogonal up to the 1/4 normalisation: <Ha, Hb> = 16 <a, b>, so <Ra, Rb> = <a, b>
        assert abs(ra @ rb - a.astype(np.float64) @ b) <= 1e-5 * (np.abs(a) @ np.abs(b) + 1)


def test_rht_sign_vector_depends_on_seed_only(orc):
    assert orc.rht_sign_word(0) == orc.rht_sign_word(0)
    assert len({orc.rht_sign_word(s) for s in range(8)}) > 1
