"""Pins for the oracle's Philox4x32-10 generator and the 16x16 random Hadamard
transform ("Pretraining Large Language Models with NVFP4", section 4.2, App. C).

Philox is checked against Triton's independent implementation (its CPU
interpreter); so are the words the stochastic-rounding draws and the RHT sign
vector are taken from. The draws are further pinned by statistics a uniform,
independent 16-bit source must pass (bit balance, chi-square over all 2^16
values, independence of draws that share a Philox word or block, distinct
streams per tensor id, step, seed and high counter word); the sign vector by
bit balance over seeds and by being the same for every tensor id and step
(section 4.2: one random sign vector for the whole run). The Hadamard transform
is checked against the Kronecker recursion the page states, against scipy's
Sylvester Hadamard matrix, and by orthogonality.
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


def _triton_philox(cases):
    """Philox4x32-10 words from Triton's implementation (CPU interpreter), which
    shares no code with the oracle: cases = [[seed, [[c0, c1, c2, c3], ...]], ...]
    (at most 64 counters per case) -> the four output words per counter."""
    pytest.importorskip("triton")
    import json
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", TRITON_PROBE], input=json.dumps(cases),
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_philox_matches_triton(orc):
    rng = np.random.default_rng(7)
    cases = []
    seeds = [0, 1, 0xFFFFFFFF, 0x123456789ABCDEF0, int(rng.integers(0, 2**63))]
    for seed in seeds:
        ctrs = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64).tolist()
        ctrs[0] = [0, 0, 0, 0]
        ctrs[1] = [0, 0, 0xFFFFFFFF, 0xFFFFFFFF]
        cases.append([seed, ctrs])
    want = _triton_philox(cases)
    for (seed, ctrs), w in zip(cases, want):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for ctr, ww in zip(ctrs, w):
            assert orc.philox4x32_10(ctr, key).tolist() == ww


def _draw_from_word(word: int, e: int) -> int:
    # the reading's byte map: the element with (e >> 1) & 1 == 0 takes bytes 2
    # (high) and 0 (low) of its word, the other bytes 3 and 1
    b = int(word).to_bytes(4, "little")
    return b[2] * 256 + b[0] if (e >> 1) & 1 == 0 else b[3] * 256 + b[1]


def test_sr_draws_and_rht_signs_from_triton_words(orc):
    """The SR draw of element e comes from word 2 ((e >> 2) & 1) + (e & 1) of
    Philox(key = seed, counter = (lo32(e >> 3), hi32(e >> 3), tensor_id,
    lo32(step))), and the RHT sign vector is the low 16 bits of word 0 at counter
    (0, 0, 0xFFFFFFFF, 0xFFFFFFFF): both checked on words Triton generates, so
    the oracle's generator, key split and counter layout are not checked against
    themselves."""
    rng = np.random.default_rng(21)
    es = [0, 1, 2, 3, 4, 5, 6, 7, 8, 15, 16, 1023, (1 << 32) + 3, (1 << 33) + 6, (1 << 35) + 1,
          (1 << 40) + 14, (1 << 47) - 1] + [int(v) for v in rng.integers(0, 2**44, size=15)]
    streams = [(0, 0, 0), (0xDEADBEEF12345, 3, 77), (1, 0xFFFFFFFE, (1 << 32) + 5),
               (0xFFFFFFFFFFFFFFFF, 12, 123456789)]
    cases, want_sr = [], []
    for seed, tid, step in streams:
        ctrs = [[(e >> 3) & 0xFFFFFFFF, (e >> 35) & 0xFFFFFFFF, tid, step & 0xFFFFFFFF] for e in es]
        cases.append([seed, ctrs])
    sign_seeds = [0, 1, 2, 99, 12345, 0xFFFFFFFF, 1 << 32, 0x0123456789ABCDEF]
    for sd in sign_seeds:
        cases.append([sd, [[0, 0, 0xFFFFFFFF, 0xFFFFFFFF]]])
    words = _triton_philox(cases)
    for (seed, tid, step), w in zip(streams, words[:len(streams)]):
        for e, ww in zip(es, w):
            want = _draw_from_word(ww[2 * ((e >> 2) & 1) + (e & 1)], e)
            assert orc.sr_bits(seed, tid, step, e) == want, (seed, tid, step, e)
    for sd, w in zip(sign_seeds, words[len(streams):]):
        assert orc.rht_sign_word(sd) == (w[0][0] & 0xFFFF), sd


def _draws(orc, seed, tid, step, es):
    return np.array([orc.sr_bits(seed, tid, step, int(e)) for e in es], dtype=np.int64)


def _chi2_indep(a, b, nbins):
    t = np.zeros((nbins, nbins))
    np.add.at(t, (a, b), 1)
    exp = np.outer(t.sum(1), t.sum(0)) / t.sum()
    return float(((t - exp) ** 2 / exp).sum()), (nbins - 1) ** 2


def test_sr_draws_are_uniform_and_independent(orc):
    """Section 4.4 needs each element's rounding decision to be an independent
    uniform draw. Over 2^20 consecutive elements of one stream: every one of
    the 16 bits is set half the time, all 2^16 values are equally frequent
    (chi-square), and draws that share a Philox word (e, e + 2), a Philox call
    (e, e + 1), (e, e + 4) or neighbouring calls (e, e + 8) are independent
    (chi-square of their top nibbles). Each bound is 6 standard deviations."""
    N = 1 << 20
    seed, tid, step = 0x1234_5678_9ABC, 3, 77
    d = _draws(orc, seed, tid, step, range(N))
    assert d.min() >= 0 and d.max() < 65536
    sigma_bit = np.sqrt(N) / 2
    for b in range(16):
        ones = int(((d >> b) & 1).sum())
        assert abs(ones - N / 2) <= 6 * sigma_bit, (b, ones)
    counts = np.bincount(d, minlength=65536)
    expect = N / 65536
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    df = 65535
    assert abs(chi2 - df) <= 6 * np.sqrt(2 * df), chi2
    e = np.arange(N)
    top = d >> 12
    for lag, sel in [(2, ((e >> 1) & 1) == 0), (1, (e & 1) == 0), (4, ((e >> 2) & 1) == 0),
                     (8, ((e >> 3) & 1) == 0)]:
        i = e[sel & (e + lag < N)]
        c2, df2 = _chi2_indep(top[i], top[i + lag], 16)
        assert abs(c2 - df2) <= 6 * np.sqrt(2 * df2), (lag, c2)


def test_sr_streams_differ_by_tensor_step_seed_and_high_counter(orc):
    """Each key (seed) and counter field (tensor id, step, high word of e >> 3)
    selects its own stream: against the base stream, equal draws occur at the
    2^-16 rate of independent streams, and the pairs pass the independence
    chi-square. A counter field left out of the generator's input would make a
    stream identical to the base one."""
    N = 1 << 17
    seed, tid, step = 0xC0FFEE, 4, 1000
    es = np.arange(N)
    base = _draws(orc, seed, tid, step, es)
    others = {
        "tensor_id": _draws(orc, seed, tid + 1, step, es),
        "step": _draws(orc, seed, tid, step + 1, es),
        "seed": _draws(orc, seed + 1, tid, step, es),
        "seed_hi": _draws(orc, seed + (1 << 32), tid, step, es),
        "hi_counter": _draws(orc, seed, tid, step, es + (1 << 35)),
    }
    for name, o in others.items():
        eq = int((o == base).sum())
        lam = N / 65536
        assert eq <= lam + 6 * np.sqrt(lam), (name, eq)
        c2, df2 = _chi2_indep(base >> 12, o >> 12, 16)
        assert abs(c2 - df2) <= 6 * np.sqrt(2 * df2), (name, c2)
    # reading: the counter holds the low 32 bits of the step only
    assert np.array_equal(_draws(orc, seed, tid, step + (1 << 32), es[:256]), base[:256])


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


def test_rht_sign_bits_balanced_over_seeds(orc):
    """The sign vector is random: over 8192 seeds each of the 16 signs is
    negative half the time (6 standard deviations), and the vectors are all
    but never equal (at most a few birthday collisions among 2^16 values)."""
    n = 8192
    words = np.array([orc.rht_sign_word(s) for s in range(n)], dtype=np.int64)
    assert words.max() < 65536
    for b in range(16):
        ones = int(((words >> b) & 1).sum())
        assert abs(ones - n / 2) <= 6 * np.sqrt(n) / 2, (b, ones)
    collisions = n - len(set(words.tolist()))
    lam = n * (n - 1) / 2 / 65536
    assert collisions <= lam + 6 * np.sqrt(lam)


def test_rht_sign_vector_shared_by_every_tensor_and_step(orc):
    """Section 4.2: one random sign vector serves every layer for the whole run.
    The colwise RHT quantization of one input with round-to-nearest gives the
    same bytes whatever its tensor id and step; with stochastic rounding the
    codes change with them (their own random stream) but the block scales,
    computed from the rotated values, do not."""
    from workloads import random_bf16
    x = random_bf16(77, (64, 48), "normal")
    ref = orc.quantize(x, colwise=True, rht=True, seed=5, tensor_id=1, step=0)
    for tid, step in [(4, 0), (9, 77), (1, 50), (8 * 31 + 4, 123456)]:
        q = orc.quantize(x, colwise=True, rht=True, seed=5, tensor_id=tid, step=step)
        assert np.array_equal(q["codes"], ref["codes"]) and np.array_equal(q["scales"], ref["scales"])
        assert q["s_dec"] == ref["s_dec"]
    sr_ref = orc.quantize(x, colwise=True, rht=True, sr=True, seed=5, tensor_id=1, step=0)
    sr_other = orc.quantize(x, colwise=True, rht=True, sr=True, seed=5, tensor_id=4, step=3)
    assert np.array_equal(sr_other["scales"], sr_ref["scales"]) and sr_other["s_dec"] == sr_ref["s_dec"]
    assert not np.array_equal(sr_other["codes"], sr_ref["codes"])
    # a different seed is a different rotation
    other = orc.quantize(x, colwise=True, rht=True, seed=6, tensor_id=1, step=0)
    assert not np.array_equal(other["codes"], ref["codes"])
