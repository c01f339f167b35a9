"""The synthetic input recipe: shapes, distributions and seeding of the
stand-in tensors for the pages' linears (CPU only; no method arithmetic)."""
import numpy as np
import torch

from workloads import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, linear_inputs, random_bf16,
                       sweep_dy)


def test_shapes_of_the_five_workloads():
    want = {"tiny": [(256, 256, 256)], "1.2b": [(8192, 2048, 6144), (8192, 6144, 2048)],
            "8b": [(8192, 4096, 21504), (8192, 21504, 4096)], "12b": [(8192, 4608, 12288), (8192, 12288, 4608)],
            "ue5m3_sweep": [(8192, 4096, 4096)]}
    assert sorted(WORKLOADS) == sorted(want)
    for name, lins in want.items():
        got = [(l.tokens, l.k_in, l.n_out) for l in WORKLOADS[name].linears]
        assert got == lins, name
        # every dimension a multiple of 128 (tensor-core tiles, the one-read quantizer)
        assert all(d % 128 == 0 for l in lins for d in l)
    assert WORKLOADS["ue5m3_sweep"].targets == (448.0, 2048.0) and WORKLOADS["ue5m3_sweep"].steps == 100
    assert WORKLOADS["12b"].rht_seed == 1 and WORKLOADS["8b"].mx_side_by_side


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
                        np.array([0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 65504.0], np.float32)])
    x = x.astype(np.float32)
    want = torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f32_to_bf16_bits(x), want)
    assert np.array_equal(bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16)).view(torch.bfloat16)
                          .float().numpy())


def test_tiny_inputs_follow_the_recipe():
    inp = linear_inputs(WORKLOADS["tiny"], 0)
    x = bf16_bits_to_f32(inp["x"]).astype(np.float64)
    # N(0,1) with 0.1 % of the 65536 elements (66) multiplied by 50
    assert np.sum(np.abs(x) > 10) >= 50 and np.sum(np.abs(x) > 10) <= 66
    w = bf16_bits_to_f32(inp["w"]).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.001 and abs(w.mean()) < 0.001
    dy = np.abs(bf16_bits_to_f32(inp["dy"]).astype(np.float64))
    assert dy.min() >= 1e-6 * (1 - 2 ** -8) and dy.max() <= 1e-2 * (1 + 2 ** -8)
    # log-uniform: log10 |dy| uniform on [-6, -2]
    l = np.log10(dy)
    assert abs(l.mean() + 4.0) < 0.05 and abs(l.std() - 4.0 / np.sqrt(12.0)) < 0.05


def test_large_workload_distributions():
    # the 1.2B up-projection's tensors: Student-t(4)/sqrt(2) activations (unit variance,
    # heavy tails), N(0, 0.02^2) weights, log-normal gradients (median 1e-4, sigma 2 in ln)
    inp = linear_inputs(WORKLOADS["1.2b"], 0)
    x = bf16_bits_to_f32(inp["x"][:1024]).astype(np.float64)
    assert abs(x.var() - 1.0) < 0.05
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert kurt > 4.0                         # a normal has 3; Student-t(4) has no finite 4th moment
    w = bf16_bits_to_f32(inp["w"][:512]).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.0005
    dy = bf16_bits_to_f32(inp["dy"][:512]).astype(np.float64)
    ln = np.log(np.abs(dy))
    assert abs(np.median(ln) - np.log(1e-4)) < 0.02 and abs(ln.std() - 2.0) < 0.02
    assert 0.49 < np.mean(dy > 0) < 0.51      # random signs
    x12 = bf16_bits_to_f32(linear_inputs(WORKLOADS["12b"], 0)["x"][:256]).astype(np.float64)
    assert abs(x12.std() - 1.0) < 0.01        # 12B activations: N(0, 1)


def test_seeding_is_deterministic_and_distinct():
    a = linear_inputs(WORKLOADS["tiny"], 0)
    b = linear_inputs(WORKLOADS["tiny"], 0)
    assert all(np.array_equal(a[k], b[k]) for k in a)
    c = linear_inputs(WORKLOADS["1.2b"], 1)
    d = linear_inputs(WORKLOADS["1.2b"], 0)
    assert not np.array_equal(c["x"][:8, :8], d["x"][:8, :8])
    assert np.array_equal(random_bf16(5, (4, 16)), random_bf16(5, (4, 16)))


def test_sweep_ramp_endpoints():
    base = f32_to_bf16_bits(np.array([[1.0, -2.0, 3.0e-4, 1.0e-30]], np.float32))
    s0 = bf16_bits_to_f32(sweep_dy(base, 0)).astype(np.float64)
    s99 = bf16_bits_to_f32(sweep_dy(base, 99)).astype(np.float64)
    b = bf16_bits_to_f32(base).astype(np.float64)
    assert np.allclose(s0, b * 1e-3, rtol=2 ** -7) and np.allclose(s99, b * 1e3, rtol=2 ** -7)
    # monotone log-uniform growth: x10^(6/99) per step
    r = bf16_bits_to_f32(sweep_dy(base, 50))[0, 0] / bf16_bits_to_f32(sweep_dy(base, 49))[0, 0]
    assert abs(np.log10(r) - 6.0 / 99.0) < 0.01
