"""Seeded synthetic inputs for the FP4 block-scaled quantized linear layer.

This module is shared by the tests, the oracle checks and the benchmark. It
holds none of the method's arithmetic: it only draws random BF16 tensors with
the shapes and value distributions of the linears the pages train (see the
workload table below) and describes each workload's recipe knobs.

The pages' workloads are model trainings on private multi-trillion-token data
("Pretraining Large Language Models with NVFP4", section A4, experimental
setup); these tensors stand in for the linear layers of those models, with the
published hidden / FFN widths and sequence length 8192.

Every tensor is drawn with numpy's PCG64 generator, seeded per workload c and
tensor: X -> 1000c + 0, W -> 1000c + 1, dY -> 1000c + 2 (the down projection
of a two-linear workload adds 10). Values are rounded once to BF16
(round-to-nearest-even) and the same bytes go to the oracle and to the GPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (nearest-even) and return the uint16 patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- distributions
def _normal(rng, shape, std):
    return rng.standard_normal(shape, dtype=np.float32) * np.float32(std)


def _student_t_unit(rng, shape):
    # Student-t with 4 degrees of freedom has variance 2; scale to unit variance.
    return (rng.standard_t(4.0, size=shape) / np.sqrt(2.0)).astype(np.float32)


def _log_uniform_signed(rng, shape, lo_exp, hi_exp):
    mag = np.power(10.0, rng.uniform(lo_exp, hi_exp, size=shape))
    sign = np.where(rng.integers(0, 2, size=shape) == 1, -1.0, 1.0)
    return (sign * mag).astype(np.float32)


def _log_normal_signed(rng, shape, median, sigma):
    mag = np.exp(rng.normal(np.log(median), sigma, size=shape))
    sign = np.where(rng.integers(0, 2, size=shape) == 1, -1.0, 1.0)
    return (sign * mag).astype(np.float32)


def _with_outliers(rng, x, frac, factor):
    n = x.size
    k = int(round(n * frac))
    idx = rng.choice(n, size=k, replace=False)
    flat = x.reshape(-1)
    flat[idx] *= np.float32(factor)
    return x


# --------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Linear:
    tokens: int
    k_in: int
    n_out: int


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: its linears and the recipe knobs that go with it."""
    index: int
    name: str
    linears: tuple
    x_dist: str
    dy_dist: str
    scale_fmt: str = "nvfp4"       # "nvfp4" (E4M3 scales) or "ue5m3"
    rht_seed: int = 0
    sr_seed: int = 0
    rht: bool = True
    held: bool = False
    targets: tuple = (448.0,)
    steps: int = 1
    mx_side_by_side: bool = False
    notes: str = ""
    extra: dict = field(default_factory=dict)

    def gemm_flops_per_step(self) -> float:
        return sum(3 * 2.0 * l.tokens * l.k_in * l.n_out for l in self.linears)


WORKLOADS = {
    "tiny": Workload(1, "tiny 256x256 NVFP4 linear", (Linear(256, 256, 256),),
                     x_dist="normal_outliers", dy_dist="log_uniform_1e-6_1e-2",
                     rht_seed=0, sr_seed=0),
    "1.2b": Workload(2, "1.2B Transformer FFN linears (T=8192, 2048->6144->2048)",
                     (Linear(8192, 2048, 6144), Linear(8192, 6144, 2048)),
                     x_dist="student_t4", dy_dist="log_normal_1e-4_2", rht_seed=0, sr_seed=0),
    "8b": Workload(3, "8B hybrid FFN linears (T=8192, 4096->21504->4096)",
                   (Linear(8192, 4096, 21504), Linear(8192, 21504, 4096)),
                   x_dist="student_t4", dy_dist="log_normal_1e-4_2", rht_seed=0, sr_seed=0,
                   mx_side_by_side=True),
    "12b": Workload(4, "12B hybrid FFN linears (T=8192, 4608->12288->4608)",
                    (Linear(8192, 4608, 12288), Linear(8192, 12288, 4608)),
                    x_dist="normal", dy_dist="log_normal_1e-4_2", rht_seed=1, sr_seed=1),
    "ue5m3_sweep": Workload(5, "UE5M3 periodic-scaling sweep (T=8192, 4096->4096, 100 steps)",
                            (Linear(8192, 4096, 4096),), x_dist="student_t4",
                            dy_dist="log_normal_1e-4_2", scale_fmt="ue5m3", rht=False,
                            held=True, targets=(448.0, 2048.0), steps=100),
}


def _draw(kind: str, rng, shape):
    if kind == "normal":
        return _normal(rng, shape, 1.0)
    if kind == "normal_outliers":
        return _with_outliers(rng, _normal(rng, shape, 1.0), 0.001, 50.0)
    if kind == "student_t4":
        return _student_t_unit(rng, shape)
    if kind == "weight":
        return _normal(rng, shape, 0.02)
    if kind == "log_uniform_1e-6_1e-2":
        return _log_uniform_signed(rng, shape, -6.0, -2.0)
    if kind == "log_normal_1e-4_2":
        return _log_normal_signed(rng, shape, 1e-4, 2.0)
    raise ValueError(kind)


def linear_inputs(w: Workload, which: int = 0) -> dict:
    """BF16 bit arrays X [T x K], W [N x K], dY [T x N] for linear `which` of `w`."""
    lin = w.linears[which]
    base = 1000 * w.index + 10 * which
    x = f32_to_bf16_bits(_draw(w.x_dist, np.random.Generator(np.random.PCG64(base + 0)),
                               (lin.tokens, lin.k_in)))
    wt = f32_to_bf16_bits(_draw("weight", np.random.Generator(np.random.PCG64(base + 1)),
                                (lin.n_out, lin.k_in)))
    dy = f32_to_bf16_bits(_draw(w.dy_dist, np.random.Generator(np.random.PCG64(base + 2)),
                                (lin.tokens, lin.n_out)))
    return {"x": x, "w": wt, "dy": dy}


def sweep_dy(base_dy_bits: np.ndarray, step: int, steps: int = 100) -> np.ndarray:
    """Gradient of sweep step s: the base gradient times 10^(-3 + 6 s / (steps-1)),
    a monotone log-uniform drift over x10^-3 .. x10^3, rounded to BF16."""
    factor = 10.0 ** (-3.0 + 6.0 * step / (steps - 1))
    return f32_to_bf16_bits(bf16_bits_to_f32(base_dy_bits) * np.float32(factor))


def random_bf16(rng_seed: int, shape, kind: str = "normal") -> np.ndarray:
    """A small seeded BF16 tensor for unit and edge-case tests."""
    return f32_to_bf16_bits(_draw(kind, np.random.Generator(np.random.PCG64(rng_seed)), shape))
