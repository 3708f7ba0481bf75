"""Seeded synthetic inputs and workload shapes for the blockwise-FP8 linear layer.

Shared by the tests and the benchmark. This module holds none of the method's
arithmetic: it only draws float32 samples with numpy's PCG64 generator and
rounds them to bfloat16 (returned as uint16 bit patterns), and it lists the
layer shapes of the Puro-2B workloads.

Shapes. The Puro-2B model is a 28-layer Transformer with hidden size 2048 and
a 4096-token context, in a Qwen3-1.7B-compatible configuration (ainews.surl.tw,
"Puro-2B Publishes a Consumer-Grade GPU Pretraining Recipe ..."). The pages do
not print the projection widths; a Qwen3-1.7B-compatible layout gives a fused
QKV projection 2048 -> 4096 (16 query heads and 2 x 8 key/value heads of width
128), an output projection 2048 -> 2048, a fused gate/up projection
2048 -> 12288 (intermediate 6144) and a down projection 6144 -> 2048.

Distributions: activations N(0,1) (or Student-t with 3 degrees of freedom for
the MLP workload, or N(0,1) with 8 outlier channels scaled x50 for the full
stack), weights N(0, 0.02^2), output gradients N(0,1). Seeds: X = seed,
W = seed + 1, dY = seed + 2; in the full stack every (layer, linear) pair j
shifts the seed by 3 * j.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import ml_dtypes
import numpy as np

HIDDEN = 2048
LAYERS = 28
SEQ = 4096
QKV_OUT = 4096
MLP_INTER = 6144


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 (round to nearest-even, by ml_dtypes) as uint16 bit patterns."""
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32).astype(ml_dtypes.bfloat16)).view(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 values (for building test inputs only)."""
    return np.asarray(b, dtype=np.uint16).view(ml_dtypes.bfloat16).astype(np.float32)


@dataclass(frozen=True)
class Linear:
    """One linear layer y = x W^T with x [M, K], W [N, K], dy [M, N]."""
    name: str
    M: int
    K: int
    N: int
    x_dist: str = "normal"      # "normal" | "student_t3" | "outliers"
    seed: int = 0

    @property
    def flops(self) -> int:
        """fwd + dgrad + wgrad, 2*M*N*K each."""
        return 3 * 2 * self.M * self.N * self.K


@dataclass(frozen=True)
class Workload:
    name: str
    linears: tuple = field(default_factory=tuple)
    passes: tuple = ("fwd", "dgrad", "wgrad")

    @property
    def flops(self) -> int:
        per = {"fwd": 1, "dgrad": 1, "wgrad": 1}
        return sum(sum(per[p] for p in self.passes) * 2 * l.M * l.N * l.K for l in self.linears)


def single_linear_256() -> Workload:
    """One linear, forward only: X [256, 256] ~ N(0,1), W [256, 256] ~ N(0, 0.02^2), seed 0."""
    return Workload("single-linear-256-fwd", (Linear("linear", 256, 256, 256, "normal", 0),), ("fwd",))


def attention_projections() -> Workload:
    """Puro-2B attention projections at M = 4096 tokens (one 4096-token sequence)."""
    return Workload("puro2b-attn-proj-M4096", (
        Linear("qkv", SEQ, HIDDEN, QKV_OUT, "normal", 0),
        Linear("o", SEQ, HIDDEN, HIDDEN, "normal", 0),
    ))


def mlp_projections() -> Workload:
    """Puro-2B MLP at M = 8192 tokens: gate/up 2048 -> 12288 and down 6144 -> 2048, Student-t(3) inputs."""
    return Workload("puro2b-mlp-M8192", (
        Linear("gate_up", 2 * SEQ, HIDDEN, 2 * MLP_INTER, "student_t3", 0),
        Linear("down", 2 * SEQ, MLP_INTER, HIDDEN, "student_t3", 0),
    ))


def full_stack(layers: int = LAYERS, M: int = 4 * SEQ) -> Workload:
    """All 28 layers' linears (QKV, O, gate/up, down) at M = 16384 tokens, outlier-channel inputs."""
    lins = []
    for layer in range(layers):
        for j, (nm, K, N) in enumerate((("qkv", HIDDEN, QKV_OUT), ("o", HIDDEN, HIDDEN),
                                        ("gate_up", HIDDEN, 2 * MLP_INTER), ("down", MLP_INTER, HIDDEN))):
            lins.append(Linear(f"L{layer}.{nm}", M, K, N, "outliers", 3 * (4 * layer + j)))
    return Workload(f"puro2b-{layers}layer-stack-M{M}", tuple(lins))


def shape_sweep() -> list:
    """M in {1000, 2048, 4000, 8192, 32768} x (K, N) in the four Puro-2B projection shapes."""
    out = []
    for M in (1000, 2048, 4000, 8192, 32768):
        for K, N in ((2048, 4096), (2048, 2048), (2048, 12288), (6144, 2048)):
            out.append(Linear(f"sweep-M{M}-K{K}-N{N}", M, K, N, "normal", 0))
    return out


def _x_samples(rng: np.random.Generator, M: int, K: int, dist: str) -> np.ndarray:
    if dist == "normal":
        return rng.standard_normal((M, K), dtype=np.float32)
    if dist == "student_t3":
        return rng.standard_t(3, size=(M, K)).astype(np.float32)
    if dist == "outliers":
        x = rng.standard_normal((M, K), dtype=np.float32)
        ch = rng.choice(K, 8, replace=False)
        x[:, ch] *= 50.0
        return x
    raise ValueError(dist)


def make_x(lin: Linear) -> np.ndarray:
    return bf16_bits(_x_samples(np.random.default_rng(lin.seed), lin.M, lin.K, lin.x_dist))


def make_w(lin: Linear) -> np.ndarray:
    rng = np.random.default_rng(lin.seed + 1)
    return bf16_bits(rng.standard_normal((lin.N, lin.K), dtype=np.float32) * np.float32(0.02))


def make_dy(lin: Linear) -> np.ndarray:
    rng = np.random.default_rng(lin.seed + 2)
    return bf16_bits(rng.standard_normal((lin.M, lin.N), dtype=np.float32))


def make_linear(lin: Linear):
    """(X bits [M,K], W bits [N,K], dY bits [M,N]) for one linear layer."""
    return make_x(lin), make_w(lin), make_dy(lin)


def random_bits(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """Plain N(0, std^2) bf16 bits of any shape (for edge-case tests)."""
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def random_codes(shape, seed: int) -> np.ndarray:
    """Uniformly random finite E4M3FN codes (NaN patterns 0x7F/0xFF excluded)."""
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    nan = (c & 0x7F) == 0x7F
    c[nan] = c[nan] - 1
    return c


def random_scales(shape, seed: int) -> np.ndarray:
    """Positive FP32 scales spread over a few decades."""
    rng = np.random.default_rng(seed)
    return (np.float32(2.0) ** rng.uniform(-12, 2, size=shape).astype(np.float32)).astype(np.float32)
