"""Seeded synthetic inputs for the sparse-plus-low-rank adapter linear layer.

This module only draws random numbers and rounds them to bf16; it holds none
of the layer's arithmetic, so both the CUDA path's tests and the CPU oracle
can take their inputs from it.

Value distributions follow the OPT-style layer shapes the library is
measured on: activations and upstream gradients ~ N(0, 1), weights and
adapter factors ~ N(0, 0.02).  Every tensor has its own stream:
``SeedSequence(seed, spawn_key=(layer, tensor))``, so any tensor can be
regenerated alone and in any order.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Tensor names, in a fixed order: their position is the stream's spawn key.
TENSORS = ("X", "W", "L", "R", "dY")
SIGMA = {"X": 1.0, "dY": 1.0, "W": 0.02, "L": 0.02, "R": 0.02}


@dataclass(frozen=True)
class Linear:
    name: str
    inp: int  # in features  (reduction dim of the forward)
    out: int  # out features


@dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    rank: int
    linears: tuple = field(default_factory=tuple)
    forward_only: bool = False
    seed: int = 0


def opt_block(d: int, ffn: int) -> tuple:
    """The six linears of one OPT decoder block: Q, K, V, O, FC1, FC2."""
    return (
        Linear("q", d, d),
        Linear("k", d, d),
        Linear("v", d, d),
        Linear("o", d, d),
        Linear("fc1", d, ffn),
        Linear("fc2", ffn, d),
    )


WORKLOADS = {
    "single-256": Workload("single-256", 64, 8, (Linear("w", 256, 256),)),
    "opt-350m-block": Workload("opt-350m-block", 4096, 16, opt_block(1024, 4096)),
    "opt-2.7b-block": Workload("opt-2.7b-block", 8192, 32, opt_block(2560, 10240)),
    "opt-33b-block-r0": Workload("opt-33b-block-r0", 16384, 0, opt_block(7168, 28672)),
    "opt-33b-block-r64": Workload("opt-33b-block-r64", 16384, 64, opt_block(7168, 28672)),
    "opt-66b-infer-t1": Workload("opt-66b-infer-t1", 1, 64, opt_block(9216, 36864), True),
    "opt-66b-infer-t16": Workload("opt-66b-infer-t16", 16, 64, opt_block(9216, 36864), True),
    "opt-66b-infer-t128": Workload("opt-66b-infer-t128", 128, 64, opt_block(9216, 36864), True),
    "opt-66b-infer-t2048": Workload("opt-66b-infer-t2048", 2048, 64, opt_block(9216, 36864), True),
}


def _rng(seed: int, layer: int, tensor: str) -> np.random.Generator:
    ss = np.random.SeedSequence(seed, spawn_key=(layer, TENSORS.index(tensor)))
    return np.random.default_rng(ss)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (torch's cast)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def normal_bf16(seed: int, layer: int, tensor: str, shape, sigma: float | None = None) -> np.ndarray:
    """bf16 bit patterns of N(0, sigma^2) draws from the tensor's own stream."""
    s = SIGMA[tensor] if sigma is None else sigma
    x = _rng(seed, layer, tensor).standard_normal(size=shape, dtype=np.float32) * np.float32(s)
    return to_bf16_bits(x)


def layer_inputs(seed: int, layer: int, tokens: int, inp: int, out: int, rank: int, rows=None):
    """All inputs of one linear, as bf16 bit patterns.

    W is out x in, X is T x in, dY is T x out, L is in x r and R is r x out
    (None when r == 0).  ``rows`` (a slice of token rows) keeps X and dY to a
    sample of the full draw; the draw itself is the same.
    """
    X = normal_bf16(seed, layer, "X", (tokens, inp))
    dY = normal_bf16(seed, layer, "dY", (tokens, out))
    W = normal_bf16(seed, layer, "W", (out, inp))
    L = R = None
    if rank:
        L = normal_bf16(seed, layer, "L", (inp, rank))
        R = normal_bf16(seed, layer, "R", (rank, out))
    if rows is not None:
        X, dY = X[rows], dY[rows]
    return {"X": X, "W": W, "L": L, "R": R, "dY": dY}


def device_normal_bf16(shape, sigma: float, seed: int, device="cuda"):
    """Seeded N(0, sigma^2) bf16 tensor drawn directly on the device (benchmark inputs)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * sigma).to(torch.bfloat16)
