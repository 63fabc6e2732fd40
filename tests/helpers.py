"""Shared test utilities: moving bf16 bit patterns between NumPy and CUDA
tensors, the float tolerance rule, and building the library once."""

import numpy as np

TOL = 2e-3  # max|gpu - oracle| <= TOL * max|oracle|, per tensor


def ensure_built():
    from sparse_rank_adapter_gb300 import build

    return build.build()


def to_dev(bits, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def u8_to_dev(a, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bits_of(t):
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close_rel(name, got, ref, tol=TOL):
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    scale = np.abs(r).max()
    err = np.abs(g - r).max()
    assert err <= tol * scale, f"{name}: max|gpu-oracle| = {err:.4e} > {tol}*max|oracle| = {tol * scale:.4e}"
    return err / scale if scale else 0.0


def hilo_bits(v):
    """bf16 hi/lo split of fp64 values as the library stores rank-r
    intermediates: [hi | lo] along the last axis, hi = bf16(v), lo = bf16(v - hi)."""
    from oracle import slope_oracle as O

    hi = O.f64_to_bf16(v)
    lo = O.f64_to_bf16(np.asarray(v, np.float64) - O.bf16_to_f64(hi))
    return np.concatenate([hi, lo], axis=-1)


def hilo_value(t):
    """fp64 value of a [hi | lo] bf16 device tensor."""
    a = t.double().cpu().numpy()
    r = a.shape[-1] // 2
    return a[..., :r] + a[..., r:]
