"""A1 and A2 on seeded random shapes and values, bit-exact against the oracle.

Shapes: rows 1 to 2048 (multiples of 8 run A2 too, others A1 alone),
columns multiples of 16 up to 2048, about half of them multiples of 128 (the
staged A2 kernels) and the rest not (the direct ones).  Values: Gaussian
weights, a tie-heavy alphabet (±0, ±0.5, ±1, ±2), or Gaussian weights with
NaN, ±Inf, the smallest subnormal and -0 planted.  Patterns: 2:4 (A1, A2 and
the one-call A1 + A2), 1:2 and 2:8 (A1, A2, and the 2:4 form of 2:8)."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import bits_of, ensure_built
from tests.test_parity_patterns import check_patterns
from tests.test_parity_prune import check_fused, gpu_double, gpu_prune

pytestmark = pytest.mark.gpu


def _values(kind, rows, cols, seed):
    rng = np.random.default_rng(seed)
    if kind == "ties":
        alphabet = synth.to_bf16_bits(np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0], np.float32))
        return rng.choice(alphabet, size=(rows, cols)).astype(np.uint16)
    W = synth.to_bf16_bits((rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)).astype(np.uint16)
    if kind == "specials":
        for bits, frac in ((0x7FC0, 0.01), (0x7F80, 0.01), (0xFF80, 0.01), (0x0001, 0.01), (0x8000, 0.02)):
            W[rng.random((rows, cols)) < frac] = bits
    return np.ascontiguousarray(W)


def _cases(n=48, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        rows = int(rng.integers(1, 257)) * 8 if rng.random() < 0.85 else int(rng.integers(1, 2048))
        cols = 128 * int(rng.integers(1, 17)) if rng.random() < 0.5 else 16 * int(rng.integers(1, 129))
        kind = str(rng.choice(["gauss", "ties", "specials"]))
        pattern = str(rng.choice(["2:4", "2:4", "2:4", "1:2", "2:8"]))
        out.append((i, rows, cols, kind, pattern))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


@pytest.mark.parametrize("i,rows,cols,kind,pattern", CASES,
                         ids=[f"{c[4]}-{c[1]}x{c[2]}-{c[3]}" for c in CASES])
def test_random_prune_bit_exact(S, i, rows, cols, kind, pattern):
    import torch

    W = _values(kind, rows, cols, 1000 + i)
    if pattern != "2:4":
        n, m = (int(x) for x in pattern.split(":"))
        check_patterns(S, W, n, m)
        return
    vals, meta = gpu_prune(S, W)
    ov, om, _ = O.prune24(W)
    np.testing.assert_array_equal(bits_of(vals), ov)
    np.testing.assert_array_equal(meta.cpu().numpy(), om)
    if rows % 8 == 0 and cols % 16 == 0:
        tv, tm = gpu_double(S, vals, meta, rows, cols)
        otv, otm, _ = O.double_prune24(ov, om, rows, cols)
        np.testing.assert_array_equal(bits_of(tv), otv)
        np.testing.assert_array_equal(tm.cpu().numpy(), otm)
        check_fused(S, W, ov, om, otv, otm)
    torch.cuda.synchronize()
    S.slope_device_status()
