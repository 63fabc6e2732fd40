"""The optimizer-side calls on seeded random shapes and masks, bit-exact.

Each case draws a shape (rows multiples of 8 up to 2048; widths multiples of
16 up to 2048, about half of them multiples of 128, which take the one-pass
kernels), an updated weight (Gaussian, tie-heavy or with special values),
the kept row mask (A1 of an older weight, or any legal one) and a legal
column mask, and checks against the oracle: re-compression + A2
(`slope_recompress_double_prune`), re-compression at both kept masks
(`slope_recompress_frozen`) and the frozen second pruning of the compressed
values (`slope_double_prune_frozen`)."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import bits_of, ensure_built, to_dev, u8_to_dev
from tests.test_parity_optimizer import gpu_recompress, random_legal_meta
from tests.test_parity_prune_random import _values

pytestmark = pytest.mark.gpu


def _cases(n=32, seed=31):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        rows = 8 * int(rng.integers(1, 257))
        cols = 128 * int(rng.integers(1, 17)) if rng.random() < 0.5 else 16 * int(rng.integers(1, 129))
        kind = str(rng.choice(["gauss", "ties", "specials"]))
        row_mask = str(rng.choice(["a1", "legal"]))
        out.append((i, rows, cols, kind, row_mask))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


@pytest.mark.parametrize("i,rows,cols,kind,row_mask", CASES,
                         ids=[f"{c[1]}x{c[2]}-{c[3]}-{c[4]}" for c in CASES])
def test_random_optimizer_calls_bit_exact(S, i, rows, cols, kind, row_mask):
    import torch

    rng = np.random.default_rng(3000 + i)
    if row_mask == "a1":
        _, meta, _ = O.prune24(synth.normal_bf16(0, 3000 + i, "W", (rows, cols)))
    else:
        meta = random_legal_meta(rng, rows, cols)
    t_meta = random_legal_meta(rng, cols, rows)
    W1 = _values(kind, rows, cols, 4000 + i)  # the updated weight

    v, tv, tm = gpu_recompress(S, W1, meta)
    ov, otv, otm = O.recompress_double_prune24(W1, meta)
    np.testing.assert_array_equal(v, ov)
    np.testing.assert_array_equal(tv, otv)
    np.testing.assert_array_equal(tm, otm)

    fv, ftv = O.recompress_frozen24(W1, meta, t_meta)
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    tvals = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    S.slope_recompress_frozen(to_dev(W1), u8_to_dev(meta), u8_to_dev(t_meta), vals, tvals)
    np.testing.assert_array_equal(bits_of(vals), fv)
    np.testing.assert_array_equal(bits_of(tvals), ftv)
    tv2 = torch.empty_like(tvals)
    S.slope_double_prune_frozen(to_dev(fv), u8_to_dev(meta), rows, cols, u8_to_dev(t_meta), tv2)
    np.testing.assert_array_equal(bits_of(tv2), ftv)
    torch.cuda.synchronize()
    S.slope_device_status()
