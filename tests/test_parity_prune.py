"""A1/A2 on the GPU against the CPU oracle, as two calls and as the one-call
A1 + A2: kept values and metadata must be bit-exact.  Small and ragged
shapes in full; the block shapes of the measured workloads in full where the
oracle is quick, sampled (rows for A1, column slabs for A2) at the largest
sizes."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import bits_of, ensure_built, to_dev, u8_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def gpu_prune(S, W_bits):
    import torch

    rows, cols = W_bits.shape
    W = to_dev(W_bits)
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(rows, cols // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(W, vals, meta)
    return vals, meta


def gpu_double(S, vals, meta, rows, cols):
    import torch

    tv = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    tm = torch.empty(cols, rows // 8, dtype=torch.uint8, device="cuda")
    S.slope_double_prune(vals, meta, rows, cols, tv, tm)
    return tv, tm


def gpu_fused(S, W_bits):
    import torch

    rows, cols = W_bits.shape
    W = to_dev(W_bits)
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(rows, cols // 8, dtype=torch.uint8, device="cuda")
    tv = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    tm = torch.empty(cols, rows // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_and_double_prune(W, vals, meta, tv, tm)
    return vals, meta, tv, tm


def check_fused(S, W, ov, om, otv, otm):
    """The one-call A1 + A2 writes the oracle's four outputs bit for bit."""
    vals, meta, tv, tm = gpu_fused(S, W)
    np.testing.assert_array_equal(bits_of(vals), ov)
    np.testing.assert_array_equal(meta.cpu().numpy(), om)
    np.testing.assert_array_equal(bits_of(tv), otv)
    np.testing.assert_array_equal(tm.cpu().numpy(), otm)


# cols % 128 == 0 takes the shared-memory staged A2 kernel (32-, 64- or
# 128-column tiles by size), other widths the direct one; 520 and 2312 rows
# leave a ragged 256-row tile.
SHAPES = [(8, 16), (1, 8), (40, 48), (264, 144), (256, 256), (1000, 1040), (1024, 1024),
          (4096, 1024), (1024, 4096), (520, 384), (2312, 2048)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_prune_and_double_prune_bit_exact(S, rows, cols):
    W = synth.normal_bf16(0, rows * 7 + cols, "W", (rows, cols))
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


def tie_heavy(rows, cols, seed):
    rng = np.random.default_rng(seed)
    alphabet = synth.to_bf16_bits(np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0], np.float32))
    return rng.choice(alphabet, size=(rows, cols)).astype(np.uint16)


@pytest.mark.parametrize("case", ["ties", "zeros", "specials", "exhaustive"])
def test_edge_values_bit_exact(S, case):
    import itertools

    if case == "ties":
        W = tie_heavy(512, 512, 1)
    elif case == "zeros":
        W = np.zeros((64, 128), np.uint16)
        W[::2, ::3] = 0x8000  # negative zeros among the zeros
    elif case == "specials":  # NaN > Inf > finite by the integer key
        W = tie_heavy(128, 256, 2)
        W[::5, ::7] = 0x7FC0
        W[1::5, ::3] = 0xFF80
        W[2::7, 1::4] = 0x0001  # smallest subnormal
    else:  # every 4-tuple of a 6-symbol alphabet, two groups per row
        alph = synth.to_bf16_bits(np.array([0.0, -0.0, 0.5, -0.5, 2.0, -2.0], np.float32))
        tup = np.array(list(itertools.product(alph, repeat=4)), dtype=np.uint16)  # 1296 groups
        W = tup.reshape(-1, 8)  # 648 x 8
        W = np.concatenate([W, W[:8]], axis=0)  # 656 rows: a multiple of 8 for A2
    rows, cols = W.shape
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


def test_double_prune_of_arbitrary_compressed_input(S):
    """A2 must accept any compressed input, including metadata that points at
    zeros and kept values that are -0."""
    rows, cols = 64, 96
    rng = np.random.default_rng(9)
    codes = np.array(sorted(O.LEGAL_NIBBLES), dtype=np.uint8)
    nib = rng.choice(codes, size=(rows, cols // 4))
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    vals = tie_heavy(rows, cols // 2, 3)
    tv, tm = gpu_double(S, to_dev(vals), u8_to_dev(meta), rows, cols)
    otv, otm, _ = O.double_prune24(vals, meta, rows, cols)
    np.testing.assert_array_equal(bits_of(tv), otv)
    np.testing.assert_array_equal(tm.cpu().numpy(), otm)


def oracle_double_prune_columns(W, cols_sel):
    """Oracle rows of D = P(Wsᵀ) for the given input columns, from the 8-column
    slabs that contain them (each row of D needs one column of Ws in full)."""
    out = {}
    for slab in sorted({c // 8 for c in cols_sel}):
        Wsl = np.ascontiguousarray(W[:, 8 * slab : 8 * slab + 8])
        v, m, _ = O.prune24(Wsl)
        tv, tm, _ = O.double_prune24(v, m, W.shape[0], 8)
        for c in range(8):
            out[8 * slab + c] = (tv[c], tm[c])
    return out


@pytest.mark.parametrize("rows,cols", [(10240, 2560), (2560, 10240), (28672, 7168), (7168, 28672)])
def test_block_shapes_sampled(S, rows, cols):
    """Full-size weights of the measured blocks, pruned on the GPU exactly as
    the benchmark does; the oracle checks sampled rows (A1) and sampled rows
    of the transposed result (A2)."""
    import torch

    W = synth.normal_bf16(0, 4, "W", (rows, cols))
    vals, meta = gpu_prune(S, W)
    tv, tm = gpu_double(S, vals, meta, rows, cols)
    # the one-call A1 + A2 writes the same four arrays in full
    for a, b in zip(gpu_fused(S, W), (vals, meta, tv, tm)):
        assert torch.equal(a, b)
    rng = np.random.default_rng(rows + cols)
    rs = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 62, replace=False)]))
    ov, om, _ = O.prune24(W[rs])
    np.testing.assert_array_equal(bits_of(vals)[rs], ov)
    np.testing.assert_array_equal(meta.cpu().numpy()[rs], om)
    cs = np.unique(np.concatenate([[0, cols - 1], rng.choice(cols, 30, replace=False)]))
    ref = oracle_double_prune_columns(W, cs)
    tvb, tmb = bits_of(tv), tm.cpu().numpy()
    for c in cs:
        np.testing.assert_array_equal(tvb[c], ref[c][0])
        np.testing.assert_array_equal(tmb[c], ref[c][1])
