"""Optimizer-side calls on the GPU against the CPU oracle.

slope_recompress_double_prune: an updated weight re-compressed at the kept
row mask and double-pruned again; values and metadata bit-exact.
slope_double_prune_frozen / slope_recompress_frozen: the second pruning
with its column mask kept (and, for the latter, the row mask too); values
bit-exact.
slope_sparse_axpby: beta·A + gamma·B on compressed values, every
combination of fp32 and bf16 arrays, within the rounding the call states
(fp32 arithmetic, then one rounding to the output type)."""

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


def gpu_recompress(S, W_bits, meta):
    import torch

    rows, cols = W_bits.shape
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    tv = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    tm = torch.empty(cols, rows // 8, dtype=torch.uint8, device="cuda")
    S.slope_recompress_double_prune(to_dev(W_bits), u8_to_dev(meta), vals, tv, tm)
    return bits_of(vals), bits_of(tv), tm.cpu().numpy()


# cols % 128 == 0 takes the one-pass kernel (128-, 64- or 32-column tiles by
# size), other widths the gather and the separate second pruning; 520 and
# 2312 rows leave a ragged 256-row tile
SHAPES = [(8, 16), (40, 48), (264, 144), (256, 256), (1000, 1040), (1024, 1024), (4096, 1024),
          (1024, 4096), (520, 384), (2312, 2048)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_recompress_updated_weight_bit_exact(S, rows, cols):
    W0 = synth.normal_bf16(0, rows + 3 * cols, "W", (rows, cols))
    _, meta, _ = O.prune24(W0)  # the mask kept from initialisation
    W1 = synth.normal_bf16(1, rows + 3 * cols, "W", (rows, cols))  # the updated weight
    v, tv, tm = gpu_recompress(S, W1, meta)
    ov, otv, otm = O.recompress_double_prune24(W1, meta)
    np.testing.assert_array_equal(v, ov)
    np.testing.assert_array_equal(tv, otv)
    np.testing.assert_array_equal(tm, otm)


def test_recompress_edge_values_and_any_legal_mask(S):
    """Tie-heavy and special values (signed zeros, NaN, Inf) under a random
    legal mask that no selection produced."""
    rng = np.random.default_rng(12)
    rows, cols = 512, 256
    alphabet = synth.to_bf16_bits(np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0], np.float32))
    W = rng.choice(alphabet, size=(rows, cols)).astype(np.uint16)
    W[::5, ::7] = 0x7FC0
    W[1::5, ::3] = 0xFF80
    codes = np.array(sorted(O.LEGAL_NIBBLES), dtype=np.uint8)
    nib = rng.choice(codes, size=(rows, cols // 4))
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    v, tv, tm = gpu_recompress(S, W, meta)
    ov, otv, otm = O.recompress_double_prune24(W, meta)
    np.testing.assert_array_equal(v, ov)
    np.testing.assert_array_equal(tv, otv)
    np.testing.assert_array_equal(tm, otm)


@pytest.mark.parametrize("rows,cols", [(10240, 2560), (28672, 7168)])
def test_recompress_block_shapes(S, rows, cols):
    """Full-size weights: at the weight's own mask the call reproduces
    prune + double prune in full; for an updated weight the oracle checks
    sampled rows of the values and sampled rows of the transposed result."""
    import torch

    W = synth.normal_bf16(0, 4, "W", (rows, cols))
    Wd = to_dev(W)
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(rows, cols // 8, dtype=torch.uint8, device="cuda")
    tv = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    tm = torch.empty(cols, rows // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(Wd, vals, meta)
    S.slope_double_prune(vals, meta, rows, cols, tv, tm)
    v2, tv2, tm2 = torch.empty_like(vals), torch.empty_like(tv), torch.empty_like(tm)
    S.slope_recompress_double_prune(Wd, meta, v2, tv2, tm2)
    for a, b in ((v2, vals), (tv2, tv), (tm2, tm)):
        assert torch.equal(a, b)
    W1 = synth.normal_bf16(1, 4, "W", (rows, cols))
    S.slope_recompress_double_prune(to_dev(W1), meta, v2, tv2, tm2)
    m_np = meta.cpu().numpy()
    rng = np.random.default_rng(rows)
    rs = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 62, replace=False)]))
    np.testing.assert_array_equal(bits_of(v2)[rs], O.recompress24(W1[rs], m_np[rs]))
    cs = np.unique(np.concatenate([[0, cols - 1], rng.choice(cols, 30, replace=False)]))
    tvb, tmb = bits_of(tv2), tm2.cpu().numpy()
    for slab in sorted({int(c) // 8 for c in cs}):
        sl = slice(8 * slab, 8 * slab + 8)
        _, otv, otm = O.recompress_double_prune24(np.ascontiguousarray(W1[:, sl]), np.ascontiguousarray(m_np[:, slab:slab + 1]))
        for c in range(8):
            if 8 * slab + c in set(cs.tolist()):
                np.testing.assert_array_equal(tvb[8 * slab + c], otv[c])
                np.testing.assert_array_equal(tmb[8 * slab + c], otm[c])


@pytest.mark.parametrize("a_dt,b_dt,o_dt", [(a, b, o) for a in ("f32", "bf16") for b in ("f32", "bf16")
                                            for o in ("f32", "bf16")])
def test_sparse_axpby_matches_oracle(S, a_dt, b_dt, o_dt):
    import torch

    dt = {"f32": torch.float32, "bf16": torch.bfloat16}
    rows, cols = 384, 1024
    _, meta, _ = O.prune24(synth.normal_bf16(0, 40, "W", (rows, cols)))
    g = torch.Generator().manual_seed(3)
    A = torch.randn(rows, cols // 2, generator=g).to(dt[a_dt])
    B = (torch.randn(rows, cols // 2, generator=g) * 1e-3).to(dt[b_dt])
    beta, gamma = 0.9999, -0.01  # a decayed weight plus a scaled step
    out = torch.empty(rows, cols // 2, dtype=dt[o_dt], device="cuda")
    S.slope_sparse_axpby(beta, A.cuda(), gamma, B.cuda(), out)
    torch.cuda.synchronize()
    ref = O.sparse_axpby24(beta, A.double().numpy(), gamma, B.double().numpy(), meta)
    got = out.double().cpu().numpy()
    scale = np.abs(beta * A.double().numpy()) + np.abs(gamma * B.double().numpy())
    # fp32 arithmetic: two roundings of at most 2^-24 of the magnitudes; a
    # bf16 output adds one rounding of 2^-9 of the result
    bound = 2.0 ** -22 * scale + (2.0 ** -8 * np.abs(ref) if o_dt == "bf16" else 0.0)
    assert (np.abs(got - ref) <= bound + 1e-30).all()


def test_sparse_axpby_in_place(S):
    import torch

    A = torch.randn(4096, device="cuda")
    B = torch.randn(4096, device="cuda")
    ref = 0.5 * A + 2.0 * B
    S.slope_sparse_axpby(0.5, A, 2.0, B, A)  # out is A
    torch.testing.assert_close(A, ref, rtol=2e-7, atol=1e-7)


def random_legal_meta(rng, rows, cols):
    codes = np.array(sorted(O.LEGAL_NIBBLES), dtype=np.uint8)
    nib = rng.choice(codes, size=(rows, cols // 4))
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_frozen_column_mask_bit_exact(S, rows, cols):
    """An updated weight under both kept masks (the row mask from A1 of the
    old weight, a column mask drawn at random among legal ones): the
    frozen second pruning of its compressed form, and the one-pass form
    from W, both against the oracle."""
    import torch

    rng = np.random.default_rng(rows * 3 + cols)
    W0 = synth.normal_bf16(0, rows + 5 * cols, "W", (rows, cols))
    _, meta, _ = O.prune24(W0)
    t_meta = random_legal_meta(rng, cols, rows)
    W1 = synth.normal_bf16(1, rows + 5 * cols, "W", (rows, cols))
    ov, otv = O.recompress_frozen24(W1, meta, t_meta)
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    tv = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    S.slope_recompress_frozen(to_dev(W1), u8_to_dev(meta), u8_to_dev(t_meta), vals, tv)
    np.testing.assert_array_equal(bits_of(vals), ov)
    np.testing.assert_array_equal(bits_of(tv), otv)
    tv2 = torch.empty_like(tv)
    S.slope_double_prune_frozen(to_dev(ov), u8_to_dev(meta), rows, cols, u8_to_dev(t_meta), tv2)
    np.testing.assert_array_equal(bits_of(tv2), otv)


@pytest.mark.parametrize("rows,cols", [(10240, 2560), (28672, 7168)])
def test_frozen_at_own_masks_block_shapes(S, rows, cols):
    """Full-size weights: frozen at the masks A1 and A2 chose, both forms
    reproduce the selecting calls' values in full."""
    import torch

    W = to_dev(synth.normal_bf16(0, 4, "W", (rows, cols)))
    vals = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(rows, cols // 8, dtype=torch.uint8, device="cuda")
    tv = torch.empty(cols, rows // 2, dtype=torch.bfloat16, device="cuda")
    tm = torch.empty(cols, rows // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_and_double_prune(W, vals, meta, tv, tm)
    v2, tv2, tv3 = torch.empty_like(vals), torch.empty_like(tv), torch.empty_like(tv)
    S.slope_recompress_frozen(W, meta, tm, v2, tv2)
    S.slope_double_prune_frozen(vals, meta, rows, cols, tm, tv3)
    assert torch.equal(v2, vals) and torch.equal(tv2, tv) and torch.equal(tv3, tv)
