"""CPU oracle for the sparse-plus-low-rank adapter linear layer (SLoPe).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its binding) never imports, links or executes it, and this
module imports nothing from the product.

The source for every step is the page "SLoPe: Double-Pruned Sparse Plus Lazy
Low-Rank Adapter Pretraining of LLMs" (an AI summary of arXiv 2405.16325v3),
cited below by its section labels:

  * §1 and §2.1 "Double-pruned backward pass": the weight is N:M pruned; the
    transposed pruned matrix is N:M pruned again so the backward input
    gradient is also an N:M-sparse product.
  * §2.2 "Lazy low-rank adapters": the pruned matrix is augmented by a
    rank-r product X·L·R.
  * §2.3 "Sparse kernels" and App. K "Implementation details": compressed
    sparse formats for the weight and its transpose; the weight gradient is
    masked with the weight's own mask and stored without its zeros.
  * §T.1 "Lemma 2.1": the expected zeros added by the second pruning.
  * App. K again, for the optimizer side: updated weights copied into the
    compressed format (with the initialised mask kept, as §2.1's training
    policy does) and linear combinations of matrices sharing a pattern.

Where the page is silent the plainest reading is taken:

  * magnitude = |bf16 value| compared exactly, as the integer key
    ``bits & 0x7FFF`` (a total order; no float arithmetic decides a mask);
  * groups are aligned at column 0; ties go to the lower index;
  * kept positions are listed in ascending order; the 2:4 metadata nibble of a
    group is ``i0 | i1 << 2`` (i0 < i1) and two groups share a byte, the lower
    group in the low nibble;
  * the second pruning sees pruned-away positions as key 0, so a group with
    fewer than two non-zeros keeps its lowest-index remaining positions;
  * all products are dense fp64 matmuls of masked matrices built from the
    exact bf16 inputs; intermediates (X·L, dY·Rᵀ) stay in fp64.

Every function here is pinned by ``tests/test_oracle.py`` against brute
force, closed forms, identity inputs and finite differences.
"""

from __future__ import annotations

import itertools

import numpy as np

# ---------------------------------------------------------------------------
# bf16 encoding (inputs arrive as raw bf16 bit patterns, uint16)
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of each bf16 bit pattern, as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even), returning bit patterns.

    The value is first rounded to fp32 (the precision of a kernel's fp32
    accumulator), then the low 16 bits are rounded away with
    round-half-to-even on the integer encoding.  NaN stays NaN.
    """
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = np.isnan(f)
    out[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x0040)).astype(np.uint16)
    return out


def magnitude_key(bits: np.ndarray) -> np.ndarray:
    """|value| as an exactly comparable integer: the bf16 pattern without its sign."""
    return np.asarray(bits, dtype=np.uint16).astype(np.int64) & 0x7FFF


# ---------------------------------------------------------------------------
# N:M magnitude pruning (§1, §2.1): per group, an explicit sort
# ---------------------------------------------------------------------------


def select_nm(bits: np.ndarray, n: int, m: int) -> np.ndarray:
    """Indices (ascending) of the n kept entries of every m-group of every row.

    ``bits`` is rows x cols bf16 patterns, cols % m == 0, groups aligned at
    column 0.  Each group is sorted by (larger magnitude first, then lower
    index first); the first n survive.  Returns int64 [rows, cols/m, n].
    """
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    if cols % m:
        raise ValueError("cols must be a multiple of m")
    keys = magnitude_key(bits).reshape(rows, cols // m, m)
    index = np.broadcast_to(np.arange(m), keys.shape)
    # np.lexsort: the LAST key is the primary one -> primary -key, then index.
    order = np.lexsort((index, -keys), axis=-1)
    return np.sort(order[..., :n], axis=-1)


def select_nm_small(bits: np.ndarray, n: int, m: int) -> np.ndarray:
    """Same selection with Python's ``sorted`` per group (tiny inputs only)."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    out = np.zeros((rows, cols // m, n), dtype=np.int64)
    for r in range(rows):
        for g in range(cols // m):
            grp = [int(bits[r, g * m + j]) & 0x7FFF for j in range(m)]
            order = sorted(range(m), key=lambda j: (-grp[j], j))
            out[r, g] = sorted(order[:n])
    return out


def mask_from_selection(sel: np.ndarray, m: int) -> np.ndarray:
    rows, groups, _ = sel.shape
    mask = np.zeros((rows, groups, m), dtype=bool)
    np.put_along_axis(mask, sel, True, axis=-1)
    return mask.reshape(rows, groups * m)


def prune_nm_mask(bits: np.ndarray, n: int, m: int) -> np.ndarray:
    """Boolean keep-mask of the N:M magnitude pruning of ``bits`` (any n:m)."""
    return mask_from_selection(select_nm(bits, n, m), m)


# ---------------------------------------------------------------------------
# 2:4 compressed format (§2.3 "sparse formats"; App. K compression)
# ---------------------------------------------------------------------------

LEGAL_NIBBLES = frozenset(i0 | (i1 << 2) for i0, i1 in itertools.combinations(range(4), 2))


def pack_meta24(sel: np.ndarray) -> np.ndarray:
    """[rows, groups, 2] ascending kept indices -> rows x groups/2 metadata bytes."""
    rows, groups, n = sel.shape
    assert n == 2 and groups % 2 == 0
    nib = (sel[..., 0] | (sel[..., 1] << 2)).astype(np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def unpack_meta24(meta: np.ndarray) -> np.ndarray:
    """rows x cols/8 metadata bytes -> [rows, cols/4, 2] kept indices."""
    meta = np.asarray(meta, dtype=np.uint8)
    rows, nbytes = meta.shape
    nib = np.empty((rows, nbytes * 2), dtype=np.int64)
    nib[:, 0::2] = meta & 0xF
    nib[:, 1::2] = meta >> 4
    return np.stack([nib & 3, nib >> 2], axis=-1)


def prune24(bits: np.ndarray):
    """2:4 prune-and-compress of a rows x cols bf16 weight (keys on |w|).

    Returns (vals uint16 rows x cols/2, meta uint8 rows x cols/8, mask bool
    rows x cols).  ``vals`` lists each group's kept entries in ascending
    column order.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    if cols % 8:
        raise ValueError("2:4 compression needs cols % 8 == 0")
    sel = select_nm(bits, 2, 4)
    grouped = bits.reshape(rows, cols // 4, 4)
    vals = np.take_along_axis(grouped, sel, axis=-1).reshape(rows, cols // 2)
    return vals.astype(np.uint16), pack_meta24(sel), mask_from_selection(sel, 4)


def decompress24(vals: np.ndarray, meta: np.ndarray, cols: int) -> np.ndarray:
    """Compressed (vals, meta) -> rows x cols bf16 patterns, zeros (0x0000) elsewhere."""
    vals = np.asarray(vals, dtype=np.uint16)
    rows = vals.shape[0]
    sel = unpack_meta24(meta)
    out = np.zeros((rows, cols // 4, 4), dtype=np.uint16)
    np.put_along_axis(out, sel, vals.reshape(rows, cols // 4, 2), axis=-1)
    return out.reshape(rows, cols)


def double_prune24(vals: np.ndarray, meta: np.ndarray, rows: int, cols: int):
    """Second 2:4 pruning of the transposed single-pruned matrix (§1, §2.1).

    The rows x cols (out x in) compressed weight is expanded (pruned entries
    are +0), transposed to cols x rows, and pruned 2:4 again along its rows,
    i.e. along the old out dimension, which is the reduction dimension of the
    input-gradient product.  Returns (t_vals cols x rows/2, t_meta cols x
    rows/8, t_mask cols x rows).
    """
    if rows % 8:
        raise ValueError("double pruning needs rows % 8 == 0")
    ws = decompress24(vals, meta, cols)
    return prune24(np.ascontiguousarray(ws.T))


# ---------------------------------------------------------------------------
# Optimizer side (App. K: updated weights copied into the compressed format,
# and sparse linear combinations of matrices that share a pattern; §2.1: the
# initialised row mask is kept while the transposed one may change; §2.3:
# both sparse representations are updated during optimisation)
# ---------------------------------------------------------------------------


def recompress24(bits: np.ndarray, meta: np.ndarray) -> np.ndarray:
    """Compressed values of a rows x cols bf16 matrix at the positions a given
    2:4 metadata names: the mask is kept, not selected again.  Group g of a
    row keeps columns 4g + i0 and 4g + i1 of ``bits``, (i0, i1) being the
    nibble's two fields, in that order."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    if cols % 8:
        raise ValueError("2:4 compression needs cols % 8 == 0")
    sel = unpack_meta24(meta)
    grouped = bits.reshape(rows, cols // 4, 4)
    return np.take_along_axis(grouped, sel, axis=-1).reshape(rows, cols // 2).astype(np.uint16)


def recompress_double_prune24(bits: np.ndarray, meta: np.ndarray):
    """The updated weight compressed with its kept mask (recompress24), and
    the second pruning of the result (double_prune24).  Returns (vals, t_vals,
    t_meta)."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    vals = recompress24(bits, meta)
    t_vals, t_meta, _ = double_prune24(vals, meta, rows, cols)
    return vals, t_vals, t_meta


def double_prune24_frozen(vals: np.ndarray, meta: np.ndarray, rows: int, cols: int,
                          t_meta: np.ndarray) -> np.ndarray:
    """The second pruning with its column-wise mask frozen: the transpose of
    the single-pruned matrix (pruned entries +0) re-compressed at the
    positions a given transposed metadata ``t_meta`` (cols x rows/8) names,
    with no new selection.  Returns t_vals (cols x rows/2)."""
    ws = decompress24(vals, meta, cols)
    return recompress24(np.ascontiguousarray(ws.T), t_meta)


def recompress_frozen24(bits: np.ndarray, meta: np.ndarray, t_meta: np.ndarray):
    """Both masks kept: the updated weight gathered at the row mask
    (recompress24), and its transpose gathered at the frozen column mask
    (double_prune24_frozen).  Returns (vals, t_vals)."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    vals = recompress24(bits, meta)
    return vals, double_prune24_frozen(vals, meta, rows, cols, t_meta)


def sparse_axpby24(beta: float, a_vals: np.ndarray, gamma: float, b_vals: np.ndarray,
                   meta: np.ndarray) -> np.ndarray:
    """beta·A + gamma·B of two rows x cols matrices that share the 2:4
    pattern ``meta``, given as real-valued compressed values (rows x cols/2):
    both are expanded to their dense masked matrices, combined in fp64 and
    compressed again with the same pattern."""
    a_vals = np.asarray(a_vals, dtype=np.float64)
    b_vals = np.asarray(b_vals, dtype=np.float64)
    rows, half = a_vals.shape
    cols = 2 * half
    sel = unpack_meta24(meta)

    def dense(v):
        out = np.zeros((rows, cols // 4, 4))
        np.put_along_axis(out, sel, v.reshape(rows, cols // 4, 2), axis=-1)
        return out.reshape(rows, cols)

    c = beta * dense(a_vals) + gamma * dense(b_vals)
    return np.take_along_axis(c.reshape(rows, cols // 4, 4), sel, axis=-1).reshape(rows, half)


# ---------------------------------------------------------------------------
# Products (§2.1 forward/backward, §2.2 adapters, App. K masked gradient)
# ---------------------------------------------------------------------------
# The *_f64 functions take real-valued fp64 matrices; the others take the bf16
# bit patterns and compressed formats the library takes, expand them exactly,
# and call the fp64 ones.


def forward_f64(X, Ws, L, R):
    """Y = X·Wsᵀ + (X·L)·R; returns (Y, XL).  L, R may be None (no adapter)."""
    Y = X @ Ws.T
    if L is None:
        return Y, np.zeros((X.shape[0], 0))
    XL = X @ L
    return Y + XL @ R, XL


def backward_input_f64(dY, D, L, R):
    """dX = dY·Dᵀ + (dY·Rᵀ)·Lᵀ with D the in x out double-pruned matrix; returns (dX, G)."""
    dX = dY @ D.T
    if L is None:
        return dX, np.zeros((dY.shape[0], 0))
    G = dY @ R.T
    return dX + G @ L.T, G


def backward_weight_f64(dY, X, mask, L, R):
    """(dW = mask ⊙ (dYᵀ·X), dL = Xᵀ·(dY·Rᵀ), dR = (X·L)ᵀ·dY)."""
    dW = np.where(mask, dY.T @ X, 0.0)
    if L is None:
        return dW, None, None
    return dW, X.T @ (dY @ R.T), (X @ L).T @ dY


def _dense(vals, meta, cols):
    return bf16_to_f64(decompress24(vals, meta, cols))


def _adapter(L, R):
    if L is None:
        return None, None
    return bf16_to_f64(L), bf16_to_f64(R)


def linear_fwd(X, Wv, Wm, L, R):
    """Y = X·Wsᵀ + (X·L)·R and XL = X·L, in fp64 from bf16 inputs.

    X: T x in, (Wv, Wm): out x in compressed 2:4, L: in x r, R: r x out
    (no adapter: pass L = R = None).
    """
    Xf = bf16_to_f64(X)
    return forward_f64(Xf, _dense(Wv, Wm, Xf.shape[1]), *_adapter(L, R))


def linear_bwd_input(dY, Dv, Dm, L, R):
    """dX = dY·Dᵀ + (dY·Rᵀ)·Lᵀ and G = dY·Rᵀ, in fp64 from bf16 inputs.

    (Dv, Dm) is the double-pruned in x out matrix, 2:4 along out, so dX only
    sees the entries that both prunings kept.
    """
    dYf = bf16_to_f64(dY)
    return backward_input_f64(dYf, _dense(Dv, Dm, dYf.shape[1]), *_adapter(L, R))


def linear_bwd_weight(dY, X, Wm, L, R):
    """Masked weight gradient and adapter gradients, in fp64 from bf16 inputs.

    dW = M ⊙ (dYᵀ·X) with M the weight's own (first-pruning) mask, returned
    compressed (out x in/2, kept entries in the metadata's ascending order)
    and dense (out x in); dL = Xᵀ·(dY·Rᵀ), dR = (X·L)ᵀ·dY (None without an
    adapter).
    """
    dYf, Xf = bf16_to_f64(dY), bf16_to_f64(X)
    out, inn = dYf.shape[1], Xf.shape[1]
    sel = unpack_meta24(Wm)
    mask = mask_from_selection(sel, 4)
    dW_dense, dL, dR = backward_weight_f64(dYf, Xf, mask, *_adapter(L, R))
    dW_comp = np.take_along_axis(dW_dense.reshape(out, inn // 4, 4), sel, axis=-1)
    return dW_comp.reshape(out, inn // 2), dW_dense, dL, dR


# ---------------------------------------------------------------------------
# Other N:M patterns (§2.1 "Double-pruned backward pass" names 1:2, 2:4 and
# 2:8, with §T.1's count of the zeros the second pruning adds to each)
# ---------------------------------------------------------------------------
#
# 1:2 keeps one entry of every aligned pair.  Two aligned pairs make an
# aligned quadruple with exactly two kept entries, one in each half, so a
# 1:2-pruned matrix is also 2:4 and is stored in the 2:4 format above
# (i0 in {0, 1}, i1 in {2, 3}).
#
# 2:8 keeps two entries of every aligned group of eight.  Its format:
#   vals: rows x cols/4, the two kept entries of each group in ascending
#         column order;
#   meta: rows x cols/8 bytes, one per group: i0 | i1 << 3 (i0 < i1).
# A 2:8-pruned matrix is also 2:4 (no quadruple holds more than two of the
# group's two entries); its 2:4 form keeps, in each quadruple, the group's
# entries that fall in it, padded to two with the quadruple's lowest-index
# remaining positions, which hold +0.


def prune12(bits: np.ndarray):
    """1:2 prune-and-compress into the 2:4 format: per aligned pair the entry
    of larger magnitude key, the lower column on ties.  Returns (vals rows x
    cols/2, meta rows x cols/8, mask rows x cols)."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    if cols % 8:
        raise ValueError("the 2:4 format needs cols % 8 == 0")
    pair = select_nm(bits, 1, 2).reshape(rows, cols // 4, 2)  # index within each pair
    sel = np.stack([pair[..., 0], 2 + pair[..., 1]], axis=-1)  # ascending quadruple indices
    grouped = bits.reshape(rows, cols // 4, 4)
    vals = np.take_along_axis(grouped, sel, axis=-1).reshape(rows, cols // 2)
    return vals.astype(np.uint16), pack_meta24(sel), mask_from_selection(sel, 4)


def double_prune12(vals: np.ndarray, meta: np.ndarray, rows: int, cols: int):
    """Second 1:2 pruning: the rows x cols 1:2-pruned weight (2:4 format) is
    expanded (pruned entries +0), transposed, and pruned 1:2 again along the
    old out dimension.  Returns (t_vals cols x rows/2, t_meta cols x rows/8,
    t_mask cols x rows), in the 2:4 format."""
    if rows % 8:
        raise ValueError("double pruning needs rows % 8 == 0")
    ws = decompress24(vals, meta, cols)
    return prune12(np.ascontiguousarray(ws.T))


def pack_meta28(sel: np.ndarray) -> np.ndarray:
    """[rows, groups, 2] ascending kept indices (0..7) -> rows x groups bytes."""
    return (sel[..., 0] | (sel[..., 1] << 3)).astype(np.uint8)


def unpack_meta28(meta: np.ndarray) -> np.ndarray:
    """rows x cols/8 bytes -> [rows, cols/8, 2] kept indices."""
    meta = np.asarray(meta, dtype=np.uint8).astype(np.int64)
    return np.stack([meta & 7, (meta >> 3) & 7], axis=-1)


def prune28(bits: np.ndarray):
    """2:8 prune-and-compress: the two entries of largest magnitude key of
    each aligned group of eight, lower columns first on ties.  Returns (vals
    rows x cols/4, meta rows x cols/8, mask rows x cols)."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    if cols % 8:
        raise ValueError("2:8 needs cols % 8 == 0")
    sel = select_nm(bits, 2, 8)
    grouped = bits.reshape(rows, cols // 8, 8)
    vals = np.take_along_axis(grouped, sel, axis=-1).reshape(rows, cols // 4)
    return vals.astype(np.uint16), pack_meta28(sel), mask_from_selection(sel, 8)


def decompress28(vals: np.ndarray, meta: np.ndarray, cols: int) -> np.ndarray:
    """2:8 (vals, meta) -> rows x cols bf16 patterns, zeros elsewhere."""
    vals = np.asarray(vals, dtype=np.uint16)
    rows = vals.shape[0]
    out = np.zeros((rows, cols // 8, 8), dtype=np.uint16)
    np.put_along_axis(out, unpack_meta28(meta), vals.reshape(rows, cols // 8, 2), axis=-1)
    return out.reshape(rows, cols)


def double_prune28(vals: np.ndarray, meta: np.ndarray, rows: int, cols: int):
    """Second 2:8 pruning of the transposed 2:8-pruned weight, along the old
    out dimension (pruned entries key 0, so a group with fewer than two
    non-zeros keeps its lowest-index remaining positions, +0).  Returns
    (t_vals cols x rows/4, t_meta cols x rows/8, t_mask cols x rows)."""
    if rows % 8:
        raise ValueError("double pruning needs rows % 8 == 0")
    ws = decompress28(vals, meta, cols)
    return prune28(np.ascontiguousarray(ws.T))


def expand28_to_24(vals: np.ndarray, meta: np.ndarray, cols: int):
    """The 2:4 form of a 2:8-compressed matrix: each quadruple keeps the
    group's entries that fall in it, padded to two with its lowest-index
    remaining positions (value +0), in ascending order.  Returns (vals24
    rows x cols/2, meta24 rows x cols/8)."""
    dense = decompress28(vals, meta, cols)
    rows = dense.shape[0]
    keep = mask_from_selection(unpack_meta28(meta), 8)
    # "kept entries first, then the lowest free index" is the 2:4 selection
    # itself, run on keys that are 1 at kept positions and 0 elsewhere
    sel = select_nm(keep.astype(np.uint16), 2, 4)
    v = np.take_along_axis(dense.reshape(rows, cols // 4, 4), sel, axis=-1).reshape(rows, cols // 2)
    return v.astype(np.uint16), pack_meta24(sel)


def linear_bwd_weight28(dY, X, Wm28, L, R):
    """A5 + A6 with a 2:8 weight: dW = M ⊙ (dYᵀ·X), M the 2:8 mask of the
    weight, compressed in the 2:8 format (out x in/4), and dense; dL, dR as
    for 2:4.  Returns (dW_compressed, dW_dense, dL, dR)."""
    dYf, Xf = bf16_to_f64(dY), bf16_to_f64(X)
    out, inn = dYf.shape[1], Xf.shape[1]
    sel = unpack_meta28(Wm28)
    mask = mask_from_selection(sel, 8)
    dW_dense, dL, dR = backward_weight_f64(dYf, Xf, mask, *_adapter(L, R))
    dW_comp = np.take_along_axis(dW_dense.reshape(out, inn // 8, 8), sel, axis=-1)
    return dW_comp.reshape(out, inn // 4), dW_dense, dL, dR


# ---------------------------------------------------------------------------
# Lemma 2.1 (§T.1): expected zeros added by the second N:M pruning
# ---------------------------------------------------------------------------


def added_sparsity_expected(n: int, m: int) -> float:
    """E[max(Y - n, 0)] / m with Y ~ Binomial(m, n/m).

    Y counts the non-zeros that an m-group of the transposed pruned matrix
    holds when each entry survived the first pruning independently with
    probability n/m; the second pruning drops all but n of them.
    """
    from math import comb

    p = n / m
    e = sum((y - n) * comb(m, y) * p**y * (1 - p) ** (m - y) for y in range(n + 1, m + 1))
    return e / m


def added_sparsity_measured(bits: np.ndarray, n: int, m: int) -> float:
    """Fraction of all entries that the second pruning zeroes (any n:m).

    Prunes ``bits`` n:m along rows, transposes, prunes n:m again (pruned
    entries carry key 0) and counts non-zeros lost per element.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    first = prune_nm_mask(bits, n, m)
    ws = np.where(first, bits, np.uint16(0)).astype(np.uint16)
    wt = np.ascontiguousarray(ws.T)
    second = prune_nm_mask(wt, n, m)
    nz_before = np.count_nonzero(magnitude_key(wt))
    nz_after = np.count_nonzero(magnitude_key(np.where(second, wt, np.uint16(0))))
    return (nz_before - nz_after) / wt.size
