"""Pins for the CPU oracle: each check fixes the oracle to something other
than itself (brute force, exhaustive alphabets, closed forms, identity
inputs, finite differences, an independent bf16 cast)."""

import itertools
import math
import os

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits_of(values):
    return synth.to_bf16_bits(np.asarray(values, dtype=np.float32))


# ---------------------------------------------------------------- bf16 -----


def test_bf16_decode_known_patterns():
    b = np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x8000, 0x3FC0], dtype=np.uint16)
    v = O.bf16_to_f64(b)
    assert v[0] == 1.0 and v[1] == -2.0 and v[2] == 2.0**-133
    assert math.isinf(v[3]) and v[4] == 0.0 and math.copysign(1, v[4]) < 0 and v[5] == 1.5


def test_bf16_encode_ties_to_even():
    one = 1.0
    ulp = 2.0**-7  # bf16 spacing just above 1.0
    cases = {
        one: 0x3F80,
        one + ulp / 2: 0x3F80,  # tie -> even (stays)
        one + 3 * ulp / 2: 0x3F82,  # tie -> even (rounds up)
        one + ulp / 2 + 2.0**-20: 0x3F81,  # above the tie
        -2.0: 0xC000,
        0.0: 0x0000,
    }
    for x, want in cases.items():
        assert int(O.f64_to_bf16(np.array([x]))[0]) == want, x


def test_bf16_encode_matches_an_independent_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    ours = O.f64_to_bf16(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)


# ------------------------------------------------------- N:M selection -----


def brute_force_select(keys, n):
    """All C(m, n) subsets; keep the largest key-sum, lexicographically first."""
    best, best_sum = None, -1
    for sub in itertools.combinations(range(len(keys)), n):
        s = sum(keys[j] for j in sub)
        if s > best_sum:  # strict: earlier (lexicographically smaller) wins ties
            best, best_sum = sub, s
    return best


def rank_select(keys, n):
    """Keep j iff fewer than n entries beat it (larger key, or equal key and lower index)."""
    m = len(keys)
    kept = [j for j in range(m) if sum(1 for l in range(m) if keys[l] > keys[j] or (keys[l] == keys[j] and l < j)) < n]
    return tuple(kept)


@pytest.mark.parametrize("n,m", [(2, 4), (1, 2), (2, 8), (1, 4)])
def test_selection_equals_brute_force_with_many_ties(n, m):
    rng = np.random.default_rng(n * 100 + m)
    # a tiny alphabet so that ties are everywhere; signs vary independently
    alphabet = bits_of([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 3.0, -3.0])
    bits = rng.choice(alphabet, size=(40, 8 * m))
    sel = O.select_nm(bits, n, m)
    keys = O.magnitude_key(bits)
    for r in range(bits.shape[0]):
        for g in range(bits.shape[1] // m):
            grp = [int(k) for k in keys[r, g * m : (g + 1) * m]]
            want = brute_force_select(grp, n)
            assert tuple(sel[r, g]) == want
            assert rank_select(grp, n) == want


def test_selection_every_4tuple_of_a_tie_alphabet():
    # every 4-tuple over {+0, -0, ±a, ±b, ±c, d}: 9^4 groups, all tie patterns
    alphabet = bits_of([0.0, -0.0, 0.25, -0.25, 0.5, -0.5, 2.0, -2.0, 1.0])
    assert len(set(alphabet.tolist())) == 9
    tuples = np.array(list(itertools.product(alphabet, repeat=4)), dtype=np.uint16)
    assert tuples.shape == (9**4, 4)
    sel = O.select_nm(tuples, 2, 4).reshape(-1, 2)  # one group per row
    keys = O.magnitude_key(tuples)
    for t in range(tuples.shape[0]):
        assert tuple(sel[t]) == brute_force_select([int(k) for k in keys[t]], 2)


def test_python_sorted_and_vectorised_selection_agree():
    rng = np.random.default_rng(3)
    bits = synth.to_bf16_bits(rng.standard_normal((16, 64)).astype(np.float32) * 0.02)
    bits[::3, ::5] = bits[::3, 1::5][:, : bits[::3, ::5].shape[1]]  # plant equal magnitudes
    for n, m in [(2, 4), (1, 2), (2, 8)]:
        np.testing.assert_array_equal(O.select_nm(bits, n, m), O.select_nm_small(bits, n, m))


def test_metadata_hand_examples():
    # group 0: |-3| and |2| are the two largest -> indices (1, 2) -> 0b1001
    # group 1: four equal magnitudes -> lowest indices (0, 1) -> 0b0100
    # group 2: all zeros (both signs) -> (0, 1) -> 0b0100
    # group 3: one non-zero at 3, rest tie at 0 -> (0, 3) -> 0b1100
    row = bits_of([0.5, -3.0, 2.0, 0.25, 1.0, -1.0, 1.0, -1.0, 0.0, -0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 5.0])
    vals, meta, mask = O.prune24(row[None, :])
    assert list(meta[0]) == [0x9 | (0x4 << 4), 0x4 | (0xC << 4)]
    np.testing.assert_array_equal(vals[0], row[[1, 2, 4, 5, 8, 9, 12, 15]])
    assert mask[0].tolist() == [False, True, True, False, True, True, False, False,
                                True, True, False, False, True, False, False, True]


def test_prune24_invariants_on_gaussian_weights():
    W = synth.normal_bf16(0, 0, "W", (64, 256))
    vals, meta, mask = O.prune24(W)
    assert mask.reshape(64, 64, 4).sum(-1).min() == 2 and mask.reshape(64, 64, 4).sum(-1).max() == 2
    assert mask.sum() == 64 * 256 // 2
    nibbles = np.concatenate([meta & 0xF, meta >> 4], axis=1)
    assert set(np.unique(nibbles).tolist()) <= O.LEGAL_NIBBLES
    np.testing.assert_array_equal(vals, W[mask].reshape(64, 128))
    # kept magnitudes dominate dropped ones within every group
    k = O.magnitude_key(W).reshape(64, 64, 4)
    mk = mask.reshape(64, 64, 4)
    kept_min = np.where(mk, k, 1 << 20).min(-1)
    drop_max = np.where(mk, -1, k).max(-1)
    assert (kept_min >= drop_max).all()
    # round trip
    np.testing.assert_array_equal(O.decompress24(vals, meta, 256), np.where(mask, W, 0))


def test_prune_is_idempotent():
    W = synth.normal_bf16(0, 1, "W", (32, 128))
    vals, meta, _ = O.prune24(W)
    v2, m2, _ = O.prune24(O.decompress24(vals, meta, 128))
    np.testing.assert_array_equal(v2, vals)
    np.testing.assert_array_equal(m2, meta)


# ------------------------------------------------------- double pruning ----


def test_double_prune_invariants():
    out, inn = 128, 64
    W = synth.normal_bf16(0, 2, "W", (out, inn))
    vals, meta, mask = O.prune24(W)
    tv, tm, tmask = O.double_prune24(vals, meta, out, inn)
    assert tv.shape == (inn, out // 2) and tm.shape == (inn, out // 8)
    assert (tmask.reshape(inn, out // 4, 4).sum(-1) == 2).all()  # 2:4 along the new reduction dim
    D = O.decompress24(tv, tm, out)
    ws_t = np.where(mask, W, 0).T
    nz = O.magnitude_key(D) > 0
    assert (O.magnitude_key(ws_t)[nz] > 0).all()  # support of D within support of Wsᵀ
    np.testing.assert_array_equal(D[nz], ws_t[nz])  # and values unchanged there
    # positions the first pruning removed are +0 (pattern 0x0000) wherever D selects them
    assert (D[~mask.T] == 0).all()
    assert (tmask & ~mask.T).any()  # some Gaussian groups had < 2 non-zeros


def test_double_prune_keeps_a_doubly_24_matrix_unchanged():
    # a 4x4 block with two non-zeros in every row AND every column is 2:4 both
    # ways, so neither pruning may drop anything
    out, inn = 16, 16
    rng = np.random.default_rng(11)
    W = np.zeros((out, inn), dtype=np.uint16)
    for bo in range(0, out, 4):
        for bi in range(0, inn, 4):
            for r in range(4):
                for c in (r, (r + 1) % 4):
                    W[bo + r, bi + c] = bits_of([rng.uniform(0.1, 1.0) * rng.choice([-1, 1])])[0]
    vals, meta, mask = O.prune24(W)
    assert (mask == (W != 0)).all()
    tv, tm, tmask = O.double_prune24(vals, meta, out, inn)
    np.testing.assert_array_equal(O.decompress24(tv, tm, out), W.T)


def test_double_prune_selection_is_brute_force_on_the_transpose():
    out, inn = 32, 16
    alphabet = bits_of([0.0, 0.5, -0.5, 1.0, 2.0, -2.0])
    W = np.random.default_rng(5).choice(alphabet, size=(out, inn))
    vals, meta, mask = O.prune24(W)
    tv, tm, tmask = O.double_prune24(vals, meta, out, inn)
    ws_t = np.where(mask, W, 0).T
    keys = O.magnitude_key(ws_t)
    sel = O.unpack_meta24(tm)
    for i in range(inn):
        for h in range(out // 4):
            assert tuple(sel[i, h]) == brute_force_select([int(k) for k in keys[i, 4 * h : 4 * h + 4]], 2)


def _golden_lemma():
    rows = {}
    with open(os.path.join(GOLDEN, "lemma21_added_sparsity.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                n, m, pct = line.split()
                rows[(int(n), int(m))] = float(pct) / 100
    return rows


def test_lemma21_closed_form_matches_the_printed_values():
    g = _golden_lemma()
    assert O.added_sparsity_expected(1, 2) == pytest.approx(g[(1, 2)], abs=1e-12)
    assert O.added_sparsity_expected(2, 4) == pytest.approx(g[(2, 4)], abs=1e-12)
    # The printed 2:8 figure does not follow from the binomial model the lemma
    # states (it gives 5.84 %); the model is kept and the mismatch recorded.
    assert O.added_sparsity_expected(2, 8) == pytest.approx(0.05840, abs=1e-4)
    assert abs(O.added_sparsity_expected(2, 8) - g[(2, 8)]) > 0.02


@pytest.mark.parametrize("n,m", [(2, 4), (1, 2), (2, 8)])
def test_lemma21_measured_on_gaussian_weights(n, m):
    W = synth.normal_bf16(0, 3, "W", (512, 512))
    measured = O.added_sparsity_measured(W, n, m)
    expect = O.added_sparsity_expected(n, m)
    # per-group variance of the dropped count, exact from the binomial
    from math import comb

    p = n / m
    pmf = [comb(m, y) * p**y * (1 - p) ** (m - y) for y in range(m + 1)]
    e1 = sum(max(y - n, 0) * pmf[y] for y in range(m + 1))
    e2 = sum(max(y - n, 0) ** 2 * pmf[y] for y in range(m + 1))
    groups = W.size // m
    sigma = math.sqrt((e2 - e1 * e1) / groups) / m
    assert abs(measured - expect) < 5 * sigma, (measured, expect, sigma)


# --------------------------------------------------------------- products --


def gather_forward(X, vals, meta, rows_out):
    """Y[t, o] = Σ over the kept (i, w) of row o of X[t, i]·w, decoded by hand."""
    Xf = O.bf16_to_f64(X)
    Y = np.zeros((X.shape[0], rows_out))
    for o in range(rows_out):
        for b, byte in enumerate(meta[o]):
            for half in range(2):
                g = 2 * b + half
                nib = (int(byte) >> (4 * half)) & 0xF
                for slot, idx in enumerate((nib & 3, nib >> 2)):
                    w = O.bf16_to_f64(np.array([vals[o, 2 * g + slot]]))[0]
                    Y[:, o] += Xf[:, 4 * g + idx] * w
    return Y


def small_layer(T=24, inn=32, out=40, r=4, layer=0):
    d = synth.layer_inputs(0, layer, T, inn, out, r)
    vals, meta, mask = O.prune24(d["W"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inn)
    return d, vals, meta, mask, tv, tm


def test_forward_equals_explicit_gather_product():
    d, vals, meta, mask, tv, tm = small_layer()
    Y0, _ = O.linear_fwd(d["X"], vals, meta, None, None)
    ref = gather_forward(d["X"], vals, meta, 40)
    np.testing.assert_allclose(Y0, ref, rtol=1e-12, atol=1e-12)
    Y, XL = O.linear_fwd(d["X"], vals, meta, d["L"], d["R"])
    adapter = np.zeros_like(Y)
    Xf, Lf, Rf = (O.bf16_to_f64(d[k]) for k in "XLR")
    for t in range(Y.shape[0]):
        for o in range(Y.shape[1]):
            adapter[t, o] = sum(sum(Xf[t, i] * Lf[i, j] for i in range(Xf.shape[1])) * Rf[j, o] for j in range(Rf.shape[0]))
    np.testing.assert_allclose(Y, ref + adapter, rtol=1e-12, atol=1e-12)


def test_identity_inputs_pin_transposes_and_metadata():
    inn, out, r = 32, 24, 4
    d = synth.layer_inputs(0, 4, 1, inn, out, r)
    vals, meta, mask = O.prune24(d["W"])
    ws = O.bf16_to_f64(np.where(mask, d["W"], 0))
    eye_in = np.where(np.eye(inn, dtype=bool), np.uint16(0x3F80), np.uint16(0))
    Y, _ = O.linear_fwd(eye_in, vals, meta, d["L"], d["R"])
    np.testing.assert_allclose(Y, ws.T + O.bf16_to_f64(d["L"]) @ O.bf16_to_f64(d["R"]), rtol=0, atol=1e-15)
    tv, tm, _ = O.double_prune24(vals, meta, out, inn)
    Dd = O.bf16_to_f64(O.decompress24(tv, tm, out))
    eye_out = np.where(np.eye(out, dtype=bool), np.uint16(0x3F80), np.uint16(0))
    dX, _ = O.linear_bwd_input(eye_out, tv, tm, d["L"], d["R"])
    np.testing.assert_allclose(dX, Dd.T + O.bf16_to_f64(d["R"]).T @ O.bf16_to_f64(d["L"]).T, rtol=0, atol=1e-15)
    # one-hot X and dY select a single gradient entry, equal to the mask bit
    for o, i in [(0, 0), (5, 7), (23, 31), (11, 2)]:
        x = np.zeros((1, inn), np.uint16)
        x[0, i] = 0x3F80
        g = np.zeros((1, out), np.uint16)
        g[0, o] = 0x3F80
        dWc, dWd, _, _ = O.linear_bwd_weight(g, x, meta, None, None)
        assert dWd.sum() == float(mask[o, i]) and dWd[o, i] == float(mask[o, i])
        assert dWc.sum() == float(mask[o, i])


def test_adapter_and_sparse_parts_separate():
    d, vals, meta, mask, tv, tm = small_layer(layer=5)
    zeroL = np.zeros_like(d["L"])
    Y, XL = O.linear_fwd(d["X"], vals, meta, zeroL, d["R"])
    Y0, _ = O.linear_fwd(d["X"], vals, meta, None, None)
    np.testing.assert_array_equal(Y, Y0)
    assert not XL.any()
    zv = np.zeros_like(vals)
    Ya, XLa = O.linear_fwd(d["X"], zv, meta, d["L"], d["R"])
    np.testing.assert_allclose(Ya, XLa @ O.bf16_to_f64(d["R"]), rtol=1e-13, atol=1e-15)


def test_gradients_by_finite_differences():
    """s = <Y, dY> is bilinear, so central differences with h = 1 are exact up
    to rounding: they pin dL, dR, the masked dW and the true input gradient."""
    T, inn, out, r = 5, 16, 16, 3
    d = synth.layer_inputs(0, 6, T, inn, out, r)
    vals, meta, mask = O.prune24(d["W"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inn)
    X, W, L, R, dY = (O.bf16_to_f64(d[k]) for k in ("X", "W", "L", "R", "dY"))

    def s(X_, W_, L_, R_):
        Y, _ = O.forward_f64(X_, np.where(mask, W_, 0.0), L_, R_)
        return float((Y * dY).sum())

    def fd(which, arr):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            up, dn = arr.copy(), arr.copy()
            up[idx] += 1.0
            dn[idx] -= 1.0
            args = {"X": X, "W": W, "L": L, "R": R}
            a_up, a_dn = dict(args, **{which: up}), dict(args, **{which: dn})
            g[idx] = (s(**{k + "_": v for k, v in a_up.items()}) - s(**{k + "_": v for k, v in a_dn.items()})) / 2
        return g

    dWc, dWd, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
    np.testing.assert_allclose(dWd, fd("W", W), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(dWc, fd("W", W)[mask].reshape(out, inn // 2), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(dL, fd("L", L), rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(dR, fd("R", R), rtol=1e-10, atol=1e-10)
    dX_true = fd("X", X)
    dX, G = O.linear_bwd_input(d["dY"], tv, tm, d["L"], d["R"])
    np.testing.assert_allclose(G, dY @ R.T, rtol=1e-12, atol=1e-14)
    D = O.bf16_to_f64(O.decompress24(tv, tm, out))
    ws = np.where(mask, W, 0.0)
    # the double-pruned dX misses exactly the entries the second pruning dropped
    np.testing.assert_allclose(dX_true - dX, dY @ (ws - D.T), rtol=1e-10, atol=1e-10)
    assert np.abs(ws - D.T).max() > 0  # something was dropped


def test_products_agree_with_a_second_library():
    torch = pytest.importorskip("torch")
    d, vals, meta, mask, tv, tm = small_layer(T=33, inn=64, out=48, r=8, layer=7)
    Y, XL = O.linear_fwd(d["X"], vals, meta, d["L"], d["R"])
    X, W, L, R, dY = (torch.from_numpy(O.bf16_to_f64(d[k])) for k in ("X", "W", "L", "R", "dY"))
    Ws = W * torch.from_numpy(mask)
    torch.testing.assert_close(torch.from_numpy(Y), X @ Ws.T + X @ L @ R, rtol=1e-12, atol=1e-12)
    dWc, dWd, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
    torch.testing.assert_close(torch.from_numpy(dL), X.T @ (dY @ R.T), rtol=1e-12, atol=1e-12)
    torch.testing.assert_close(torch.from_numpy(dR), (X @ L).T @ dY, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- optimizer side


def test_recompress_at_own_mask_is_prune():
    """Gathering a weight at the mask selected from it returns the values the
    selection kept: the gather and the selection agree on layout and order."""
    W = synth.normal_bf16(0, 31, "W", (64, 96))
    v, m, _ = O.prune24(W)
    np.testing.assert_array_equal(O.recompress24(W, m), v)


def test_recompress_worked_example():
    """One row of eight weights 1..8 and metadata byte 0xD8: the low nibble 0x8
    names positions 0 and 2 of group 0, the high nibble 0xD positions 1 and 3
    of group 1, so the values are 1, 3, 6, 8."""
    W = synth.to_bf16_bits(np.arange(1, 9, dtype=np.float32)).reshape(1, 8)
    vals = O.recompress24(W, np.array([[0xD8]], dtype=np.uint8))
    np.testing.assert_array_equal(O.bf16_to_f64(vals), [[1.0, 3.0, 6.0, 8.0]])


def test_recompress_is_masked_weight():
    """Expanding the gathered values gives W where the (kept) mask is set and
    zero elsewhere; the mask is rebuilt here from the nibbles one by one."""
    rng = np.random.default_rng(5)
    W = synth.normal_bf16(0, 32, "W", (16, 32))
    codes = np.array(sorted(O.LEGAL_NIBBLES), dtype=np.uint8)
    nib = rng.choice(codes, size=(16, 8))
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    mask = np.zeros((16, 32), dtype=bool)
    for r in range(16):
        for g in range(8):
            mask[r, 4 * g + (nib[r, g] & 3)] = True
            mask[r, 4 * g + (nib[r, g] >> 2)] = True
    dense = O.decompress24(O.recompress24(W, meta), meta, 32)
    np.testing.assert_array_equal(dense, np.where(mask, W, 0).astype(np.uint16))


def test_recompress_double_prune_matches_the_two_steps():
    """With the weight unchanged, re-compressing at its own mask and double
    pruning gives what prune24 and double_prune24 give; with an updated
    weight the transposed result still keeps 2 of 4 along its rows and only
    positions the kept row mask allows."""
    W = synth.normal_bf16(0, 33, "W", (64, 48))
    v, m, mask = O.prune24(W)
    tv, tm, _ = O.double_prune24(v, m, 64, 48)
    v2, tv2, tm2 = O.recompress_double_prune24(W, m)
    np.testing.assert_array_equal(v2, v)
    np.testing.assert_array_equal(tv2, tv)
    np.testing.assert_array_equal(tm2, tm)
    W2 = synth.normal_bf16(0, 34, "W", (64, 48))  # the optimizer's new values
    v3, tv3, tm3 = O.recompress_double_prune24(W2, m)
    t_mask = O.decompress24(np.full_like(tv3, 0x3F80), tm3, 64) != 0  # positions D keeps
    assert (t_mask.reshape(48, 16, 4).sum(-1) == 2).all()
    nz = O.decompress24(tv3, tm3, 64) != 0
    assert not (nz & ~mask.T).any()  # D's non-zeros lie inside the kept row mask


def test_sparse_axpby_cases():
    """beta·A + gamma·B on a shared pattern: (1, 0) gives A, (0, 1) gives B,
    A = B gives (beta + gamma)·A, and it is linear in (beta, gamma); the
    result equals the element-wise combination of the compressed values
    because both matrices keep the same positions."""
    rng = np.random.default_rng(7)
    _, meta, _ = O.prune24(synth.normal_bf16(0, 35, "W", (32, 64)))
    A = rng.standard_normal((32, 32))
    B = rng.standard_normal((32, 32))
    np.testing.assert_array_equal(O.sparse_axpby24(1.0, A, 0.0, B, meta), A)
    np.testing.assert_array_equal(O.sparse_axpby24(0.0, A, 1.0, B, meta), B)
    np.testing.assert_allclose(O.sparse_axpby24(0.3, A, 0.5, A, meta), 0.8 * A, rtol=1e-15)
    c1 = O.sparse_axpby24(0.9, A, -0.01, B, meta)
    c2 = O.sparse_axpby24(0.9, A, 0.0, B, meta) + O.sparse_axpby24(0.0, A, -0.01, B, meta)
    np.testing.assert_allclose(c1, c2, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(c1, 0.9 * A - 0.01 * B, rtol=1e-14, atol=1e-15)


def test_frozen_double_prune_fixed_point_and_gather():
    """With the column mask frozen at what the second pruning selected, the
    frozen variant returns the same values; with any other frozen mask each
    value is the transposed single-pruned entry at the named position (zero
    where the first pruning removed it)."""
    W = synth.normal_bf16(0, 36, "W", (64, 48))
    v, m, mask = O.prune24(W)
    tv, tm, _ = O.double_prune24(v, m, 64, 48)
    np.testing.assert_array_equal(O.double_prune24_frozen(v, m, 64, 48, tm), tv)
    rng = np.random.default_rng(8)
    codes = np.array(sorted(O.LEGAL_NIBBLES), dtype=np.uint8)
    nib = rng.choice(codes, size=(48, 16))
    tmf = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    got = O.double_prune24_frozen(v, m, 64, 48, tmf)
    ws = np.where(mask, W, 0).astype(np.uint16)
    for i in range(48):
        for g in range(16):
            i0, i1 = nib[i, g] & 3, nib[i, g] >> 2
            assert got[i, 2 * g] == ws[4 * g + i0, i]
            assert got[i, 2 * g + 1] == ws[4 * g + i1, i]
    vals, tvals = O.recompress_frozen24(W, m, tmf)
    np.testing.assert_array_equal(vals, v)
    np.testing.assert_array_equal(tvals, got)


# ---------------------------------------------------- 1:2 and 2:8 patterns --


def _keys(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.int64) & 0x7FFF)


def _best_pair(keys8):
    """Brute force over all C(8, 2) pairs: the largest key sum, then the
    lexicographically smallest pair (ascending indices)."""
    best = None
    for a, b in itertools.combinations(range(len(keys8)), 2):
        cand = (keys8[a] + keys8[b], -a, -b)
        if best is None or cand > best[0]:
            best = (cand, (a, b))
    return best[1]


def test_prune12_hand_example():
    # pairs: (1, -3) keeps -3; (2, 2) a tie, the lower; (0, -0) a tie at key 0,
    # the lower; (5, -5) a tie, the lower
    row = bits_of([[1, -3, 2, 2, 0, -0.0, 5, -5]])
    vals, meta, mask = O.prune12(row)
    np.testing.assert_array_equal(vals[0], row[0, [1, 2, 4, 6]])
    # quadruple 0 keeps (1, 2) -> 0b1001, quadruple 1 keeps (0, 2) -> 0b1000
    assert meta[0, 0] == 0x89
    assert mask[0].tolist() == [False, True, True, False, True, False, True, False]


def test_prune12_invariants():
    W = synth.normal_bf16(0, 7, "W", (64, 96))
    vals, meta, mask = O.prune12(W)
    sel = O.unpack_meta24(meta)
    assert ((sel[..., 0] < 2) & (sel[..., 1] >= 2)).all()  # one kept in each half
    assert (mask.reshape(64, 48, 2).sum(-1) == 1).all()
    np.testing.assert_array_equal(O.decompress24(vals, meta, 96), np.where(mask, W, np.uint16(0)))
    # each pair keeps the entry of larger key, the lower on ties
    k = _keys(W).reshape(64, 48, 2)
    np.testing.assert_array_equal(mask.reshape(64, 48, 2)[..., 1], k[..., 1] > k[..., 0])


def test_double_prune12_is_brute_force_on_the_transpose():
    rng = np.random.default_rng(3)
    W = bits_of(rng.integers(-3, 4, size=(16, 24)).astype(np.float32))  # many ties and zeros
    vals, meta, mask = O.prune12(W)
    tv, tm, tmask = O.double_prune12(vals, meta, 16, 24)
    ws = np.where(mask, W, np.uint16(0))
    wt, kt = ws.T, _keys(ws.T)
    for i in range(24):
        for p in range(8):
            keep = 2 * p + (1 if kt[i, 2 * p + 1] > kt[i, 2 * p] else 0)
            assert tmask[i, keep] and not tmask[i, keep ^ 1]
    np.testing.assert_array_equal(O.decompress24(tv, tm, 16), np.where(tmask, wt, np.uint16(0)))
    # the second pruning only removes: D's support is inside Wsᵀ's
    assert not (np.where(tmask, kt, 0) > 0)[~mask.T].any()


def test_prune28_hand_example():
    row = bits_of([[1, -7, 3, 7, 0, 2, -2, 5, 2, 2, 2, 2, 2, 2, 2, 2]])
    vals, meta, mask = O.prune28(row)
    # group 0: |-7| and |7| at 1 and 3 -> 1 | 3 << 3 = 0x19; group 1: all tie -> (0, 1)
    assert meta[0].tolist() == [0x19, 0x08]
    np.testing.assert_array_equal(vals[0], row[0, [1, 3, 8, 9]])
    assert mask[0].sum() == 4


def test_prune28_invariants_and_decompress():
    W = synth.normal_bf16(0, 8, "W", (40, 64))
    vals, meta, mask = O.prune28(W)
    assert (meta >> 6 == 0).all()
    sel = O.unpack_meta28(meta)
    assert (sel[..., 0] < sel[..., 1]).all()
    assert (mask.reshape(40, 8, 8).sum(-1) == 2).all()
    np.testing.assert_array_equal(O.decompress28(vals, meta, 64), np.where(mask, W, np.uint16(0)))
    k = _keys(W).reshape(40, 8, 8)
    for r in range(40):
        for g in range(8):
            assert tuple(sel[r, g]) == _best_pair([int(x) for x in k[r, g]])


def test_double_prune28_is_brute_force_on_the_transpose():
    rng = np.random.default_rng(4)
    W = bits_of(rng.integers(-2, 3, size=(32, 16)).astype(np.float32))
    vals, meta, mask = O.prune28(W)
    tv, tm, tmask = O.double_prune28(vals, meta, 32, 16)
    ws = np.where(mask, W, np.uint16(0))
    kt = _keys(ws.T)
    sel = O.unpack_meta28(tm)
    for i in range(16):
        for h in range(4):
            assert tuple(sel[i, h]) == _best_pair([int(x) for x in kt[i, 8 * h:8 * h + 8]])
    np.testing.assert_array_equal(O.decompress28(tv, tm, 32), np.where(tmask, ws.T, np.uint16(0)))


@pytest.mark.parametrize("n,m", [(1, 2), (2, 8)])
def test_double_prunes_drop_what_lemma21_counts(n, m):
    """The zeros each double prune adds equal the count of the lemma's
    measurement helper, and sit within 5 sigma of its binomial value."""
    W = synth.normal_bf16(0, 9, "W", (512, 512))
    if (n, m) == (1, 2):
        v, mt, mask = O.prune12(W)
        _, _, tmask = O.double_prune12(v, mt, 512, 512)
    else:
        v, mt, mask = O.prune28(W)
        _, _, tmask = O.double_prune28(v, mt, 512, 512)
    ws = np.where(mask, W, np.uint16(0)).T
    before = np.count_nonzero(_keys(ws))
    after = np.count_nonzero(_keys(np.where(tmask, ws, np.uint16(0))))
    added = (before - after) / W.size
    assert added == pytest.approx(O.added_sparsity_measured(W, n, m), abs=0)
    expect = O.added_sparsity_expected(n, m)
    assert expect == pytest.approx(0.125 if m == 2 else 0.05840, abs=1e-4)
    assert abs(added - expect) < 0.01


def test_expand28_to_24_hand_example_and_invariants():
    row = bits_of([[1, -7, 3, 7, 0, 2, -2, 5, 9, 0, 0, 0, 0, 0, 0, 8]])
    vals, meta, _ = O.prune28(row)
    v24, m24 = O.expand28_to_24(vals, meta, 16)
    # group 0: both kept in quadruple 0 at (1, 3) -> 0xD; quadruple 1 pads (0, 1) -> 0x4
    # group 1: 9 at 0 and 8 at 7: quadruple 2 keeps 0 and pads 1 -> 0x4; quadruple 3 keeps 3, pads 0 -> 0xC
    assert m24[0].tolist() == [0x4D, 0xC4]
    z = np.uint16(0)
    np.testing.assert_array_equal(v24[0], [row[0, 1], row[0, 3], z, z, row[0, 8], z, z, row[0, 15]])
    W = synth.normal_bf16(0, 10, "W", (24, 64))
    vals, meta, mask = O.prune28(W)
    v24, m24 = O.expand28_to_24(vals, meta, 64)
    np.testing.assert_array_equal(O.decompress24(v24, m24, 64), O.decompress28(vals, meta, 64))
    sel24 = O.mask_from_selection(O.unpack_meta24(m24), 4)
    assert (sel24 | ~mask).all()  # the 2:4 form keeps every 2:8 entry


def test_weight_grad28_is_an_explicit_gather():
    d = synth.layer_inputs(0, 12, 10, 32, 16, 4)
    vals, meta, mask = O.prune28(d["W"])
    dWc, dWd, dL, dR = O.linear_bwd_weight28(d["dY"], d["X"], meta, d["L"], d["R"])
    dY, X = O.bf16_to_f64(d["dY"]), O.bf16_to_f64(d["X"])
    sel = O.unpack_meta28(meta)
    for o in range(16):
        for g in range(4):
            for j in range(2):
                i = 8 * g + int(sel[o, g, j])
                assert dWc[o, 2 * g + j] == pytest.approx(sum(dY[t, o] * X[t, i] for t in range(10)), rel=1e-12)
    assert (dWd[~mask] == 0).all()
    _, _, dL24, dR24 = O.linear_bwd_weight(d["dY"], d["X"], O.prune24(d["W"])[1], d["L"], d["R"])
    np.testing.assert_allclose(dL, dL24, rtol=1e-12)  # the adapter gradients ignore the mask
    np.testing.assert_allclose(dR, dR24, rtol=1e-12)


def test_stacked_linears_decompose_block_by_block():
    """The identities a caller relies on when stacking Q, K and V: A1 of the
    stacked weights is each weight's A1 stacked (rows prune alone); A2 of the
    stack is each A2 side by side (groups along 3·out never straddle two
    linears); with L side by side and R block-diagonal, the forward's column
    blocks, the weight gradient's row blocks, dL's column blocks and dR's
    diagonal blocks are each linear's own, and the stacked input gradient is
    the sum of the three."""
    T, inp, out, r = 12, 32, 16, 4
    ds = [synth.layer_inputs(0, 40 + j, T, inp, out, r) for j in range(3)]
    X = ds[0]["X"]
    W = np.concatenate([d["W"] for d in ds])
    dY = np.concatenate([d["dY"] for d in ds], axis=1)
    L = np.concatenate([d["L"] for d in ds], axis=1)
    R = np.zeros((3 * r, 3 * out), np.uint16)  # bf16 bits; +0 off the diagonal blocks
    for j, d in enumerate(ds):
        R[j * r:(j + 1) * r, j * out:(j + 1) * out] = d["R"]
    vals, meta, _ = O.prune24(W)
    tv, tm, _ = O.double_prune24(vals, meta, 3 * out, inp)
    Y, _ = O.linear_fwd(X, vals, meta, L, R)
    dX, _ = O.linear_bwd_input(dY, tv, tm, L, R)
    dWc, _, dL, dR = O.linear_bwd_weight(dY, X, meta, L, R)
    dX_sum = 0.0
    for j, d in enumerate(ds):
        vj, mj, _ = O.prune24(d["W"])
        tvj, tmj, _ = O.double_prune24(vj, mj, out, inp)
        rows, cols = slice(j * out, (j + 1) * out), slice(j * r, (j + 1) * r)
        np.testing.assert_array_equal(vals[rows], vj)
        np.testing.assert_array_equal(meta[rows], mj)
        np.testing.assert_array_equal(tv[:, j * out // 2:(j + 1) * out // 2], tvj)
        np.testing.assert_array_equal(tm[:, j * out // 8:(j + 1) * out // 8], tmj)
        Yj, _ = O.linear_fwd(X, vj, mj, d["L"], d["R"])
        np.testing.assert_allclose(Y[:, rows], Yj, rtol=1e-12, atol=1e-12)
        dXj, _ = O.linear_bwd_input(d["dY"], tvj, tmj, d["L"], d["R"])
        dX_sum = dX_sum + dXj
        dWj, _, dLj, dRj = O.linear_bwd_weight(d["dY"], X, mj, d["L"], d["R"])
        np.testing.assert_allclose(dWc[rows], dWj, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dL[:, cols], dLj, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dR[cols, rows], dRj, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dX, dX_sum, rtol=1e-12, atol=1e-12)
