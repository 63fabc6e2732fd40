"""The 1:2 and 2:8 patterns on the GPU against the CPU oracle.

Masks, kept values and metadata bit-exact: A1 and A2 of both patterns, and
the 2:4 form of a 2:8 matrix.  Products within 2e-3·max|oracle| per tensor:
1:2 runs the 2:4 sparse GEMMs on its 2:4-format output as it is; 2:8 runs
them on its 2:4 form, and the weight gradient is masked by the 2:8 mask."""

import itertools
import math

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import assert_close_rel, bits_of, ensure_built, to_dev, u8_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def vcols(cols, m):
    return cols // 4 if m == 8 else cols // 2


def gpu_prune(S, W_bits, n, m):
    import torch

    rows, cols = W_bits.shape
    vals = torch.empty(rows, vcols(cols, m), dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(rows, cols // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(to_dev(W_bits), vals, meta, n=n, m=m)
    return vals, meta


def gpu_double(S, vals, meta, rows, cols, n, m):
    import torch

    tv = torch.empty(cols, vcols(rows, m), dtype=torch.bfloat16, device="cuda")
    tm = torch.empty(cols, rows // 8, dtype=torch.uint8, device="cuda")
    S.slope_double_prune_nm(vals, meta, rows, cols, tv, tm, n=n, m=m)
    return tv, tm


def gpu_expand(S, vals, meta, rows, cols):
    import torch

    v24 = torch.empty(rows, cols // 2, dtype=torch.bfloat16, device="cuda")
    m24 = torch.empty(rows, cols // 8, dtype=torch.uint8, device="cuda")
    S.slope_expand_nm_to_24(vals, meta, rows, cols, v24, m24)
    return v24, m24


ORACLE = {(1, 2): (O.prune12, O.double_prune12), (2, 8): (O.prune28, O.double_prune28)}


def check_patterns(S, W, n, m):
    """A1 (and A2 and the 2:4 form where the shape allows) bit-exact."""
    import torch

    prune, double = ORACLE[(n, m)]
    rows, cols = W.shape
    vals, meta = gpu_prune(S, W, n, m)
    ov, om, _ = prune(W)
    np.testing.assert_array_equal(bits_of(vals), ov)
    np.testing.assert_array_equal(meta.cpu().numpy(), om)
    if m == 8:
        v24, m24 = gpu_expand(S, vals, meta, rows, cols)
        ev, em = O.expand28_to_24(ov, om, cols)
        np.testing.assert_array_equal(bits_of(v24), ev)
        np.testing.assert_array_equal(m24.cpu().numpy(), em)
    if rows % 8 == 0 and cols % 16 == 0:
        tv, tm = gpu_double(S, vals, meta, rows, cols, n, m)
        otv, otm, _ = double(ov, om, rows, cols)
        np.testing.assert_array_equal(bits_of(tv), otv)
        np.testing.assert_array_equal(tm.cpu().numpy(), otm)
    torch.cuda.synchronize()


SHAPES = [(8, 16), (1, 8), (7, 40), (40, 48), (264, 144), (256, 1024), (1000, 1040), (2312, 2048)]


@pytest.mark.parametrize("n,m", [(1, 2), (2, 8)])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_patterns_bit_exact(S, n, m, rows, cols):
    check_patterns(S, synth.normal_bf16(0, rows + 3 * cols + m, "W", (rows, cols)), n, m)


def tie_heavy(rows, cols, seed):
    rng = np.random.default_rng(seed)
    alphabet = synth.to_bf16_bits(np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0], np.float32))
    return rng.choice(alphabet, size=(rows, cols)).astype(np.uint16)


@pytest.mark.parametrize("n,m", [(1, 2), (2, 8)])
@pytest.mark.parametrize("case", ["ties", "zeros", "specials", "exhaustive"])
def test_pattern_edge_values_bit_exact(S, n, m, case):
    if case == "ties":
        W = tie_heavy(512, 512, 11)
    elif case == "zeros":
        W = np.zeros((64, 128), np.uint16)
        W[::2, ::3] = 0x8000  # negative zeros among the zeros
    elif case == "specials":  # NaN > Inf > finite by the integer key
        W = tie_heavy(128, 256, 12)
        W[::5, ::7] = 0x7FC0
        W[1::5, ::3] = 0xFF80
        W[2::7, 1::4] = 0x0001  # smallest subnormal
    else:
        # 1:2: every ordered pair of a 9-symbol alphabet; 2:8: every group of
        # eight over a 3-symbol alphabet with at most three non-zeros
        alph = synth.to_bf16_bits(np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0, 4.0], np.float32))
        if m == 2:
            flat = np.array(list(itertools.product(alph, repeat=2)), dtype=np.uint16).ravel()
        else:
            a3 = alph[[0, 2, 5]]
            flat = np.array([t for t in itertools.product(a3, repeat=8) if sum(int(x) != 0 for x in t) <= 3],
                            dtype=np.uint16).ravel()
        n_rows = math.ceil(math.ceil(flat.size / 8) / 8) * 8  # rows of 8 values, a multiple of 8 rows
        W = np.zeros(n_rows * 8, np.uint16)
        W[: flat.size] = flat
        W = W.reshape(n_rows, 8)
        W = np.ascontiguousarray(np.concatenate([W, W[::-1]], axis=1))  # 16 columns: A2 runs too
    check_patterns(S, W, n, m)


def test_double_prune12_of_arbitrary_24_input(S):
    """The 1:2 A2 accepts any 2:4-format input: metadata pointing at zeros,
    kept values that are -0, and quadruples keeping both entries of a pair."""
    rows, cols = 64, 96
    rng = np.random.default_rng(5)
    legal = [i0 | (i1 << 2) for i0, i1 in itertools.combinations(range(4), 2)]
    nib = rng.choice(legal, size=(rows, cols // 4))
    meta = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    vals = tie_heavy(rows, cols // 2, 6)
    vals[::3, ::5] = 0x8000
    tv, tm = gpu_double(S, to_dev(vals), u8_to_dev(meta), rows, cols, 1, 2)
    otv, otm, _ = O.double_prune12(vals, meta, rows, cols)
    np.testing.assert_array_equal(bits_of(tv), otv)
    np.testing.assert_array_equal(tm.cpu().numpy(), otm)


@pytest.mark.parametrize("n,m", [(1, 2), (2, 8)])
def test_block_weight_bit_exact(S, n, m):
    """An OPT-2.7B FC1 weight (10240 x 2560), whole."""
    check_patterns(S, synth.normal_bf16(0, 4, "W", (10240, 2560)), n, m)


def np64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("n,m", [(1, 2), (2, 8)])
@pytest.mark.parametrize("T,inp,out,r", [(200, 384, 512, 16), (4096, 1024, 4096, 16), (64, 2048, 1024, 0)])
def test_pattern_products_match_oracle(S, n, m, T, inp, out, r):
    """Forward, input gradient and the weight and adapter gradients of a
    1:2 or 2:8 layer through the 2:4 sparse GEMMs (2:8: on its 2:4 form;
    dW masked by the 2:8 mask, compressed and dense)."""
    import torch

    d = synth.layer_inputs(0, 40 + T + r + m, T, inp, out, r)
    X, dY = to_dev(d["X"]), to_dev(d["dY"])
    L = to_dev(d["L"]) if r else None
    R = to_dev(d["R"]) if r else None
    prune, double = ORACLE[(n, m)]
    vals, meta = gpu_prune(S, d["W"], n, m)
    tv, tm = gpu_double(S, vals, meta, out, inp, n, m)
    if m == 8:
        Wv, Wm = gpu_expand(S, vals, meta, out, inp)
        Dv, Dm = gpu_expand(S, tv, tm, inp, out)
    else:
        Wv, Wm, Dv, Dm = vals, meta, tv, tm
    Y = torch.empty(T, out, dtype=torch.float32, device="cuda")
    dX = torch.empty(T, inp, dtype=torch.float32, device="cuda")
    XL = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda") if r else None
    G = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda") if r else None
    dW = torch.full((out, inp // 4 if m == 8 else inp // 2), float("nan"), device="cuda")
    dWd = torch.full((out, inp), float("nan"), device="cuda")
    dL = torch.empty(inp, r, dtype=torch.float32, device="cuda") if r else None
    dR = torch.empty(r, out, dtype=torch.float32, device="cuda") if r else None
    S.slope_linear_fwd(X, Wv, Wm, L, R, Y, XL)
    S.slope_linear_bwd_input(dY, Dv, Dm, L, R, dX, G)
    f28 = S.DW_NM28 if m == 8 else 0
    S.slope_linear_bwd_weight(dY, X, meta, XL, G, dW, dL, dR, flags=f28)
    S.slope_linear_bwd_weight(dY, X, meta, XL, G, dWd, flags=f28 | S.DW_DENSE | S.SKIP_ADAPTER)
    torch.cuda.synchronize()
    S.slope_device_status()

    ov, om, mask = prune(d["W"])
    otv, otm, _ = double(ov, om, out, inp)
    Lr, Rr = (d["L"], d["R"]) if r else (None, None)
    if m == 8:
        v24, m24 = O.expand28_to_24(ov, om, inp)
        tv24, tm24 = O.expand28_to_24(otv, otm, out)
        dWc, dWdense, dLr, dRr = O.linear_bwd_weight28(d["dY"], d["X"], om, Lr, Rr)
    else:
        v24, m24, tv24, tm24 = ov, om, otv, otm
        dWc, dWdense, dLr, dRr = O.linear_bwd_weight(d["dY"], d["X"], om, Lr, Rr)
    assert_close_rel("Y", np64(Y), O.linear_fwd(d["X"], v24, m24, Lr, Rr)[0])
    assert_close_rel("dX", np64(dX), O.linear_bwd_input(d["dY"], tv24, tm24, Lr, Rr)[0])
    assert_close_rel("dW", np64(dW), dWc)
    gd = np64(dWd)
    assert (gd[~mask] == 0).all()  # exact zeros off the pattern's mask
    assert_close_rel("dW dense", gd, dWdense)
    if r:
        assert_close_rel("dL", np64(dL), dLr)
        assert_close_rel("dR", np64(dR), dRr)
