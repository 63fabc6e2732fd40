"""A3-A6 on seeded random shapes against the CPU oracle.

Token counts from 1 to 513 reach every tile width the dispatcher picks
(16, 64 and 128 tokens with and without a cluster split of K, the CTA-pair
kernels beyond); widths of 128 to 2048 give odd and even weight-tile counts
(one-CTA and pair kernels) and K-loops with and without splits; ranks
include values that are not multiples of 16 and ranks above 64 (two adapter
blocks).  Some cases write bf16 outputs and a dense masked dW.  Every output
is compared with the oracle: fp32 within 2e-3·max|oracle| per tensor, bf16
within that plus one bf16 rounding of the value, pruned dW positions exactly
zero."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import TOL, assert_close_rel, ensure_built, hilo_value
from tests.test_parity_linear import run_layer

pytestmark = pytest.mark.gpu


def _cases(n=64, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.choice([1, 3, 16, 17, 40, 64, 65, 100, 128, 129, 200, 257, 400, 513]))
        inp = 128 * int(rng.integers(1, 17))
        o = 128 * int(rng.integers(1, 17))
        r = int(rng.choice([0, 8, 16, 24, 40, 64, 72, 96]))
        out.append((i, T, inp, o, r, bool(rng.integers(0, 2)), bool(rng.integers(0, 2))))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def np64(t):
    return t.double().cpu().numpy()


def close_bf16(name, got, ref):
    bound = TOL * np.abs(ref).max() + 2.0**-8 * np.abs(ref)
    assert (np.abs(got - ref) <= bound).all(), name


@pytest.mark.parametrize("i,T,inp,out,r,y_bf16,dense_dw", CASES,
                         ids=[f"T{c[1]}-in{c[2]}-out{c[3]}-r{c[4]}{'-bf16' if c[5] else ''}{'-dense' if c[6] else ''}"
                              for c in CASES])
def test_random_shape_matches_oracle(S, i, T, inp, out, r, y_bf16, dense_dw):
    d = synth.layer_inputs(0, 500 + i, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r, y_bf16=y_bf16, dense_dw=dense_dw)
    vals, meta, mask = O.prune24(d["W"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inp)
    L, R = (d["L"], d["R"]) if r else (None, None)
    Y, XL = O.linear_fwd(d["X"], vals, meta, L, R)
    dX, G = O.linear_bwd_input(d["dY"], tv, tm, L, R)
    dWc, dWd, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, L, R)
    for name, ref in (("Y", Y), ("dX", dX)):
        got = np64(g[name])
        if y_bf16:
            close_bf16(name, got, ref)
        else:
            assert_close_rel(name, got, ref)
    if dense_dw:
        gd = np64(g["dW"])
        assert (gd[~mask] == 0).all()
        assert_close_rel("dW dense", gd, dWd)
    else:
        assert_close_rel("dW", np64(g["dW"]), dWc)
    if r:
        assert_close_rel("XL", hilo_value(g["XL"]), XL, tol=1e-4)
        assert_close_rel("G", hilo_value(g["G"]), G, tol=1e-4)
        assert_close_rel("dL", np64(g["dL"]), dL)
        assert_close_rel("dR", np64(g["dR"]), dR)
