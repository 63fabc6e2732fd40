"""Full-size parity: the FC1 / FC2 linears of the measured blocks run whole on
the GPU through the same calls the benchmark makes; the oracle recomputes
sampled outputs exactly.  Each sample decomposes exactly:

  Y[t, o]    needs X[t, :], the pruned row o of W, XL[t, :] and R[:, o];
  dX[t, i]   needs dY[t, :], row i of D (the 8-column slab of W holding
             column i, pruned and double-pruned), G[t, :] and L[i, :];
  dW[o, :]   needs dY[:, o], all of X and row o of the mask;
  dL[i, :]   needs X[:, i] and all of G, so 8-column slabs of `in`;
  dR[:, o]   needs all of XL and dY[:, o].

Tolerance as everywhere: max|gpu - oracle| <= 2e-3 * max|oracle| per tensor,
over the sampled entries."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import assert_close_rel, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def np64(t):
    return t.double().cpu().numpy()


def run_gpu(S, d, T, inp, out, r, forward_only=False):
    import torch

    dev = "cuda"
    X, W = to_dev(d["X"]), to_dev(d["W"])
    L = to_dev(d["L"]) if r else None
    R = to_dev(d["R"]) if r else None
    Wv = torch.empty(out, inp // 2, dtype=torch.bfloat16, device=dev)
    Wm = torch.empty(out, inp // 8, dtype=torch.uint8, device=dev)
    Y = torch.empty(T, out, dtype=torch.float32, device=dev)
    XL = torch.empty(T, 2 * r, dtype=torch.bfloat16, device=dev) if r else None
    S.slope_prune_nm(W, Wv, Wm)
    S.slope_linear_fwd(X, Wv, Wm, L, R, Y, XL)
    res = {"Y": Y, "Wm": Wm}
    if not forward_only:
        dY = to_dev(d["dY"])
        Dv = torch.empty(inp, out // 2, dtype=torch.bfloat16, device=dev)
        Dm = torch.empty(inp, out // 8, dtype=torch.uint8, device=dev)
        dX = torch.empty(T, inp, dtype=torch.float32, device=dev)
        G = torch.empty(T, 2 * r, dtype=torch.bfloat16, device=dev) if r else None
        dW = torch.empty(out, inp // 2, dtype=torch.float32, device=dev)
        dL = torch.empty(inp, r, dtype=torch.float32, device=dev) if r else None
        dR = torch.empty(r, out, dtype=torch.float32, device=dev) if r else None
        S.slope_double_prune(Wv, Wm, out, inp, Dv, Dm)
        S.slope_linear_bwd_input(dY, Dv, Dm, L, R, dX, G)
        # the benchmark's weight-gradient call: dW, dL and dR together
        S.slope_linear_bwd_weight(dY, X, Wm, XL, G, dW, dL, dR)
        res.update(dX=dX, dW=dW, dL=dL, dR=dR)
    torch.cuda.synchronize()
    S.slope_device_status()
    return res


def check_layer(S, layer, T, inp, out, r, forward_only=False, n_t=48, n_o=256, n_i=256, n_slab=4):
    d = synth.layer_inputs(0, layer, T, inp, out, r)
    g = run_gpu(S, d, T, inp, out, r, forward_only)
    rng = np.random.default_rng(layer + T)
    ts = np.unique(np.concatenate([[0, T - 1], rng.choice(T, min(T, n_t), replace=False)]))
    os_ = np.unique(np.concatenate([[0, out - 1], rng.choice(out, n_o, replace=False)]))
    L, R = (d["L"], d["R"]) if r else (None, None)

    # Y on (ts x os_): pruned rows os_ of W; R restricted to columns os_
    v, m, _ = O.prune24(d["W"][os_])
    Yr, _ = O.linear_fwd(d["X"][ts], v, m, L, None if R is None else np.ascontiguousarray(R[:, os_]))
    assert_close_rel("Y", np64(g["Y"])[np.ix_(ts, os_)], Yr)
    if forward_only:
        return

    # dX on (ts x is_): rows is_ of D from the 8-column slabs of W holding them
    is_ = np.unique(np.concatenate([[0, inp - 1], rng.choice(inp, n_i, replace=False)]))
    slabs = sorted({int(i) // 8 for i in is_})
    Dv_rows, Dm_rows, col_of = [], [], {}
    for sb in slabs:
        vs, ms, _ = O.prune24(np.ascontiguousarray(d["W"][:, 8 * sb:8 * sb + 8]))
        tv, tm, _ = O.double_prune24(vs, ms, out, 8)
        for c in range(8):
            col_of[8 * sb + c] = len(Dv_rows)
            Dv_rows.append(tv[c])
            Dm_rows.append(tm[c])
    pick = [col_of[int(i)] for i in is_]
    Dv_s, Dm_s = np.stack(Dv_rows)[pick], np.stack(Dm_rows)[pick]
    dXr, _ = O.linear_bwd_input(d["dY"][ts], Dv_s, Dm_s, None if L is None else L[is_], R)
    assert_close_rel("dX", np64(g["dX"])[np.ix_(ts, is_)], dXr)

    # dW rows os_ (compressed) and dR columns os_: dY[:, os_], all of X (and XL)
    dWr, _, _, dRr = O.linear_bwd_weight(np.ascontiguousarray(d["dY"][:, os_]), d["X"], m, L,
                                         None if R is None else np.ascontiguousarray(R[:, os_]))
    assert_close_rel("dW", np64(g["dW"])[os_], dWr)
    if not r:
        return
    assert_close_rel("dR", np64(g["dR"])[:, os_], dRr)
    # dL on 8-column slabs of `in`: X[:, slab], all of G = dY·Rᵀ
    sl = rng.choice(inp // 8, n_slab, replace=False)
    cols = np.concatenate([np.arange(8 * s, 8 * s + 8) for s in sl])
    Wm_s = np.ascontiguousarray(O.pack_meta24(O.select_nm(np.ascontiguousarray(d["W"][:, cols]), 2, 4)))
    _, _, dLr, _ = O.linear_bwd_weight(d["dY"], np.ascontiguousarray(d["X"][:, cols]), Wm_s,
                                       np.ascontiguousarray(L[cols]), R)
    assert_close_rel("dL", np64(g["dL"])[cols], dLr)


@pytest.mark.parametrize("name,inp,out", [("q", 2560, 2560), ("fc1", 2560, 10240), ("fc2", 10240, 2560)])
def test_opt27b_block_linears(S, name, inp, out):
    check_layer(S, {"q": 0, "fc1": 4, "fc2": 5}[name], 8192, inp, out, 32)


@pytest.mark.parametrize("r", [0, 64])
def test_opt33b_fc1(S, r):
    check_layer(S, 4, 16384, 7168, 28672, r, n_t=32, n_o=192, n_i=192, n_slab=2)


@pytest.mark.parametrize("name,inp,out", [("q", 7168, 7168), ("fc2", 28672, 7168)])
def test_opt33b_q_and_fc2_r64(S, name, inp, out):
    """The other two shapes of the OPT-33B block at rank 64 (Q stands for
    K, V and O), whole on the GPU in the benchmark's launch configuration."""
    check_layer(S, {"q": 0, "fc2": 5}[name], 16384, inp, out, 64, n_t=32, n_o=192, n_i=192, n_slab=2)


@pytest.mark.parametrize("T", [1, 16, 128, 2048])
def test_opt66b_inference_fc1(S, T):
    check_layer(S, 4, T, 9216, 36864, 64, forward_only=True, n_t=64, n_o=512)


@pytest.mark.parametrize("name,T,inp,out", [("q", 16, 9216, 9216), ("fc2", 1, 36864, 9216),
                                             ("q", 128, 9216, 9216), ("fc2", 128, 36864, 9216)])
def test_opt66b_inference_split_k(S, name, T, inp, out):
    """72 weight tiles: the sparse product splits K over CTA pairs (16- and
    128-token tiles) and XL over clusters of eight."""
    check_layer(S, 0 if name == "q" else 5, T, inp, out, 64, forward_only=True, n_t=16, n_o=512)
