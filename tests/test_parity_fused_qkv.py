"""Q, K and V of one block as one call per step, against the oracle per linear.

The three weights are stacked (3·out x in) and pruned as one matrix; the
adapter is one rank-3r adapter with L = [L_q L_k L_v] and R block-diagonal.
A1 ranks each row's groups on their own, so the stacked compressed weight is
the three compressed weights stacked, bit for bit; and the block-diagonal R
gives each column block exactly its own linear's (X·L)·R, so Y's column
blocks must each match the oracle's forward of that linear alone (within
2e-3·max|oracle|)."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import assert_close_rel, bits_of, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


@pytest.mark.parametrize("T,inp,out,r", [(1, 1024, 512, 16), (16, 2048, 1024, 64), (100, 4096, 1024, 64),
                                         (128, 2048, 1536, 32), (300, 1024, 768, 0)])
def test_stacked_qkv_matches_three_linears(S, T, inp, out, r):
    import torch

    ds = [synth.layer_inputs(0, 700 + 10 * j + r, T, inp, out, r) for j in range(3)]
    X = ds[0]["X"]  # one input for all three
    W = np.concatenate([d["W"] for d in ds])
    Wv = torch.empty(3 * out, inp // 2, dtype=torch.bfloat16, device="cuda")
    Wm = torch.empty(3 * out, inp // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(to_dev(W), Wv, Wm)
    L = R = XL = None
    if r:
        L = torch.cat([to_dev(d["L"]) for d in ds], dim=1).contiguous()
        R = torch.block_diag(*[to_dev(d["R"]) for d in ds]).contiguous()
        XL = torch.empty(T, 6 * r, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, 3 * out, dtype=torch.float32, device="cuda")
    S.slope_linear_fwd(to_dev(X), Wv, Wm, L, R, Y, XL)
    torch.cuda.synchronize()
    S.slope_device_status()
    Yg = Y.double().cpu().numpy()
    vb, mb = bits_of(Wv), Wm.cpu().numpy()
    for j, d in enumerate(ds):
        vals, meta, _ = O.prune24(d["W"])
        rows = slice(j * out, (j + 1) * out)
        np.testing.assert_array_equal(vb[rows], vals)
        np.testing.assert_array_equal(mb[rows], meta)
        ref, _ = O.linear_fwd(X, vals, meta, d["L"] if r else None, d["R"] if r else None)
        assert_close_rel(f"Y[{'qkv'[j]}]", Yg[:, rows], ref)


@pytest.mark.parametrize("T,inp,out,r", [(200, 512, 384, 16), (64, 256, 256, 0), (1000, 1024, 512, 48),
                                         (4096, 1024, 1024, 16)])
def test_stacked_qkv_training_step(S, T, inp, out, r):
    """The training calls on the stack: A2 of the stacked weight is each
    linear's A2 side by side (its 2:4 groups run along 3·out and never
    straddle two linears); dX is the sum of the three input gradients (the
    block's shared X); dW, dL and the diagonal blocks of dR are each
    linear's own.  3r = 144 takes the separate dL, dR launches."""
    import torch

    ds = [synth.layer_inputs(0, 800 + 10 * j + r, T, inp, out, r) for j in range(3)]
    X = ds[0]["X"]
    W = np.concatenate([d["W"] for d in ds])
    dY = np.ascontiguousarray(np.concatenate([d["dY"] for d in ds], axis=1))
    dev = "cuda"
    n = 3
    Wv = torch.empty(n * out, inp // 2, dtype=torch.bfloat16, device=dev)
    Wm = torch.empty(n * out, inp // 8, dtype=torch.uint8, device=dev)
    Dv = torch.empty(inp, n * out // 2, dtype=torch.bfloat16, device=dev)
    Dm = torch.empty(inp, n * out // 8, dtype=torch.uint8, device=dev)
    L = R = XL = G = dL = dR = None
    if r:
        L = torch.cat([to_dev(d["L"]) for d in ds], dim=1).contiguous()
        R = torch.block_diag(*[to_dev(d["R"]) for d in ds]).contiguous()
        XL = torch.empty(T, 2 * n * r, dtype=torch.bfloat16, device=dev)
        G = torch.empty(T, 2 * n * r, dtype=torch.bfloat16, device=dev)
        dL = torch.empty(inp, n * r, dtype=torch.float32, device=dev)
        dR = torch.empty(n * r, n * out, dtype=torch.float32, device=dev)
    Y = torch.empty(T, n * out, dtype=torch.float32, device=dev)
    dX = torch.empty(T, inp, dtype=torch.float32, device=dev)
    dW = torch.empty(n * out, inp // 2, dtype=torch.float32, device=dev)
    Xd, dYd = to_dev(X), to_dev(dY)
    S.slope_prune_nm(to_dev(W), Wv, Wm)
    S.slope_double_prune(Wv, Wm, n * out, inp, Dv, Dm)
    S.slope_linear_fwd(Xd, Wv, Wm, L, R, Y, XL)
    S.slope_linear_bwd_input(dYd, Dv, Dm, L, R, dX, G)
    S.slope_linear_bwd_weight(dYd, Xd, Wm, XL, G, dW, dL, dR)
    torch.cuda.synchronize()
    S.slope_device_status()

    def f64(t):
        return t.double().cpu().numpy()

    Dvb, Dmb = bits_of(Dv), Dm.cpu().numpy()
    dX_ref = 0.0
    for j, d in enumerate(ds):
        Lj, Rj = (d["L"], d["R"]) if r else (None, None)
        vals, meta, _ = O.prune24(d["W"])
        tv, tm, _ = O.double_prune24(vals, meta, out, inp)
        np.testing.assert_array_equal(Dvb[:, j * out // 2:(j + 1) * out // 2], tv)
        np.testing.assert_array_equal(Dmb[:, j * out // 8:(j + 1) * out // 8], tm)
        cols = slice(j * out, (j + 1) * out)
        Yj, _ = O.linear_fwd(X, vals, meta, Lj, Rj)
        assert_close_rel(f"Y[{'qkv'[j]}]", f64(Y)[:, cols], Yj)
        dXj, _ = O.linear_bwd_input(d["dY"], tv, tm, Lj, Rj)
        dX_ref = dX_ref + dXj
        dWj, _, dLj, dRj = O.linear_bwd_weight(d["dY"], X, meta, Lj, Rj)
        assert_close_rel(f"dW[{'qkv'[j]}]", f64(dW)[cols], dWj)
        if r:
            assert_close_rel(f"dL[{'qkv'[j]}]", f64(dL)[:, j * r:(j + 1) * r], dLj)
            assert_close_rel(f"dR[{'qkv'[j]}]", f64(dR)[j * r:(j + 1) * r, cols], dRj)
    assert_close_rel("dX (sum of three)", f64(dX), dX_ref)
