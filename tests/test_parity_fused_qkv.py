"""Q, K and V of one block as one forward call, against the oracle per linear.

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
