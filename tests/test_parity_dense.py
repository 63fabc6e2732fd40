"""A5/A6 alone (dense tcgen05 GEMMs only): the weight gradient with its mask
epilogue and the adapter gradients, on XL and G taken from the oracle in the
library's hi/lo bf16 form, so this file needs no sparse kernel."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import assert_close_rel, ensure_built, hilo_bits, to_dev, u8_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


# An even number of 128-row weight tiles (out = 256, 512, 768, 1024) takes the
# launch that computes dW, dL and dR together (2r up to 256); odd ones the
# separate adapter-gradient GEMMs.
@pytest.mark.parametrize("T,inp,out,r", [(64, 256, 256, 8), (200, 384, 512, 16), (1, 128, 128, 8),
                                         (4096, 1024, 1024, 16), (1000, 640, 896, 64), (333, 256, 384, 24),
                                         (777, 640, 1024, 64), (300, 512, 768, 120)])
@pytest.mark.parametrize("dense", [False, True])
def test_weight_and_adapter_grads(S, T, inp, out, r, dense):
    import torch

    d = synth.layer_inputs(0, 300 + T + r, T, inp, out, r)
    vals, meta, mask = O.prune24(d["W"])
    _, XL = O.linear_fwd(d["X"], vals, meta, d["L"], d["R"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inp)
    _, G = O.linear_bwd_input(d["dY"], tv, tm, d["L"], d["R"])
    dWc, dWd, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
    dW = torch.full((out, inp) if dense else (out, inp // 2), float("nan"), device="cuda")
    gdL = torch.full((inp, r), float("nan"), device="cuda")
    gdR = torch.full((r, out), float("nan"), device="cuda")
    S.slope_linear_bwd_weight(to_dev(d["dY"]), to_dev(d["X"]), u8_to_dev(meta), to_dev(hilo_bits(XL)),
                              to_dev(hilo_bits(G)), dW, gdL, gdR, flags=S.DW_DENSE if dense else 0)
    torch.cuda.synchronize()
    S.slope_device_status()
    got = dW.double().cpu().numpy()
    if dense:
        assert (got[~mask] == 0).all()
        assert_close_rel("dW dense", got, dWd)
    else:
        assert_close_rel("dW", got, dWc)
    assert_close_rel("dL", gdL.double().cpu().numpy(), dL)
    assert_close_rel("dR", gdR.double().cpu().numpy(), dR)


@pytest.mark.parametrize("T,inp,out,r", [(2048, 4096, 4096, 16), (16384, 1024, 1024, 8), (4096, 2048, 6144, 0)])
def test_weight_grad_with_waves_in_step(S, T, inp, out, r):
    """With a workspace the dW launch keeps its waves of tiles in step (a
    grid-wide counter between waves).  The tiles and their arithmetic are
    unchanged: the outputs match the call without a workspace (bit for bit
    where K is not split) and the oracle."""
    import torch

    d = synth.layer_inputs(0, 60 + r, T, inp, out, r)
    X, dY = to_dev(d["X"]), to_dev(d["dY"])
    W = to_dev(d["W"])
    Wv = torch.empty(out, inp // 2, dtype=torch.bfloat16, device="cuda")
    Wm = torch.empty(out, inp // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(W, Wv, Wm)
    XL = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda") if r else None
    G = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda") if r else None
    L = to_dev(d["L"]) if r else None
    R = to_dev(d["R"]) if r else None
    if r:
        S.slope_linear_fwd(X, Wv, Wm, L, R, torch.empty(T, out, device="cuda"), XL)
        Dv = torch.empty(inp, out // 2, dtype=torch.bfloat16, device="cuda")
        Dm = torch.empty(inp, out // 8, dtype=torch.uint8, device="cuda")
        S.slope_double_prune(Wv, Wm, out, inp, Dv, Dm)
        S.slope_linear_bwd_input(dY, Dv, Dm, L, R, torch.empty(T, inp, device="cuda"), G)
    ws = torch.full((256,), 0x5A, dtype=torch.uint8, device="cuda")  # contents must not matter
    outs = []
    for workspace in (None, ws, ws):  # twice with the workspace: the counter restarts
        dW = torch.full((out, inp // 2), float("nan"), device="cuda")
        dL = torch.full((inp, r), float("nan"), device="cuda") if r else None
        dR = torch.full((r, out), float("nan"), device="cuda") if r else None
        S.slope_linear_bwd_weight(dY, X, Wm, XL, G, dW, dL, dR, workspace=workspace)
        torch.cuda.synchronize()
        S.slope_device_status()
        outs.append((dW, dL, dR))
    vals, meta, _ = O.prune24(d["W"])
    dWc, _, dLr, dRr = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"] if r else None, d["R"] if r else None)
    for dW, dL, dR in outs[1:]:
        assert_close_rel("dW", dW.double().cpu().numpy(), dWc)
        if r:
            assert_close_rel("dL", dL.double().cpu().numpy(), dLr)
            assert_close_rel("dR", dR.double().cpu().numpy(), dRr)
    if T <= 4096:  # no split of K: the same tiles, the same sums
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[1][0], outs[2][0])


def test_weight_grads_with_workspaces_on_two_streams(S):
    """Two weight-gradient calls with their own workspaces, issued on two
    streams so that their launches can overlap: waves that cannot come
    together (the two grids share the SMs) stop waiting, and both results
    still match the oracle with no device-side error."""
    import torch

    T, inp, out, r = 2048, 4096, 4096, 16
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    cases = []
    for k, st in enumerate(streams):
        d = synth.layer_inputs(0, 80 + k, T, inp, out, r)
        X, dY, W = to_dev(d["X"]), to_dev(d["dY"]), to_dev(d["W"])
        Wv = torch.empty(out, inp // 2, dtype=torch.bfloat16, device="cuda")
        Wm = torch.empty(out, inp // 8, dtype=torch.uint8, device="cuda")
        S.slope_prune_nm(W, Wv, Wm)
        XL = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda")
        G = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda")
        S.slope_linear_fwd(X, Wv, Wm, to_dev(d["L"]), to_dev(d["R"]), torch.empty(T, out, device="cuda"), XL)
        Dv = torch.empty(inp, out // 2, dtype=torch.bfloat16, device="cuda")
        Dm = torch.empty(inp, out // 8, dtype=torch.uint8, device="cuda")
        S.slope_double_prune(Wv, Wm, out, inp, Dv, Dm)
        S.slope_linear_bwd_input(dY, Dv, Dm, to_dev(d["L"]), to_dev(d["R"]), torch.empty(T, inp, device="cuda"), G)
        cases.append((d, X, dY, Wm, XL, G))
    torch.cuda.synchronize()
    outs = []
    for (d, X, dY, Wm, XL, G), st in zip(cases, streams):
        dW = torch.full((out, inp // 2), float("nan"), device="cuda")
        dL = torch.empty(inp, r, device="cuda")
        dR = torch.empty(r, out, device="cuda")
        ws = torch.empty(256, dtype=torch.uint8, device="cuda")
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            for _ in range(3):  # several launches in flight on each stream
                S.slope_linear_bwd_weight(dY, X, Wm, XL, G, dW, dL, dR, workspace=ws, stream=st)
        outs.append((dW, dL, dR, ws))
    torch.cuda.synchronize()
    S.slope_device_status()
    for (d, *_), (dW, dL, dR, _) in zip(cases, outs):
        vals, meta, _ = O.prune24(d["W"])
        dWc, _, dLr, dRr = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
        assert_close_rel("dW", dW.double().cpu().numpy(), dWc)
        assert_close_rel("dL", dL.double().cpu().numpy(), dLr)
        assert_close_rel("dR", dR.double().cpu().numpy(), dRr)
