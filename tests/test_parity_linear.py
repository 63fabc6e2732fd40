"""A3-A6 on the GPU against the CPU oracle.

Each case prunes and double-prunes on the GPU (bit-exactness of that step is
checked in test_parity_prune), then runs the forward, the input gradient and
the weight/adapter gradients; every float output must satisfy
max|gpu - oracle| <= 2e-3 * max|oracle|.  The oracle recomputes everything
from the same seeded bf16 inputs in fp64."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import TOL, assert_close_rel, bits_of, ensure_built, hilo_value, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def run_layer(S, d, T, inp, out, r, y_bf16=False, dense_dw=False):
    import torch

    dev = "cuda"
    X, W, dY = to_dev(d["X"]), to_dev(d["W"]), to_dev(d["dY"])
    L = to_dev(d["L"]) if r else None
    R = to_dev(d["R"]) if r else None
    Wv = torch.empty(out, inp // 2, dtype=torch.bfloat16, device=dev)
    Wm = torch.empty(out, inp // 8, dtype=torch.uint8, device=dev)
    Dv = torch.empty(inp, out // 2, dtype=torch.bfloat16, device=dev)
    Dm = torch.empty(inp, out // 8, dtype=torch.uint8, device=dev)
    ydt = torch.bfloat16 if y_bf16 else torch.float32
    Y = torch.full((T, out), float("nan"), dtype=ydt, device=dev)
    dX = torch.full((T, inp), float("nan"), dtype=ydt, device=dev)
    XL = torch.empty(T, 2 * r, dtype=torch.bfloat16, device=dev) if r else None
    G = torch.empty(T, 2 * r, dtype=torch.bfloat16, device=dev) if r else None
    dW = torch.full((out, inp) if dense_dw else (out, inp // 2), float("nan"), dtype=torch.float32, device=dev)
    dL = torch.full((inp, r), float("nan"), dtype=torch.float32, device=dev) if r else None
    dR = torch.full((r, out), float("nan"), dtype=torch.float32, device=dev) if r else None
    S.slope_prune_nm(W, Wv, Wm)
    S.slope_double_prune(Wv, Wm, out, inp, Dv, Dm)
    S.slope_linear_fwd(X, Wv, Wm, L, R, Y, XL)
    S.slope_linear_bwd_input(dY, Dv, Dm, L, R, dX, G)
    S.slope_linear_bwd_weight(dY, X, Wm, XL, G, dW, dL, dR, flags=S.DW_DENSE if dense_dw else 0)
    torch.cuda.synchronize()
    S.slope_device_status()
    return dict(Y=Y, dX=dX, XL=XL, G=G, dW=dW, dL=dL, dR=dR, Wv=Wv, Wm=Wm, Dv=Dv, Dm=Dm)


def np64(t):
    return t.double().cpu().numpy()


CASES = [
    # T, in, out, r
    (64, 256, 256, 8),      # the single-linear workload
    (1, 128, 128, 8),       # one token
    (16, 256, 384, 0),      # no adapter
    (200, 384, 512, 16),    # ragged token count (not a multiple of any tile)
    (300, 640, 384, 24),    # rank not a multiple of 16
    (130, 256, 128, 72),    # rank above 64: two adapter blocks
    (777, 1152, 896, 64),
    (16, 4096, 2048, 64),   # few token tiles: K split over clusters (4 and 2 CTAs)
    (48, 6144, 3072, 32),   # odd cluster sizes (6 and 3 CTAs), ragged T
    (100, 4096, 5120, 16),  # 128-token tiles with K split over CTA pairs (forward), ragged T
    (100, 4736, 5120, 16),  # the same with 37 K-blocks: 19 and 18 per CTA; 37 weight tiles in dX
    (4096, 1024, 1024, 16),  # OPT-350M block linears
    (4096, 1024, 4096, 16),
    (4096, 4096, 1024, 16),
    (300, 256, 384, 256),   # the largest rank the ABI takes: four adapter blocks per part
]


@pytest.mark.parametrize("T,inp,out,r", CASES)
def test_linear_matches_oracle(S, T, inp, out, r):
    d = synth.layer_inputs(0, T + inp + out + r, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r)
    vals, meta, _ = O.prune24(d["W"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inp)
    L, R = (d["L"], d["R"]) if r else (None, None)
    Y, XL = O.linear_fwd(d["X"], vals, meta, L, R)
    dX, G = O.linear_bwd_input(d["dY"], tv, tm, L, R)
    dWc, _, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, L, R)
    assert_close_rel("Y", np64(g["Y"]), Y)
    assert_close_rel("dX", np64(g["dX"]), dX)
    assert_close_rel("dW", np64(g["dW"]), dWc)
    if r:
        assert_close_rel("XL", hilo_value(g["XL"]), XL, tol=1e-4)
        assert_close_rel("G", hilo_value(g["G"]), G, tol=1e-4)
        assert_close_rel("dL", np64(g["dL"]), dL)
        assert_close_rel("dR", np64(g["dR"]), dR)


def test_dense_dw_and_bf16_outputs(S):
    T, inp, out, r = 333, 512, 256, 16
    d = synth.layer_inputs(0, 99, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r, y_bf16=True, dense_dw=True)
    vals, meta, mask = O.prune24(d["W"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inp)
    Y, _ = O.linear_fwd(d["X"], vals, meta, d["L"], d["R"])
    dX, _ = O.linear_bwd_input(d["dY"], tv, tm, d["L"], d["R"])
    _, dWd, _, _ = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
    gd = np64(g["dW"])
    assert (gd[~mask] == 0).all()  # pruned positions are exact zeros
    assert_close_rel("dW dense", gd, dWd)
    # bf16 outputs: within the fp32 tolerance plus one bf16 rounding of the value
    for name, got, ref in (("Y", g["Y"], Y), ("dX", g["dX"], dX)):
        gg = np64(got)
        bound = TOL * np.abs(ref).max() + 2.0**-8 * np.abs(ref)
        assert (np.abs(gg - ref) <= bound).all(), name


def test_weight_grad_accumulates(S):
    import torch

    T, inp, out, r = 96, 256, 256, 8
    d = synth.layer_inputs(0, 5, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r)
    dW1, dL1, dR1 = g["dW"].clone(), g["dL"].clone(), g["dR"].clone()
    S.slope_linear_bwd_weight(to_dev(d["dY"]), to_dev(d["X"]), g["Wm"], g["XL"], g["G"],
                              g["dW"], g["dL"], g["dR"], flags=S.ACCUMULATE)
    torch.cuda.synchronize()
    for a, b in ((g["dW"], dW1), (g["dL"], dL1), (g["dR"], dR1)):
        torch.testing.assert_close(a, 2 * b, rtol=1e-5, atol=1e-6)


def test_zero_tokens_writes_zero_gradients(S):
    import torch

    inp, out, r = 256, 128, 8
    Wm = torch.zeros(out, inp // 8, dtype=torch.uint8, device="cuda")
    dW = torch.full((out, inp // 2), 5.0, device="cuda")
    dL = torch.full((inp, r), 5.0, device="cuda")
    dR = torch.full((r, out), 5.0, device="cuda")
    X = torch.empty(0, inp, dtype=torch.bfloat16, device="cuda")
    dY = torch.empty(0, out, dtype=torch.bfloat16, device="cuda")
    XL = torch.empty(0, 2 * r, dtype=torch.bfloat16, device="cuda")
    S.lib()  # load
    st = S.lib().slope_linear_bwd_weight(0, 0, 0, inp, out, Wm.data_ptr(), 0, 0, r, dW.data_ptr(), 0,
                                         dL.data_ptr(), dR.data_ptr(), None, 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert not dW.any() and not dL.any() and not dR.any()
    del X, dY, XL


def test_identity_inputs_expose_layout(S):
    """X = I makes Y = Wsᵀ + L·R exactly (bf16 products are exact in fp32),
    pinning the kernel's reading of the compressed values and metadata."""
    import torch

    inp, out, r = 256, 256, 16
    d = synth.layer_inputs(0, 11, inp, inp, out, r)
    d["X"] = np.where(np.eye(inp, dtype=bool), np.uint16(0x3F80), np.uint16(0))
    g = run_layer(S, d, inp, inp, out, r)
    vals, meta, mask = O.prune24(d["W"])
    ws = O.bf16_to_f64(np.where(mask, d["W"], 0))
    ref = ws.T + O.bf16_to_f64(d["L"]) @ O.bf16_to_f64(d["R"])
    got = np64(g["Y"])
    np.testing.assert_allclose(got, ref, rtol=2e-6, atol=1e-7)


def test_weight_grad_skip_flags(S):
    """SLOPE_SKIP_ADAPTER computes dW alone and leaves dL, dR untouched;
    SLOPE_SKIP_DW computes dL, dR alone and leaves dW untouched."""
    import torch

    T, inp, out, r = 300, 512, 256, 16
    d = synth.layer_inputs(0, 21, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r)
    X, dY = to_dev(d["X"]), to_dev(d["dY"])
    dW = torch.full_like(g["dW"], 7.0)
    dL = torch.full_like(g["dL"], 7.0)
    dR = torch.full_like(g["dR"], 7.0)
    S.slope_linear_bwd_weight(dY, X, g["Wm"], g["XL"], g["G"], dW, dL, dR, flags=S.SKIP_ADAPTER)
    torch.cuda.synchronize()
    torch.testing.assert_close(dW, g["dW"], rtol=0, atol=0)
    assert (dL == 7.0).all() and (dR == 7.0).all()
    dW.fill_(7.0)
    S.slope_linear_bwd_weight(dY, X, g["Wm"], g["XL"], g["G"], dW, dL, dR, flags=S.SKIP_DW)
    torch.cuda.synchronize()
    assert (dW == 7.0).all()
    torch.testing.assert_close(dL, g["dL"], rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(dR, g["dR"], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("T,inp,out,r", [(200, 384, 512, 16), (4096, 1024, 4096, 16), (16, 4096, 2048, 64)])
def test_rank_plane_in_workspace(S, T, inp, out, r):
    """XL and G passed as NULL: the rank-r plane lives in the caller's
    workspace (slope_workspace_size bytes).  The same kernels run, so Y and
    dX are bit for bit those of the calls that keep XL and G, and match the
    oracle."""
    import torch

    d = synth.layer_inputs(0, 7 * T + r, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r)
    need = S.slope_workspace_size(T, inp, out, r)
    assert need == 4 * T * r + (-4 * T * r) % 256
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")  # contents must not matter
    X, dY, L, R = to_dev(d["X"]), to_dev(d["dY"]), to_dev(d["L"]), to_dev(d["R"])
    Y = torch.empty(T, out, dtype=torch.float32, device="cuda")
    dX = torch.empty(T, inp, dtype=torch.float32, device="cuda")
    S.slope_linear_fwd(X, g["Wv"], g["Wm"], L, R, Y, None, workspace=ws)
    S.slope_linear_bwd_input(dY, g["Dv"], g["Dm"], L, R, dX, None, workspace=ws)
    torch.cuda.synchronize()
    S.slope_device_status()
    assert torch.equal(Y, g["Y"]) and torch.equal(dX, g["dX"])
    # the plane holds the last call's G (hi | lo), exactly as the output G
    assert torch.equal(ws[: T * 4 * r].view(torch.bfloat16).view(T, 2 * r), g["G"])
    vals, meta, _ = O.prune24(d["W"])
    tv, tm, _ = O.double_prune24(vals, meta, out, inp)
    assert_close_rel("Y", np64(Y), O.linear_fwd(d["X"], vals, meta, d["L"], d["R"])[0])
    assert_close_rel("dX", np64(dX), O.linear_bwd_input(d["dY"], tv, tm, d["L"], d["R"])[0])


def test_weight_grad_accumulates_under_split_k(S):
    """Many tokens on a small weight: the dW launch splits K and adds its
    parts atomically.  With SLOPE_ACCUMULATE the call adds dW, dL and dR
    onto what the buffers held: result = before + oracle."""
    import torch

    T, inp, out, r = 16384, 256, 256, 8
    d = synth.layer_inputs(0, 31, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r)
    gen = torch.Generator(device="cuda").manual_seed(5)
    before = {k: torch.randn(g[k].shape, generator=gen, device="cuda") * 50 for k in ("dW", "dL", "dR")}
    acc = {k: v.clone() for k, v in before.items()}
    S.slope_linear_bwd_weight(to_dev(d["dY"]), to_dev(d["X"]), g["Wm"], g["XL"], g["G"],
                              acc["dW"], acc["dL"], acc["dR"], flags=S.ACCUMULATE)
    torch.cuda.synchronize()
    S.slope_device_status()
    vals, meta, _ = O.prune24(d["W"])
    dWc, _, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
    for name, ref in (("dW", dWc), ("dL", dL), ("dR", dR)):
        assert_close_rel(name, np64(acc[name]), np64(before[name]) + ref)
    # and the overwriting call on the same split matches the oracle alone
    assert_close_rel("dW", np64(g["dW"]), dWc)
