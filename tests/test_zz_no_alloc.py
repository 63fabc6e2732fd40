"""slope_linear_fwd_static_scratch: the forward for callers that cannot
allocate device memory (a plugin whose host runtime owns every allocation,
a serving loop that must not call cudaMalloc), which keeps its rank-r plane
in the library's own fixed device array instead of a caller's buffer.

Called through the C ABI, twice in a row on different inputs (the array
keeps the first call's plane when the second starts), and compared with
slope_linear_fwd, the entry point that takes XL from the caller, within the
tolerance every parity test here uses.  Sizes beyond the array are refused.

This file is named to be collected last, so that a run stopping at the
first failure has already run every other test."""

import numpy as np
import pytest

from sparse_rank_adapter_gb300 import synth
from tests.helpers import TOL, assert_close_rel, ensure_built, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def _layer(S, seed, T, inp, out, r):
    import torch

    d = synth.layer_inputs(seed, 0, T, inp, out, r)
    X, W = to_dev(d["X"]), to_dev(d["W"])
    L, R = to_dev(d["L"]), to_dev(d["R"])
    Wv = torch.empty(out, inp // 2, dtype=torch.bfloat16, device="cuda")
    Wm = torch.empty(out, inp // 8, dtype=torch.uint8, device="cuda")
    S.slope_prune_nm(W, Wv, Wm)
    return X, Wv, Wm, L, R


def _reference(S, X, Wv, Wm, L, R):
    """The existing entry point, with the caller's XL buffer."""
    import torch

    T, out, r = X.shape[0], Wv.shape[0], L.shape[1]
    Y = torch.empty(T, out, dtype=torch.float32, device="cuda")
    XL = torch.empty(T, 2 * r, dtype=torch.bfloat16, device="cuda")
    S.slope_linear_fwd(X, Wv, Wm, L, R, Y, XL)
    return Y


def test_static_scratch_forward_matches_the_forward_twice(S):
    import torch

    # two calls in a row with different shapes and inputs: the second finds
    # the first's plane in the shared array and must not depend on it
    cases = [(777, 1152, 896, 64, 1), (4096, 1024, 4096, 16, 2)]
    for T, inp, out, r, seed in cases:
        X, Wv, Wm, L, R = _layer(S, seed, T, inp, out, r)
        Y = torch.full((T, out), float("nan"), dtype=torch.float32, device="cuda")
        S.slope_linear_fwd_static_scratch(X, Wv, Wm, L, R, Y)
        ref = _reference(S, X, Wv, Wm, L, R)
        torch.cuda.synchronize()
        S.slope_device_status()
        assert torch.isfinite(Y).all()
        assert_close_rel("Y", Y.double().cpu().numpy(), ref.double().cpu().numpy(), tol=TOL)


def test_static_scratch_forward_bf16_output_and_no_adapter(S):
    import torch

    T, inp, out, r = 200, 384, 512, 16
    X, Wv, Wm, L, R = _layer(S, 3, T, inp, out, r)
    Y = torch.empty(T, out, dtype=torch.bfloat16, device="cuda")
    S.slope_linear_fwd_static_scratch(X, Wv, Wm, L, R, Y)
    ref = _reference(S, X, Wv, Wm, L, R)
    torch.cuda.synchronize()
    # bf16 output: the fp32 tolerance plus one bf16 rounding of the value
    got, want = Y.double().cpu().numpy(), ref.double().cpu().numpy()
    assert (np.abs(got - want) <= TOL * np.abs(want).max() + 2.0**-8 * np.abs(want)).all()
    # r == 0 needs no plane at all
    Y0 = torch.empty(T, out, dtype=torch.float32, device="cuda")
    S.slope_linear_fwd_static_scratch(X, Wv, Wm, None, None, Y0)
    Y0ref = torch.empty(T, out, dtype=torch.float32, device="cuda")
    S.slope_linear_fwd(X, Wv, Wm, None, None, Y0ref)
    torch.cuda.synchronize()
    assert_close_rel("Y r=0", Y0.double().cpu().numpy(), Y0ref.double().cpu().numpy(), tol=TOL)


def test_static_scratch_refuses_planes_beyond_the_array(S):
    import torch

    inp, out, r = 128, 128, 64
    limit = S.STATIC_SCRATCH_BYTES
    T_max = limit // (4 * r)  # the largest T whose plane fits exactly (32768 tokens)
    assert S.slope_workspace_size(T_max, inp, out, r) == limit
    for T, fits in ((T_max, True), (T_max + 1, False)):
        X, Wv, Wm, L, R = _layer(S, 4, T, inp, out, r)
        Y = torch.zeros(T, out, dtype=torch.float32, device="cuda")
        if fits:
            S.slope_linear_fwd_static_scratch(X, Wv, Wm, L, R, Y)
            ref = _reference(S, X, Wv, Wm, L, R)
            torch.cuda.synchronize()
            assert_close_rel("Y", Y.double().cpu().numpy(), ref.double().cpu().numpy(), tol=TOL)
        else:
            with pytest.raises(S.SlopeError) as e:
                S.slope_linear_fwd_static_scratch(X, Wv, Wm, L, R, Y)
            assert e.value.status == S.ERR_SHAPE
            torch.cuda.synchronize()
            assert not Y.any()  # refused before any work
