"""A5 + A6 on seeded random shapes and flags against the CPU oracle.

Many tokens on small weights make the weight-gradient launch split K (its
parts added atomically); widths give odd and even weight-tile counts (the
dense fallback and the pair kernel with dL and dR fused).  Each case draws
its flags: SLOPE_ACCUMULATE (outputs added onto random contents: the result
minus those contents must match the oracle), SLOPE_DW_DENSE (masked dense dW,
exact zeros off the mask when not accumulating), SLOPE_SKIP_DW or
SLOPE_SKIP_ADAPTER (the skipped buffers keep their contents bit for bit),
and whether a workspace is passed.  Tolerance as everywhere: 2e-3·max|oracle|
per tensor."""

import numpy as np
import pytest

from oracle import slope_oracle as O
from sparse_rank_adapter_gb300 import synth
from tests.helpers import assert_close_rel, ensure_built, to_dev
from tests.test_parity_linear import run_layer

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=4096):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        T = int(rng.choice([512, 1000, 2048, 4096, 8192, 12288]))
        inp = 128 * int(rng.integers(1, 9))
        o = 128 * int(rng.integers(1, 9))
        r = int(rng.choice([0, 8, 16, 64, 128]))
        acc, dense, ws = (bool(rng.integers(0, 2)) for _ in range(3))
        skip = str(rng.choice(["none", "none", "dw", "adapter"])) if r else "none"
        out.append((i, T, inp, o, r, acc, dense, skip, ws))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def S():
    ensure_built()
    from sparse_rank_adapter_gb300 import slope

    return slope


def np64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("i,T,inp,out,r,acc,dense,skip,ws", CASES,
                         ids=[f"T{c[1]}-in{c[2]}-out{c[3]}-r{c[4]}{'-acc' if c[5] else ''}"
                              f"{'-dense' if c[6] else ''}-skip_{c[7]}{'-ws' if c[8] else ''}" for c in CASES])
def test_random_weight_grad_flags(S, i, T, inp, out, r, acc, dense, skip, ws):
    import torch

    d = synth.layer_inputs(0, 900 + i, T, inp, out, r)
    g = run_layer(S, d, T, inp, out, r)  # Wm, XL and G as the step makes them
    gen = torch.Generator(device="cuda").manual_seed(i)
    dw_shape = (out, inp) if dense else (out, inp // 2)
    before = {"dW": torch.randn(dw_shape, generator=gen, device="cuda")}
    if r:
        before["dL"] = torch.randn(inp, r, generator=gen, device="cuda")
        before["dR"] = torch.randn(r, out, generator=gen, device="cuda")
    bufs = {k: v.clone() for k, v in before.items()}
    flags = (S.ACCUMULATE if acc else 0) | (S.DW_DENSE if dense else 0)
    flags |= {"none": 0, "dw": S.SKIP_DW, "adapter": S.SKIP_ADAPTER}[skip]
    workspace = torch.empty(256, dtype=torch.uint8, device="cuda") if ws else None
    S.slope_linear_bwd_weight(to_dev(d["dY"]), to_dev(d["X"]), g["Wm"], g["XL"], g["G"], bufs["dW"],
                              bufs.get("dL"), bufs.get("dR"), flags=flags, workspace=workspace)
    torch.cuda.synchronize()
    S.slope_device_status()

    vals, meta, mask = O.prune24(d["W"])
    L, R = (d["L"], d["R"]) if r else (None, None)
    dWc, dWd, dL, dR = O.linear_bwd_weight(d["dY"], d["X"], meta, L, R)
    refs = {"dW": dWd if dense else dWc, "dL": dL, "dR": dR}
    skipped = {"dw": ("dW",), "adapter": ("dL", "dR"), "none": ()}[skip]
    for name, buf in bufs.items():
        if name in skipped:
            assert torch.equal(buf, before[name]), f"{name} changed although skipped"
            continue
        got = np64(buf) - (np64(before[name]) if acc else 0.0)
        assert_close_rel(name, got, refs[name])
        if name == "dW" and dense and not acc:
            assert (np64(buf)[~mask] == 0).all()
