"""The library's first calls in a process may be made inside CUDA graph
capture (kernel attributes, occupancy queries and the status word are set up
lazily on first use).  A fresh process captures prune, double prune, forward
and both gradients as its very first library calls, replays the graph, then
makes the same calls eagerly: masks and values must agree bit for bit, the
float outputs within 2e-3·max|eager| (the weight gradient adds split-K parts
with atomics, so its last bits may differ)."""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent(r"""
    import sys
    import torch
    sys.path.insert(0, sys.argv[1])
    from sparse_rank_adapter_gb300 import build
    build.build()
    from sparse_rank_adapter_gb300 import slope as S

    dev = "cuda"
    T, inp, out, r = 2048, 1024, 512, 16
    g = torch.Generator(device=dev).manual_seed(0)
    W = (torch.randn(out, inp, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    X = torch.randn(T, inp, device=dev, generator=g).to(torch.bfloat16)
    dY = torch.randn(T, out, device=dev, generator=g).to(torch.bfloat16)
    L = (torch.randn(inp, r, device=dev, generator=g) * 0.02).to(torch.bfloat16)
    R = (torch.randn(r, out, device=dev, generator=g) * 0.02).to(torch.bfloat16)

    def buffers():
        return dict(Wv=torch.empty(out, inp // 2, dtype=torch.bfloat16, device=dev),
                    Wm=torch.empty(out, inp // 8, dtype=torch.uint8, device=dev),
                    Dv=torch.empty(inp, out // 2, dtype=torch.bfloat16, device=dev),
                    Dm=torch.empty(inp, out // 8, dtype=torch.uint8, device=dev),
                    Y=torch.empty(T, out, dtype=torch.float32, device=dev),
                    XL=torch.empty(T, 2 * r, dtype=torch.bfloat16, device=dev),
                    dX=torch.empty(T, inp, dtype=torch.float32, device=dev),
                    G=torch.empty(T, 2 * r, dtype=torch.bfloat16, device=dev),
                    dW=torch.empty(out, inp // 2, dtype=torch.float32, device=dev),
                    dL=torch.empty(inp, r, dtype=torch.float32, device=dev),
                    dR=torch.empty(r, out, dtype=torch.float32, device=dev))

    def step(b, st):
        S.slope_prune_nm(W, b["Wv"], b["Wm"], stream=st)
        S.slope_double_prune(b["Wv"], b["Wm"], out, inp, b["Dv"], b["Dm"], stream=st)
        S.slope_linear_fwd(X, b["Wv"], b["Wm"], L, R, b["Y"], b["XL"], stream=st)
        S.slope_linear_bwd_input(dY, b["Dv"], b["Dm"], L, R, b["dX"], b["G"], stream=st)
        S.slope_linear_bwd_weight(dY, X, b["Wm"], b["XL"], b["G"], b["dW"], b["dL"], b["dR"], stream=st)

    st = torch.cuda.Stream()
    cap = buffers()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        step(cap, st)  # the library's first calls in this process
    with torch.cuda.stream(st):
        graph.replay()
    st.synchronize()
    S.slope_device_status(st)

    ref = buffers()
    with torch.cuda.stream(st):
        step(ref, st)
    st.synchronize()
    S.slope_device_status(st)
    for k in ("Wv", "Wm", "Dv", "Dm"):
        assert torch.equal(cap[k], ref[k]), k
    for k in ("Y", "XL", "dX", "G", "dW", "dL", "dR"):
        a, b = cap[k].double(), ref[k].double()
        assert (a - b).abs().max().item() <= 2e-3 * b.abs().max().item(), k
    print("capture-first-use ok")
""")


def test_first_library_calls_inside_graph_capture():
    res = subprocess.run([sys.executable, "-c", SCRIPT, REPO], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "capture-first-use ok" in res.stdout
