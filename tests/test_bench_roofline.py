"""The benchmark's roofline arithmetic (host logic, no GPU): the work counted
for each call and the peak it is judged against."""

import bench
from sparse_rank_adapter_gb300 import synth


def test_masked_weight_gradient_counts_half_the_dense_product():
    T, i, o, r = 16384, 7168, 28672, 64
    adapter = 2.0 * T * r * (i + o)
    assert bench.call_flops("bwd_weight", T, i, o, r) == 2.0 * T * i * o + adapter
    assert bench.method_flops("bwd_weight", T, i, o, r) == 1.0 * T * i * o + adapter
    # the sparse products count their dense-equivalent work either way
    for c in ("fwd", "bwd_input"):
        assert bench.method_flops(c, T, i, o, r) == bench.call_flops(c, T, i, o, r)


def test_step_flops_are_the_sum_of_the_calls():
    wl = synth.WORKLOADS["opt-33b-block-r64"]
    tot = sum(bench.call_flops(c, wl.tokens, x.inp, x.out, wl.rank)
              for x in wl.linears for c in ("fwd", "bwd_input", "bwd_weight"))
    assert abs(bench.flops_per_step(wl) - tot) <= 1e-9 * tot
    assert abs(bench.flops_per_step(wl) / 1e12 - 61.4) < 0.1  # the block's 61.4 TFLOP


def test_peak_follows_the_power_cap():
    p, why = bench.pick_peak({"reasons": ["sw_power_cap"]}, 1900.0, 1700.0)
    assert p == 1700.0 and "sustained" in why
    p, why = bench.pick_peak({"reasons": []}, 1900.0, 1700.0)
    assert p == 1900.0 and "burst" in why


def test_default_workload_is_the_largest_training_block():
    src = open(bench.__file__).read()
    assert 'ap.add_argument("--workload", default="opt-33b-block-r64"' in src


def test_sub_workload_keeps_one_linear():
    wl = bench.sub_workload(synth.WORKLOADS["opt-33b-block-r64"], "fc2")
    assert [(x.inp, x.out) for x in wl.linears] == [(28672, 7168)]
    assert wl.tokens == 16384 and wl.rank == 64


def test_oracle_slabs_cover_each_weight_exactly_once():
    s = bench.OracleSampler(synth.WORKLOADS["opt-350m-block"])
    for li, lin in enumerate(s.wl.linears):
        rows = sorted((o0, n) for l2, _, o0, n in s.units if l2 == li)
        assert sum(n for _, n in rows) == lin.out
        assert all(o0 % 8 == 0 and n % 8 == 0 for o0, n in rows)
    # a unit counts its exact share of the workload's flops
    tot = sum(s.unit_flops(lin, n) for _, lin, _, n in s.units)
    wl_T = synth.Workload("x", s.T, s.wl.rank, s.wl.linears)
    assert abs(tot - bench.flops_per_step(wl_T)) <= 1e-9 * tot


def test_fuse_qkv_rejects_what_it_cannot_stack():
    """--fuse-qkv stacks the block's Q, K and V: it refuses a single linear,
    the optimizer step and the other N:M patterns (argparse error, exit 2)."""
    import os
    import subprocess
    import sys

    script = os.path.abspath(bench.__file__)
    for extra in (["--linear", "q"], ["--optimizer"], ["--pattern", "1:2"]):
        res = subprocess.run([sys.executable, script, "--fuse-qkv", *extra], capture_output=True, text=True,
                             timeout=120)
        assert res.returncode == 2, (extra, res.stderr[-500:])
        assert "--fuse-qkv" in res.stderr
