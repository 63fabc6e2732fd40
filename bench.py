"""Benchmark of the 2:4-sparse + low-rank adapter linear path on GB300.

One step = the whole path over one OPT-shaped decoder block (six linears:
Q, K, V, O, FC1, FC2) for one batch of synthetic tokens:
    prune (A1) -> double prune (A2) -> forward (A3) -> input gradient (A4)
    -> masked weight gradient and adapter gradients (A5, A6)
all through the C ABI (libslope.so), on one stream, captured once as a CUDA
graph per input set and replayed.  Inputs are seeded synthetic bf16 tensors
resident in HBM; four input sets are rotated so that consecutive steps never
find their inputs in L2.

Metric: dense-equivalent TFLOP/s of fwd + bwd (2·T·in·out for each of the
forward, input-gradient and weight-gradient products plus 6·T·r·(in+out)
for the adapter), whole job, summed over ranks.

The default workload is the largest single-GPU block, OPT-33B-shaped
(d = 7168, FFN 28672, T = 16384, adapter rank 64).  `--linear NAME` keeps
one linear of the block (profiling runs of one launch).

--impl reference times the CPU oracle (the plain fp64 NumPy definition of
the same step) on the host cores, on a bounded sample of the same workload:
row slabs of each weight (a slab of output rows is an exact share of the
linear's work) over a token sample.

--gpus N (N > 1, not already under torchrun) starts N replica processes, one
per GPU, with RANK / LOCAL_RANK / WORLD_SIZE set, as torchrun would.

Step variants (the default is the five path calls per linear):
  --fused-prune      A1 and A2 as one call (slope_prune_and_double_prune);
  --optimizer        the training step with the row mask kept from
                     initialisation: the updated weight re-compressed and
                     double-pruned (slope_recompress_double_prune) in place of
                     A1 and A2, and beta·A + gamma·B (slope_sparse_axpby) on an
                     fp32 master copy of the kept values after the gradients;
  --frozen-columns   with --optimizer, the column mask kept too
                     (slope_recompress_frozen);
  --streams N        the block's linears (independent in this synthetic
                     step) issued on N streams, linear i on stream i % N,
                     forked from and joined into the step's stream; the
                     default, one stream, runs them as a dependent chain;
  --fuse-qkv         Q, K and V read one X and run as one call each on their
                     stacked compressed weights, with one rank-3r adapter (L
                     side by side, R block-diagonal); in training their input
                     gradients are summed by the stacked dX call, as the
                     block's shared X needs.
Every memory-bound call's achieved bandwidth is reported in `hbm_calls`, and
the library's tensor-pipe rate self test in `mma_rate_selftest`.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_rank_adapter_gb300 import synth  # noqa: E402

L2_BYTES = 129 * 2**20


def flops_per_step(wl) -> float:
    T, r = wl.tokens, wl.rank
    f = 0.0
    for lin in wl.linears:
        f += 2.0 * T * lin.inp * lin.out * (1 if wl.forward_only else 3)
        if r:
            f += (2.0 if wl.forward_only else 6.0) * T * r * (lin.inp + lin.out)
    return f


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (x itself without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, world: int, ms_step_max: float) -> float:
    """Every rank's work over the slowest rank's step time (weak scaling)."""
    return flops_per_rank * world / (ms_step_max * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------ clocks -------


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


class NvmlClockSampler:
    """Polls the SM clock and the clock-event reasons through NVML (the
    driver's libnvidia-ml, loaded with ctypes) about every millisecond from a
    background thread, so that even a timed region of a few milliseconds
    gets samples.  Reads only; changes no setting."""

    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, device):
        import ctypes
        import threading

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        import torch

        props = torch.cuda.get_device_properties(device)
        ok = False
        uuid = str(getattr(props, "uuid", ""))
        for u in (uuid, "GPU-" + uuid):
            if u and self.lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.handle)) == 0:
                ok = True
                break
        if not ok and hasattr(props, "pci_bus_id"):
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle)) == 0
        if not ok:
            self.lib.nvmlShutdown()
            raise RuntimeError("no NVML handle for this device")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = (float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0 else None)
        self.samples = []
        self.stop = threading.Event()
        self.thread = threading.Thread(target=self._poll, daemon=True)

    def _poll(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop.is_set():
            if (self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ct.byref(clk)) == 0
                    and self.reasons_fn(self.handle, ct.byref(rs)) == 0):
                self.samples.append((float(clk.value), int(rs.value)))
            self.stop.wait(0.001)

    def __enter__(self):
        self.thread.start()
        while not self.samples and self.thread.is_alive():  # running before the region starts
            time.sleep(0.0005)
        self.samples.clear()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "samples": 0}
        reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "sm_min_mhz": min(c for c, _ in self.samples), "reasons": reasons,
                "samples": len(self.samples), "source": "nvml, 1 ms polling"}


def clock_sampler(device, index):
    try:
        return NvmlClockSampler(device)
    except Exception:
        return ClockSampler(index)


# ------------------------------------------------------------- GPU arm ----


class BlockStep:
    """Device buffers and the ordered ABI calls of one block step."""

    def __init__(self, wl, seed: int, device, fused_prune: bool = False, optimizer: bool = False,
                 frozen_columns: bool = False, pattern: str = "2:4", fuse_qkv: bool = False):
        import torch

        from sparse_rank_adapter_gb300 import slope

        self.S = slope
        self.wl = wl
        # N:M pattern of the weights: 2:4, 1:2 (in the 2:4 format) or 2:8
        # (its own format, expanded to its 2:4 form for the sparse products)
        self.n, self.m = (int(x) for x in pattern.split(":"))
        self.extra_streams = []  # streams beside the step's own (see run)
        self.fused_prune = fused_prune
        self.optimizer = optimizer  # kept row mask: re-compression + A2, then beta·A + gamma·B
        self.frozen_columns = frozen_columns  # the column mask kept too: no second selection
        T, r = wl.tokens, wl.rank
        # workspaces of the weight-gradient calls (their wave counters), one
        # per stream the step may use: calls on one stream run one after
        # another, calls on two streams may overlap
        self.workspaces = [torch.empty(256, dtype=torch.uint8, device=device) for _ in range(8)]
        self.layers = []
        for li, lin in enumerate(wl.linears):
            inp, out = lin.inp, lin.out
            s = seed * 1000 + li
            b = dict(
                W=synth.device_normal_bf16((out, inp), 0.02, s * 8 + 0, device),
                X=synth.device_normal_bf16((T, inp), 1.0, s * 8 + 1, device),
                dY=synth.device_normal_bf16((T, out), 1.0, s * 8 + 2, device),
                L=synth.device_normal_bf16((inp, r), 0.02, s * 8 + 3, device) if r else None,
                R=synth.device_normal_bf16((r, out), 0.02, s * 8 + 4, device) if r else None,
                Wv=torch.empty(out, inp // 2, dtype=torch.bfloat16, device=device),
                Wm=torch.empty(out, inp // 8, dtype=torch.uint8, device=device),
                Dv=torch.empty(inp, out // 2, dtype=torch.bfloat16, device=device),
                Dm=torch.empty(inp, out // 8, dtype=torch.uint8, device=device),
                # activations and their gradients in bf16, the mixed-precision
                # convention; weight and adapter gradients in fp32
                Y=torch.empty(T, out, dtype=torch.bfloat16, device=device),
                XL=torch.empty(T, 2 * r, dtype=torch.bfloat16, device=device) if r else None,
                dX=torch.empty(T, inp, dtype=torch.bfloat16, device=device),
                G=torch.empty(T, 2 * r, dtype=torch.bfloat16, device=device) if r else None,
                dW=torch.empty(out, inp // 4 if self.m == 8 else inp // 2, dtype=torch.float32, device=device),
                # 2:8: the weight and its double pruning in the 2:8 format
                Wv8=torch.empty(out, inp // 4, dtype=torch.bfloat16, device=device) if self.m == 8 else None,
                Wm8=torch.empty(out, inp // 8, dtype=torch.uint8, device=device) if self.m == 8 else None,
                Dv8=torch.empty(inp, out // 4, dtype=torch.bfloat16, device=device) if self.m == 8 else None,
                Dm8=torch.empty(inp, out // 8, dtype=torch.uint8, device=device) if self.m == 8 else None,
                dL=torch.empty(inp, r, dtype=torch.float32, device=device) if r else None,
                dR=torch.empty(r, out, dtype=torch.float32, device=device) if r else None,
                # the optimizer's fp32 master copy of the kept values
                Wmaster=torch.empty(out, inp // 2, dtype=torch.float32, device=device) if optimizer else None,
                inp=inp, out=out)
            self.layers.append(b)
        if fuse_qkv:
            self.layers = [self._stack_qkv(self.layers[:3], device, not wl.forward_only)] + self.layers[3:]

    @staticmethod
    def _stack_qkv(parts, device, training):
        """Q, K and V of one block read the same X: one call computes all
        three with their weights stacked (3·out x in; A1 prunes rows on their
        own, so the stack prunes to the three compressed weights stacked) and
        one rank-3r adapter, L side by side and R block-diagonal, whose
        product is each linear's own (X·L)·R on its columns.  Backward, the
        stacked dY (T x 3·out) against the stacked double-pruned weight (its
        2:4 groups along 3·out never straddle two linears) sums the three
        input gradients, as the block's shared X needs; the weight gradient
        call gives the three dW and dL blocks, and dR on its diagonal blocks
        (the off-diagonal ones are computed and not used)."""
        import torch

        inp, out = parts[0]["inp"], parts[0]["out"]
        assert all(p["inp"] == inp and p["out"] == out for p in parts), "Q, K, V of one shape"
        T = parts[0]["X"].shape[0]
        r = 0 if parts[0]["L"] is None else parts[0]["L"].shape[1]
        n = len(parts)
        bf, f32 = torch.bfloat16, torch.float32

        def new(shape, dt, cond=True):
            return torch.empty(shape, dtype=dt, device=device) if cond else None

        b = dict(W=torch.cat([p["W"] for p in parts]), X=parts[0]["X"],
                 dY=torch.cat([p["dY"] for p in parts], dim=1) if training else None,
                 L=torch.cat([p["L"] for p in parts], dim=1) if r else None,
                 R=torch.block_diag(*[p["R"] for p in parts]).contiguous() if r else None,
                 Wv=new((n * out, inp // 2), bf), Wm=new((n * out, inp // 8), torch.uint8),
                 Dv=new((inp, n * out // 2), bf, training), Dm=new((inp, n * out // 8), torch.uint8, training),
                 Y=new((T, n * out), bf), XL=new((T, 2 * n * r), bf, r > 0),
                 dX=new((T, inp), bf, training), G=new((T, 2 * n * r), bf, training and r > 0),
                 dW=new((n * out, inp // 2), f32, training),
                 dL=new((inp, n * r), f32, training and r > 0), dR=new((n * r, n * out), f32, training and r > 0),
                 inp=inp, out=n * out, parts=[(inp, out)] * n)
        for k in ("Wv8", "Wm8", "Dv8", "Dm8", "Wmaster"):
            b[k] = None
        return b

    def input_names(self):
        if self.wl.forward_only:  # weights stay resident (pre-compressed); a request brings X
            return ["X"]
        return ["W", "X", "dY", "L", "R"]

    def output_names(self):
        return ["Y", "dX", "dW", "dL", "dR"] if not self.wl.forward_only else ["Y"]

    def prepare(self, stream):
        """Inference workloads take their weights pre-compressed, and the
        optimizer step keeps the mask chosen at initialisation: prune once
        here (and fill the master copy from the kept values)."""
        if self.wl.forward_only or self.optimizer:
            for b in self.layers:
                if self.frozen_columns:  # both masks from initialisation
                    self.S.slope_prune_and_double_prune(b["W"], b["Wv"], b["Wm"], b["Dv"], b["Dm"], stream=stream)
                elif self.m == 8:  # the 2:8 weight's 2:4 form is what the forward reads
                    self.S.slope_prune_nm(b["W"], b["Wv8"], b["Wm8"], n=2, m=8, stream=stream)
                    self.S.slope_expand_nm_to_24(b["Wv8"], b["Wm8"], b["out"], b["inp"], b["Wv"], b["Wm"],
                                                 stream=stream)
                else:
                    self.S.slope_prune_nm(b["W"], b["Wv"], b["Wm"], n=self.n, m=self.m, stream=stream)
                if self.optimizer:
                    b["Wmaster"].copy_(b["Wv"].float())

    def run(self, stream, marks=None, only=None):
        """Issues the step on `stream` (or, with `only`, the calls of that one
        linear); `marks` (optional) records an event pair around every ABI
        call, keyed by call name.  A training step prunes (the row mask is
        re-derived from the current weights), double-prunes, runs the forward
        and both gradients; an inference step runs the forward on the
        pre-compressed weights."""
        S = self.S
        # the block's linears are independent: with extra streams, linear i
        # goes to stream i % n (forked from and joined back into `stream`).
        # A marked pass stays on `stream`, so that each call's events time
        # that call alone.
        lanes = [stream] + (list(self.extra_streams) if only is None and marks is None else [])
        for x in lanes[1:]:
            x.wait_stream(stream)
        for li, b in enumerate(self.layers if only is None else [self.layers[only]]):
            sl = lanes[li % len(lanes)]
            if self.wl.forward_only:
                calls = []
            elif self.optimizer and self.frozen_columns:  # the updated W at both kept masks
                calls = [("recompress_frozen", lambda b=b: S.slope_recompress_frozen(
                    b["W"], b["Wm"], b["Dm"], b["Wv"], b["Dv"], stream=sl))]
            elif self.optimizer:  # the updated W at the kept mask, and the second pruning
                calls = [("recompress_double", lambda b=b: S.slope_recompress_double_prune(
                    b["W"], b["Wm"], b["Wv"], b["Dv"], b["Dm"], stream=sl))]
            elif self.fused_prune:  # A1 and A2 from one read of W
                calls = [("prune_double", lambda b=b: S.slope_prune_and_double_prune(
                    b["W"], b["Wv"], b["Wm"], b["Dv"], b["Dm"], stream=sl))]
            elif self.m == 2:  # 1:2, written in the 2:4 format
                calls = [
                    ("prune12", lambda b=b: S.slope_prune_nm(b["W"], b["Wv"], b["Wm"], n=1, m=2, stream=sl)),
                    ("double_prune12", lambda b=b: S.slope_double_prune_nm(
                        b["Wv"], b["Wm"], b["out"], b["inp"], b["Dv"], b["Dm"], n=1, m=2, stream=sl)),
                ]
            elif self.m == 8:  # 2:8, and the 2:4 forms the sparse products read
                calls = [
                    ("prune28", lambda b=b: S.slope_prune_nm(b["W"], b["Wv8"], b["Wm8"], n=2, m=8, stream=sl)),
                    ("expand28", lambda b=b: S.slope_expand_nm_to_24(
                        b["Wv8"], b["Wm8"], b["out"], b["inp"], b["Wv"], b["Wm"], stream=sl)),
                    ("double_prune28", lambda b=b: S.slope_double_prune_nm(
                        b["Wv8"], b["Wm8"], b["out"], b["inp"], b["Dv8"], b["Dm8"], n=2, m=8, stream=sl)),
                    ("expand28_t", lambda b=b: S.slope_expand_nm_to_24(
                        b["Dv8"], b["Dm8"], b["inp"], b["out"], b["Dv"], b["Dm"], stream=sl)),
                ]
            else:
                calls = [
                    ("prune", lambda b=b: S.slope_prune_nm(b["W"], b["Wv"], b["Wm"], stream=sl)),
                    ("double_prune", lambda b=b: S.slope_double_prune(b["Wv"], b["Wm"], b["out"], b["inp"],
                                                                      b["Dv"], b["Dm"], stream=sl)),
                ]
            calls += [
                ("fwd", lambda b=b: S.slope_linear_fwd(b["X"], b["Wv"], b["Wm"], b["L"], b["R"], b["Y"],
                                                       b["XL"], stream=sl)),
            ]
            if not self.wl.forward_only:
                calls += [
                    ("bwd_input", lambda b=b: S.slope_linear_bwd_input(b["dY"], b["Dv"], b["Dm"], b["L"], b["R"],
                                                                       b["dX"], b["G"], stream=sl)),
                    # dW and the adapter gradients dL, dR in one call (one
                    # launch: the dW GEMM computes the two rank-r products too)
                    ("bwd_weight", lambda b=b: S.slope_linear_bwd_weight(
                        b["dY"], b["X"], b["Wm8"] if self.m == 8 else b["Wm"], b["XL"], b["G"], b["dW"],
                        b["dL"], b["dR"], flags=S.DW_NM28 if self.m == 8 else 0,
                        workspace=self.workspaces[li % len(lanes)],
                        stream=sl)),
                ]
                if self.optimizer:  # decayed master values plus the scaled gradient, in place
                    calls += [("axpby", lambda b=b: S.slope_sparse_axpby(
                        0.9999, b["Wmaster"], -1e-3, b["dW"], b["Wmaster"], stream=sl))]
            for name, fn in calls:
                if marks is not None:
                    e0, e1 = marks.new(name, b)
                    e0.record(sl)
                    fn()
                    e1.record(sl)
                else:
                    fn()
        for x in lanes[1:]:
            stream.wait_stream(x)

    def launches_per_step(self):
        import torch

        slots = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count // 2
        n = 0
        for b in self.layers:
            n += 0 if self.wl.forward_only else (1 if self.fused_prune or self.optimizer else 2)  # prune(s)
            n += 2 if self.m == 8 and not self.wl.forward_only else 0  # the two 2:4 forms
            n += 1 if self.optimizer else 0  # beta·A + gamma·B
            r = 0 if b["L"] is None else b["L"].shape[1]  # the layer's own rank (3r when Q, K, V are stacked)
            n += 2 if r else 1  # fwd: (XL) + sparse
            if not self.wl.forward_only:
                n += 2 if r else 1  # bwd_input: (G) + sparse
                pair = (b["out"] // 128) % 2 == 0  # the dW GEMM on CTA pairs
                fuse = r > 0 and r <= 128 and pair  # dL, dR inside the dW launch
                n += 1  # dW
                # the zero-fill before it: on CTA pairs always (the workspace's
                # wave counter, and the outputs the launch adds into); otherwise
                # when its K is split
                if pair or dw_splits(self.wl.tokens, b["inp"], b["out"], slots) > 1:
                    n += 1
                if r and not fuse:
                    n += 3  # zero-fill of dL, dR, then their two GEMMs
        return n


def dw_splits(T: int, inp: int, out: int, slots: int) -> int:
    """Split count the library picks for the pair dW GEMM without the adapter
    (the same round-count model): 256 x 256 output tiles over `slots` SM
    pairs, K = T in blocks of 64."""
    tiles = (out // 256) * ((inp + 255) // 256)
    num_kb = (T + 63) // 64
    best, best_cost = 1, None
    for s in range(1, max(num_kb // 4, 1) + 1):
        waves = (tiles * s + slots - 1) // slots
        per_unit = (num_kb + s - 1) // s + (8 if s > 1 else 4)
        cost = waves * per_unit + (8 if s > 1 else 0)
        if best_cost is None or cost < best_cost:
            best, best_cost = s, cost
    kbs = (num_kb + best - 1) // best
    return (num_kb + kbs - 1) // kbs


class Marks:
    def __init__(self):
        self.pairs = []

    def new(self, name, b):
        import torch

        # external: inside a captured graph these become event-record nodes
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
        # the linears the call computes: one, or Q, K and V stacked
        self.pairs.append((name, b.get("parts", [(b["inp"], b["out"])]), e0, e1))
        return e0, e1


def call_flops(name, T, inp, out, r):
    """Dense-equivalent flops the tensor cores execute in one ABI call: every
    GEMM call runs its main product 2·T·in·out (forward, input gradient,
    weight gradient) and two rank-r products 2·T·r·(in + out) (XL and the
    adapter term; G and the adapter term; dL and dR)."""
    if name in ("fwd", "bwd_input", "bwd_weight"):
        return 2.0 * T * inp * out + 2.0 * T * r * (inp + out)
    return 0.0


def method_flops(name, T, inp, out, r, keep=0.5):
    """The method's own work in one ABI call.  The sparse products count
    their dense-equivalent 2·T·in·out (judged against twice the dense
    peak); the masked weight gradient counts T·in·out, because only the
    kept half of dYᵀ·X is needed (the tensor cores still compute all of
    it); the rank-r products count 2·T·r·(in + out).  `keep` is the
    pattern's density (0.5 for 2:4 and 1:2, 0.25 for 2:8)."""
    if name in ("fwd", "bwd_input"):
        return 2.0 * T * inp * out + 2.0 * T * r * (inp + out)
    if name == "bwd_weight":
        return 2.0 * keep * T * inp * out + 2.0 * T * r * (inp + out)
    return 0.0


def fwd_bytes(T, inp, out, r):
    """Bytes a forward call must move at least: the compressed weight (values
    and metadata, 1.125 B per weight), X in and Y out (bf16), L and R, and XL
    out and back in (hi/lo bf16)."""
    return out * inp * 1.125 + 2.0 * T * (inp + out) + 2.0 * r * (inp + out) + 2 * 4.0 * T * r


def dw_bytes(T, inp, out, r):
    """Bytes a weight-gradient call must move at least: dY and X in (bf16),
    the metadata, the compressed fp32 dW out, XL and G in (hi/lo bf16), and
    dL, dR out (fp32)."""
    return 2.0 * T * (inp + out) + out * inp / 8 + out * inp / 2 * 4 + 2 * 4.0 * T * r + 4.0 * r * (inp + out)


# DRAM bytes (read + write) per launch of the dominant kernel, averaged over
# its launches in one step, from an ncu capture of the same workload
# (dram__bytes_read.sum + dram__bytes_write.sum; outputs a short kernel
# leaves dirty in L2 are not yet written).  Only kernels unchanged since their
# capture are listed.
NCU_TRAFFIC = {("opt-350m-block", "bwd_weight"): 30.44e6,
               # one launch of each linear shape, averaged over the block's six
               ("opt-33b-block-r64", "bwd_weight"): 4.442e9}


def sub_workload(wl, linear):
    """The workload restricted to one of its linears (by name)."""
    keep = tuple(x for x in wl.linears if x.name == linear)
    if not keep:
        raise SystemExit(f"{wl.name} has no linear {linear!r}: {[x.name for x in wl.linears]}")
    return synth.Workload(f"{wl.name}:{linear}", wl.tokens, wl.rank, keep, wl.forward_only)


def pick_peak(clocks, bf16, bf16_sus):
    """The dense bf16 peak a kernel timed inside this run is judged against:
    the sustained figure (measured under the power cap) when the clock
    record of the timed region shows the power cap, else the burst one."""
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    if capped:
        return bf16_sus, "sustained (sw_power_cap seen in the timed region)"
    return bf16, "burst (no power cap seen in the timed region)"


def call_bytes(name, T, inp, out, r):
    if name in ("prune", "prune12"):  # W in; values (half) and metadata out
        return out * inp * (2 + 1 + 0.125)
    if name in ("double_prune", "double_prune12"):
        return out * inp * (1.125 + 1.125)
    if name == "prune28":  # W in; a quarter of the values and the metadata out
        return out * inp * (2 + 0.5 + 0.125)
    if name == "double_prune28":
        return out * inp * (0.625 + 0.625)
    if name in ("expand28", "expand28_t"):  # 2:8 format in, 2:4 form out
        return out * inp * (0.625 + 1.125)
    if name == "prune_double":  # W in once; both compressed formats out
        return out * inp * (2 + 1.125 + 1.125)
    if name == "recompress_double":  # W and the kept metadata in; values, D values and metadata out
        return out * inp * (2 + 0.125 + 1 + 1.125)
    if name == "recompress_frozen":  # W and both metadata in; values and D values out
        return out * inp * (2 + 0.125 + 0.125 + 1 + 1)
    if name == "axpby":  # fp32 master and fp32 compressed dW in, master out
        return out * inp / 2 * (4 + 4 + 4)
    return 0.0


def mma_rates(stream, iters: int = 2048, reps: int = 3):
    """Tensor-core rate self test of the library (resident shared-memory
    operands, N = 256): dense and 2:4-sparse kind::f16 (random legal
    metadata, as pruned weights have; and one fixed pattern) on one SM and
    on SM pairs, dense-equivalent TFLOP/s, best of `reps` launches timed with
    events on `stream`."""
    import torch

    from sparse_rank_adapter_gb300 import slope as S

    out = {}
    with torch.cuda.stream(stream):
        for kind, name in ((0, "dense"), (1, "sparse_fixed_meta"), (2, "sparse")):
            for pair in (False, True):
                S.slope_selftest_mma_rate(kind, pair, 64, stream=stream)  # warm-up
                best = 0.0
                for _ in range(reps):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fl = S.slope_selftest_mma_rate(kind, pair, iters, stream=stream)
                    e1.record(stream)
                    e1.synchronize()
                    best = max(best, fl / (e0.elapsed_time(e1) * 1e-3) / 1e12)
                out[f"{name}_{'pair' if pair else 'one_sm'}"] = round(best, 1)
    S.slope_device_status(stream)
    out["unit"] = "TFLOP/s dense-equivalent, kind::f16 bf16, N = 256, operands resident in shared memory"
    return out


def gpu_arm(args):
    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from sparse_rank_adapter_gb300 import build as B

    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        dist.barrier()
    wl = synth.WORKLOADS[args.workload]
    if args.linear:
        wl = sub_workload(wl, args.linear)
    stream = torch.cuda.Stream(device=dev)
    n_sets = max(1, args.sets)
    sets = [BlockStep(wl, seed=s + 10 * rank, device=dev, fused_prune=args.fused_prune, optimizer=args.optimizer,
                      frozen_columns=args.frozen_columns, pattern=args.pattern, fuse_qkv=args.fuse_qkv)
            for s in range(n_sets)]
    extra = [torch.cuda.Stream(device=dev) for _ in range(min(max(1, args.streams), 8) - 1)]
    for st in sets:
        st.extra_streams = extra
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for st in sets:
            st.prepare(stream)
    # warm-up (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            sets[i % n_sets].run(stream)
    stream.synchronize()

    # Two graphs per input set: a plain one for the timed steps, and one with
    # an event pair around every ABI call (event-record nodes between the
    # kernels), replayed after the timed steps for the per-call breakdown, so
    # that the headline time carries no timing nodes.
    graphs, mgraphs, marks = [], [], []
    for st in sets:
        m = Marks()
        if args.graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                st.run(stream)
            graphs.append(g)
            gm = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gm, stream=stream):
                st.run(stream, m)
            mgraphs.append(gm)
        marks.append(m)
    for i in range(args.warmup):  # warm the graphs too
        if args.graph:
            graphs[i % n_sets].replay()
            mgraphs[i % n_sets].replay()
    torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with clock_sampler(dev, local) as clk:  # samples the timed region only
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                if args.graph:
                    graphs[i % n_sets].replay()
                else:
                    sets[i % n_sets].run(stream)
        t_end.record(stream)
        t_end.synchronize()
    clocks = clk.summary()
    ms_step = t_start.elapsed_time(t_end) / args.steps
    S = sets[0].S
    S.slope_device_status(stream)  # raises if a kernel-side wait ran out during the timed steps

    # Per-call breakdown: `call_reps` marked passes over every input set; a
    # call's time per step is the median over the passes of its summed
    # event times in that pass.  The marked passes issue every call on the
    # step's own stream (with --streams, so that calls do not overlap).
    reps = max(1, args.call_reps)
    per_rep = []  # one {call: ms per step} per pass
    obs = {}  # call -> [(in, out)] of one step, one per linear
    n_calls = {}  # call -> launches of it in one step
    for rep in range(reps):
        with torch.cuda.stream(stream):
            for i in range(n_sets):
                if args.graph:
                    mgraphs[i].replay()
                else:
                    marks[i].pairs.clear()
                    sets[i].run(stream, marks[i])
        stream.synchronize()
        tot = {}
        for m in marks:
            for name, parts, e0, e1 in m.pairs:
                tot[name] = tot.get(name, 0.0) + e0.elapsed_time(e1)
                if rep == 0 and m is marks[0]:
                    obs.setdefault(name, []).extend(parts)  # per linear (algorithmic work and bytes)
                    n_calls[name] = n_calls.get(name, 0) + 1
        per_rep.append({k: v / n_sets for k, v in tot.items()})
    calls_ms = {k: statistics.median(r[k] for r in per_rep) for k in per_rep[0]}
    if world > 1:
        dist.barrier()

    ms_step = max_over_ranks(ms_step, dev)
    fl = flops_per_step(wl)
    value = whole_job_tflops(fl, world, ms_step)

    # roofline of the dominant call
    T, r = wl.tokens, wl.rank
    hbm, bf16, bf16_sus, src = peaks()
    dense_peak, peak_why = pick_peak(clocks, bf16, bf16_sus)
    dom = max(calls_ms, key=calls_ms.get)
    n_launch = n_calls[dom]
    if dom == "fwd" and wl.forward_only and T <= 128:
        # small-batch inference streams the compressed weights: bytes-bound
        byts = sum(fwd_bytes(T, i, o, r) for i, o in obs[dom])
        ach = byts / (calls_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"{src} hbm"}
    elif call_bytes(dom, T, 1, 1, r) > 0:  # a memory-bound call
        alg = sum(call_bytes(dom, T, i, o, r) for i, o in obs[dom])
        ach = alg / (calls_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"{src} hbm"}
    else:
        work = sum(method_flops(dom, T, i, o, r, keep=0.25 if sets[0].m == 8 else 0.5) for i, o in obs[dom])
        ach = work / (calls_ms[dom] * 1e-3) / 1e12
        sparse = dom in ("fwd", "bwd_input")
        peak = dense_peak * (2.0 if sparse else 1.0)
        roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "work_flops_per_step": work,
                "work": ("dense-equivalent 2*T*in*out + 2*T*r*(in+out) per linear, against 2x the dense peak"
                         if sparse else
                         "masked outputs T*in*out + adapter 2*T*r*(in+out) per linear, against the dense peak"),
                "peak_source": f"{src} {'2x ' if sparse else ''}bf16 {peak_why}"}
        if not sparse:
            # what the tensor cores execute: the whole dYᵀ·X product
            exe = sum(call_flops(dom, T, i, o, r) for i, o in obs[dom])
            roof["dense_gemm_achieved"] = exe / (calls_ms[dom] * 1e-3) / 1e12
            roof["dense_gemm_frac"] = roof["dense_gemm_achieved"] / peak
    kernel_of = {"prune": "prune24_kernel (slope_prune_nm)", "double_prune": "double_prune24_kernel (slope_double_prune)",
                 "fwd": "slope_linear_fwd (XL GEMM + sparse GEMM)", "bwd_input": "slope_linear_bwd_input (G GEMM + sparse GEMM)",
                 "bwd_weight": "dW GEMM with dL, dR (slope_linear_bwd_weight)",
                 "prune_double": "prune_double24_kernel (slope_prune_and_double_prune)",
                 "recompress_double": "prune_double24_kernel, kept mask (slope_recompress_double_prune)",
                 "recompress_frozen": "prune_double24_kernel, both masks kept (slope_recompress_frozen)",
                 "axpby": "axpby_kernel (slope_sparse_axpby)",
                 "prune12": "prune12_kernel (slope_prune_nm 1:2)",
                 "double_prune12": "double_prune12_kernel (slope_double_prune_nm 1:2)",
                 "prune28": "prune28_kernel (slope_prune_nm 2:8)",
                 "double_prune28": "double_prune28_kernel (slope_double_prune_nm 2:8)",
                 "expand28": "expand28_kernel (slope_expand_nm_to_24)",
                 "expand28_t": "expand28_kernel (slope_expand_nm_to_24)"}
    # achieved bandwidth of every memory-bound call (algorithmic bytes over its time)
    hbm_calls = {}
    for name, o_ in obs.items():
        byts = sum(call_bytes(name, T, i, o, r) for i, o in o_)
        if byts > 0 and calls_ms.get(name):
            gbs = byts / (calls_ms[name] * 1e-3) / 1e9
            hbm_calls[name] = {"GB/s": round(gbs, 1), "frac": round(gbs / hbm, 3)}
    traffic = NCU_TRAFFIC.get((wl.name, dom))
    if traffic is not None:
        roof["traffic_unit"] = "bytes per launch (dram read + write, ncu)"
        if dom == "bwd_weight":
            roof["algorithmic_bytes"] = sum(dw_bytes(T, i, o, r) for i, o in obs[dom]) / n_launch
    roof.update({"kernel": kernel_of.get(dom, dom), "traffic": traffic, "launches_per_step": n_launch,
                 "call_ms_per_step": round(calls_ms[dom], 4),
                 "call_time": f"median over {reps} marked passes of the step"
                              + (", its calls on one stream" if args.streams > 1 else "")})

    rates = mma_rates(stream) if args.mma_rate else None
    if rates and roof["bound"] == "tensor":
        key = "sparse_pair" if dom in ("fwd", "bwd_input") else "dense_pair"
        roof["frac_of_mma_selftest"] = roof["achieved"] / rates[key]
    e2e = e2e_measure(args, wl, sets[0], stream, dev) if args.e2e else None
    cpu = None
    if rank == 0 and args.cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": "sparse+LoRA linear fwd+bwd TFLOP/s (dense-equiv) and % of 2:4-sparse bf16 peak",
            "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "tokens_per_gpu": wl.tokens, "rank": wl.rank,
                       "outputs": "Y, dX bf16; dW (compressed), dL, dR fp32",
                       "linears": [f"{x.name}:{x.inp}->{x.out}" for x in wl.linears],
                       "l2": f"{n_sets} rotating input sets of {set_bytes(sets[0]) / 2**20:.0f} MiB (> L2 {L2_BYTES // 2**20} MiB)",
                       "graph": bool(args.graph), "parallelism": f"replicas x{world}",
                       "streams": max(1, min(args.streams, 8)),
                       "fuse_qkv": bool(args.fuse_qkv),
                       "prune": ("both masks kept: re-compression, then beta*A + gamma*B"
                                 if args.optimizer and args.frozen_columns
                                 else "kept mask: re-compression + A2, then beta*A + gamma*B" if args.optimizer
                                 else "one call (A1 + A2)" if args.fused_prune else "two calls (A1, A2)"),
                       "pattern": args.pattern + (" (2:8 format; the sparse products on its 2:4 form)"
                                                  if args.pattern == "2:8" else
                                                  " (in the 2:4 format)" if args.pattern == "1:2" else "")},
            "pct_of_sparse_peak": round(100 * value / (2 * bf16), 2),
            "composite_roofline_frac": composite_frac(wl, ms_step, dense_peak),
            "composite_peak": f"{src} bf16 {peak_why}",
            "calls_ms_per_step": {k: round(v, 4) for k, v in calls_ms.items()},
            "hbm_calls": hbm_calls,
            "roofline": roof, "clocks": clocks, "gpu_launches": sets[0].launches_per_step() * args.steps,
            "e2e": e2e, "cpu_baseline": cpu, "mma_rate_selftest": rates,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def set_bytes(st):
    tot = 0
    for b in st.layers:
        for k, v in b.items():
            if hasattr(v, "numel"):
                tot += v.numel() * v.element_size()
    return tot


def composite_frac(wl, ms_step, dense_peak):
    """Time the composite roofline allows (sparse products at 2x the dense
    peak, dense ones at the dense peak) over the measured step time."""
    T, r = wl.tokens, wl.rank
    t = 0.0
    for lin in wl.linears:
        sparse = 2.0 * T * lin.inp * lin.out * (1 if wl.forward_only else 2)
        dense = 0.0 if wl.forward_only else 2.0 * T * lin.inp * lin.out
        if r:
            dense += (2.0 if wl.forward_only else 6.0) * T * r * (lin.inp + lin.out)
        t += sparse / (2 * dense_peak * 1e12) + dense / (dense_peak * 1e12)
    return round(t / (ms_step * 1e-3), 4)


def e2e_measure(args, wl, st, stream, dev):
    """The same step through the C ABI with inputs in pinned host memory:
    host->device copies of every input and device->host copies of every
    result are inside the timed region."""
    import torch

    def pinned_copy(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    host_in, host_out = [], []
    for b in st.layers:
        host_in.append({k: pinned_copy(b[k]) for k in st.input_names() if b[k] is not None})
        host_out.append({k: torch.empty(b[k].shape, dtype=b[k].dtype, pin_memory=True)
                         for k in st.output_names() if b[k] is not None})
    h2d = sum(v.numel() * v.element_size() for d in host_in for v in d.values())
    d2h = sum(v.numel() * v.element_size() for d in host_out for v in d.values())

    # Pipelined per linear, as a caller streaming a block would: one copy
    # stream brings linear i+1's inputs in while linear i computes, another
    # takes linear i's results out.  Events keep each device buffer from
    # being overwritten before the work that reads it is done.
    n_lin = len(st.layers)
    cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(n_lin)]
    ev_done = [torch.cuda.Event() for _ in range(n_lin)]
    ev_out = [torch.cuda.Event() for _ in range(n_lin)]
    started = [False] * n_lin

    def one():
        for i, (b, hi, ho) in enumerate(zip(st.layers, host_in, host_out)):
            if started[i]:
                cin.wait_event(ev_done[i])  # last step's compute has read these inputs
            with torch.cuda.stream(cin):
                for k, v in hi.items():
                    b[k].copy_(v, non_blocking=True)
            ev_in[i].record(cin)
            stream.wait_event(ev_in[i])
            if started[i]:
                stream.wait_event(ev_out[i])  # last step's results of this linear are out
            with torch.cuda.stream(stream):
                st.run(stream, only=i)
            ev_done[i].record(stream)
            cout.wait_event(ev_done[i])
            with torch.cuda.stream(cout):
                for k, v in ho.items():
                    v.copy_(b[k], non_blocking=True)
            ev_out[i].record(cout)
            started[i] = True

    def join():  # the compute stream waits for the last copies out
        for i in range(n_lin):
            stream.wait_event(ev_out[i])

    for _ in range(2):
        one()
    join()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, min(args.steps, 20))
    e0.record(stream)
    cin.wait_event(e0)
    cout.wait_event(e0)
    for _ in range(n):
        one()
    join()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"value": round(flops_per_step(wl) / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}


# ------------------------------------------------------------- CPU arm ----


SLAB_ROWS = 512  # output rows of W per oracle sample unit
SAMPLE_TOKENS = 2048  # token rows of X and dY per oracle sample unit


class OracleSampler:
    """The oracle (as it stands) over row slabs of a workload's weights.

    A unit is one linear restricted to a slab of `SLAB_ROWS` output rows
    (rows of W) on `SAMPLE_TOKENS` tokens: prune the slab, run the forward
    for its output columns, double-prune it (the slab's rows are whole
    groups of the transposed pruning, so its columns of D are exact), add
    its share of the input gradient, and take its rows of dW and columns of
    dR (and the full dL product).  A slab of o of the linear's `out` rows is
    exactly o/out of the linear's work, which is what a unit counts; the
    oracle also recomputes the rank-r products X·L and dY·Rᵀ per slab, which
    is not counted.  Units rotate over the linears and their slabs."""

    def __init__(self, wl):
        from oracle import slope_oracle as O

        self.O = O
        self.wl = wl
        self.T = min(wl.tokens, SAMPLE_TOKENS)
        self.units = []
        for li, lin in enumerate(wl.linears):
            rows = min(SLAB_ROWS, lin.out)
            for o0 in range(0, lin.out - rows + 1, rows):
                self.units.append((li, lin, o0, rows))
        # rotate linears first, so a short sample still touches every shape
        self.units.sort(key=lambda u: (u[2], u[0]))
        self.cache = {}
        self.next = 0

    def inputs(self, li, lin, o0, rows):
        key = (li, o0)
        if key not in self.cache:
            T, r = self.T, self.wl.rank
            X = synth.normal_bf16(1, li, "X", (T, lin.inp))
            d = {"X": X, "W": synth.normal_bf16(1 + o0, li, "W", (rows, lin.inp)),
                 "dY": synth.normal_bf16(1 + o0, li, "dY", (T, rows)),
                 "L": synth.normal_bf16(1, li, "L", (lin.inp, r)) if r else None,
                 "R": synth.normal_bf16(1 + o0, li, "R", (r, rows)) if r else None}
            if len(self.cache) > 64:
                self.cache.clear()
            self.cache[key] = d
        return self.cache[key]

    def unit_flops(self, lin, rows):
        one = synth.Workload(self.wl.name, self.T, self.wl.rank, (lin,), self.wl.forward_only)
        return flops_per_step(one) * rows / lin.out

    def run(self, budget_s: float, min_units: int = 1):
        """Units until `budget_s` seconds of oracle time (at least
        `min_units`); returns (flops counted, seconds, units done)."""
        O = self.O
        done, t_total, n = 0.0, 0.0, 0
        while n < min_units or t_total < budget_s:
            li, lin, o0, rows = self.units[self.next % len(self.units)]
            self.next += 1
            d = self.inputs(li, lin, o0, rows)
            s = time.perf_counter()
            vals, meta, _ = O.prune24(d["W"])
            O.linear_fwd(d["X"], vals, meta, d["L"], d["R"])
            if not self.wl.forward_only:
                tv, tm, _ = O.double_prune24(vals, meta, rows, lin.inp)
                O.linear_bwd_input(d["dY"], tv, tm, d["L"], d["R"])
                O.linear_bwd_weight(d["dY"], d["X"], meta, d["L"], d["R"])
            t_total += time.perf_counter() - s
            done += self.unit_flops(lin, rows)
            n += 1
        return done, t_total, n

    def describe(self, n):
        wl = self.wl
        steps = "prune, forward" if wl.forward_only else "prune, double prune, forward, both gradients"
        return (f"{n} units of {wl.name}: row slabs of up to {SLAB_ROWS} output rows of each of its "
                f"{len(wl.linears)} weights ({steps}) on {self.T} of {wl.tokens} tokens, counted as "
                f"their exact share of the workload's flops; oracle fp64 NumPy")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def one_core_sample(wl_name, linear, budget_s):
    """The same oracle sample in a child process held to one core (BLAS
    threads 1, CPU affinity one core); returns its JSON dict or None."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               VECLIB_MAXIMUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", wl_name,
           "--oracle-sample", str(budget_s)]
    if linear:
        cmd += ["--linear", linear]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 4 + 300)
        if res.returncode == 0:
            return json.loads(res.stdout.strip().splitlines()[-1])
    except Exception:
        pass
    return None


def cpu_baseline(wl, budget_s):
    """The oracle on all host cores, and on one core (a child process)."""
    smp = OracleSampler(wl)
    smp.run(0.0, 1)  # warm-up: first-touch costs and input generation
    done, secs, n = smp.run(budget_s)
    out = {"value": round(done / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_cores(),
           "kind": "oracle", "sample": smp.describe(n), "seconds": round(secs, 2)}
    name, _, linear = wl.name.partition(":")
    one = one_core_sample(name, linear, budget_s)
    if one is not None:
        out["one_core"] = {"value": one["value"], "unit": "TFLOP/s", "cores": 1, "sample": one["sample"],
                           "seconds": one["seconds"]}
    return out


def oracle_sample_child(args):
    """--oracle-sample: time the oracle alone on this process's first
    allowed core and print one JSON line (used for the one-core figure)."""
    try:
        core = sorted(os.sched_getaffinity(0))[0]
        os.sched_setaffinity(0, {core})
    except Exception:
        pass
    wl = synth.WORKLOADS[args.workload]
    if args.linear:
        wl = sub_workload(wl, args.linear)
    smp = OracleSampler(wl)
    smp.run(0.0, 1)
    done, secs, n = smp.run(args.oracle_sample)
    print(json.dumps({"value": round(done / secs / 1e12, 6), "seconds": round(secs, 2),
                      "sample": smp.describe(n), "cores": 1}), flush=True)


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    if args.linear:
        wl = sub_workload(wl, args.linear)
    smp = OracleSampler(wl)
    tot_flops, tot_s, n_units = 0.0, 0.0, 0
    for i in range(args.warmup + args.steps):
        if i < args.warmup:  # warm-up steps: one unit each, untimed
            smp.run(0.0, 1)
            continue
        f, s, n = smp.run(args.ref_seconds)
        tot_flops += f
        tot_s += s
        n_units += n
    value = tot_flops / tot_s / 1e12
    desc = smp.describe(n_units) + f"; {args.steps} steps of about {args.ref_seconds:g} s"
    line = {
        "impl": "reference",
        "metric": "sparse+LoRA linear fwd+bwd TFLOP/s (dense-equiv) and % of 2:4-sparse bf16 peak",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * tot_s / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "tokens_per_gpu": wl.tokens, "rank": wl.rank},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def tiling_study(args):
    """SLoPe §2.4 / App. E split the "upsample" weights (FC1: d -> 4d) into
    square tiles to avoid a dip of the sparse product's speed-up at some
    dimensions.  This times, on this library's kernels, each FC1 forward as
    one call against its four square d x d row tiles (four calls, each
    writing its own T x d output), for the OPT hidden sizes and token
    counts; rank 0 (the sparse product alone), weights pre-compressed, L2
    flushed before every timed call, median of `reps` calls.  Prints one
    JSON line."""
    import torch

    from sparse_rank_adapter_gb300 import build as B
    from sparse_rank_adapter_gb300 import slope as S

    B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    reps = 10

    def timed(fn):
        out = []
        with torch.cuda.stream(stream):
            for i in range(reps + 2):
                flush.fill_(i & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    out.append(e0.elapsed_time(e1))
        return statistics.median(out)

    rows = []
    for d in (2560, 4096, 7168, 9216):
        W = synth.device_normal_bf16((4 * d, d), 0.02, d, dev)
        Wv = torch.empty(4 * d, d // 2, dtype=torch.bfloat16, device=dev)
        Wm = torch.empty(4 * d, d // 8, dtype=torch.uint8, device=dev)
        S.slope_prune_nm(W, Wv, Wm, stream=stream)
        tiles = [(Wv[k * d:(k + 1) * d], Wm[k * d:(k + 1) * d]) for k in range(4)]
        del W
        for T in (16, 2048, 16384):
            X = synth.device_normal_bf16((T, d), 1.0, d + T, dev)
            Y = torch.empty(T, 4 * d, dtype=torch.bfloat16, device=dev)
            Yk = [torch.empty(T, d, dtype=torch.bfloat16, device=dev) for _ in range(4)]
            one = timed(lambda: S.slope_linear_fwd(X, Wv, Wm, None, None, Y, stream=stream))

            def four():
                for (v, m), y in zip(tiles, Yk):
                    S.slope_linear_fwd(X, v, m, None, None, y, stream=stream)

            sq = timed(four)
            flops = 2.0 * T * d * 4 * d
            rows.append({"d": d, "T": T, "one_call_ms": round(one, 4), "square_tiles_ms": round(sq, 4),
                         "tiles_over_one": round(sq / one, 3),
                         "one_call_tflops": round(flops / (one * 1e-3) / 1e12, 1)})
            del X, Y, Yk
        del Wv, Wm, tiles
    S.slope_device_status(stream)
    print(json.dumps({"study": "FC1 (d -> 4d) forward: one call vs four square d x d tiles",
                      "source": "SLoPe §2.4 and App. E (weight tiling)", "unit": "ms", "rank": 0,
                      "pattern": "2:4", "timing": f"median of {reps} calls, L2 flushed before each",
                      "rows": rows}), flush=True)


def free_port():
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_replicas(n, argv):
    """Runs this script as n processes, one per GPU, with the environment a
    torchrun launch would give them; returns the first non-zero exit code
    (0 if every rank succeeded).  Only rank 0 prints."""
    port = free_port()
    procs = []
    for rank in range(n):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        out = None if rank == 0 else subprocess.DEVNULL
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + list(argv), env=env,
                                      stdout=out))
    rcs = [p.wait() for p in procs]
    return next((rc for rc in rcs if rc != 0), 0)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="slope", choices=["slope", "reference"])
    ap.add_argument("--workload", default="opt-33b-block-r64", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--linear", default="", help="keep only this linear of the block (e.g. fc1)")
    ap.add_argument("--sets", type=int, default=4, help="rotating input sets (L2 defeat)")
    ap.add_argument("--call-reps", type=int, default=5,
                    help="marked passes for the per-call breakdown (median)")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle seconds of the GPU arm's cpu_baseline (all cores, then one core)")
    ap.add_argument("--ref-seconds", type=float, default=6.0,
                    help="oracle seconds per step of --impl reference")
    ap.add_argument("--oracle-sample", type=float, default=0.0, help=argparse.SUPPRESS)
    ap.add_argument("--no-mma-rate", dest="mma_rate", action="store_false",
                    help="skip the tensor-core rate self test")
    ap.add_argument("--optimizer", action="store_true",
                    help="training step with the mask kept from initialisation: re-compression + A2 "
                         "(slope_recompress_double_prune) in place of A1, A2, and beta*A + gamma*B "
                         "(slope_sparse_axpby) on an fp32 master copy")
    ap.add_argument("--frozen-columns", action="store_true",
                    help="with --optimizer: the column mask kept from initialisation too "
                         "(slope_recompress_frozen in place of the re-compression + A2)")
    ap.add_argument("--fuse-qkv", action="store_true",
                    help="Q, K and V of the block read one X and run as one call each on their stacked "
                         "weights (rank-3r adapter, block-diagonal R; in training the dX call sums theirs)")
    ap.add_argument("--fused-prune", action="store_true",
                    help="A1 and A2 through the one-call slope_prune_and_double_prune")
    ap.add_argument("--streams", type=int, default=1,
                    help="issue the block's independent linears on this many streams")
    ap.add_argument("--tiling-study", action="store_true",
                    help="time FC1 forwards as one call against four square tiles (one JSON line)")
    ap.add_argument("--pattern", default="2:4", choices=["2:4", "1:2", "2:8"],
                    help="N:M pattern of the weights (1:2 in the 2:4 format; 2:8 with its 2:4 form)")
    args = ap.parse_args()
    if args.pattern != "2:4" and (args.fused_prune or args.optimizer):
        ap.error("--pattern 1:2 / 2:8 runs the plain training step (no --fused-prune, --optimizer)")
    if args.fuse_qkv:
        wl0 = synth.WORKLOADS[args.workload]
        if args.linear or [x.name for x in wl0.linears[:3]] != ["q", "k", "v"]:
            ap.error("--fuse-qkv applies to a whole block (Q, K, V first)")
        if args.optimizer or args.pattern != "2:4":
            ap.error("--fuse-qkv runs the plain 2:4 step (no --optimizer, --pattern)")
    if args.warmup < 3:
        args.warmup = 3
    if args.oracle_sample > 0:
        oracle_sample_child(args)
        return
    if args.tiling_study:
        tiling_study(args)
        return
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus, sys.argv[1:]))
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
