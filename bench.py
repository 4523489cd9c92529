#!/usr/bin/env python
"""Benchmark of the tensor-parallel MLP block on one GB300 (per GPU).

Workload (one "step" = one pass of the whole hot path): the Megatron MLP
block, forward and backward, with p = 4 shards held in one GPU's memory,
4096 tokens, h = 4096, ffn = 16384 -- FC1 column-parallel [4096, 4096] per
shard with GeLU, FC2 row-parallel [4096, 4096] per shard with the fused
AllReduce, then FC2's backward (dZ_k = dY W2_k^T * GeLU'(H_k), dW2_k) and
FC1's backward (the fused dX = sum_k dZ_k W1_k^T, dW1_k).  Six GEMMs, 3.30
TFLOP per step, in five ABI calls and five launches: FC2's backward is one
call whose two products share one launch.  Inputs: X N(0,1), dY N(0,1), weights N(0, 0.02), bf16,
drawn by the seeded generator.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --sweep      # chunk_m sweep report (GPT-3-scale FC pair)

Prints one JSON line.  ``value`` is TFLOP/s of the whole job with inputs
resident in HBM; ``e2e`` is the same through the C-ABI with host buffers:
the weights stay on the device like a model's parameters, and every step's
data (X, dY) is uploaded from pinned host memory and its results (Y, dX)
downloaded inside the timed region.  ``e2e_streamed_weights`` also moves
W1, W2 up and dW1, dW2 down every step.  ``--impl reference`` times the CPU oracle on a bounded token sample
of the same workload instead.  With N > 1 (torchrun, one rank per GPU) every
rank runs an independent replica (the path has no cross-GPU exchange on one
box) and ``value`` is the sum over ranks of the work divided by the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import signal
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded GEMM+reduce TFLOP/s and % of GB300 dense BF16 peak (1 GPU)"
P, M, H, FFN = 4, 4096, 4096, 16384
NK = FFN // P
GEMM_FLOPS = 2.0 * M * H * NK * P            # every one of the six GEMMs
STEP_FLOPS = 6 * GEMM_FLOPS
WORKLOAD = (f"Megatron MLP block fwd+bwd, p={P}: tokens {M}, h={H}, ffn={FFN}; FC1 column-parallel "
            f"[{H},{NK}]/shard + GeLU, FC2 row-parallel [{NK},{H}]/shard with fused AllReduce; "
            f"backward: FC2 dZ (GeLU') + dW2, FC1 fused dX reduce + dW1")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["gemm_reduce_fusion_gb300/csrc/gemm_kernel.cuh", "gemm_reduce_fusion_gb300/csrc/ptx.cuh",
                  "gemm_reduce_fusion_gb300/csrc/tp_fused.cu"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the end-to-end run (host buffers, copies overlapped with compute); "
                         "0: as many as --steps, so both runs see the same sustained clocks")
    ap.add_argument("--sweep", action="store_true",
                    help="chunk_m sweep of the GPT-3-scale FC pair: fused time vs the timeline model")
    ap.add_argument("--configs", action="store_true",
                    help="one JSON line per workload (all five), TFLOP/s and roofline fraction")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="leave out the per-workload table of the headline line")
    ap.add_argument("--workload-steps", type=int, default=20,
                    help="timed steps per workload in the headline line's workload table")
    ap.add_argument("--tile-mode", type=int, default=0, choices=[0, 1, 2],
                    help="0: planner chooses 128x256 or CTA-pair 256x256 tiles; 1: 128x256 only; 2: pairs")
    ap.add_argument("--profile-case", action="store_true",
                    help="run each GEMM variant of the step twice at the step's shapes (for ncu)")
    ap.add_argument("--profile-workload", default="", metavar="NAME",
                    help="set up one workload of --configs and run its calls twice (for ncu)")
    ap.add_argument("--trace", action="store_true",
                    help="per-chunk timeline of single fused launches (the two-engine timeline, measured)")
    ap.add_argument("--precision-report", action="store_true",
                    help="output error of the fused path vs the unfused baseline with fp32 or bf16 collectives")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------------ distributed plumbing

def dist_init(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def aggregate_value(flops_per_step: float, steps: int, world: int, t_max_ms: float) -> float:
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's time."""
    return flops_per_step * steps * world / (t_max_ms / 1e3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.send_signal(signal.SIGTERM)
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ the step

class MLPStep:
    """Device buffers and the five ABI calls of one MLP fwd+bwd step."""

    def __init__(self, tp, torch, host):
        bf = dict(dtype=torch.bfloat16, device="cuda")
        self.tp = tp
        self.torch = torch
        self.X = torch.empty((M, H), **bf)
        self.W1 = [torch.empty((H, NK), **bf) for _ in range(P)]
        self.W2 = [torch.empty((NK, H), **bf) for _ in range(P)]
        self.DY = torch.empty((M, H), **bf)
        self.Z = [torch.empty((M, NK), **bf) for _ in range(P)]
        self.Hp = [torch.empty((M, NK), **bf) for _ in range(P)]
        self.Y = torch.empty((M, H), **bf)
        self.DZ = [torch.empty((M, NK), **bf) for _ in range(P)]
        self.DW2 = [torch.empty((NK, H), **bf) for _ in range(P)]
        self.DX = torch.empty((M, H), **bf)
        self.DW1 = [torch.empty((H, NK), **bf) for _ in range(P)]
        need = max(tp.tp_workspace_size(op, P, mm, nn, kk, 0) for op, mm, nn, kk in [
            (tp.TP_OP_COL_FWD, M, NK, H), (tp.TP_OP_ROW_AR, M, H, NK),
            (tp.TP_OP_ROW_BWD, M, H, NK), (tp.TP_OP_COL_BWD, M, NK, H)])
        self.ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        self.upload(host)

    def inputs(self):
        return [self.X, *self.W1, *self.W2, self.DY]

    def outputs(self):
        return [self.Y, self.DX, *self.DW1, *self.DW2]

    def data_inputs(self):
        """What changes from step to step: the activation X and the gradient dY."""
        return [self.X, self.DY]

    def data_outputs(self):
        """What the step hands on: the output Y and the input gradient dX."""
        return [self.Y, self.DX]

    def upload(self, host):
        for d, h in zip(self.inputs(), host):
            d.copy_(h, non_blocking=True)

    def upload_data(self, host):
        for d, h in zip(self.data_inputs(), [host[0], host[-1]]):
            d.copy_(h, non_blocking=True)

    def calls(self):
        tp, ws = self.tp, self.ws
        return [
            ("col_fwd_gelu", lambda: tp.tp_col_linear_fwd(self.X, self.W1, self.Z, ws, epi=tp.TP_EPI_GELU,
                                                          preact=self.Hp)),
            ("row_fwd_allreduce", lambda: tp.tp_row_linear_fwd_allreduce(self.Z, self.W2, [self.Y], ws)),
            ("row_bwd", lambda: tp.tp_row_linear_bwd(self.Z, self.W2, self.DY, self.DZ, self.DW2, ws,
                                                     preact=self.Hp)),
            ("col_bwd_dx", lambda: tp.tp_col_linear_bwd(None, self.W1, self.DZ, self.DX, None, ws)),
            ("col_bwd_dw", lambda: tp.tp_col_linear_bwd(self.X, self.W1, self.DZ, None, self.DW1, ws)),
        ]


# which kernel variant each call launches (one launch per call at these
# sizes) and the GEMMs it computes.  The row backward is one call for dZ and
# dW2, which the library runs as one launch of both products (2 x 13.5 waves
# as 27); the column backward's two products would run as two launches even
# from one call (its fused makespan is longer), so the step issues them as two
# calls and each is timed on its own.
CALL_KERNEL = {
    "col_fwd_gelu": ("tp_gemm_pair_kernel<0,1,128,0> (X.W, 256x256 tiles on CTA pairs)", 1),
    "row_fwd_allreduce": ("tp_gemm_pair_kernel<0,1,128,1> (X.W, 256x256 tiles on CTA pairs, last wave in k-slices)", 1),
    "row_bwd": ("tp_gemm_pair2_kernel<0,0,1,1,128> (dY.W^T with GeLU' then X^T.dY, one launch on CTA pairs)", 2),
    "col_bwd_dx": ("tp_gemm_pair_kernel<0,0,128,1> (dY.W^T, 256x256 tiles on CTA pairs, last wave in k-slices)", 1),
    "col_bwd_dw": ("tp_gemm_pair_kernel<1,1,128,0> (X^T.dY, 256x256 tiles on CTA pairs)", 1),
}


def host_inputs(torch):
    import synth
    gen = [synth.normal_bf16((M, H), synth.seed_for(1, 0), 1.0)]
    gen += [synth.normal_bf16((H, NK), synth.seed_for(1, 1 + k), 0.02) for k in range(P)]
    gen += [synth.normal_bf16((NK, H), synth.seed_for(1, 5 + k), 0.02) for k in range(P)]
    gen += [synth.normal_bf16((M, H), synth.seed_for(1, 9), 1.0)]
    import numpy as np
    out = []
    for a in gen:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        out.append(t.pin_memory() if torch.cuda.is_available() else t)
    return out


# ------------------------------------------------------------------ CPU oracle leg

def oracle_step(x, w1, w2, dy):
    """The same MLP step in the fp64 oracle on the given token sample."""
    import oracle
    z, h = oracle.col_fwd(x, w1, apply_gelu=True)
    zb = [oracle.round_bf16(a) for a in z]
    hb = [oracle.round_bf16(a) for a in h]
    oracle.row_fwd_allreduce(zb, w2)
    dz = oracle.row_bwd_dx(w2, dy, preacts=hb)
    oracle.row_bwd_dw(zb, dy)
    dzb = [oracle.round_bf16(a) for a in dz]
    oracle.col_bwd_dx(w1, dzb)
    oracle.col_bwd_dw(x, dzb)


def cpu_inputs(tokens):
    import synth
    x = synth.normal_bf16((M, H), synth.seed_for(1, 0), 1.0)[:tokens]
    w1 = [synth.normal_bf16((H, NK), synth.seed_for(1, 1 + k), 0.02) for k in range(P)]
    w2 = [synth.normal_bf16((NK, H), synth.seed_for(1, 5 + k), 0.02) for k in range(P)]
    dy = synth.normal_bf16((M, H), synth.seed_for(1, 9), 1.0)[:tokens]
    return x, w1, w2, dy


def cpu_baseline(target_s=12.0):
    """Time the oracle on a token sample sized for about `target_s` seconds
    (the sample grows until one timed step takes at least half of that)."""
    tokens = 64
    x, w1, w2, dy = cpu_inputs(M)
    while True:
        t0 = time.perf_counter()
        oracle_step(x[:tokens], w1, w2, dy[:tokens])
        dt = time.perf_counter() - t0
        if dt >= target_s / 2 or tokens >= M:
            break
        tokens = int(min(M, max(2 * tokens, tokens * target_s / max(dt, 1e-3))) // 64 * 64)
    flops = STEP_FLOPS * tokens / M
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"one MLP fwd+bwd step over {tokens} of the {M} tokens with the full weights "
                      f"(fp64 numpy oracle, {dt:.1f} s, {flops / 1e9:.0f} GFLOP)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    tokens = 64
    x, w1, w2, dy = cpu_inputs(tokens)
    for _ in range(args.warmup):
        oracle_step(x, w1, w2, dy)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(x, w1, w2, dy)
    dt = time.perf_counter() - t0
    flops = STEP_FLOPS * tokens / M
    v = flops * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded splitmix64 normals)",
            "config": {"workload": WORKLOAD, "sample_tokens": tokens},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"each step: the MLP fwd+bwd over {tokens} of the {M} tokens, full weights"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU leg

def _dist(v):
    """median, min and p90 of a list of per-step times."""
    s = sorted(v)
    return s[len(s) // 2], s[0], s[int(0.9 * (len(s) - 1))]


def choose_peak(pk, src, clocks):
    """The bf16 roofline denominator for what the timed region saw: the
    measured burst peak while no sample showed the power cap (the SM clock at
    its maximum), the measured sustained peak once sw_power_cap was seen."""
    burst = pk.get("bf16_tflops", FALLBACK["bf16_tflops"])
    sust = pk.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    if capped:
        return sust, f"{src} bf16 dense, sustained: sw_power_cap was active during the timed region"
    return burst, (f"{src} bf16 dense, burst: no sw_power_cap sample during the timed region "
                   f"(SM clock median {clocks.get('sm_mhz')} of max {clocks.get('sm_max_mhz')} MHz)")


def run_ours(args):
    import torch
    rank, world, local = dist_init(args.gpus)
    torch.cuda.set_device(local)
    import gemm_reduce_fusion_gb300 as tp

    host = host_inputs(torch)
    step = MLPStep(tp, torch, host)
    calls = step.calls()
    stream = torch.cuda.current_stream()

    for _ in range(max(3, args.warmup)):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    st = tp.tp_get_device_status(step.ws)
    if st != tp.TP_OK:
        raise RuntimeError(f"device status after warm-up: {tp.tp_status_string(st)}")

    # Headline: K steps back to back, events at step boundaries only (no
    # event between the launches of a step, which keeps the programmatic
    # dependent launch overlap of consecutive kernels intact).
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for k in range(K):
            for _, fn in calls:
                fn()
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = clk.summary()
    total_ms = ev[0].elapsed_time(ev[K])
    step_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(K)]
    med, mn, p90 = _dist(step_ms)

    # Per-call durations, in a separate pass of K steps with an event around
    # every launch (used for the dominant kernel's roofline only).
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
    torch.cuda.synchronize()
    for k in range(K):
        evc[k][0].record(stream)
        for i, (_, fn) in enumerate(calls):
            fn()
            evc[k][i + 1].record(stream)
    torch.cuda.synchronize()
    per_call = {name: 0.0 for name, _ in calls}
    for k in range(K):
        for i, (name, _) in enumerate(calls):
            per_call[name] += evc[k][i].elapsed_time(evc[k][i + 1])
    st = tp.tp_get_device_status(step.ws)
    if st != tp.TP_OK:
        raise RuntimeError(f"device status after timing: {tp.tp_status_string(st)}")

    t_max = max_over_ranks(total_ms, world)
    value = aggregate_value(STEP_FLOPS, K, world, t_max)

    # dominant kernel variant: the one with the largest total time
    per_kernel = {}
    for name, ms in per_call.items():
        kname, gemms = CALL_KERNEL[name]
        d = per_kernel.setdefault(kname, {"ms": 0.0, "launches": 0, "gemms": gemms})
        d["ms"] += ms
        d["launches"] += K
    dom = max(per_kernel, key=lambda n: per_kernel[n]["ms"])
    dom_avg_s = per_kernel[dom]["ms"] / per_kernel[dom]["launches"] / 1e3
    dom_flops = GEMM_FLOPS * per_kernel[dom]["gemms"]
    pk, src = peaks()
    peak, peak_why = choose_peak(pk, src, clocks)
    burst = pk.get("bf16_tflops", FALLBACK["bf16_tflops"])
    sust = pk.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"])
    achieved = dom_flops / dom_avg_s / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": peak_why,
                "frac_of_burst": achieved / burst, "frac_of_sustained": achieved / sust,
                "traffic": dram_traffic(dom),
                "per_call_ms": {n: per_call[n] / K for n in per_call},
                "per_call_pass": f"a separate pass of {K} steps with an event around every launch",
                "dominant_launches_per_step": per_kernel[dom]["launches"] // K,
                "algorithmic_flops_per_launch": dom_flops,
                "value_frac_of_peak": value / world / peak,
                "value_frac_of_burst": value / world / burst,
                "value_frac_of_sustained": value / world / sust}

    # End to end through the ABI with host buffers, double-buffered: two
    # device buffer sets alternate, so step i+1's upload (copy stream) and
    # step i-1's download (second copy stream) overlap step i's kernels.
    # Headline: the weights live on the device like a model's parameters
    # (uploaded once, before timing); every step uploads its data (X, dY)
    # from pinned host memory and downloads its results (Y, dX).  Context:
    # the same with W1, W2 uploaded and dW1, dW2 downloaded every step too.
    E = max(1, args.e2e_steps if args.e2e_steps > 0 else args.steps)
    steps = [step, MLPStep(tp, torch, host)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()

    def e2e_run(n, streamed):
        outs = [st.outputs() if streamed else st.data_outputs() for st in steps]
        houts = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs[0]]
        done_up = [torch.cuda.Event() for _ in range(n)]
        done_comp = [torch.cuda.Event() for _ in range(n)]
        done_down = [torch.cuda.Event() for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(up)
        for i in range(n):
            st = steps[i % 2]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(done_comp[i - 2])     # this buffer set's previous step is done
                if streamed:
                    st.upload(host)
                else:
                    st.upload_data(host)
                done_up[i].record(up)
            comp.wait_event(done_up[i])
            if i >= 2:
                comp.wait_event(done_down[i - 2])       # its outputs have left the device
            for _, fn in st.calls():
                fn()
            done_comp[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done_comp[i])
                for h, d in zip(houts, outs[i % 2]):
                    h.copy_(d, non_blocking=True)
                done_down[i].record(down)
        t1.record(down)
        torch.cuda.synchronize()
        nb_in = sum(t.numel() * t.element_size() for t in (st.inputs() if streamed else st.data_inputs()))
        nb_out = sum(t.numel() * t.element_size() for t in houts)
        return t0.elapsed_time(t1), nb_in, nb_out

    for st in steps:                                     # resident weights
        st.upload(host)
    torch.cuda.synchronize()
    e2e_run(2, False)
    barrier(world)
    e2e_ms, h2d, d2h = e2e_run(E, False)
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e_run(2, True)
    barrier(world)
    s_ms, s_h2d, s_d2h = e2e_run(E, True)
    s_ms = max_over_ranks(s_ms, world)
    barrier(world)
    e2e = {"value": aggregate_value(STEP_FLOPS, E, world, e2e_ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": E,
           "ms_per_step": e2e_ms / E,
           "how": "weights resident on the device (uploaded once); every step uploads X and dY from pinned "
                  "host memory and downloads Y and dX, on two copy streams overlapping the kernels of the "
                  "neighbouring steps (double-buffered)"}
    e2e_streamed = {"value": aggregate_value(STEP_FLOPS, E, world, s_ms), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": s_h2d, "d2h_bytes_per_step": s_d2h, "steps": E,
                    "ms_per_step": s_ms / E,
                    "how": "as e2e, but W1 and W2 are also uploaded and dW1 and dW2 downloaded every step"}

    if rank != 0:
        return
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": t_max / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded splitmix64 normals: X, dY N(0,1); weights N(0,0.02))",
            "config": {"workload": WORKLOAD, "p": P, "tokens": M, "h": H, "ffn": FFN,
                       "flops_per_step": STEP_FLOPS, "chunk_m": "scheduler (0)",
                       "l2": "no flush: every step streams inputs larger than L2 "
                             "(X 32 MiB, W1 128 MiB, W2 128 MiB, dY 32 MiB, 129 MB L2)",
                       "parallelism": f"{world} independent replica(s), all {P} ranks on each GPU"},
            "roofline": roofline, "clocks": clocks, "e2e": e2e, "e2e_streamed_weights": e2e_streamed,
            "gpu_launches": len(calls) * K}
    line.update({"ms_per_step_median": med, "ms_per_step_min": mn, "ms_per_step_p90": p90,
                 "timing": "CUDA events at step boundaries on the launching stream; value = work of all "
                           "K steps / their total time; median, min and p90 over the K steps"})
    if world == 1 and not args.no_workloads:
        del step, calls
        torch.cuda.empty_cache()
        headline = {"ms_median": med, "ms_min": mn, "ms_p90": p90, "steps": K,
                    "tflops": STEP_FLOPS / (med / 1e3) / 1e12, "peak": peak, "clocks": clocks}
        line["workloads"] = workload_table(torch, tp, args, pk, src, headline)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
        line["cpu_baseline"]["per_core"] = cpu_rate_one_core()
    print(json.dumps(line), flush=True)


# Targets per workload: fraction of the dense bf16 peak for the tensor-bound
# ones, of the measured HBM copy bandwidth for the decode-like one; the
# worked example is a parity and latency case, reported as % of HBM.
WORKLOAD_TABLE = [
    ("worked_example_p2", "hbm", None),
    ("mlp_block_p4", "tensor", 0.70),
    ("mha_projections_p4", "tensor", 0.70),
    ("sp_pair_fwd_p8", "tensor", 0.70),
    ("gpt3_mlp_p8_m2048", "tensor", 0.70),
    ("gpt3_mlp_p8_m16", "hbm", 0.60),
]


def _time_steps(torch, calls, steps, warmup, flush_buf=None):
    """Per-step ms of the calls: back to back with events at step boundaries,
    or, with flush_buf, each step timed alone after the L2 is overwritten."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    if flush_buf is None:
        ev[0].record(stream)
        for k in range(steps):
            for _, fn in calls:
                fn()
            ev[k + 1].record(stream)
        torch.cuda.synchronize()
        return [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    for k in range(steps):
        flush_buf.fill_(float(k))
        ev[2 * k].record(stream)
        for _, fn in calls:
            fn()
        ev[2 * k + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(steps)]


def workload_table(torch, tp, args, pk, src, headline):
    """Every workload at full size, timed like the headline (median, min and
    p90 over --workload-steps steps), each against its roofline: TFLOP/s as
    a fraction of the bf16 peak chosen from the clocks seen during this pass,
    or GB/s as a fraction of the measured HBM copy bandwidth (L2 flushed
    before each step)."""
    table = dict(workloads(torch, tp))
    flush = torch.empty(256 << 20, dtype=torch.float32, device="cuda")   # 1 GiB > 2 x L2
    hbm = pk.get("hbm_gbs", FALLBACK["hbm_gbs"])
    out, raw = {}, {}
    with ClockSampler(torch.cuda.current_device()) as clk:
        for name, bound, target in WORKLOAD_TABLE:
            if name == "mlp_block_p4":
                continue
            w = table[name]()
            ms = _time_steps(torch, w["calls"], args.workload_steps, 3, flush if w["flush"] else None)
            graph_ms = None
            if name == "worked_example_p2":
                # the same step captured once in a CUDA graph and replayed: the
                # calls' device time without the host's per-call work
                g = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        for _, fn in w["calls"]:
                            fn()
                torch.cuda.current_stream().wait_stream(s)
                graph_ms = _time_steps(torch, [("graph", g.replay)], args.workload_steps, 3,
                                       flush if w["flush"] else None)
                del g
            st = tp.tp_get_device_status(w["ws"])
            if st != tp.TP_OK:
                raise RuntimeError(f"{name}: device status {tp.tp_status_string(st)}")
            raw[name] = ({k: w.get(k) for k in ("desc", "flops", "bytes", "flush")}, ms, graph_ms)
            del w
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
    clocks = clk.summary()
    peak, why = choose_peak(pk, src, clocks)
    for name, bound, target in WORKLOAD_TABLE:
        if name == "mlp_block_p4":
            h = headline
            e = {"desc": WORKLOAD, "bound": "tensor", "ms_median": h["ms_median"], "ms_min": h["ms_min"],
                 "ms_p90": h["ms_p90"], "steps": h["steps"], "tflops": h["tflops"],
                 "peak_tflops": h["peak"], "frac_of_peak": h["tflops"] / h["peak"],
                 "l2": "inputs larger than L2", "timed_in": "the headline run above"}
            e["target"] = f">= {target} of the dense bf16 peak"
            e["meets_target"] = e["frac_of_peak"] >= target
            out[name] = e
            continue
        w, ms, graph_ms = raw[name]
        med, mn, p90 = _dist(ms)
        e = {"desc": w["desc"], "bound": bound, "ms_median": med, "ms_min": mn, "ms_p90": p90,
             "steps": len(ms), "flops_per_step": w["flops"], "tflops": w["flops"] / (med / 1e3) / 1e12,
             "l2": "flushed before each step" if w["flush"] else "inputs larger than L2"}
        e["peak_tflops"] = peak
        e["frac_of_peak"] = e["tflops"] / peak
        if w.get("bytes"):
            e["bytes_per_step"] = w["bytes"]
            e["hbm_gbs"] = w["bytes"] / (med / 1e3) / 1e9
            e["frac_of_hbm"] = e["hbm_gbs"] / hbm
        if graph_ms is not None:
            gmed, gmn, _ = _dist(graph_ms)
            e["graph_replay"] = {"ms_median": gmed, "ms_min": gmn,
                                 "hbm_gbs": w["bytes"] / (gmed / 1e3) / 1e9 if w.get("bytes") else None,
                                 "how": "the step's calls captured once in a CUDA graph, replayed each step "
                                        "(L2 flushed before each): device time without per-call host work"}
        if target is not None:
            frac = e["frac_of_hbm"] if bound == "hbm" else e["frac_of_peak"]
            e["target"] = f">= {target} of {'HBM bandwidth' if bound == 'hbm' else 'the dense bf16 peak'}"
            e["meets_target"] = frac >= target
        out[name] = e
    del raw, flush
    torch.cuda.empty_cache()
    return {"entries": out, "peak_tflops": peak, "peak_source": why, "hbm_gbs_peak": hbm,
            "clocks": clocks, "steps_each": args.workload_steps,
            "how": "each workload set up once (seeded inputs), 3 warm-up steps, then --workload-steps "
                   "steps timed with CUDA events at step boundaries; the MLP block is the headline run"}


def cpu_rate_one_core(tokens=64):
    """The oracle's rate on one host core: the same MLP step on a token
    sample in a child process whose BLAS and OpenMP pools have one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    code = ("import time, bench\n"
            f"x, w1, w2, dy = bench.cpu_inputs({tokens})\n"
            "bench.oracle_step(x[:8], w1, w2, dy[:8])\n"
            "t0 = time.perf_counter()\n"
            "bench.oracle_step(x, w1, w2, dy)\n"
            "print(time.perf_counter() - t0)\n")
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=600)
        dt = float(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, never fatal
        return {"error": f"one-core run failed: {e}"}
    flops = STEP_FLOPS * tokens / M
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": 1,
            "gflops_per_core": flops / dt / 1e9,
            "sample": f"one MLP fwd+bwd step over {tokens} of the {M} tokens with the full weights, "
                      f"fp64 numpy oracle with one BLAS/OpenMP thread ({dt:.1f} s, {flops / 1e9:.0f} GFLOP)"}


def profile_case():
    """Each kernel variant of the step at the step's shapes (about 1 GB
    resident), a bounded case for ncu captures.  Launch order:
    [col fwd + GeLU (X.W), row fwd AllReduce (X.W, last wave in k-slices),
    row bwd dZ with GeLU' and dW2 in one launch (dY.W^T then X^T.dY), col bwd
    fused dX (dY.W^T, last wave in k-slices)] x 2,
    then col bwd dW1 (X^T.dZ) x 2."""
    import torch
    import gemm_reduce_fusion_gb300 as tp
    import synth
    import numpy as np

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    bf = dict(dtype=torch.bfloat16, device="cuda")
    x = [dev(synth.normal_bf16((M, NK), synth.seed_for(2, r))) for r in range(P)]
    w = [dev(synth.normal_bf16((NK, H), synth.seed_for(2, 4 + r), 0.02)) for r in range(P)]
    w1 = [dev(synth.normal_bf16((H, NK), synth.seed_for(2, 8 + r), 0.02)) for r in range(P)]
    z = [torch.empty((M, NK), **bf) for _ in range(P)]
    hh = [torch.empty((M, NK), **bf) for _ in range(P)]
    y = torch.empty((M, H), **bf)
    g = [torch.empty((M, NK), **bf) for _ in range(P)]
    ws = _ws_for(torch, tp, [(tp.TP_OP_COL_FWD, P, M, NK, H, 0), (tp.TP_OP_ROW_AR, P, M, H, NK, 0),
                             (tp.TP_OP_ROW_BWD, P, M, H, NK, 0), (tp.TP_OP_COL_BWD, P, M, NK, H, 0)])
    dx = torch.empty((M, H), **bf)
    wgrad2 = [torch.empty((NK, H), **bf) for _ in range(P)]
    for _ in range(2):
        tp.tp_col_linear_fwd(y, w1, z, ws, epi=tp.TP_EPI_GELU, preact=hh)   # X.W + GeLU
        tp.tp_row_linear_fwd_allreduce(x, w, [y], ws)                         # X.W, fused AllReduce
        tp.tp_row_linear_bwd(x, w, y, g, wgrad2, ws, preact=hh)               # dY.W^T * GeLU'(H), X^T.dY
        tp.tp_col_linear_bwd(None, w1, g, dx, None, ws)                       # dY.W^T, fused dX
    wgrad = [torch.empty((H, NK), **bf) for _ in range(P)]
    for _ in range(2):
        tp.tp_col_linear_bwd(y, w1, g, None, wgrad, ws)                       # X^T.dZ
    torch.cuda.synchronize()
    assert tp.tp_get_device_status(ws) == tp.TP_OK
    print("profile case done")


def profile_workload(name):
    """One workload of --configs, set up once and its calls run twice: a
    bounded case for ncu (at most about 3 GB resident, a few launches)."""
    import torch
    torch.cuda.set_device(0)
    import gemm_reduce_fusion_gb300 as tp
    table = dict(workloads(torch, tp))
    if name not in table:
        raise SystemExit(f"unknown workload {name!r}; one of {sorted(table)}")
    w = table[name]()
    for _ in range(2):
        for _, fn in w["calls"]:
            fn()
    torch.cuda.synchronize()
    print(f"profile workload {name} done: {[n for n, _ in w['calls']]} x 2")


# ------------------------------------------------------------------ all workloads / chunk sweep

def _dev_all(torch, tree):
    import numpy as np
    conv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return {k: ([conv(a) for a in v] if isinstance(v, list) else conv(v)) for k, v in tree.items()}


def _ws_for(torch, tp, calls):
    n = max(tp.tp_workspace_size(*c) for c in calls)
    return torch.zeros(n, dtype=torch.uint8, device="cuda")


def workloads(torch, tp):
    """(name, setup) pairs; setup() -> dict(calls=[(name, fn)], flops=..., bytes=..., bound=...)."""
    import synth
    bf = dict(dtype=torch.bfloat16, device="cuda")

    def w1():
        d = _dev_all(torch, synth.worked_example_inputs())
        p, M, K, N = 2, 128, 1024, 2048
        y = torch.empty((M, N), **bf)
        ys = [torch.empty((M // p, N), **bf) for _ in range(p)]
        ws = _ws_for(torch, tp, [(tp.TP_OP_ROW_AR, p, M, N, K, 32), (tp.TP_OP_ROW_RS, p, M, N, K, 32)])
        return dict(calls=[("row_fwd_allreduce", lambda: tp.tp_row_linear_fwd_allreduce(d["x"], d["w"], [y], ws, 32)),
                           ("row_fwd_reducescatter",
                            lambda: tp.tp_row_linear_fwd_reducescatter(d["x"], d["w"], ys, ws, 32))],
                    flops=2 * 2.0 * M * N * K * p, bytes=2 * (2 * (p * M * K + p * K * N) + 2 * M * N),
                    bound="hbm", flush=True,
                    row_reduce=dict(call="row_fwd_allreduce", x=d["x"], w=d["w"], y=y, chunk=32),
                    desc="row-parallel p=2, X_r[128,1024], W_r[1024,2048], AllReduce + ReduceScatter, chunk_m=32", ws=ws)

    def w2():
        d = _dev_all(torch, synth.mlp_block_inputs())
        p, M, h, nk = 4, 4096, 4096, 4096
        Z = [torch.empty((M, nk), **bf) for _ in range(p)]
        Hh = [torch.empty((M, nk), **bf) for _ in range(p)]
        Y = torch.empty((M, h), **bf)
        DZ = [torch.empty((M, nk), **bf) for _ in range(p)]
        DW2 = [torch.empty((nk, h), **bf) for _ in range(p)]
        DX = torch.empty((M, h), **bf)
        DW1 = [torch.empty((h, nk), **bf) for _ in range(p)]
        ws = _ws_for(torch, tp, [(tp.TP_OP_COL_FWD, p, M, nk, h, 0), (tp.TP_OP_ROW_AR, p, M, h, nk, 0),
                                 (tp.TP_OP_ROW_BWD, p, M, h, nk, 0), (tp.TP_OP_COL_BWD, p, M, nk, h, 0)])
        return dict(calls=[
            ("col_fwd_gelu", lambda: tp.tp_col_linear_fwd(d["x"], d["w1"], Z, ws, epi=tp.TP_EPI_GELU, preact=Hh)),
            ("row_fwd_allreduce", lambda: tp.tp_row_linear_fwd_allreduce(Z, d["w2"], [Y], ws)),
            ("row_bwd", lambda: tp.tp_row_linear_bwd(Z, d["w2"], d["dy"], DZ, DW2, ws, preact=Hh)),
            ("col_bwd_dx", lambda: tp.tp_col_linear_bwd(None, d["w1"], DZ, DX, None, ws)),
            ("col_bwd_dw", lambda: tp.tp_col_linear_bwd(d["x"], d["w1"], DZ, None, DW1, ws))],
            flops=6 * 2.0 * M * h * nk * p, bytes=None, bound="tensor", flush=False,
            row_reduce=dict(call="row_fwd_allreduce", x=Z, w=d["w2"], y=Y, chunk=0),
            desc="Megatron MLP block fwd+bwd p=4, 4096 tokens, h=4096, ffn=16384", ws=ws)

    def w3():
        d = _dev_all(torch, synth.mha_projection_inputs())
        p, M, h, nq, no = 4, 4096, 4096, 3072, 1024
        QKV = [torch.empty((M, nq), **bf) for _ in range(p)]
        Y = torch.empty((M, h), **bf)
        DO = [torch.empty((M, no), **bf) for _ in range(p)]
        DWO = [torch.empty((no, h), **bf) for _ in range(p)]
        DX = torch.empty((M, h), **bf)
        DWQ = [torch.empty((h, nq), **bf) for _ in range(p)]
        ws = _ws_for(torch, tp, [(tp.TP_OP_COL_FWD, p, M, nq, h, 0), (tp.TP_OP_ROW_AR, p, M, h, no, 0),
                                 (tp.TP_OP_ROW_BWD, p, M, h, no, 0), (tp.TP_OP_COL_BWD, p, M, nq, h, 0)])
        return dict(calls=[
            ("qkv_col_fwd", lambda: tp.tp_col_linear_fwd(d["x"], d["wqkv"], QKV, ws)),
            ("wo_row_fwd_allreduce", lambda: tp.tp_row_linear_fwd_allreduce(d["o"], d["wo"], [Y], ws)),
            ("wo_row_bwd", lambda: tp.tp_row_linear_bwd(d["o"], d["wo"], d["dy"], DO, DWO, ws)),
            ("qkv_col_bwd", lambda: tp.tp_col_linear_bwd(d["x"], d["wqkv"], d["dqkv"], DX, DWQ, ws))],
            flops=3 * (2.0 * M * h * nq * p + 2.0 * M * no * h * p), bytes=None, bound="tensor", flush=False,
            row_reduce=dict(call="wo_row_fwd_allreduce", x=d["o"], w=d["wo"], y=Y, chunk=0),
            desc="MHA projections fwd+bwd p=4, 4096 tokens, h=4096, QKV [4096,3072]/shard, W_O [1024,4096]/shard", ws=ws)

    def w4():
        d = _dev_all(torch, synth.sequence_parallel_pair_inputs())
        p, Mp, h, nk = 8, 1024, 8192, 3584
        M = p * Mp
        Z = [torch.empty((M, nk), **bf) for _ in range(p)]
        Hh = [torch.empty((M, nk), **bf) for _ in range(p)]
        YS = [torch.empty((Mp, h), **bf) for _ in range(p)]
        ws = _ws_for(torch, tp, [(tp.TP_OP_AG_MM, p, M, nk, h, 0), (tp.TP_OP_ROW_RS, p, M, h, nk, 0)])
        return dict(calls=[
            ("ag_matmul_gelu", lambda: tp.tp_ag_matmul(d["x"], d["w1"], Z, ws, epi=tp.TP_EPI_GELU, preact=Hh)),
            ("row_fwd_reducescatter", lambda: tp.tp_row_linear_fwd_reducescatter(Z, d["w2"], YS, ws))],
            flops=2 * 2.0 * M * h * nk * p, bytes=None, bound="tensor", flush=False,
            row_reduce=dict(call="row_fwd_reducescatter", x=Z, w=d["w2"], y=None, chunk=0, op=tp.TP_OP_ROW_RS),
            desc="sequence-parallel pair fwd p=8, 8192 tokens (1024/rank), h=8192, ffn=28672", ws=ws)

    def w4b():
        d = _dev_all(torch, synth.sequence_parallel_pair_inputs())
        p, Mp, h, nk = 8, 1024, 8192, 3584
        M = p * Mp
        dys = _dev_all(torch, {"dy": [synth.normal_bf16((Mp, h), synth.seed_for(43, s)) for s in range(p)]})["dy"]
        Z = [torch.empty((M, nk), **bf) for _ in range(p)]
        Hh = [torch.empty((M, nk), **bf) for _ in range(p)]
        YS = [torch.empty((Mp, h), **bf) for _ in range(p)]
        DZ = [torch.empty((M, nk), **bf) for _ in range(p)]
        DW2 = [torch.empty((nk, h), **bf) for _ in range(p)]
        DXS = [torch.empty((Mp, h), **bf) for _ in range(p)]
        DW1 = [torch.empty((h, nk), **bf) for _ in range(p)]
        ws = _ws_for(torch, tp, [(tp.TP_OP_AG_MM, p, M, nk, h, 0), (tp.TP_OP_ROW_RS, p, M, h, nk, 0),
                                 (tp.TP_OP_ROW_RS_BWD, p, M, h, nk, 0), (tp.TP_OP_AG_MM_BWD, p, M, nk, h, 0)])
        return dict(calls=[
            ("ag_matmul_gelu", lambda: tp.tp_ag_matmul(d["x"], d["w1"], Z, ws, epi=tp.TP_EPI_GELU, preact=Hh)),
            ("row_fwd_reducescatter", lambda: tp.tp_row_linear_fwd_reducescatter(Z, d["w2"], YS, ws)),
            ("row_bwd_allgather", lambda: tp.tp_row_linear_bwd_reducescatter(Z, d["w2"], dys, DZ, DW2, ws,
                                                                             preact=Hh)),
            ("ag_matmul_bwd", lambda: tp.tp_ag_matmul_bwd(d["x"], d["w1"], DZ, DXS, DW1, ws))],
            flops=6 * 2.0 * M * h * nk * p, bytes=None, bound="tensor", flush=False,
            desc="sequence-parallel pair fwd+bwd p=8, 8192 tokens (1024/rank), h=8192, ffn=28672", ws=ws)

    gpt3_weights = {}

    def w5(M):
        def setup():
            # the weights are shared by both token counts: drawn and uploaded once
            if not gpt3_weights:
                gpt3_weights.update(_dev_all(torch, synth.gpt3_mlp_weights()))
            d = dict(gpt3_weights, **_dev_all(torch, {"x": synth.gpt3_mlp_activations(M)}))
            p, h, nk = 8, 12288, 6144
            Z = [torch.empty((M, nk), **bf) for _ in range(p)]
            Hh = [torch.empty((M, nk), **bf) for _ in range(p)]
            Y = torch.empty((M, h), **bf)
            ws = _ws_for(torch, tp, [(tp.TP_OP_COL_FWD, p, M, nk, h, 0), (tp.TP_OP_ROW_AR, p, M, h, nk, 0)])
            wbytes = 2 * 2.0 * h * nk * p
            return dict(calls=[
                ("col_fwd_gelu", lambda: tp.tp_col_linear_fwd(d["x"], d["w1"], Z, ws, epi=tp.TP_EPI_GELU, preact=Hh)),
                ("row_fwd_allreduce", lambda: tp.tp_row_linear_fwd_allreduce(Z, d["w2"], [Y], ws))],
                flops=2 * 2.0 * M * h * nk * p,
                bytes=wbytes + 4.0 * M * h + 6.0 * M * nk * p,
                bound="hbm" if M <= 64 else "tensor", flush=M <= 64,
                row_reduce=dict(call="row_fwd_allreduce", x=Z, w=d["w2"], y=Y, chunk=0),
                desc=f"GPT-3-scale MLP fwd p=8, h=12288, ffn=49152, M={M}", ws=ws)
        return setup

    return [("worked_example_p2", w1), ("mlp_block_p4", w2), ("mha_projections_p4", w3), ("sp_pair_fwd_p8", w4), ("sp_pair_fwd_bwd_p8", w4b),
            ("gpt3_mlp_p8_m2048", w5(2048)), ("gpt3_mlp_p8_m16", w5(16))]


def _time_calls(torch, calls, steps, warmup, flush_buf=None):
    """Median per-step ms of the calls (L2 flushed before each step when asked)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    times, per = [], {n: [] for n, _ in calls}
    for _ in range(steps):
        if flush_buf is not None:
            flush_buf.fill_(1.0)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
        ev[0].record(stream)
        for i, (_, fn) in enumerate(calls):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        times.append(ev[0].elapsed_time(ev[-1]))
        for i, (n, _) in enumerate(calls):
            per[n].append(ev[i].elapsed_time(ev[i + 1]))
    med = lambda v: sorted(v)[len(v) // 2]
    return med(times), {n: med(v) for n, v in per.items()}, min(times), sorted(times)[int(0.9 * (len(times) - 1))]


# The same GEMMs on the unsharded problem, (M, K, N) each, as plain library
# matmuls: context for each workload (a GEMM library on the concatenated
# weights, with no reduction or gather to do), not part of the measured path.
UNSHARDED_GEMMS = {
    "worked_example_p2": [(128, 2048, 2048)] * 2,
    "mlp_block_p4": [(4096, 4096, 16384), (4096, 16384, 4096), (4096, 4096, 16384), (16384, 4096, 4096),
                (4096, 16384, 4096), (4096, 4096, 16384)],
    "mha_projections_p4": [(4096, 4096, 12288), (4096, 4096, 4096), (4096, 4096, 4096), (4096, 4096, 4096),
                (4096, 12288, 4096), (4096, 4096, 12288)],
    "sp_pair_fwd_p8": [(8192, 8192, 28672), (8192, 28672, 8192)],
    "sp_pair_fwd_bwd_p8": [(8192, 8192, 28672), (8192, 28672, 8192), (8192, 8192, 28672), (28672, 8192, 8192),
                        (8192, 28672, 8192), (8192, 8192, 28672)],
    "gpt3_mlp_p8_m2048": [(2048, 12288, 49152), (2048, 49152, 12288)],
    "gpt3_mlp_p8_m16": [(16, 12288, 49152), (16, 49152, 12288)],
}


def _time_unsharded(torch, gemms, steps, warmup, flush_buf):
    """Median per-step ms of torch.matmul over the unsharded GEMMs."""
    bufs = []
    for m, k, n in gemms:
        bufs.append((torch.randn((m, k), device="cuda").to(torch.bfloat16),
                     torch.randn((k, n), device="cuda").mul_(0.02).to(torch.bfloat16),
                     torch.empty((m, n), dtype=torch.bfloat16, device="cuda")))
    calls = [(f"matmul{i}", (lambda a=a, b=b, c=c: torch.matmul(a, b, out=c))) for i, (a, b, c) in enumerate(bufs)]
    ms, _, _, _ = _time_calls(torch, calls, steps, warmup, flush_buf)
    del bufs, calls
    torch.cuda.empty_cache()
    return ms


def _row_timeline(torch, tp, rr, fused_ms, steps, warmup, flush_buf):
    """The two-engine timeline of a workload's row-parallel reduction
    ([M027] §03): c = one chunk's per-rank partial GEMMs and m = its
    rank-order reduce, both timed on the unfused baseline on chunk_m rows;
    the modelled T = c + (n-1) max(c, m) + m beside the fused call and the
    whole unfused call.  A ReduceScatter is modelled by the AllReduce of the
    same partials: it sums the same terms and routes row slices."""
    x, w = rr["x"], rr["w"]
    p = len(x)
    M, K = x[0].shape
    N = w[0].shape[1]
    y = rr["y"] if rr["y"] is not None else torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    chunk = min(rr["chunk"] or tp.tp_choose_chunk_m(rr.get("op", tp.TP_OP_ROW_AR), p, M, N, K), M)
    n = tp.tp_num_chunks(M, chunk)
    ws = _ws_for(torch, tp, [(tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, chunk)])
    xc, yc = [a[:chunk] for a in x], y[:chunk]
    c, _, _, _ = _time_calls(torch, [("c", lambda: tp.tp_row_linear_fwd_unfused(xc, w, yc, ws, chunk, phases=1))],
                             steps, warmup, flush_buf)
    m, _, _, _ = _time_calls(torch, [("m", lambda: tp.tp_row_linear_fwd_unfused(xc, w, yc, ws, chunk, phases=2))],
                             steps, warmup, flush_buf)
    u, _, _, _ = _time_calls(torch, [("u", lambda: tp.tp_row_linear_fwd_unfused(x, w, y, ws, chunk, phases=3))],
                             steps, warmup, flush_buf)
    del ws
    return {"call": rr["call"], "chunk_m": chunk, "n_chunks": n, "c_ms": c, "m_ms": m,
            "model_pipelined_ms": tp.tp_pipeline_time(c, m, n), "model_serial_ms": n * (c + m),
            "fused_ms": fused_ms, "unfused_ms": u}


def run_configs(args):
    import torch
    torch.cuda.set_device(0)
    import gemm_reduce_fusion_gb300 as tp
    pk, src = peaks()
    flush = torch.empty(256 << 20, dtype=torch.float32, device="cuda")   # 1 GiB > 2 x L2
    for name, setup in workloads(torch, tp):
        w = setup()
        steps, warmup = max(50, args.steps), max(10, args.warmup)
        ms, per, mn, p90 = _time_calls(torch, w["calls"], steps, warmup, flush if w["flush"] else None)
        tflops = w["flops"] / (ms / 1e3) / 1e12
        line = {"workload": name, "desc": w["desc"], "ms_per_step": ms, "ms_min": mn, "ms_p90": p90,
                "tflops": tflops, "frac_of_bf16_sustained": tflops / pk["bf16_tflops_sustained"],
                "per_call_ms": per, "l2": "flushed before each step" if w["flush"] else "inputs larger than L2",
                "peak_source": src}
        if w["bytes"]:
            gbs = w["bytes"] / (ms / 1e3) / 1e9
            line.update({"hbm_gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"], "bytes_per_step": w["bytes"]})
        if w.get("row_reduce"):
            rr = w["row_reduce"]
            line["timeline"] = _row_timeline(torch, tp, rr, per[rr["call"]], steps, warmup,
                                             flush if w["flush"] else None)
        del w
        torch.cuda.empty_cache()
        if name in UNSHARDED_GEMMS:
            cms = _time_unsharded(torch, UNSHARDED_GEMMS[name], steps, warmup,
                                  flush if line["l2"].startswith("flushed") else None)
            line.update({"unsharded_torch_matmul_ms": cms,
                         "fused_speed_vs_unsharded_torch_matmul": cms / ms,
                         "context": "torch.matmul (library GEMM) on the unsharded problem's GEMMs, same FLOPs, "
                                    "no reduction or gather; not part of the measured path"})
        print(json.dumps(line), flush=True)


def run_sweep(args):
    """chunk_m sweep of the GPT-3-scale FC pair at M = 2048 ([M027] §03-§04):
    fused time per chunk_m beside the two-engine timeline T = c + (n-1) max(c, m) + m
    with c = one chunk's per-rank GEMMs and m = its reduce, both measured on
    the unfused baseline."""
    import torch
    torch.cuda.set_device(0)
    import gemm_reduce_fusion_gb300 as tp
    import synth
    M, p, h, nk = 2048, 8, 12288, 6144
    d = _dev_all(torch, synth.gpt3_mlp_inputs(M))
    bf = dict(dtype=torch.bfloat16, device="cuda")
    Z = [torch.empty((M, nk), **bf) for _ in range(p)]
    Hh = [torch.empty((M, nk), **bf) for _ in range(p)]
    Y = torch.empty((M, h), **bf)
    chunks = [16, 64, 256, 1024, 2048]
    ws = _ws_for(torch, tp, [(op, p, M, n, k, c) for c in chunks for op, n, k in
                             [(tp.TP_OP_COL_FWD, nk, h), (tp.TP_OP_ROW_AR, h, nk), (tp.TP_OP_ROW_AR_UNFUSED, h, nk)]])
    tp.tp_col_linear_fwd(d["x"], d["w1"], Z, ws, epi=tp.TP_EPI_GELU, preact=Hh)
    measured = []   # (chunk_m, c, m, fused FC2 ms)
    for c in chunks:
        n = tp.tp_num_chunks(M, c)
        fc1, _, _, _ = _time_calls(torch, [("f", lambda: tp.tp_col_linear_fwd(d["x"], d["w1"], Z, ws, epi=tp.TP_EPI_GELU,
                                                                               preact=Hh, chunk_m=c))], 5, 2)
        fc2, _, _, _ = _time_calls(torch, [("f", lambda: tp.tp_row_linear_fwd_allreduce(Z, d["w2"], [Y], ws, chunk_m=c))], 5, 2)
        zc = [z[:min(c, M)] for z in Z]
        yc = Y[:min(c, M)]
        cm, _, _, _ = _time_calls(torch, [("c", lambda: tp.tp_row_linear_fwd_unfused(zc, d["w2"], yc, ws, c, phases=1))], 5, 2)
        mm, _, _, _ = _time_calls(torch, [("m", lambda: tp.tp_row_linear_fwd_unfused(zc, d["w2"], yc, ws, c, phases=2))], 5, 2)
        full_unfused, _, _, _ = _time_calls(torch, [("u", lambda: tp.tp_row_linear_fwd_unfused(Z, d["w2"], Y, ws, c, phases=3))], 3, 1)
        flops_fc = 2.0 * M * h * nk * p
        print(json.dumps({"sweep": "GPT-3-scale FC pair, p=8, M=2048", "chunk_m": c, "n_chunks": n,
                          "fc1_fused_ms": fc1, "fc2_fused_ms": fc2,
                          "fc1_tflops": flops_fc / fc1 / 1e9, "fc2_tflops": flops_fc / fc2 / 1e9,
                          "fc2_c_ms": cm, "fc2_m_ms": mm,
                          "fc2_model_pipelined_ms": tp.tp_pipeline_time(cm, mm, n),
                          "fc2_model_serial_ms": n * (cm + mm),
                          "fc2_unfused_whole_ms": full_unfused}), flush=True)
        measured.append((c, cm, mm, fc2))
    pick = tp.tp_choose_chunk_m_measured(M, [r[0] for r in measured], [r[1] for r in measured],
                                         [r[2] for r in measured])
    fastest = min(measured, key=lambda r: r[3])[0]
    print(json.dumps({"sweep": "GPT-3-scale FC pair, p=8, M=2048", "chunk_m_from_measured_c_m": pick,
                      "chunk_m_scheduler_model": tp.tp_choose_chunk_m(tp.TP_OP_ROW_AR, p, M, h, nk),
                      "chunk_m_fastest_fused_fc2": fastest}), flush=True)


def _err_stats(torch, got, ref):
    """Error of a bf16 result against an fp32 reference: max|d|/max|ref|,
    rms(d)/rms(ref), and the share of elements that differ from bf16(ref)."""
    g = got.float()
    d = (g - ref).abs()
    return {"max_rel": float(d.max() / ref.abs().max()),
            "rms_rel": float(d.pow(2).mean().sqrt() / ref.pow(2).mean().sqrt()),
            "frac_not_rounded_ref": float((got != ref.to(torch.bfloat16)).float().mean())}


def run_precision_report(args):
    """Whole-layer output (and gradient) error of the fused path against the
    separate baseline ([M027] §04: compare the layer's output error, and for
    training its backward and parameter gradients; §06: record the output and
    gradient error and the workspace peak).  For each row-parallel layer of
    the workloads, bf16 outputs of
      fused        -- all p partials in one fp32 accumulator, rounded once;
      unfused_fp32 -- per-rank fp32 partials, then an fp32 rank-order sum;
      unfused_bf16 -- per-rank partials rounded to bf16, summed as a bf16
                      collective would (bf16 running sum, rank order);
    are compared with the library's own fp32-output result, which the parity
    tests hold within 1e-5 of max|Y| of the exact fp64 sum (far below the
    bf16 errors measured here).  Every element of the layer is compared."""
    import torch
    torch.cuda.set_device(0)
    import gemm_reduce_fusion_gb300 as tp
    import synth
    bf = dict(dtype=torch.bfloat16, device="cuda")

    def ws(calls):
        return _ws_for(torch, tp, calls)

    def row_layer(name, xs, wsh, extra=None):
        p = len(xs)
        M, K = xs[0].shape
        N = wsh[0].shape[1]
        calls = [(tp.TP_OP_ROW_AR, p, M, N, K, 0, tp.TP_FP32), (tp.TP_OP_ROW_AR, p, M, N, K, 0),
                 (tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, 0)]
        w_ = ws(calls)
        ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
        tp.tp_row_linear_fwd_allreduce(xs, wsh, [ref], w_)
        out = {}
        y = torch.empty((M, N), **bf)
        tp.tp_row_linear_fwd_allreduce(xs, wsh, [y], w_)
        out["fused"] = _err_stats(torch, y, ref)
        tp.tp_row_linear_fwd_unfused(xs, wsh, y, w_)
        out["unfused_fp32"] = _err_stats(torch, y, ref)
        tp.tp_row_linear_fwd_unfused(xs, wsh, y, w_, flags=tp.TP_UNFUSED_BF16_COLLECTIVE)
        out["unfused_bf16"] = _err_stats(torch, y, ref)
        line = {"precision_report": name, "p": p, "M": M, "N": N, "K_per_rank": K, "errors_vs_fp32": out,
                "workspace_bytes": {"fused_bf16_out": tp.tp_workspace_size(tp.TP_OP_ROW_AR, p, M, N, K, 0),
                                    "unfused": tp.tp_workspace_size(tp.TP_OP_ROW_AR_UNFUSED, p, M, N, K, 0)}}
        if extra:
            line.update(extra)
        print(json.dumps(line), flush=True)
        del ref, y, w_
        torch.cuda.empty_cache()

    # worked example: p = 2
    d = _dev_all(torch, synth.worked_example_inputs())
    row_layer("row-parallel worked example (p=2, X_r[128,1024], W_r[1024,2048])", d["x"], d["w"])
    # MLP block: FC2 forward on the GPU's own GeLU output, then the backward's gradients
    d = _dev_all(torch, synth.mlp_block_inputs())
    p, M, h, nk = 4, 4096, 4096, 4096
    Z = [torch.empty((M, nk), **bf) for _ in range(p)]
    Hh = [torch.empty((M, nk), **bf) for _ in range(p)]
    w0 = ws([(tp.TP_OP_COL_FWD, p, M, nk, h, 0), (tp.TP_OP_ROW_BWD, p, M, h, nk, 0, tp.TP_FP32),
             (tp.TP_OP_COL_BWD, p, M, nk, h, 0, tp.TP_FP32), (tp.TP_OP_ROW_BWD, p, M, h, nk, 0),
             (tp.TP_OP_COL_BWD, p, M, nk, h, 0)])
    tp.tp_col_linear_fwd(d["x"], d["w1"], Z, w0, epi=tp.TP_EPI_GELU, preact=Hh)
    row_layer("MLP FC2 forward (p=4, 4096 tokens, h=4096, ffn=16384)", Z, d["w2"])
    # gradients: bf16 results of the fused backward vs its fp32-output results
    grads = {}
    DZ = [torch.empty((M, nk), **bf) for _ in range(p)]
    DZf = [torch.empty((M, nk), dtype=torch.float32, device="cuda") for _ in range(p)]
    tp.tp_row_linear_bwd(None, d["w2"], d["dy"], DZ, None, w0, preact=Hh)
    tp.tp_row_linear_bwd(None, d["w2"], d["dy"], DZf, None, w0, preact=Hh)
    grads["dZ_k (FC2 dX * GeLU')"] = _err_stats(torch, torch.cat(DZ, 1), torch.cat(DZf, 1))
    del DZf
    DW2 = [torch.empty((nk, h), **bf) for _ in range(p)]
    DW2f = [torch.empty((nk, h), dtype=torch.float32, device="cuda") for _ in range(p)]
    tp.tp_row_linear_bwd(Z, d["w2"], d["dy"], None, DW2, w0)
    tp.tp_row_linear_bwd(Z, d["w2"], d["dy"], None, DW2f, w0)
    grads["dW2_k"] = _err_stats(torch, torch.cat(DW2, 1), torch.cat(DW2f, 1))
    del DW2, DW2f
    DX = torch.empty((M, h), **bf)
    DXf = torch.empty((M, h), dtype=torch.float32, device="cuda")
    tp.tp_col_linear_bwd(None, d["w1"], DZ, DX, None, w0)
    tp.tp_col_linear_bwd(None, d["w1"], DZ, DXf, None, w0)
    grads["dX (fused reduce over k)"] = _err_stats(torch, DX, DXf)
    DW1 = [torch.empty((h, nk), **bf) for _ in range(p)]
    DW1f = [torch.empty((h, nk), dtype=torch.float32, device="cuda") for _ in range(p)]
    tp.tp_col_linear_bwd(d["x"], d["w1"], DZ, None, DW1, w0)
    tp.tp_col_linear_bwd(d["x"], d["w1"], DZ, None, DW1f, w0)
    grads["dW1_k"] = _err_stats(torch, torch.cat(DW1, 1), torch.cat(DW1f, 1))
    del DW1, DW1f, DXf, w0
    print(json.dumps({"precision_report": "MLP backward gradients, bf16 vs the fp32-output result",
                      "errors_vs_fp32": grads}), flush=True)
    # FC1's dX reduce as an unfused collective would do it: X_k = dZ_k, W_k = W1_k^T
    w1t = [w.t().contiguous() for w in d["w1"]]
    row_layer("MLP FC1 backward dX = sum_k dZ_k W1_k^T (p=4)", DZ, w1t)
    del w1t, DZ, Z, Hh, d
    torch.cuda.empty_cache()
    # MHA output projection
    d = _dev_all(torch, synth.mha_projection_inputs())
    row_layer("MHA W_O forward (p=4, 4096 tokens, K_r=1024, h=4096)", d["o"], d["wo"])
    del d
    torch.cuda.empty_cache()
    # GPT-3-scale FC2, p = 8
    d = _dev_all(torch, synth.gpt3_mlp_inputs(2048))
    p, M, h, nk = 8, 2048, 12288, 6144
    Z = [torch.empty((M, nk), **bf) for _ in range(p)]
    w0 = ws([(tp.TP_OP_COL_FWD, p, M, nk, h, 0)])
    tp.tp_col_linear_fwd(d["x"], d["w1"], Z, w0, epi=tp.TP_EPI_GELU)
    row_layer("GPT-3-scale FC2 forward (p=8, M=2048, K_r=6144, N=12288)", Z, d["w2"])


def _trace_launch(torch, tp, fn, cap=1 << 16):
    """Run fn() once with the timeline trace on; per-unit records, time-ordered."""
    buf = torch.zeros((cap, 4), dtype=torch.int64, device="cuda")
    fn()                                   # warm: tensor maps, caches
    torch.cuda.synchronize()
    buf.zero_()
    tp.tp_trace_set(buf, cap)
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        tp.tp_trace_set(None)
    rec = [tuple(int(v) for v in r) for r in buf.cpu().tolist() if r[0] != 0]
    return rec


def _timeline(rec):
    """Per-chunk compute and drain windows of one traced launch ([M027] §03:
    compute c and communication m per chunk; here c is the chunk's MMA
    window and m the drain after its last accumulator completes) and the
    share of drain time that overlapped later MMAs on the same CTA/cluster."""
    t0 = min(r[0] for r in rec)
    chunks = {}
    for start, full, drained, tag in rec:
        chunks.setdefault(tag >> 32, []).append((start, full, drained))
    per = []
    for ch in sorted(chunks):
        u = chunks[ch]
        c0, c1 = min(x[0] for x in u), max(x[1] for x in u)
        d1 = max(x[2] for x in u)
        per.append({"chunk": ch, "mma_us": [round((c0 - t0) / 1e3, 2), round((c1 - t0) / 1e3, 2)],
                    "drained_us": round((d1 - t0) / 1e3, 2), "c_us": round((c1 - c0) / 1e3, 2),
                    "m_us": round((d1 - c1) / 1e3, 2)})
    by_who = {}
    for start, full, drained, tag in rec:
        by_who.setdefault(tag & 0xFFFFFFFF, []).append((start, full, drained))
    drain = over = 0
    for units in by_who.values():
        units.sort()
        for a, b in zip(units, units[1:] + [None]):
            drain += a[2] - a[1]
            if b is not None:
                over += max(0, min(a[2], b[1]) - max(a[1], b[0]))
    total = (max(r[2] for r in rec) - t0) / 1e3
    return per, total, (over / drain if drain else 0.0)


def run_trace(args):
    """Measured chunk timelines of single fused launches beside the pages'
    model T = c + (n-1) max(c, m) + m built from the measured c and m."""
    import torch
    torch.cuda.set_device(0)
    import gemm_reduce_fusion_gb300 as tp
    import synth
    cases = []
    d1 = _dev_all(torch, synth.worked_example_inputs())
    y1 = torch.empty((128, 2048), dtype=torch.bfloat16, device="cuda")
    ws1 = _ws_for(torch, tp, [(tp.TP_OP_ROW_AR, 2, 128, 2048, 1024, 32)])
    cases.append(("worked example: row AllReduce p=2, M=128, chunk_m=32",
                  lambda: tp.tp_row_linear_fwd_allreduce(d1["x"], d1["w"], [y1], ws1, 32)))
    M, p, h, nk = 2048, 8, 12288, 6144
    d5 = _dev_all(torch, synth.gpt3_mlp_inputs(M))
    z5 = [torch.empty((M, nk), dtype=torch.bfloat16, device="cuda") for _ in range(p)]
    y5 = torch.empty((M, h), dtype=torch.bfloat16, device="cuda")
    for c in (256, 1024, 2048):
        ws5 = _ws_for(torch, tp, [(tp.TP_OP_ROW_AR, p, M, h, nk, c)])
        cases.append((f"GPT-3-scale FC2 row AllReduce p=8, M=2048, chunk_m={c}",
                      lambda c=c, ws5=ws5: tp.tp_row_linear_fwd_allreduce(z5, d5["w2"], [y5], ws5, c)))
    for name, fn in cases:
        rec = _trace_launch(torch, tp, fn)
        per, total, overlap = _timeline(rec)
        n = len(per)
        cbar = sum(x["c_us"] for x in per) / n
        mbar = sum(x["m_us"] for x in per) / n
        print(json.dumps({"trace": name, "units": len(rec), "n_chunks": n, "launch_us": round(total, 2),
                          "mean_c_us": round(cbar, 2), "mean_m_us": round(mbar, 2),
                          "model_pipelined_us": round(tp.tp_pipeline_time(cbar, mbar, n), 2),
                          "model_serial_us": round(n * (cbar + mbar), 2),
                          "drain_overlapped_with_mma": round(overlap, 3), "chunks": per[:8]}), flush=True)


def main():
    args = parse()
    if args.tile_mode and args.impl == "ours":
        import gemm_reduce_fusion_gb300 as tp
        tp.tp_debug_set(tp.TP_DEBUG_TILE_MODE, args.tile_mode)
    if args.profile_case:
        profile_case()
        return
    if args.profile_workload:
        profile_workload(args.profile_workload)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.configs:
        run_configs(args)
        return
    if args.precision_report:
        run_precision_report(args)
        return
    if args.trace:
        run_trace(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
