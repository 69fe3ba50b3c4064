#!/usr/bin/env python
"""Benchmark: one MoE MLP layer step (forward + backward, every kernel of the
hot path) on synthetic inputs of the DeepSeek-V3-shaped expert shard.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Timed regions (CUDA events on the launching
stream, synchronize + barrier on both sides, max over ranks):
  1. K replays of the step captured as one CUDA graph -> value, ms_per_step;
  2. K eager steps with an event between kernels -> per-kernel durations,
     the roofline of the dominant kernel, launch count;
  3. K end-to-end steps: pinned-host -> device copies of the step's inputs,
     the graph replay, and the device -> host copy of the layer output -> e2e
     (the copies of neighbouring steps overlap the compute on copy streams).
Inputs (weights 2.8 GB, activations > 0.5 GB) are larger than the 129 MB L2,
so no flush is needed between steps.  N > 1: one process per GPU, each an
independent expert-parallel shard (experts [r*E, (r+1)*E) of 256) of the same
token batch; no collective on the data path (weak scaling).
--impl reference times the CPU oracle on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fused grouped FC1+GLU+MXFP8 fwd/bwd TFLOP/s and % of GB300 tensor peak"
WORKLOAD = "dsv3"
CAPACITY_FACTOR = 2.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d.get("bf16_tflops_sustained",
                d["bf16_tflops"]), "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


SHAPE = {"dsv3": "DeepSeek-V3-shaped expert-parallel shard", "gptoss": "GPT-OSS-shaped layer",
         "skew": "skewed-routing 64-expert layer", "skew_srelu": "skewed-routing 64-expert layer",
         "tiny": "tiny MoE MLP"}


def workload_desc(w):
    fwd = ("NVFP4 (forward: FC1 bf16 + amax -> E2M1/E4M3 casts -> block-scaled NVFP4 FC2; backward: dGLU "
           "bf16 + amax + rotated amax -> NVFP4 dX, random-Hadamard-rotated NVFP4 weight gradients)"
           if w.out == "nvfp4" else "MXFP8 E4M3/E8M0 outputs + transposed copies")
    return (f"{w.name}: {SHAPE.get(w.name, w.name)}, T={w.T} H={w.H} experts "
            f"{w.expert_begin}..{w.expert_begin + w.E - 1} of {w.n_experts}, top-{w.k}, F={w.F}, {w.act}, "
            f"{fwd}; forward + backward")


def kernel_model(name, w, R, Rp):
    """Algorithmic FLOPs, minimal HBM bytes and the arithmetic type of one
    launch of each step kernel (R real rows, Rp padded rows)."""
    E, H, F, N1, T, k = w.E, w.H, w.F, w.N1, w.T, w.k
    nv = 1 / 2 + 1 / 16  # bytes per NVFP4 element: E2M1 code + E4M3 scale per 16
    m = {
        "route_permute": (0, T * k * 8 + 2 * R * H * 2 + (Rp - R) * H * 2, None),
        "fc1_glu_quant": (2 * R * H * N1, E * N1 * H * 2 + R * H * 2 + R * N1 * 2 + 2 * R * F * (1 + 1 / 32),
                          "bf16"),
        "quant_w2": (0, E * F * H * 2 + E * F * H * (1 + 1 / 32), None),
        "fc2": (2 * R * F * H, E * H * F * (1 + 1 / 32) + R * F * (1 + 1 / 32) + R * H * 2, "fp8"),
        "combine": (0, R * H * 2 + T * H * 2, None),
        "combine_bwd": (0, T * H * 2 + R * H * 2 + Rp * H * 2 + T * k * 8, None),
        "dglu_quant": (2 * R * H * F, E * F * H * 2 + R * H * 2 + R * N1 * 2 + 2 * R * N1 * (1 + 1 / 32), "bf16"),
        "quant_w1": (0, E * N1 * H * 2 + E * N1 * H * (1 + 1 / 32), None),
        "dx": (2 * R * N1 * H, E * H * N1 * (1 + 1 / 32) + R * N1 * (1 + 1 / 32) + R * H * 2, "fp8"),
        "quant_x_col": (0, R * H * 2 + R * H * (1 + 1 / 32), None),
        "quant_dy_col": (0, R * H * 2 + R * H * (1 + 1 / 32), None),
        # the gather / combine backward that also write the column-wise MXFP8 copy
        "route_permute_qcol": (0, T * k * 8 + 2 * R * H * 2 + (Rp - R) * H * 2 + Rp * H * (1 + 1 / 32), None),
        "combine_bwd_qcol": (0, T * H * 2 + R * H * 2 + Rp * H * 2 + T * k * 8 + Rp * H * (1 + 1 / 32), None),
        "wgrad_w1": (2 * R * N1 * H, (N1 + H) * R * (1 + 1 / 32) + E * N1 * H * 2, "fp8"),
        "wgrad_w2": (2 * R * F * H, (F + H) * R * (1 + 1 / 32) + E * F * H * 2, "fp8"),
        "permute_bwd": (0, R * H * 2 + T * H * 2 + T * k * 4, None),
        # NVFP4 forward: FC1 writes bf16 y + amax; casts to E2M1 + E4M3 per 16; FP4 FC2
        "fc1_glu_nvfp4": (2 * R * H * N1, E * N1 * H * 2 + R * H * 2 + R * N1 * 2 + R * F * 2, "bf16"),
        "quant_a_nvfp4": (0, R * F * 2 + R * F * (1 / 2 + 1 / 16), None),
        "amax_w2": (0, E * F * H * 2, None),
        "quant_w2_nvfp4": (0, E * F * H * 2 + E * F * H * (1 / 2 + 1 / 16), None),
        "fc2_nvfp4": (2 * R * F * H, E * H * F * (1 / 2 + 1 / 16) + R * F * (1 / 2 + 1 / 16) + R * H * 2, "fp4"),
        # NVFP4 backward: dGLU writes bf16 dFC1 + its amax and rotated amax; NVFP4 rows of dFC1
        # and W1 (along 2F) for dX; rotated column-wise NVFP4 casts (with their amax passes)
        # of dFC1, x, a and dY for the weight gradients
        "dglu_nvfp4": (2 * R * H * F, E * F * H * 2 + R * H * 2 + R * N1 * 2 + R * N1 * 2, "bf16"),
        "quant_d_nvfp4": (0, R * N1 * 2 + R * N1 * nv, None),
        "amax_w1": (0, E * N1 * H * 2, None),
        "quant_w1_nvfp4": (0, E * N1 * H * 2 + E * N1 * H * nv, None),
        "dx_nvfp4": (2 * R * N1 * H, E * H * N1 * nv + R * N1 * nv + R * H * 2, "fp4"),
        "quant_d_rht": (0, R * N1 * 2 + R * N1 * nv, None),
        "rht_amax_x": (0, R * H * 2, None),
        "quant_x_rht": (0, R * H * 2 + R * H * nv, None),
        "wgrad_w1_nvfp4": (2 * R * N1 * H, (N1 + H) * R * nv + E * N1 * H * 2, "fp4"),
        "rht_amax_a": (0, R * F * 2, None),
        "quant_a_rht": (0, R * F * 2 + R * F * nv, None),
        "rht_amax_dy": (0, R * H * 2, None),
        "quant_dy_rht": (0, R * H * 2 + R * H * nv, None),
        "wgrad_w2_nvfp4": (2 * R * F * H, (F + H) * R * nv + E * F * H * 2, "fp4"),
    }
    return m[name]


# dense tensor peak of an arithmetic type: the measured bf16 figure times the
# nominal dense ratio (fp8 2x, fp4 6x bf16)
PEAK_RATIO = {"bf16": 1.0, "fp8": 2.0, "fp4": 6.0}


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed regions run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": n}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (the reference arm and the cpu_baseline key)
# ---------------------------------------------------------------------------

def oracle_sample_step(inp, w, E_s, f_s=None):
    """The oracle's forward + backward of the same layer restricted to the
    shard's first E_s experts and, within them, to the first f_s of the F
    FFN columns (the matching input, gate and FC2 rows).  Returns the
    algorithmic FLOPs of the sample and its routed rows."""
    from oracle import moe_oracle as O
    f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()
    F = w.F
    f_s = f_s or F
    prm = O.ActParams(O.ACT_SWIGLU)
    rt = O.route(inp["topk_idx"].numpy(), w.expert_begin, E_s)
    R, Rp = int(rt.counts.sum()), rt.R_pad
    xp = O.permute(f64(inp["x"]), rt)
    W1 = inp["W1"][:E_s]
    W1 = f64(torch.cat([W1[:, :f_s], W1[:, F:F + f_s]], dim=1))
    W1p = O.repack_fc1(W1)
    W2 = f64(inp["W2"][:E_s, :f_s])
    fo = O.fc1_glu_fwd(xp, W1p, None, rt, prm)
    aq, asc = O.mx_quantize_rows(fo.y)
    W2q = [O.mx_quantize_cols(W2[e]) for e in range(E_s)]
    W2d = np.stack([O.mx_dequantize(q, s) for q, s in W2q])
    y = O.bf16_round(O.grouped_gemm_rows(O.mx_dequantize(aq, asc), W2d, rt))
    O.unpermute_combine(y, rt.row_of, inp["topk_prob"].numpy())
    dY, _ = O.combine_bwd(f64(inp["dOut"]), y, rt.row_of, inp["topk_prob"].numpy(), Rp)
    dY = O.bf16_round(dY)
    d = O.dglu_bwd(dY, W2, fo.pre_bf16, rt, prm)
    dq, ds = O.mx_quantize_rows(d)
    W1q = np.stack([O.mx_dequantize(*O.mx_quantize_cols(W1p[e])) for e in range(E_s)])
    dX = O.bf16_round(O.grouped_gemm_rows(O.mx_dequantize(dq, ds), W1q, rt))
    O.permute_bwd(dX, rt.row_of, w.T, w.k)
    xqc = O.mx_dequantize(*O.mx_quantize_cols(xp))
    dyqc = O.mx_dequantize(*O.mx_quantize_cols(dY))
    O.grouped_wgrad(O.mx_dequantize(*O.mx_quantize_cols(d)), xqc, rt)
    O.grouped_wgrad(O.mx_dequantize(*O.mx_quantize_cols(fo.y)), dyqc, rt)
    H = w.H
    return 2 * R * H * (2 * f_s) * 3 + 2 * R * f_s * H * 3, R


def cpu_threads():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count()


def size_oracle_sample(inp, w, budget_s):
    """Smallest-to-larger samples (FFN slice, then experts) until one step
    takes about budget_s / 2 or more."""
    E_s, f_s = 1, 64
    while True:
        t = time.perf_counter()
        oracle_sample_step(inp, w, E_s, f_s)
        dt = time.perf_counter() - t
        if dt >= budget_s / 2:
            return E_s, f_s
        if f_s * 2 <= w.F:
            f_s *= 2
        elif E_s * 2 <= w.E:
            E_s *= 2
        else:
            return E_s, f_s


def run_oracle_timed(inp, w, steps, warmup, budget_s):
    """Times `steps` oracle sample steps after `warmup` untimed ones; each
    step's sample is sized to about budget_s seconds."""
    E_s, f_s = size_oracle_sample(inp, w, budget_s)
    for _ in range(max(0, warmup - 1)):
        oracle_sample_step(inp, w, E_s, f_s)
    times, fl, R = [], 0, 0
    for _ in range(steps):
        t = time.perf_counter()
        fl, R = oracle_sample_step(inp, w, E_s, f_s)
        times.append(time.perf_counter() - t)
    mean = sum(times) / len(times)
    return {"value": fl / mean / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
            "sample": f"forward+backward of the first {E_s} of {w.E} experts ({R} routed rows), FFN columns "
                      f"0..{f_s - 1} of {w.F}; {steps} timed step(s) of {mean:.2f} s"}, mean


# ---------------------------------------------------------------------------

def profile_traffic(call_name):
    """DRAM bytes (read + write) per launch of one step call, from the
    committed ncu capture of that kernel (taken on the 8-expert shard and
    scaled to this workload), if it was taken on the current kernel sources
    (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic_dsv3.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get("calls", {}).get(call_name)
    if not d:
        return None
    h = hashlib.sha256()
    for f in d.get("sources", []):
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != d.get("sources_sha256"):
        return None
    return d.get("dram_bytes_per_launch")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sm-margin", type=int, default=0)
    ap.add_argument("--experts", type=int, default=0,
                    help="local experts of the shard (default: the workload's); a smaller shard for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from grouped_gemm_glu_gb300 import synth
    base = synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return
        w = base
        R_cap = w.capped_R(CAPACITY_FACTOR)
        inp = synth.make_inputs(w, seed=0, R_cap=R_cap)
        budget = max(0.3, 150.0 / (args.steps + args.warmup))
        cpu, mean = run_oracle_timed(inp, w, args.steps, args.warmup, budget)
        line = {"impl": "reference", "metric": METRIC, "value": cpu["value"], "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": workload_desc(w), "sample": cpu["sample"]},
                "cpu_baseline": cpu,
                "e2e": {"value": cpu["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    from grouped_gemm_glu_gb300 import build as B
    from grouped_gemm_glu_gb300 import lib as L
    from grouped_gemm_glu_gb300 import ops
    from grouped_gemm_glu_gb300.layer import MoeLayer
    B.build()
    lib = L.load()

    if args.experts:
        base = synth.scaled(base, E=args.experts)
    from grouped_gemm_glu_gb300 import shard
    w = synth.scaled(base, expert_begin=shard.shard_expert_begin(rank, base.E, base.n_experts))
    R_cap = w.capped_R(CAPACITY_FACTOR)
    inp = synth.make_inputs(w, seed=0, R_cap=R_cap)
    host = {k: inp[k].pin_memory() for k in ("x", "topk_idx", "topk_prob", "dOut")}
    g = {k: v.to(dev) for k, v in inp.items() if v is not None}
    if w.gpt_oss:   # GPT-OSS SwiGLU: gate clamp +-7, alpha 1.702, (up + 1), FC1 bias
        params = L.glu_params("swiglu", alpha=1.702, up_offset=1.0, gate_lo=-7.0, gate_hi=7.0)
    else:
        params = L.glu_params(w.act)
    layer = MoeLayer(g["W1"], g["W2"], w.T, w.k, R_cap, params, b1=g.get("b1"), expert_begin=w.expert_begin,
                     sm_margin=args.sm_margin, gated=w.gated, nvfp4=w.out == "nvfp4")
    X, I, P, DO = g["x"], g["topk_idx"], g["topk_prob"], g["dOut"]
    for _ in range(args.warmup):
        layer.step(X, I, P, DO)
    torch.cuda.synchronize()
    st = ops.read_status(layer.status)
    if st:
        raise SystemExit(f"device status {st} after warm-up")
    counts = layer.counts.cpu().numpy()
    R = int(counts.sum())
    Rp = int(layer.offsets[-1].item())

    graph = layer.capture(X, I, P, DO)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    # -- timed region 1: graph replays
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier()
    ms_graph = e0.elapsed_time(e1) / args.steps

    # -- timed region 2: eager, an event between kernels
    calls = layer.step_calls(X, I, P, DO)
    names = [n for n, _ in calls]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    launches0 = lib.moe_launch_count()
    barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        layer.run(calls, evs[s])
    torch.cuda.synchronize()
    barrier()
    launches = lib.moe_launch_count() - launches0
    per_kernel = {n: 0.0 for n in names}
    for s in range(args.steps):
        for i, n in enumerate(names):
            per_kernel[n] += evs[s][i].elapsed_time(evs[s][i + 1]) / args.steps
    ms_eager = sum(evs[s][0].elapsed_time(evs[s][-1]) for s in range(args.steps)) / args.steps

    # -- timed region 3: end to end with host buffers.  Every step copies its
    #    inputs from pinned host memory and reads its output back; the copies
    #    of step i+1 and the read-back of step i-1 run on copy streams while
    #    step i computes (two input sets, one captured graph per set, and two
    #    device output slots, as a training loop that prefetches would).
    out_host = [torch.empty(w.T, w.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in host)
    d2h = out_host[0].numel() * out_host[0].element_size()
    sets = [(X, I, P, DO), tuple(t.clone() for t in (X, I, P, DO))]
    # one graph per input set, each writing the layer output into its own
    # device slot (no device-to-device copy of the output per step)
    out_dev = [torch.empty_like(layer.out) for _ in range(2)]
    out0, graphs = layer.out, []
    for b in range(2):
        layer.out = out_dev[b]
        graphs.append(layer.capture(*sets[b]))
    layer.out = out0
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps(n, t0=None, t1=None):
        ev = lambda: torch.cuda.Event()
        copied, done, fetched = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        if t0 is not None:
            t0.record(comp)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(done[b])      # graph i-2 has finished reading set b
                for t, k in zip(sets[b], ("x", "topk_idx", "topk_prob", "dOut")):
                    t.copy_(host[k], non_blocking=True)
                copied[b].record(h2d_s)
            comp.wait_event(copied[b])
            if i >= 2:
                comp.wait_event(fetched[b])        # the read-back of step i-2 has left out_dev[b]
            graphs[b].replay()
            done[b].record(comp)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                fetched[b].record(d2h_s)
        for b in range(min(2, n)):
            comp.wait_event(fetched[b])
        if t1 is not None:
            t1.record(comp)

    # untimed warm-up of this region: the second graph's first replays and
    # the copy streams' first use are one-time costs
    e2e_steps(max(args.warmup, 2))
    barrier()
    torch.cuda.synchronize()
    e2e_steps(args.steps, e0, e1)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = e0.elapsed_time(e1) / args.steps
    # -- ablation: fused kernels vs the unfused path (same GEMM writing bf16,
    #    separate activation and quantize kernels), per direction
    def timed_on(lay, calls, n):
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            lay.run(calls)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    timed = lambda calls, n: timed_on(layer, calls, n)

    ufwd, ubwd = layer.forward_unfused_calls(), layer.backward_unfused_calls(layer.dY_perm)
    fused_fc1 = [("fc1_glu_quant", layer.fc1_mxfp8_call())]
    fused_dglu = [("dglu_quant", layer.dglu_mxfp8_call())]
    for calls in (fused_fc1, ufwd, fused_dglu, ubwd):
        layer.run(calls)  # warm-up
    na = max(3, min(args.steps, 20))
    f_ms = timed(fused_fc1, na)
    uf_ms = timed(ufwd, na)
    b_ms = timed(fused_dglu, na)
    ub_ms = timed(ubwd, na)
    ablation = {
        "forward": {"fused_ms": round(f_ms, 4), "unfused_ms": round(uf_ms, 4), "speedup": round(uf_ms / f_ms, 3),
                    "unfused": "gemm(bf16 pre) -> act -> mxfp8 rows -> mxfp8 cols"},
        "backward": {"fused_ms": round(b_ms, 4), "unfused_ms": round(ub_ms, 4), "speedup": round(ub_ms / b_ms, 3),
                     "unfused": "gemm(bf16 da) -> dact -> mxfp8 rows -> mxfp8 cols"},
        "pages": "up to 1.3x forward, 2.1x backward over unfused paths (unit microbenchmarks; GB200 figure)",
    }
    # -- the MXFP8-input FC1 (same fused epilogue on the block-scaled product
    #    of the row-wise MXFP8 x_perm and W1p): its two casts and the GEMM,
    #    each timed alone; not part of the step above, whose FC1 is bf16
    import ctypes as C
    from grouped_gemm_glu_gb300.ops import _p, _s
    # -- the MXFP8-input FC1 variant: the whole step with it (x_perm cast
    #    row-wise after the gather, both MXFP8 copies of W1 from one read in
    #    the forward, no W1 cast in the backward), as one graph, and its three
    #    forward calls one by one
    fc1_mx = None
    if w.out != "nvfp4":
        layer_mx = MoeLayer(g["W1"], g["W2"], w.T, w.k, R_cap, params, b1=g.get("b1"), expert_begin=w.expert_begin,
                            sm_margin=args.sm_margin, gated=w.gated, fc1_mxfp8=True)
        for _ in range(args.warmup):
            layer_mx.step(X, I, P, DO)
        graph_mx = layer_mx.capture(X, I, P, DO)
        for _ in range(args.warmup):
            graph_mx.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            graph_mx.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_graph_mx = e0.elapsed_time(e1) / args.steps
        by_name_mx = dict(layer_mx.step_calls(X, I, P, DO))
        mx_ms = {}
        for n_ in ("quant_x_rows", "quant_w1_dual", "fc1_mxfp8"):
            c_ = [(n_, by_name_mx[n_])]
            layer_mx.run(c_)
            mx_ms[n_] = timed_on(layer_mx, c_, na)
        st_mx = ops.read_status(layer_mx.status)
        if st_mx:
            raise SystemExit(f"device status {st_mx} in the MXFP8-FC1 step")
        E_, N1_, H_, F_ = w.E, w.N1, w.H, w.F
        fl_mx = 2 * R * H_ * N1_
        by_mx = (E_ * N1_ * H_ + R * H_) * (1 + 1 / 32) + R * N1_ * 2 + 2 * R * F_ * (1 + 1 / 32)
        by_dual = E_ * N1_ * H_ * 2 + 2 * E_ * N1_ * H_ * (1 + 1 / 32)
        peaks_ = load_peaks()
        fc1_mx = {"step_graph_ms": round(ms_graph_mx, 4),
                  "step_graph_ms_bf16_fc1": round(ms_graph, 4),
                  "x rows cast ms": round(mx_ms["quant_x_rows"], 4),
                  "W1 dual cast ms": round(mx_ms["quant_w1_dual"], 4),
                  "W1 dual cast frac_of_hbm_peak": round(by_dual / mx_ms["quant_w1_dual"] / 1e6 / peaks_["hbm"], 4),
                  "fc1 ms": round(mx_ms["fc1_mxfp8"], 4), "fc1 TFLOP/s": round(fl_mx / mx_ms["fc1_mxfp8"] / 1e9, 1),
                  "fc1 frac_of_fp8_peak": round(fl_mx / mx_ms["fc1_mxfp8"] / 1e9 / (2 * peaks_["bf16"]), 4),
                  "fc1 frac_of_hbm_roof": round(by_mx / mx_ms["fc1_mxfp8"] / 1e6 / peaks_["hbm"], 4),
                  "note": "layer with fc1_mxfp8=True: FC1 on MXFP8 x and W1 (fp8 = 2 x bf16 burst peak), W1's two "
                          "MXFP8 copies in one pass; the headline step keeps the bf16 FC1"}
        del graph_mx, layer_mx
    clocks = sampler.stop()
    st = ops.read_status(layer.status)
    if st:
        raise SystemExit(f"device status {st} after the timed regions")

    peaks = load_peaks()
    total_flops = 0.0
    kern = {}
    for n in names:
        fl, by, dt = kernel_model(n, w, R, Rp)
        total_flops += fl
        ms = per_kernel[n]
        ent = {"ms": round(ms, 4), "GB/s": round(by / ms / 1e6, 1)}
        if fl:
            # kernels timed one by one inside a short region run at the
            # burst clocks: the burst peak applies (fp8 = 2 x bf16, the
            # nominal dense ratio); the sustained figure is kept beside it
            peak = PEAK_RATIO[dt] * peaks["bf16"]
            peak_sus = PEAK_RATIO[dt] * peaks["bf16_sus"]
            ent["TFLOP/s"] = round(fl / ms / 1e9, 1)
            ent["frac_of_tensor_peak"] = round(fl / ms / 1e9 / peak, 4)
            ent["frac_of_sustained_tensor_peak"] = round(fl / ms / 1e9 / peak_sus, 4)
        ent["frac_of_hbm_peak"] = round(by / ms / 1e6 / peaks["hbm"], 4)
        kern[n] = ent

    times = torch.tensor([ms_graph, ms_eager, ms_e2e], dtype=torch.float64, device=dev)
    flops_t = torch.tensor([total_flops], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(times, op=dist.ReduceOp.MAX)
        dist.all_reduce(flops_t, op=dist.ReduceOp.SUM)
    ms_graph, ms_eager, ms_e2e = times.tolist()
    job_flops = flops_t.item()

    # dominant kernel and its roofline
    dom = max(names, key=lambda n: per_kernel[n])
    fl, by, dt = kernel_model(dom, w, R, Rp)
    ms = per_kernel[dom]
    peak_t = PEAK_RATIO[dt] * peaks["bf16"] if fl else None
    t_tensor = fl / (peak_t * 1e12) if fl else 0.0
    t_hbm = by / (peaks["hbm"] * 1e9)
    if fl and t_tensor >= t_hbm:
        roof = {"bound": "tensor", "achieved": round(fl / ms / 1e9, 1), "peak": round(peak_t, 1), "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": round(by / ms / 1e6, 1), "peak": peaks["hbm"], "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    tr = profile_traffic(dom) if w.E == base.E and w.name == WORKLOAD and not args.experts else None
    roof["traffic"] = tr
    if tr is not None:
        roof["traffic_source"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of this kernel on the 8-expert "
                                  "shard, x 32/8 (profiles/traffic_dsv3.json)")
    roof["kernel"] = dom
    if roof["bound"] == "hbm":
        roof["peak_source"] = f"of {peaks['src']} (HBM copy)"
    else:
        roof["peak_source"] = f"of {peaks['src']} ({dt} = {PEAK_RATIO[dt]:g} x bf16 burst)"
    roof["algorithmic"] = {"flops": fl, "bytes": by}

    # the metric's own quantity: TFLOP/s of the fused forward
    # (GroupGemm + Activation + Quantize/Transpose) and backward
    # (GroupGemm + dActivation + Quantize/Transpose) kernels and their
    # fraction of the dense bf16 tensor peak (burst: each is timed alone in a
    # short region), then both together
    fused = {}
    fl_sum = ms_sum = 0.0
    for n in (("fc1_glu_nvfp4", "dglu_nvfp4") if w.out == "nvfp4" else ("fc1_glu_quant", "dglu_quant")):
        fl_n, by_n, _ = kernel_model(n, w, R, Rp)
        tf = fl_n / per_kernel[n] / 1e9
        fused[n] = {"ms": round(per_kernel[n], 4), "TFLOP/s": round(tf, 1),
                    "frac_of_bf16_peak": round(tf / peaks["bf16"], 4),
                    "frac_of_bf16_sustained_peak": round(tf / peaks["bf16_sus"], 4),
                    "frac_of_hbm_roof": round(by_n / per_kernel[n] / 1e6 / peaks["hbm"], 4)}
        fl_sum += fl_n
        ms_sum += per_kernel[n]
    fused["fwd+bwd"] = {"ms": round(ms_sum, 4), "TFLOP/s": round(fl_sum / ms_sum / 1e9, 1),
                        "frac_of_bf16_peak": round(fl_sum / ms_sum / 1e9 / peaks["bf16"], 4)}
    fused["peak"] = {"bf16_burst_tflops": peaks["bf16"], "bf16_sustained_tflops": peaks["bf16_sus"],
                     "source": peaks["src"]}

    line = {
        "metric": METRIC,
        "value": round(job_flops / ms_graph / 1e9, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_graph, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16+nvfp4" if w.out == "nvfp4" else "bf16+mxfp8",
        "data": "synthetic (seeded; random-init weights N(0,1/H), x N(0,1), router logits N(0,1))",
        "config": {"workload": workload_desc(w), "T": w.T, "H": w.H, "E_local": w.E, "experts": w.n_experts,
                   "top_k": w.k, "F": w.F, "R_cap": R_cap, "routed_rows": R, "padded_rows": Rp,
                   "capacity_factor": CAPACITY_FACTOR, "l2": "inputs larger than L2 (no flush)",
                   "step": "one CUDA graph: " + " -> ".join(names), "parallelism": f"ep-shards x{world}",
                   "bf16_gemm_schedule": "dynamic (atomic tile counter)", "tail_swap_max_rows": 32},
        "roofline": roof,
        "fused_kernels": fused,
        "kernels": kern,
        "ablation_fused_vs_unfused": ablation,
        "fc1_mxfp8_variant": fc1_mx,
        "eager_ms_per_step": round(ms_eager, 4),
        # counted: the eager region's launches plus, for the two graph
        # regions, the kernel launches recorded into the captured step graph
        # times its replays
        "gpu_launches": int(launches + layer.graph_launches * 2 * args.steps),
        "clocks": clocks,
        "e2e": {"value": round(job_flops / ms_e2e / 1e9, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4)},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, _ = run_oracle_timed(inp, w, 1, 1, 20.0)
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
