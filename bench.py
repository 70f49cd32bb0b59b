#!/usr/bin/env python
"""MoE-layer throughput on GB300: the Kimi-K3-shape MXFP4 MoE layer through libk3moe.so.

Shapes (all workloads): d_model 7168, d_ff 1536, 896 routed experts top-16 + 2 shared, fp32 N(0,1/d)
router, MXFP4 experts with uniform E2M1 codes and E8M0 exponents uniform in -6..-2. Synthetic inputs
(no checkpoint exists here): see synth/.

Headline (`value`): single-token decode, bf16 token N(0,1). One step = one layer call (router, top-k,
permutation, gate/up + GLU, down + combine) on one token. Steps rotate over `--layers` independent
weight sets, so each step's inputs (341.6 MB) are larger than L2 and were not touched by the
previous step. Exactly --steps steps are timed, with nothing else inside the timed region; the
per-kernel times come from a separate pass of event-bracketed steps afterwards.

The same JSON line carries, under "workloads", the other configurations the metric names, each timed
the same way: batched decode (64 tokens, Zipf(1.1)-skewed routing bias), prefill (4096 tokens) and a
4-layer stack with pre-norm residual at 1 and 64 tokens.

Prints ONE JSON line (rank 0). Under torchrun (--gpus N > 1) every rank runs an independent replica
(the layer has no exchange step on one GPU; weak scaling) and the time is the max over ranks.
`--impl reference` times the CPU oracle (fp64, plain loops) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

WORKLOADS = {
    # name: (tokens per step, seed, zipf s, weight sets rotated)
    "decode_b1": (1, 1, None, 8),
    "decode_b64_zipf": (64, 2, 1.1, 2),
    "prefill_4096": (4096, 3, None, 1),
}
# Activation mode of the library per workload: from 3 tokens on the layer runs with h as two E4M3 terms
# (K3MOE_ACT_BF16H, bf16-class h, output within the same 2e-3 bound); each such line also reports the
# exact mode's time. One token is the same in both modes (eight E2M1 terms).
BF16H_MIN_T = 3
STACK_TOKENS = (1, 64)
LAUNCH_COVER_CYCLES = 200_000  # ~100 us at 2 GHz: longer than the host needs to queue the first step
FALLBACK_HBM_GBS = 6800.0
NOMINAL_FP4_TFLOPS = 13500.0   # dense FP4 tensor peak of a GB300 (nominal)
NOMINAL_FP8_TFLOPS = 4500.0    # dense FP8/FP6/FP4-as-f8f6f4 tensor peak (nominal)
# the metric of both arms (this library, and the oracle as the reference arm)
METRIC = "MoE-layer tokens/s (K3 shape, one layer) and fraction of HBM roofline"

# Counters from ncu captures of the projection kernels, per launch, keyed by (kernel, workload); valid
# only while the kernel sources hash to the recorded value (the summaries under profiles/ give the
# commands): dram__bytes_read.sum + dram__bytes_write.sum of a decode launch (the capture used 128
# routed experts: a launch reads the same 16 + 2 records as at 896), and the tensor pipe's active
# fraction (sm__pipe_tensor_cycles_active, of elapsed) at the prefill proxy of 512 tokens x 128 experts.
NCU_COUNTERS = {
    ("k_tc<gate/up>", "decode_b1"): {"traffic": 213953024, "hash": "4a8581d337f38b99"},
    ("k_tc<down>", "decode_b1"): {"traffic": 108093440, "hash": "4a8581d337f38b99"},
    ("k_tc<gate/up>", "prefill_4096"): {"tensor_active": 0.3122, "hash": "4a8581d337f38b99",
                                        "case": "ncu at 512 tokens x 128 experts (64 tokens per expert), "
                                                "h as two E4M3 terms"},
    ("k_tc<down>", "prefill_4096"): {"tensor_active": 0.2375, "hash": "4a8581d337f38b99",
                                     "case": "ncu at 512 tokens x 128 experts (64 tokens per expert), "
                                             "h as two E4M3 terms"},
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=list(WORKLOADS), default="decode_b1", help="the headline workload")
    p.add_argument("--extra", default="decode_b64_zipf,prefill_4096,stack4_zipf",
                   help="other workloads reported in the same line ('' for none)")
    p.add_argument("--layers", type=int, default=None, help="weight sets rotated (default per workload)")
    p.add_argument("--experts", type=int, default=None, help="override routed experts (small profiling case)")
    p.add_argument("--tokens", type=int, default=None, help="override tokens per layer call (small profiling case)")
    p.add_argument("--phase-steps", type=int, default=24, help="event-bracketed steps of the per-kernel pass")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--ref-budget-s", type=float, default=150.0)
    return p.parse_args()


def kernel_hash():
    """Hash of the sources of the projection kernels' device code (k_tc and the device headers it
    includes; k3moe_kernels.h holds host-side launch declarations only), without comments, blank
    lines and indentation, so that a change of the comments keeps the counters taken on the code."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp4_routed_expert_k3moe_gb300", "csrc")
    for f in ("k3moe_tc.cu", "k3moe_ptx.cuh", "k3moe_common.cuh"):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"//[^\n]*", "", text)  # (no // inside string literals in these files)
        lines = [ln.strip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle (CPU baseline)
def oracle_sample(shape, seed, zipf_s, x_dtype, n_tokens):
    """Time the oracle on n_tokens tokens of layer 0 (records generated outside the timed part)."""
    import oracle
    W = synth.router_weights(shape, seed, 0)
    bias = None if zipf_s is None else synth.zipf_bias(shape, seed, zipf_s, 0)
    x = synth.tokens(shape, seed, n_tokens, x_dtype, batch=999)
    xf = synth.tokens_as_f64(x, x_dtype)
    experts = set()
    for t in range(n_tokens):
        experts.update(int(e) for e in oracle.route_token(xf[t], W, shape.top_k, bias)[1])
    ids = sorted(experts)
    recs = synth.records_host(shape, seed, 0, ids + [shape.n_routed + s for s in range(shape.n_shared)])
    routed = {e: recs[i] for i, e in enumerate(ids)}
    shared = list(recs[len(ids):])
    t0 = time.perf_counter()
    oracle.layer(x, x_dtype, W, bias, routed, shared, shape.d_model, shape.d_ff, shape.top_k)
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(workload, seed, zipf_s):
    n = max(1, min(cpu_cores(), 16))
    secs = oracle_sample(synth.K3, seed, zipf_s, "bf16", n)
    return {"value": n / secs, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{n} tokens of layer 0 ({workload} shape), one oracle call, OpenMP over tokens, {secs:.1f} s"}


def workload_config(workload, T, shape):
    """The keys that name the workload (the same in both arms' lines)."""
    return {"workload": workload, "tokens_per_layer_call": T, "d_model": shape.d_model, "d_ff": shape.d_ff,
            "n_routed": shape.n_routed, "top_k": shape.top_k, "n_shared": shape.n_shared}


def run_reference(args, rank, world):
    if rank != 0:
        return
    T, seed, zipf_s, _ = WORKLOADS[args.workload]
    shape = synth.K3
    cores = cpu_cores()
    n = max(1, min(cores, 16))
    # warmup: the first oracle call also compiles the C oracle
    warm = min(args.warmup, 1)
    for _ in range(warm):
        oracle_sample(shape, seed, zipf_s, "bf16", 1)
    times = []
    t_start = time.perf_counter()
    while len(times) < args.steps:
        times.append(oracle_sample(shape, seed, zipf_s, "bf16", n))
        if time.perf_counter() - t_start > args.ref_budget_s:
            break
    total = sum(times)
    value = len(times) * n / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 0, "steps": len(times), "warmup": warm, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, T, shape),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(n, cores), "kind": "oracle",
                         "sample": f"{len(times)} oracle layer calls x {n} tokens of the {args.workload} shape "
                                   f"(each step a bounded sample; stops after {args.ref_budget_s:.0f} s)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
class LayerWeights:
    """One layer's weights on the device, loaded the way a user loads them: records generated on the
    device, put into the device order (k3moe_pack_records) and the router's bf16 parts prepared
    (k3moe_prepare_router), once, outside any timed region."""

    def __init__(self, k3, cfg, shape, seed, layer, zipf_s, stride, dev):
        import torch
        self.W = torch.from_numpy(synth.router_weights(shape, seed, layer)).to(dev)
        self.bias = None if zipf_s is None else torch.from_numpy(synth.zipf_bias(shape, seed, zipf_s, layer)).to(dev)
        self.routed = torch.empty(shape.n_routed * stride, dtype=torch.uint8, device=dev)
        self.shared = torch.empty(max(1, shape.n_shared) * stride, dtype=torch.uint8, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        synth.records_device(shape, seed, layer, 0, shape.n_routed, self.routed.data_ptr(), stride, st)
        synth.records_device(shape, seed, layer, shape.n_routed, shape.n_shared, self.shared.data_ptr(), stride, st)
        k3.pack_records(cfg, self.routed, shape.n_routed)
        k3.pack_records(cfg, self.shared, shape.n_shared)
        self.parts = torch.empty(k3.router_parts_bytes(cfg) // 2, dtype=torch.int16, device=dev)
        k3.prepare_router(cfg, self.W, self.parts)


def max_over_ranks(ms, world, device="cuda"):
    """The slowest rank's time: every rank gets the largest of the ranks' `ms` (all-reduce MAX over the
    default process group; `device` is where the collective's tensor lives: cuda for NCCL, cpu for
    gloo). One rank returns its own time."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_step, steps, ms):
    """Whole-job throughput: the units all `world` ranks processed in `steps` steps (each rank
    `units_per_step` per step: replicas, weak scaling) over the slowest rank's `ms` milliseconds."""
    return world * units_per_step * steps / (ms * 1e-3)


def timed(step, steps, world, local_rank, warmup=0, check=None):
    """Device time of exactly `steps` calls of step(i), bracketed by a barrier and synchronize on both
    sides (CUDA events on the launching stream), with nvidia-smi clocks sampled meanwhile. The sampler
    starts first; the `warmup` untimed calls run right before the timed ones (then `check()`), so that
    the timed region does not start from an idle GPU."""
    import torch
    st = torch.cuda.current_stream()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if check:
        check()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a short sleep kernel ahead of the start event keeps the host's launch latency of the first step
    # out of the device timing (the first steps are queued by the time the GPU reaches the event)
    torch.cuda._sleep(LAUNCH_COVER_CYCLES)
    a.record(st)
    for i in range(steps):
        step(i)
    b.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = a.elapsed_time(b)
    if world > 1:
        ms = max_over_ranks(ms, world, "cuda")
        torch.distributed.barrier()
    return ms, clk


def run_layer_workload(args, k3, name, T, seed, zipf_s, n_sets, steps, warmup, world, local_rank, with_cpu):
    """One layer workload: timed steps, the per-kernel pass, e2e and the CPU baseline."""
    import torch
    dev = torch.device("cuda", local_rank)
    base = synth.K3
    E = args.experts or base.n_routed
    shape = synth.LayerShape(base.d_model, base.d_ff, E, base.top_k, base.n_shared)
    stride = shape.record_stride
    d, f, k, S = shape.d_model, shape.d_ff, shape.top_k, shape.n_shared
    bf16h = T >= BF16H_MIN_T
    cfg = k3.Config.make(d, f, E, k, S, x_dtype=k3.X_BF16, record_stride=stride,
                         act_mode=k3.ACT_BF16H if bf16h else k3.ACT_EXACT)
    layers = [LayerWeights(k3, cfg, shape, seed, l, zipf_s, stride, dev) for l in range(n_sets)]
    nb = 64 if T <= 64 else 2
    xs_host = np.stack([synth.tokens(shape, seed, T, "bf16", batch=b) for b in range(nb)])  # [nb, T, d] uint16
    xs = torch.from_numpy(xs_host.view(np.int16)).to(dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    ws = torch.zeros(k3.workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def step(i):
        L = layers[i % len(layers)]
        k3.layer(cfg, xs[i % nb], T, L.W, L.bias, L.routed, L.shared, y, ws, w_parts=L.parts)

    def check_warm():
        if k3.check_device_status(ws) != k3.OK:
            raise RuntimeError(f"{name}: device status check failed after warm-up")

    elapsed_ms, clk = timed(step, steps, world, local_rank, warmup=warmup, check=check_warm)
    if k3.check_device_status(ws) != k3.OK:
        raise RuntimeError(f"{name}: device status check failed in the timed region")
    exact = None
    if bf16h:  # the same steps in the exact mode (h as three E4M3 terms), timed the same way
        cfg_x = k3.Config.make(d, f, E, k, S, x_dtype=k3.X_BF16, record_stride=stride, act_mode=k3.ACT_EXACT)

        def step_x(i):
            L = layers[i % len(layers)]
            k3.layer(cfg_x, xs[i % nb], T, L.W, L.bias, L.routed, L.shared, y, ws, w_parts=L.parts)

        ms_x, _ = timed(step_x, steps, world, local_rank, warmup=warmup)
        if k3.check_device_status(ws) != k3.OK:
            raise RuntimeError(f"{name}: device status check failed in the exact-mode pass")
        exact = {"act_mode": "exact (h as three E4M3 terms, within 2^-12 of each block maximum)", "value": job_rate(world, T, steps, ms_x),
                 "unit": "tokens/s", "ms_per_step": ms_x / steps}

    # per-kernel pass (after the headline timing): events recorded between the kernels of each step on
    # the launching stream; the gate/up kernel finishes h itself, so its two closing events are adjacent
    st = torch.cuda.current_stream()
    n_samp = max(3, args.phase_steps if T <= 64 else min(args.phase_steps, 6))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_samp)]
    for e6 in ev:  # materialise the handles
        for e in e6:
            e.record(st)
    idx_samples = torch.empty((n_samp, T, k), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    for s in range(n_samp):
        L = layers[s % len(layers)]
        k3.layer_timed(cfg, xs[s % nb], T, L.W, L.bias, L.routed, L.shared, y, ws, [e.cuda_event for e in ev[s]],
                       topk_idx=idx_samples[s], w_parts=L.parts)
    torch.cuda.synchronize()
    ph = np.array([[ev[s][j].elapsed_time(ev[s][j + 1]) for j in range(5)] for s in range(n_samp)])
    route_ms, gateup_ms, _, down_ms, combine_ms = ph.mean(axis=0)
    idxs = idx_samples.cpu().numpy()
    U = float(np.mean([len(np.unique(idxs[s])) for s in range(n_samp)]))

    rec = shape.record_bytes
    mat = f * d // 2 + f * d // 32
    # algorithmic bytes: the expert records the step must read, the router weights, x read once and
    # y written once; activation terms, partial sums and h are implementation traffic (not counted)
    bytes_gateup = (U + S) * 2 * mat
    bytes_down = (U + S) * mat
    bytes_route = E * d * 4 + T * d * 2
    bytes_layer = (U + S) * rec + E * d * 4 + T * d * 2 + T * d * 4
    # implementation traffic the layer adds on top (written and read back once each): the
    # per-position down outputs [P, d] fp32 (h's E4M3 terms and x's in position order are not counted)
    P = T * (k + S)
    bytes_partials = 2 * P * d * 4
    # algorithmic flops: 2 per multiply-add of the three projections of every selected (token, expert)
    flops_ffn = 2.0 * 3 * d * f * P
    peak, peak_kind = hbm_peak()
    kernels = {"k_tc<gate/up>": (gateup_ms, bytes_gateup, flops_ffn * 2 / 3),
               "k_tc<down>": (down_ms, bytes_down, flops_ffn / 3), "k_route": (route_ms, bytes_route, 0.0)}
    dom = max(kernels, key=lambda n: kernels[n][0])
    dom_ms, dom_bytes, dom_flops = kernels[dom]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    cnt = NCU_COUNTERS.get((dom, name))
    valid = cnt is not None and cnt["hash"] == kernel_hash() and T == WORKLOADS[name][0] and E == 896
    if valid and "traffic" not in cnt:
        cnt = {**cnt, "traffic": None}
    ms_per_step = elapsed_ms / steps
    out = {
        "value": job_rate(world, T, steps, elapsed_ms), "unit": "tokens/s", "steps": steps, "warmup": warmup,
        "ms_per_step": ms_per_step,
        "config": {**workload_config(name, T, shape), "weight_sets_rotated": n_sets,
                   "act_mode": "bf16h (h as two E4M3 terms, bf16-class)" if bf16h else "exact",
                   "l2": f"inputs larger than L2: each step reads {bytes_layer / 1e6:.1f} MB of weights "
                         f"({n_sets} weight set(s) rotated, {nb} token batch(es))"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": cnt["traffic"] if valid else None,
                     "peak_kind": "measured (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms},
        "kernels_ms": {"router": route_ms, "k_tc<gate/up> (with the GLU)": gateup_ms, "k_tc<down>": down_ms,
                       "k_combine": combine_ms, "steps": n_samp,
                       "note": "separate pass after the timed steps; events between the kernels remove their "
                               "launch overlap"},
        "layer_roofline": {"bytes_per_step": bytes_layer, "achieved_gbs": bytes_layer / (ms_per_step * 1e-3) / 1e9,
                           "frac": bytes_layer / (ms_per_step * 1e-3) / 1e9 / peak,
                           "implementation_bytes_per_step": bytes_partials,
                           "frac_with_implementation_bytes":
                               (bytes_layer + bytes_partials) / (ms_per_step * 1e-3) / 1e9 / peak},
        "distinct_experts_per_step": U,
        "gpu_launches": (4 if T < 16 else (5 if T < 256 else 6)) * steps,
        "clocks": clk,
    }
    if T >= 16:
        tc = {"algorithmic_tflop_per_step": flops_ffn / 1e12,
              "fp4_frac_nominal": flops_ffn / (ms_per_step * 1e-3) / 1e12 / NOMINAL_FP4_TFLOPS,
              "dominant_kernel_fp4_frac_nominal": dom_flops / (dom_ms * 1e-3) / 1e12 / NOMINAL_FP4_TFLOPS,
              "peak_kind": f"nominal dense FP4 {NOMINAL_FP4_TFLOPS:.0f} TFLOP/s"}
        if valid and "tensor_active" in cnt:
            tc["tensor_pipe_active_ncu"] = {"value": cnt["tensor_active"], "kernel": dom, "case": cnt["case"]}
        out["tensor"] = tc
    if exact is not None:
        out["exact_mode"] = exact
    if not args.no_e2e:
        out["e2e"] = e2e(k3, cfg, layers, xs_host, T, d, dev, steps, warmup)
    if with_cpu and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(name, seed, zipf_s)
    del layers, xs, ws, y
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def e2e(k3, cfg, layers, xs_host, T, d, dev, steps, warmup):
    """Same metric through the public call with host buffers: pinned x -> device, layer, y -> pinned host."""
    import torch
    nb = xs_host.shape[0]
    xh = torch.from_numpy(xs_host.view(np.int16)).pin_memory()
    yh = torch.empty((T, d), dtype=torch.float32).pin_memory()
    xd = torch.empty((T, d), dtype=torch.int16, device=dev)
    yd = torch.empty((T, d), dtype=torch.float32, device=dev)
    ws = torch.zeros(k3.workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()

    def one(i):
        L = layers[i % len(layers)]
        xd.copy_(xh[i % nb], non_blocking=True)
        k3.layer(cfg, xd, T, L.W, L.bias, L.routed, L.shared, yd, ws, w_parts=L.parts)
        yh.copy_(yd, non_blocking=True)

    for i in range(max(3, min(warmup, 20))):
        one(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for i in range(steps):
        one(i)
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": T * steps / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": T * d * 2,
            "d2h_bytes_per_step": T * d * 4, "steps": steps}


def run_stack(args, k3, world, local_rank):
    """stack4_zipf: 4 independent layers (seeds 40-43, Zipf 1.1 routing bias), pre-norm residual
    x <- x + Layer_l(RMSNorm(x)) with fp32 activations. One step = the 4 layers on one batch. Timed
    two ways: with the residual add and the next layer's norm fused in k3moe_residual_rmsnorm (whose
    early launch lets the next layer's router stream its weights during it), and with the separate
    k3moe_residual_add + k3moe_rmsnorm calls."""
    import torch
    dev = torch.device("cuda", local_rank)
    shape = synth.K3
    stride = shape.record_stride
    d, E, k, S = shape.d_model, shape.n_routed, shape.top_k, shape.n_shared
    cfg = k3.Config.make(d, shape.d_ff, E, k, S, x_dtype=k3.X_F32, record_stride=stride)
    layers = [LayerWeights(k3, cfg, shape, 40 + l, l, 1.1, stride, dev) for l in range(4)]
    peak, peak_kind = hbm_peak()
    res = {}
    for T in STACK_TOKENS:
        x0 = torch.from_numpy(synth.tokens(shape, 40, T, "f32")).to(dev)
        x = x0.clone()
        xn = torch.empty_like(x)
        y = torch.empty_like(x)
        ws = torch.zeros(k3.workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
        idx = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in range(4)]

        def fused(keep_idx=False):
            k3.rmsnorm(x, T, d, 1e-6, xn)
            for l, L in enumerate(layers):
                k3.layer(cfg, xn, T, L.W, L.bias, L.routed, L.shared, y, ws, topk_idx=idx[l] if keep_idx else None,
                         w_parts=L.parts)
                k3.residual_rmsnorm(x, y, T, d, 1e-6, xn)

        def separate():
            for L in layers:
                k3.rmsnorm(x, T, d, 1e-6, xn)
                k3.layer(cfg, xn, T, L.W, L.bias, L.routed, L.shared, y, ws, w_parts=L.parts)
                k3.residual_add(x, y, T * d)

        steps = max(3, min(args.steps, 200 if T <= 64 else 20))
        out = {}
        for label, fn in (("fused", fused), ("separate", separate)):
            x.copy_(x0)
            ms, clk = timed(lambda i: fn(), steps, world, local_rank, warmup=3)
            out[label] = {"layer_tokens_per_s": job_rate(world, 4 * T, steps, ms), "ms_per_step": ms / steps,
                          "steps": steps, "clocks": clk}
        x.copy_(x0)
        fused(keep_idx=True)
        torch.cuda.synchronize()
        if k3.check_device_status(ws) != k3.OK:
            raise RuntimeError("device status check failed in the stack")
        U = [int(torch.unique(i).numel()) for i in idx]
        rec = shape.record_bytes
        bytes_step = sum((u + S) * rec + E * d * 4 + T * d * 4 * 2 for u in U)
        ms = out["fused"]["ms_per_step"]
        res[f"T{T}"] = {**out, "distinct_experts_per_layer": U,
                        "layer_roofline": {"bytes_per_step": bytes_step, "frac": bytes_step / (ms * 1e-3) / 1e9 / peak,
                                           "peak": peak, "peak_kind": peak_kind}}
        del ws, x, x0, xn, y
    del layers
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {"metric": "layer-tokens/s of a 4-layer stack with pre-norm residual (x <- x + Layer(RMSNorm(x)))",
            "config": {"workload": "stack4_zipf", "layers": 4, "x_dtype": "f32", "zipf_s": 1.1}, **res}


def run_ours(args, rank, world, local_rank):
    import torch
    import mxfp4_routed_expert_k3moe_gb300 as k3

    torch.cuda.set_device(local_rank)
    T, seed, zipf_s, n_sets = WORKLOADS[args.workload]
    T = args.tokens or T
    n_sets = args.layers or n_sets
    head = run_layer_workload(args, k3, args.workload, T, seed, zipf_s, n_sets, args.steps, args.warmup, world,
                              local_rank, with_cpu=rank == 0 and world == 1)
    extra = {}
    for name in [w for w in args.extra.split(",") if w]:
        if name == args.workload:
            continue
        if name == "stack4_zipf":
            extra[name] = run_stack(args, k3, world, local_rank)
            continue
        Tw, sw, zw, nw = WORKLOADS[name]
        # the same step count as the headline, capped so that a workload takes seconds
        steps = max(3, min(args.steps, 400 if Tw <= 64 else 40))
        extra[name] = run_layer_workload(args, k3, name, Tw, sw, zw, nw, steps, max(3, min(args.warmup, 5)), world,
                                         local_rank, with_cpu=rank == 0 and world == 1)
    launches = head["gpu_launches"] + sum(v.get("gpu_launches", 0) for v in extra.values())
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp4 weights x bf16 activations, fp32 accumulate", "data": "synthetic",
        "config": {**head["config"], "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": head["roofline"], "layer_roofline": head["layer_roofline"], "kernels_ms": head["kernels_ms"],
        "distinct_experts_per_step": head["distinct_experts_per_step"],
        "gpu_launches": head["gpu_launches"], "gpu_launches_all_workloads": launches, "clocks": head["clocks"],
    }
    for key in ("e2e", "cpu_baseline"):
        if key in head:
            line[key] = head[key]
    line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
