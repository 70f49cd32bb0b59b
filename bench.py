#!/usr/bin/env python
"""MoE-layer throughput on GB300: the Kimi-K3-shape MXFP4 MoE layer through libk3moe.so.

Default workload: single-token decode (d_model 7168, d_ff 1536, 896 routed experts top-16 + 2 shared,
bf16 token N(0,1), fp32 N(0,1/d) router, MXFP4 experts with uniform E2M1 codes and E8M0 exponents
uniform in -6..-2). One step = one layer call (router, top-k, permutation, gate/up + GLU, down +
combine) on one batch of tokens. Steps rotate over `--layers` independent weight sets (4 x 15.8 GB),
so each step's inputs (341 MB at decode b=1) are larger than L2 and were not touched by the
previous step. Synthetic inputs (no checkpoint exists here): see synth/.

Prints ONE JSON line (rank 0). Under torchrun (--gpus N > 1) every rank runs an independent replica
(the layer has no exchange step on one GPU; weak scaling) and the time is the max over ranks.
`--impl reference` times the CPU oracle (fp64, plain loops) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
    # name: (tokens per step, seed, zipf s)
    "decode_b1": (1, 1, None),
    "decode_b64_zipf": (64, 2, 1.1),
    "prefill_4096": (4096, 3, None),
}
FALLBACK_HBM_GBS = 6800.0
# the metric of both arms (this library, and the oracle as the reference arm)
METRIC = "MoE-layer tokens/s (K3 shape, one layer) and fraction of HBM roofline"

# DRAM traffic per launch from an ncu capture, keyed by kernel; valid only while the kernel sources
# hash to the recorded value (see profiles/).
NCU_TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum of one launch (decode b=1: 16 routed + 2 shared
    # records, the same per launch at any expert count), profiles/k_tc_ffn_decode_b1.md
    "k_tc<gate/up>": (213776128, "220f8b4c3ca7401f"),
    "k_tc<down>": (107876352, "220f8b4c3ca7401f"),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=list(WORKLOADS) + ["stack4_zipf"], default="decode_b1")
    p.add_argument("--sweep", default="1,8,64,512,4096,16384",
                   help="stack4_zipf: token counts per layer call (one JSON line each)")
    p.add_argument("--layers", type=int, default=8,
                   help="independent weight sets rotated across steps (8: the router weights alone, 206 MB, exceed L2)")
    p.add_argument("--experts", type=int, default=None, help="override routed experts (small profiling case)")
    p.add_argument("--tokens", type=int, default=None, help="override tokens per layer call (small profiling case)")
    p.add_argument("--batches", type=int, default=64, help="distinct token batches rotated across steps")
    p.add_argument("--sample-every", type=int, default=8, help="phase-timed step every N steps")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--ref-budget-s", type=float, default=150.0)
    return p.parse_args()


def kernel_hash():
    """Hash of the sources of the projection kernels' device code (k_tc and the device headers it
    includes; k3moe_kernels.h holds host-side launch declarations only)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mxfp4_routed_expert_k3moe_gb300", "csrc")
    for f in ("k3moe_tc.cu", "k3moe_ptx.cuh", "k3moe_common.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
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
def kernels_per_layer(T, x_dtype):
    """Kernels one layer call launches: router, gate/up (with the GLU), down, combine, plus the
    tensor-core router GEMM and the bf16 splits of its operands from 16 tokens on."""
    n = 4
    if T >= 16:
        n += 2 + (1 if x_dtype == "f32" else 0)
    return n


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


def workload_config(workload, T, shape):
    """The keys that name the workload (the same in both arms' lines)."""
    return {"workload": workload, "tokens_per_layer_call": T, "d_model": shape.d_model, "d_ff": shape.d_ff,
            "n_routed": shape.n_routed, "top_k": shape.top_k, "n_shared": shape.n_shared}


def run_reference(args, rank, world):
    if rank != 0:
        return
    T, seed, zipf_s = WORKLOADS[args.workload]
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
    def __init__(self, shape, seed, layer, zipf_s, stride, dev):
        import torch
        self.W = torch.from_numpy(synth.router_weights(shape, seed, layer)).to(dev)
        self.bias = None if zipf_s is None else torch.from_numpy(synth.zipf_bias(shape, seed, zipf_s, layer)).to(dev)
        self.routed = torch.empty(shape.n_routed * stride, dtype=torch.uint8, device=dev)
        self.shared = torch.empty(max(1, shape.n_shared) * stride, dtype=torch.uint8, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        synth.records_device(shape, seed, layer, 0, shape.n_routed, self.routed.data_ptr(), stride, st)
        synth.records_device(shape, seed, layer, shape.n_routed, shape.n_shared, self.shared.data_ptr(), stride, st)
        # weight loading: records into the device order the kernels read (once, not timed)
        import mxfp4_routed_expert_k3moe_gb300 as k3
        cfg = k3.Config.make(shape.d_model, shape.d_ff, shape.n_routed, shape.top_k, shape.n_shared,
                             record_stride=stride)
        k3.pack_records(cfg, self.routed, shape.n_routed)
        k3.pack_records(cfg, self.shared, shape.n_shared)


def run_ours(args, rank, world, local_rank):
    import torch
    import mxfp4_routed_expert_k3moe_gb300 as k3

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    T, seed, zipf_s = WORKLOADS[args.workload]
    T = args.tokens or T
    base = synth.K3
    E = args.experts or base.n_routed
    shape = synth.LayerShape(base.d_model, base.d_ff, E, base.top_k, base.n_shared)
    stride = shape.record_stride
    d, f, k, S = shape.d_model, shape.d_ff, shape.top_k, shape.n_shared
    cfg = k3.Config.make(d, f, E, k, S, x_dtype=k3.X_BF16, record_stride=stride)
    layers = [LayerWeights(shape, seed, l, zipf_s, stride, dev) for l in range(args.layers)]
    nb = max(1, args.batches if T <= 64 else min(args.batches, 4))
    xs_host = np.stack([synth.tokens(shape, seed, T, "bf16", batch=b) for b in range(nb)])  # [nb, T, d] uint16
    xs = torch.from_numpy(xs_host.view(np.int16)).to(dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    ws = torch.zeros(k3.workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
    idx_out = torch.empty((T, k), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    def step(i, events=None, idx=None):
        L = layers[i % len(layers)]
        x = xs[i % nb]
        if events is None:
            k3.layer(cfg, x, T, L.W, L.bias, L.routed, L.shared, y, ws)
        else:
            k3.layer_timed(cfg, x, T, L.W, L.bias, L.routed, L.shared, y, ws, events, topk_idx=idx)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if k3.check_device_status(ws) != k3.OK:
        raise RuntimeError("device status check failed after warm-up")

    # phase events for sampled steps (all recorded inside the timed region, on the launching stream)
    n_samp = (args.steps + args.sample_every - 1) // args.sample_every
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_samp)]
    st = torch.cuda.current_stream()
    for e4 in ev:  # materialise the handles
        for e in e4:
            e.record(st)
    idx_samples = torch.empty((n_samp, T, k), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(st)
    for i in range(args.steps):
        if i % args.sample_every == 0:
            s = i // args.sample_every
            step(i, [e.cuda_event for e in ev[s]], idx_samples[s])
        else:
            step(i)
    end.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed_ms = start.elapsed_time(end)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
        torch.distributed.barrier()
    if k3.check_device_status(ws) != k3.OK:
        raise RuntimeError("device status check failed in the timed region")

    # per-kernel device times of the sampled steps (events between the kernels; the gate/up kernel
    # finishes h itself, so its two closing events are adjacent)
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
    peak, peak_kind = hbm_peak()
    kernels = {"k_tc<gate/up>": (gateup_ms, bytes_gateup), "k_tc<down>": (down_ms, bytes_down),
               "k_route": (route_ms, bytes_route)}
    dom = max(kernels, key=lambda n: kernels[n][0])
    dom_ms, dom_bytes = kernels[dom]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = None
    # (the recorded counters are those of the decode b=1 launch; other workloads report none)
    if args.workload == "decode_b1" and T == 1 and dom in NCU_TRAFFIC and NCU_TRAFFIC[dom][1] == kernel_hash():
        traffic = NCU_TRAFFIC[dom][0]
    ms_per_step = elapsed_ms / args.steps
    value = world * T * args.steps / (elapsed_ms * 1e-3)

    line = {
        "metric": METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp4 weights x bf16 activations, fp32 accumulate", "data": "synthetic",
        "config": {**workload_config(args.workload, T, shape), "weight_sets_rotated": args.layers,
                   "l2": f"inputs larger than L2: each step reads {bytes_layer / 1e6:.1f} MB of weights from a "
                         f"different layer than the previous step ({args.layers} layers rotated)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)"
                     if peak_kind == "measured" else "fallback",
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms},
        "kernels_ms": {"k_route": route_ms, "k_tc<gate/up> (with the GLU)": gateup_ms, "k_tc<down>": down_ms,
                       "k_combine": combine_ms, "sampled_steps": n_samp,
                       "note": "events between the kernels remove their launch overlap in the sampled steps"},
        "layer_roofline": {"bytes_per_step": bytes_layer, "achieved_gbs": bytes_layer / (ms_per_step * 1e-3) / 1e9,
                           "frac": bytes_layer / (ms_per_step * 1e-3) / 1e9 / peak},
        "distinct_experts_per_step": U,
        "gpu_launches": kernels_per_layer(T, "bf16") * args.steps,
        "clocks": clk,
    }

    if not args.no_e2e:
        line["e2e"] = e2e(args, k3, cfg, layers, xs_host, T, d, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = max(1, min(cpu_cores(), 16))
        secs = oracle_sample(synth.K3, seed, zipf_s, "bf16", n)
        line["cpu_baseline"] = {"value": n / secs, "unit": "tokens/s", "cores": n, "kind": "oracle",
                                "sample": f"{n} tokens of layer 0 ({args.workload} shape), one oracle call, "
                                          f"OpenMP over tokens, {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def e2e(args, k3, cfg, layers, xs_host, T, d, dev):
    """Same metric through the public call with host buffers: pinned x -> device, layer, y -> pinned host."""
    import torch
    nb = xs_host.shape[0]
    xh = torch.from_numpy(xs_host.view(np.int16)).pin_memory()
    yh = torch.empty((T, d), dtype=torch.float32).pin_memory()
    xd = torch.empty((T, d), dtype=torch.int16, device=dev)
    yd = torch.empty((T, d), dtype=torch.float32, device=dev)
    ws = torch.zeros(k3.workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
    steps = max(10, args.steps // 4)
    st = torch.cuda.current_stream()

    def one(i):
        L = layers[i % len(layers)]
        xd.copy_(xh[i % nb], non_blocking=True)
        k3.layer(cfg, xd, T, L.W, L.bias, L.routed, L.shared, yd, ws)
        yh.copy_(yd, non_blocking=True)

    for i in range(min(args.warmup, 20)):
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


def run_stack(args, rank, world, local_rank):
    """stack4_zipf: 4 independent layers (seeds 40-43, Zipf 1.1 routing bias), pre-norm residual
    x <- x + Layer_l(RMSNorm(x)) with fp32 activations, for each token count of --sweep. One step =
    the 4 layers on one batch; one JSON line per token count (a curve, not the headline)."""
    import torch
    import mxfp4_routed_expert_k3moe_gb300 as k3

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shape = synth.K3
    stride = shape.record_stride
    d, E, k, S = shape.d_model, shape.n_routed, shape.top_k, shape.n_shared
    layers = [LayerWeights(shape, 40 + l, l, 1.1, stride, dev) for l in range(4)]
    cfg = k3.Config.make(d, shape.d_ff, E, k, S, x_dtype=k3.X_F32, record_stride=stride)
    peak, peak_kind = hbm_peak()
    for T in [int(t) for t in args.sweep.split(",")]:
        x = torch.from_numpy(synth.tokens(shape, 40, T, "f32")).to(dev)
        xn = torch.empty_like(x)
        y = torch.empty_like(x)
        ws = torch.zeros(k3.workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
        idx = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in range(4)]

        def step(keep_idx=False):
            for l, L in enumerate(layers):
                k3.rmsnorm(x, T, d, 1e-6, xn)
                k3.layer(cfg, xn, T, L.W, L.bias, L.routed, L.shared, y, ws, topk_idx=idx[l] if keep_idx else None)
                k3.residual_add(x, y, T * d)

        steps = max(3, min(args.steps, int(2e5 // max(T, 1))))
        for _ in range(max(3, min(args.warmup, 5))):
            step()
        step(keep_idx=True)
        torch.cuda.synchronize()
        if k3.check_device_status(ws) != k3.OK:
            raise RuntimeError("device status check failed in the stack")
        U = [int(torch.unique(i).numel()) for i in idx]
        clocks = ClockSampler(local_rank)
        clocks.start()
        time.sleep(0.2)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            step()
        b.record()
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = a.elapsed_time(b) / steps
        rec = shape.record_bytes
        bytes_step = sum((u + S) * rec + E * d * 4 + T * d * 4 * 2 for u in U)
        line = {"metric": "MoE-layer tokens/s (K3 shape, 4-layer stack with pre-norm residual)",
                "value": 4 * T / (ms * 1e-3), "unit": "layer-tokens/s", "stack_tokens_per_s": T / (ms * 1e-3),
                "ms_per_step": ms, "steps": steps, "higher_is_better": True, "dtype": "mxfp4 weights x fp32 activations, fp32 accumulate",
                "data": "synthetic", "config": {"workload": "stack4_zipf", "tokens_per_layer_call": T, "layers": 4},
                "distinct_experts_per_layer": U,
                "layer_roofline": {"bytes_per_step": bytes_step, "achieved_gbs": bytes_step / (ms * 1e-3) / 1e9,
                                   "frac": bytes_step / (ms * 1e-3) / 1e9 / peak, "peak": peak, "peak_kind": peak_kind},
                "clocks": clk}
        if rank == 0:
            print(json.dumps(line), flush=True)
        del ws, x, xn, y
        torch.cuda.empty_cache()


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
    if args.workload == "stack4_zipf":
        run_stack(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
