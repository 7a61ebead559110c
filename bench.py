#!/usr/bin/env python
"""Throughput of the routed Q8_0 MoE feed-forward step on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl fw|reference]

With no --workload, every workload of the layer shapes is timed in one run and
the headline line is the largest one, large2048 (H=7168, I=2048, 256 routed
experts top-8 + 1 shared, T=2048 tokens per call, 2 layers of 12.7 GB cycled);
the others (tiny, dec1, dec16, pre4096, large1) are reported under
"per_config", each with its own roofline. --workload NAME times one workload
as the headline.

A step of a workload is one pass of the whole hot path (route, experts,
combine) over every layer of the workload for each of its hidden batches
(64 rows for T = 1, fewer batches for larger T), all on one stream, captured
once as a CUDA graph by the library (fw_moe_graph_create) and replayed. value = tokens x layer-calls per second.
Every workload cycles more layers than L2 holds (no flush needed). Timing: CUDA
events around K graph replays, repeated 5 times, median.

The path does not shard: under torch.distributed.run with N processes (one
per GPU) every rank runs an independent replica of the same workload on its
own GPU (weak scaling; the only collectives are the barriers around the timed
region and the max over ranks of its time). --gpus N > 1 without such a launch
reports that it is unavailable.

--impl reference times the fp64 oracle on the host cores instead (rank 0),
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

HEADLINE = "large2048"
ALL_WORKLOADS = ("tiny", "dec1", "dec16", "pre4096", "large1", "large2048")
REPEATS = 5
# Workloads that run on another workload's layers (same shapes; the weights
# are made once): multi-slot decode on the batch-1 decode layers, and the
# large MoE's decode run on its prefill layers.
SHARED_LAYERS = {"dec16": "dec1", "large1": "large2048"}


def n_x_rows(w):
    """Distinct hidden batches cycled per step: 64 rows at T=1, fewer for larger T."""
    return max(1, 64 // w.T)


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default=None, choices=sorted(synth.WORKLOADS))
    p.add_argument("--impl", default="fw", choices=["fw", "reference"])
    p.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    p.add_argument("--experts", type=int, default=0,
                   help="override E (a smaller case for profiling: at T = 1 the expert work per call is the same)")
    p.add_argument("--tokens", type=int, default=0,
                   help="override T (with --experts: a smaller case with the same rows per expert, for profiling)")
    p.add_argument("--repeats", type=int, default=REPEATS)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--act-q8", action="store_true",
                   help="Q8 activations on the decode path (an option of the layer; the default is bf16)")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="host time budget of the oracle baseline (and of the whole reference arm)")
    return p.parse_args(argv)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's time: all_reduce MAX (NCCL on GPU ranks, gloo on CPU)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Units all ranks processed over the slowest rank's time (weak scaling)."""
    return units_per_rank * world / seconds_max


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# Source files each timed kernel is built from: a profile summary under
# profiles/ records their hash, and its DRAM traffic is reported only while
# the kernel is unchanged since the counters were taken.
KERNEL_SOURCES = {
    "decode_experts": ("decode.cu", "routing.cuh", "internal.cuh"),
    "prefill_gateup": ("prefill.cu", "internal.cuh"),
}


def code_only(text: str) -> str:
    """A CUDA source without its comments, trailing blanks and empty lines: a
    change of comments alone leaves the measured code, and so the hash, as it
    was."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def source_hash(texts) -> str:
    h = hashlib.sha256()
    for t in texts:
        h.update(code_only(t).encode())
    return h.hexdigest()


def kernel_source_hash(kernel: str) -> str:
    texts = []
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "quantized_sparse_moe_router_gb300", "csrc", f)) as fh:
            texts.append(fh.read())
    return source_hash(texts)


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (read + write) of `kernel` from the committed ncu
    summary profiles/<kernel>_<workload>.md, or None when there is none or it
    was taken on other source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if kernel not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    with open(path) as f:
        txt = f.read()
    m = re.search(r"^traffic_bytes_per_launch:\s*([0-9.]+)\s*$", txt, re.M)
    h = re.search(r"^source_sha256:\s*([0-9a-f]{64})\s*$", txt, re.M)
    if not m or not h or h.group(1) != kernel_source_hash(kernel):
        return None
    return float(m.group(1))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- layers
def build_layers(w, n_layers, device, T_max, act_q8=False):
    """n_layers seeded layers of workload w's shapes, quantised to Q8_0 on the GPU."""
    import torch
    import quantized_sparse_moe_router_gb300 as fw
    layers = []
    H, I, E, S = w.H, w.I, w.E, w.S
    tmp = torch.empty(I * H, dtype=torch.float32, device=device)
    gu = fw.q8_0_bytes(I, H)
    dn = fw.q8_0_bytes(H, I)
    for l in range(n_layers):
        q = {k: torch.empty((E + S, gu if k < 2 else dn), dtype=torch.uint8, device=device) for k in (0, 1, 2)}
        for e in range(E + S):
            for kind in (0, 1, 2):
                synth.fill_normal_f32_device(tmp, w.seed, synth.stream_id(l, e, kind), w.sigma_w)
                rows, K = (I, H) if kind < 2 else (H, I)
                fw.quantize_q8_0(tmp.view(rows, K), out=q[kind][e].view(rows, K // 32 * 34))
        Wr = torch.from_numpy(synth.router_weight_f32(w, l)).to(device)
        b = synth.router_bias_f32(w, l)
        weights = {"router_w": Wr, "router_bias": None if b is None else torch.from_numpy(b).to(device),
                   "w_gate": q[0][:E], "w_up": q[1][:E], "w_down": q[2][:E]}
        if S:
            weights.update(shared_gate=q[0][E], shared_up=q[1][E], shared_down=q[2][E])
        layers.append(fw.MoELayer(H, I, E, w.k, n_shared=S, T_max=T_max, weights=weights, act_q8=act_q8))
        del q, Wr, weights
    del tmp
    torch.cuda.synchronize()
    return layers


def hidden_rows(w, n_rows):
    """n_rows independent [T, H] hidden-state batches (bf16 bits)."""
    return [synth.normal_bf16_bits(w.seed, synth.stream_id(9999, r, synth.KIND_X), w.T * w.H, 1.0).reshape(w.T, w.H)
            for r in range(n_rows)]


# ------------------------------------------------------- algorithmic work
def algorithmic(w, ids_list):
    """Bytes and FLOPs the method must move/compute for the given calls' routing
    (each touched expert's Q8_0 once, router once, x once, out once)."""
    bq = 34.0 / 32.0
    per_expert_gu = 2 * w.I * w.H * bq
    per_expert_d = w.H * w.I * bq
    tot = {"bytes": 0.0, "gu_bytes": 0.0, "d_bytes": 0.0, "flops": 0.0, "U": []}
    for ids in ids_list:
        U = len(np.unique(ids)) + w.S
        T = ids.shape[0]
        tot["U"].append(U)
        tot["gu_bytes"] += U * per_expert_gu + T * w.H * 2 + T * (w.k + w.S) * w.I * 4
        tot["d_bytes"] += U * per_expert_d + T * (w.k + w.S) * w.I * 4 + T * w.H * 2
        tot["bytes"] += U * (per_expert_gu + per_expert_d) + w.E * w.H * 4 + 2 * T * w.H * 2
        tot["flops"] += T * (w.k + w.S) * 3 * 2 * w.H * w.I
    return tot


def work_bytes_layer(w):
    return (w.E + w.S) * 3 * w.I * w.H * (1 + 4 / 32)


def gemm_roofline(fl, gb, k_us, hbm, bf16, peak_src):
    """Roofline of a GEMM launch doing fl FLOPs over gb algorithmic bytes in k_us: bound by
    whichever of the two takes longer at its peak (bf16 TFLOP/s, HBM GB/s); the other beside it."""
    tf = fl / (k_us / 1e6) / 1e12
    bw = gb / (k_us / 1e6) / 1e9
    tensor_side = {"achieved": round(tf, 1), "peak": bf16, "unit": "TFLOP/s", "frac": round(tf / bf16, 4),
                   "algorithmic_flops_per_launch": round(fl), "peak_source": f"{peak_src} bf16_tflops (cuBLAS burst)"}
    hbm_side = {"achieved": round(bw, 1), "peak": hbm, "unit": "GB/s", "frac": round(bw / hbm, 4),
                "algorithmic_bytes_per_launch": round(gb), "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"}
    if fl / (bf16 * 1e12) >= gb / (hbm * 1e9):
        return {"bound": "tensor", **tensor_side, "hbm": hbm_side}
    return {"bound": "hbm", **hbm_side, "tensor": tensor_side}


# ------------------------------------------------------------ fw arm
def time_workload(w, layers, args, world, dev, e2e: bool):
    """Time one workload on its layers: graph of one step, REPEATS x K replays,
    median; a per-kernel event pass; e2e through the host-buffer entry point."""
    import torch
    import quantized_sparse_moe_router_gb300 as fw
    n_layers = len(layers)
    NX = n_x_rows(w)
    xs_host = hidden_rows(w, NX)
    xs = [torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in xs_host]
    T, k = w.T, w.k
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    out = torch.empty((T, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    calls_per_step = NX * n_layers

    def step(s_=None):
        for r in range(NX):
            for L in layers:
                fw.fw_moe_forward(L.handle, xs[r].data_ptr(), T, ids.data_ptr(), None, out.data_ptr(),
                                  s_ if s_ is not None else sp)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for L in layers:
        L.status()

    # the step as one CUDA graph through the library's own capture (fw_moe_graph_create):
    # the same calls as step(), replayed by one fw_moe_graph_launch
    order = [(xs[r], L) for r in range(NX) for L in layers]
    graph = fw.MoEGraph([L for _, L in order], [x for x, _ in order], [out] * len(order), [ids] * len(order))
    replay = lambda: graph.launch(sp)
    for _ in range(max(3, args.warmup)):
        replay()
    torch.cuda.synchronize()

    def timed(fn, n):
        barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n):
            fn()
        t1.record(stream)
        t1.synchronize()
        barrier()
        return max_over_ranks(t0.elapsed_time(t1), world, dev)

    reps = [timed(replay, args.steps) for _ in range(max(1, args.repeats))]
    ms = statistics.median(reps)
    for L in layers:
        L.status()
    value = whole_job_rate(T * calls_per_step * args.steps, ms / 1e3, world)
    ms_eager = timed(step, 1)
    graph.close()

    # ---- per-kernel event pass (events serialise the kernels: a pass of its own, one step)
    for L in layers:
        fw.fw_moe_profile_begin(L.handle, 16 * NX)
    ids_all = torch.empty((NX, n_layers, T, k), dtype=torch.int32, device=dev)
    for r in range(NX):
        for li, L in enumerate(layers):
            fw.fw_moe_forward(L.handle, xs[r].data_ptr(), T, ids_all[r, li].data_ptr(), None, out.data_ptr(), sp)
    torch.cuda.synchronize()
    prof = {}
    for L in layers:
        for kname, (kms, cnt) in fw.fw_moe_profile_end(L.handle).items():
            a = prof.setdefault(kname, [0.0, 0])
            a[0] += kms
            a[1] += cnt
    work = algorithmic(w, ids_all.cpu().numpy().reshape(-1, T, k))
    n_calls = calls_per_step
    launches_per_call = sum(c for _, c in prof.values()) / n_calls
    call_us = ms / args.steps / calls_per_step * 1e3

    def avg_us(name):
        tot, cnt = prof.get(name, (0.0, 0))
        return tot / cnt * 1e3 if cnt else 0.0

    hbm, bf16_burst, _, peak_src = load_peaks()
    if T <= 16:
        dom = "decode_experts"  # the experts' one kernel (gate/up, down, combine): one launch per call
        dom_bytes = (work["gu_bytes"] + work["d_bytes"]) / n_calls
        ev_us = avg_us(dom)
        # the event pass serialises the kernels; inside the timed graph the
        # kernel overlaps its router, so its time there is at most the call's
        k_us = min(ev_us, call_us) if ev_us else call_us
        achieved = dom_bytes / (k_us / 1e6) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4),
                    # the committed captures are of the bf16-activation kernel: none for the Q8 one
                    "traffic": None if args.act_q8 else measured_traffic(dom, w.name), "kernel": dom,
                    "avg_launch_us": round(k_us, 3), "event_pass_us": round(ev_us, 3),
                    "algorithmic_bytes_per_launch": round(dom_bytes),
                    "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"}
    else:
        # the gate/up "launch": the GEMM launches of one call (big, mid and small token tiles).
        # Its bound is the binding one of its own work: its FLOPs at the bf16 peak or its
        # bytes (the touched experts' gate/up weights once, x in, h out) at the HBM peak;
        # the other is reported beside it.
        dom = "prefill_gateup"
        k_us = avg_us(dom) + avg_us("prefill_gateup_mid") + avg_us("prefill_gateup_small")
        roofline = gemm_roofline(work["flops"] * 2 / 3 / n_calls, work["gu_bytes"] / n_calls, k_us, hbm, bf16_burst,
                                 peak_src)
        roofline.update({"traffic": measured_traffic(dom, w.name), "kernel": dom, "avg_launch_us": round(k_us, 3)})
    step_bytes = work["bytes"]
    call_roof_us = max(step_bytes / calls_per_step / (hbm * 1e9), work["flops"] / calls_per_step / (bf16_burst * 1e12)) * 1e6
    whole = {"us_per_call": round(call_us, 3), "roofline_us_per_call": round(call_roof_us, 3),
             "frac_of_roofline": round(call_roof_us / call_us, 4),
             "algorithmic_GBps": round(step_bytes / (ms / args.steps / 1e3) / 1e9, 1),
             "algorithmic_TFLOPs": round(work["flops"] / (ms / args.steps / 1e3) / 1e12, 1),
             "touched_experts_mean": round(float(np.mean(work["U"])), 2),
             "repeats_ms_per_step": [round(r / args.steps, 4) for r in reps]}
    kernels = {n: {"total_ms": round(v[0], 3), "launches": v[1], "avg_us": round(v[0] / v[1] * 1e3, 3)}
               for n, v in prof.items()}

    e2e_res = None
    if e2e:
        xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs_host]
        ids_h = torch.empty((T, k), dtype=torch.int32).pin_memory()
        out_h = torch.empty((T, w.H), dtype=torch.bfloat16).pin_memory()
        e2e_steps = max(1, min(args.steps, 3))
        for r in range(min(4, NX)):
            layers[0].forward_host(xh[r], ids_h, out_h)
        barrier()
        t_s = time.perf_counter()
        for _ in range(e2e_steps):
            for r in range(NX):
                for L in layers:
                    fw.fw_moe_forward_host(L.handle, xh[r].data_ptr(), T, ids_h.data_ptr(), out_h.data_ptr(), sp)
        el = max_over_ranks(time.perf_counter() - t_s, world, dev)
        e2e_res = {"value": round(whole_job_rate(T * calls_per_step * e2e_steps, el, world), 1), "unit": "tokens/s",
                   "h2d_bytes_per_step": calls_per_step * T * w.H * 2,
                   "d2h_bytes_per_step": calls_per_step * (T * k * 4 + T * w.H * 2),
                   "steps": e2e_steps, "api": "fw_moe_forward_host (pinned host buffers, synchronous per call)"}
    return {
        "value": round(value, 1), "unit": "tokens/s", "ms_per_step": round(ms / args.steps, 4),
        "config": {"workload": w.name, "H": w.H, "I": w.I, "E": w.E, "k": w.k, "n_shared": w.S, "T": w.T,
                   "layers": n_layers, "x_rows": NX, "calls_per_step": calls_per_step,
                   "l2": f"inputs larger than L2: {n_layers} layers x {round(work_bytes_layer(w) / 1e9, 2)} GB "
                         "of repacked experts cycled (L2 129 MB), no flush"},
        "eager_ms_per_step": round(ms_eager, 4),
        "roofline": roofline, "whole_step": whole, "kernels": kernels, "e2e": e2e_res,
        "gpu_launches": int(round(launches_per_call * args.steps * calls_per_step)),
    }


def metric_name(w):
    return (f"MoE-FFN tokens/s ({w.name}: H={w.H} I={w.I} E={w.E} top-{w.k}"
            f"{' +1 shared' if w.S else ''} T={w.T}); decode HBM GB/s / prefill TFLOP/s as fraction of peak")


def workload_of(args, name):
    w = synth.WORKLOADS[name]
    if args.experts:
        w = w.with_(E=args.experts)
    if args.tokens:
        w = w.with_(T=args.tokens)
    return w


def run_fw(args, rank, world, local_rank):
    import torch
    import quantized_sparse_moe_router_gb300 as fw
    fw.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    head = args.workload or HEADLINE
    names = [head] if args.workload else [n for n in ALL_WORKLOADS if n != head] + [head]
    results = {}
    built = {}  # layer-set owner -> layers
    clocks = ClockSampler(local_rank)
    clk = None
    for name in names:
        w = workload_of(args, name)
        owner = SHARED_LAYERS.get(name, name) if not args.workload else name
        users = [n for n in names if SHARED_LAYERS.get(n, n) == owner] if not args.workload else [name]
        if owner not in built:
            wo = workload_of(args, owner)
            n_layers = args.layers or max(synth.WORKLOADS[u].layers for u in users)
            T_max = max(workload_of(args, u).T for u in users)
            built[owner] = build_layers(wo, n_layers, dev, T_max, act_q8=args.act_q8)
        layers = built[owner][:(args.layers or w.layers)]
        if name == head:
            clocks.start()
            time.sleep(0.3)
        results[name] = time_workload(w, layers, args, world, dev, e2e=(name == head and not args.no_e2e))
        if name == head:
            clk = clocks.stop()
        if all(n in results for n in users):  # last user of this layer set: free it
            for L in built.pop(owner):
                L.close()
            torch.cuda.empty_cache()
    w = workload_of(args, head)
    res = results.pop(head)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)
        # the 4096-token prefill's baseline on its first 256 tokens (one call, about 25 s)
        pre = "pre4096" if "pre4096" in results else None
        if pre:
            results[pre]["cpu_baseline"] = cpu_baseline_tokens(workload_of(args, pre), 256)
    line = {
        "metric": metric_name(w), "value": res["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("int32 dot products (Q8_0 weights x Q8 activations), fp32 scales and sums" if args.act_q8
                  else "fp32 (Q8_0 weights x bf16 activations, fp32 accumulate)") if w.T <= 16
        else "bf16 tensor-core (Q8_0 dequantised to bf16), fp32 accumulate",
        "data": "synthetic (seeded Irwin-Hall normals; experts quantised to Q8_0 on the GPU)",
        "config": dict(res["config"], parallelism=f"replicas x{world}", activations="q8" if args.act_q8 else "bf16"),
        "timing": f"CUDA events on the launch stream around K replays of one step's CUDA graph "
                  f"(fw_moe_graph_create / fw_moe_graph_launch); median of {args.repeats} repeats",
        "roofline": res["roofline"], "whole_step": res["whole_step"], "kernels": res["kernels"],
        "e2e": res["e2e"], "cpu_baseline": cpu, "gpu_launches": res["gpu_launches"], "clocks": clk,
        "eager_ms_per_step": res["eager_ms_per_step"],
    }
    if results:
        line["per_config"] = {n: {"metric": metric_name(workload_of(args, n)), **r} for n, r in results.items()}
        line["gpu_launches_all_configs"] = line["gpu_launches"] + sum(r["gpu_launches"] for r in results.values())
    return line


# ------------------------------------------------------------ oracle arm
def _prep_expert(args):
    """(workload, layer, expert) -> its three Q8_0 matrices by the oracle's quantiser (worker process)."""
    import oracle
    w, l, e = args
    return e, [oracle.q8_0_quantize(synth.expert_weight_f32(w, l, e, kind)) for kind in (0, 1, 2)]


def oracle_prepare(w, n_tokens, n_layers=2):
    """Hidden rows and the Q8_0 experts their routing needs, for the first
    n_layers layers of w: quantised by the oracle over a spawn pool (untimed)."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    xs = hidden_rows(w, 1)[0][:n_tokens]
    jobs, routed = [], []
    for l in range(min(w.layers, n_layers)):
        Wr = synth.router_weight_f32(w, l)
        b = synth.router_bias_f32(w, l)
        ids, _ = oracle.topk_gates(oracle.router_logits(xs, Wr, b), w.k)
        need = sorted(set(np.unique(ids).tolist()) | set(range(w.E, w.E + w.S)))
        routed.append((Wr, b, need))
        jobs += [(w, l, e) for e in need]
    procs = max(1, min(os.cpu_count() or 1, 32))
    with mp.get_context("spawn").Pool(procs) as pool:
        done = pool.map(_prep_expert, jobs)
    prepared, i = [], 0
    for Wr, b, need in routed:
        lists = [[None] * (w.E + w.S) for _ in range(3)]
        for e in need:
            _, q = done[i]
            i += 1
            for kind in range(3):
                lists[kind][e] = q[kind]
        prepared.append((Wr, b, lists))
    return xs, prepared


def oracle_tokens(w, seconds):
    """Tokens of the bounded oracle sample: about `seconds` of single-thread work."""
    per_token = 3 * 2 * w.H * w.I * (w.k + w.S) / 0.8e9 + 2 * w.E * w.H / 1e9  # ~0.8 GMAC/s fp64 with dequant
    return int(max(1, min(w.T, 256, seconds / per_token)))


def oracle_sample(w, seconds, xs, prepared, max_calls=64):
    """Time the oracle, as it stands, single-threaded, on calls of the workload
    (the prepared layers cycled; each call all prepared tokens)."""
    import oracle
    done_tokens, el, calls = 0, 0.0, 0
    while calls < max_calls and (calls == 0 or el < seconds):
        Wr, b, (g, u, d) = prepared[calls % len(prepared)]
        t = time.perf_counter()
        oracle.moe_forward(xs, Wr, b, g, u, d, k=w.k, S=w.S)
        el += time.perf_counter() - t
        done_tokens += xs.shape[0]
        calls += 1
    return done_tokens, el, calls


def cpu_baseline(w, seconds):
    n_tok = oracle_tokens(w, seconds / 2)
    xs, prepared = oracle_prepare(w, n_tok)
    tokens, el, calls = oracle_sample(w, seconds, xs, prepared)
    return {"value": round(tokens / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{calls} route+FFN calls of the first {n_tok} token(s) of the workload's hidden batch, "
                      f"cycling {len(prepared)} of its layers ({el:.1f} s of single-thread fp64 work; expert "
                      f"quantisation untimed)",
            "host_cores": os.cpu_count()}


def cpu_baseline_tokens(w, n_tok):
    """The oracle on one call of the workload's first n_tok tokens (one layer)."""
    n_tok = min(n_tok, w.T)
    xs, prepared = oracle_prepare(w, n_tok, n_layers=1)
    tokens, el, calls = oracle_sample(w, 0.0, xs, prepared, max_calls=1)
    return {"value": round(tokens / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"one route+FFN call of the first {n_tok} tokens of the workload's hidden batch "
                      f"({el:.1f} s of single-thread fp64 work; expert quantisation untimed)",
            "host_cores": os.cpu_count()}


def run_reference(args):
    w = workload_of(args, args.workload or HEADLINE)
    total = args.steps + args.warmup
    per_step = max(0.2, args.cpu_seconds / max(1, total))
    n_tok = oracle_tokens(w, per_step)
    xs, prepared = oracle_prepare(w, n_tok)
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, xs, prepared, max_calls=1)
    tot_tokens, tot_el, tot_calls = 0, 0.0, 0
    for _ in range(args.steps):
        tokens, el, calls = oracle_sample(w, 0.0, xs, prepared, max_calls=1)
        tot_tokens += tokens
        tot_el += el
        tot_calls += calls
    value = tot_tokens / tot_el
    return {
        "impl": "reference", "metric": metric_name(w),
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp64", "data": "synthetic",
        "config": {"workload": w.name, "H": w.H, "I": w.I, "E": w.E, "k": w.k, "n_shared": w.S, "T": w.T},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle", "cores": 1,
                         "sample": f"{tot_calls} calls (one per step) of the first {n_tok} token(s) of the "
                                   f"workload, cycling {len(prepared)} layers (single-thread fp64 oracle; expert "
                                   "quantisation untimed)"},
        "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.gpus > 1 and world == 1:
        print(json.dumps({"metric": metric_name(workload_of(args, args.workload or HEADLINE)),
                          "n_gpus": args.gpus, "unavailable":
                          "replicas only: launch one process per GPU with torch.distributed.run"}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_fw(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
