#!/usr/bin/env python
"""Throughput of the routed Q8_0 MoE feed-forward step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dec1] [--impl fw|reference]

Default workload: decode batch-1 (H=2048, I=768, E=128, top-8, T=1) over 48
independently generated layers cycled so the working set (32.6 GB of repacked
Q8_0 experts) is far larger than L2. One step = every one of 64 synthetic
hidden rows through all 48 layers in turn (3072 route+ffn calls; 64/T batches
for T > 1), all on one stream. value = tokens x layer-calls per second, i.e. the token throughput of
one MoE layer, summed over ranks. The path does not shard: N GPUs run N
independent replicas (weak scaling) and the only collective is the timing's
max over ranks.

--impl reference times the fp64 oracle on the host cores instead, on a
bounded sample of the same workload (rank 0 only).
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

def n_x_rows(w):
    """Distinct hidden batches cycled per step: 64 rows at T=1, fewer for larger T."""
    return max(1, 64 // w.T)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="dec1", choices=sorted(synth.WORKLOADS))
    p.add_argument("--impl", default="fw", choices=["fw", "reference"])
    p.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    p.add_argument("--experts", type=int, default=0,
                   help="override E (a smaller case for profiling: at T = 1 the expert work per call is the same)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0,
                   help="host time budget of the oracle baseline (and of the whole reference arm)")
    return p.parse_args()


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
def build_layers(w, n_layers, device):
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
        layers.append(fw.MoELayer(H, I, E, w.k, n_shared=S, T_max=w.T, weights=weights))
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


# ------------------------------------------------------------ fw arm
def run_fw(args, rank, world, local_rank):
    import torch
    import quantized_sparse_moe_router_gb300 as fw
    fw.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synth.WORKLOADS[args.workload]
    if args.experts:
        w = w.with_(E=args.experts)
    n_layers = args.layers or w.layers
    layers = build_layers(w, n_layers, dev)
    N_X_ROWS = n_x_rows(w)
    xs_host = hidden_rows(w, N_X_ROWS)
    xs = [torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in xs_host]
    T, k = w.T, w.k
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    out = torch.empty((T, w.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    calls_per_step = N_X_ROWS * n_layers

    def step():
        for r in range(N_X_ROWS):
            x = xs[r]
            for L in layers:
                fw.fw_moe_forward(L.handle, x.data_ptr(), T, ids.data_ptr(), None, out.data_ptr(), sp)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for L in layers:
        L.status()

    # ---- the step captured once as a CUDA graph (the serving mode: decode replays graphs)
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(stream)
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            csp = torch.cuda.current_stream().cuda_stream
            for r in range(N_X_ROWS):
                for L in layers:
                    fw.fw_moe_forward(L.handle, xs[r].data_ptr(), T, ids.data_ptr(), None, out.data_ptr(), csp)
    stream.wait_stream(cap_stream)
    for _ in range(max(1, args.warmup)):
        graph.replay()
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

    # ---- timed region (graph replays)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ms = timed(graph.replay, args.steps)
    clk = clocks.stop()
    for L in layers:
        L.status()
    ms_eager = timed(step, max(1, min(args.steps, 5)))
    eager_steps = max(1, min(args.steps, 5))
    value = whole_job_rate(T * calls_per_step * args.steps, ms / 1e3, world)
    value_eager = whole_job_rate(T * calls_per_step * eager_steps, ms_eager / 1e3, world)

    # ---- per-kernel timing pass (events around every kernel; same K steps)
    ids_log = []
    for L in layers:
        # room for every launch: 2 kernels per decode call, at most 12 per prefill call
        fw.fw_moe_profile_begin(L.handle, (2 if T <= 16 else 12) * N_X_ROWS * max(args.steps, 1))
    ids_all = torch.empty((args.steps, N_X_ROWS, n_layers, T, k), dtype=torch.int32, device=dev)
    for s_ in range(args.steps):
        for r in range(N_X_ROWS):
            for li, L in enumerate(layers):
                fw.fw_moe_forward(L.handle, xs[r].data_ptr(), T, ids_all[s_, r, li].data_ptr(), None,
                                  out.data_ptr(), sp)
    torch.cuda.synchronize()
    prof = {}
    for L in layers:
        for kname, (kms, cnt) in fw.fw_moe_profile_end(L.handle).items():
            a = prof.setdefault(kname, [0.0, 0])
            a[0] += kms
            a[1] += cnt
    ids_np = ids_all.cpu().numpy().reshape(-1, T, k)
    work = algorithmic(w, ids_np)
    n_calls = args.steps * calls_per_step
    launches_per_call = sum(c for _, c in prof.values()) / n_calls

    def avg_launch_ms(name):  # mean duration of one launch of this kind
        tot, cnt = prof.get(name, (0.0, 0))
        return tot / cnt if cnt else 0.0

    hbm, bf16_burst, bf16_sus, peak_src = load_peaks()
    decode = T <= 16
    if decode:
        dom = "decode_experts"  # gate/up + down + combine in one kernel (one launch per call)
        dom_bytes = (work["gu_bytes"] + work["d_bytes"]) / n_calls
        t_ms = avg_launch_ms(dom)
        achieved = dom_bytes / (t_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4), "traffic": measured_traffic(dom, w.name), "kernel": dom,
                    "avg_launch_us": round(t_ms * 1e3, 3),
                    "algorithmic_bytes_per_launch": round(dom_bytes),
                    "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"}
    else:
        # the gate/up "launch": the pair of GEMM launches of one call (192-row tiles, then the small tiles)
        dom = "prefill_gateup"
        t_ms = avg_launch_ms(dom) + avg_launch_ms("prefill_gateup_small")
        fl = work["flops"] * 2 / 3 / n_calls
        achieved = fl / (t_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16_burst, "unit": "TFLOP/s",
                    "frac": round(achieved / bf16_burst, 4), "traffic": measured_traffic(dom, w.name), "kernel": dom,
                    "avg_launch_us": round(t_ms * 1e3, 3), "algorithmic_flops_per_launch": round(fl),
                    "peak_source": f"{peak_src} bf16_tflops (cuBLAS burst)"}
    step_bytes = work["bytes"] / args.steps
    whole = {"algorithmic_GBps": round(step_bytes / (ms / args.steps / 1e3) / 1e9, 1),
             "frac_of_hbm": round(step_bytes / (ms / args.steps / 1e3) / 1e9 / hbm, 4),
             "us_per_call": round(ms / args.steps / calls_per_step * 1e3, 3),
             "roofline_us_per_call": round(step_bytes / calls_per_step / (hbm * 1e9) * 1e6, 3),
             "touched_experts_mean": round(float(np.mean(work["U"])), 2)}
    kernels = {n: {"total_ms": round(v[0], 3), "launches": v[1], "avg_us": round(v[0] / v[1] * 1e3, 3)}
               for n, v in prof.items()}

    # ---- end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e:
        xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs_host]
        ids_h = torch.empty((T, k), dtype=torch.int32).pin_memory()
        out_h = torch.empty((T, w.H), dtype=torch.bfloat16).pin_memory()
        e2e_steps = max(1, min(args.steps, 3))
        for r in range(min(4, N_X_ROWS)):
            layers[0].forward_host(xh[r], ids_h, out_h)
        barrier()
        t_s = time.perf_counter()
        for _ in range(e2e_steps):
            for r in range(N_X_ROWS):
                for L in layers:
                    fw.fw_moe_forward_host(L.handle, xh[r].data_ptr(), T, ids_h.data_ptr(), out_h.data_ptr(), sp)
        el = max_over_ranks(time.perf_counter() - t_s, world, dev)
        e2e = {"value": round(whole_job_rate(T * calls_per_step * e2e_steps, el, world), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": calls_per_step * T * w.H * 2,
               "d2h_bytes_per_step": calls_per_step * (T * k * 4 + T * w.H * 2),
               "steps": e2e_steps, "api": "fw_moe_forward_host (pinned host buffers, synchronous per call)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)

    for L in layers:
        L.close()
    return {
        "metric": f"MoE-FFN tokens/s ({w.name}: H={w.H} I={w.I} E={w.E} top-{w.k}"
                  f"{' +1 shared' if w.S else ''} T={w.T}); decode HBM GB/s / prefill TFLOP/s as fraction of peak",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 (Q8_0 weights x bf16 activations, fp32 accumulate)" if decode
        else "bf16 tensor-core (Q8_0 dequantised to bf16), fp32 accumulate",
        "data": "synthetic (seeded Irwin-Hall normals; experts quantised to Q8_0 on the GPU)",
        "config": {"workload": w.name, "H": w.H, "I": w.I, "E": w.E, "k": w.k, "n_shared": w.S, "T": w.T,
                   "layers": n_layers, "x_rows": n_x_rows(w), "calls_per_step": calls_per_step,
                   "l2": f"inputs larger than L2: {n_layers} layers x {round(work_bytes_layer(w) / 1e9, 2)} GB "
                         "of repacked experts cycled (L2 129 MB), no flush",
                   "parallelism": f"replicas x{world}"},
        "eager": {"value": round(value_eager, 1), "ms_per_step": round(ms_eager / eager_steps, 4),
                  "note": "same step launched call by call from Python (no graph)"},
        "timing": "CUDA events on the launch stream around K replays of a CUDA graph of one step",
        "roofline": roofline, "whole_step": whole, "kernels": kernels, "e2e": e2e, "cpu_baseline": cpu,
        "gpu_launches": int(round(launches_per_call * args.steps * calls_per_step)),
        "clocks": clk,
    }


def work_bytes_layer(w):
    return (w.E + w.S) * 3 * w.I * w.H * (1 + 4 / 32)


# ------------------------------------------------------------ oracle arm
def oracle_sample(w, seconds, max_calls=64):
    """Time the oracle, as it stands, on calls of the workload (layers cycled,
    the same hidden rows); the experts a call needs are quantised by the oracle
    beforehand, untimed."""
    import oracle
    oracle.build()
    xs = hidden_rows(w, 4)
    n_layers = min(w.layers, 4)
    prepared = []
    for l in range(n_layers):
        Wr = synth.router_weight_f32(w, l)
        b = synth.router_bias_f32(w, l)
        T_s = min(w.T, 8)
        x = xs[l % 4][:T_s]
        ids, _ = oracle.topk_gates(oracle.router_logits(x, Wr, b), w.k)
        need = set(np.unique(ids).tolist()) | set(range(w.E, w.E + w.S))
        lists = [[oracle.q8_0_quantize(synth.expert_weight_f32(w, l, e, kind)) if e in need else None
                  for e in range(w.E + w.S)] for kind in (0, 1, 2)]
        prepared.append((x, Wr, b, lists))
    done_tokens, el, calls = 0, 0.0, 0
    while el < seconds and calls < max_calls:
        x, Wr, b, (g, u, d) = prepared[calls % n_layers]
        t = time.perf_counter()
        oracle.moe_forward(x, Wr, b, g, u, d, k=w.k, S=w.S)
        el += time.perf_counter() - t
        done_tokens += x.shape[0]
        calls += 1
    return done_tokens, el, calls, min(w.T, 8)


def cpu_baseline(w, seconds):
    tokens, el, calls, T_s = oracle_sample(w, seconds)
    return {"value": round(tokens / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{calls} route+FFN calls of {T_s} token(s) each over {min(w.layers, 4)} layers of the "
                      f"workload ({el:.1f} s of single-thread fp64 work; expert quantisation untimed)",
            "host_cores": os.cpu_count()}


def run_reference(args):
    w = synth.WORKLOADS[args.workload]
    per_step = max(0.2, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, per_step / 4, max_calls=1)
    tot_tokens, tot_el, tot_calls = 0, 0.0, 0
    for _ in range(args.steps):
        tokens, el, calls, T_s = oracle_sample(w, per_step, max_calls=4)
        tot_tokens += tokens
        tot_el += el
        tot_calls += calls
    value = tot_tokens / tot_el
    return {
        "impl": "reference",
        "metric": f"MoE-FFN tokens/s ({w.name}: H={w.H} I={w.I} E={w.E} top-{w.k}"
                  f"{' +1 shared' if w.S else ''} T={w.T}); decode HBM GB/s / prefill TFLOP/s as fraction of peak",
        "value": round(value, 3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp64", "data": "synthetic",
        "config": {"workload": w.name, "H": w.H, "I": w.I, "E": w.E, "k": w.k, "n_shared": w.S, "T": w.T},
        "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "kind": "oracle", "cores": 1,
                         "sample": f"{tot_calls} calls of up to 8 tokens over <=4 layers (single-thread fp64 oracle)"},
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
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_fw(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
