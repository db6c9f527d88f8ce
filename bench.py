#!/usr/bin/env python
"""Benchmark of the causal packed MXFP8 attention training call on GB300.

One step = one pass of the whole hot path over one microbatch: the GPU work
list (plan), token-block quantization of Q, K and V, the forward, and the
backward (dO encoding with D, dQ boosts, backward attention, dQ finalise).
FLOPs per step follow the pages' convention: 14 * head_dim * hq * visible
pairs (2 FLOPs per multiply-add, causal pairs only; forward 4d, backward 10d).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs its
own replica of the workload (the attention call has no exchange step) and the
timed region is bracketed by barriers; value = work of all ranks / max time.
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

import flamia_workloads as W  # noqa: E402

METRIC = "causal packed MXFP8 attn fwd+bwd TFLOPS and % of GB300 dense FP8 peak"
DEFAULT_WORKLOAD = "packed_16k_h16_d128"
# kernels launched per step: plan, 3 quantize, fwd, fwd tail, dO prep, dQ boost, bwd, dQ finalise;
# strict: the ordered dQ kernel and the zeroing of rows outside every document replace the
# finalise; mixed: 3 more quantize launches (NVFP4 Q and K, per-token V)
LAUNCHES_PER_STEP = {"default": 10, "strict": 11, "mixed": 13}
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--mode", default="default", choices=["default", "strict", "mixed"],
                    help="strict options or the mixed NVFP4/FP8 route (head_dim 128)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of CUDA-graph replays")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        return dict(bf16=m["bf16_tflops"], bf16_sust=m["bf16_tflops_sustained"], hbm=m["hbm_gbs"], src="measured")
    return dict(bf16=1900.0, bf16_sust=1700.0, hbm=6800.0, src="fallback")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.lines

    @staticmethod
    def summarize(lines, t0, t1):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [l for (t, l) in lines if t0 - 0.15 <= t <= t1 + 0.15] or [l for (_, l) in lines]
        for l in window:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- oracle sample

def oracle_opts(mode):
    import oracle as O
    return O.Options(strict=mode == "strict", mixed=mode == "mixed")


def oracle_sample(w, budget_s, max_tokens=None, mode="default"):
    """Time the oracle (as it stands) on a bounded sample of the workload: the
    first S tokens of the longest document for G kv-head groups, S doubled from
    256 (up to the document length), then G doubled (up to hkv), until about
    budget_s seconds of CPU work.  Returns the last sample's throughput."""
    import oracle as O
    L = min(max(w.lengths), max_tokens or max(w.lengths))
    g = w.hq // w.hkv
    inp = W.make_inputs(W.custom([L], w.hq, w.hkv, w.d, dist=w.dist, seed=w.seed))
    vals = {n: W.bf16_bits_to_f32(b).astype(np.float64) for n, b in inp.items()}
    S, G, best, spent = 256, 1, None, 0.0
    while True:
        S = min(S, L)
        sub = {n: v[:S, :(G * g if n in ("q", "do") else G)] for n, v in vals.items()}
        t0 = time.perf_counter()
        O.run_training_call(sub["q"], sub["k"], sub["v"], sub["do"], [0, S], G * g, G, opts=oracle_opts(mode))
        dt = time.perf_counter() - t0
        spent += dt
        flops = 14.0 * w.d * G * g * S * (S + 1) / 2
        best = dict(tokens=S, heads=G * g, seconds=dt, flops=flops, tflops=flops / dt / 1e12)
        if spent + 2.5 * dt > budget_s:
            break
        if S < L:
            S *= 2
        elif G < w.hkv:
            G = min(2 * G, w.hkv)
        else:
            break
    return best


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v):
            return int(os.environ[v])
    return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = W.WORKLOADS[args.workload]
    probe = oracle_sample(w, budget_s=6.0, mode=args.mode)
    S, Hs = probe["tokens"], probe["heads"]
    import oracle as O
    g = w.hq // w.hkv
    inp = W.make_inputs(W.custom([S], Hs, Hs // g, w.d, dist=w.dist, seed=w.seed))
    vals = {n: W.bf16_bits_to_f32(b).astype(np.float64) for n, b in inp.items()}
    step = lambda: O.run_training_call(vals["q"], vals["k"], vals["v"], vals["do"], [0, S], Hs, Hs // g,
                                       opts=oracle_opts(args.mode))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = 14.0 * w.d * Hs * S * (S + 1) / 2
    value = flops / dt / 1e12
    sample = f"oracle fwd+bwd (fp64 numpy) on the first {S} tokens of the longest document, {Hs} query heads"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "mode": args.mode, "sample_tokens": S, "sample_heads": Hs, "head_dim": w.d},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": blas_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- our arm

def kernel_source_sha(name):
    with open(os.path.join(ROOT, "microscaled_precision_causal_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_for(kernel_file, workload):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel_file)
    if not rec or rec.get("source_sha256") != kernel_source_sha(kernel_file):
        return None
    per_unit = rec["dram_bytes_per_launch"] / rec["flops_per_launch"]
    return {"bytes_per_flop": per_unit, "workload": rec.get("workload")}


def quantizer_roofline(w, mode, ms, hbm_gbs):
    """Algorithmic bytes of the Q/K/V quantization (token-block codes, scale bytes,
    the K/V row stats; mixed: also the NVFP4 copies of Q and K and the per-token V
    copy) over its measured time (the three or six launches of one step)."""
    T, hq, hkv, d = w.total_tokens, w.hq, w.hkv, w.d
    per = lambda H: T * H * d * (2 + 1) + T * H          # bf16 in, E4M3 out, one scale byte per row
    total = per(hq) + 2 * per(hkv) + 2 * T * hkv * 8     # + (||x^||, max |x^|) of K and V
    if mode == "mixed":
        nv = lambda H: T * H * d * (2 + 0.5) + T * H * d / 16
        total += nv(hq) + nv(hkv) + per(hkv)
    gbs = total / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
            "bytes_per_step": total, "ms": ms, "traffic": None}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from microscaled_precision_causal_gb300 import build as _b
    _b.build()
    import microscaled_precision_causal_gb300 as F

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.WORKLOADS[args.workload]
    T, N, hq, hkv, d = w.total_tokens, len(w.lengths), w.hq, w.hkv, w.d
    pairs = W.visible_pair_count(w.lengths)
    flops_step = 14.0 * d * hq * pairs
    flops_fwd, flops_bwd = 4.0 * d * hq * pairs, 10.0 * d * hq * pairs

    inp = W.make_inputs(w)
    host = {n: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory() for n, b in inp.items()}
    x = {n: t.to(dev) for n, t in host.items()}
    cu_host = torch.tensor(w.cu_seqlens, dtype=torch.int32).pin_memory()
    cu = cu_host.to(dev)
    att = F.FlamiaAttention(T, N, hq, hkv, d, device=dev, strict=args.mode == "strict",
                            mixed=args.mode == "mixed")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    import ctypes

    def make_opts(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)          # creates the underlying cudaEvent_t
        arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
        o = F.Options()
        ctypes.pointer(o)[0] = att.opts          # the mode's flags and operands
        o.timing_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        return evs, arr, o

    o_plain = F.Options()
    ctypes.pointer(o_plain)[0] = att.opts

    def step(o_fwd=None, o_bwd=None, qev=None):
        att.plan_build(cu)
        if qev:
            qev[0].record(stream)
        att.quantize(x["q"], x["k"], x["v"], cu)
        if qev:
            qev[1].record(stream)
        att.opts = o_fwd or o_plain
        att.forward(cu)
        att.opts = o_bwd or o_plain
        att.backward(x["do"], cu)
        att.opts = o_plain

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert att.device_status() == 0, "device status error during warm-up"

    gpu_index = local_rank
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local_rank])
        except ValueError:
            pass
    sampler = ClockSampler(gpu_index)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.3)

    # Per-kernel phases: eager steps with the timing_events hook (a bounded sample).
    n_ph = min(args.steps, 50)
    per_step = [(make_opts(2), make_opts(8)) for _ in range(n_ph)]
    qevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_ph)]
    for i in range(n_ph):
        flush.zero_()
        step(per_step[i][0][2], per_step[i][1][2], qevs[i])
    torch.cuda.synchronize()
    # The whole step (plan, quantize, forward, backward) as one CUDA graph: the same
    # launches, replayed without host launch gaps ([EN] Appendix D times CUDA graphs).
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        for _ in range(max(args.warmup, 3)):
            graph.replay()
        torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()                      # L2 flush between timed steps (outside the events)
        starts[i].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall1 = time.time()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kf = [f[0][0].elapsed_time(f[0][1]) for f, _ in per_step]
    kb = [b[0][4].elapsed_time(b[0][5]) for _, b in per_step]
    kbp = [b[0][0].elapsed_time(b[0][1]) for _, b in per_step]
    kfin = [b[0][6].elapsed_time(b[0][7]) for _, b in per_step]
    kq = [q0.elapsed_time(q1) for q0, q1 in qevs]
    total_ms = float(sum(ms))
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    assert att.device_status() == 0, "device status error during the timed steps"

    # end to end: pinned host inputs -> device, the training call, results -> pinned host
    out_host = {n: torch.empty_like(t, device="cpu").pin_memory() for n, t in
                (("o", att.out), ("dq", att.dq), ("dk", att.dk), ("dv", att.dv))}
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + cu_host.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The copies run on a second stream so that they overlap the compute they do not
    # feed: dO comes in while the forward runs and O goes out while the backward runs
    # (Q, K, V and cu_seqlens before the forward, dQ, dK, dV after the backward).  More
    # copy streams were measured slower: the host link is the limit, not the engines.
    copy_stream = torch.cuda.Stream(dev)
    ev_qkv, ev_do, ev_fwd, ev_bwd, ev_out = (torch.cuda.Event() for _ in range(5))
    e2e_ms = []
    for i in range(args.e2e_steps + 1):
        flush.zero_()
        e0.record(stream)
        copy_stream.wait_event(e0)
        with torch.cuda.stream(copy_stream):
            cu.copy_(cu_host, non_blocking=True)
            for n in ("q", "k", "v"):
                x[n].copy_(host[n], non_blocking=True)
            ev_qkv.record(copy_stream)
            x["do"].copy_(host["do"], non_blocking=True)
            ev_do.record(copy_stream)
        stream.wait_event(ev_qkv)
        att.plan_build(cu)
        att.quantize(x["q"], x["k"], x["v"], cu)
        att.forward(cu)
        ev_fwd.record(stream)
        stream.wait_event(ev_do)
        att.backward(x["do"], cu)
        ev_bwd.record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_fwd)
            out_host["o"].copy_(att.out, non_blocking=True)
            copy_stream.wait_event(ev_bwd)
            for n, t in (("dq", att.dq), ("dk", att.dk), ("dv", att.dv)):
                out_host[n].copy_(t, non_blocking=True)
            ev_out.record(copy_stream)
        stream.wait_event(ev_out)
        e1.record(stream)
        e1.synchronize()
        if i > 0:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_mean = float(np.mean(e2e_ms))
    if world > 1:
        t = torch.tensor([e2e_mean], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_mean = float(t.item())

    lines = sampler.stop() if not args.no_clocks else None
    clocks = ClockSampler.summarize(lines, t_wall0, t_wall1) if lines else None
    if rank != 0:
        return None

    pk = peaks()
    fp8_peak = 2.0 * pk["bf16"]          # FP8 dense = 2 x BF16 dense (4.5 / 2.25 nominal ratio)
    kf_ms, kb_ms = float(np.mean(kf)), float(np.mean(kb))
    if kb_ms >= kf_ms:
        dom, dom_ms, dom_flops, dom_src = "attn_bwd_kernel", kb_ms, flops_bwd, "attn_bwd.cu"
    else:
        dom, dom_ms, dom_flops, dom_src = "attn_fwd_kernel", kf_ms, flops_fwd, "attn_fwd.cu"
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    tr = traffic_for(dom_src, w.name)
    traffic = tr["bytes_per_flop"] * dom_flops if tr else None
    value = world * flops_step / (total_ms / args.steps * 1e-3) / 1e12
    res = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": w.name, "mode": args.mode, "cuda_graph": graph is not None, "total_tokens": T, "num_docs": N, "hq": hq, "hkv": hkv, "head_dim": d,
                   "visible_pairs": pairs, "flops_per_step": flops_step,
                   "l2": "flushed between timed steps (256 MiB write); step inputs 256 MiB > L2",
                   "frac_of_fp8_peak": value / world / fp8_peak,
                   "fp8_peak_tflops": fp8_peak, "peak_source": pk["src"] + " (2 x bf16 burst)"},
        "phases_ms": {"quantize_qkv": float(np.mean(kq)), "fwd_kernel": kf_ms, "bwd_kernel": kb_ms,
                      "bwd_prep": float(np.mean(kbp)), "bwd_finalise": float(np.mean(kfin))},
        "quantizer_roofline": quantizer_roofline(w, args.mode, float(np.mean(kq)), pk["hbm"]),
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak, "traffic": traffic,
                     "per_unit": "FLOPs per launch = %s * head_dim * hq * visible pairs" % ("10" if "bwd" in dom else "4")},
        "e2e": {"value": world * flops_step / (e2e_mean * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_mean,
                "copies": "pinned host buffers; a second stream brings dO in during the forward and takes O out "
                          "during the backward"},
        "gpu_launches": LAUNCHES_PER_STEP[args.mode] * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        s = oracle_sample(w, args.cpu_seconds, mode=args.mode)
        res["cpu_baseline"] = {
            "value": s["tflops"], "unit": "TFLOPS", "cores": blas_threads(), "kind": "oracle",
            "sample": (f"oracle fwd+bwd (fp64 numpy) on the first {s['tokens']} tokens of the longest document, "
                       f"{s['heads']} query heads: {s['seconds']:.1f} s")}
    return res


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        res = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
