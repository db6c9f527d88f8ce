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
# kernels launched per step: plan, Q/K/V quantize (one launch), fwd, fwd tail, dO prep, dQ boost,
# bwd, dQ finalise; strict: the ordered dQ kernel and the zeroing of rows outside every document
# replace the finalise; mixed: 3 more quantize launches (NVFP4 Q and K, per-token V)
LAUNCHES_PER_STEP = {"default": 8, "strict": 9, "mixed": 11}
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
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--rounds", type=int, default=4, help="the timed steps are split into this many rounds")
    ap.add_argument("--no-secondary", action="store_true", help="skip the other workloads")
    ap.add_argument("--secondary-steps", type=int, default=30)
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

def oracle_opts(mode, window=(-1, 0)):
    import oracle as O
    return O.Options(strict=mode == "strict", mixed=mode == "mixed", window=tuple(window))


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
        O.run_training_call(sub["q"], sub["k"], sub["v"], sub["do"], [0, S], G * g, G,
                            opts=oracle_opts(mode, w.window))
        dt = time.perf_counter() - t0
        spent += dt
        flops = 14.0 * w.d * G * g * W.visible_pair_count([S], w.window)
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
                                       opts=oracle_opts(args.mode, w.window))
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = 14.0 * w.d * Hs * W.visible_pair_count([S], w.window)
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

# The other workloads of the pages' shapes, timed in the same run after the headline
# (parity cases in the tests; here for their throughput): (workload, route).
SECONDARY = (
    ("causal_b1_h2_s256_d64", "default"),
    ("skewed_8192_224x256_h16_d128", "default"),
    ("packed_16x4096_h16_d128", "default"),
    ("gqa_b4_s8192_hq32_hkv8_d128", "default"),
    ("mixed_nvfp4_gqa_b4_s8192", "mixed"),
    ("strict_packed_4x8192_h16_t3", "strict"),
    ("strict_packed_4x8192_h16_t3", "default"),
    ("noncausal_packed_16k_h16_d128", "default"),
    ("noncausal_b2_s8192_h16_d128", "default"),
)
# whole training calls (forward and backward with quantization) that the pages time on B300
# for the same shapes (FLAMIA technical review section 8, Table 1): context for those lines
PAGES_CALL_MS = {
    "skewed_8192_224x256_h16_d128": (1.67, "B300, MXFP8, FLAMIA technical review section 8, Table 1"),
    "packed_16x4096_h16_d128": (3.17, "B300, MXFP8, FLAMIA technical review section 8, Table 1"),
}
EX2_PER_CLK_PER_SM = 32      # MUFU ex2 issue rate of B300-class SMs ([EN] section 7; probe in the design notes)


def kernel_source_sha(name):
    with open(os.path.join(ROOT, "microscaled_precision_causal_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def traffic_record(kernel_file, workload):
    """DRAM bytes per launch of a kernel from profiles/traffic.json (one ncu capture),
    valid only while the kernel's source is unchanged and for the same workload."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel_file)
    if not rec or rec.get("source_sha256") != kernel_source_sha(kernel_file) or rec.get("workload") != workload:
        return None
    return rec


def quantizer_bytes(w, mode):
    """Algorithmic bytes of the Q/K/V quantization of one step: bf16 in, E4M3 codes and one
    scale byte per row out, plus the K/V row stats; mixed: also the NVFP4 copies of Q and K
    and the per-token V copy."""
    T, hq, hkv, d = w.total_tokens, w.hq, w.hkv, w.d
    per = lambda H: T * H * d * (2 + 1) + T * H
    total = per(hq) + 2 * per(hkv) + 2 * T * hkv * 8
    if mode == "mixed":
        nv = lambda H: T * H * d * (2 + 0.5) + T * H * d / 16
        total += nv(hq) + nv(hkv) + per(hkv)
    return total


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the process group (the slowest rank's
    time is the job's time); the values unchanged without a group of more than one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def measure_fp8_peak(dev):
    """Dense E4M3 GEMM throughput of this GPU: torch._scaled_mm at 8192^3 (per-tensor
    scales, bf16 out), best of 10 after warm-up, CUDA events.  None if unavailable."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            mm()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:
        return None


def timing_event(torch_mod):
    """A timing event that, recorded inside a stream capture, becomes a graph node."""
    try:
        return torch_mod.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


class WorkloadRun:
    """One workload on one route: buffers, the captured training call, and its timings."""

    def __init__(self, F, w, mode, dev, flush):
        import torch
        self.torch, self.F, self.w, self.mode, self.dev, self.flush = torch, F, w, mode, dev, flush
        self.T, self.N = w.total_tokens, len(w.lengths)
        self.pairs = W.visible_pair_count(w.lengths, w.window)
        self.flops = 14.0 * w.d * w.hq * self.pairs
        inp = W.make_inputs(w)
        self.host = {n: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory() for n, b in inp.items()}
        self.x = {n: t.to(dev) for n, t in self.host.items()}
        self.cu_host = torch.tensor(w.cu_seqlens, dtype=torch.int32).pin_memory()
        self.cu = self.cu_host.to(dev)
        self.att = F.FlamiaAttention(self.T, self.N, w.hq, w.hkv, w.d, device=dev, strict=mode == "strict",
                                     mixed=mode == "mixed", causal=w.causal, window=w.window)
        self.stream = torch.cuda.current_stream(dev)
        self.o_plain = F.Options()
        import ctypes
        ctypes.pointer(self.o_plain)[0] = self.att.opts

    def step(self, o_fwd=None, o_bwd=None, qev=None):
        att, cu = self.att, self.cu
        att.plan_build(cu)
        cur = self.torch.cuda.current_stream()     # the capture stream while a graph is captured
        if qev:
            qev[0].record(cur)
        att.quantize(self.x["q"], self.x["k"], self.x["v"], cu)
        if qev:
            qev[1].record(cur)
        att.opts = o_fwd or self.o_plain
        att.forward(cu)
        att.opts = o_bwd or self.o_plain
        att.backward(self.x["do"], cu)
        att.opts = self.o_plain

    def _opts_with_events(self, n):
        import ctypes
        torch = self.torch
        evs = [timing_event(torch) for _ in range(n)]
        if any(e is None for e in evs):
            return None
        for e in evs:
            e.record(self.stream)          # creates the underlying cudaEvent_t
        arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
        o = self.F.Options()
        ctypes.pointer(o)[0] = self.att.opts
        o.timing_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
        return evs, arr, o

    def warm_and_capture(self, warmup):
        torch = self.torch
        for _ in range(max(warmup, 3)):
            self.step()
        torch.cuda.synchronize()
        assert self.att.device_status() == 0, "device status error during warm-up"
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize()
        for _ in range(max(warmup, 3)):
            self.graph.replay()
        torch.cuda.synchronize()

    def phases(self, n):
        """Per-kernel times inside a CUDA graph of the step: the library's timing hook and
        two events around the Q/K/V quantization are captured as event-record nodes; each
        replay follows an L2 flush and is read before the next one."""
        torch = self.torch
        ef, eb = self._opts_with_events(2), self._opts_with_events(8)
        qev = [timing_event(torch), timing_event(torch)]
        if ef is None or eb is None or qev[0] is None:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(ef[2], eb[2], qev)
        torch.cuda.synchronize()
        rows = []
        for i in range(n + 2):
            self.flush.zero_()
            g.replay()
            torch.cuda.synchronize()
            if i >= 2:
                e, b = ef[0], eb[0]
                rows.append(dict(quantize_qkv=qev[0].elapsed_time(qev[1]), fwd_kernel=e[0].elapsed_time(e[1]),
                                 bwd_prep=b[0].elapsed_time(b[1]), bwd_boost=b[2].elapsed_time(b[3]),
                                 bwd_kernel=b[4].elapsed_time(b[5]), bwd_finalise=b[6].elapsed_time(b[7])))
        assert self.att.device_status() == 0, "device status error during the phase replays"
        del g
        return {k: float(np.median([r[k] for r in rows])) for k in rows[0]}

    def timed(self, steps, rounds, world):
        """`steps` graph replays, each after an L2 flush (outside its events), bracketed
        by a barrier and a synchronize; per-round mean, median over rounds."""
        torch = self.torch
        import torch.distributed as dist
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(steps):
            self.flush.zero_()
            starts[i].record(self.stream)
            self.graph.replay()
            ends[i].record(self.stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t1 = time.time()
        ms = np.array([s.elapsed_time(e) for s, e in zip(starts, ends)])
        assert self.att.device_status() == 0, "device status error during the timed steps"
        per_round = [float(c.mean()) for c in np.array_split(ms, max(1, min(rounds, len(ms))))]
        return dict(mean=float(ms.mean()), median_of_rounds=float(np.median(per_round)), rounds=per_round,
                    t_wall=(t0, t1))

    def _out_host(self):
        att = self.att
        return {n: self.torch.empty_like(t, device="cpu").pin_memory() for n, t in
                (("o", att.out), ("dq", att.dq), ("dk", att.dk), ("dv", att.dv))}

    def e2e_serial(self, steps):
        """The training call through the public API with host buffers, one step at a time:
        pinned inputs in and results out inside each step's events.  The copies run on a
        second stream: dO comes in while the forward runs and O goes out while the
        backward runs (Q, K, V and cu_seqlens before the forward, dQ, dK, dV after the
        backward).  Returns the median ms per step and the bytes each way."""
        torch, att, x, host, stream = self.torch, self.att, self.x, self.host, self.stream
        out_host = self._out_host()
        h2d = sum(t.numel() * t.element_size() for t in host.values()) + self.cu_host.numel() * 4
        d2h = sum(t.numel() * t.element_size() for t in out_host.values())
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy_stream = torch.cuda.Stream(self.dev)
        ev_qkv, ev_do, ev_fwd, ev_bwd, ev_out = (torch.cuda.Event() for _ in range(5))
        res = []
        for i in range(steps + 1):
            self.flush.zero_()
            e0.record(stream)
            copy_stream.wait_event(e0)
            with torch.cuda.stream(copy_stream):
                self.cu.copy_(self.cu_host, non_blocking=True)
                for n in ("q", "k", "v"):
                    x[n].copy_(host[n], non_blocking=True)
                ev_qkv.record(copy_stream)
                x["do"].copy_(host["do"], non_blocking=True)
                ev_do.record(copy_stream)
            stream.wait_event(ev_qkv)
            att.plan_build(self.cu)
            att.quantize(x["q"], x["k"], x["v"], self.cu)
            att.forward(self.cu)
            ev_fwd.record(stream)
            stream.wait_event(ev_do)
            att.backward(x["do"], self.cu)
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
                res.append(e0.elapsed_time(e1))
        assert att.device_status() == 0, "device status error during the end-to-end steps"
        return float(np.median(res)), h2d, d2h

    def e2e_pipelined(self, steps, rounds=3):
        """The same steps as a training loop runs them: the inputs of step i + 1 (Q, K, V,
        dO, cu_seqlens; two device buffer sets) are copied in on one stream while step i
        computes and its results (O after the forward, dQ, dK, dV after the backward) are
        copied out on another, so the two link directions overlap.  Every step's copies
        are inside the timed region: ms per step = (the whole run of `steps` steps,
        pipeline fill and drain included) / steps, median of `rounds` runs.  The inputs
        (268 MB at the headline size) are larger than L2, so there is no flush."""
        torch, att, host, stream = self.torch, self.att, self.host, self.stream
        xs = [(self.x, self.cu), ({n: torch.empty_like(t) for n, t in self.x.items()}, torch.empty_like(self.cu))]
        out_host = self._out_host()
        cin, cout = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_used = [torch.cuda.Event() for _ in range(2)]
        ev_fwd, ev_bwd, ev_o, ev_out = (torch.cuda.Event() for _ in range(4))

        def copy_in(i):
            b = i % 2
            x, cu = xs[b]
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(ev_used[b])        # step i - 2 is done with this buffer set
                cu.copy_(self.cu_host, non_blocking=True)
                for n in ("q", "k", "v", "do"):
                    x[n].copy_(host[n], non_blocking=True)
                ev_in[b].record(cin)

        res = []
        for _ in range(rounds):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            cin.wait_event(e0)
            cout.wait_event(e0)
            copy_in(0)
            for i in range(steps):
                x, cu = xs[i % 2]
                if i + 1 < steps:
                    copy_in(i + 1)
                stream.wait_event(ev_in[i % 2])
                if i > 0:
                    stream.wait_event(ev_o)            # O of step i - 1 has been read
                att.plan_build(cu)
                att.quantize(x["q"], x["k"], x["v"], cu)
                att.forward(cu)
                ev_fwd.record(stream)
                if i > 0:
                    stream.wait_event(ev_out)          # dQ, dK, dV of step i - 1 have been read
                att.backward(x["do"], cu)
                ev_used[i % 2].record(stream)
                ev_bwd.record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(ev_fwd)
                    out_host["o"].copy_(att.out, non_blocking=True)
                    ev_o.record(cout)
                    cout.wait_event(ev_bwd)
                    for n in ("dq", "dk", "dv"):
                        out_host[n].copy_(getattr(att, n), non_blocking=True)
                    ev_out.record(cout)
            stream.wait_event(ev_out)
            e1.record(stream)
            e1.synchronize()
            res.append(e0.elapsed_time(e1) / steps)
        assert att.device_status() == 0, "device status error during the end-to-end steps"
        del xs[1]
        torch.cuda.empty_cache()
        return float(np.median(res)), res

    def link_bandwidth(self, h2d_bytes, d2h_bytes):
        """Pinned host <-> device copy rates of this machine for the step's byte counts: each
        direction alone and both at once (one stream each), best of 3, CUDA events."""
        torch, dev = self.torch, self.dev
        hi = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
        di = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
        ho = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
        do_ = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
        s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def best(which):
            t = float("inf")
            for _ in range(4):
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                cur = torch.cuda.current_stream(dev)
                e0.record(cur)
                for st, dst, src, on in ((s1, di, hi, "in"), (s2, ho, do_, "out")):
                    if on in which:
                        st.wait_event(e0)
                        with torch.cuda.stream(st):
                            dst.copy_(src, non_blocking=True)
                        ev = torch.cuda.Event()
                        ev.record(st)
                        cur.wait_event(ev)
                e1.record(cur)
                e1.synchronize()
                t = min(t, e0.elapsed_time(e1))
            return t

        t_in, t_out, t_both = best(("in",)), best(("out",)), best(("in", "out"))
        del hi, di, ho, do_
        torch.cuda.empty_cache()
        return {"h2d_gbs": h2d_bytes / (t_in * 1e-3) / 1e9, "d2h_gbs": d2h_bytes / (t_out * 1e-3) / 1e9,
                "both_directions_gbs": (h2d_bytes + d2h_bytes) / (t_both * 1e-3) / 1e9,
                "both_directions_ms": t_both}

    def kernel_roofline(self, ph, fp8_peak):
        d, hq = self.w.d, self.w.hq
        f_fwd, f_bwd = 4.0 * d * hq * self.pairs, 10.0 * d * hq * self.pairs
        if ph["bwd_kernel"] >= ph["fwd_kernel"]:
            name, ms, flops, src = "attn_bwd_kernel", ph["bwd_kernel"], f_bwd, "attn_bwd.cu"
        else:
            name, ms, flops, src = "attn_fwd_kernel", ph["fwd_kernel"], f_fwd, "attn_fwd.cu"
        ach = flops / (ms * 1e-3) / 1e12
        rec = traffic_record(src, self.w.name) if self.mode == "default" else None
        traffic = rec["dram_bytes_per_launch"] if rec else None
        return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": ach / fp8_peak, "traffic": traffic, "algorithmic_flops": flops,
                "per_unit": "FLOPs per launch = %s * head_dim * hq * visible pairs" % ("10" if "bwd" in name else "4")}

    def release(self):
        del self.graph
        self.att = self.x = self.host = None
        self.torch.cuda.empty_cache()


def exp_ceiling(d, sms, sm_mhz):
    """Upper bounds set by the MUFU exponentials: one ex2 per visible pair in the forward
    and one in the backward, against 4d (forward), 10d (backward) and 14d (call) FLOPs."""
    rate = EX2_PER_CLK_PER_SM * sms * sm_mhz * 1e6          # ex2 per second
    return {"ex2_per_clk_per_sm": EX2_PER_CLK_PER_SM, "sms": sms, "sm_mhz": sm_mhz,
            "fwd_tflops": 4.0 * d * rate / 1e12, "bwd_tflops": 10.0 * d * rate / 1e12,
            "call_tflops": 7.0 * d * rate / 1e12}


def run_ours(args, rank, world, local_rank):
    import torch
    from microscaled_precision_causal_gb300 import build as _b
    _b.build()
    import microscaled_precision_causal_gb300 as F

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pk = peaks()
    fp8_meas = measure_fp8_peak(dev) if rank == 0 else None
    fp8_peak = max(fp8_meas or 0.0, 2.0 * pk["bf16"])
    fp8_src = ("measured E4M3 _scaled_mm 8192^3 burst" if fp8_meas and fp8_meas >= 2.0 * pk["bf16"]
               else "2 x %s bf16 burst (nominal FP8/BF16 ratio)" % pk["src"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    w = W.WORKLOADS[args.workload]
    run = WorkloadRun(F, w, args.mode, dev, flush)
    run.warm_and_capture(args.warmup)

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
    ph = run.phases(min(args.steps, 30))
    tm = run.timed(args.steps, args.rounds, world)
    (ms_step,) = max_over_ranks([tm["median_of_rounds"]], dev)
    e2e_serial_ms, h2d, d2h = run.e2e_serial(5)
    e2e_ms, e2e_rounds = run.e2e_pipelined(args.e2e_steps)
    link = run.link_bandwidth(h2d, d2h)
    e2e_ms, e2e_serial_ms = max_over_ranks([e2e_ms, e2e_serial_ms], dev)
    lines = sampler.stop() if not args.no_clocks else None
    clocks = ClockSampler.summarize(lines, *tm["t_wall"]) if lines else None
    if rank != 0:
        return None
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = clocks["sm_mhz"] if clocks else 2070.0
    value = world * run.flops / (ms_step * 1e-3) / 1e12
    q_ms = ph["quantize_qkv"] if ph else None
    qb = quantizer_bytes(w, args.mode)
    qrec = traffic_record("quantize.cu", w.name) if args.mode == "default" else None
    res = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": w.name, "mode": args.mode, "causal": w.causal, "window": list(w.window),
                   "cuda_graph": True, "total_tokens": run.T,
                   "num_docs": run.N, "hq": w.hq, "hkv": w.hkv, "head_dim": w.d, "visible_pairs": run.pairs,
                   "flops_per_step": run.flops,
                   "l2": "flushed between timed steps (256 MiB write); step inputs 256 MiB > L2",
                   "timing": "%d graph replays in %d rounds; ms_per_step = median of the round means "
                             "(mean %.4f ms)" % (args.steps, args.rounds, tm["mean"]),
                   "frac_of_fp8_peak": value / world / fp8_peak, "fp8_peak_tflops": fp8_peak,
                   "fp8_peak_source": fp8_src, "fp8_measured_tflops": fp8_meas},
        "phases_ms": ph,
        "roofline": run.kernel_roofline(ph, fp8_peak) if ph else None,
        "exp_ceiling": exp_ceiling(w.d, sms, sm_mhz),
        "quantizer_roofline": ({"bound": "hbm", "achieved": qb / (q_ms * 1e-3) / 1e9, "peak": pk["hbm"],
                                "unit": "GB/s", "frac": qb / (q_ms * 1e-3) / 1e9 / pk["hbm"],
                                "bytes_per_step": qb, "ms": q_ms,
                                "traffic": qrec["dram_bytes_per_launch"] if qrec else None,
                                "measured": "inside the CUDA graph (event-record nodes), median of replays"}
                               if ph else None),
        "e2e": {"value": world * run.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "rounds_ms": e2e_rounds,
                "copies": ("pinned host buffers, %d steps as a training loop runs them: step i + 1's inputs come in "
                           "on one stream while step i computes and its results go out on another (two device "
                           "input sets); ms_per_step = whole run / steps, fill and drain included, median of 3 "
                           "runs; inputs > L2, no flush" % args.e2e_steps),
                "serial": {"value": world * run.flops / (e2e_serial_ms * 1e-3) / 1e12, "ms_per_step": e2e_serial_ms,
                           "copies": "one step at a time: Q, K, V in, then the call (dO in during the forward, "
                                     "O out during the backward), then dQ, dK, dV out"},
                "link": dict(link, floor_ms_per_step=link["both_directions_ms"],
                             note="pinned copies of the step's bytes, each direction alone and both at once; "
                                  "the pipelined loop cannot beat both_directions_ms per step")},
        "gpu_launches": LAUNCHES_PER_STEP[args.mode] * args.steps,
        "clocks": clocks,
    }
    run.release()
    if not args.no_cpu_baseline:
        s = oracle_sample(w, args.cpu_seconds, mode=args.mode)
        res["cpu_baseline"] = {
            "value": s["tflops"], "unit": "TFLOPS", "cores": blas_threads(), "kind": "oracle",
            "sample": (f"oracle fwd+bwd (fp64 numpy) on the first {s['tokens']} tokens of the longest document, "
                       f"{s['heads']} query heads: {s['seconds']:.1f} s")}
    if not args.no_secondary and world == 1:
        res["workloads"] = {}
        for wname, mode in SECONDARY:
            if wname == w.name and mode == args.mode:
                continue
            ws = W.WORKLOADS[wname]
            r = WorkloadRun(F, ws, mode, dev, flush)
            r.warm_and_capture(3)
            p2 = r.phases(10)
            t2 = r.timed(args.secondary_steps, 3, 1)
            v2 = r.flops / (t2["median_of_rounds"] * 1e-3) / 1e12
            ent = {"mode": mode, "causal": ws.causal, "value": v2, "unit": "TFLOPS", "ms_per_step": t2["median_of_rounds"],
                   "rounds_ms": t2["rounds"], "frac_of_fp8_peak": v2 / fp8_peak, "phases_ms": p2,
                   "roofline": r.kernel_roofline(p2, fp8_peak) if p2 else None,
                   "exp_ceiling_call_tflops": exp_ceiling(ws.d, sms, sm_mhz)["call_tflops"]}
            if mode == "default" and wname in PAGES_CALL_MS:
                ms_p, src = PAGES_CALL_MS[wname]
                ent["pages_call_ms"] = {"value": ms_p, "source": src,
                                        "ratio": ms_p / t2["median_of_rounds"]}
            r.release()
            if not args.no_cpu_baseline:
                s = oracle_sample(ws, args.cpu_seconds / 3, mode=mode)
                ent["cpu_baseline"] = {"value": s["tflops"], "unit": "TFLOPS", "cores": blas_threads(),
                                       "kind": "oracle",
                                       "sample": f"first {s['tokens']} tokens, {s['heads']} query heads: "
                                                 f"{s['seconds']:.1f} s"}
            res["workloads"][f"{wname}/{mode}"] = ent
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
