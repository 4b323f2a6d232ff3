#!/usr/bin/env python3
"""Benchmark of the per-layer MoE expert step on one GB300 (or N replicas).

A step is one decode token through every MoE layer of the workload: per
layer moe_layer_forward (router, control step, expert FFN + combine carrying
the fill copies), through the C ABI on inputs already resident in HBM.  The
FFN's own duration (roofline) is taken from a separate replay of the same
steps as moe_route / moe_cache_step / moe_expert_ffn calls with CUDA events
around each moe_expert_ffn.  `e2e` repeats the measurement
through moe_layer_forward with the step's hidden states copied in from pinned
host memory and the layer outputs copied back every step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Multi-GPU: the decode step does not shard in this build (one control step
per shared cache); N GPUs run N independent replicas, no collective.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer decode tok/s & expert-weight HBM GB/s vs peak; prefill TFLOPS"

WORKLOADS = {
    "qwen_decode": dict(
        desc="Qwen3.6-35B-A3B-shaped decode: 40 MoE layers, H=2048, I=512, E=256, top-8 "
             "softmax + 1 shared expert (I=512), int4 affine g64, batch 1, 2560 slots (25% of "
             "pairs), K=8, B_P/B_H=52.7/77.3 GB/s, AR(1) hidden states rho=0.9",
        L=40, H=2048, I=512, E=256, k=8, T=1, shared=True, router="softmax", slots=2560, K=8,
        bp=52700, bh=77300),
    "deepseek_decode_b1": dict(
        desc="DeepSeek-V3-style decode: 8 MoE layers, H=7168, I=2048, E=256 in 8 groups, top-4 "
             "groups, top-8, scale 2.5, selection bias N(0,0.01), int4 affine g64, batch 1, 307 "
             "slots (15%), K=8, B_P/B_H=11.8/47.5 GB/s",
        L=8, H=7168, I=2048, E=256, k=8, T=1, shared=False, router="sigmoid_group", ng=8, G=4,
        scale=2.5, slots=307, K=8, bp=11800, bh=47500),
    "deepseek_decode_b8": dict(
        desc="DeepSeek-V3-style decode, batch 8 (8 independent AR(1) streams), otherwise as "
             "deepseek_decode_b1",
        L=8, H=7168, I=2048, E=256, k=8, T=8, shared=False, router="sigmoid_group", ng=8, G=4,
        scale=2.5, slots=307, K=8, bp=11800, bh=47500),
    "qwen_decode_nvfp4": dict(
        desc="qwen_decode with NVFP4 experts (E2M1 elements, one E4M3 scale per 16, fp32 "
             "matrix scales), the format the pages deploy Qwen3.6 in",
        L=40, H=2048, I=512, E=256, k=8, T=1, shared=True, router="softmax", slots=2560, K=8,
        bp=52700, bh=77300, fmt=2),
    "deepseek_decode_b1_mxfp4": dict(
        desc="deepseek_decode_b1 with MXFP4 experts (E2M1 elements, one E8M0 scale per 32), "
             "the format the pages deploy DeepSeek-V4-Flash in",
        L=8, H=7168, I=2048, E=256, k=8, T=1, shared=False, router="sigmoid_group", ng=8, G=4,
        scale=2.5, slots=307, K=8, bp=11800, bh=47500, fmt=1),
    "qwen_prefill": dict(
        desc="Whole-layer prefill, Qwen3.6-35B-A3B layer shape: H=2048, I=512, E=256, top-8 "
             "softmax + shared expert, 8192 tokens of N(0,1) bf16 hidden states with the router "
             "logit of expert (t mod 256) raised by 3 (routing union = all 256 experts), int4 "
             "affine g64 dequantised to bf16 into tcgen05 grouped GEMMs; 2 layers alternating, "
             "the next layer copied bank -> buffer on a second stream (double buffer)",
        L=2, H=2048, I=512, E=256, k=8, T=8192, shared=True, router="softmax", prefill=True),
    "elastic_resize": dict(
        desc="Elastic slot pool on the qwen_decode shape and inputs (40 layers, H=2048, I=512, "
             "E=256, top-8 + shared, int4 g64, K=8, B_P/B_H=52.7/77.3 GB/s): each step fills "
             "the 2560-slot pool with a random resident set and runs one decode step through "
             "all layers (both untimed), then the pool shrinks to 2048 slots (the KV cache takes "
             "0.9 GB: the 512 least recently routed experts are evicted, the kept ones past slot "
             "2048 move down) and grows back to 2560; the two re-divisions are timed",
        L=40, H=2048, I=512, E=256, k=8, T=1, shared=True, router="softmax", slots=2560, K=8,
        bp=52700, bh=77300, elastic=True, slots_lo=2048),
    "qwen_prefill_nvfp4": dict(
        desc="qwen_prefill with NVFP4 experts (E2M1 elements, one E4M3 scale per 16, fp32 "
             "matrix scales; dequantised exactly to bf16 inside the tcgen05 grouped GEMMs)",
        L=2, H=2048, I=512, E=256, k=8, T=8192, shared=True, router="softmax", prefill=True,
        fmt=2),
    "cache_sweep": dict(
        desc="Cache stress sweep: 40 layers x 256 experts, top-8, Zipf(1.1) routing traces of "
             "2048 steps per layer with 70% step-to-step overlap fed straight to the control "
             "step (no router, no fill); capacity 5/10/25/50% of pairs x B_P/B_H in "
             "{52.7/77.3, 11.8/47.5, 77.3/77.3} GB/s, K=8; replacement policies (shared LRU, "
             "per-layer LRU, static hot set, static whole layers) replayed on the same traces "
             "and on phased ones (popular experts redrawn every 256 steps)",
        L=40, H=64, I=64, E=256, k=8, T=1, shared=False, router="softmax", K=8, sweep=True,
        trace_steps=2048, caps=(0.05, 0.10, 0.25, 0.50),
        ratios=((52700, 77300), (11800, 47500), (77300, 77300)), slots=2560, bp=52700, bh=77300,
        phase_steps=256),
}


def run_config(args, w, world):
    """The `config` object of a bench line; the same for the GPU arm and the
    reference arm of a workload."""
    par = f"replicas x{world}" if world > 1 else "single GPU"
    if w.get("prefill"):
        return {"workload": args.workload, "desc": w["desc"], "tokens": w["T"], "layers": w["L"],
                "parallelism": par,
                "l2": "inputs larger than L2: 453 MB of int4 experts per layer + 32 MB x"}
    if w.get("sweep"):
        return {"workload": args.workload, "desc": w["desc"], "layers": w["L"],
                "headline_point": "capacity 25%, B_P/B_H 52.7/77.3", "parallelism": par,
                "l2": "integer tables (<1 MB) stay in L2; this is a latency measurement"}
    se = 27 * w["H"] * w["I"] // 16  # int4 blob bytes (codes + bf16 scales / biases)
    per_layer = min(w["T"] * w["k"], w["E"]) + (1 if w["shared"] else 0)
    return {"workload": args.workload, "desc": w["desc"], "layers": w["L"], "batch": w["T"],
            "parallelism": par,
            "l2": f"inputs larger than L2: up to {per_layer * se * w['L'] / 1e6:.0f} MB of expert "
                  "weights touched per step vs 129 MB L2"}


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def max_over_ranks(ms, world, device=None):
    """The slowest rank's time (the job's time) when N replicas run; ms itself for N = 1."""
    if world <= 1:
        return ms
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_barrier(world):
    if world > 1:
        import torch

        torch.distributed.barrier()


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("ffn_coop.cu", "control_common.cuh", "route_select.cuh", "stream_common.cuh",
              "moe_internal.cuh"):
        h.update(open(os.path.join(ROOT, "moe_expert_offload_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, experts_per_launch, router_bytes):
    """DRAM bytes per launch of the timed kernel from the committed ncu summary,
    if it was taken on the current kernel source (else None).  The summary holds
    the bytes per expert of a smaller capture of the same expert shape (reads and
    writes, less the router weights); they are scaled by the experts each launch
    executes, plus this workload's router weights."""
    p = os.path.join(ROOT, "profiles", "ffn_decode_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return float(e["bytes_per_expert"]) * experts_per_launch + router_bytes


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ inputs
def make_inputs(w, n_steps, seed_base=0):
    from moe_expert_offload_gb300 import synth

    L, H, E, T = w["L"], w["H"], w["E"], w["T"]
    xs = np.stack([synth.ar1_stream(seed_base + l, n_steps, H, n_streams=T) for l in range(L)],
                  axis=1)  # [steps][L][T][H]
    wr = np.stack([synth.router_weights(100 + l, E, H) for l in range(L)])  # [L][E][H]
    bias = (np.stack([synth.selection_bias(300 + l, E) for l in range(L)])
            if w["router"] == "sigmoid_group" else None)
    return xs, wr, bias


def spec_of(w):
    import moe_expert_offload_gb300 as m

    fmt = w.get("fmt", m.FORMAT_INT4)
    if w["router"] == "sigmoid_group":
        return m.make_spec(w["L"], w["H"], w["I"], w["E"], w["k"], router="sigmoid_group",
                           n_groups=w["ng"], topk_groups=w["G"], routed_scale=w["scale"],
                           has_shared=w["shared"], fmt=fmt)
    return m.make_spec(w["L"], w["H"], w["I"], w["E"], w["k"], has_shared=w["shared"], fmt=fmt)


def make_bank(w, n, seed, dev):
    """The workload's expert bank in device memory (int4 or FP4 blobs)."""
    from moe_expert_offload_gb300 import synth

    if w.get("fmt", 0):
        return synth.make_fp4_bank_torch(n, w["H"], w["I"], w["fmt"] - 1, seed, dev)
    return synth.make_bank_torch(n, w["H"], w["I"], seed, dev)


# --------------------------------------------------------------- CPU oracle
class OracleRunner:
    """Times the CPU oracle on the same workload (its row loops on
    oracle.set_threads() host threads).  Expert blobs are generated on the host
    on first use (untimed); only oracle calls count."""

    def __init__(self, w, xs, wr, bias):
        import oracle
        from moe_expert_offload_gb300 import synth

        oracle.build()
        self.o, self.synth, self.w = oracle, synth, w
        self.xs, self.wr, self.bias = xs, wr, bias
        self.state = oracle.CacheState(w["L"] * w["E"], w["slots"])
        self.blobs = {}
        self.fp4 = w.get("fmt", 0) - 1  # the oracle's FP4 format, or -1 for int4
        rng = np.random.default_rng(12345)
        self.shared = self.make(rng) if w["shared"] else None
        self.spent = 0.0
        self.tokens = 0

    def make(self, rng):
        if self.fp4 >= 0:
            return self.synth.make_fp4_expert(rng, self.w["H"], self.w["I"], self.fp4)
        return self.synth.make_expert_bytes(rng, self.w["H"], self.w["I"])

    def blob(self, gid):
        b = self.blobs.get(gid)
        if b is None:
            b = self.make(np.random.default_rng(gid + 1))
            self.blobs[gid] = b
        return b

    def step(self, s):
        w, o = self.w, self.o
        for l in range(w["L"]):
            xb = self.xs[s, l]
            t0 = time.perf_counter()
            lg = o.router_logits(xb, self.wr[l])
            if w["router"] == "sigmoid_group":
                ids, wt = o.route_sigmoid_group(lg, self.bias[l], w["ng"], w["G"], w["k"],
                                                w["scale"])
            else:
                ids, wt = o.route_softmax_topk(lg, w["k"])
            o.cache_step(self.state, w["E"], l, ids, w["K"], w["bp"], w["bh"])
            self.spent += time.perf_counter() - t0
            need = {int(e) for e in ids.reshape(-1)}
            if self.fp4 >= 0:
                # FP4: the oracle's FP4 expert per routed expert, weighted sum in float64
                blobs = {e: self.blob(l * w["E"] + e) for e in need}
                t0 = time.perf_counter()
                y = np.zeros((xb.shape[0], w["H"]))
                for e in need:
                    ye = o.fp4_expert_forward(blobs[e], w["H"], w["I"], self.fp4, xb)
                    for t in range(xb.shape[0]):
                        for j in range(ids.shape[1]):
                            if ids[t, j] == e:
                                y[t] += float(wt[t, j]) * ye[t]
                if self.shared is not None:
                    y += o.fp4_expert_forward(self.shared, w["H"], w["I"], self.fp4, xb)
                self.spent += time.perf_counter() - t0
            else:
                full = [self.blob(l * w["E"] + (e if e in need else next(iter(need))))
                        for e in range(w["E"])]
                t0 = time.perf_counter()
                o.moe_ffn(full, w["H"], w["I"], xb, ids, wt, self.shared, w["I"])
                self.spent += time.perf_counter() - t0
        self.tokens += w["T"]


def cpu_baseline(w, xs, wr, bias, budget_s=8.0, max_steps=64):
    """The oracle on a bounded sample of the workload, twice: on one thread (the
    oracle as it stands) and with its row loops on every host core (the same
    arithmetic and results)."""
    import oracle

    oracle.build()
    ncores = host_cores()

    def run(threads):
        used = oracle.set_threads(threads)
        r = OracleRunner(w, xs, wr, bias)
        s = 0
        while s < min(max_steps, xs.shape[0]) and (r.spent < budget_s or s == 0):
            r.step(s)
            s += 1
        oracle.set_threads(1)
        return r.tokens / r.spent, used, (f"{s} decode steps x {w['L']} layers x batch {w['T']} "
                                          f"(route, control, float64 FFN) in {r.spent:.1f} s of "
                                          f"oracle time, {used} thread(s)")

    v1, _, s1 = run(1)
    vn, used, sn = run(ncores)
    return {"value": v1, "unit": "tok/s", "cores": 1, "kind": "oracle", "sample": s1,
            "host_cores": ncores,
            "all_cores": {"value": vn, "unit": "tok/s", "cores": used,
                          "kind": "oracle, row loops on every host core", "sample": sn}}


def reference_line(args, w, world, val, unit, spent, sample, dtype, cores=1):
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic", "config": run_config(args, w, world),
            "cpu_baseline": {"value": val, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference_prefill(args, w, world):
    """Each step is one token of the prefill layer through the oracle (route +
    float64 FFN, the token's experts dequantised per call): a bounded sample."""
    import oracle

    x_h, wr_h = prefill_inputs(w)
    oracle.build()
    used = oracle.set_threads(host_cores())
    r = PrefillOracle(w, x_h, wr_h)
    for t in range(args.warmup):
        r.token(t)
    r.spent, r.n = 0.0, 0
    for t in range(args.warmup, args.warmup + args.steps):
        r.token(t % w["T"])
    val = r.flops_per_token * r.n / r.spent / 1e12
    sample = (f"{r.n} tokens of the {w['T']}-token prefill layer (route + float64 FFN, row loops "
              f"on {used} host thread(s)), {r.spent:.1f} s of oracle time")
    print(json.dumps(reference_line(args, w, world, val, "TFLOP/s", r.spent, sample, "f64",
                                    cores=used)), flush=True)


def run_reference_sweep(args, w, world):
    """Each step is one trace step through all layers' oracle control steps at the
    capacity-25%, B_P/B_H 52.7/77.3 point of the sweep."""
    import oracle
    from moe_expert_offload_gb300 import synth

    oracle.build()
    L, E, K = w["L"], w["E"], w["K"]
    n = args.warmup + args.steps
    tr = np.stack([synth.zipf_trace(1000 + l, n, E, w["k"]) for l in range(L)], axis=1)
    state = oracle.CacheState(L * E, int(round(0.25 * L * E)))
    spent = 0.0
    for s in range(n):
        if s == args.warmup:
            spent = 0.0
        for l in range(L):
            t0 = time.perf_counter()
            oracle.cache_step(state, E, l, tr[s, l:l + 1], K, 52700, 77300)
            spent += time.perf_counter() - t0
    val = args.steps * L / spent
    sample = (f"{args.steps} trace steps x {L} layers of oracle control steps, single thread, "
              f"{spent:.3f} s of oracle time")
    print(json.dumps(reference_line(args, w, world, val, "layer-steps/s", spent, sample, "int32")),
          flush=True)


def run_reference_elastic(args, w, world):
    """Each step is the oracle's shrink and growth of a full pool of the workload's
    size (tables only: the oracle has no slot pool), on tables of random recency."""
    import oracle

    oracle.build()
    n_ids = w["L"] * w["E"]
    rng = np.random.default_rng(11)
    spent = 0.0
    for s in range(args.warmup + args.steps):
        if s == args.warmup:
            spent = 0.0
        st = oracle.CacheState(n_ids, w["slots"])
        oracle.cache_place(st, w["E"], w["L"], rng.choice(n_ids, w["slots"], replace=False))
        st.ts[:] = rng.integers(1, 1000, w["slots"])
        t0 = time.perf_counter()
        oracle.cache_resize(st, w["slots_lo"])
        oracle.cache_resize(st, w["slots"])
        spent += time.perf_counter() - t0
    val = 2 * args.steps / spent
    sample = (f"{args.steps} shrink + growth pairs of a full {w['slots']}-slot pool, single "
              f"thread, {spent:.3f} s of oracle time")
    print(json.dumps(reference_line(args, w, world, val, "re-divisions/s", spent, sample,
                                    "int32")), flush=True)


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    if w.get("prefill"):
        return run_reference_prefill(args, w, world)
    if w.get("sweep"):
        return run_reference_sweep(args, w, world)
    if w.get("elastic"):
        return run_reference_elastic(args, w, world)
    import oracle

    n = args.warmup + args.steps
    xs, wr, bias = make_inputs(w, n)
    oracle.build()
    used = oracle.set_threads(host_cores())
    r = OracleRunner(w, xs, wr, bias)
    for s in range(args.warmup):
        r.step(s)
    r.spent, r.tokens = 0.0, 0
    for s in range(args.warmup, n):
        r.step(s)
    val = r.tokens / r.spent
    sample = (f"{args.steps} decode steps x {w['L']} layers x batch {w['T']} (route, control, "
              f"float64 FFN, row loops on {used} host thread(s)), {r.spent:.1f} s of oracle time")
    print(json.dumps(reference_line(args, w, world, val, "tok/s", r.spent, sample, "f64",
                                    cores=used)), flush=True)


# ----------------------------------------------------------------- GPU arm
def run_gpu(args, w, rank, world, local_rank):
    import torch

    import moe_expert_offload_gb300 as m
    from moe_expert_offload_gb300 import _build, synth

    _build.build()
    m.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    L, H, I, E, k, T = w["L"], w["H"], w["I"], w["E"], w["k"], w["T"]
    spec = spec_of(w)
    se = m.moe_expert_bytes(spec)
    n_in = 2 * (args.warmup + args.steps)
    xs_h, wr_h, bias_h = make_inputs(w, n_in)
    bank = make_bank(w, L * E + (1 if w["shared"] else 0), 7, dev)
    shared = bank[L * E] if w["shared"] else None
    cache = m.DeviceCache(spec, w["slots"], w["K"], w["bp"], w["bh"], bank[:L * E], device=dev)
    plan = m.DevicePlan(T * k, w["K"], device=dev)
    xs = torch.from_numpy(xs_h.view(np.int16)).to(dev)          # [steps][L][T][H]
    wr = torch.from_numpy(wr_h.view(np.int16)).to(dev)          # [L][E][H]
    bias = None if bias_h is None else torch.from_numpy(bias_h).to(dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    y = torch.empty((L, T, H), dtype=torch.float32, device=dev)
    fws = m.moe_ffn_workspace_bytes(spec, T)
    ws = torch.empty(max(fws, m.moe_layer_workspace_bytes(spec, T)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    def bias_l(l):
        return None if bias is None else bias[l]

    def layer(x, l, sh, ev=None):
        m.moe_route(spec, x, T, wr[l], bias_l(l), logits, ids, wts, sh)
        m.moe_cache_step(spec, cache.c, l, ids, T, plan.c, 1, sh)
        if ev is not None:
            ev[0].record(torch.cuda.current_stream())
        m.moe_expert_ffn(spec, cache.c, l, plan.c, x, T, ids, wts, shared, ws, fws, y[l], sh)
        if ev is not None:
            ev[1].record(torch.cuda.current_stream())

    lws = m.moe_layer_workspace_bytes(spec, T)
    # the whole layer step is one cooperative kernel for this shape (the cache has sync words)
    one_kernel = m.moe_layer_kernel_count(spec, cache.c, T) == 1

    def step(s, ev=None):
        # the timed step: one moe_layer_forward per layer (route, control, FFN
        # carrying the fill copy).  With events: around each layer call when the
        # step is one kernel, else the same work as separate calls so that the
        # FFN launches can be bracketed
        sh = torch.cuda.current_stream().cuda_stream
        for l in range(L):
            if ev is None or one_kernel:
                if ev is not None:
                    ev[l][0].record(torch.cuda.current_stream())
                m.moe_layer_forward(spec, cache.c, l, xs[s, l], T, wr[l], bias_l(l), shared,
                                    plan.c, ids, wts, ws, lws, y[l], sh)
                if ev is not None:
                    ev[l][1].record(torch.cuda.current_stream())
            else:
                layer(xs[s, l], l, sh, ev[l])

    def barrier():
        rank_barrier(world)

    # B_P / B_H measured on this device and shape (untimed); with --adaptive-q they
    # replace the configured rates for the whole run
    pws_bytes = m.moe_profile_workspace_bytes(spec)
    pws = torch.empty(pws_bytes, dtype=torch.uint8, device=dev)
    m.moe_cache_reset(spec, cache.c, sp)
    bp_meas, bh_meas = m.moe_profile_bandwidths(spec, cache.c, 0, pws, pws_bytes, reps=10)
    del pws
    if args.adaptive_q:
        cache.c.bp_mbps, cache.c.bh_mbps = bp_meas, bh_meas
    m.moe_cache_reset(spec, cache.c, sp)
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()

    # The timed region is one CUDA graph holding all K steps back to back (each
    # step reads its own resident inputs), with nothing between the kernels.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for s in range(args.steps):
            step(args.warmup + s)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    # The timed region is the one replay of the K steps.  The clock sampler runs
    # from before it until the GPU has been kept busy for >= 1 s by untimed
    # replays of the same graph after it, so that the clock record reflects the
    # sustained state of this load (a K-step region alone can be a few ms).
    with ClockSampler(local_rank) as clk:
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        soak_t0 = time.perf_counter()
        while time.perf_counter() - soak_t0 < 1.0:
            graph.replay()
            torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    del graph

    # Per-launch duration of the dominant kernel for the roofline (the layer
    # kernel, or the FFN kernel of the multi-kernel form): a second graph of the
    # same steps with timing events around every such launch (event nodes sit
    # between kernels, so this graph is replayed outside the timed region).
    ev_steps = min(args.steps, 16)
    try:
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        mk()
        evs = [[[mk(), mk()] for _ in range(L)] for _ in range(ev_steps)]
        g_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ev):
            for s in range(ev_steps):
                step(args.warmup + s, evs[s])
        g_ev.replay()
        torch.cuda.synchronize()
        ffn_ms = [evs[s][l][0].elapsed_time(evs[s][l][1]) for s in range(ev_steps)
                  for l in range(L)]
        ffn_timing = (f"CUDA events around every {'layer' if one_kernel else 'FFN'} launch, "
                      f"{ev_steps} steps replayed as a graph outside the timed region")
        del g_ev
    except TypeError:
        ffn_ms = []
        ffn_timing = "unavailable (this torch build has no external events)"
    ffn_avg_s = statistics.mean(ffn_ms) * 1e-3 if ffn_ms else float("nan")

    # statistics of the control decisions (untimed replay of more steps)
    n_uniq = n_fill = n_direct = n_miss = 0
    stat_steps = min(args.steps, 16)
    for s in range(stat_steps):
        for l in range(L):
            m.moe_layer_forward(spec, cache.c, l, xs[args.warmup + args.steps + s, l], T, wr[l],
                                bias_l(l), shared, plan.c, ids, wts, ws, lws, y[l], sp)
            c = plan.counts.cpu().numpy()
            n_uniq += int(c[0])
            n_miss += int(c[2])
            n_fill += int(c[4])
            n_direct += int(c[5])
    layer_steps = stat_steps * L

    # end to end through the public API, on the timed steps' own inputs and from
    # the same cache state (reset, then the warm-up steps): pinned host hidden
    # states -> device, the layers' moe_layer_forward calls (one captured graph),
    # layer outputs -> pinned host, every step, no host sync in the timed region.
    x_host = torch.from_numpy(
        xs_h[args.warmup:args.warmup + args.steps].view(np.int16).copy()).pin_memory()
    y_host = torch.empty((args.steps, L, T, H), dtype=torch.float32).pin_memory()
    x_dev = torch.empty((L, T, H), dtype=torch.int16, device=dev)

    def fwd_layers():
        sh = torch.cuda.current_stream().cuda_stream
        for l in range(L):
            m.moe_layer_forward(spec, cache.c, l, x_dev[l], T, wr[l], bias_l(l), shared, plan.c,
                                ids, wts, ws, lws, y[l], sh)

    fwd_layers()
    torch.cuda.synchronize()
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1):
        fwd_layers()

    def e2e_step(s):
        x_dev.copy_(x_host[s], non_blocking=True)
        g1.replay()
        y_host[s].copy_(y, non_blocking=True)

    m.moe_cache_reset(spec, cache.c, sp)
    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        e2e_step(s)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, dev)

    if rank != 0:
        return
    hbm, _, peak_kind = peaks()
    ffn_bytes = (n_uniq / layer_steps + (1 if w["shared"] else 0)) * se  # per FFN launch
    if one_kernel:
        # the layer kernel also reads the router weights and writes the fills
        ffn_bytes += E * H * 2 + (n_fill / layer_steps) * se
    achieved = ffn_bytes / ffn_avg_s / 1e9
    tokens = args.steps * T * world
    value = tokens / (ms * 1e-3)
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm,
            "traffic": ncu_traffic(args.workload, n_uniq / layer_steps + (1 if w["shared"] else 0),
                                   E * H * 2 if one_kernel else 0),
            "kernel": ("decode layer step (moe_layer_forward as one cooperative kernel: router "
                       "logits, selection, control step, gate/up + down carrying the fill)"
                       if one_kernel else
                       "decode expert FFN (moe_expert_ffn: counter memset + one cooperative "
                       "gate/up + down kernel)"),
            "algorithmic_bytes_per_launch": ffn_bytes, "avg_launch_us": ffn_avg_s * 1e6,
            "peak_kind": peak_kind, "timing": ffn_timing}
    cpu = cpu_baseline(w, xs_h, wr_h, bias_h) if world == 1 and not args.no_cpu else None
    # moe_layer_forward: logits, control step (+ selection for T <= 16, E <= 256, else a
    # separate select kernel), gate/up, down (+ a fill copy kernel for shapes whose FFN
    # does not carry the fill); the library reports the count for the shape
    launches_per_layer = m.moe_layer_kernel_count(spec, cache.c, T)
    # the FFN carries the fill when no copy kernel is counted: one kernel, or logits,
    # control, FFN (+ a separate selection kernel past 16 tokens or 256 experts)
    fused = launches_per_layer in (1, 3 + (0 if T <= 16 and E <= 256 else 1))
    out = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": run_config(args, w, world),
        "roofline": roof,
        "e2e": {"value": tokens / (ms_e2e * 1e-3), "unit": "tok/s",
                "h2d_bytes_per_step": L * T * H * 2, "d2h_bytes_per_step": L * T * H * 4},
        "gpu_launches": launches_per_layer * L * args.steps,
        "clocks": clk.summary(),
        "calibration": {"bp_mbps": bp_meas, "bh_mbps": bh_meas,
                        "configured_mbps": [w["bp"], w["bh"]], "used": "measured" if args.adaptive_q
                        else "configured",
                        "how": "moe_profile_bandwidths: the fill copy (B_P) and the decode FFN "
                               "(B_H) timed on this device, layer 0, untimed"},
        "cache": {"miss_rate": n_miss / max(n_uniq, 1), "fill_per_layer": n_fill / layer_steps,
                  "direct_per_layer": n_direct / layer_steps,
                  "uniq_per_layer": n_uniq / layer_steps},
        "ffn_gbs": achieved,
        # per layer-step: the experts read, the router weights and the fills (a fill
        # carried by the FFN writes the slot, S_e; a fill copy kernel reads and writes
        # it, 2 S_e), over the graph-timed step
        "step_gbs": ((n_uniq / layer_steps + (1 if w["shared"] else 0)) * se + E * H * 2 +
                     (1 if fused else 2) * se * n_fill / layer_steps) * L /
                    (ms * 1e-3 / args.steps) / 1e9,
    }
    if cpu:
        out["cpu_baseline"] = cpu
    print(json.dumps(out), flush=True)


def prefill_flops(w):
    """Algorithmic flops of the expert FFN per layer: 6*H*I per (token, expert)."""
    return 6.0 * w["H"] * w["I"] * w["T"] * (w["k"] + (1 if w["shared"] else 0))


def run_prefill(args, w, rank, world, local_rank):
    import torch

    import moe_expert_offload_gb300 as m
    from moe_expert_offload_gb300 import _build, synth

    _build.build()
    m.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    L, H, I, E, k, T = w["L"], w["H"], w["I"], w["E"], w["k"], w["T"]
    spec = spec_of(w)
    se = m.moe_expert_bytes(spec)
    bank = make_bank(w, L * E + 1, 7, dev)
    shared = bank[L * E]
    bufs = [torch.empty((E, se), dtype=torch.uint8, device=dev) for _ in range(2)]
    wr_h = [synth.router_weights(100 + l, E, H) for l in range(L)]
    x_h = [synth.prefill_hidden(500 + l, T, H, wr_h[l]) for l in range(L)]
    wr = [torch.from_numpy(a.view(np.int16)).to(dev) for a in wr_h]
    xs = [torch.from_numpy(a.view(np.int16)).to(dev) for a in x_h]
    wsb = m.moe_prefill_workspace_bytes(spec, T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream(priority=-1)  # the layer copy's CTAs are placed first
    copy_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    fws = m.moe_prefill_workspace_bytes(spec, T)

    def compute(s, buf, ev=None):
        l = s % L
        sp = main.cuda_stream
        if ev is not None:
            ev[0].record(main)
        m.moe_route(spec, xs[l], T, wr[l], None, logits, ids, wts, sp)
        if ev is not None:
            ev[1].record(main)
        m.moe_expert_ffn_prefill(spec, buf, xs[l], T, ids, wts, shared, err, ws, fws, y, sp)
        if ev is not None:
            ev[2].record(main)

    def step_overlap(s, ev=None):
        # layer s % L computes from bufs[s % 2] while layer (s+1) % L streams into the
        # other.  The copy starts with the step, beside the routing: the router's
        # FMA-bound CTAs leave room on every SM for the copy kernel's, while the
        # expert GEMMs that follow would lose HBM bandwidth to it
        main.wait_event(copy_done[s % 2])
        side.wait_event(comp_done[(s + 1) % 2])
        m.moe_layer_prefetch(spec, bank, (s + 1) % L, bufs[(s + 1) % 2], side.cuda_stream)
        copy_done[(s + 1) % 2].record(side)
        compute(s, bufs[s % 2], ev)
        comp_done[s % 2].record(main)

    def step_serial(s, ev=None):
        m.moe_layer_prefetch(spec, bank, s % L, bufs[0], main.cuda_stream)
        compute(s, bufs[0], ev)

    def timed(fn, n, with_ev):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(main)
        for s in range(n):
            fn(s, evs[s] if with_ev else None)
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b), evs

    m.moe_layer_prefetch(spec, bank, 0, bufs[0], main.cuda_stream)
    copy_done[0].record(main)
    comp_done[1].record(main)
    for s in range(args.warmup):
        step_overlap(s)
    torch.cuda.synchronize()
    rank_barrier(world)
    with ClockSampler(local_rank) as clk:
        ms, evs = timed(step_overlap, args.steps, True)
        # untimed steps after the timed ones keep the GPU busy for >= 1 s, so that
        # the clock record reflects the sustained state of this load
        soak_t0, s = time.perf_counter(), args.steps
        while time.perf_counter() - soak_t0 < 1.0:
            step_overlap(s)
            s += 1
            if s % 8 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
    ms = max_over_ranks(ms, world, dev)
    route_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ffn_ms = max_over_ranks(statistics.mean(e[1].elapsed_time(e[2]) for e in evs), world, dev)
    for s in range(min(args.warmup, 3)):
        step_serial(s)
    ms_serial, _ = timed(step_serial, args.steps, False)
    # the double buffer's parts: the layer copy alone, and the layer step with no
    # copy anywhere (its FFN time against the FFN time beside the copy)
    ms_copy, _ = timed(lambda s, ev=None: m.moe_layer_prefetch(spec, bank, (s + 1) % L, bufs[1],
                                                              main.cuda_stream),
                       args.steps, False)
    ms_nocopy, evs_nc = timed(lambda s, ev=None: compute(s, bufs[0], ev), args.steps, True)
    ffn_nocopy = statistics.mean(e[1].elapsed_time(e[2]) for e in evs_nc)
    assert int(err.cpu()[0]) == 0, "device error flag set"

    # end to end: hidden states in from pinned host memory, y back, every step.  The
    # transfers run on streams of their own (the copy engines), one step apart: step
    # s + 1's x comes in and step s's y goes out while the GPU computes step s + 1
    x_host = [torch.from_numpy(a.view(np.int16)).pin_memory() for a in x_h]
    y_host = [torch.empty((T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [torch.empty((T, H), dtype=torch.int16, device=dev) for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    x_in = [torch.cuda.Event() for _ in range(2)]
    y_out = [torch.cuda.Event() for _ in range(2)]
    lws = m.moe_prefill_workspace_bytes(spec, T)

    def x_copy(s):
        h2d.wait_event(comp_done[s % 2])  # step s - 2 has read x_dev[s % 2]
        with torch.cuda.stream(h2d):
            x_dev[s % 2].copy_(x_host[s % L], non_blocking=True)
        x_in[s % 2].record(h2d)

    def e2e_step(s, last):
        main.wait_event(copy_done[s % 2])
        side.wait_event(comp_done[(s + 1) % 2])
        m.moe_layer_prefetch(spec, bank, (s + 1) % L, bufs[(s + 1) % 2], side.cuda_stream)
        copy_done[(s + 1) % 2].record(side)
        main.wait_event(x_in[s % 2])
        main.wait_event(y_out[s % 2])  # step s - 2's y has left y_dev[s % 2]
        m.moe_layer_forward_prefill(spec, bufs[s % 2], x_dev[s % 2], T, wr[s % L], None, shared,
                                    ids, wts, err, ws, lws, y_dev[s % 2], main.cuda_stream)
        comp_done[s % 2].record(main)
        if not last:
            x_copy(s + 1)
        d2h.wait_event(comp_done[s % 2])
        with torch.cuda.stream(d2h):
            y_host[s % 2].copy_(y_dev[s % 2], non_blocking=True)
        y_out[s % 2].record(d2h)

    def timed_e2e(s0, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(main)
        h2d.wait_stream(main)
        x_copy(s0)
        for s in range(s0, s0 + n):
            e2e_step(s, s == s0 + n - 1)
        main.wait_stream(d2h)
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    m.moe_layer_prefetch(spec, bank, 0, bufs[0], main.cuda_stream)
    copy_done[0].record(main)
    comp_done[1].record(main)
    nw = min(args.warmup, 3)
    timed_e2e(0, nw)
    rank_barrier(world)
    ms_e2e = timed_e2e(nw, args.steps)
    ms_e2e = max_over_ranks(ms_e2e, world, dev)
    if rank != 0:
        return
    _, bf16_peak, peak_kind = peaks()
    sustained = None
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pp):
        sustained = json.load(open(pp)).get("bf16_tflops_sustained")
    peak = float(sustained or bf16_peak)
    flops = prefill_flops(w)
    tflops = flops / (ffn_ms * 1e-3) / 1e12
    step_ms = ms / args.steps
    tokens = args.steps * T * world
    # value: the whole layer step (route + expert FFN with the next layer's copy
    # overlapped); the roofline entry is the expert FFN call alone
    out = {
        "metric": METRIC, "value": world * flops / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": run_config(args, w, world),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": tflops / peak, "traffic": None,
                     "kernel": "prefill expert FFN (moe_expert_ffn_prefill: permute, 2 grouped "
                               "tcgen05 GEMMs, combine)",
                     "algorithmic_flops_per_launch": flops, "avg_launch_us": ffn_ms * 1e3,
                     "peak_kind": f"{peak_kind} bf16 dense, sustained"},
        "prefill_tok_s": tokens / (ms * 1e-3),
        "ffn_tflops": tflops,
        "layer_ms": {"overlapped_copy": step_ms, "serial_copy": ms_serial / args.steps,
                     "copy_alone": ms_copy / args.steps, "without_copy": ms_nocopy / args.steps,
                     "route": route_ms, "ffn": ffn_ms, "ffn_without_copy": ffn_nocopy},
        "e2e": {"value": flops * args.steps * world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                "tok_s": tokens / (ms_e2e * 1e-3),
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 4},
        "gpu_launches": 10 * args.steps,  # logits, select, 7 FFN kernels, the layer copy
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline_prefill(w, x_h, wr_h)
    print(json.dumps(out), flush=True)


def prefill_inputs(w):
    from moe_expert_offload_gb300 import synth

    L, H, E, T = w["L"], w["H"], w["E"], w["T"]
    wr_h = [synth.router_weights(100 + l, E, H) for l in range(L)]
    x_h = [synth.prefill_hidden(500 + l, T, H, wr_h[l]) for l in range(L)]
    return x_h, wr_h


class PrefillOracle:
    """The oracle on single tokens of prefill layer 0: routing and the float64 FFN
    (the token's experts dequantised per call).  Blob generation is untimed."""

    def __init__(self, w, x_h, wr_h):
        import oracle
        from moe_expert_offload_gb300 import synth

        oracle.build()
        self.o, self.synth, self.w, self.x, self.wr = oracle, synth, w, x_h[0], wr_h[0]
        self.blobs = {}
        self.fp4 = w.get("fmt", 0) - 1  # the oracle's FP4 format, or -1 for int4
        self.shared = self.make(np.random.default_rng(12345))
        self.flops_per_token = 6.0 * w["H"] * w["I"] * (w["k"] + 1)
        self.spent, self.n = 0.0, 0

    def make(self, rng):
        if self.fp4 >= 0:
            return self.synth.make_fp4_expert(rng, self.w["H"], self.w["I"], self.fp4)
        return self.synth.make_expert_bytes(rng, self.w["H"], self.w["I"])

    def token(self, t):
        o, w = self.o, self.w
        xb = self.x[t:t + 1]
        t0 = time.perf_counter()
        ids, wt = o.route_softmax_topk(o.router_logits(xb, self.wr), w["k"])
        self.spent += time.perf_counter() - t0
        for e in ids.reshape(-1):
            if int(e) not in self.blobs:
                self.blobs[int(e)] = self.make(np.random.default_rng(int(e) + 1))
        if self.fp4 >= 0:
            # the oracle's FP4 expert per routed expert, weighted sum in float64
            t0 = time.perf_counter()
            y = o.fp4_expert_forward(self.shared, w["H"], w["I"], self.fp4, xb)
            for j in range(ids.shape[1]):
                y += float(wt[0, j]) * o.fp4_expert_forward(self.blobs[int(ids[0, j])], w["H"],
                                                            w["I"], self.fp4, xb)
            self.spent += time.perf_counter() - t0
        else:
            anyb = self.blobs[int(ids[0, 0])]
            full = [self.blobs.get(e, anyb) for e in range(w["E"])]
            t0 = time.perf_counter()
            o.moe_ffn(full, w["H"], w["I"], xb, ids, wt, self.shared, w["I"])
            self.spent += time.perf_counter() - t0
        self.n += 1


def cpu_baseline_prefill(w, x_h, wr_h, budget_s=8.0):
    """The oracle on a bounded sample of the prefill layer (successive tokens until
    the budget is spent; TFLOP/s), on one thread and with its row loops on every
    host core (the same arithmetic and results)."""
    import oracle

    oracle.build()
    ncores = host_cores()

    def run(threads):
        used = oracle.set_threads(threads)
        r = PrefillOracle(w, x_h, wr_h)
        t = 0
        while r.spent < budget_s and t < w["T"]:
            r.token(t)
            t += 1
        oracle.set_threads(1)
        return (r.flops_per_token * r.n / r.spent / 1e12, used,
                f"{r.n} prefill tokens (route + float64 FFN, experts dequantised per call) in "
                f"{r.spent:.1f} s, {used} thread(s)")

    v1, _, s1 = run(1)
    out = {"value": v1, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": s1,
           "host_cores": ncores}
    if w.get("fmt", 0):
        # the oracle's FP4 expert is a single-threaded loop: no multi-core variant
        return out
    vn, used, sn = run(ncores)
    out["all_cores"] = {"value": vn, "unit": "TFLOP/s", "cores": used,
                        "kind": "oracle, row loops on every host core", "sample": sn}
    return out


# ------------------------------------------------------------- cache sweep
def sweep_traces(w):
    """Zipf routing traces int32 [steps][L][k], layer l drawn with seed 1000 + l."""
    from moe_expert_offload_gb300 import synth

    per_layer = [synth.zipf_trace(1000 + l, w["trace_steps"], w["E"], w["k"]) for l in range(w["L"])]
    return np.ascontiguousarray(np.stack(per_layer, axis=1))


def sweep_points(w):
    return [(cap, int(round(cap * w["L"] * w["E"])), bp, bh)
            for cap in w["caps"] for bp, bh in w["ratios"]]


def run_elastic(args, w, rank, world, local_rank):
    """Re-divisions of the slot pool between decode steps (moe_cache_resize), each
    bracketed by CUDA events; the decode steps between them are not timed.  The
    first shrink's tables are checked against the oracle's re-division of the same
    tables (the oracle's own time on them is the CPU baseline)."""
    import torch

    import moe_expert_offload_gb300 as m
    from moe_expert_offload_gb300 import _build

    _build.build()
    m.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    L, H, E, k, T = w["L"], w["H"], w["E"], w["k"], w["T"]
    S_hi, S_lo = w["slots"], w["slots_lo"]
    spec = spec_of(w)
    se = m.moe_expert_bytes(spec)
    n_in = args.warmup + args.steps
    xs_h, wr_h, _ = make_inputs(w, n_in)
    bank = make_bank(w, L * E + 1, 7, dev)
    cache = m.DeviceCache(spec, S_hi, w["K"], w["bp"], w["bh"], bank[:L * E], device=dev)
    plan = m.DevicePlan(T * k, w["K"], device=dev)
    xs = torch.from_numpy(xs_h.view(np.int16)).to(dev)
    wr = torch.from_numpy(wr_h.view(np.int16)).to(dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, k), dtype=torch.float32, device=dev)
    y = torch.empty((T, H), dtype=torch.float32, device=dev)
    lws = m.moe_layer_workspace_bytes(spec, T)
    lw = torch.empty(lws, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    rwb = m.moe_cache_resize_workspace_bytes(cache.c, S_lo)
    rws = torch.zeros((n_in, 2, rwb // 4), dtype=torch.int32, device=dev)
    rng = np.random.default_rng(3)

    def fill_pool():
        # a full pool: a random resident set (ts 0); the decode step after it stamps
        # the experts it routes (synchronises the stream)
        m.moe_cache_place(spec, cache.c, rng.choice(L * E, S_hi, replace=False).astype(np.int32),
                          sp)

    def decode_step(s):
        for l in range(L):
            m.moe_layer_forward(spec, cache.c, l, xs[s, l], T, wr[l], None, bank[L * E], plan.c,
                                ids, wts, lw, lws, y, sp)

    def redivide(s, ev=None):
        if ev is not None:
            ev[0].record(stream)
        m.moe_cache_resize(spec, cache.c, S_lo, rws[s, 0], rwb, sp)
        if ev is not None:
            ev[1].record(stream)
        m.moe_cache_resize(spec, cache.c, S_hi, rws[s, 1], rwb, sp)
        if ev is not None:
            ev[2].record(stream)

    for s in range(args.warmup):
        fill_pool()
        decode_step(s)
        redivide(s)
    torch.cuda.synchronize()
    # parity of one shrink against the oracle, on the tables as they stand
    import oracle

    oracle.build()
    fill_pool()
    decode_step(args.warmup)
    torch.cuda.synchronize()
    soi, ios, ts, clk = cache.host_tables()
    ost = oracle.CacheState(L * E, S_hi)
    ost.slot_of_id[:], ost.id_of_slot[:], ost.ts[:], ost.clock[:] = soi, ios, ts, clk
    t0 = time.perf_counter()
    want = oracle.cache_resize(ost, S_lo)
    cpu_s = time.perf_counter() - t0
    m.moe_cache_resize(spec, cache.c, S_lo, rws[0, 0], rwb, sp)
    torch.cuda.synchronize()
    got = cache.host_tables()
    if not (np.array_equal(got[0], ost.slot_of_id) and np.array_equal(got[1], ost.id_of_slot)
            and np.array_equal(got[2], ost.ts) and int(rws[0, 0, 1]) == want["n_moved"]):
        raise RuntimeError("elastic re-division differs from the oracle's")
    m.moe_cache_resize(spec, cache.c, S_hi, rws[0, 1], rwb, sp)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    rank_barrier(world)
    with ClockSampler(local_rank) as clk:
        for j in range(args.steps):
            s = args.warmup + j
            fill_pool()
            decode_step(s)
            redivide(s, evs[j])
        torch.cuda.synchronize()
    rank_barrier(world)
    shrink_ms = [e[0].elapsed_time(e[1]) for e in evs]
    grow_ms = [e[1].elapsed_time(e[2]) for e in evs]
    res_ms = max_over_ranks(sum(shrink_ms) + sum(grow_ms), world, dev)
    r = rws[args.warmup:].cpu().numpy()
    if np.any(r[:, :, 3] != 0):
        raise RuntimeError("re-division reported inconsistent tables")
    moved = r[:, 0, 1].astype(np.int64)
    evicted = r[:, 0, 0].astype(np.int64)

    # end to end through the public API: each re-division's counts read back to
    # pinned host memory inside the timed region
    cnt_host = torch.empty((args.steps, 2, 4), dtype=torch.int32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for j in range(args.steps):
        fill_pool()
        decode_step(args.warmup + j)
        e0.record(stream)
        m.moe_cache_resize(spec, cache.c, S_lo, rws[j, 0], rwb, sp)
        cnt_host[j, 0].copy_(rws[j, 0, :4], non_blocking=True)
        m.moe_cache_resize(spec, cache.c, S_hi, rws[j, 1], rwb, sp)
        cnt_host[j, 1].copy_(rws[j, 1, :4], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        tot += e0.elapsed_time(e1)
    ms_e2e = max_over_ranks(tot, world, dev)
    if rank != 0:
        return
    hbm, _, peak_kind = peaks()
    mv_bytes = 2.0 * float(moved.sum()) * se  # each moved blob read once and written once
    t_shrink = sum(shrink_ms) * 1e-3
    out = {
        "metric": METRIC, "value": 2 * args.steps * world / (res_ms * 1e-3),
        "unit": "re-divisions/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": run_config(args, w, world),
        "roofline": {"bound": "hbm", "achieved": mv_bytes / t_shrink / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": mv_bytes / t_shrink / 1e9 / hbm, "traffic": None,
                     "kernel": "shrink (moe_cache_resize: one-CTA plan kernel + blob move "
                               "kernel), moved blob bytes read + written per shrink",
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": mv_bytes / args.steps,
                     "avg_launch_us": 1e6 * t_shrink / args.steps},
        "elastic": {"slots": [S_hi, S_lo], "mean_evicted": float(evicted.mean()),
                    "mean_moved": float(moved.mean()),
                    "shrink_us": 1e3 * statistics.mean(shrink_ms),
                    "grow_us": 1e3 * statistics.mean(grow_ms),
                    "timing": "CUDA events around each moe_cache_resize call; decode steps "
                              "between them untimed"},
        "e2e": {"value": 2 * args.steps * world / (ms_e2e * 1e-3), "unit": "re-divisions/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 2 * 16},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu:
        out["cpu_baseline"] = {
            "value": 1.0 / cpu_s, "unit": "re-divisions/s", "cores": 1, "kind": "oracle",
            "sample": f"one shrink {S_hi} -> {S_lo} of the GPU's own tables after a fill and "
                      f"a decode step (tables only; the oracle has no slot pool), single thread, "
                      f"{cpu_s * 1e3:.2f} ms", "host_cores": host_cores()}
    print(json.dumps(out), flush=True)


def run_sweep(args, w, rank, world, local_rank):
    """Config 5: every (capacity, B_P/B_H) point runs the 2048-step x 40-layer trace
    through moe_cache_step from a reset cache; one CUDA graph per 64 trace steps.
    Each call's counts land in their own row of a device array (the plan struct of
    call i points there), so the statistics cost no extra work in the timed region."""
    import torch

    import moe_expert_offload_gb300 as m
    from moe_expert_offload_gb300 import _build

    _build.build()
    m.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    L, E, k, K, n = w["L"], w["E"], w["k"], w["K"], w["trace_steps"]
    spec = spec_of(w)
    tr_h = sweep_traces(w)                                   # [n][L][k]
    tr = torch.from_numpy(tr_h).to(dev)
    calls = n * L
    base = m.DevicePlan(k, K, device=dev)
    stats = torch.zeros((calls, 8), dtype=torch.int32, device=dev)
    b = base.buf
    bp_ = [m._ptr(b[x]) for x in m.DevicePlan.NAMES]
    plans = [m.MoePlan(k, *bp_, m._ptr(base.victims), stats.data_ptr() + 32 * i,
                       m._ptr(base.err)) for i in range(calls)]
    tr_ptr = tr.data_ptr()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    chunk = 64

    def capture(cache):
        graphs = []
        for s0 in range(0, n, chunk):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                sh = torch.cuda.current_stream().cuda_stream
                for st in range(s0, min(n, s0 + chunk)):
                    for l in range(L):
                        i = st * L + l
                        m.moe_cache_step(spec, cache.c, l, tr_ptr + 4 * k * i, 1, plans[i], 0, sh)
            graphs.append(g)
        return graphs

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rows, head = [], None
    with ClockSampler(local_rank) as clk:
        for cap, S, bp, bh in sweep_points(w):
            cache = m.DeviceCache(spec, S, K, bp, bh, bank=None, device=dev, with_pool=False)
            graphs = capture(cache)
            for rep in range(2):          # a warm pass, then the timed pass, each from reset
                m.moe_cache_reset(spec, cache.c, sp)
                torch.cuda.synchronize()
                e0.record(stream)
                for g in graphs:
                    g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            st = stats.cpu().numpy().astype(np.int64)
            if int(base.err.cpu()[0]) != 0:
                raise RuntimeError("control step flagged an error in the sweep")
            row = {"capacity": cap, "slots": S, "bp_bh": f"{bp / 1000:.1f}/{bh / 1000:.1f}",
                   "miss_rate": float(st[:, 2].sum() / max(st[:, 0].sum(), 1)),
                   "mean_uniq": float(st[:, 0].mean()), "mean_hits": float(st[:, 1].mean()),
                   "mean_F": float(st[:, 4].mean()), "mean_C": float(st[:, 5].mean()),
                   "mean_q": float(st[:, 3].mean()),
                   "control_us_per_layer": 1e3 * ms / calls}
            rows.append(row)
            if cap == 0.25 and (bp, bh) == (52700, 77300):
                head = (row, ms, cache, graphs)
            else:
                del graphs
            torch.cuda.synchronize()
    row, ms, cache, graphs = head
    ms = max_over_ranks(ms, world, dev)

    # end to end at the headline point: each 64-step chunk of the trace is copied
    # in from pinned host memory and its counts copied back, inside the timed region
    tr_host = torch.from_numpy(tr_h).pin_memory()
    st_host = torch.empty((calls, 8), dtype=torch.int32).pin_memory()
    m.moe_cache_reset(spec, cache.c, sp)
    torch.cuda.synchronize()
    e0.record(stream)
    for j, g in enumerate(graphs):
        s0, s1 = j * chunk, min(n, (j + 1) * chunk)
        tr[s0:s1].copy_(tr_host[s0:s1], non_blocking=True)
        g.replay()
        st_host[s0 * L:s1 * L].copy_(stats[s0 * L:s1 * L], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world, dev)
    policies = policy_rows(m, spec, w, dev, plans, stats, base)
    if rank != 0:
        return
    hbm, _, peak_kind = peaks()
    t_call = ms * 1e-3 / calls
    scan = row["slots"] * 8 + (k + K) * 16            # ts + id_of_slot scan, plan rows
    out = {
        "metric": METRIC, "value": world * calls / (ms * 1e-3), "unit": "layer-steps/s",
        "n_gpus": world, "steps": n, "warmup": 1, "ms_per_step": ms / n,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": run_config(args, w, world),
        "roofline": {"bound": "hbm", "achieved": scan / t_call / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": scan / t_call / 1e9 / hbm, "traffic": None,
                     "kernel": "control step (one CTA, latency-bound)", "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": scan, "avg_launch_us": t_call * 1e6},
        "sweep": rows,
        "policies": policies,
        "e2e": {"value": world * calls / (ms_e2e * 1e-3), "unit": "layer-steps/s",
                "h2d_bytes_per_step": L * k * 4, "d2h_bytes_per_step": L * 32},
        "gpu_launches": calls,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline_sweep(w, tr_h)
    print(json.dumps(out), flush=True)


POLICIES = ("shared_lru", "layer_lru", "static_hot", "static_layers")


def policy_rows(m, spec, w, dev, plans, stats, base):
    """Miss rate of each replacement policy at each capacity, replayed on the
    same traces (stationary Zipf, and the same recipe with the popular experts
    redrawn every `phase_steps` steps) through moe_cache_step on the device:
    shared LRU, per-layer LRU (floor(S/L) slots per layer), static hot set
    (the S most routed pairs of the replayed trace, placed once) and static
    whole layers.  B_P/B_H 52.7/77.3 GB/s for the LRU policies; the static
    ones never fill.  Plain stream launches (not timed)."""
    import torch

    from moe_expert_offload_gb300 import placement, synth

    L, E, k, K, n = w["L"], w["E"], w["k"], w["K"], w["trace_steps"]
    sp = torch.cuda.current_stream().cuda_stream
    kinds = {"shared_lru": m.POLICY_SHARED_LRU, "layer_lru": m.POLICY_LAYER_LRU}
    sets = [("stationary", sweep_traces(w)),
            (f"phased_{w['phase_steps']}", np.ascontiguousarray(np.stack(
                [synth.zipf_trace(1000 + l, n, E, k, phase_steps=w["phase_steps"])
                 for l in range(L)], axis=1)))]
    out = []
    for tname, tr_h in sets:
        tr = torch.from_numpy(tr_h).to(dev)
        ptr = tr.data_ptr()
        for cap in w["caps"]:
            S = int(round(cap * L * E))
            for pol in POLICIES:
                cache = m.DeviceCache(spec, S, K, 52700, 77300, bank=None, device=dev,
                                      with_pool=False, policy=kinds.get(pol, m.POLICY_STATIC))
                if pol == "static_hot":
                    m.moe_cache_place(spec, cache.c, placement.hot_placement(tr_h, E, S), sp)
                elif pol == "static_layers":
                    m.moe_cache_place(spec, cache.c, placement.layer_placement(L, E, S), sp)
                else:
                    m.moe_cache_reset(spec, cache.c, sp)
                for i in range(n * L):
                    m.moe_cache_step(spec, cache.c, i % L, ptr + 4 * k * i, 1, plans[i], 0, sp)
                torch.cuda.synchronize()
                if int(base.err.cpu()[0]) != 0:
                    raise RuntimeError("control step flagged an error in the policy replay")
                st = stats.cpu().numpy().astype(np.int64)
                out.append({"trace": tname, "capacity": cap, "slots": S, "policy": pol,
                            "miss_rate": float(st[:, 2].sum() / max(st[:, 0].sum(), 1)),
                            "mean_F": float(st[:, 4].mean()), "mean_C": float(st[:, 5].mean())})
                del cache
    return out


def cpu_baseline_sweep(w, tr_h, budget_s=10.0):
    """The oracle control step (single thread) at the headline sweep point, on the
    first trace steps until the budget is spent; layer-steps/s."""
    import oracle

    oracle.build()
    L, E, K = w["L"], w["E"], w["K"]
    state = oracle.CacheState(L * E, int(round(0.25 * L * E)))
    spent, calls, s = 0.0, 0, 0
    while s < tr_h.shape[0] and (spent < budget_s or s == 0):
        for l in range(L):
            t0 = time.perf_counter()
            oracle.cache_step(state, E, l, tr_h[s, l:l + 1], K, 52700, 77300)
            spent += time.perf_counter() - t0
            calls += 1
        s += 1
    return {"value": calls / spent, "unit": "layer-steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{s} trace steps x {L} layers at capacity 25%, B_P/B_H 52.7/77.3 in "
                      f"{spent:.1f} s, single thread (each control step depends on the last: "
                      "no multi-core variant)",
            "host_cores": host_cores()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="qwen_decode", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu", action="store_true", help="skip the timed CPU oracle baseline")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small cases for profiling)")
    ap.add_argument("--adaptive-q", action="store_true",
                    help="decode: use B_P / B_H measured on the device instead of the configured "
                         "rates")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the experts per layer (small cases for profiling; same expert "
                         "shape, slot count scaled in proportion)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = dict(WORKLOADS[args.workload])
    if args.layers or args.experts:
        L0, E0 = w["L"], w["E"]
        w["L"] = args.layers or L0
        w["E"] = args.experts or E0
        if "slots" in w:
            w["slots"] = max(2 * w["k"], round(w["slots"] * w["L"] * w["E"] / (L0 * E0)))
        w["desc"] += f" [profiling case: {w['L']} layers x {w['E']} experts]"
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return
    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if w.get("prefill"):
        run_prefill(args, w, rank, world, local_rank)
    elif w.get("sweep"):
        run_sweep(args, w, rank, world, local_rank)
    elif w.get("elastic"):
        run_elastic(args, w, rank, world, local_rank)
    else:
        run_gpu(args, w, rank, world, local_rank)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
