"""Benchmark of the MoE layer local data path on one GB300 (or N replicas).

Default workload: fine-grained-bf16 (T=4096 tokens, D=2048, H=1408, E=64
experts, top-6, softmax renormalised; bf16 activations and weights, fp32
accumulation), seeded synthetic inputs from moe_inputs.py, resident in HBM.
``--workload NAME`` times another workload of moe_inputs.WORKLOADS instead
(``--workload all``: one line per workload, in the specification's order).

One step = router top-k -> permute -> grouped SwiGLU (GEMM1 + gate, GEMM2)
-> weighted combine, issued as one moe_layer_forward call of the C ABI (the
layer call a user makes; every intermediate in its workspace).  A second loop
times the four step calls one by one for the per-call breakdown.  The line
reports tokens/s (value: T tokens per step, each routed to
k experts), the dominant kernel against its roof (roofline: the grouped
SwiGLU on the tensor cores, on HBM for the masked decode layout, on the FP32
ALUs for the fp32 workload), permute and combine GB/s (breakdown), an
end-to-end figure with host buffers through the host pipeline, every step
copying its input in and its output out (e2e; the one-call-at-a-time figure
beside it), and the CPU oracle timed on a bounded sample (cpu_baseline).

Multi-GPU: the path does not exchange data; each rank runs an independent
replica on its own GPU ("scaling": "weak") and value = all ranks' tokens / the
slowest rank's time.

--impl reference times the CPU oracle (the reference arm) on
the same workload and prints the same kind of line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import dataclasses
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

WORKLOAD = "fine-grained-bf16"   # the default line
METRIC = "MoE layer routed tokens/s"
UNIT = "tokens/s"
L2_BYTES = 129 * 1000 * 1000        # GB300 L2 (126 MiB)
VALUE_COUNTS = ("tokens: T per step (every token routed to k experts; the expert rows per "
                "step are T*k)")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def algorithmic(w, R=None, touched=None):
    """Algorithmic work of one step: R routed expert rows (T*k unless given),
    `touched` experts with at least one row (all E unless given)."""
    R = w.T * w.k if R is None else R
    touched = w.E if touched is None else touched
    b = 2 if w.dtype == "bf16" else 4
    return dict(
        ffn_flops=6.0 * R * w.D * w.H,
        permute_bytes=float(w.T * w.D * b + R * w.D * b),
        # the method's combine bytes: y rows read once, out written once, the
        # row index and weight of every slot
        combine_bytes=float(R * w.D * b + w.T * w.D * b + R * 8),
        # what the combine moves here: y_perm is fp16 (bf16 layers) or fp32
        combine_bytes_moved=float(R * w.D * b + w.T * w.D * b + R * 8),
        # the grouped call when it streams weights (masked decode): the touched
        # experts' w1, w3, w2 once, x_perm rows read, h written and read, y written
        grouped_bytes=float(touched * 3 * w.D * w.H * b + R * w.D * b + 2 * R * w.H * b
                            + R * w.D * b),
        weight_bytes=float(w.E * 3 * w.D * w.H * b),
    )


def workload_config(moe, w):
    """The C ABI configuration of a workload (its layout, router and dtype)."""
    return moe.Config(T=w.T, D=w.D, H_local=w.H, E=w.E, k=w.k,
                      dtype=moe.MOE_F32 if w.dtype == "f32" else moe.MOE_BF16,
                      score=moe.MOE_SCORE_SOFTMAX if w.score == "softmax" else moe.MOE_SCORE_SIGMOID,
                      renorm=int(w.renorm),
                      layout=moe.MOE_LAYOUT_MASKED if w.layout == "masked"
                      else moe.MOE_LAYOUT_CONTIGUOUS,
                      align_m=128, capacity=w.T if w.layout == "masked" else 0,
                      n_group=w.n_group, topk_group=w.topk_group)


def needs_l2_flush(w):
    """Whether one step's inputs fit in L2 (then every timed step is preceded
    by an L2 flush and timed on its own)."""
    return algorithmic(w)["weight_bytes"] < 2 * L2_BYTES


def l2_note(w):
    if needs_l2_flush(w):
        return ("L2 flushed (256 MB write) before every timed step; each step timed between "
                "its own CUDA events")
    gb = algorithmic(w)["weight_bytes"] / 1e9
    return f"inputs larger than L2: {gb:.1f} GB of expert weights per step, no flush"


def workload_data_note(w):
    return (f"synthetic (seeded N(0,1) activations, N(0,{w.wstd}) weights"
            + (", Zipf(1.2)-shaped router bias" if w.zipf_s else "") + ")")


def router_note(w):
    r = f"{w.score}, renormalised over top-k" if w.renorm else f"{w.score}, not renormalised"
    if w.n_group:
        r += f", {w.topk_group} of {w.n_group} groups"
    return r


def layout_note(w):
    return ("masked, capacity = T" if w.layout == "masked" else "contiguous, align_m=128")


def max_over_ranks(value_ms, dev):
    """The slowest rank's time: every rank gets the maximum over the process
    group (the value itself when there is no group or only one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value_ms
    t = torch.tensor([float(value_ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_tokens_per_s(world, tokens_per_rank, ms_per_step):
    """Whole-job throughput of `world` replicas that each route tokens_per_rank
    tokens per step, over the slowest rank's step time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                sm_max_mhz=2070.0, source="fallback")


# grouped SwiGLU kernel that dominates each workload's step, and its sources
GROUPED_KERNEL = {
    "tiny-fp32": ("grouped_f32_kernel (fp32 SIMT FFMA, GEMM1 + SwiGLU and GEMM2)",
                  ("grouped_f32.cu", "common.cuh")),
    "decode-masked": ("grouped_tc_kernel (tcgen05, one CTA per 128x256 tile, masked tile table)",
                      ("grouped_tc.cu", "common.cuh")),
}
PAIR_KERNEL = ("grouped_pair_kernel (tcgen05 cta_group::2, GEMM1 + SwiGLU, GEMM2)",
               ("grouped_tc2.cu", "common.cuh"))


def grouped_kernel(workload):
    return GROUPED_KERNEL.get(workload, PAIR_KERNEL)


def kernel_source_hash(workload=WORKLOAD):
    h = hashlib.sha256()
    for f in grouped_kernel(workload)[1]:
        h.update(open(os.path.join(ROOT, "routing_grouped_gemm_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload=WORKLOAD):
    """DRAM bytes per call of the grouped SwiGLU from a committed ncu summary
    (profiles/grouped_swiglu_traffic.json, one entry per workload), only if it
    was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "grouped_swiglu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    entry = d.get(workload) if isinstance(d, dict) else None
    if not isinstance(entry, dict):
        return None
    if entry.get("kernel_source_hash") != kernel_source_hash(workload):
        return None
    return entry.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_tokens_per_s(x, wg, bias, expert, w, n_tokens, seed=0, nthreads=None):
    """Time the oracle's whole layer (router + per-token experts) on a sample
    of n_tokens tokens.  x, wg: host arrays; bias: host fp64 or None;
    expert(e) -> host (w1[e], w3[e], w2[e]).  Only the experts the sample
    reaches are fetched, before the timed part."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    toks = np.sort(rng.choice(w.T, size=n_tokens, replace=False)).astype(np.int32)
    nth = nthreads or oracle.default_threads()
    score = oracle.SOFTMAX if w.score == "softmax" else oracle.SIGMOID
    xs = x[toks]
    _, _, idx, _, _ = oracle.route(xs, wg, bias, w.k, score, w.renorm, nthreads=nth,
                                   n_group=w.n_group, topk_group=w.topk_group)
    used = sorted(set(int(e) for e in np.unique(idx)))
    w1s, w3s, w2s = [None] * w.E, [None] * w.E, [None] * w.E
    for e in used:
        w1s[e], w3s[e], w2s[e] = expert(e)
    t0 = time.perf_counter()
    _, _, idx, wts, _ = oracle.route(xs, wg, bias, w.k, score, w.renorm, nthreads=nth,
                                     n_group=w.n_group, topk_group=w.topk_group)
    oracle.moe_tokens(np.arange(n_tokens), xs, w1s, w3s, w2s, idx, wts,
                      round_h=(w.dtype == "bf16"), nthreads=nth)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt, nth


def host_router_inputs(inp):
    """Host copies of x, W_g and the bias (fp64) in the oracle's conventions."""
    import numpy as np
    import moe_inputs
    H = moe_inputs.host_array
    bias = None if inp.bias is None else inp.bias.detach().cpu().numpy().astype(np.float64)
    return H(inp.x), H(inp.wg), bias


def host_expert(inp):
    """expert(e) -> host copies of the GPU's w1[e], w3[e], w2[e]."""
    import moe_inputs
    H = moe_inputs.host_array
    return lambda e: (H(inp.w1[e]), H(inp.w3[e]), H(inp.w2[e]))


def cpu_baseline(inp, w, seconds, seed=7):
    """The oracle as it stands on a token sample sized to about `seconds`."""
    x, wg, bias = host_router_inputs(inp)
    expert = host_expert(inp)
    tps, _, nth = oracle_tokens_per_s(x, wg, bias, expert, w, min(w.T, 16), seed=99)
    n = int(max(16, min(w.T, tps * seconds)))
    tps, dt, nth = oracle_tokens_per_s(x, wg, bias, expert, w, n, seed=seed)
    # the same on one thread, on a sample of about a second
    n1 = int(max(4, min(w.T, tps / nth)))
    tps1, dt1, _ = oracle_tokens_per_s(x, wg, bias, expert, w, n1, seed=seed + 1, nthreads=1)
    return {"value": tps, "unit": UNIT, "cores": nth, "kind": "oracle",
            "sample": f"{n} sampled tokens of the {w.name} batch, router + per-token experts in "
                      f"fp64 ({dt:.1f} s)",
            "single_thread": {"value": tps1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} sampled tokens ({dt1:.1f} s)"},
            "cpu": cpu_model()}


def cpu_model():
    try:
        for l in open("/proc/cpuinfo"):
            if l.lower().startswith(("model name", "cpu part")):
                return l.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_reference(args):
    """Reference arm: the CPU oracle as it stands, on the host cores, on a
    bounded token sample of the workload per step."""
    import torch
    import moe_inputs
    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = getattr(args, "workload", None) or WORKLOAD
    if name == "all":
        name = WORKLOAD
    w = moe_inputs.WORKLOADS[name]
    inp = moe_inputs.make_inputs(w, device="cpu", seed=0, weights=False)
    x, wg, bias = host_router_inputs(inp)
    cache = {}

    def expert(e):
        # the weights of the experts the samples reach, drawn on the host
        # with the workload's distribution
        if e not in cache:
            cache[e] = tuple(moe_inputs.host_array(t) for t in moe_inputs.expert_weights(w, e))
        return cache[e]

    # calibrate so the whole run stays within about two minutes
    tps, _, nth = oracle_tokens_per_s(x, wg, bias, expert, w, min(w.T, 16), seed=99)
    budget_s = 120.0
    per_step = max(1, min(w.T, int(tps * budget_s / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        oracle_tokens_per_s(x, wg, bias, expert, w, per_step, seed=i)
    times = []
    for i in range(args.steps):
        _, dt, _ = oracle_tokens_per_s(x, wg, bias, expert, w, per_step, seed=1000 + i)
        times.append(dt)
    total = sum(times)
    value = per_step * args.steps / total
    sample = (f"{per_step} sampled tokens per step of the {name} batch of {w.T} "
              f"(router + per-token experts in fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        # measured: the mean time of one timed step, i.e. of `per_step` tokens
        "ms_per_step": 1e3 * total / args.steps,
        "tokens_per_step": per_step, "value_counts": VALUE_COUNTS,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": name, "T": w.T, "D": w.D, "H": w.H, "E": w.E, "k": w.k,
                   "parallelism": "replicas" if world > 1 else "single", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": nth, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_e2e(moe, cfg, inp, out, stream, dev, world, args):
    """End to end through host buffers: every step copies its pinned x in and
    its output out.  The headline figure runs the steps through the host
    pipeline (moe_host_pipeline: each step's copies overlap the neighbouring
    steps' compute, as a serving loop would run them); the single-call figure
    through moe_layer_forward_host, one step at a time on one stream."""
    import torch
    w = inp.w
    e_steps = args.steps  # the same number of timed steps as the device-resident loop
    x_host = inp.x.cpu().pin_memory()
    out_host = torch.empty((w.T, w.D), dtype=inp.x.dtype).pin_memory()
    eb = inp.x.element_size()

    # single call: copy in, layer, copy out, all on `stream`
    lws = moe.alloc_workspace(cfg, host=True, device=dev)

    def single_step():
        moe.moe_layer_forward_host(cfg, x_host, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out_host,
                                   lws, stream)

    for _ in range(max(3, args.warmup)):
        single_step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        single_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    single_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)
    st = moe.moe_get_device_status(lws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after e2e: {moe.status_string(st)}")
    del lws

    # pipelined: the timed region opens on an idle device and closes after
    # the pipeline's sync (every output copy done)
    pipe = moe.HostPipeline(cfg, device=dev)
    try:
        def piped_step():
            pipe.submit(x_host, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out_host, stream)

        for _ in range(max(3, args.warmup)):
            piped_step()
        pipe.sync()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(e_steps):
            piped_step()
        pipe.sync()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        piped_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)
    finally:
        pipe.close()
    return {"value": replica_tokens_per_s(world, w.T, piped_ms), "unit": UNIT,
            "h2d_bytes_per_step": int(x_host.numel() * eb),
            "d2h_bytes_per_step": int(out_host.numel() * eb),
            "ms_per_step": piped_ms, "steps": e_steps,
            "api": "moe_host_pipeline (C ABI, depth 2): every step copies its pinned x in and its "
                   "output out on the pipeline's copy streams, overlapping the neighbouring steps' "
                   "compute",
            "single_call": {"value": replica_tokens_per_s(world, w.T, single_ms), "unit": UNIT,
                            "ms_per_step": single_ms,
                            "api": "moe_layer_forward_host (C ABI): copy in, layer, copy out on one "
                                   "stream, one step at a time"}}


def run_fused(moe, cfg, inp, stream, dev, args):
    """The same step through moe_layer_forward_fused: the combine fused into
    GEMM2's epilogue (fp32 atomic adds into a [T, D] accumulator, then one
    rounding kernel), so y_perm is never written or read back."""
    import torch
    w = inp.w
    lws = moe.alloc_workspace(cfg, layer=True, device=dev)
    out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)

    def step():
        moe.moe_layer_forward_fused(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out,
                                    lws, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    n = max(20, args.steps // 4)
    n0 = moe.kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    launches = (moe.kernel_launches() - n0) / n
    st = moe.moe_get_device_status(lws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after the fused leg: {moe.status_string(st)}")
    ms = e0.elapsed_time(e1) / n
    return {"api": "moe_layer_forward_fused (C ABI): combine in GEMM2's epilogue, fp32 atomics",
            "ms_per_step": ms, "value": w.T / (ms * 1e-3), "unit": UNIT,
            "launches_per_step": launches, "deterministic": False}


def run_gather(moe, cfg, inp, stream, dev, args):
    """The dispatch fused into GEMM1's operand load: moe_layer_forward_gather
    against moe_layer_forward in the same loop shape, and the step through
    the step calls (route, permute_index, grouped_swiglu_gather, combine)
    with CUDA events between them.  Bitwise the same output."""
    import torch
    w = inp.w
    lws = moe.alloc_workspace(cfg, layer=True, device=dev)
    out = torch.empty((w.T, w.D), dtype=inp.x.dtype, device=dev)
    views = moe.layer_views(cfg, lws)

    def layer_gather():
        moe.moe_layer_forward_gather(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out,
                                     lws, stream)

    def layer_copy():
        moe.moe_layer_forward(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, lws,
                              stream)

    n = max(20, args.steps // 2)
    res = {}
    for _ in range(2):  # two rounds, alternating, so drift hits both alike
        for name, fn in (("layer_forward_ms", layer_copy), ("layer_forward_gather_ms", layer_gather)):
            for _ in range(3):
                fn()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            res.setdefault(name, []).append(e0.elapsed_time(e1) / n)
    st = moe.moe_get_device_status(lws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after the gather leg: {moe.status_string(st)}")
    # per-call breakdown of the gather step
    v = views
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        moe.moe_route_topk(cfg, inp.x, inp.wg, inp.bias, None, v["topk_idx"], v["topk_w"], lws, stream)
        ev[i][1].record(stream)
        moe.moe_permute_index(cfg, v["topk_idx"], v["tokens_per_expert"], v["seg_offsets"],
                              v["row_of"], v["token_of_row"], lws, stream)
        ev[i][2].record(stream)
        moe.moe_grouped_swiglu_gather(cfg, inp.x, v["token_of_row"], v["seg_offsets"],
                                      v["tokens_per_expert"], inp.w1, inp.w3, inp.w2, v["h"],
                                      v["y_perm"], lws, stream)
        ev[i][3].record(stream)
        moe.moe_unpermute_combine(cfg, v["y_perm"], v["row_of"], v["topk_w"], out, lws, stream)
        ev[i][4].record(stream)
    torch.cuda.synchronize(dev)
    parts = [sum(e[j].elapsed_time(e[j + 1]) for e in ev) / n for j in range(4)]
    st = moe.moe_get_device_status(lws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after the gather breakdown: {moe.status_string(st)}")
    lf, lg = min(res["layer_forward_ms"]), min(res["layer_forward_gather_ms"])
    return {"api": "moe_layer_forward_gather (C ABI): GEMM1 reads x[token_of_row[r]], no x_perm",
            "layer_forward_ms": lf, "layer_forward_gather_ms": lg,
            "value": w.T / (lg * 1e-3), "unit": UNIT, "speedup": lf / lg,
            "breakdown_ms": {"route": parts[0], "permute_index": parts[1],
                             "grouped_swiglu_gather": parts[2], "combine": parts[3]},
            "rounds_ms": res}


def run_fp8(moe, cfg, inp, stream, dev, args, peaks):
    """The FP8 variant of the same step: moe_layer_forward_fp8 (e4m3 dispatch,
    GEMM1 on e4m3 codes with per-row scales, GEMM2 in bf16), the weights
    quantised once before timing, as in inference.  Also times the grouped
    call alone.  Its FLOPs are 4 R D H in e4m3 and 2 R D H in bf16; the
    peak fraction compares the time both would take at the measured bf16
    peak and twice it for e4m3 (the nominal dense fp8 : bf16 ratio)."""
    import torch
    w = inp.w
    w1q, w1s = moe.quantize_weights_fp8(inp.w1)
    w3q, w3s = moe.quantize_weights_fp8(inp.w3)
    lws = moe.alloc_workspace(cfg, layer=True, device=dev)
    out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    views = moe.layer_views(cfg, lws)

    def step():
        moe.moe_layer_forward_fp8(cfg, inp.x, inp.wg, inp.bias, w1q, w1s, w3q, w3s, inp.w2, out,
                                  lws, stream)

    def grouped():
        moe.moe_grouped_swiglu_fp8(cfg, views["x_perm_q"], views["x_scale"], views["seg_offsets"],
                                   views["tokens_per_expert"], w1q, w1s, w3q, w3s, inp.w2,
                                   views["h"], views["y_perm"], lws, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    res = {}
    for name, fn in (("step", step), ("grouped", grouped)):
        n = max(20, args.steps // 4)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = e0.elapsed_time(e1) / n
    st = moe.moe_get_device_status(lws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after the fp8 leg: {moe.status_string(st)}")
    R = w.T * w.k
    f8_flops, bf_flops = 4.0 * R * w.D * w.H, 2.0 * R * w.D * w.H
    ideal_ms = (f8_flops / (2 * peaks["bf16_tflops"] * 1e12) + bf_flops / (peaks["bf16_tflops"] * 1e12)) * 1e3
    return {"api": "moe_layer_forward_fp8 (C ABI), weights quantised once",
            "dtype": "e4m3 GEMM1 operands (one fp32 scale per row), bf16 GEMM2",
            "ms_per_step": res["step"], "value": w.T / (res["step"] * 1e-3), "unit": UNIT,
            "grouped_ms": res["grouped"],
            "grouped_tflops": (f8_flops + bf_flops) / (res["grouped"] * 1e-3) / 1e12,
            "grouped_frac_of_peak": ideal_ms / res["grouped"],
            "peak_note": "e4m3 at 2x the measured bf16 burst peak, bf16 at the measured peak"}


def run_backward(moe, cfg, inp, stream, dev, args, peaks):
    """The training step's backward on the same batch: moe_layer_forward_train,
    then moe_layer_backward (all gradients), timed with CUDA events on the
    launching stream.  The expert GEMMs of the backward do 12 R D H FLOPs
    (dgrad 6 R D H, wgrad 6 R D H)."""
    import torch
    w = inp.w
    tws = moe.alloc_workspace(cfg, train=True, device=dev)
    out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
    g = torch.Generator(device=dev).manual_seed(1)
    dout = torch.randn((w.T, w.D), generator=g, device=dev).to(torch.bfloat16)
    dx = torch.empty_like(out)
    dwg = torch.empty((w.E, w.D), device=dev)
    dbias = torch.empty((w.E,), device=dev)
    dw1 = torch.empty((w.E, w.H, w.D), device=dev)
    dw3 = torch.empty((w.E, w.H, w.D), device=dev)
    dw2 = torch.empty((w.E, w.D, w.H), device=dev)

    def fwd():
        moe.moe_layer_forward_train(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, tws,
                                    stream)

    def bwd():
        moe.moe_layer_backward(cfg, inp.x, inp.wg, inp.w1, inp.w3, inp.w2, dout, dx, dwg, dbias,
                               dw1, dw3, dw2, tws, stream)

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    st = moe.moe_get_device_status(tws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after backward warm-up: {moe.status_string(st)}")
    n = max(10, args.steps // 8)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    n0 = moe.kernel_launches()
    for i in range(n):
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    launches = (moe.kernel_launches() - n0) / n
    torch.cuda.synchronize(dev)
    st = moe.moe_get_device_status(tws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after backward: {moe.status_string(st)}")
    # the same backward with bf16 expert weight gradients
    b1, b3, b2 = (torch.empty(t.shape, dtype=torch.bfloat16, device=dev) for t in (dw1, dw3, dw2))

    def bwd16():
        moe.moe_layer_backward(cfg, inp.x, inp.wg, inp.w1, inp.w3, inp.w2, dout, dx, dwg, dbias,
                               b1, b3, b2, tws, stream)

    for _ in range(3):
        bwd16()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        bwd16()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    b16_ms = e0.elapsed_time(e1) / n
    f_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    b_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / n
    flops = 12.0 * w.T * w.k * w.D * w.H
    tf = flops / (b_ms * 1e-3) / 1e12
    fl32 = backward_floors(w, peaks, 4)
    fl16 = backward_floors(w, peaks, 2)
    del tws, dw1, dw3, dw2, b1, b3, b2
    return {"api": "moe_layer_forward_train + moe_layer_backward (dx, dwg, dbias, dw1, dw3, dw2)",
            "forward_train_ms": f_ms, "backward_ms": b_ms,
            "training_step_tokens_per_s": w.T / ((f_ms + b_ms) * 1e-3),
            "backward_expert_flops": flops, "backward_tflops": tf,
            "backward_frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "backward_floor_ms": fl32["total_floor_ms"],
            "backward_frac_of_floor": fl32["total_floor_ms"] / b_ms,
            "backward_bf16_weight_grads_ms": b16_ms,
            "backward_bf16_weight_grads_tflops": flops / (b16_ms * 1e-3) / 1e12,
            "backward_bf16_weight_grads_floor_ms": fl16["total_floor_ms"],
            "backward_bf16_weight_grads_frac_of_floor": fl16["total_floor_ms"] / b16_ms,
            "floor_note": "per kernel the larger of its FLOPs at the bf16 burst peak and its "
                          "algorithmic bytes at the copy rate, summed; with fp32 weight "
                          "gradients all four expert GEMMs are byte-bound",
            "floors_by_kernel": {k: {"bound": v["bound"],
                                     "floor_ms": max(v["compute_floor_ms"], v["hbm_floor_ms"])}
                                 for k, v in fl32.items() if k != "total_floor_ms"},
            "launches_per_forward_and_backward": launches}


def backward_floors(w, peaks, wgrad_bytes=4):
    """Lower bounds of the layer backward, kernel by kernel: each kernel's
    FLOPs at the bf16 tensor peak or its algorithmic bytes at the copy rate,
    whichever is larger, summed over the kernels.  Bytes count the valid rows
    (R = T k) once per read or write of each operand; dx_perm and the router's
    dense dx part are fp32, the expert weight gradients `wgrad_bytes` wide."""
    R, T, D, H, E = w.T * w.k, w.T, w.D, w.H, w.E
    b = 2
    dense = w.score == "softmax" and not w.renorm   # dl nonzero on every expert
    parts = {
        # dout read, y_perm (fp16) read, gy written, slot index and weight, dw
        "combine_bwd": (0.0, T * D * b + 2 * R * D * b + R * 12),
        # gy, w2, the saved gate/up read; dg/du written
        "dgrad2_swiglu_bwd": (2.0 * R * D * H, R * D * b + E * D * H * b + 2 * R * 2 * H * b),
        # dg/du, w1 and w3 read; dx_perm written (fp32)
        "dgrad1": (4.0 * R * D * H, R * 2 * H * b + 2 * E * H * D * b + R * D * 4),
        # gy and h read; dw2 written
        "wgrad2": (2.0 * R * D * H, R * D * b + R * H * b + E * D * H * wgrad_bytes),
        # dg/du and x_perm read; dw1 and dw3 written
        "wgrad13": (4.0 * R * D * H, R * 2 * H * b + R * D * b + 2 * E * H * D * wgrad_bytes),
        # logits, dw read, dl written; dW_g = dl^T x (x read once); where dl is
        # dense (softmax without renorm) the dx part dl wg is a GEMM (fp32 out)
        "router_bwd": (4.0 * T * E * D, T * E * 4 * 2 + R * 4 + T * D * b + E * D * 4 + E * D * b
                       + T * D * 4) if dense else
                      (2.0 * R * D, T * E * 4 * 2 + R * 4 + T * D * b + E * D * 4),
        # dx_perm (fp32) and the router's dx part read (dense: the fp32 GEMM
        # output; else wg and each slot's dl), dx written
        "dispatch_bwd": (0.0, R * D * 4 + R * 4 + T * D * 4 + T * D * b) if dense else
                        (2.0 * R * D, R * D * 4 + R * 4 + E * D * b + R * 4 + T * D * b),
    }
    out = {}
    for name, (flops, nbytes) in parts.items():
        c = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
        m = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e3
        out[name] = {"flops": flops, "bytes": float(nbytes), "compute_floor_ms": c,
                     "hbm_floor_ms": m, "bound": "hbm" if m > c else "tensor"}
    out["total_floor_ms"] = sum(max(v["compute_floor_ms"], v["hbm_floor_ms"])
                                for v in out.values())
    return out


def floors(w, R, touched, peaks):
    """The grouped call's two lower bounds in ms: its FLOPs at the bf16 tensor
    peak and its algorithmic bytes at the copy rate.  The larger one is the
    roof that binds (the classic roofline: attainable = min(peak, intensity x
    bandwidth))."""
    alg = algorithmic(w, R, touched)
    return (alg["ffn_flops"] / (peaks["bf16_tflops"] * 1e12) * 1e3,
            alg["grouped_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e3)


def grouped_bound(w, R, touched, peaks):
    """"alu" for fp32, else "hbm" when the call's byte floor is above its FLOP
    floor (the masked decode layout, and the 256-expert layer whose ~256 rows
    per expert give each weight byte fewer FLOPs than the ridge point), else
    "tensor"."""
    if w.dtype == "f32":
        return "alu"
    compute_ms, hbm_ms = floors(w, R, touched, peaks)
    return "hbm" if w.layout == "masked" or hbm_ms > compute_ms else "tensor"


def roofline(w, moe, cfg, gemm_ms, R, touched, peaks, gemm_launches, dev):
    """The dominant kernel of the step (the grouped SwiGLU call) against the
    roof that binds it: the bf16 tensor peak, or HBM where the call's
    algorithmic bytes take longer at the copy rate than its FLOPs at the tensor
    peak (it streams the touched experts' weights once); the FP32 FFMA rate
    for fp32.  Both floors are reported beside the fraction."""
    import torch
    alg = algorithmic(w, R, touched)
    name = grouped_kernel(w.name)[0]
    kernel = f"{name}: {gemm_launches} launch{'es' if gemm_launches != 1 else ''} per call"
    compute_ms, hbm_ms = floors(w, R, touched, peaks)
    both = {"compute_floor_ms": compute_ms, "hbm_floor_ms": hbm_ms,
            "frac_of_tensor": compute_ms / gemm_ms, "frac_of_hbm": hbm_ms / gemm_ms}
    bound = grouped_bound(w, R, touched, peaks)
    if bound == "hbm":
        achieved = alg["grouped_bytes"] / (gemm_ms * 1e-3) / 1e9
        return {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_source": f"{peaks['source']} copy bandwidth",
                "traffic": recorded_traffic(w.name),
                "algorithmic_bytes_per_call": alg["grouped_bytes"],
                "algorithmic_bytes_note": "touched experts' w1, w3, w2 once + x_perm rows read + "
                                          "h written and read + y written (fp16)",
                "touched_experts": touched, "tflops": alg["ffn_flops"] / (gemm_ms * 1e-3) / 1e12,
                **both}
    achieved = alg["ffn_flops"] / (gemm_ms * 1e-3) / 1e12
    if w.dtype == "f32":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12   # FFMA lanes x 2 FLOP x clock
        return {"kernel": kernel, "bound": "alu", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 FLOP x {peaks['sm_max_mhz']:.0f} MHz",
                "traffic": recorded_traffic(w.name),
                "algorithmic_flops_per_call": alg["ffn_flops"],
                "note": "0.1 GFLOP per call: bound by launch and pipeline latency, not by the ALUs"}
    return {"kernel": kernel, "bound": "tensor", "achieved": achieved,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"],
            "peak_source": f"{peaks['source']} bf16 burst",
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
            "traffic": recorded_traffic(w.name),
            "algorithmic_flops_per_call": alg["ffn_flops"], **both}


def run_gpu(args, name):
    import numpy as np
    import torch
    import torch.distributed as dist

    import moe_inputs
    import routing_grouped_gemm_gb300 as moe

    rank, world, local = dist_env()
    dev = torch.device("cuda", local)

    w = moe_inputs.WORKLOADS[name]
    if args.scale:
        # a reduced case of the same workload (profiling captures only)
        over = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.scale.split(",")}
        w = w.scaled(**over)
    default = name == WORKLOAD and not args.shard
    inp = moe_inputs.make_inputs(w, device=dev, seed=rank)
    cfg = workload_config(moe, w)
    if args.shard:
        # the first expert range and H shard of an EP x TP split (profiling
        # captures only): experts [0, E/EP), hidden units [0, H/TP)
        ep, tp = (int(v) for v in args.shard.split(","))
        el, hl = w.E // ep, w.H // tp
        inp.w1 = inp.w1[:el, :hl].contiguous()
        inp.w3 = inp.w3[:el, :hl].contiguous()
        inp.w2 = inp.w2[:el, :, :hl].contiguous()
        torch.cuda.empty_cache()
        w = w.scaled(H=hl)
        cfg = dataclasses.replace(cfg, H_local=hl, E_local=el)
    dt = moe_inputs.torch_dtype(w)
    if args.fp8_only:
        fp8 = run_fp8(moe, cfg, inp, torch.cuda.current_stream(dev), dev, args, load_peaks())
        if rank == 0:
            print(json.dumps({"workload": name, "fp8": fp8}), flush=True)
        return
    if args.backward_only:
        backward = run_backward(moe, cfg, inp, torch.cuda.current_stream(dev), dev, args,
                                load_peaks())
        if rank == 0:
            print(json.dumps({"workload": name, "scale": args.scale or None,
                              "T": w.T, "D": w.D, "H": w.H, "E": w.E, "k": w.k,
                              "backward": backward}), flush=True)
        return
    ra = moe.rows_alloc(cfg)
    ws = moe.alloc_workspace(cfg, device=dev)
    logits = None
    topk_idx = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    topk_w = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    tpe = torch.empty(w.E, dtype=torch.int32, device=dev)
    seg = torch.empty(cfg.e_local + 1, dtype=torch.int32, device=dev)
    row_of = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    tor = torch.empty(ra, dtype=torch.int32, device=dev)
    x_perm = torch.empty((ra, w.D), dtype=dt, device=dev)
    h = torch.empty((ra, w.H), dtype=dt, device=dev)
    y_perm = torch.empty((ra, w.D), dtype=cfg.y_dtype, device=dev)
    out = torch.empty((w.T, w.D), dtype=dt, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev) if needs_l2_flush(w) else None

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        moe.moe_route_topk(cfg, inp.x, inp.wg, inp.bias, logits, topk_idx, topk_w, ws, stream)
        if ev is not None:
            ev[1].record(stream)
        moe.moe_permute(cfg, inp.x, topk_idx, tpe, seg, row_of, tor, x_perm, ws, stream)
        if ev is not None:
            ev[2].record(stream)
        moe.moe_grouped_swiglu(cfg, x_perm, seg, tpe, inp.w1, inp.w3, inp.w2, h, y_perm, ws, stream)
        if ev is not None:
            ev[3].record(stream)
        moe.moe_unpermute_combine(cfg, y_perm, row_of, topk_w, out, ws, stream)
        if ev is not None:
            ev[4].record(stream)

    # the timed step is the layer call a user makes (one C-ABI call: route,
    # permute, grouped SwiGLU, combine on one stream, every intermediate in
    # its workspace); the per-call breakdown below times the four step calls
    # one by one
    lws = moe.alloc_workspace(cfg, device=dev, layer=True)

    def layer_step():
        moe.moe_layer_forward(cfg, inp.x, inp.wg, inp.bias, inp.w1, inp.w3, inp.w2, out, lws,
                              stream)

    for _ in range(max(3, args.warmup)):
        step()
        layer_step()
    # launches of one grouped SwiGLU call (one cooperative launch or two)
    n0 = moe.kernel_launches()
    moe.moe_grouped_swiglu(cfg, x_perm, seg, tpe, inp.w1, inp.w3, inp.w2, h, y_perm, ws, stream)
    gemm_launches = moe.kernel_launches() - n0
    torch.cuda.synchronize(dev)
    for wsx in (ws, lws):
        st = moe.moe_get_device_status(wsx, stream)
        if st != moe.MOE_OK:
            raise RuntimeError(f"device status after warm-up: {moe.status_string(st)}")

    # the timed loop has events only at its two ends: events between the
    # calls would cut the programmatic launch overlap of consecutive kernels;
    # the per-call breakdown comes from a second, separately timed loop.
    # Where the inputs fit in L2, every step is timed on its own after a flush.
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        n_launch0 = moe.kernel_launches()
        if flush is None:
            t_start = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            for i in range(args.steps):
                layer_step()
            t_end.record(stream)
            n_launches = moe.kernel_launches() - n_launch0
            torch.cuda.synchronize(dev)
            local_ms = t_start.elapsed_time(t_end)
        else:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for i in range(args.steps):
                flush.zero_()
                evs[i][0].record(stream)
                layer_step()
                evs[i][1].record(stream)
            n_launches = moe.kernel_launches() - n_launch0
            torch.cuda.synchronize(dev)
            local_ms = sum(a.elapsed_time(b) for a, b in evs)
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(local_ms, dev)
    st = moe.moe_get_device_status(lws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after timing: {moe.status_string(st)}")

    n_parts = max(20, args.steps // 4)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_parts)]
    for i in range(n_parts):
        if flush is not None:
            flush.zero_()
        step(evs[i])
    torch.cuda.synchronize(dev)
    st = moe.moe_get_device_status(ws, stream)
    if st != moe.MOE_OK:
        raise RuntimeError(f"device status after the breakdown: {moe.status_string(st)}")
    parts = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in evs])  # ms
    mean_parts = parts.mean(0)
    ms_per_step = elapsed_ms / args.steps
    value = replica_tokens_per_s(world, w.T, ms_per_step)

    # end to end: host x in and host out every step, through the C ABI
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(moe, cfg, inp, out, stream, dev, world, args)
    fused = fp8 = backward = gather = None
    if w.dtype == "bf16" and not args.no_gather:
        gather = run_gather(moe, cfg, inp, stream, dev, args)
    if default and not args.no_fused:
        fused = run_fused(moe, cfg, inp, stream, dev, args)
    if default and not args.no_fp8:
        fp8 = run_fp8(moe, cfg, inp, stream, dev, args, load_peaks())
    if default and not args.no_backward:
        backward = run_backward(moe, cfg, inp, stream, dev, args, load_peaks())
    tpe_h = tpe.cpu().numpy()
    local_cnt = tpe_h[cfg.e_first:cfg.e_first + cfg.e_local]
    R = int(np.minimum(local_cnt, cfg.capacity).sum() if w.layout == "masked" else local_cnt.sum())
    touched = int((local_cnt > 0).sum())
    alg = algorithmic(w, R, touched)
    peaks = load_peaks()
    gemm_ms = float(mean_parts[2])
    roof = roofline(w, moe, cfg, gemm_ms, R, touched, peaks, gemm_launches, dev)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": workload_data_note(w),
        "value_counts": VALUE_COUNTS, "tokens_per_step": w.T, "routed_rows_per_step": R,
        "config": {"workload": name, "T": w.T, "D": w.D, "H": w.H, "E": w.E, "k": w.k,
                   "shard": args.shard or None,
                   "router": router_note(w), "layout": layout_note(w),
                   "parallelism": f"replicas x{world}" if world > 1 else "single", "l2": l2_note(w)},
        "roofline": roof,
        "api": "moe_layer_forward (C ABI): one call per step; intermediates in its workspace",
        "breakdown_ms": {"route": float(mean_parts[0]), "permute": float(mean_parts[1]),
                         "grouped_swiglu": gemm_ms, "combine": float(mean_parts[3])},
        "breakdown_note": "the four step calls (moe_route_topk, moe_permute, moe_grouped_swiglu, "
                          "moe_unpermute_combine) one by one, CUDA events between them; the "
                          "layer call also lets the router write the dispatch's count input "
                          "where the count matrix is small, one launch fewer",
        "bandwidth": {
            "permute_gbs": alg["permute_bytes"] / (mean_parts[1] * 1e-3) / 1e9,
            "combine_gbs": alg["combine_bytes"] / (mean_parts[3] * 1e-3) / 1e9,
            "combine_gbs_moved": alg["combine_bytes_moved"] / (mean_parts[3] * 1e-3) / 1e9,
            "combine_note": "combine_gbs counts the method's bytes (y rows at the activation "
                            "width); combine_gbs_moved counts the y_perm actually read (fp16 for "
                            "bf16 layers, so the two agree there)",
            "hbm_peak_gbs": peaks["hbm_gbs"]},
        "gemm_tflops": alg["ffn_flops"] / (gemm_ms * 1e-3) / 1e12,
        "tokens_per_expert": {"min": int(tpe_h.min()), "max": int(tpe_h.max()),
                              "zeros": int((tpe_h == 0).sum())},
        "e2e": e2e,
        "gather": gather,
        "gpu_launches": n_launches,
        "clocks": clk.summary(),
    }
    if default:
        line.update({"fused_combine": fused, "fp8": fp8, "backward": backward})

    if rank == 0 and not args.no_cpu_baseline and not args.shard:
        line["cpu_baseline"] = cpu_baseline(inp, w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    del inp, ws, x_perm, h, y_perm, out, flush
    torch.cuda.empty_cache()


def run_gpu_arm(args):
    import torch
    import torch.distributed as dist
    import moe_inputs
    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    try:
        names = moe_inputs.WORKLOAD_ORDER if args.workload == "all" else [args.workload]
        for name in names:
            run_gpu(args, name)
    finally:
        if world > 1:
            dist.destroy_process_group()


def run_dispatch_bandwidth(args):
    """--dispatch-bandwidth: the permute and combine calls alone on the contiguous bf16
    workloads, each call timed between CUDA events after an L2 flush (a 256 MB write);
    one JSON line per workload, rates against the measured copy bandwidth."""
    import torch

    import moe_inputs
    import routing_grouped_gemm_gb300 as moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    cases = [moe_inputs.WORKLOADS[n] for n in ("fine-grained-bf16", "zipf-skewed",
                                               "deepseek-v3-shaped")]
    # a long prefill batch: 128 count blocks x 256 experts = 32768 count cells,
    # above both single-pass limits, so the permute runs its four-launch chain
    # (D = 1024 keeps the case near 2 GB on the device)
    cases.append(moe_inputs.WORKLOADS["zipf-skewed"].scaled(
        name="prefill-32k-e256-d1024", T=32768, D=1024, E=256, zipf_s=None))
    if args.workload not in ("all", WORKLOAD):
        cases = [c for c in cases if c.name == args.workload]
    for w in cases:
        name = w.name
        inp = moe_inputs.make_inputs(w, device=dev, seed=0, weights=False)
        cfg = moe.Config(T=w.T, D=w.D, H_local=w.H, E=w.E, k=w.k, dtype=moe.MOE_BF16,
                         score=moe.MOE_SCORE_SOFTMAX if w.score == "softmax"
                         else moe.MOE_SCORE_SIGMOID,
                         renorm=int(w.renorm), align_m=128, n_group=w.n_group,
                         topk_group=w.topk_group)
        ws = moe.alloc_workspace(cfg, device=dev)
        idx = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        wts = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        moe.moe_route_topk(cfg, inp.x, inp.wg, inp.bias, None, idx, wts, ws)
        ra = moe.rows_alloc(cfg)
        tpe = torch.empty(w.E, dtype=torch.int32, device=dev)
        seg = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
        row_of = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        tor = torch.empty(ra, dtype=torch.int32, device=dev)
        xp = torch.empty((ra, w.D), dtype=torch.bfloat16, device=dev)
        y = torch.randn((ra, w.D), dtype=torch.float32, device=dev).to(cfg.y_dtype)
        out = torch.empty((w.T, w.D), dtype=torch.bfloat16, device=dev)
        calls = {
            "permute": lambda: moe.moe_permute(cfg, inp.x, idx, tpe, seg, row_of, tor, xp, ws),
            "combine": lambda: moe.moe_unpermute_combine(cfg, y, row_of, wts, out, ws),
        }
        calls["permute"]()
        assert moe.moe_get_device_status(ws) == moe.MOE_OK
        R = int((row_of >= 0).sum().item())
        nbytes = {"permute": w.T * w.D * 2 + R * w.D * 2,
                  "combine": R * w.D * 2 + w.T * w.D * 2 + w.T * w.k * 8}
        line = {"workload": name, "T": w.T, "D": w.D, "E": w.E, "k": w.k, "routed_rows": R,
                "l2": "flushed before every call", "steps": args.steps, "warmup": args.warmup}
        for key, fn in calls.items():
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.warmup + args.steps):
                flush.zero_()
                if i >= args.warmup:
                    ev[i - args.warmup][0].record()
                fn()
                if i >= args.warmup:
                    ev[i - args.warmup][1].record()
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
            gbs = nbytes[key] / (ms * 1e-3) / 1e9
            line[key] = {"us": ms * 1e3, "bytes": nbytes[key], "gbs": gbs,
                         "frac_of_copy_peak": gbs / peaks["hbm_gbs"]}
        print(json.dumps(line), flush=True)
        del inp, xp, y, out, ws
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    help="a workload of moe_inputs.WORKLOADS, or 'all' (one line each)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--no-backward", action="store_true", help="skip the training backward leg")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 (e4m3 GEMM1) leg")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused-combine leg")
    ap.add_argument("--no-gather", action="store_true",
                    help="skip the leg with the dispatch fused into GEMM1's operand load")
    ap.add_argument("--fp8-only", action="store_true", help="time only the FP8 leg, print its JSON")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the training step (forward_train + backward), print its JSON")
    ap.add_argument("--dispatch-bandwidth", action="store_true",
                    help="time only the permute and combine calls on three workloads")
    ap.add_argument("--scale", default="",
                    help="with --backward-only: override workload sizes, e.g. E=16,k=2 (profiling)")
    ap.add_argument("--shard", default="",
                    help="EP,TP: time the first expert range and H shard only, e.g. 8,4 (profiling)")
    args = ap.parse_args()
    if args.scale and not args.backward_only:
        ap.error("--scale is for --backward-only profiling runs")
    import moe_inputs
    if (args.workload != "all" and args.workload not in moe_inputs.WORKLOADS
            and not args.dispatch_bandwidth):
        ap.error(f"unknown workload {args.workload!r}")
    if (args.fp8_only or args.backward_only) and args.workload != WORKLOAD:
        ap.error("--fp8-only and --backward-only time the default workload")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.dispatch_bandwidth:
        run_dispatch_bandwidth(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
