"""Benchmark of the GB300 MoE layer.

One step = one whole MoE layer (router GEMM, top-8 + weights, histogram, scan,
scatter, block map, gate/up grouped GEMM + SwiGLU, down grouped GEMM + weighted
combine) over the T=8192 prefill workload, 4 distinct weight sets and 4
activation sets cycled so every step streams its weights from HBM (inputs
larger than L2).  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload per step.  Under torchrun (N>1)
every rank runs an independent replica of the layer on its own GPU (the path
has no exchange step); rank 0 prints the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer prefill tokens/s @T=2048/8192; decode µs/layer; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def gateup_traffic():
    """DRAM bytes per gate/up launch from the committed ncu summary, or None when
    the kernel sources changed since the counters were taken."""
    import hashlib
    try:
        txt = open(os.path.join(ROOT, "profiles", "grouped_gemm_t8192_dram.md")).read()
        csrc = os.path.join(ROOT, "bit_grouped_expert_top_gb300", "csrc")
        h = hashlib.sha256()
        for f in ("grouped_gemm.cu", "lily_device.cuh"):
            h.update(open(os.path.join(csrc, f), "rb").read())
    except OSError:
        return None
    vals = {}
    for ln in txt.splitlines():
        if ":" in ln:
            k, v = ln.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_prefix") != h.hexdigest()[:16]:
        return None
    try:
        return int(vals["traffic_bytes_per_launch gateup"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = [ln.split(",") for ln in open(self.path).read().strip().splitlines() if ln.count(",") >= 8]
        os.remove(self.path)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ distributed plumbing
def dist_setup(n_gpus: int):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_config(cfg, world: int) -> dict:
    """The `config` object of the JSON line; both arms report the same one."""
    return {"workload": "prefill_t8192: one MoE layer, T=8192, d=2048, E=256 top-8 + 1 shared, I=512, "
                        "int4 group-64 bf16 scale/bias, 4 weight+activation sets cycled",
            "global_batch": cfg.T * world, "seq_len": cfg.T, "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (each step reads a 456 MB weight set)"}


def job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput of independent replicas: the units every rank processed in
    one step, over the slowest rank's step time (ms)."""
    return units_per_rank * world / (ms_max * 1e-3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU baseline (oracle)
def oracle_sample_rate(cfg, layer_np, x_bits, logits_f32, n_tokens: int):
    """Tokens/s of the fp64 oracle on n_tokens of the workload (all host threads)."""
    import numpy as np
    import oracle
    toks = np.arange(n_tokens, dtype=np.int64)
    t0 = time.perf_counter()
    idx, w = oracle.select(logits_f32[:n_tokens].astype(np.float64), cfg.top_k)
    lg = oracle.logits(x_bits[:n_tokens], layer_np["router_w"], layer_np.get("router_bias"))
    oracle.moe_tokens(layer_np, x_bits[:n_tokens], idx, w, None, d=cfg.d, E=cfg.E, I=cfg.I,
                      I_shared=cfg.I_shared)
    dt = time.perf_counter() - t0
    del lg, toks
    return n_tokens / dt, dt


def input_digests(ctx):
    """sha256 (first 16 hex digits) of every input buffer of the timed workload:
    each weight set (its tensors in name order) and each activation set."""
    import hashlib
    out = {}
    for i, (layer, x) in enumerate(zip(ctx["layers"], ctx["xs"])):
        h = hashlib.sha256()
        for k in sorted(layer):
            h.update(layer[k].detach().contiguous().view(-1).view(torch_uint8()).cpu().numpy().tobytes())
        out[f"weights_{i}"] = h.hexdigest()[:16]
        out[f"x_{i}"] = hashlib.sha256(x.detach().contiguous().view(-1).view(torch_uint8()).cpu().numpy().tobytes()
                                       ).hexdigest()[:16]
    return out


def torch_uint8():
    import torch
    return torch.uint8


def oracle_single_thread_rates(peaks_unused=None):
    """Tokens/s of the fp64 oracle on one host thread, on the tiny workload and on
    16 tokens of the T=512 workload (a bounded sample)."""
    import oracle
    from bit_grouped_expert_top_gb300.inputs import CONFIGS, make_layer, make_x
    res = {}
    n_all = oracle.num_threads()
    oracle.set_threads(1)
    try:
        for name, n in (("tiny", 32), ("prefill_t512", 16)):
            cfg = CONFIGS[name]
            layer = _np_layer(make_layer(cfg, "cpu"))
            xb = _bits(make_x(cfg, "cpu"))[:n]
            lg = oracle.logits(xb, layer["router_w"], layer.get("router_bias")).astype("float32")
            rate, dt = oracle_sample_rate(cfg, layer, xb, lg, n)
            res[name] = {"tokens_per_s": round(rate, 3), "tokens": n, "seconds": round(dt, 2), "threads": 1}
    finally:
        oracle.set_threads(n_all)
    return res


def _np_layer(layer_t):
    import numpy as np
    import torch
    out = {}
    for k, v in layer_t.items():
        v = v.detach().cpu().contiguous()
        out[k] = v.view(torch.int16).numpy().view(np.uint16) if v.dtype == torch.bfloat16 else v.numpy()
    return out


def _bits(t):
    import numpy as np
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ our arm
def prefill_flops(cfg, T):
    per_tok = 2 * 3 * cfg.d * cfg.I * (cfg.top_k + 1) + 2 * cfg.d * cfg.E
    return T * per_tok, T * 2 * 2 * cfg.d * cfg.I * (cfg.top_k + 1), T * 2 * cfg.d * cfg.I * (cfg.top_k + 1)


def tensor_peak(peaks, clocks):
    """Dense bf16 tensor peak to divide by (the fp16 dense rate is the same).
    The burst figure applies while the SM clock stays at its maximum during the
    timed region (the step is short and under the power limit); the sustained
    one, measured under the power cap, when the clock was held down."""
    burst, sust = peaks["bf16_tflops"], peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm and mx and sm < 0.95 * mx:
        return sust, f"{peaks['source']} bf16 sustained (SM clock {sm:.0f} of {mx:.0f} MHz under load)"
    return burst, (f"{peaks['source']} bf16 burst (SM clock {sm:.0f} of {mx:.0f} MHz under load; "
                   f"sustained figure {sust})" if sm and mx else f"{peaks['source']} bf16 burst")


def routing_counts(ctx, stream):
    """Expert histogram of the first weight/activation set (one routing call)."""
    import bit_grouped_expert_top_gb300 as lm
    rt = lm.alloc_routing(ctx["shape"])
    stream.wait_stream(__import__("torch").cuda.current_stream())
    lm.lily_moe_route(ctx["shape"], ctx["ws_l"][0], ctx["xs"][0], lm.make_routing(rt), ctx["ws"], stream=stream)
    stream.synchronize()
    return rt["counts"].cpu().numpy()


def config_roofline(cfg, ms, counts, peaks, peak_tc):
    """Roofline of one prefill workload from its realised expert counts: the
    method's FLOPs (9 experts per token + router) against the tensor peak, and
    its bytes (int4 + scale/bias of every expert with a token, the shared
    expert, the router, x in and out) against HBM; the bound is the larger time."""
    from bit_grouped_expert_top_gb300.inputs import weight_bytes
    wb = weight_bytes(cfg)
    touched = int((counts > 0).sum())
    nbytes = (touched + 1) * wb["expert"] + wb["router"] + cfg.T * cfg.d * 2 + cfg.T * cfg.d * 4
    flops = prefill_flops(cfg, cfg.T)[0]
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peak_tc * 1e12)
    t = ms * 1e-3
    return {"bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": round(max(t_hbm, t_tc) / t, 4),
            "hbm_gbs": round(nbytes / t / 1e9, 1), "hbm_peak": peaks["hbm_gbs"],
            "tflops": round(flops / t / 1e12, 1), "tensor_peak": peak_tc,
            "algorithmic_bytes": int(nbytes), "algorithmic_flops": int(flops), "experts_touched": touched}


def time_prefill(cfg, steps, warmup, n_sets, stream, with_stages=True):
    """Device time of `steps` forward passes cycling n_sets weight/activation sets."""
    import torch
    import bit_grouped_expert_top_gb300 as lm
    from bit_grouped_expert_top_gb300.inputs import make_layer, make_x
    layers = [make_layer(cfg, "cuda", i) for i in range(n_sets)]
    ws_l = [lm.make_weights(L) for L in layers]
    xs = [make_x(cfg, "cuda", seed_offset=i) for i in range(n_sets)]
    s = lm.make_shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.top_k, I=cfg.I, I_shared=cfg.I_shared,
                      group=cfg.group, block_rows=cfg.block_rows)
    ws = lm.alloc_workspace(s)
    out = torch.empty((cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    # inputs and the zeroed workspace were made on the default stream
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for i in range(warmup):
            lm.lily_moe_forward(s, ws_l[i % n_sets], xs[i % n_sets], out, ws, stream=stream)
    stream.synchronize()
    status = lm.lily_moe_device_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)] if with_stages else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    return dict(layers=layers, ws_l=ws_l, xs=xs, shape=s, ws=ws, out=out, evs=evs, start=start, end=end)


def run_timed(ctx, steps, stream, n_sets, stages=True):
    """`steps` forward passes; with stages, lily_moe_forward_timed records the
    stage events of every pass (which breaks the overlap of consecutive
    kernels), else plain lily_moe_forward."""
    import bit_grouped_expert_top_gb300 as lm
    s, ws, out = ctx["shape"], ctx["ws"], ctx["out"]
    ctx["start"].record(stream)
    for i in range(steps):
        j = i % n_sets
        if stages and ctx["evs"] is not None:
            lm.lily_moe_forward_timed(s, ctx["ws_l"][j], ctx["xs"][j], out, ws, ctx["evs"][i], stream=stream)
        else:
            lm.lily_moe_forward(s, ctx["ws_l"][j], ctx["xs"][j], out, ws, stream=stream)
    ctx["end"].record(stream)


def time_e2e(ctx, steps, n_sets, stream):
    """ms per step of the layer through lily_moe_forward with host buffers: each
    step copies its x from pinned host memory to the device and its out back.
    Three streams: the input copy of step i, the layer of step i - 1 and the
    output copy of step i - 2 run at the same time; device and host buffers are
    double buffered, and events order each buffer's reuse."""
    import torch
    import bit_grouped_expert_top_gb300 as lm
    cfg_T, d = ctx["out"].shape
    x_host = [x.cpu().pin_memory() for x in ctx["xs"]]
    out_host = [torch.empty((cfg_T, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(ctx["xs"][0]) for _ in range(2)]
    out_dev = [torch.empty_like(ctx["out"]) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    loaded, computed, stored = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def run(n):
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(h2d):
                if used[b]:
                    h2d.wait_event(computed[b])        # the layer that read x_dev[b] is done
                x_dev[b].copy_(x_host[i % n_sets], non_blocking=True)
                loaded[b].record(h2d)
            stream.wait_event(loaded[b])
            if used[b]:
                stream.wait_event(stored[b])           # out_dev[b] copied out by the step before last
            lm.lily_moe_forward(ctx["shape"], ctx["ws_l"][i % n_sets], x_dev[b], out_dev[b], ctx["ws"], stream=stream)
            computed[b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                stored[b].record(d2h)
            used[b] = True
        stream.wait_stream(h2d)
        stream.wait_stream(d2h)

    stream.wait_stream(torch.cuda.current_stream())
    run(3)
    stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    h2d.wait_event(a)
    d2h.wait_event(a)
    run(steps)
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / steps


def stage_means(ctx):
    evs = ctx["evs"]
    names = ["route", "route_tables", "prep", "gateup", "down"]
    acc = {n: [] for n in names}
    for e in evs:
        for k, n in enumerate(names):
            acc[n].append(e[k].elapsed_time(e[k + 1]) * 1e3)  # us
    return {n: statistics.mean(v) for n, v in acc.items()}


def bench_decode(cfg, Ts, reps, stream, peaks):
    """µs per layer of lily_moe_decode over cfg.n_layers distinct layers."""
    import numpy as np
    import torch
    import bit_grouped_expert_top_gb300 as lm
    from bit_grouped_expert_top_gb300.inputs import make_layer, make_x, weight_bytes
    L = cfg.n_layers
    layers = [make_layer(cfg, "cuda", i) for i in range(L)]
    wl = [lm.make_weights(x) for x in layers]
    wb = weight_bytes(cfg)
    res = {}
    for T in Ts:
        s = lm.make_shape(T=T, d=cfg.d, E=cfg.E, top_k=cfg.top_k, I=cfg.I, I_shared=cfg.I_shared,
                          group=cfg.group, block_rows=cfg.block_rows)
        ws = lm.alloc_workspace(s, n_layers_decode=L)
        x = make_x(cfg, "cuda", seed_offset=500 + T, T=T)
        out = torch.empty((L, T, cfg.d), dtype=torch.float32, device="cuda")
        idx = torch.empty((L, T, cfg.top_k), dtype=torch.int32, device="cuda")
        stream.wait_stream(torch.cuda.current_stream())
        for _ in range(3):
            lm.lily_moe_decode(s, wl, x, out, ws, trace={"topk_idx": idx}, stream=stream)
        stream.synchronize()
        assert lm.lily_moe_device_status(ws, stream) == 0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            lm.lily_moe_decode(s, wl, x, out, ws, trace={"topk_idx": idx}, stream=stream)
        b.record(stream)
        b.synchronize()
        us_layer = a.elapsed_time(b) * 1e3 / (reps * L)
        ids = idx.cpu().numpy()
        distinct = np.mean([len(np.unique(ids[l])) for l in range(L)])
        expert_bytes = (distinct + 1) * wb["expert"]
        total_bytes = expert_bytes + wb["router"]
        res[f"T{T}"] = {"us_per_layer": round(us_layer, 3), "experts_read_per_layer": round(float(distinct) + 1, 2),
                        "weight_bytes_per_layer": int(total_bytes),
                        "achieved_gbs": round(total_bytes / (us_layer * 1e-6) / 1e9, 1),
                        "frac_of_hbm": round(total_bytes / (us_layer * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                        "expert_bytes_gbs": round(expert_bytes / (us_layer * 1e-6) / 1e9, 1)}
    return res


def bench_attention(names, reps, stream, peaks):
    """µs per call of lily_attn_decode (batch-1 grouped-query decode attention)
    at the given context lengths, against HBM on the K/V bytes read; the caches
    of n_sets workloads are cycled so that the bytes of consecutive calls
    exceed L2."""
    import torch
    import bit_grouped_expert_top_gb300 as lm
    from bit_grouped_expert_top_gb300.attn_inputs import ATTN_CONFIGS, kv_bytes, make_attn
    res = {}
    for name in names:
        cfg = ATTN_CONFIGS[name]
        sets = [{k: v.cuda() for k, v in make_attn(cfg, "cpu", i).items()} for i in range(cfg.n_sets)]
        s = lm.make_attn_shape(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.block_size, cfg.max_blocks)
        ws = lm.alloc_attn_workspace(s)
        out = torch.empty((cfg.B, cfg.H_q, cfg.D), dtype=torch.float32, device="cuda")
        stream.wait_stream(torch.cuda.current_stream())

        def call(a):
            lm.lily_attn_decode(s, a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"], out, ws,
                                stream=stream)
        for i in range(3 * cfg.n_sets):
            call(sets[i % cfg.n_sets])
        stream.synchronize()
        assert lm.lily_moe_device_status(ws, stream) == 0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            call(sets[i % cfg.n_sets])
        b.record(stream)
        b.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        nbytes = kv_bytes(cfg)
        res[name] = {"context_tokens": sum(cfg.seq_lens), "heads": f"{cfg.H_q}q/{cfg.H_kv}kv", "D": cfg.D,
                     "block_size": cfg.block_size, "us_per_call": round(us, 2), "kv_bytes": nbytes,
                     "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac_of_hbm": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                     "bytes_cycled": nbytes * cfg.n_sets}
        del sets
        torch.cuda.empty_cache()
    return res


def bench_gdn(names, reps, stream, clocks):
    """µs per call of lily_gdn_scan; the scan is a sequential fp32 recurrence, so
    its roofline is the fp32 FMA rate of the CUDA cores (152 SMs x 128 lanes x 2
    flops per cycle at the sampled SM clock)."""
    import torch
    import bit_grouped_expert_top_gb300 as lm
    from bit_grouped_expert_top_gb300.gdn_inputs import GDN_CONFIGS, gdn_bytes, gdn_flops, make_gdn
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = (clocks or {}).get("sm_mhz") or 2070.0
    peak = sms * 128 * 2 * mhz * 1e6 / 1e12  # TFLOP/s
    res = {}
    for name in names:
        cfg = GDN_CONFIGS[name]
        g = {k: v.cuda() for k, v in make_gdn(cfg, "cpu").items()}
        out = torch.empty((cfg.T, cfg.H_v, cfg.d_v), dtype=torch.float32, device="cuda")
        st = torch.empty((cfg.H_v, cfg.d_v, cfg.d_k), dtype=torch.float32, device="cuda")
        stream.wait_stream(torch.cuda.current_stream())

        def call():
            lm.lily_gdn_scan(g["q"], g["k"], g["v"], g["alpha"], g["beta"], out, st, state_in=g["state"],
                             stream=stream)
        for _ in range(3):
            call()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            call()
        b.record(stream)
        b.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        fl = gdn_flops(cfg)
        res[name] = {"tokens": cfg.T, "heads": f"{cfg.H_k}qk/{cfg.H_v}v", "d": cfg.d_k, "us_per_call": round(us, 1),
                     "tokens_per_s": round(cfg.T / (us * 1e-6)),
                     "roofline": {"bound": "alu", "achieved": round(fl / (us * 1e-6) / 1e12, 2), "peak": round(peak, 1),
                                  "unit": "TFLOP/s", "frac": round(fl / (us * 1e-6) / 1e12 / peak, 4),
                                  "peak_note": "fp32 FMA: SMs x 128 lanes x 2 flops x sampled SM clock"},
                     "hbm_gbs": round(gdn_bytes(cfg) / (us * 1e-6) / 1e9, 1)}
        del g
    return res


def run_ours(args):
    import numpy as np
    import torch
    import bit_grouped_expert_top_gb300 as lm
    from bit_grouped_expert_top_gb300.inputs import CONFIGS
    import oracle

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    lm.load()
    peaks = load_peaks()
    cfg = CONFIGS["prefill_t8192"]
    n_sets = cfg.n_weight_sets
    stream = torch.cuda.Stream()
    ctx = time_prefill(cfg, args.steps, args.warmup, n_sets, stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = ClockSampler(local)
    clk.start()
    # the timed steps: the layer as a caller runs it (lily_moe_forward, no events)
    run_timed(ctx, args.steps, stream, n_sets, stages=False)
    stream.synchronize()
    clocks = clk.stop()
    ms = ctx["start"].elapsed_time(ctx["end"]) / args.steps
    ms = max_over_ranks(ms, world)
    if lm.lily_moe_device_status(ctx["ws"], stream) != 0:
        raise RuntimeError("device status error in timed region")
    # stage times from a second pass with CUDA events at the stage boundaries (the
    # events break the programmatic dependent launches, so its steps take longer)
    run_timed(ctx, args.steps, stream, n_sets)
    stream.synchronize()
    st = stage_means(ctx)
    ms_staged = ctx["start"].elapsed_time(ctx["end"]) / args.steps
    tokens_per_s = job_rate(cfg.T, world, ms)
    flops_total, flops_gu, flops_down = prefill_flops(cfg, cfg.T)
    peak_tc, peak_note = tensor_peak(peaks, clocks)
    achieved = flops_gu / (st["gateup"] * 1e-6) / 1e12
    layer_tflops = flops_total / (ms * 1e-3) / 1e12

    # e2e: host buffers through the public call, H2D of x and D2H of out of every step inside the
    # timed region; the copies run on their own streams, double buffered, so step i's input copy
    # and step i-2's output copy overlap step i-1's layer (a serving loop's pipeline)
    e2e_steps = max(5, min(args.steps, 40))
    e2e_ms = max_over_ranks(time_e2e(ctx, e2e_steps, n_sets, stream), world)

    also = {}
    if not args.quick:
        for name in ("prefill_t2048_zipf", "prefill_t512"):
            c = CONFIGS[name]
            cx = time_prefill(c, 50, 5, 1, stream, with_stages=True)
            run_timed(cx, 50, stream, 1, stages=False)
            stream.synchronize()
            ms_c = cx["start"].elapsed_time(cx["end"]) / 50
            run_timed(cx, 50, stream, 1)
            stream.synchronize()
            stc = stage_means(cx)
            counts = routing_counts(cx, stream)
            also[name] = {"tokens_per_s": round(c.T / (ms_c * 1e-3)), "us_per_layer": round(ms_c * 1e3, 2),
                          "stage_us": {k: round(v, 2) for k, v in stc.items()},
                          "roofline": config_roofline(c, ms_c, counts, peaks, peak_tc),
                          "inputs_vs_l2": "weights 456 MB > L2"}
            del cx
        torch.cuda.empty_cache()
        also["decode_l40"] = bench_decode(CONFIGS["decode_t1_l40"], (1, 2, 4, 8), 20, stream, peaks)
        also["attn_decode"] = bench_attention(("attn_32k", "attn_64k", "attn_128k"), 50, stream, peaks)
        also["gdn_scan"] = bench_gdn(("gdn_t512", "gdn_t8192"), 10, stream, clocks)

    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xint4 (fp32 accumulate); router bf16",
        "data": "synthetic (seeded; int4 g64 affine weights, N(0,1) activations)",
        "config": workload_config(cfg, world),
        "stage_us": {k: round(v, 2) for k, v in st.items()},
        "stage_note": "stage times from a second pass with CUDA events at the stage boundaries; that pass "
                      "takes %.4f ms per step (the events stop consecutive kernels from overlapping)" % ms_staged,
        "roofline": {"kernel": "grouped_gemm_kernel (gate/up + SwiGLU)", "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tc, 4), "traffic": gateup_traffic(),
                     "traffic_unit": "bytes per launch (ncu dram read+write of the current kernel source, "
                                     "null if the source changed since the capture)",
                     "peak_note": peak_note,
                     "algorithmic_flops_per_launch": flops_gu},
        "roofline_layer": {"what": "whole layer: router + routing tables + expert GEMMs, ms_per_step",
                           "bound": "tensor", "achieved": round(layer_tflops, 1), "peak": peak_tc,
                           "unit": "TFLOP/s", "frac": round(layer_tflops / peak_tc, 4),
                           "algorithmic_flops_per_step": flops_total, "peak_note": peak_note},
        "layer_tflops": round(layer_tflops, 1),
        "clocks": clocks,
        "e2e": {"value": round(job_rate(cfg.T, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 4},
        "gpu_launches": 7 * args.steps,  # router GEMM, top-8, scan, scatter, prep, gate/up, down
        "also": also,
    }
    if rank == 0:
        # CPU baseline: the oracle as it stands, on a bounded token sample of the same workload
        lg = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
        rt = lm.alloc_routing(ctx["shape"])
        rt["logits"] = lg
        r = lm.make_routing(rt)
        stream.wait_stream(torch.cuda.current_stream())
        lm.lily_moe_route(ctx["shape"], ctx["ws_l"][0], ctx["xs"][0], r, ctx["ws"], stream=stream)
        stream.synchronize()
        n_tok = args.cpu_baseline_tokens
        rate, dt = oracle_sample_rate(cfg, _np_layer(ctx["layers"][0]), _bits(ctx["xs"][0]), lg.cpu().numpy(), n_tok)
        line["cpu_baseline"] = {"value": round(rate, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                                "kind": "oracle",
                                "sample": f"{n_tok} tokens of prefill_t8192 (router + top-8 + 9 experts each), "
                                          f"{dt:.1f} s wall"}
        if not args.quick:
            line["cpu_baseline"]["single_thread"] = oracle_single_thread_rates()
            line["inputs_sha256"] = input_digests(ctx)
        print(json.dumps(line), flush=True)
    barrier(world)


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args):
    import numpy as np
    import torch
    from bit_grouped_expert_top_gb300.inputs import CONFIGS, make_layer, make_x
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = CONFIGS["prefill_t8192"]
    L = _np_layer(make_layer(cfg, "cpu", 0))
    xb = _bits(make_x(cfg, "cpu"))
    n_tok = args.cpu_tokens
    lg = oracle.logits(xb[:n_tok], L["router_w"], L.get("router_bias")).astype(np.float32)
    for _ in range(args.warmup if args.warmup < 2 else 1):
        oracle_sample_rate(cfg, L, xb, lg, max(1, n_tok // 4))
    times = []
    for _ in range(args.steps):
        _, dt = oracle_sample_rate(cfg, L, xb, lg, n_tok)
        times.append(dt)
    total = sum(times)
    rate = n_tok * len(times) / total
    line = {"impl": "reference", "metric": METRIC, "value": round(rate, 3), "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": workload_config(cfg, args.gpus),
            "cpu_baseline": {"value": round(rate, 3), "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{n_tok} tokens of the prefill_t8192 workload per step (router + top-8 "
                                       f"+ 9 experts each), weight set 0"},
            "e2e": {"value": round(rate, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=24,
                    help="oracle sample per step of the reference arm (tokens)")
    ap.add_argument("--cpu-baseline-tokens", type=int, default=1024,
                    help="oracle sample of the cpu_baseline entry (tokens; about 10 s on 16 cores)")
    ap.add_argument("--quick", action="store_true", help="headline workload only (no extra configs / decode)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
