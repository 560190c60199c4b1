#!/usr/bin/env python
"""Benchmark of the fused MXFP4-weight MoE layer on one GB300: tokens/s and the
fraction of the block-scaled roofline.

One step = one pass of the layer's hot path over one batch: top-k routing
from router logits, permutation, MXFP8 activation quantisation, FC1 +
SwiGLU + requant, FC2 + combine (``kt_moe_route_permute`` then
``kt_mxfp4_moe_forward_routed``, which reuses the routing call's
permutation; decode-sized layers: ``kt_mxfp4_moe_decode``, one launch).
Inputs are seeded and synthetic, resident in HBM when the timed region
starts; ``e2e`` repeats the measurement with the
step's inputs (hidden, logits) copied from pinned host memory and the output
copied back inside the timed region.

Default workload: the Kimi-K3-shaped layer at T=8192 prefill tokens (H=7168,
E=896 experts, top-16, I=3584, uniform router logits; 36.7 GB of packed
experts, all resident), the largest configuration that fits one GPU.  The
DeepSeek-V4-Flash-shaped layer (T=4096, H=4096, E=256, top-6, I=2048,
Zipf(1.1) skew) is measured after it and nested under "secondary".  Expert
weights far exceed L2, so every step streams them from HBM (no L2 flush is
needed between steps).

``--impl reference`` times the fp64 CPU oracle (the only reference
implementation; the pages ship no code) on the host cores, on a bounded
token sample per step, and prints the same JSON line with "impl":
"reference".

The layer runs on one GPU: it is not sharded and has no collective step.
Multi-GPU runs (``--gpus N`` with N > 1, or WORLD_SIZE > 1 under torchrun)
print an "unavailable" line on rank 0 and exit without touching a GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import mxfp4_weight_moe_gb300 as kt  # noqa: E402
from mxfp4_weight_moe_gb300 import synthetic as syn  # noqa: E402

METRIC = "MXFP4 fused-MoE layer tokens/s at 1 GB300; % of block-scaled roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0     # nominal dense ratio (4.5 / 2.25 PFLOP/s); mxf8f6f4 runs at the fp8 rate

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one FC1 launch
# from an ncu capture (the summaries under profiles/ give the command), keyed
# by workload and by the SHA-256 of the GEMM source it was taken on: once the
# kernel changes, the figure no longer applies and the bench line reports
# traffic null.
GEMM_SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "mxfp4_weight_moe_gb300", "csrc", "kt_gemm_mx.cu")
FC1_TRAFFIC = {
    ("dsv4", "fd79b72d69a1d01a24bf2389aa0c7423ce2fb39c693b30cf8ab916b6e1eae91a"): 2386266368 + 52687872,
    ("kimi_T8192", "fd79b72d69a1d01a24bf2389aa0c7423ce2fb39c693b30cf8ab916b6e1eae91a"): 25473608448 + 485629696,
    ("kimi_T16", "fd79b72d69a1d01a24bf2389aa0c7423ce2fb39c693b30cf8ab916b6e1eae91a"): 6206675456 + 4165632,
    ("small_T32", "fd79b72d69a1d01a24bf2389aa0c7423ce2fb39c693b30cf8ab916b6e1eae91a"): 8587776,
    ("small_T1", "fd79b72d69a1d01a24bf2389aa0c7423ce2fb39c693b30cf8ab916b6e1eae91a"): 2334976,
    ("tiny", "fd79b72d69a1d01a24bf2389aa0c7423ce2fb39c693b30cf8ab916b6e1eae91a"): 132864,
}


def fc1_traffic(workload: str):
    import hashlib

    try:
        sha = hashlib.sha256(open(GEMM_SRC, "rb").read()).hexdigest()
    except OSError:
        return None
    return FC1_TRAFFIC.get((workload, sha))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:  # noqa: BLE001
            self.ident = str(device.index or 0)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows]
        mx = [num(r[2]) for r in rows]
        power = [num(r[3]) for r in rows]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6), ("sw_thermal_slowdown", 7),
                              ("sw_power_cap", 8)):
                if r[col].lower().startswith("active"):
                    reasons.add(name)
        loaded = [s for s, p in zip(sm, power) if p == p] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(p for p in power if p == p) if any(p == p for p in power)
                else None}


# ------------------------------------------------------------------ work accounting
def algorithmic(cfg, touched: int):
    """Algorithmic FLOPs and HBM bytes of one layer step and of each GEMM launch.

    FLOPs = 6*H*I*S (FC1 4HI + FC2 2HI per slot).  Bytes = touched experts x
    (w13 + w2 + their e8m0 scales = 1.59375*H*I) + bf16 hidden in and out
    (4*T*H) + ids and weights (8*S); intermediates are implementation traffic."""
    H, I, S, T = cfg.H, cfg.I, cfg.S, cfg.T
    w13_bytes = 2 * I * H // 2 + 2 * I * H // 32
    w2_bytes = H * I // 2 + H * I // 32
    return {
        "layer_flops": 6.0 * H * I * S,
        "layer_bytes": float(touched * (w13_bytes + w2_bytes) + 4 * T * H + 8 * S),
        "fc1_bytes": float(touched * w13_bytes), "fc1_flops": 4.0 * H * I * S,
        "fc2_bytes": float(touched * w2_bytes), "fc2_flops": 2.0 * H * I * S,
        "w13_bytes_per_expert": w13_bytes, "w2_bytes_per_expert": w2_bytes,
    }


def workload_desc(cfg):
    return (f"{cfg.name}: T={cfg.T} H={cfg.H} E={cfg.E} top_k={cfg.k} I={cfg.I} "
            f"logits={cfg.logits} seed={cfg.seed}")


# ------------------------------------------------------------------ CPU oracle on token samples
# A step whose weights and activations total less than this is timed one step at a time, with an L2 scrub
# between steps (outside the timed events): otherwise its experts would stay resident in the 129 MB L2.
L2_FLUSH_BELOW = 1 << 30
L2_SCRUB_BYTES = 256 << 20


def needs_l2_flush(work: dict) -> bool:
    return work["layer_bytes"] < L2_FLUSH_BELOW


def config_block(cfg, touched: int, work: dict) -> dict:
    """The line's "config" (identical for this arm and the reference arm)."""
    if needs_l2_flush(work):
        l2 = (f"flushed between steps: {L2_SCRUB_BYTES >> 20} MB written before each step, outside its timed "
              f"events ({work['layer_bytes'] / 1e6:.1f} MB of weights+activations per step)")
    else:
        l2 = f"inputs larger than L2 ({work['layer_bytes'] / 1e9:.2f} GB of weights+activations per step)"
    return {"workload": workload_desc(cfg), "T": cfg.T, "H": cfg.H, "E": cfg.E, "top_k": cfg.k, "I": cfg.I,
            "touched_experts": touched, "parallelism": "single", "l2": l2}


def timed_ms(fn, n: int, stream, scrub=None) -> float:
    """Device milliseconds of n calls fn(0..n-1) on `stream`.  Without a scrub
    buffer: one event pair around all n calls.  With one: an event pair per
    call, and the buffer rewritten before each call, outside the pair, so that
    every call starts with nothing of the step in L2."""
    if scrub is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    pairs = []
    for i in range(n):
        scrub.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(i)
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs)


class ExpertSource:
    """Packed weights of chosen experts, as host arrays for the oracle.

    Either slices of device-resident weight tensors, or each expert
    regenerated by the seeded input generator (every expert has its own
    generator, so a subset comes out byte-identical to the full tensors made
    on the same kind of device).  Only the experts a token sample touches
    are ever copied to the host: the Kimi-K3-shaped layer holds 36.7 GB."""

    def __init__(self, cfg, W=None, device="cpu"):
        self.cfg, self.W, self.device = cfg, W, device

    def fetch(self, experts: np.ndarray):
        if self.W is not None:
            idx = torch.from_numpy(experts.astype(np.int64)).to(self.W[0].device)
            return [t.index_select(0, idx).cpu().numpy() for t in self.W]
        parts = [syn.make_expert(int(e), self.cfg.H, self.cfg.I, self.cfg.seed, self.device) for e in experts]
        out = [torch.stack([p[i] for p in parts]).cpu().numpy() for i in range(4)]
        del parts
        return out


def oracle_batch(hb, ids, w, src: ExpertSource, tokens: np.ndarray, E: int) -> float:
    """The oracle forward for `tokens` (routing given), using only the experts
    they touch (ids remapped to that compact list).  Returns the seconds the
    oracle call took (the weight fetch is not counted)."""
    import oracle as O

    sub = ids[tokens]
    ok = (sub >= 0) & (sub < E)
    used = np.unique(sub[ok])
    remap = np.full(E, -1, np.int64)
    remap[used] = np.arange(used.shape[0])
    rid = np.where(ok, remap[np.clip(sub, 0, E - 1)], -1).astype(np.int32)
    Wh = src.fetch(used)
    t0 = time.perf_counter()
    O.moe_forward(np.ascontiguousarray(hb[tokens]), rid, np.ascontiguousarray(w[tokens]), *Wh, want=("out",))
    return time.perf_counter() - t0


def cpu_baseline(cfg, hidden, ids_np, w_np, W, target_s=12.0):
    """The fp64 oracle on the host cores, on seeded batches of tokens until
    about target_s seconds of oracle time have run (routing excluded)."""
    import oracle as O

    threads = O.max_threads()
    batch = max(1, threads)
    hb = hidden.cpu().view(torch.int16).numpy().view(np.uint16)
    order = np.random.default_rng(1).permutation(cfg.T).astype(np.int32)
    src = ExpertSource(cfg, W=W)
    spent, done = 0.0, 0
    while done < cfg.T and (spent < target_s or done == 0):
        toks = np.sort(order[done:done + batch])
        spent += oracle_batch(hb, ids_np, w_np, src, toks, cfg.E)
        done += toks.shape[0]
    return {"value": done / spent, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of {cfg.T} tokens (seeded, in batches of {batch}, all {cfg.k} experts each) "
                      f"through the fp64 oracle forward ({spent:.1f} s of oracle time); routing excluded"}


# ------------------------------------------------------------------ arms
def run_reference(args, cfg):
    """The fp64 oracle as the reference arm: every step routes and runs the
    layer forward on a seeded token sample on the host cores."""
    import oracle as O

    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"   # the seeded input generator only
    hidden = syn.make_hidden(cfg.T, cfg.H, cfg.seed, device=gen_dev).cpu()
    logits = syn.make_logits(cfg.T, cfg.E, cfg.logits, cfg.seed, device=gen_dev).cpu()
    hb = hidden.view(torch.int16).numpy().view(np.uint16)
    lg = logits.numpy()
    ids_all, _ = O.route(lg, cfg.k)
    touched = int((np.bincount(ids_all.reshape(-1), minlength=cfg.E) > 0).sum())
    work = algorithmic(cfg, touched)
    full_bytes = cfg.E * (work["w13_bytes_per_expert"] + work["w2_bytes_per_expert"])
    if full_bytes <= 8e9:   # small enough to hold every expert on the host once
        W = syn.make_weights(cfg.E, cfg.H, cfg.I, seed=cfg.seed, device=gen_dev)
        src = ExpertSource(cfg, W=W)
    else:                   # regenerate only the experts each step's tokens touch
        src = ExpertSource(cfg, device=gen_dev)
    threads = O.max_threads()
    order = np.random.default_rng(0).permutation(cfg.T).astype(np.int32)

    cache = {}   # expert -> its four packed arrays, fetched once for the run

    def prepare(n):
        """The first n tokens of the seeded order, and the experts they touch (fetched once)."""
        toks = np.sort(order[:n])
        sub = ids_all[toks]
        used = np.unique(sub[(sub >= 0) & (sub < cfg.E)])
        missing = [int(e) for e in used if int(e) not in cache]
        if missing:
            got = src.fetch(np.array(missing, dtype=np.int64))
            for j, e in enumerate(missing):
                cache[e] = [got[i][j] for i in range(4)]
        return toks, used, [np.stack([cache[int(e)][i] for e in used]) for i in range(4)]

    def step(toks, used, Wh):
        """One timed step: route the sample's logits, then the layer forward on them (seconds)."""
        t0 = time.perf_counter()
        ids, w = O.route(lg[toks], cfg.k)
        remap = np.full(cfg.E, -1, np.int64)
        remap[used] = np.arange(used.shape[0])
        ok = (ids >= 0) & (ids < cfg.E)
        rid = np.where(ok, remap[np.clip(ids, 0, cfg.E - 1)], -1).astype(np.int32)
        O.moe_forward(np.ascontiguousarray(hb[toks]), rid, np.ascontiguousarray(w), *Wh, want=("out",))
        return time.perf_counter() - t0

    # size the sample so that the whole run takes about ref_budget_s of oracle time; the same sample (and
    # its experts, fetched once) serves every step, so the run's wall time stays close to that budget
    per_step = float(args.ref_budget_s) / max(1, args.steps + args.warmup)
    t_cal = step(*prepare(max(1, threads)))
    n_per_step = int(max(1, min(cfg.T, threads * per_step / max(t_cal, 1e-6))))
    sample_args = prepare(n_per_step)
    for _ in range(args.warmup):
        step(*sample_args)
    dt = sum(step(*sample_args) for _ in range(args.steps))
    value = n_per_step * args.steps / dt
    sample = (f"{n_per_step} of {cfg.T} tokens (seeded; the same sample every step), route + forward in fp64 on "
              f"the host cores ({threads} threads); {args.steps} steps, {dt:.1f} s of oracle time (input "
              f"generation and the one weight fetch excluded)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(cfg, touched, work),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ours(args, cfg, full: bool = True):
    """Device-resident timing, e2e with host copies, CUDA-graph replay, the
    roofline of the dominant kernel and (full=True) the CPU baseline."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    hidden = syn.make_hidden(cfg.T, cfg.H, cfg.seed, device=dev)
    logits = syn.make_logits(cfg.T, cfg.E, cfg.logits, cfg.seed, device=dev)
    W = syn.make_weights(cfg.E, cfg.H, cfg.I, seed=cfg.seed, device=dev)
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    route_out = (torch.empty(T, k, dtype=torch.int32, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
                 torch.empty(E + 1, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
                 torch.empty(T * k, dtype=torch.int32, device=dev))
    ws_route = torch.empty(int(kt.lib().kt_moe_route_workspace_bytes(T, E, k)), dtype=torch.uint8, device=dev)
    ws = torch.empty(kt.workspace_bytes(T, H, I, E, k), dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    # auto runs the separate launches (routing, then the forward on its permutation).  The single-launch
    # decode kernel is there with --path decode: measured on GB300 with every step starting from DRAM (the
    # L2 flush below), the separate launches were 0-8 us faster on the tiny and small layers and 10-17 us
    # faster replayed in a CUDA graph; on the 9 GB Kimi-shaped T=16 layer the separate GEMM launches are
    # faster too.
    use_decode = args.path == "decode"

    def step(h=hidden, lg=logits, o=out, s=stream):
        if use_decode:
            kt.decode(lg, h, k, *W, out=o, topk=route_out[:2], workspace=ws, stream=s)
        else:
            ids, w, offs, perm, inv = kt.route_permute(lg, k, out=route_out, workspace=ws_route, stream=s)
            kt.forward(h, ids, w, *W, out=o, workspace=ws, stream=s, routing=(offs, perm, inv))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert kt.read_device_error(ws) == 0, "device error word set during warm-up"
    if use_decode:   # the offsets live in the workspace on this path
        lay = kt.workspace_layout(T, H, I, E, k)
        offs = ws[lay["expert_offsets"]:lay["expert_offsets"] + 4 * (E + 1)].view(torch.int32)
        counts = (offs[1:] - offs[:-1]).cpu()
    else:
        counts = (route_out[2][1:] - route_out[2][:-1]).cpu()
    touched = int((counts > 0).sum())
    work = algorithmic(cfg, touched)
    scrub = torch.empty(L2_SCRUB_BYTES, dtype=torch.uint8, device=dev) if needs_l2_flush(work) else None

    # ---- timed region: device-resident inputs
    sampler = ClockSampler(dev)
    sampler.start()
    torch.cuda.synchronize(dev)
    launches0 = kt.kernel_launches()
    # inside the timed region only the roofline kernel (FC1) is bracketed by
    # events: each recorded stage adds two event records to every step
    kt.profile_enable(True, stages=("fc1",))
    elapsed_ms = timed_ms(lambda i: step(), args.steps, stream, scrub)
    launches = kt.kernel_launches() - launches0
    prof_fc1 = kt.profile_read()["fc1"]
    kt.profile_enable(False)
    clocks = sampler.stop()
    # per-stage breakdown: a few more steps with every stage bracketed, after the timed region
    n_prof = max(3, min(args.steps, 20))
    kt.profile_enable(True)
    for _ in range(n_prof):
        step()
    prof = kt.profile_read()
    kt.profile_enable(False)
    if use_decode:   # one kernel for the whole layer: its time is the step's
        prof_fc1 = (elapsed_ms, args.steps)
    ms_per_step = elapsed_ms / args.steps
    value = T / (ms_per_step / 1e3)

    # ---- e2e: host buffers in, host buffer out, copies inside the timed region.  As a serving
    # loop would run it: inputs and outputs double-buffered, host->device copies on one stream
    # and device->host copies on another, so step i's copies overlap steps i-1 and i+1.
    h_host = hidden.cpu().pin_memory()
    lg_host = logits.cpu().pin_memory()
    out_host = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h_dev = [torch.empty_like(hidden) for _ in range(2)]
    lg_dev = [torch.empty_like(logits) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        s_in.wait_event(ev_done[b])            # step i-2 finished reading this input buffer
        with torch.cuda.stream(s_in):
            h_dev[b].copy_(h_host, non_blocking=True)
            lg_dev[b].copy_(lg_host, non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])           # step i-2's result left this output buffer
        step(h_dev[b], lg_dev[b], out_dev[b])
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            out_host[b].copy_(out_dev[b], non_blocking=True)
        ev_out[b].record(s_out)

    # decode-sized steps (inputs under 1 MB) move a few KB: there the cross-stream events cost more
    # than they hide, and a single stream runs copy -> compute -> copy in order
    overlap = hidden.numel() * 2 >= (1 << 20) and scrub is None
    if not overlap:
        s_in = s_out = stream

        def e2e_step(i):   # noqa: F811 - the in-order variant
            b = i % 2
            h_dev[b].copy_(h_host, non_blocking=True)
            lg_dev[b].copy_(lg_host, non_blocking=True)
            step(h_dev[b], lg_dev[b], out_dev[b])
            out_host[b].copy_(out_dev[b], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if overlap:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        s_in.wait_stream(stream)               # the first copy starts inside the timed region
        for i in range(e2e_steps):
            e2e_step(i)
        stream.wait_stream(s_out)              # ... and the last result is on the host before it ends
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = ev0.elapsed_time(ev1) / e2e_steps
    else:
        e2e_ms = timed_ms(e2e_step, e2e_steps, stream, scrub) / e2e_steps
    last = (e2e_steps - 1) % 2
    assert torch.equal(out_host[last].view(torch.int16), out.cpu().view(torch.int16))

    # ---- the same step captured once in a CUDA graph and replayed (device-resident inputs)
    graph = None
    try:
        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            step(s=gstream)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        reps = max(3, min(args.steps, 50))
        g_ms = timed_ms(lambda i: g.replay(), reps, stream, scrub) / reps
        graph = {"value": T / (g_ms / 1e3), "unit": "tokens/s", "ms_per_step": g_ms, "replays": reps}
        del g
    except Exception as exc:  # noqa: BLE001 - reported, never fatal to the bench line
        graph = {"error": f"{type(exc).__name__}: {exc}"[:200]}

    # ---- roofline of the dominant kernel (FC1 grouped GEMM) and of the layer
    fc1_ms = prof_fc1[0] / max(1, prof_fc1[1])
    fc2_ms = prof["fc2"][0] / max(1, prof["fc2"][1])
    hbm = float(peaks["hbm_gbs"])
    mx_tflops = float(peaks["bf16_tflops"]) * FP8_OVER_BF16
    # the decode path's one kernel moves the whole layer's bytes
    dom_bytes = work["layer_bytes"] if use_decode else work["fc1_bytes"]
    fc1_gbs = dom_bytes / (fc1_ms / 1e3) / 1e9
    t_roof_ms = 1e3 * max(work["layer_flops"] / (mx_tflops * 1e12), work["layer_bytes"] / (hbm * 1e9))
    res = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8xmxfp4", "data": "synthetic",
        "config": config_block(cfg, touched, work),
        "e2e": {"value": T / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "copies": "overlapped (separate H2D and D2H streams, double-buffered)" if overlap else "in order",
                "h2d_bytes_per_step": hidden.numel() * 2 + logits.numel() * 4,
                "d2h_bytes_per_step": out.numel() * 2},
        "gpu_launches": int(launches),
        "graph": graph,
        "clocks": clocks,
        "roofline": {"bound": "hbm", "achieved": fc1_gbs, "peak": hbm, "unit": "GB/s", "frac": fc1_gbs / hbm,
                     "traffic": None if use_decode else fc1_traffic(cfg.name),
                     "kernel": "moe_decode_kernel (whole layer, one launch)" if use_decode
                     else "mx_gemm_kernel<SwiGLU> (FC1)",
                     "peak_source": f"{peak_src} hbm_gbs",
                     "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": fc1_ms},
        "path": "decode: one launch (route, permute, quantise, FC1, FC2, combine)" if use_decode
        else "route_permute + forward_routed (separate launches)",
        "layer_roofline": {"t_roof_ms": t_roof_ms, "frac": t_roof_ms / ms_per_step,
                           "bytes": work["layer_bytes"], "flops": work["layer_flops"],
                           "hbm_gbs": hbm, "mx_tflops": mx_tflops,
                           "peaks": f"{peak_src}: hbm_gbs; bf16_tflops x {FP8_OVER_BF16} (nominal fp8/bf16)"},
        "stage_ms": {name: (ms / max(1, n)) for name, (ms, n) in prof.items()},
        "stage_ms_note": f"CUDA events around every stage over {n_prof} steps after the timed region; "
                         "the roofline's FC1 time is measured inside it",
        "fc2_gbs": work["fc2_bytes"] / (fc2_ms / 1e3) / 1e9 if fc2_ms > 0 else None,
    }
    if full and not args.no_cpu_baseline:
        ids_np = route_out[0].cpu().numpy()
        w_np = route_out[1].cpu().numpy()
        res["cpu_baseline"] = cpu_baseline(cfg, hidden, ids_np, w_np, W)
    del W
    torch.cuda.empty_cache()
    return res


def secondary_summary(res: dict) -> dict:
    keep = ("value", "unit", "ms_per_step", "config", "e2e", "gpu_launches", "graph", "roofline", "layer_roofline",
            "stage_ms", "fc2_gbs", "clocks", "path")
    return {k: res[k] for k in keep if k in res}


def _h2d_best(pack, dst, stream, reps: int) -> float:
    """Best pinned host -> device copy rate (GB/s) of one pack over `reps` copies."""
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = 0.0
    for _ in range(reps):
        ev0.record(stream)
        dst.copy_(pack, non_blocking=True)
        ev1.record(stream)
        torch.cuda.synchronize()
        best = max(best, pack.numel() / (ev0.elapsed_time(ev1) / 1e3) / 1e9)
    return best


def run_layerwise(args, cfg):
    """Layerwise prefill over cfg.layers DSV4-shaped layers at T tokens.

    Expert weights live in pinned host memory: P distinct layer stores used
    cyclically (layer l streams store l mod P), so the host link moves one
    full 3.42 GB pack per layer while the pinned footprint stays P packs.
    The link's rate is the best of several pack copies taken before and after
    the timed prefills; the library's per-layer events give each layer's copy
    and compute busy times; the serialized control (upload -> compute ->
    synchronise per layer) is timed over the same number of steps."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    L, T, H, E, k, I = cfg.layers, cfg.T, cfg.H, cfg.E, cfg.k, cfg.I
    P = max(1, min(args.layer_stores, L))
    packs = []
    for i in range(P):
        W = syn.make_weights(E, H, I, seed=cfg.seed + 1000 * i, device=dev)
        packs.append(kt.Layerwise.pack(*[t.cpu() for t in W]))
        del W
    pack_bytes = kt.Layerwise.pack_bytes(H, I, E)
    hidden = syn.make_hidden(T, H, cfg.seed, device=dev)
    logits = [syn.make_logits(T, E, cfg.logits, seed=l, device=dev) for l in range(L)]
    lw = kt.Layerwise([packs[l % P] for l in range(L)], H, I, E, k, T_max=T, zero_copy=args.zero_copy)
    out = torch.empty_like(hidden)
    stream = torch.cuda.current_stream(dev)
    probe_dst = torch.empty(pack_bytes, dtype=torch.uint8, device=dev)
    link_before = max(_h2d_best(p, probe_dst, stream, 2) for p in packs)
    for _ in range(args.warmup):
        lw.prefill(hidden, logits, out=out)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev)
    sampler.start()
    launches0 = kt.kernel_launches()
    lw.enable_timing(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        lw.prefill(hidden, logits, out=out)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / args.steps
    launches = kt.kernel_launches() - launches0
    clocks = sampler.stop()
    per_layer = lw.timing()          # the last prefill's per-layer copy / compute busy times
    lw.enable_timing(False)
    link_after = max(_h2d_best(p, probe_dst, stream, 2) for p in packs)
    del probe_dst
    # serialized control over the same number of steps
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        lw.prefill(hidden, logits, out=out, serialized=True)
    torch.cuda.synchronize(dev)
    ms_serial = 1e3 * (time.perf_counter() - t0) / args.steps
    lw.close()
    h2d_gbs = max(link_before, link_after)
    link_gbs = L * pack_bytes / (ms / 1e3) / 1e9
    t_roof_ms = 1e3 * L * pack_bytes / (h2d_gbs * 1e9)
    touched = E
    work = algorithmic(cfg, touched)
    cfgb = config_block(cfg, touched, work)
    cfgb.update({"workload": f"layerwise: {L} layers x ({workload_desc(cfg)}), {P} distinct pinned host stores "
                             f"cycled", "layers": L, "pinned_host_GB": P * pack_bytes / 1e9,
                 "weights": "read in place from pinned host memory" if args.zero_copy else
                            "streamed into two device slots, double-buffered",
                 "l2": "inputs larger than L2 (3.42 GB streamed per layer)"})
    copy_ms = [c for c, _ in per_layer["layers"]]
    comp_ms = [m for _, m in per_layer["layers"]]
    return {
        "metric": METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8xmxfp4", "data": "synthetic", "config": cfgb,
        "e2e": {"value": T / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": L * pack_bytes,
                "d2h_bytes_per_step": 0},
        "gpu_launches": int(launches), "clocks": clocks,
        "roofline": {"bound": "h2d", "achieved": link_gbs, "peak": h2d_gbs, "unit": "GB/s",
                     "frac": link_gbs / h2d_gbs, "traffic": None,
                     "kernel": "host->device expert streaming" + (" (GEMM loads from host memory)" if args.zero_copy
                                                                   else " (copy engine)"),
                     "peak_source": "best pinned H2D copy of one pack, measured in this run before "
                                    f"({link_before:.1f} GB/s) and after ({link_after:.1f} GB/s) the timed prefills"},
        "layer_roofline": {"t_roof_ms": t_roof_ms, "frac": t_roof_ms / ms},
        "per_layer": {"copy_ms_mean": float(np.mean(copy_ms)) if copy_ms else None,
                      "compute_ms_mean": float(np.mean(comp_ms)) if comp_ms else None,
                      "copy_ms": copy_ms, "compute_ms": comp_ms, "span_ms": per_layer["span_ms"],
                      "note": "CUDA events the library records on the copy and compute streams, last timed prefill"},
        "serialized_control_ms": ms_serial,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="kimi_T8192", choices=sorted(syn.CONFIGS))
    ap.add_argument("--secondary", default="dsv4", help="a second workload measured after the first and nested "
                                                          "under 'secondary' ('none' to skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=("auto", "decode", "multi"), default="auto",
                    help="decode: the single-launch decode kernel (T * top_k <= 2048); auto and multi: "
                         "route_permute + forward_routed")
    ap.add_argument("--ref-budget-s", type=float, default=150.0)
    ap.add_argument("--layer-stores", type=int, default=4,
                    help="layerwise workload: distinct pinned host layer stores, cycled over the layers")
    ap.add_argument("--zero-copy", action="store_true",
                    help="layerwise workload: the GEMMs read each layer's experts in place from pinned host memory")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.gpus != 1 or world != 1:
        # one GPU only: the layer is not sharded and has no collective step
        if rank == 0:
            print(json.dumps({"metric": METRIC, "impl": args.impl, "n_gpus": max(args.gpus, world),
                              "unavailable": "single-GPU only: the MoE layer runs on one GPU with no sharding and "
                                             "no collective; multi-GPU runs are out of scope"}), flush=True)
        return
    cfg = syn.CONFIGS[args.workload]
    if args.impl == "reference":
        res = run_reference(args, cfg)
    elif cfg.layers > 1:
        res = run_layerwise(args, cfg)
    else:
        res = run_ours(args, cfg)
        if args.secondary not in ("none", "", args.workload):
            res["secondary"] = {args.secondary: secondary_summary(run_ours(args, syn.CONFIGS[args.secondary],
                                                                           full=False))}
    print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
