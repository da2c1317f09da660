"""Benchmark of the NVFP4 MoE layer on GB300: one JSON line on stdout (rank 0).

A step is one layer call on one synthetic layer instance: for one token the routed decode
(ft_moe_nvfp4_decode_routed, routing inside the one launch); for several tokens the router
(ft_moe_route) + experts (ft_moe_nvfp4_decode, or ft_moe_nvfp4_prefill for the prefill
workload). The decode workloads rotate over distinct instances (weights far larger than L2,
so every call streams its experts from HBM). Exactly K steps are timed: CUDA graphs of whole
passes over the instances, then one of the remaining steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

The default run times the one-token 288-expert layer as the headline (K steps) and then, in
the same process and one after the other, the one-token 512-expert layer with its shared
expert, the 32-token decode batch and the 2048-token prefill, each with its own default step
count; those land in the line's "configs" object (µs per call, roofline, e2e, CPU oracle).
--only skips them. --gpus N without torchrun re-launches itself under torchrun with N ranks.

--impl reference times the CPU oracle (the plain float32 reference) on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 MoE layer µs/call & achieved HBM GB/s vs GB300 peak (batch 1–32)"
DEFAULT_WORKLOAD = "decode_t1_e288_k8_h3072_i1024"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NVFP4_BYTES_PER_ELEM = 0.5625       # 4-bit code + one E4M3 byte per 16 elements


# ----------------------------------------------------------------------- helpers
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed layer calls (default: about a quarter second of GPU time)")
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--instances", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=0,
                    help="streams the end-to-end steps take in turn (default 3)")
    ap.add_argument("--only", action="store_true",
                    help="time the --workload alone (no companion configs)")
    ap.add_argument("--unrouted", action="store_true",
                    help="one-token decode as ft_moe_route + ft_moe_nvfp4_decode (two launches) "
                         "instead of the routed call; the roofline then times the decode launch")
    return ap.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    hbm, bf16, src = FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(o, pre=""):
                if isinstance(o, dict):
                    for k, v in o.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = o
            walk(d)
            for k, v in flat.items():
                kl = k.lower()
                if isinstance(v, (int, float)) and "hbm" in kl and "gbs" in kl:
                    hbm, src = float(v), "measured"
                if isinstance(v, (int, float)) and kl.endswith("bf16_tflops"):
                    bf16 = float(v)
        except Exception:
            pass
    return hbm, bf16, src


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works.

    Started before the warm-up and stopped after the kernel replays, so that even a timed
    region of a fraction of a second falls inside a run of samples; __enter__ waits (up to
    5 s) for the first sample. summary() reports the samples taken between mark_start() and
    mark_end() (the timed region and the replays) when there are any, else all of them."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}",
                                          f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "20"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.t_start = time.monotonic()

    def mark_end(self):
        self.t_end = time.monotonic()

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.05)          # one more sample after the last replay
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [ln for t, ln in self.lines
                  if self.t_start is not None and self.t_end is not None
                  and self.t_start - 0.025 <= t <= self.t_end + 0.025]
        scope = "timed region and kernel replays"
        if not window:
            window = [ln for _, ln in self.lines]
            scope = "warm-up, timed region and kernel replays"
        sm, mx, reasons = [], None, set()
        for ln in window:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "window": scope}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def layer_bytes(spec, n_experts_touched: int) -> float:
    """Algorithmic HBM bytes of one layer call: every touched expert's NVFP4 W13 and W2
    (codes + block scales) and its two tensor scales, plus x, logits, gate and output."""
    per_expert = 3 * spec.H * spec.I * NVFP4_BYTES_PER_ELEM + 8
    n = n_experts_touched + (1 if spec.shared else 0)
    io = spec.T * spec.H * 2 * 2 + spec.T * spec.E * 4 + (spec.H * 2 if spec.shared else 0)
    return n * per_expert + io


def layer_flops(spec, n_pairs: int) -> float:
    return 2.0 * n_pairs * 3 * spec.H * spec.I


# ------------------------------------------------------------------ our implementation
def run_ours(args, spec, rank, world, local, cpu_seconds=20.0):
    import torch
    from nvfp4_mixture_experts_02_gb300 import ftmoe
    from synth.device import make_device_layer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    n_inst = args.instances or spec.instances
    prefill = spec.prefill
    t_setup = time.perf_counter()
    layers, exps, shs, wss, idxs, ws_ = [], [], [], [], [], []
    touched, pairs = [], []
    for inst in rank_instances(rank, n_inst):
        lay = make_device_layer(spec, instance=inst, device=dev)
        ex = ftmoe.NvFP4Experts(lay.w13, lay.s13, lay.g13, lay.w2, lay.s2, lay.g2)
        sh = None
        if lay.shared is not None:
            s = lay.shared
            sh = ftmoe.NvFP4Shared(s["w13"], s["s13"], s["g13"], s["w2"], s["s2"], s["g2"],
                                   s["gate"])
        idx = torch.empty((spec.T, spec.k), dtype=torch.int32, device=dev)
        w = torch.empty((spec.T, spec.k), dtype=torch.float32, device=dev)
        ftmoe.route(lay.logits, spec.k, idx, w)
        torch.cuda.synchronize()
        touched.append(int(torch.unique(idx).numel()))
        pairs.append(spec.T * spec.k)
        layers.append(lay)
        exps.append(ex)
        shs.append(sh)
        idxs.append((idx, w))
    ws = ftmoe.new_workspace(spec.T, spec.k, exps[0], spec.shared, prefill=prefill)
    outs = [torch.empty((spec.T, spec.H), dtype=torch.bfloat16, device=dev) for _ in range(n_inst)]
    call = ftmoe.prefill if prefill else ftmoe.decode
    # one-token decode: the routed call is one launch (the kernel routes the token itself),
    # so the call and the expert kernel are the same launch
    fused = not prefill and spec.T == 1 and not getattr(args, "unrouted", False)

    def step(i, with_route=True):
        lay = layers[i]
        idx, w = idxs[i]
        if fused:
            ftmoe.decode_routed(lay.x, lay.logits, spec.k, exps[i], shs[i],
                                limit=spec.swiglu_limit, out=outs[i], workspace=ws)
            return
        if with_route:
            ftmoe.route(lay.logits, spec.k, idx, w)
        call(lay.x, idx, w, exps[i], shs[i], limit=spec.swiglu_limit, out=outs[i], workspace=ws)

    setup_s = time.perf_counter() - t_setup
    # warm up eagerly (also sets kernel attributes outside capture)
    for i in range(min(n_inst, 3)):
        step(i)
    torch.cuda.synchronize()
    assert ftmoe.get_error(ws) == 0

    # exactly K timed steps (and W warm-up steps): q whole passes over the instances, one
    # CUDA graph per pass, then a graph of the first r = K mod n instances
    steps_done = max(1, args.steps)
    passes_k, rem_k = divmod(steps_done, n_inst)
    stream = torch.cuda.Stream(device=dev)

    def capture(n_steps, with_route=True):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_steps):
                    step(i, with_route)
        return g

    g_step = capture(n_inst) if passes_k else None
    g_dec = capture(n_inst, with_route=False) if passes_k else None
    g_step_r = capture(rem_k) if rem_k else None
    g_dec_r = capture(rem_k, with_route=False) if rem_k else None
    torch.cuda.synchronize()

    def run(g_pass, g_rem):
        for _ in range(passes_k):
            g_pass.replay()
        if g_rem is not None:
            g_rem.replay()

    # W warm-up steps in the same rotation, ending on the last instance, so the timed region
    # starts on the instance read longest ago (the rotated inputs are larger than L2)
    n_w = max(0, args.warmup)
    with ClockSampler(local) as clk:
        for j in range(n_w):
            step((j - n_w) % n_inst)
        torch.cuda.synchronize()
        barrier(world)

        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clk.mark_start()
        torch.cuda.synchronize()
        barrier(world)
        ev0.record()
        run(g_step, g_step_r)
        ev1.record()
        torch.cuda.synchronize()
        barrier(world)
        step_ms = ev0.elapsed_time(ev1)
        # the expert kernel's duration for the roofline: the median over at least 5 timed
        # replays of a graph of decode launches only (one per instance, cold L2 each time)
        g_roof, n_roof = (g_dec, n_inst) if g_dec is not None else (g_dec_r, rem_k)
        reps = max(5, min(31, int(0.25e6 / max(1.0, step_ms * 1e3 / steps_done * n_roof))))
        rep_ms = []
        for _ in range(reps):
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record()
            g_roof.replay()
            d1.record()
            torch.cuda.synchronize()
            rep_ms.append(d0.elapsed_time(d1))
        clk.mark_end()
        dec_ms = statistics.median(rep_ms) / n_roof * steps_done
    assert ftmoe.get_error(ws) == 0
    step_ms = max_over_ranks(step_ms, world)

    bytes_call = statistics.mean(layer_bytes(spec, t) for t in touched)
    flops_call = statistics.mean(layer_flops(spec, p) for p in pairs)
    us_call = step_ms * 1e3 / steps_done
    dec_us = dec_ms * 1e3 / steps_done
    total_bytes = bytes_call * steps_done * world
    gbs = total_bytes / (step_ms * 1e-3) / 1e9

    # end to end through the public API with host buffers (pinned), copies timed
    e2e = run_e2e(args, spec, layers, exps, shs, ws, dev, bytes_call, world)

    hbm, bf16, src = measured_peaks()
    traffic = measured_traffic(spec.name)
    if prefill:
        achieved = flops_call / (dec_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": bf16,
                "unit": "TFLOP/s", "frac": round(achieved / bf16, 4), "traffic": traffic,
                "peak_source": src, "us_per_launch": round(dec_us, 3),
                "replays": reps, "launches_per_replay": n_roof,
                "kernel": "ft_moe_nvfp4_prefill (plan, activations, W13 and W2 tcgen05 "
                          "grouped GEMMs, reduce; the whole call's time)",
                "hbm_bound_frac": round((bytes_call / (hbm * 1e9)) / (dec_us * 1e-6), 4)}
    else:
        achieved = bytes_call / (dec_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": src,
                "kernel": decode_kernel_name(spec, fused),
                "us_per_launch": round(dec_us, 3), "replays": reps,
                "launches_per_replay": n_roof}
    res = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": steps_done, "warmup": max(0, args.warmup), "ms_per_step": step_ms / steps_done,
        "us_per_call": round(us_call, 3), "tokens_per_s": round(spec.T * steps_done * world /
                                                                 (step_ms * 1e-3), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4/f16/f32",
        "data": "synthetic (seeded N(0,0.02) weights quantised to NVFP4, N(0,1) bf16 x)",
        "config": {"workload": spec.name, "T": spec.T, "E": spec.E, "k": spec.k, "H": spec.H,
                   "I": spec.I, "shared_expert": spec.shared, "instances": n_inst,
                   "l2": f"inputs larger than L2: {n_inst} distinct layer instances rotated",
                   "graph": "CUDA graphs: whole passes over the instances, then the rest",
                   "arith": ("NVFP4 weights (e2m1 x e4m3) as exact f16 products, f16 tcgen05 MMA, "
                             "f32 accumulate, bf16 in/out" if prefill else
                             "NVFP4 weights (e2m1 x e4m3), f16x2 FMA per 16-element block, "
                             "f32 accumulate, bf16 in/out"),
                   "bytes_per_call": round(bytes_call), "experts_touched_mean":
                   statistics.mean(touched)},
        "roofline": roof, "e2e": e2e,
        "gpu_launches": (6 if prefill else 1 if fused else 2) * steps_done,
        "setup_s": round(setup_s, 1),
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(spec, layers[:2], bytes_call, cpu_seconds)
    return res


def decode_kernel_name(spec, fused):
    if fused:
        return ("k_decode1 (ft_moe_nvfp4_decode_routed, one token: routing, W13+SwiGLU, "
                "W2+weighted sum in one launch)")
    if spec.T == 1:
        return "k_decode1 (ft_moe_nvfp4_decode, one token: W13+SwiGLU, W2+weighted sum)"
    return ("k_decode (ft_moe_nvfp4_decode: plan, W13+SwiGLU, W2+weighted sum in one "
            "launch)")


def measured_traffic(workload):
    """DRAM bytes per launch from profiles/dram_traffic.md (an ncu capture), or None when
    the table has no row for the workload or the kernel source changed since the capture."""
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    path = os.path.join(here, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) < 4 or cells[0] != workload:
            continue
        src = os.path.join(here, "nvfp4_mixture_experts_02_gb300", "csrc", cells[1])
        if not os.path.exists(src):
            return None
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return int(cells[3]) if sha == cells[2] else None
    return None


def run_e2e(args, spec, layers, exps, shs, ws, dev, bytes_call, world):
    """The same layer calls end to end through the host-buffer entry point
    (ft_moe_layer_from_host): every step copies its x and logits from pinned host memory,
    runs the layer and copies the output back to pinned host memory, one C call per step."""
    import torch
    from nvfp4_mixture_experts_02_gb300 import ftmoe
    n = min(len(layers), 48)
    hx = [torch.from_numpy(l.x_bits.view(np.int16).copy()).view(spec.T, spec.H).pin_memory()
          for l in layers[:n]]
    hl = [torch.from_numpy(np.ascontiguousarray(l.logits_np)).pin_memory() for l in layers[:n]]
    # streams take the steps in turn, each with its own device buffers and workspace, so one
    # step's copies overlap the neighbouring steps' kernels (with two, a step's input copy
    # waits behind the output copy of the step two before it, on the same buffers)
    nb = max(1, args.e2e_streams or 3)
    prefill = spec.prefill
    streams = [torch.cuda.Stream(device=dev) for _ in range(nb)]
    wss = [ws] + [ftmoe.new_workspace(spec.T, spec.k, exps[0], spec.shared, prefill=prefill)
                  for _ in range(nb - 1)]
    mk = lambda shape, dt: [torch.empty(shape, dtype=dt, device=dev) for _ in range(nb)]
    xd, ld, od = (mk((spec.T, spec.H), torch.bfloat16), mk((spec.T, spec.E), torch.float32),
                  mk((spec.T, spec.H), torch.bfloat16))
    idd, wd = mk((spec.T, spec.k), torch.int32), mk((spec.T, spec.k), torch.float32)
    houts = [torch.empty((spec.T, spec.H), dtype=torch.int16).pin_memory() for _ in range(nb)]
    torch.cuda.synchronize()

    def one(i, b):
        ftmoe.layer_from_host(hx[i], hl[i], spec.k, exps[i], shs[i], limit=spec.swiglu_limit,
                              out_host=houts[b], x_dev=xd[b], logits_dev=ld[b], out_dev=od[b],
                              topk_idx_dev=idd[b], topk_w_dev=wd[b], workspace=wss[b],
                              stream=streams[b])

    for i in range(min(n, 4)):
        one(i, i % nb)
    torch.cuda.synchronize()
    steps = max(n, min(args.steps, 4 * n))
    main = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    for st in streams:
        st.wait_stream(main)
    for s_ in range(steps):
        one(s_ % n, s_ % nb)
    for st in streams:
        main.wait_stream(st)
    e1.record(main)
    torch.cuda.synchronize()
    for w_ in wss:
        assert ftmoe.get_error(w_) == 0
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    return {"value": round(bytes_call * steps * world / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "us_per_call": round(ms * 1e3 / steps, 3),
            "h2d_bytes_per_step": spec.T * spec.H * 2 + spec.T * spec.E * 4,
            "d2h_bytes_per_step": spec.T * spec.H * 2, "streams": nb,
            "call": "ft_moe_layer_from_host (pinned host x and logits in, pinned host output "
                    "out, one C call per step)"}


# --------------------------------------------------------------------- CPU oracle arm
def oracle_call_seconds(spec, lay, tokens=None):
    from oracle import moe as om
    from synth.device import HostExperts
    host = HostExperts(lay)
    if tokens is None:
        tokens = np.arange(spec.T)
    idx = np.argsort(-lay.logits_np[tokens], axis=1, kind="stable")[:, :spec.k]
    for e in np.unique(idx):                  # fetch first: device reads are not timed
        host._fetch(int(e))
    sh = host.shared_host()
    t0 = time.perf_counter()
    om.moe_layer(lay.x_bits, lay.logits_np, spec.k, host, shared=sh, tokens=tokens)
    return time.perf_counter() - t0, len(tokens)


def cpu_baseline(spec, layers, bytes_call, seconds=20.0):
    """The oracle timed on the host cores on a bounded sample: whole calls for decode
    batches of up to 32 tokens, else the first tokens of a call (scaled to the whole call),
    until 2 calls per instance or `seconds` have been spent (at least one call)."""
    secs, calls = 0.0, 0
    tokens = None if spec.T <= 32 else np.arange(8)
    deadline = time.perf_counter() + seconds
    while calls < 2 * len(layers) and time.perf_counter() < deadline:
        s, ntok = oracle_call_seconds(spec, layers[calls % len(layers)], tokens)
        secs += s * (spec.T / ntok)            # scale a token sample to a whole call
        calls += 1
    per_call = secs / max(calls, 1)
    return {"value": round(bytes_call / per_call / 1e9, 4), "unit": "GB/s", "cores": host_threads(),
            "kind": "oracle", "us_per_call": round(per_call * 1e6, 1),
            "sample": f"{calls} layer calls of instances 0-{len(layers) - 1}"
                      + ("" if tokens is None else f" ({len(tokens)} of {spec.T} tokens, scaled)")
                      + "; numpy float32, BLAS threads default"}


def run_reference(args, spec, rank, world, local):
    if rank != 0:
        return None
    import torch
    from synth.device import make_device_layer
    torch.cuda.set_device(local)
    n_inst = min(args.instances or spec.instances, 4)
    layers = [make_device_layer(spec, instance=i) for i in range(n_inst)]
    torch.cuda.synchronize()
    tokens = None if spec.T <= 32 else np.arange(16)
    W = min(args.warmup, 2)          # the oracle is slow: a bounded warm-up
    for s in range(W):
        oracle_call_seconds(spec, layers[s % n_inst], tokens)
    total, ntoks = 0.0, 0
    K = max(1, min(args.steps, 20))
    for s in range(K):
        sec, nt = oracle_call_seconds(spec, layers[s % n_inst], tokens)
        total += sec * (spec.T / nt)
    per_call = total / K
    touched = [len(np.unique(np.argsort(-l.logits_np, axis=1, kind="stable")[:, :spec.k]))
               for l in layers]
    bytes_call = statistics.mean(layer_bytes(spec, t) for t in touched)
    v = bytes_call / per_call / 1e9
    sample = (f"{K} layer calls over instances 0-{n_inst - 1}"
              + ("" if tokens is None else f", {len(tokens)} of {spec.T} tokens per call, scaled"))
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": per_call * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": spec.name, "T": spec.T, "E": spec.E, "k": spec.k,
                       "H": spec.H, "I": spec.I, "shared_expert": spec.shared},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": host_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------------ plumbing
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """Max of a per-rank timing over all ranks (the slowest rank sets the job time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_threads():
    """Host threads the oracle's numpy/BLAS may use: the CPUs this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def rank_instances(rank: int, n_inst: int):
    """Layer instances a rank generates and times: ranks run independent replicas, each on
    its own disjoint set of instances (weak scaling, no collective on the data path)."""
    return [rank * n_inst + i for i in range(n_inst)]


DEFAULT_STEPS = {1: 24000, 32: 240, 2048: 40}   # by batch size T
# timed after the headline in a default run, one after the other (each freed before the next)
COMPANIONS = ["decode_t1_e512_k10_h4096_i1024_shared", "decode_t32_e512_k10_h4096_i1024_shared",
              "prefill_t2048_e512_k10_h4096_i1024"]
COMPANION_KEYS = ("value", "unit", "us_per_call", "tokens_per_s", "steps", "warmup",
                  "ms_per_step", "roofline", "e2e", "cpu_baseline", "clocks", "gpu_launches",
                  "config", "setup_s")


def default_steps(spec):
    return DEFAULT_STEPS.get(spec.T, 480)


def default_warmup(steps):
    return max(3, min(steps // 10, 480))


def spawn_ranks(n):
    """--gpus N outside torchrun: run this same command under torchrun with N ranks."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    args = parse()
    from synth import BY_NAME
    spec = BY_NAME[args.workload]
    rank, world, local = dist_env()
    if "RANK" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {world}", file=sys.stderr)
        sys.exit(2)
    explicit_steps = args.steps is not None
    if args.steps is None:
        args.steps = default_steps(spec)
    if args.warmup is None:
        args.warmup = default_warmup(args.steps)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        res = run_reference(args, spec, rank, world, local)
    else:
        res = run_ours(args, spec, rank, world, local)
        if args.workload == DEFAULT_WORKLOAD and not args.only:
            res["configs"] = run_companions(args, rank, world, local, explicit_steps)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_companions(args, rank, world, local, explicit_steps):
    """The other configs, each in turn with its own default steps (at most K when --steps K
    was given) and warm-up; the previous config's device memory is freed first."""
    import gc
    import torch
    from synth import BY_NAME
    out = {}
    for name in COMPANIONS:
        gc.collect()
        torch.cuda.empty_cache()
        spec = BY_NAME[name]
        a = argparse.Namespace(**vars(args))
        a.workload, a.instances, a.unrouted = name, None, False
        a.steps = default_steps(spec)
        if explicit_steps:
            a.steps = max(1, min(a.steps, args.steps))
        a.warmup = default_warmup(a.steps)
        r = run_ours(a, spec, rank, world, local, cpu_seconds=8.0)
        out[name] = {k: r[k] for k in COMPANION_KEYS if k in r}
        del r
    gc.collect()
    torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    main()
