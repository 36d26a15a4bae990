#!/usr/bin/env python
"""Layer-end compress benchmark on GB300.

One step = one full layer-end compress (pass 1, pass 2 + pooling, per-head
top-k, gather) of one layer of the chosen workload, through the C ABI
(kvc_compress_layer).  Default workload: Mistral-7B layer shape at S=131072
(B=1, H_q=32, H_kv=8, D=128, W=64, K_l=4096, sink 4, recent 64, avgpool 7,
b_s 4096), seeded synthetic bf16 inputs drawn on the device.  Four distinct
layers' inputs (512 MiB of K+V each) are cycled, so every step reads inputs
larger than L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0).  Under torchrun each rank compresses its own
layers on its own GPU (independent replicas, no data-path collective).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "layer-end compress: prefix keys scored/s per KV head; HBM GB/s vs ~8 TB/s peak"
UNIT = "prefix keys scored/s (per KV head)"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", default="mistral128k")
    ap.add_argument("--layers", type=int, default=4, help="distinct layer inputs cycled")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-full-layer", action="store_true",
                    help="time the oracle on every KV head of layer 0 (a whole layer), whatever --cpu-seconds "
                         "says; for multi-layer workloads the N-layer time is extrapolated linearly")
    ap.add_argument("--path", choices=["two_pass", "rawdot_int8", "append_chunk", "overlap"], default="two_pass",
                    help="two_pass: the layer compress (default, the headline); rawdot_int8: the single-pass "
                         "INT8 raw inner-product scorer, then the same selection and gather; append_chunk: the "
                         "layer-major chunk append; overlap: the HeteroCache overlap coefficient")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override the workload's S (smaller profiling captures); 0 keeps it")
    return ap.parse_args(argv)


def config_of(args):
    from synth import get_config
    return get_config(args.config, **({"S": args.seq_len} if args.seq_len > 0 else {}))


# ---- replica bookkeeping (no CUDA needed; the multi-process CPU tests use it)
def replica_layer_ids(rank, n_local, n_layers):
    """Layers rank `rank` compresses: n_local distinct ones, disjoint across
    ranks while world * n_local <= n_layers."""
    return [(rank * n_local + l) % n_layers for l in range(n_local)]


def max_over_ranks(value, world, device=None):
    """The slowest rank's elapsed time (all_reduce MAX), or value at N=1."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_step, steps, ms):
    """Units processed by all ranks per second over the slowest rank's time."""
    return world * units_per_step * steps / (ms / 1e3)


def workload_desc(cfg):
    kl = f"K_l={cfg.K_l}" if not cfg.inverse_stability else f"K_l~1/s, {cfg.budget_frac:.0%} of S*H_kv"
    return (f"{cfg.name}: N={cfg.N} B={cfg.B} H_q={cfg.H_q} H_kv={cfg.H_kv} D={cfg.D} S={cfg.S} C={cfg.C} "
            f"W={cfg.W} {kl} sink={cfg.sink} recent={cfg.recent} avgpool={cfg.pool_k} b_s={cfg.b_s} "
            f"heavy_hitters={cfg.hh_frac:.0%}")


def budgets(cfg, K, layer):
    if not cfg.inverse_stability:
        return [cfg.K_l] * cfg.H_kv
    from synth import stability_scores
    s = stability_scores(cfg, layer).numpy()
    total = round(cfg.budget_frac * cfg.S * cfg.H_kv)
    rsz = min(cfg.sink, cfg.S) + min(cfg.recent, max(cfg.S - cfg.sink, 0))
    return K.kvc_budget_inverse_stability(s, total, rsz, cfg.S)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


NOMINAL_HBM_GBS = 7900.0   # HBM3e of one GB300, nominal


def oracle_sample(cfg, inp_cpu, heads, budget_s, K_l):
    """Time the CPU oracle on whole KV heads of one layer (bounded sample)."""
    from oracle import kvc_oracle as O
    keys, t_used, done = 0, 0.0, []
    for (b, h) in heads:
        t0 = time.perf_counter()
        O.compress_layer(inp_cpu["q"], inp_cpu["k"], inp_cpu["v"], K_l, cfg.sink, cfg.recent, cfg.pool_k,
                         heads=[(b, h)])
        t_used += time.perf_counter() - t0
        keys += cfg.S
        done.append((b, h))
        if t_used >= budget_s:
            break
    return keys / t_used, t_used, done


def run_reference(args):
    """The CPU oracle as the reference arm: each step a bounded sample, one KV
    head of the workload's layer.  The head is whole when K + W such steps fit
    the time budget; otherwise its first S_s keys, S_s halved until they fit,
    are taken as a prompt of S_s keys.  The oracle's arithmetic per key does
    not depend on S, but its dense logit arrays outgrow the caches as S grows,
    so a shortened head runs faster per key than a whole one."""
    import torch
    from synth import get_config, make_layer_inputs
    from oracle import kvc_oracle as O
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = config_of(args)
    S_s = cfg.S
    budget_total = 150.0
    inp = make_layer_inputs(cfg.with_(S=S_s, C=min(cfg.C, S_s)), 0)
    q, k, v = inp.q_win, inp.k, inp.v
    K_l = [min(cfg.K_l if not cfg.inverse_stability else int(0.3 * S_s), S_s)] * cfg.H_kv
    K_l = [max(x, cfg.sink + cfg.recent) for x in K_l]

    def step(i):
        b, h = i % cfg.B, i % cfg.H_kv
        O.compress_layer(q, k, v, K_l, cfg.sink, cfg.recent, cfg.pool_k, heads=[(b, h)])

    t0 = time.perf_counter()
    step(0)
    t_one = time.perf_counter() - t0
    # one timed step is a noisy estimate: keep a margin of 1.5x
    while S_s > 512 and 1.5 * t_one * (args.steps + args.warmup) > budget_total:
        S_s //= 2
        inp = make_layer_inputs(cfg.with_(S=S_s, C=min(cfg.C, S_s), W=min(cfg.W, S_s)), 0)
        q, k, v = inp.q_win, inp.k, inp.v
        K_l = [max(min(x, S_s), cfg.sink + cfg.recent) for x in K_l]
        t0 = time.perf_counter()
        step(0)
        t_one = time.perf_counter() - t0
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = args.steps * S_s / dt
    sample = (f"one KV head per step (cycling b, h) of layer 0, "
              + ("whole" if S_s == cfg.S else f"its first {S_s} keys as a prompt of {S_s}")
              + f"; dense fp64 softmax over G*W={cfg.GW} window rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(cfg), "sample_S": S_s},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_rawdot(args):
    """One step = INT8 raw-product scores, selection, gather over one layer
    (1 GPU).  Prints one JSON line like the headline's, with the scorer as
    the dominant kernel of the roofline."""
    import torch
    from attention_score_kv_gb300 import build as _b
    _b.build()
    import attention_score_kv_gb300.kvc as K
    from synth import make_layer_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cfg = config_of(args)
    layers = []
    for layer_id in replica_layer_ids(0, args.layers, cfg.N):
        inp = make_layer_inputs(cfg, layer_id, device=dev)
        kl = budgets(cfg, K, layer_id)
        k_out, v_out, pos, off = K.retained_outputs(cfg.B, cfg.H_kv, cfg.S, cfg.D, kl, device=dev)
        layers.append(dict(q=inp.q_win, k=inp.k, v=inp.v, K_l=kl, k_out=k_out, v_out=v_out, pos=pos, T=off[-1]))
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, max(max(L["K_l"]) for L in layers),
                     cfg.pool_k, device=dev)
    scores = torch.empty((cfg.B, cfg.H_kv, cfg.S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_prof = min(args.steps, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_prof)]

    def step(i, marks=False):
        L = layers[i % len(layers)]
        ev = evs[i] if marks else None
        if marks:
            ev[0].record(stream)
        K.kvc_score_rawdot_int8(L["q"], L["k"], cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, scores, ws,
                                stream=stream)
        if marks:
            ev[1].record(stream)
        K.kvc_select_topk(scores, cfg.B, cfg.H_kv, cfg.S, L["K_l"], cfg.sink, cfg.recent, L["pos"], ws,
                          stream=stream)
        if marks:
            ev[2].record(stream)
        K.kvc_gather(L["k"], L["v"], L["pos"], cfg.B, cfg.H_kv, cfg.S, cfg.D, L["K_l"], L["k_out"], L["v_out"],
                     L["pos"], stream=stream)
        if marks:
            ev[3].record(stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    K.kvc_check_status(stream)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.15)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    stage = [0.0, 0.0, 0.0]
    for i in range(n_prof):
        step(i, marks=True)
    torch.cuda.synchronize(dev)
    for i in range(n_prof):
        for t in range(3):
            stage[t] += evs[i][t].elapsed_time(evs[i][t + 1])
    K.kvc_check_status(stream)
    stage = [x / n_prof for x in stage]
    units = cfg.B * cfg.H_kv * cfg.S
    Tmean = sum(L["T"] for L in layers) / len(layers)
    kbytes = cfg.B * cfg.H_kv * cfg.S * cfg.D * 2
    hbm_peak, _, peak_kind = load_peaks()
    alg = [kbytes + cfg.B * cfg.H_q * cfg.W * cfg.D * 2 + 4 * units, 4 * units + 4 * cfg.B * Tmean,
           cfg.B * Tmean * (4 * cfg.D * 2 + 4)]
    dom = max(range(3), key=lambda t: stage[t])
    names = ["rawdot_int8", "select_topk", "gather"]
    achieved = alg[dom] / (stage[dom] / 1e3) / 1e9
    path_bytes = sum(alg)
    line = {
        "metric": METRIC, "value": job_throughput(1, units, args.steps, ms), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 scores, bf16 rows", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "path": "rawdot_int8 (HillInfer raw q.k, INT8 keys)",
                   "parallelism": "replicas x1",
                   "l2": f"inputs larger than L2: {len(layers)} distinct layers cycled"},
        "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": None, "peak_kind": peak_kind,
                     "alg_bytes_per_launch": alg[dom], "ms_per_launch": stage[dom]},
        "path_hbm_gbs": path_bytes / (ms / args.steps / 1e3) / 1e9,
        "stage_ms_per_launch": {n: round(t, 5) for n, t in zip(names, stage)},
        "gpu_launches": 4 * args.steps, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_next_rows(args):
    """Measurements of two "next" rows on one GPU: the layer-major chunk
    append (one step = all C-key chunks of one layer's K and V appended to
    the active buffers; bytes moved per second against the HBM peak) and the
    HeteroCache overlap coefficient (one step = one call over 256 pairs of
    4096-index sets; index bytes read per second).  One JSON line each."""
    import numpy as np
    import torch
    from attention_score_kv_gb300 import build as _b
    _b.build()
    import attention_score_kv_gb300.kvc as K
    from synth import make_layer_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    hbm_peak, _, peak_kind = load_peaks()

    def timed(fn, steps, warmup):
        for i in range(max(3, warmup)):
            fn(i)
        torch.cuda.synchronize(dev)
        K.kvc_check_status(stream)
        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.15)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        K.kvc_check_status(stream)
        return e0.elapsed_time(e1) / steps, clk

    if args.path == "append_chunk":
        cfg = config_of(args)
        nch = -(-cfg.S // cfg.C)
        srcs = []
        for layer_id in replica_layer_ids(0, min(args.layers, 2), cfg.N):
            inp = make_layer_inputs(cfg, layer_id, device=dev)
            srcs.append([(inp.k[:, :, j * cfg.C:(j + 1) * cfg.C].contiguous(),
                          inp.v[:, :, j * cfg.C:(j + 1) * cfg.C].contiguous()) for j in range(nch)])
            del inp
        k_act = torch.empty((cfg.B, cfg.H_kv, cfg.S, cfg.D), dtype=torch.bfloat16, device=dev)
        v_act = torch.empty_like(k_act)

        def step(i):
            for j, (kc, vc) in enumerate(srcs[i % len(srcs)]):
                K.kvc_append_chunk(kc, vc, cfg.B, cfg.H_kv, cfg.S, cfg.C, cfg.D, j, k_act, v_act, stream=stream)

        ms, clk = timed(step, args.steps, args.warmup)
        moved = 2 * 2 * cfg.B * cfg.H_kv * cfg.S * cfg.D * 2      # K and V, read once and written once
        gbs = moved / (ms / 1e3) / 1e9
        line = {
            "metric": "layer-major chunk append: bytes moved per second (K and V chunks into the active layer)",
            "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "path": f"append_chunk ({nch} chunks of C={cfg.C} per step)",
                       "parallelism": "replicas x1", "l2": "each step moves 1.07 GB, far above L2"},
            "roofline": {"bound": "hbm", "kernel": "append_chunk", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "traffic": None, "peak_kind": peak_kind,
                         "alg_bytes_per_launch": moved / nch, "ms_per_launch": ms / nch},
            "gpu_launches": nch * args.steps, "clocks": clk,
        }
    else:
        rng = np.random.default_rng(5)
        n_pairs, k_sel, S = 256, 4096, 131072

        def sets():
            out = []
            for _ in range(n_pairs):
                out.append(np.sort(rng.choice(S, k_sel, replace=False)).astype(np.int32))
            return out
        A, B = sets(), sets()
        off = np.arange(n_pairs + 1, dtype=np.int64) * k_sel
        a = torch.from_numpy(np.concatenate(A)).to(dev)
        b = torch.from_numpy(np.concatenate(B)).to(dev)
        a_off = torch.from_numpy(off).to(dev)
        b_off = a_off.clone()
        out = torch.empty(n_pairs, dtype=torch.float32, device=dev)
        ms, clk = timed(lambda i: K.kvc_overlap_coefficient(a, a_off, b, b_off, n_pairs, out, stream=stream),
                        args.steps, args.warmup)
        read = 2 * n_pairs * k_sel * 4
        gbs = read / (ms / 1e3) / 1e9
        line = {
            "metric": "HeteroCache overlap coefficient: index-set pairs per second",
            "value": n_pairs / (ms / 1e3), "unit": "pairs/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": {"workload": f"{n_pairs} pairs of ascending {k_sel}-index sets drawn from [0, {S})",
                       "path": "overlap", "parallelism": "replicas x1", "l2": f"{read / 1e6:.1f} MB of indices (in L2)"},
            "roofline": {"bound": "hbm", "kernel": "overlap", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "traffic": None, "peak_kind": peak_kind,
                         "alg_bytes_per_launch": read, "ms_per_launch": ms},
            "gpu_launches": args.steps, "clocks": clk,
        }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.path == "rawdot_int8":
        run_rawdot(args)
        return
    if args.path in ("append_chunk", "overlap"):
        run_next_rows(args)
        return
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from attention_score_kv_gb300 import build as _b
    _b.build()
    import attention_score_kv_gb300.kvc as K
    from synth import get_config, make_layer_inputs

    cfg = config_of(args)
    NL = args.layers
    layers = []
    for layer_id in replica_layer_ids(rank, NL, cfg.N):
        inp = make_layer_inputs(cfg, layer_id, device=dev)
        kl = budgets(cfg, K, layer_id)
        k_out, v_out, pos, off = K.retained_outputs(cfg.B, cfg.H_kv, cfg.S, cfg.D, kl, device=dev)
        layers.append(dict(id=layer_id, q=inp.q_win, k=inp.k, v=inp.v, K_l=kl, k_out=k_out, v_out=v_out,
                           pos=pos, T=off[-1]))
    kmax = max(max(L["K_l"]) for L in layers)
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, kmax, cfg.pool_k, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        L = layers[i % NL]
        K.kvc_compress_layer(cfg.N, L["id"], cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, L["K_l"],
                             cfg.sink, cfg.recent, cfg.pool_k, cfg.b_s, L["q"], L["k"], L["v"], L["k_out"],
                             L["v_out"], L["pos"], ws, stream=stream)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    K.kvc_check_status(stream)

    # ---- timed region: device-resident inputs
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.15)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    # Per-stage times from the library's events between its kernels, on a
    # separate run: an event between two kernels keeps the next one from
    # starting while the previous one drains, so these are whole-kernel
    # durations, and the timed run above does not carry them.
    K.kvc_profile_begin()
    for i in range(min(args.steps, 50)):
        step(i)
    torch.cuda.synchronize(dev)
    stage_ms, calls, launches = K.kvc_profile_end()
    launches = launches * args.steps // max(calls, 1)
    ms = max_over_ranks(ms, world, dev)
    if world > 1:
        dist.barrier()
    K.kvc_check_status(stream)

    units_per_step = cfg.B * cfg.H_kv * cfg.S
    value = job_throughput(world, units_per_step, args.steps, ms)

    # ---- roofline of the dominant kernel (algorithmic bytes per launch)
    hbm_peak, _, peak_kind = load_peaks()
    Tmean = sum(L["T"] for L in layers) / NL
    kbytes = cfg.B * cfg.H_kv * cfg.S * cfg.D * 2
    qbytes = cfg.B * cfg.H_q * cfg.W * cfg.D * 2
    ncand = cfg.B * cfg.H_kv * max(0, cfg.S - cfg.sink - cfg.recent)
    alg = {
        "pass1": kbytes + qbytes,
        "pass2_pool": kbytes + qbytes,
        "select_topk": 8 * ncand + 4 * cfg.B * Tmean,
        "gather": cfg.B * Tmean * (4 * cfg.D * 2 + 4),
    }
    names = K.STAGE_NAMES
    per_launch_ms = [x / max(calls, 1) for x in stage_ms]
    dom = max(range(len(names)), key=lambda i: per_launch_ms[i])
    achieved = alg[names[dom]] / (per_launch_ms[dom] / 1e3) / 1e9
    path_bytes = 2 * kbytes + 2 * qbytes + cfg.B * Tmean * (4 * cfg.D * 2 + 4)
    traffic = None
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tfile):
        try:
            tj = json.load(open(tfile))
            ent = tj.get(args.config, {}).get(names[dom])
            if ent and ent.get("source_digest") == _source_digest(names[dom]):
                traffic = ent["bytes_per_launch"]
        except (ValueError, KeyError):
            traffic = None
    roofline = {"bound": "hbm", "kernel": names[dom], "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "frac_of": f"the dominant kernel ({names[dom]}) alone",
                "traffic": traffic, "peak_kind": peak_kind,
                "alg_bytes_per_launch": alg[names[dom]], "ms_per_launch": per_launch_ms[dom]}
    stages = {n: round(t, 5) for n, t in zip(names, per_launch_ms)}
    path_gbs = path_bytes / (ms / args.steps / 1e3) / 1e9

    # ---- end to end: host buffers, H2D + compress + D2H inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        nl_e = min(2, NL)
        host = []
        for L in layers[:nl_e]:
            host.append(dict(q=L["q"].cpu().pin_memory(), k=L["k"].cpu().pin_memory(),
                             v=L["v"].cpu().pin_memory(),
                             ko=torch.empty(L["k_out"].shape, dtype=torch.bfloat16).pin_memory(),
                             vo=torch.empty(L["v_out"].shape, dtype=torch.bfloat16).pin_memory(),
                             po=torch.empty(L["pos"].shape, dtype=torch.int32).pin_memory()))
        # Two slots of device buffers (steps alternate), so a step never
        # overwrites what the previous one still reads.  Per step: Q and K go
        # up on the main stream, then V on a side stream (after K, so the
        # host link carries one copy at a time) while the scans run; only
        # the gather waits for V (kvc_compress_layer_deferred_v).  The
        # outputs come down on a third stream, overlapping the next step's
        # uploads.
        dev_in = [dict(q=torch.empty_like(layers[0]["q"]), k=torch.empty_like(layers[0]["k"]),
                       v=torch.empty_like(layers[0]["v"])) for _ in range(nl_e)]
        s_v = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        ev_k = [torch.cuda.Event() for _ in range(nl_e)]
        ev_v = [torch.cuda.Event() for _ in range(nl_e)]
        ev_done = [torch.cuda.Event() for _ in range(nl_e)]
        ev_out = [torch.cuda.Event() for _ in range(nl_e)]
        for e in ev_out:
            e.record(s_out)

        def e2e_step(i):
            p = i % nl_e
            H, L, Dv = host[p], layers[p], dev_in[p]
            stream.wait_event(ev_out[p])                 # slot p's outputs have been copied out
            Dv["q"].copy_(H["q"], non_blocking=True)
            Dv["k"].copy_(H["k"], non_blocking=True)
            ev_k[p].record(stream)
            s_v.wait_event(ev_k[p])                      # after K (and after the gather that last read slot p)
            with torch.cuda.stream(s_v):
                Dv["v"].copy_(H["v"], non_blocking=True)
            ev_v[p].record(s_v)
            K.kvc_compress_layer_deferred_v(cfg.N, L["id"], cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W,
                                            L["K_l"], cfg.sink, cfg.recent, cfg.pool_k, cfg.b_s, Dv["q"], Dv["k"],
                                            Dv["v"], L["k_out"], L["v_out"], L["pos"], ws, ev_v[p], stream=stream)
            ev_done[p].record(stream)
            s_out.wait_event(ev_done[p])
            with torch.cuda.stream(s_out):
                H["ko"].copy_(L["k_out"], non_blocking=True)
                H["vo"].copy_(L["v_out"], non_blocking=True)
                H["po"].copy_(L["pos"], non_blocking=True)
            ev_out[p].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(args.e2e_steps):
            e2e_step(i)
        stream.wait_stream(s_out)                        # the last outputs are on the host
        stream.wait_stream(s_v)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        ems = a0.elapsed_time(a1)
        ems = max_over_ranks(ems, world, dev)
        L0 = layers[0]
        e2e = {"value": job_throughput(world, units_per_step, args.e2e_steps, ems), "unit": UNIT,
               "h2d_bytes_per_step": (L0["q"].numel() + L0["k"].numel() + L0["v"].numel()) * 2,
               "d2h_bytes_per_step": (L0["k_out"].numel() + L0["v_out"].numel()) * 2 + L0["pos"].numel() * 4,
               "ms_per_step": ems / args.e2e_steps}
        K.kvc_check_status(stream)

    # ---- CPU baseline: the oracle on whole KV heads of layer 0 (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        L0 = layers[0]
        heads = [(b, h) for b in range(cfg.B) for h in range(cfg.H_kv)]
        inp_cpu = {"q": L0["q"].cpu(), "k": L0["k"].cpu(), "v": L0["v"].cpu()}
        budget_s = float("inf") if args.cpu_full_layer else args.cpu_seconds
        v_cpu, t_cpu, done = oracle_sample(cfg, inp_cpu, heads, budget_s, L0["K_l"])
        whole = len(done) == len(heads)
        cpu = {"value": v_cpu, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": (f"{'the whole layer: ' if whole else ''}{len(done)} KV head(s) of layer 0 "
                          f"({cfg.S} keys each, dense fp64 softmax over G*W={cfg.GW} rows), {t_cpu:.1f} s")}
        if whole:
            cpu["layer_s"] = t_cpu
            cpu["job_s"] = t_cpu * cfg.N
            cpu["job_s_is"] = ("measured (one layer)" if cfg.N == 1 else
                               f"extrapolated linearly from one measured layer to the {cfg.N} layers")

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {NL} distinct layers of "
                             f"{2 * kbytes / 2**20:.0f} MiB K+V cycled"},
            "roofline": roofline,
            "path_hbm_gbs": path_gbs, "path_alg_bytes_per_step": path_bytes,
            "path_frac_measured": path_gbs / hbm_peak, "path_frac_nominal": path_gbs / NOMINAL_HBM_GBS,
            "stage_ms_per_launch": stages,
            "gpu_launches": launches, "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# Sources behind each stage's kernels: a profiled traffic figure is only
# reported while these files are unchanged since the capture.
_STAGE_SOURCES = {
    "pass1": ["kvc_pass1_tc.cu", "kvc_scan_common.cuh", "kvc_tc.cuh", "kvc_device.cuh", "kvc_internal.cuh"],
    "pass2_pool": ["kvc_pass2_tc.cu", "kvc_scan_common.cuh", "kvc_tc.cuh", "kvc_device.cuh", "kvc_internal.cuh"],
    "select_topk": ["kvc_select.cu", "kvc_device.cuh", "kvc_internal.cuh"],
    "gather": ["kvc_select.cu", "kvc_device.cuh", "kvc_internal.cuh"],
}


def _source_digest(stage):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_score_kv_gb300", "csrc")
    for f in _STAGE_SOURCES[stage]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    main()
