#!/usr/bin/env python
"""MoE-layer throughput at the Qwen3-30B-A3B shape on GB300, through the C ABI.

One step = one pass of the whole sparse MoE block (router GEMM, softmax / top-k /
renormalisation, expert histogram + scan + stable permutation, grouped SwiGLU
experts, weighted un-permute) over one batch of seeded synthetic tokens, as one
``moe_forward`` call captured in a CUDA graph.  Weights are random-init with the
model's shapes (no checkpoint); inputs are resident in HBM when timing starts.

The headline line is the decode workload (T=8, bf16).  In the same process, at one
GPU, every other workload (Zipf decode, 4-bit decode, the 4-layer prefill stack and
4-bit prefill) is measured the same way and reported under ``configs``, each with its
own roofline, clock record and per-op breakdown.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle (plain C
loops in double, on every host core) on the same workload instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode8|...] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/sec at Qwen3-30B-A3B shape; achieved HBM GB/s vs roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FALLBACK_L2_BYTES = 129 * 1024 * 1024

DESCR = {
    "tiny": "tiny MoE block fp32: T=16 H=64 E=8 k=2 I=32",
    "decode8": "Qwen3-30B-A3B MoE layer decode, bf16: T=8 H=2048 E=128 k=8 I=768, norm_topk",
    "decode64z": "Qwen3-30B-A3B MoE layer decode, bf16, Zipf(1.1) router bias: T=64 H=2048 E=128 k=8 I=768",
    "decode48q": "Qwen3-30B-A3B MoE layer decode, 4-bit codebook expert weights: T=48 H=2048 E=128 k=8 I=768",
    "prefill": "Qwen3-30B-A3B MoE layer prefill, bf16: 4 independent layers x T=4096 H=2048 E=128 k=8 I=768",
    "prefill4q": "Qwen3-30B-A3B MoE layer prefill, 4-bit codebook expert weights: T=4096 H=2048 E=128 k=8 I=768",
}
EXTRA_WORKLOADS = ("decode64z", "decode48q", "prefill", "prefill4q")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode8", choices=sorted(DESCR))
    ap.add_argument("--extras", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated workloads also measured at one GPU ('none' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--copies", type=int, default=0, help="weight copies to rotate (0 = automatic)")
    ap.add_argument("--layers", type=int, default=0, help="use only the first N layers (profiling; 0 = all)")
    ap.add_argument("--lora-unpacked", action="store_true",
                    help="with --entry lora: pass the fp32 adapters without a pack (CUDA-core adapter products)")
    ap.add_argument("--entry", choices=["forward", "rmsnorm", "lora"], default="forward",
                    help="moe_forward, moe_forward_rmsnorm (pre-router RMSNorm and residual fused in) or "
                         "moe_forward_lora (synthetic rank-16 fp32 adapters on the expert projections)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region (every 100 ms)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def src_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (every rank times the same number of steps)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, steps: int, ms_total: float) -> float:
    """Whole-job tokens/s: every replica processes its own batch each step (weak scaling)."""
    return world * tokens_per_step * steps / (ms_total / 1e3)


def layer_inputs(workload):
    import synth
    c = synth.WORKLOADS[workload]
    return [synth.make_inputs(workload, layer=l) for l in range(c["layers"])]


def expert_bytes_per_expert(inp):
    if inp.w == "q4":
        return 3 * inp.I * inp.H // 2 + 3 * inp.I * inp.H // inp.q_block * 2
    return 3 * inp.I * inp.H * (4 if inp.w == "f32" else 2)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_throughput(inp, seconds: float, threads: int):
    """Tokens/s of the oracle as it stands on `threads` host threads: every thread evaluates
    single tokens of the batch (token i, i + threads, ... cycling) through
    oracle.forward_tokens until the time is up.  The oracle's C call releases the GIL, so
    the threads run on separate cores.  Returns (tokens/s, tokens done, seconds)."""
    import numpy as np
    import oracle
    oracle.build()
    deadline = time.perf_counter() + seconds
    T = inp.T

    def worker(i):
        done, j = 0, i
        while True:
            oracle.forward_tokens(inp, np.array([j % T], dtype=np.int32))
            done += 1
            j += threads
            if time.perf_counter() >= deadline:
                return done

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(threads) as pool:
        n = sum(pool.map(worker, range(threads)))
    dt = time.perf_counter() - t0
    return n / dt, n, dt


def cpu_baseline(layers, seconds: float):
    """The oracle as it stands (plain C, double) on a bounded sample of the workload: single
    tokens of layer 0, on every host core, plus a single-thread figure."""
    inp = layers[0]
    cores = host_cores()
    v1, n1, d1 = oracle_throughput(inp, seconds / 4, 1)
    vn, nn, dn = oracle_throughput(inp, seconds, cores)
    return {"value": vn, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"oracle.forward_tokens on single tokens of layer 0 ({inp.T}-token batch, cycled), "
                      f"{nn} tokens in {dn:.1f} s on {cores} threads",
            "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{n1} tokens in {d1:.1f} s"}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    layers = layer_inputs(args.workload)
    oracle.build()
    inp = layers[0]
    cores = host_cores()
    t0 = time.perf_counter()
    oracle.forward_tokens(inp, np.array([0], dtype=np.int32))
    per_tok = max(time.perf_counter() - t0, 1e-4)
    # each step: n single-token evaluations spread over the host cores, bounded so that the
    # whole run stays within about two minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(inp.T * 8, budget * cores / per_tok)))
    toks = [np.array([i % inp.T], dtype=np.int32) for i in range(n)]

    def step(pool):
        list(pool.map(lambda t: oracle.forward_tokens(inp, t), toks))

    with cf.ThreadPoolExecutor(cores) as pool:
        for _ in range(args.warmup):
            step(pool)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(pool)
        dt = time.perf_counter() - t0
    value = args.steps * n / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCR[args.workload], "tokens_per_step": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} single-token evaluations per step (tokens of the {inp.T}-token batch, "
                                   f"cycled) through oracle.forward_tokens (C, double) on {cores} threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class Ctx:
    """What every measurement shares: device, stream, peaks, the library."""

    def __init__(self, args, world, local):
        import torch
        import top_routing_grouped_router_gb300 as moe
        from top_routing_grouped_router_gb300 import build as moe_build
        self.torch, self.moe = torch, moe
        self.args, self.world, self.local = args, world, local
        self.dev = torch.device("cuda", local)
        moe_build.build()
        self.peaks, self.peak_kind = load_peaks()
        props = torch.cuda.get_device_properties(self.dev)
        self.l2_bytes = int(getattr(props, "L2_cache_size", 0) or FALLBACK_L2_BYTES)
        self.l2_source = "device property" if getattr(props, "L2_cache_size", 0) else "fallback"
        self.stream = torch.cuda.Stream(device=self.dev)


def measure(ctx: Ctx, workload: str, steps: int, warmup: int, *, headline: bool):
    """One workload: graph-replayed steps (timed), then each entry point timed alone, the
    roofline of the grouped expert op, and (headline only) the end-to-end C-ABI run."""
    torch, moe, args, dev, stream = ctx.torch, ctx.moe, ctx.args, ctx.dev, ctx.stream
    import synth
    from top_routing_grouped_router_gb300.device import upload, to_device

    layers = layer_inputs(workload)
    if headline and args.layers > 0:
        layers = layers[:args.layers]
    inp0 = layers[0]
    T, H, E, k, I = inp0.T, inp0.H, inp0.E, inp0.k, inp0.I
    # enough weight copies that a replay never finds the previous replay's weights in L2
    per_copy = sum(expert_bytes_per_expert(l) * E for l in layers)
    n_copies = args.copies if (headline and args.copies > 0) else (1 if per_copy > 32 * ctx.l2_bytes else 3)
    dl = [[upload(l, dev) for l in layers] for _ in range(n_copies)]
    for c in range(1, n_copies):  # copies share x / router / bias with copy 0 (the same tokens each step)
        for l in range(len(layers)):
            dl[c][l].x, dl[c][l].w_router, dl[c][l].b_router = dl[0][l].x, dl[0][l].w_router, dl[0][l].b_router
    out_dt = dl[0][0].out_dtype()
    outs = [torch.empty((T, H), dtype=out_dt, device=dev) for _ in layers]
    wss = [d.new_workspace() for d in dl[0]]
    entry = args.entry if headline else "forward"

    gammas = [to_device(synth.make_norm_weight(l.H, l.act, seed=l.T, layer=i), dev) for i, l in enumerate(layers)]
    loras, lora_keep = [], []
    if entry == "lora":
        names = ("a_gate", "b_gate", "a_up", "b_up", "a_down", "b_down")
        for i, l in enumerate(layers):
            ad = synth.make_lora(l.E, l.H, l.I, rank=16, seed=l.T, layer=i)
            t = [to_device(ad[n], dev) for n in names]
            lo = moe.make_lora(ad["rank"], ad["scale"], *t)
            if l.w in ("bf16", "q4") and not args.lora_unpacked:
                # adapters are static: packed once, before timing, like the weights
                lo = moe.pack_lora(dl[0][i].shape, lo, device=dev)
                t.append(lo.pack_tensor)
            lora_keep.append(t)
            loras.append(lo)

    def forward(c, st=None):
        for l, L in enumerate(dl[c]):
            if entry == "lora":
                moe.moe_forward_lora(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4,
                                     loras[l], outs[l], workspace=wss[l], stream=st)
            elif entry == "rmsnorm":
                moe.moe_forward_rmsnorm(L.shape, L.x, gammas[l], 1e-6, L.w_router, L.b_router, L.w_gate, L.w_up,
                                        L.w_down, L.q4, outs[l], workspace=wss[l], stream=st)
            else:
                moe.moe_forward(L.shape, L.x, L.w_router, L.b_router, L.w_gate, L.w_up, L.w_down, L.q4, outs[l],
                                workspace=wss[l], stream=st)

    with torch.cuda.stream(stream):
        for c in range(n_copies):
            forward(c)
    torch.cuda.synchronize()
    graphs = []
    for c in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            forward(c)
        graphs.append(g)
    # the copies' forwards back to back in one graph, as a model replays its consecutive MoE
    # layers: each forward's first kernel overlaps the previous one's tail (programmatic
    # dependent launch) instead of waiting for a new graph launch
    chain = n_copies
    gchain = None
    if chain > 1:
        gchain = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gchain, stream=stream):
            for c in range(n_copies):
                forward(c)

    def run_steps(n):
        """Exactly n forwards: whole chains, then single-copy graphs for the rest."""
        if gchain is not None:
            for _ in range(n // chain):
                gchain.replay()
            for i in range(n % chain):
                graphs[i].replay()
        else:
            for i in range(n):
                graphs[i % n_copies].replay()

    # active experts (fixed by the seeded tokens) -> algorithmic bytes of the expert kernel
    counts = []
    for l, L in enumerate(dl[0]):
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        moe.moe_route(L.shape, L.x, L.w_router, L.b_router, ids, w, workspace=wss[l])
        counts.append(torch.bincount(ids.view(-1).long(), minlength=E).cpu().numpy())
    torch.cuda.synchronize()
    n_active = [int((c > 0).sum()) for c in counts]
    act_b = 2 if inp0.act == "bf16" else 4
    grouped_bytes = sum(na * expert_bytes_per_expert(l) + T * H * act_b + T * k * H * act_b
                        for na, l in zip(n_active, layers))
    step_bytes = grouped_bytes + sum(E * H * act_b + T * H * act_b for _ in layers)
    expert_flops = sum(2 * T * k * 3 * I * H for _ in layers)
    flops = expert_flops + sum(2 * T * H * E for _ in layers)

    clocks = ClockSampler(ctx.local)
    clocks.start()
    with torch.cuda.stream(stream):
        run_steps(max(3, warmup))
        # bring the GPU under load before the timed region so the clock samples mean something
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            run_steps(3 * n_copies)
            stream.synchronize()
    if ctx.world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        run_steps(steps)
        ev1.record(stream)
    torch.cuda.synchronize()
    if ctx.world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), ctx.world, dev)
    ms_step = ms_total / steps
    tokens_per_step = T * len(layers)
    value = job_throughput(ctx.world, tokens_per_step, steps, ms_total)

    # each entry point timed alone with events on its stream, eager launches back to back
    kt_steps = max(20, min(steps, 200))
    ids_b = [torch.empty((T, k), dtype=torch.int32, device=dev) for _ in layers]
    w_b = [torch.empty((T, k), dtype=torch.float32, device=dev) for _ in layers]
    cnt_b = [torch.empty(E, dtype=torch.int32, device=dev) for _ in layers]
    off_b = [torch.empty(E + 1, dtype=torch.int32, device=dev) for _ in layers]
    ord_b = [torch.empty(T * k, dtype=torch.int32, device=dev) for _ in layers]
    pos_b = [torch.empty(T * k, dtype=torch.int32, device=dev) for _ in layers]
    y_b = [torch.empty((T * k, H), dtype=out_dt, device=dev) for _ in layers]
    ops = ("route", "permute", "grouped_swiglu", "unpermute")
    kev = {o: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(kt_steps)] for o in ops}
    out_b = [torch.empty((T, H), dtype=out_dt, device=dev) for _ in layers]

    def timed(name, i, fn):
        if i >= 3:
            kev[name][i - 3][0].record(stream)
        fn()
        if i >= 3:
            kev[name][i - 3][1].record(stream)

    with torch.cuda.stream(stream):
        for i in range(kt_steps + 3):
            c = i % n_copies
            timed("route", i, lambda: [moe.moe_route(L.shape, dl[0][l].x, L.w_router, L.b_router, ids_b[l], w_b[l],
                                                     workspace=wss[l], stream=stream) for l, L in enumerate(dl[c])])
            timed("permute", i, lambda: [moe.moe_permute(L.shape, ids_b[l], cnt_b[l], off_b[l], ord_b[l], pos_b[l],
                                                         wss[l], stream=stream) for l, L in enumerate(dl[c])])
            timed("grouped_swiglu", i, lambda: [moe.moe_grouped_swiglu(L.shape, dl[0][l].x, off_b[l], ord_b[l],
                                                                       L.w_gate, L.w_up, L.w_down, L.q4, y_b[l],
                                                                       wss[l], stream=stream)
                                                for l, L in enumerate(dl[c])])
            timed("unpermute", i, lambda: [moe.moe_unpermute(L.shape, y_b[l], w_b[l], pos_b[l], out_b[l],
                                                             stream=stream) for l, L in enumerate(dl[c])])
    torch.cuda.synchronize()
    breakdown = {o: statistics.mean(a.elapsed_time(b) for a, b in kev[o]) * 1e3 for o in ops}
    k_ms = breakdown["grouped_swiglu"] / 1e3

    peaks = ctx.peaks
    tensor_bound = workload.startswith("prefill")
    peak_src = "measured (MEASURED_PEAKS.json)" if ctx.peak_kind == "measured" else "fallback"
    if tensor_bound:
        # the grouped op is timed on its own (eager launches of a few hundred microseconds):
        # the burst bf16 peak applies, and only the expert flops count (the op does no router GEMM)
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        achieved = expert_flops / (k_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{peak_src}, bf16 burst", "algorithmic_flops": expert_flops}
    else:
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        achieved = grouped_bytes / (k_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": peak_src}
    roof["kernel"] = "moe_grouped_swiglu (grouped SwiGLU expert kernels)"
    roof["kernel_ms"] = k_ms
    roof["algorithmic_bytes"] = grouped_bytes
    roof["traffic"] = None
    tr_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tr_path):
        tr = json.load(open(tr_path)).get(workload)
        if tr and tr.get("src_digest") == src_digest(tr["sources"]):
            roof["traffic"] = tr["dram_bytes_per_launch"]

    res = {
        "workload": DESCR[workload], "value": value, "unit": "tokens/s", "steps": steps, "ms_per_step": ms_step,
        "roofline": roof, "clocks": clk, "active_experts": n_active, "layers": len(layers),
        "weights": inp0.w, "T": T, "H": H, "E": E, "k": k, "I": I,
        "step_hbm_gbs": step_bytes / (ms_step / 1e3) / 1e9,
        "step_tflops": flops / (ms_step / 1e3) / 1e12,
        "l2": f"inputs larger than L2 ({ctx.l2_bytes / 2**20:.0f} MiB, {ctx.l2_source}): {n_copies} rotating "
              f"weight cop{'y' if n_copies == 1 else 'ies'} ({n_copies * per_copy / 1e9:.1f} GB)",
        "graph": (f"the {n_copies} copies' forwards back to back in one CUDA graph (consecutive MoE layers; "
                  f"programmatic dependent launch across them), single-forward graphs for a remainder"
                  if n_copies > 1 else "one CUDA graph per step"),
        "breakdown_us": {**breakdown, "note": "each entry point timed alone (eager launches, CUDA events)"},
        "gpu_launches_per_step": sum(moe.moe_forward_launches(L.shape) for L in dl[0]),
    }
    if tensor_bound:
        peak_s = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
        res["step_frac_of_sustained_bf16"] = res["step_tflops"] / peak_s

    if headline:
        res["e2e"] = end_to_end(ctx, layers, dl, outs, graphs, n_copies, steps)
        res["entry"] = entry
        res["n_copies"] = n_copies
        res["per_copy"] = per_copy
    del graphs, dl, wss, outs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, layers


def end_to_end(ctx, layers, dl, outs, graphs, n_copies, steps):
    """The same metric through the C ABI with HOST buffers: each step copies the step's tokens
    from pinned host memory, runs the block and copies the result back to pinned host memory.
    Decode batches use moe_graphs_run (the library's bucketed decode graphs: with pinned
    buffers one graph launch whose first kernel reads the step's rows from pinned host memory
    and whose last kernel writes the result there); larger batches copy around the block's
    graph replay."""
    torch, moe, dev, stream = ctx.torch, ctx.moe, ctx.dev, ctx.stream
    from top_routing_grouped_router_gb300.device import to_device
    T, H = layers[0].T, layers[0].H
    out_dt = outs[0].dtype
    x_host = [to_device(l.x, "cpu", pin=True) for l in layers]
    out_host = [torch.empty((T, H), dtype=out_dt, pin_memory=True) for _ in layers]
    e2e_steps = min(steps, 500)
    use_graph_api = len(layers) == 1 and T <= 64 and ctx.args.entry == "forward"
    if use_graph_api:
        dgs = [moe.DecodeGraphs(dl[c][0].shape, T, dl[c][0].w_router, dl[c][0].b_router, dl[c][0].w_gate,
                                dl[c][0].w_up, dl[c][0].w_down, dl[c][0].q4, device=dev, stream=stream)
               for c in range(n_copies)]
        run = lambda i: dgs[i % n_copies].run(T, x_host[0], out_host[0], stream=stream)
        how = "moe_graphs_run (C ABI) with pinned host x and out"
    else:
        def run(i):
            for l in range(len(layers)):
                dl[0][l].x.copy_(x_host[l], non_blocking=True)
            graphs[i % n_copies].replay()
            for l in range(len(layers)):
                out_host[l].copy_(outs[l], non_blocking=True)
        how = "pinned host copies around the moe_forward graph replay"
    with torch.cuda.stream(stream):
        for i in range(3):
            run(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            run(i)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    # the host result equals the device path's result on the same tokens
    with torch.cuda.stream(stream):
        graphs[(e2e_steps - 1) % n_copies].replay()
    torch.cuda.synchronize()
    same = all(torch.equal(out_host[l], outs[l].cpu()) for l in range(len(layers)))
    if use_graph_api:
        for g in dgs:
            g.close()
    bi = sum(x.numel() * x.element_size() for x in x_host)
    bo = sum(o.numel() * o.element_size() for o in out_host)
    return {"value": ctx.world * T * len(layers) / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms, "steps": e2e_steps, "how": how,
            "host_result_equals_device_result": bool(same)}


def run_ours(args, rank, world, local):
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ctx = Ctx(args, world, local)
    head, layers = measure(ctx, args.workload, args.steps, args.warmup, headline=True)
    inp0 = layers[0]
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if inp0.act == "bf16" else "f32",
        "data": "synthetic: seeded N(0,1) tokens, N(0,1/fan_in) random-init weights of the model's shapes",
        "config": {"workload": head["workload"],
                   "entry": {"forward": "moe_forward", "rmsnorm": "moe_forward_rmsnorm (pre-router RMSNorm + residual)",
                             "lora": "moe_forward_lora (rank-16 fp32 adapters on the expert projections"
                                      + (", packed: tensor-core adapter products)" if inp0.w == "bf16" and not args.lora_unpacked
                                         else ", packed: tensor-core adapter products)"
                                         if inp0.w == "q4" and not args.lora_unpacked
                                         else ", CUDA-core adapter products)")}[head["entry"]],
                   "T": head["T"], "H": head["H"], "E": head["E"], "k": head["k"], "I": head["I"],
                   "layers": head["layers"], "weights": head["weights"], "active_experts": head["active_experts"],
                   "l2": head["l2"], "l2_bytes": ctx.l2_bytes, "graph": head["graph"],
                   "step_hbm_gbs": head["step_hbm_gbs"], "step_tflops": head["step_tflops"],
                   "parallelism": f"replicas x{world}"},
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "breakdown_us": head["breakdown_us"],
        "clocks": head["clocks"],
    }
    extras = [] if args.extras.strip().lower() in ("", "none") else [w.strip() for w in args.extras.split(",")]
    if world == 1 and args.entry == "forward":
        configs = {}
        for wl in extras:
            if wl == args.workload:
                continue
            # a few hundred microseconds (decode) to 1.6 ms (prefill) per step
            st = max(50, min(args.steps, 500)) if not wl.startswith("prefill") else max(20, min(args.steps, 100))
            r, _ = measure(ctx, wl, st, max(3, args.warmup), headline=False)
            configs[wl] = r
        if configs:
            line["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(layers, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
