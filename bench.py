"""Benchmark: routed bit-plane MoE layers on GB300.

One step = the whole hot path (router top-K -> permutation -> bit-plane expert
FFN -> fp16 shared FFN -> weighted combine) over one batch of T tokens.  The
default headline is the largest configuration: 32 Mixtral-8x7B-shaped layers
decoding 64 tokens per step, a seeded quarter of the (layer, expert) pairs
changing bitwidth by page-table unmap/remap every step.  Beside it, in the same
run ("sub_runs"): the single Mixtral-shaped layer at decode 1/8/64/256 and
prefill 4096 tokens, the 128-expert layer at decode 128 and prefill 8192, the
Qwen1.5-MoE-shaped layer at decode 1/8/64/256, and the throughput loss of
asynchronous paging.  Layer copies (same synthetic weights, distinct pages)
are visited round-robin so weights stream from HBM, not L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload W --tokens T] [--impl reference]

Prints one JSON line (rank 0).  With torchrun (N > 1) every rank runs an
independent replica of the layer on its own GPU ("replicas only": the path has
no exchange step); value = tokens of all ranks / max over ranks of the time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at 1 GB300; achieved HBM GB/s (decode) / tensor util (prefill)"

# name -> (description, default tokens, default layer copies)
WORKLOADS = {
    "qwen": ("qwen1.5-moe-a2.7b-shaped layer (d=2048, 60 experts ffn 1408 top-4, fp16 shared FFN 5632, "
             "Zipf(1.1) router bias, greedy floor-respecting bitwidth plan)", 64, 6),
    "mixtral": ("mixtral-8x7b-shaped layer (d=4096, 8 experts ffn 14336 top-2, bitwidths 6/5/4/3 cycled)", 4096, 2),
    "e128": ("128-expert layer (d=2816, ffn 704, top-8, Zipf(1.2) bias, 45@3 45@4 30@6 8@16 bits)", 8192, 2),
    "tiny": ("tiny layer (d=512, 8 experts ffn 1024 top-2, mixed 3/4/5/6/16 bits)", 16, 8),
    "sweep": ("32-layer mixtral-8x7b-shaped decode step (d=4096, 8 experts ffn 14336 top-2 per layer, "
              "bits [6,5,4,3,16][(e+l) mod 5], 2 MiB plane pages; every step a seeded 25% of the "
              "(layer, expert) pairs get a new bitwidth by page-table unmap / remap)", 64, 1),
}


# The headline: the largest configuration that runs on one GPU, 32
# Mixtral-shaped layers decoding 64 tokens per step with bitwidth changes.
DEFAULT_WORKLOAD = "sweep"


def _load_json(path):
    try:
        with open(path) as f:
            return json.load(f)
    except Exception:
        return None


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def build_workload(cfg_name="qwen", n_copies=6, seed=0, T=64, device="cuda", src=None, vmm=False):
    """Upload n_copies of one synthetic layer; returns a dict with host copies for the oracle.

    src: a layer of the same shape holding this config's experts at 16 bits
    (all six planes and the fp16 page); the copies then take device copies of
    them (pw_layer_copy_expert) instead of generating and uploading from the
    host.  The sweep's source layer holds exactly the Mixtral-shaped experts
    (same seeded codes and LUTs), so the Mixtral sub-runs are built from it.
    vmm: the pool is a virtual-memory pool over physical pages this caller
    creates (pw_pool_create_vmm), instead of one buffer."""
    import torch

    import any_precision_expert_gb300 as pw
    from synth import bits_plan, get_config, make_expert, make_router, make_shared

    cfg = get_config(cfg_name)
    bits = bits_plan(cfg, seed)
    wr, bias = make_router(cfg, seed)
    experts = None if src is not None else [make_expert(cfg, e, seed) for e in range(cfg.E)]
    shared = make_shared(cfg, seed)
    plane = 3 * cfg.d * cfg.f // 8
    page = 2 << 20
    per_layer = 0
    for b in bits:
        np_ = 6 if b == 16 else int(b)
        per_layer += np_ * (plane // page + 2) * page
        if b == 16:
            per_layer += (3 * cfg.d * cfg.f * 2 // page + 3) * page
    per_layer += cfg.E * (2 * cfg.f + cfg.d) * 240 + 3 * cfg.d * cfg.shared_ffn * 2 + 4 * page
    nbytes = n_copies * per_layer + (64 << 20)
    phys = None
    if vmm:
        from any_precision_expert_gb300.vmm import PhysicalPages
        phys = PhysicalPages((nbytes + page - 1) // page, page, torch.cuda.current_device())
        pool = pw.Pool.from_vmm_handles(phys.handles, page, torch.cuda.current_device())
    else:
        pool = pw.Pool(nbytes, page_bytes=page, device=device)
    layers = []
    for _ in range(n_copies):
        L = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize, cfg.shared_ffn)
        for e in range(cfg.E):
            if src is not None:
                L.copy_expert(e, src, e, int(bits[e]))
            else:
                ex = experts[e]
                L.load_expert(e, int(bits[e]), ex["code6"], ex["lut"], ex["w16"])
        if shared is not None:
            L.load_shared(shared)
        layers.append(L)
    wl = dict(cfg=cfg, name=cfg_name, seed=seed, bits=bits, wr=wr, bias=bias, experts=experts, shared=shared,
              pool=pool, phys=phys, layers=layers, wr_d=torch.from_numpy(wr).to(device),
              bias_d=torch.from_numpy(bias).to(device) if bias is not None else None, bufs=None)
    set_tokens(wl, T, device)
    return wl


def set_tokens(wl, T, device="cuda"):
    """Seeded inputs and device buffers of every layer copy for batches of T tokens."""
    import torch

    import any_precision_expert_gb300 as pw
    from synth import make_tokens

    cfg = wl["cfg"]
    wl["bufs"] = None  # the previous batch size's buffers go back to torch first
    wl["xs"] = [make_tokens(cfg, T, wl["seed"], stream=i) for i in range(len(wl["layers"]))]
    wl["xs_d"] = [torch.from_numpy(x).to(device) for x in wl["xs"]]
    wl["bufs"] = [pw.Buffers(L, T, device=device) for L in wl["layers"]]
    wl["T"] = T
    torch.cuda.synchronize()


def free_workload(wl):
    for L in wl["layers"]:
        L.destroy()
    wl["bufs"] = None
    wl["pool"].close()
    if wl.get("phys") is not None:
        wl["phys"].release()


def algorithmic_bytes(cfg, bits, offsets, T):
    """Bytes the method must move: (expert-FFN call, whole step).  The FFN call
    reads the weights of the routed experts at their bitwidth plus their LUT_b
    rows and the shared FFN; the step adds the router weights, x in and y out."""
    d, f = cfg.d, cfg.f
    n = np.diff(offsets)
    ffn = 0
    for e in range(cfg.E):
        if n[e] == 0:
            continue
        b = int(bits[e])
        ffn += 3 * d * f * 2 if b == 16 else 3 * d * f * b // 8 + (2 * f + d) * (1 << b) * 2
    shared = 3 * d * cfg.shared_ffn * 2
    router = d * cfg.E * 2
    io = 2 * T * d * 2
    return ffn + shared, ffn + shared + router + io


def _peaks():
    """(HBM GB/s, its source, 16-bit tensor TFLOP/s, its source)."""
    peaks = _load_json(os.path.join(ROOT, "MEASURED_PEAKS.json"))
    if peaks and peaks.get("hbm_gbs"):
        hbm, hbm_src = float(peaks["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    else:
        hbm, hbm_src = 6800.0, "fallback 6.8 TB/s"
    if peaks and peaks.get("bf16_tflops"):
        tc, tc_src = float(peaks["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops; fp16 runs at the bf16 rate)"
    else:
        tc, tc_src = 1900.0, "fallback 1.9 PFLOP/s"
    return hbm, hbm_src, tc, tc_src


def measure_steps(wl, K, W, stream, soak=0.0):
    """Time K decode/prefill steps of the workload's current batch size.

    W eager warm-up steps fix the routing of every layer copy (and with it
    the algorithmic bytes); then one CUDA graph of K steps, copies visited
    round-robin, with CUDA events (graph nodes, on the launching stream)
    around each expert-FFN call -- or around the whole-layer call when the
    step is the router plus one fused kernel.  `soak` seconds of untimed
    replays come first (the clock record of the headline).  Returns the
    total and per-call times with the bytes and FLOPs behind them."""
    import inspect

    import torch

    import any_precision_expert_gb300 as pw

    cfg, layers, bufs, xs_d, T = wl["cfg"], wl["layers"], wl["bufs"], wl["xs_d"], wl["T"]
    NL = len(layers)
    fused = _fused_step(cfg, T)
    # one router (layer copies) or one per layer (the sweep's layers)
    per_layer = isinstance(wl["wr_d"], list)
    wr_of = (lambda j: wl["wr_d"][j]) if per_layer else (lambda j: wl["wr_d"])
    bias_of = (lambda j: wl["bias_d"][j]) if per_layer else (lambda j: wl["bias_d"])
    bits_of = (lambda j: wl["bits"][j]) if per_layer else (lambda j: wl["bits"])

    with torch.cuda.stream(stream):
        for i in range(max(W, NL)):
            j = i % NL
            pw.moe_forward_fused(layers[j], xs_d[j], wr_of(j), bias_of(j), bufs[j], stream=stream)
    torch.cuda.synchronize()
    ffn_bytes, step_bytes = [], []
    for j in range(NL):
        counts = np.bincount(bufs[j].idx[:T].cpu().numpy().reshape(-1), minlength=cfg.E)
        off = np.concatenate([[0], np.cumsum(counts)])
        fb, sb = algorithmic_bytes(cfg, bits_of(j), off, T)
        ffn_bytes.append(fb)
        step_bytes.append(sb)

    external = "external" in inspect.signature(torch.cuda.Event.__new__).parameters

    def mk_event():
        return torch.cuda.Event(enable_timing=True, external=True) if external else \
            torch.cuda.Event(enable_timing=True)

    ev_a = [mk_event() for _ in range(K)]
    ev_b = [mk_event() for _ in range(K)]

    def part_a(j):
        if not fused:
            L, b, x = layers[j], bufs[j], xs_d[j]
            L.route_topk(x, wr_of(j), bias_of(j), T, b.idx, b.w, None, stream)
            L.permute(b.idx, T, x, b.offsets, b.perm_src, b.inv_slot, b.x_perm, b.ws, stream)

    def part_f(j):
        L, b, x = layers[j], bufs[j], xs_d[j]
        if fused:
            L.forward(x, wr_of(j), bias_of(j), T, b.idx, b.w, b.y, b.fws, stream)
        else:
            L.moe_ffn(x, b.x_perm, b.offsets, T, b.y_perm, b.y_shared if cfg.shared_ffn else None, b.ws, stream)

    def part_c(j):
        if not fused:
            L, b = layers[j], bufs[j]
            L.combine(b.y_perm, b.inv_slot, b.w, T, b.y_shared if cfg.shared_ffn else None, b.y, stream)

    if external:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                j = i % NL
                part_a(j)
                ev_a[i].record(stream)
                part_f(j)
                ev_b[i].record(stream)
                part_c(j)

        def region():
            g.replay()
    else:
        graphs = []
        for j in range(NL):
            trio = []
            for part in (part_a, part_f, part_c):
                gg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gg, stream=stream):
                    part(j)
                trio.append(gg)
            graphs.append(trio)

        def region():
            torch.cuda._sleep(int(60e6))  # hold the GPU while the host queues the region
            for i in range(K):
                ga, gf, gc = graphs[i % NL]
                ga.replay()
                ev_a[i].record(stream)
                gf.replay()
                ev_b[i].record(stream)
                gc.replay()
    torch.cuda.synchronize()
    t_soak = time.time()
    while time.time() - t_soak < soak:
        with torch.cuda.stream(stream):
            region()
        torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0.record(stream)
        region()
        t1.record(stream)
    torch.cuda.synchronize()
    call_ms = [ev_a[i].elapsed_time(ev_b[i]) for i in range(K)]
    return {"ms": t0.elapsed_time(t1), "K": K, "NL": NL, "fused": fused, "external": external,
            "call_ms": sum(call_ms) / K,
            "ffn_bytes": sum(ffn_bytes[i % NL] for i in range(K)) / K,
            "step_bytes": sum(step_bytes[i % NL] for i in range(K)) / K,
            "ffn_flops": 2.0 * T * 3 * cfg.d * (cfg.K * cfg.f + cfg.shared_ffn)}


def roofline_of(m, cfg, T):
    """Roofline of the timed call: HBM for decode batches (algorithmic bytes of
    the call over its time), 16-bit tensor for prefill-sized ones."""
    hbm, hbm_src, tc, tc_src = _peaks()
    call_bytes = m["step_bytes"] if m["fused"] else m["ffn_bytes"]
    call_s = m["call_ms"] * 1e-3
    gbs = call_bytes / call_s / 1e9
    tflops = m["ffn_flops"] / call_s / 1e12
    name = ("whole-layer call pw_moe_forward (one persistent kernel: router, permutation, routed experts, "
            "shared FFN, combine)" if m["fused"] else "expert FFN call pw_moe_ffn (routed experts + shared FFN)")
    if T * cfg.K / cfg.E >= 256:  # tokens per expert: prefill-sized, the tensor pipe bounds it
        return {"kernel": name, "bound": "tensor", "achieved": tflops, "peak": tc, "unit": "TFLOP/s",
                "frac": tflops / tc, "algorithmic_flops_per_launch": m["ffn_flops"],
                "algorithmic_bytes_per_launch": m["ffn_bytes"], "hbm_GBps": gbs, "avg_launch_ms": m["call_ms"],
                "peak_source": tc_src}
    return {"kernel": name, "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
            "algorithmic_bytes_per_launch": call_bytes, "TFLOPs": tflops, "avg_launch_ms": m["call_ms"],
            "peak_source": hbm_src}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def rank_max(v, ws, device):
    """Max of v over the ranks of the process group (the job's time is the
    slowest rank's)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank, ws, seconds_max):
    """Whole-job throughput: the tokens of all ranks over the slowest rank's time."""
    return ws * tokens_per_rank / seconds_max


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import any_precision_expert_gb300 as pw

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    T, K, W = args.tokens, args.steps, args.warmup
    wl = build_workload(args.workload, n_copies=args.copies, T=T)
    cfg, layers, bufs = wl["cfg"], wl["layers"], wl["bufs"]
    NL = len(layers)
    stream = torch.cuda.Stream()

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    m = measure_steps(wl, K, W, stream, soak=args.soak)
    barrier()
    clk = clocks.stop()
    ms_max = rank_max(m["ms"], ws, "cuda")
    fused = m["fused"]

    # end to end through the public API with pinned host buffers: every step
    # copies its input in and its result out; the next step is enqueued
    # before the host waits for the previous result (two steps in flight)
    x_host = [torch.from_numpy(x).pin_memory() for x in wl["xs"]]
    y_host = [torch.empty((T, cfg.d), dtype=torch.float16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty((T, cfg.d), dtype=torch.float16, device="cuda") for _ in range(2)]
    y_done = [torch.cuda.Event() for _ in range(2)]
    KE = min(K, args.e2e_steps)
    barrier()
    te = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(KE + 1):
            if i < KE:
                j, b = i % NL, i & 1
                x_dev[b].copy_(x_host[j], non_blocking=True)
                y = pw.moe_forward_fused(layers[j], x_dev[b], wl["wr_d"], wl["bias_d"], bufs[j], stream=stream)
                y_host[b].copy_(y, non_blocking=True)
                y_done[b].record(stream)
            if i > 0:
                y_done[(i - 1) & 1].synchronize()  # step i - 1's result is on the host
    barrier()
    e2e_s = rank_max(time.perf_counter() - te, ws, "cuda")

    paging = measure_paging(wl, stream, args.paging) if args.paging > 0 else None
    roof = roofline_of(m, cfg, T)
    roof["traffic"] = _traffic_from_profile(args.workload, T)
    ok = all(L.check_device() == 0 for L in layers)

    out = None
    if rank == 0:
        cpu = cpu_baseline(wl, seconds=args.cpu_seconds) if (ws == 1 and args.cpu_seconds > 0) else None
        out = {
            "metric": METRIC,
            "value": job_value(T * K, ws, ms_max * 1e-3),
            "unit": "tokens/s",
            "n_gpus": ws,
            "steps": K,
            "warmup": W,
            "ms_per_step": ms_max / K,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16",
            "data": "synthetic",
            "config": {
                "workload": f"{WORKLOADS[args.workload][0]}, {T} tokens per step",
                "tokens_per_step": T,
                "bits_plan": {str(b): int((wl["bits"] == b).sum()) for b in (3, 4, 5, 6, 16)},
                "layer_copies": NL,
                "l2": f"inputs larger than L2: {NL} layer copies visited round-robin "
                      f"({m['step_bytes'] * (NL - 1) / 1e6:.0f} MB streamed between reuses of a copy)",
                "timing": ("one CUDA graph of K steps with timed event nodes" if m["external"] else
                           "three CUDA graphs per step, queued ahead of the GPU") + "; CUDA events on the launching stream",
                "step_algorithmic_bytes": m["step_bytes"],
                "hbm_GBps_step": m["step_bytes"] / ((ms_max / K) * 1e-3) / 1e9,
                "parallelism": "replicas" if ws > 1 else "single GPU",
                "device_errors": not ok,
            },
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": ws * T * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": T * cfg.d * 2,
                    "d2h_bytes_per_step": T * cfg.d * 2, "steps": KE,
                    "note": "public API (pw_moe_forward) per step: pinned H2D of x, layer, D2H of y, host wait for y; two steps in flight (step i+1 enqueued before the host waits for step i)"},
            "gpu_launches": _launches_per_step(cfg, T) * K,
            "clocks": clk,
        }
        if paging is not None:
            out["config"]["paging"] = paging
    free_workload(wl)
    if rank == 0 and args.sub_runs and ws == 1:
        out["sub_runs"] = sub_runs(stream)
    if ws > 1:
        dist.destroy_process_group()
    return out


# The other workloads of the layer's configurations, measured in the same run
# beside the headline: every decode batch size and prefill size they name.
SUB_RUNS = (("mixtral", 2, (1, 8, 64, 256, 4096), False),
            ("mixtral", 2, (64,), True),  # the same layer on the virtual-memory page table
            ("e128", 2, (128, 8192), False),
            ("qwen", 6, (1, 8, 64, 256), False))


def sub_runs(stream, src=None, steps_decode=50, steps_prefill=10, warmup=3, paging_steps=48):
    """One record per (workload, batch size): tokens/s and the roofline of the
    timed call, plus the throughput loss of asynchronous paging on the
    Qwen-shaped layer.  src: the sweep's source layer (Mixtral-shaped experts
    at 16 bits) to copy the Mixtral layers from."""
    recs = []
    for name, copies, Ts, vmm in SUB_RUNS:
        wl = build_workload(name, n_copies=copies, T=Ts[0], src=src if name == "mixtral" else None, vmm=vmm)
        cfg = wl["cfg"]
        for T in Ts:
            if T != wl["T"]:
                set_tokens(wl, T)
            prefill = T * cfg.K / cfg.E >= 256
            m = measure_steps(wl, steps_prefill if prefill else steps_decode, warmup, stream)
            roof = roofline_of(m, cfg, T)
            recs.append({"workload": name + (" (virtual-memory page table)" if vmm else ""), "tokens": T,
                         "kind": "prefill" if prefill else "decode",
                         "value": T * m["K"] / (m["ms"] * 1e-3), "unit": "tokens/s",
                         "ms_per_step": m["ms"] / m["K"], "steps": m["K"], "layer_copies": m["NL"],
                         "timed_call": "pw_moe_forward (one fused kernel, router included)" if m["fused"] else "pw_moe_ffn",
                         "call_ms": m["call_ms"],
                         "roofline": {k: roof[k] for k in ("bound", "achieved", "unit", "peak", "frac")},
                         "hbm_GBps_call": roof.get("hbm_GBps", roof["achieved"] if roof["bound"] == "hbm" else None),
                         "device_errors": not all(L.check_device() == 0 for L in wl["layers"])})
        if name == "qwen" and paging_steps > 0:
            set_tokens(wl, 64)
            recs.append({"workload": name, "tokens": 64, "kind": "paging",
                         "paging": measure_paging(wl, stream, paging_steps)})
        free_workload(wl)
    return recs


def _decode_plan(cfg, T):
    """The library's split of a T-token batch (pw_decode_plan): routed and
    shared decode thresholds, and whether pw_moe_forward takes the fused step."""
    import any_precision_expert_gb300 as pw
    return pw.decode_plan(cfg.d, cfg.f, cfg.E, cfg.K, T, cfg.shared_ffn)


def _fused_step(cfg, T):
    """pw_moe_forward runs one fused kernel (router included) for small decode batches."""
    return _decode_plan(cfg, T)["fused"]


def _launches_per_step(cfg, T):
    """Kernels one step launches: one fused kernel (router included) when
    every group is decode-sized; otherwise the router, the permutation
    (histogram + scatter for more than 1024 slots, or one kernel), row
    gather, the persistent decode kernel, the tcgen05 GEMM pair for experts
    above the token threshold and for a shared FFN above its own, and the
    combine."""
    plan = _decode_plan(cfg, T)
    thr, thr_s = plan["routed_max"], plan["shared_max"]
    if plan["fused"]:
        return 1
    S = T * cfg.K
    n = 1 + (2 if S > 1024 else 1) + 1
    n += 1
    if T > thr:
        n += 2
    if cfg.shared_ffn and T > thr_s:
        n += 2
    return n + 1


# ---------------------------------------------------------------------------
# 32-layer decode sweep with bitwidth changes between steps
# ---------------------------------------------------------------------------

def _expert_pages(cfg, b, page):
    plane = 3 * cfg.d * cfg.f // 8
    n = (6 if b == 16 else b) * (plane // page + 3)
    if b == 16:
        n += 3 * cfg.d * cfg.f * 2 // page + 4
    return n


def build_sweep(T, seed=0, device="cuda"):
    """32 layers built from one uploaded set of experts: a source layer holds the
    8 synthetic experts at 16 bits (six planes + fp16 page) and every layer gets
    device copies of them at its initial bitwidths (distinct pages, so each
    layer streams its own bytes); routers and inputs differ per layer."""
    import torch

    import any_precision_expert_gb300 as pw
    from synth import bits_plan, get_config, make_expert, make_router, make_tokens

    cfg = get_config("sweep")
    page = 2 << 20
    n_layers = cfg.n_layers
    init = [bits_plan(cfg, seed, layer=l) for l in range(n_layers)]
    lut = cfg.E * (2 * cfg.f + cfg.d) * 240
    pages = cfg.E * _expert_pages(cfg, 16, page)
    for l in range(n_layers):
        pages += sum(_expert_pages(cfg, int(b), page) for b in init[l])
    nbytes = pages * page + (n_layers + 1) * (lut + 4 * page) + (256 << 20)
    pool = pw.Pool(nbytes, page_bytes=page, device=device)
    src = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize, 0)
    experts = []
    for e in range(cfg.E):
        ex = make_expert(cfg, e, seed, layer=0, with_w16=True)
        src.load_expert(e, 16, ex["code6"], ex["lut"], ex["w16"])
        experts.append({"code6": ex["code6"], "lut": ex["lut"], "w16": ex["w16"]})
    layers, wr, bias, xs = [], [], [], []
    for l in range(n_layers):
        L = pw.Layer(pool, cfg.d, cfg.f, cfg.E, cfg.K, cfg.renormalize, 0)
        for e in range(cfg.E):
            L.copy_expert(e, src, e, int(init[l][e]))
        layers.append(L)
        w, bb = make_router(cfg, seed, layer=l)
        wr.append(w)
        bias.append(bb)
        xs.append(make_tokens(cfg, T, seed, layer=l))
    return dict(cfg=cfg, pool=pool, src=src, layers=layers, init=init, experts=experts, wr=wr, bias=bias, xs=xs,
                wr_d=[torch.from_numpy(w).to(device) for w in wr],
                bias_d=[torch.from_numpy(b).to(device) if b is not None else None for b in bias],
                xs_d=[torch.from_numpy(x).to(device) for x in xs],
                bufs=[pw.Buffers(L, T, device=device) for L in layers], T=T)


def run_sweep(args):
    import torch
    import torch.distributed as dist

    import any_precision_expert_gb300 as pw
    from synth.workloads import sweep_changes

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return rank_max(v, ws, "cuda")

    T, K, W = args.tokens, args.steps, args.warmup
    sw = build_sweep(T)
    cfg, layers, bufs = sw["cfg"], sw["layers"], sw["bufs"]
    NL = len(layers)
    stream = torch.cuda.Stream()

    def forward_all():
        for l in range(NL):
            pw.moe_forward_fused(layers[l], sw["xs_d"][l], sw["wr_d"][l], sw["bias_d"][l], bufs[l], stream=stream)

    cur = [b.copy() for b in sw["init"]]
    plan = [sweep_changes(cfg, i, sw["init"]) for i in range(W + K)]

    def apply(i):
        for l, e, b in plan[i]:
            layers[l].set_expert_bitwidth(e, b, stream=stream)
            cur[l][e] = b

    with torch.cuda.stream(stream):
        for i in range(W):
            apply(i)
            forward_all()
    torch.cuda.synchronize()
    # routing is fixed per layer: experts with tokens, from the router's output
    active = [np.bincount(bufs[l].idx[:T].cpu().numpy().reshape(-1), minlength=cfg.E) > 0 for l in range(NL)]

    def step_bytes():
        tot = 0
        for l in range(NL):
            for e in range(cfg.E):
                if active[l][e]:
                    b = int(cur[l][e])
                    tot += 3 * cfg.d * cfg.f * 2 if b == 16 else 3 * cfg.d * cfg.f * b // 8 + (2 * cfg.f + cfg.d) * (1 << b) * 2
            tot += cfg.d * cfg.E * 2 + 2 * T * cfg.d * 2
        return tot

    # the 32 layers run as one CUDA graph; it reads bitwidths and page tables
    # from device memory, so the changes made between replays take effect
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        forward_all()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t_soak = time.time()
    while time.time() - t_soak < args.soak:
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
    byts = []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(W, W + K):
            apply(i)
            byts.append(step_bytes())
            g.replay()
        t1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1))
    # the dominant kernel: each layer's expert-FFN call, timed once more in a
    # graph of the 32 layers with events around every call (bitwidths as
    # after the last timed step)
    fm = measure_steps(dict(cfg=cfg, layers=layers, bufs=bufs, xs_d=sw["xs_d"], T=T, wr_d=sw["wr_d"],
                            bias_d=sw["bias_d"], bits=[np.array(c) for c in cur]), NL, 0, stream)
    froof = roofline_of(fm, cfg, T)
    ok = all(L.check_device() == 0 for L in layers)

    # end to end: every step makes its bitwidth changes, then every layer
    # copies its x in from pinned host memory, runs pw_moe_forward and copies
    # y back; the host waits for each step
    x_host = [torch.from_numpy(x).pin_memory() for x in sw["xs"]]
    y_host = [torch.empty((T, cfg.d), dtype=torch.float16).pin_memory() for _ in range(NL)]
    x_dev = [torch.empty((T, cfg.d), dtype=torch.float16, device="cuda") for _ in range(NL)]
    KE = min(K, args.e2e_steps)
    plan_e = [sweep_changes(cfg, W + K + i, sw["init"]) for i in range(KE)]
    barrier()
    te = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(KE):
            for l, e, b in plan_e[i]:
                layers[l].set_expert_bitwidth(e, b, stream=stream)
                cur[l][e] = b
            for l in range(NL):
                x_dev[l].copy_(x_host[l], non_blocking=True)
                y = pw.moe_forward_fused(layers[l], x_dev[l], sw["wr_d"][l], sw["bias_d"][l], bufs[l], stream=stream)
                y_host[l].copy_(y, non_blocking=True)
            stream.synchronize()
    barrier()
    e2e_s = max_over_ranks(time.perf_counter() - te)

    peaks = _load_json(os.path.join(ROOT, "MEASURED_PEAKS.json"))
    if peaks and peaks.get("hbm_gbs"):
        peak, peak_src = float(peaks["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    else:
        peak, peak_src = 6800.0, "fallback 6.8 TB/s"
    avg_bytes = sum(byts) / len(byts)
    gbs = avg_bytes / (ms / K * 1e-3) / 1e9
    out = None
    if rank == 0:
        cpu = sweep_cpu_baseline(sw, args.cpu_seconds) if (ws == 1 and args.cpu_seconds > 0) else None
        out = {
            "metric": METRIC, "value": job_value(T * K, ws, ms * 1e-3), "unit": "tokens/s", "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"{WORKLOADS['sweep'][0]}, {T} tokens per step through all {NL} layers",
                       "tokens_per_step": T, "layers": NL,
                       "bitwidth_changes_per_step": len(plan[W]),
                       "l2": f"inputs larger than L2: {avg_bytes / 1e6:.0f} MB of weights streamed per step",
                       "timing": "bitwidth calls (host page lists + one stream-ordered 4-byte write each) and "
                                 "one CUDA graph of the 32 layers per step, inside CUDA events on the stream",
                       "step_algorithmic_bytes": avg_bytes, "parallelism": "replicas" if ws > 1 else "single GPU",
                       "device_errors": not ok},
            "roofline": dict(froof, traffic=_traffic_from_profile("sweep", T),
                             note="per layer: the expert-FFN call (one persistent decode launch over the layer's "
                                  "8 experts), timed by CUDA events in a graph of the 32 layers; traffic: mean "
                                  "DRAM bytes of those launches from the committed ncu summary (null once the "
                                  "kernel sources change)"),
            "step_roofline": {"kernel": "32-layer decode step (per layer: router, permutation, persistent FFN, "
                                        "combine; bitwidth changes)",
                              "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                              "algorithmic_bytes_per_step": avg_bytes, "ms_per_step": ms / K,
                              "peak_source": peak_src},
            "cpu_baseline": cpu,
            "e2e": {"value": ws * T * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": NL * T * cfg.d * 2,
                    "d2h_bytes_per_step": NL * T * cfg.d * 2, "steps": KE,
                    "note": "per step: the step's bitwidth changes, then per layer a pinned H2D of x, pw_moe_forward "
                            "and a D2H of y (eager calls); host sync per step"},
            # bitwidth words are written by stream memory operations, not kernels
            "gpu_launches": NL * _launches_per_step(cfg, T) * K,
            "clocks": clk,
        }
    for L in layers:
        L.destroy()
    sw["bufs"] = None
    if rank == 0 and args.sub_runs and ws == 1:
        out["sub_runs"] = sub_runs(stream, src=sw["src"])
    sw["src"].destroy()
    sw["pool"].close()
    if ws > 1:
        dist.destroy_process_group()
    return out


def sweep_cpu_baseline(sw, seconds=20.0):
    """The oracle on one decode token of layer 0, extrapolated to the 32 layers."""
    from oracle import pw_oracle as O

    cfg = sw["cfg"]
    t_start = time.perf_counter()
    n = 0
    while n < 1 or (time.perf_counter() - t_start < seconds and n < 4):
        O.moe_tokens(sw["xs"][0], sw["wr"][0], sw["bias"][0], lambda e: sw["experts"][e], sw["init"][0], cfg.K,
                     cfg.renormalize, [n % sw["T"]])
        n += 1
    per_layer = (time.perf_counter() - t_start) / n
    return {"value": 1.0 / (per_layer * len(sw["layers"])), "unit": "tokens/s", "cores": _threads(),
            "kind": "oracle",
            "sample": f"{n} decode tokens through layer 0 at its initial bitwidths, x{len(sw['layers'])} extrapolated "
                      f"to the 32 layers ({per_layer:.1f} s per token-layer, numpy fp64)"}


def measure_paging(wl, stream, n_steps):
    """Decode throughput while precision is raised in the background (the
    pages' asynchronous paging, write-up section 安全边界与异步搬运).  Every
    step, on the step's layer copy: the expert raised at the copy's previous
    visit goes back to 3 bits, the expert prefetched then is raised to 6 bits
    (pw_set_expert_bitwidth: the commit, in stream order), and the next 3-bit
    expert's three missing planes are uploaded from pinned host memory on a
    copy stream (pw_prefetch_expert), to be committed at the copy's next
    visit, i.e. a step ahead.  Each step replays the copy's captured CUDA
    graph of the whole layer (it reads bitwidths and page tables from device
    memory); the paging calls run on the host between replays.  Same routing
    with and without the paging."""
    import torch

    import any_precision_expert_gb300 as pw

    layers, bufs, xs_d, T = wl["layers"], wl["bufs"], wl["xs_d"], wl["T"]
    NL = len(layers)
    three = [e for e in range(len(wl["bits"])) if int(wl["bits"][e]) == 3]
    n_steps = min(n_steps, (len(three) - 1) * NL)
    hold = {}

    def planes_of(e):
        if e not in hold:
            hold[e] = [[torch.from_numpy(q).pin_memory() if p >= 3 else None
                        for p, q in enumerate(pw.pack_planes(wl["experts"][e]["code6"][m]))] for m in range(3)]
        return hold[e]

    for e in three:
        planes_of(e)
    copy = torch.cuda.Stream()
    graphs = []
    with torch.cuda.stream(stream):
        for j in range(NL):  # warm the copy once eagerly, then capture its whole-layer call
            pw.moe_forward_fused(layers[j], xs_d[j], wl["wr_d"], wl["bias_d"], bufs[j], stream=stream)
    torch.cuda.synchronize()
    for j in range(NL):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            pw.moe_forward_fused(layers[j], xs_d[j], wl["wr_d"], wl["bias_d"], bufs[j], stream=stream)
        graphs.append(g)
    torch.cuda.synchronize()

    def run(with_paging):
        raised, fetched = {}, {}
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(n_steps):
                j = i % NL
                if with_paging:
                    if j in raised:
                        layers[j].set_expert_bitwidth(raised.pop(j), 3, stream=stream)
                    if j in fetched:
                        e = fetched.pop(j)
                        layers[j].set_expert_bitwidth(e, 6, stream=stream)
                        raised[j] = e
                    e = three[(i // NL) % len(three)]
                    layers[j].prefetch_expert(e, 6, planes=planes_of(e), copy_stream=copy)
                    fetched[j] = e
                graphs[j].replay()
            t1.record(stream)
        torch.cuda.synchronize()
        for j, e in list(raised.items()) + list(fetched.items()):
            layers[j].set_expert_bitwidth(e, 6, stream=stream)   # commit any pending prefetch first
            layers[j].set_expert_bitwidth(e, 3, stream=stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(False)  # warm-up
    base_ms = min(run(False), run(False))
    pag_ms = min(run(True), run(True))
    upload = 3 * 3 * (wl["cfg"].d * wl["cfg"].f // 8)
    return {"steps": n_steps, "tokens_per_s_without": T * n_steps / (base_ms * 1e-3),
            "tokens_per_s_with": T * n_steps / (pag_ms * 1e-3),
            "loss_pct": 100.0 * (1.0 - base_ms / pag_ms), "upload_bytes_per_step": upload,
            "pages_figure_context": "the write-up reports at most 4.1% for its system (hardware not stated)",
            "note": "CUDA-graph replay of the whole layer per step; per step one lower, one raise committing the "
                    "previous visit's prefetch, one prefetch (three planes uploaded on a copy stream a step "
                    "ahead); best of two passes each"}


def _traffic_from_profile(workload, T):
    """DRAM bytes per FFN call from the committed ncu summary, if it matches the current kernel."""
    prof = _load_json(os.path.join(ROOT, "profiles", f"ffn_traffic_{workload}_T{T}.json"))
    if not prof or int(prof.get("tokens", -1)) != T:
        return None
    if prof.get("source_hash") != kernel_source_hash():
        return None
    return prof.get("dram_bytes_per_call")


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("pw_ffn.cu", "pw_decode.cu", "pw_gemv.cuh", "pw_prefill.cu", "pw_device.cuh", "pw_tc.cuh"):
        with open(os.path.join(ROOT, "any_precision_expert_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle as it stands
# ---------------------------------------------------------------------------

def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def _blas_name():
    try:
        import numpy as np
        blas = np.show_config(mode="dicts")["Build Dependencies"]["blas"]
        return f"{blas.get('name', '?')} {blas.get('version', '')}".strip()
    except Exception:
        return "unknown"


# One oracle run in a fresh interpreter with every BLAS pool at one thread:
# the first n_tok tokens of the layer's seeded batch, one per call, repeated
# until `seconds` have passed (only the experts those tokens use are drawn).
_ONE_THREAD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
from oracle import pw_oracle as O
from synth import bits_plan, get_config, make_expert, make_router, make_shared, make_tokens
name, seconds, n_tok, T = sys.argv[2], float(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5])
cfg = get_config(name)
bits = bits_plan(cfg, 0)
wr, bias = make_router(cfg, 0)
shared = make_shared(cfg, 0)
x = make_tokens(cfg, T, 0, stream=0)
cache = {}
def expert(e):
    if e not in cache:
        cache[e] = make_expert(cfg, e, 0)
    return cache[e]
for t in range(n_tok):  # draws the sample's experts outside the timed loop
    O.moe_tokens(x, wr, bias, expert, bits, cfg.K, cfg.renormalize, [t], shared=shared)
n, t0 = 0, time.perf_counter()
while time.perf_counter() - t0 < seconds and n < 1024:
    O.moe_tokens(x, wr, bias, expert, bits, cfg.K, cfg.renormalize, [n % n_tok], shared=shared)
    n += 1
print(json.dumps({"value": n / (time.perf_counter() - t0), "calls": n}))
"""


def cpu_single_thread(names=("tiny", "qwen"), seconds=4.0, n_tok=4, T=64):
    """The oracle on one host thread for the tiny and Qwen-shaped layers (a
    bounded sample each); failures are reported, never raised."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    out = {"unit": "tokens/s", "threads": 1,
           "sample": f"tokens 0..{n_tok - 1} of the seeded {T}-token batch, one per oracle call, {seconds:.0f} s each"}
    for name in names:
        try:
            r = subprocess.run([sys.executable, "-c", _ONE_THREAD, ROOT, name, str(seconds), str(n_tok), str(T)],
                               env=env, capture_output=True, text=True, timeout=300)
            out[name] = json.loads(r.stdout.strip().splitlines()[-1])["value"] if r.returncode == 0 else \
                f"failed: {(r.stderr.strip().splitlines() or ['?'])[-1][:200]}"
        except Exception as e:  # noqa: BLE001 -- a baseline must not break the bench
            out[name] = f"failed: {e}"[:200]
    return out


def cpu_baseline(wl, seconds=20.0):
    """Time the oracle on a bounded sample: tokens of the batch one per call
    until `seconds` of CPU work (at most 1024 calls); then the one-thread runs."""
    from oracle import pw_oracle as O

    cfg = wl["cfg"]
    x = wl["xs"][0]
    done, tokens, t_start = 0, 0, time.perf_counter()
    n = 1
    while time.perf_counter() - t_start < seconds and done < 1024:
        O.moe_tokens(x, wl["wr"], wl["bias"], lambda e: wl["experts"][e], wl["bits"], cfg.K, cfg.renormalize,
                     list(range(done % x.shape[0], done % x.shape[0] + n)), shared=wl["shared"])
        done += 1
        tokens += n
    el = time.perf_counter() - t_start
    return {"value": tokens / el, "unit": "tokens/s", "cores": _threads(), "kind": "oracle",
            "sample": f"{tokens} decode tokens of the same layer, one token per oracle call "
                      f"({el:.1f} s of CPU work, numpy fp64, BLAS threads={_threads()}, os.cpu_count={os.cpu_count()})",
            "blas": _blas_name(), "single_thread": cpu_single_thread()}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    from synth import bits_plan, get_config, make_expert, make_router, make_shared, make_tokens
    from oracle import pw_oracle as O

    cfg = get_config(args.workload)
    T = args.tokens
    bits = bits_plan(cfg, 0)
    wr, bias = make_router(cfg, 0)
    experts = [make_expert(cfg, e, 0) for e in range(cfg.E)]
    shared = make_shared(cfg, 0)
    x = make_tokens(cfg, T, 0, stream=0)

    def one(i):
        t = i % T
        O.moe_tokens(x, wr, bias, lambda e: experts[e], bits, cfg.K, cfg.renormalize, [t], shared=shared)

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(args.warmup + i)
    el = time.perf_counter() - t0
    # the sweep's metric counts a token through all of its layers: one timed
    # layer, extrapolated
    n_layers = cfg.n_layers if args.workload == "sweep" else 1
    v = args.steps / (el * n_layers)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{WORKLOADS[args.workload][0]}, {T} tokens per step (same layer as the GPU arm)",
                       "tokens_per_step": 1},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": _threads(), "kind": "oracle",
                             "sample": "one decode token of the batch per step (numpy fp64 oracle)"
                                       + (f", one layer timed, x{n_layers} extrapolated" if n_layers > 1 else "")},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(WORKLOADS),
                    help="one workload only (default: the 32-layer sweep, with every other "
                         "configuration as sub-runs)")
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--copies", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed load for the clock record")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--paging", type=int, default=0,
                    help="steps of the async-paging measurement (0: skip)")
    ap.add_argument("--sub-runs", choices=["auto", "on", "off"], default="auto",
                    help="measure the other workloads and batch sizes beside the headline "
                         "(auto: only when no workload is named)")
    args = ap.parse_args()
    args.sub_runs = args.sub_runs == "on" or (args.sub_runs == "auto" and args.workload is None)
    if args.workload is None:
        args.workload = DEFAULT_WORKLOAD
    args.warmup = max(args.warmup, 3) if args.impl != "reference" else args.warmup
    if args.tokens is None:
        args.tokens = WORKLOADS[args.workload][1]
    if args.copies is None:
        args.copies = WORKLOADS[args.workload][2]
    if args.impl == "reference":
        out = run_reference(args)
    elif args.workload == "sweep":
        out = run_sweep(args)
    else:
        out = run_gpu(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
