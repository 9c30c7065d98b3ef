#!/usr/bin/env python
"""MoE-layer tokens/s of the NVFP4 expert FFN on one GB300 (per GPU replica).

One step = the whole forward pass on one batch of synthetic tokens:
route -> quantise into the grouped slot layout -> L1 grouped GEMM with fused
alpha/SiLU*up/amax -> requantise -> L2 grouped GEMM -> weighted reduce,
through the one-call layer entry point (moe_nvfp4_layer_forward): a single
cooperative kernel for small batches, route / quantise / GEMM / reduce
launches above that (the library counts its own launches).  The step is
replayed as one CUDA graph.  --api calls times the four-call composition
(route, quantise, forward, reduce) instead.

Default workload: the large prefill case (E=48 experts, H=7168, I=3072,
T=16384 tokens, top-8 with one expert in every token's list and six experts
idle, Student-t activations), the largest of the workloads, whose roofline is
the dense FP4 tensor peak.  --config decode1 (one token) and the others
select the smaller workloads; decode workloads are bound by HBM bandwidth on
the weight + scale bytes of the experts that receive a token.  The L2 cache
is flushed (256 MiB write) before every timed step of the large workloads;
decode steps instead alternate two routings with disjoint expert sets (each
step's weights are larger than L2 and were not read by the step before), and
the flushed decode time is reported in config.  Inputs are resident in HBM
before the timed region.

Also reported:
  roofline      the dominant kernel (the single layer kernel for small batches,
                else the L1 GEMM) timed alone with CUDA events recorded by
                the library on the launching stream, against the measured
                HBM copy bandwidth (MEASURED_PEAKS.json) for decode, and for
                prefill against the dense FP4 tensor peak that the library's
                own probe (nvmoe_fp4_mma_probe) measures on this GPU, with the
                datasheet figure beside it
  e2e           the same metric through the public API from pinned host
                buffers: H2D of x / topk ids / topk weights, forward, D2H of y
  cpu_baseline  the CPU oracle (numpy, fp64) timed on a bounded sample of the
                same workload (rank 0, N = 1)
--impl reference times the oracle alone on the same workload and metric.

Under torchrun each rank runs an independent replica on its own GPU (the
path has no cross-GPU exchange: replicas only), value = all ranks' tokens /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/sec on 1 GB300; % HBM roofline (decode), % FP4 TC peak (prefill)"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20            # > 129 MB L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: 2000 for decode workloads, 200 for prefill)")
    p.add_argument("--warmup", type=int, default=None,
                   help="untimed warm-up steps (default: 50 decode, 10 prefill)")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="prefill16k")
    p.add_argument("--api", choices=["layer", "calls"], default="layer",
                   help="one-call layer entry point, or route/quantise/forward/reduce")
    p.add_argument("--gate-up-scales", choices=["joint", "split"], default="joint",
                   help="one L1 weight global scale per expert, or separate gate/up scales")
    p.add_argument("--mid-scale", choices=["dynamic", "static"], default="dynamic",
                   help="the pages' dynamic intermediate scale, or a static per-expert one "
                        "(calibrated as one dynamic forward's scale)")
    p.add_argument("--part", choices=["layer", "router", "peak"], default="layer",
                   help="the MoE layer (steps 1-7), the router front-end alone, or the "
                        "dense FP4 tensor-core probe alone")
    p.add_argument("--pdl", choices=["on", "off"], default="off",
                   help="programmatic dependent launch on the multi-launch path "
                        "(off by default: measured slower on the prefill step)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--profile-steps", type=int, default=0,
                   help="run this many eager steps and exit (for ncu launch lists)")
    a = p.parse_args()
    big = a.config.startswith("prefill")
    if a.steps is None:
        a.steps = 200 if big else 2000
    if a.warmup is None:
        a.warmup = 10 if big else 50
    return a


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------ clocks ----
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # the timed region starts only once samples are flowing
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- oracle sample ----
def oracle_sample(cfg, n_tok, x_h=None, ids_h=None, w_h=None, weight_device=None):
    """Inputs of a CPU-oracle sample and a function that times one pass.

    The sample is the first n_tok tokens of the workload (activations and
    routing as drawn for the whole batch) with the workload's weights of the
    experts those tokens use: drawn by the seeded generator on
    `weight_device` (the GPU, i.e. the values the GPU arm quantises; the
    host when there is none) and quantised by the oracle (set-up, untimed).
    One pass is the C++ oracle's whole forward (route, quantise, L1 with
    alpha, SiLU*up, requantise, L2 with alpha, weighted reduce) on all host
    cores; it returns the seconds of that pass."""
    import numpy as np
    import torch
    from oracle import cpp as ocpp
    from nvfp4_block_scaled_route_gb300 import synthetic as syn
    if x_h is None:
        x_h = syn.draw_activations(cfg)
        ids_h, w_h = syn.draw_routing(cfg)
    x = x_h[:n_tok].float().numpy()
    ids = ids_h[:n_tok].numpy()
    w = w_h[:n_tok].numpy()
    used = sorted(set(ids.reshape(-1).tolist()))
    E, H, I = cfg.E, cfg.H, cfg.I
    W1q = np.zeros((E, H // 2, 2 * I), np.uint8)
    W1s = np.zeros((E, H // 16, 2 * I), np.uint8)
    W2q = np.zeros((E, I // 2, H), np.uint8)
    W2s = np.zeros((E, I // 16, H), np.uint8)
    g1 = np.ones(E, np.float32)
    g2 = np.ones(E, np.float32)
    dev = weight_device if weight_device is not None else "cpu"
    for e in used:
        W1q[e], W1s[e], g1[e] = ocpp.nvfp4.quantize_weight(
            syn.draw_weight(cfg, 1, e, device=dev).cpu().numpy())
        W2q[e], W2s[e], g2[e] = ocpp.nvfp4.quantize_weight(
            syn.draw_weight(cfg, 2, e, device=dev).cpu().numpy())
    if dev != "cpu":
        torch.cuda.empty_cache()

    def one_pass():
        return ocpp.moe.forward(x, ids, w, W1q, W1s, g1, W2q, W2s, g2)["seconds"]

    desc = (f"the first {n_tok} token(s) of the workload ({len(used)} experts) through the "
            f"C++ oracle's whole forward (fp64 GEMMs), the workload's own weights "
            f"(drawn on {'the GPU' if dev != 'cpu' else 'the host'}), "
            f"{ocpp.threads()} OpenMP threads")
    return one_pass, ocpp.threads(), desc


def oracle_tokens(cfg, budget_tokens: int) -> int:
    return max(1, min(cfg.T, budget_tokens))


# ---------------------------------------------------------------- main ----
def workload_desc(cfg):
    return (f"{cfg.name}: E={cfg.E} H={cfg.H} I={cfg.I} T={cfg.T} top-{cfg.k} "
            f"routing={cfg.routing} act={cfg.act}")


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores: each step one pass of
    the C++ oracle over a one-token sample of the workload (its token, its
    routing, the workload's weights of its experts)."""
    from nvfp4_block_scaled_route_gb300 import synthetic as syn
    import torch
    cfg = syn.CONFIGS[args.config]
    if rank != 0:
        return
    n_tok = oracle_tokens(cfg, 1)
    dev = "cuda" if torch.cuda.is_available() else None
    one_pass, cores, desc = oracle_sample(cfg, n_tok, weight_device=dev)
    times = []
    for i in range(args.warmup + args.steps):
        t = one_pass()
        if i >= args.warmup:
            times.append(t)
    sec = sum(times)
    value = n_tok * len(times) / sec
    ms = 1000.0 * sec / max(len(times), 1)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(cfg)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: " + desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_router(args, nb, syn, cfg, dev, world, torch):
    """The router front-end alone (moe_router_topk) on the workload's tokens:
    logits over the E experts, top-k, softmax; one CUDA graph per step, L2
    flushed before every step."""
    x = syn.draw_activations(cfg).to(dev)
    w = syn.draw_router_weight(cfg).to(dev)
    mode = nb.ROUTER_ALL if cfg.routing == "softmax_topk_probs" else nb.ROUTER_SELECTED
    ws = nb._workspace(nb.lib().moe_router_workspace_size(cfg.T, cfg.H, cfg.E), dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            nb.router_topk(x, w, cfg.k, mode, ws=ws)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        nb.router_topk(x, w, cfg.k, mode, ws=ws)
    times = []
    with torch.cuda.stream(stream):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.warmup + args.steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    times = [a.elapsed_time(b) for a, b in evs[args.warmup:]]
    ms = sum(times) / len(times)
    nbytes = x.nbytes + w.nbytes + cfg.T * cfg.k * 8
    flops = 2.0 * cfg.T * cfg.H * cfg.E
    hbm_gbs, _, peak_src = peaks()
    achieved = nbytes / (ms / 1000.0) / 1e9
    line = {"metric": "router tokens/sec on 1 GB300", "value": world * cfg.T / (ms / 1000.0),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 in, fp32 sums", "data": "synthetic",
            "config": {"workload": workload_desc(cfg), "part": "router (logits, top-k, softmax)",
                       "l2_flush": "256 MiB write before every step",
                       "graph": "one CUDA graph per step", "launches_per_step": 2,
                       "flops_per_step": flops},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                         "frac": achieved / hbm_gbs, "peak_source": peak_src,
                         "algorithmic_bytes_per_step": nbytes}}
    print(json.dumps(line), flush=True)


FP4_DATASHEET_TFLOPS = 13500.0       # GB300 dense NVFP4, nominal (no sparsity)


def measure_fp4_peak(nb, torch, dev, sustain_s: float = 2.0):
    """Dense NVFP4 tensor-core peak of this GPU from the library's own probe
    (tcgen05.mma kind::mxf4nvf4 back to back on every SM, operands resident
    in shared memory).  Burst: the best single launch of the faster of the
    one-CTA and CTA-pair forms; sustained: that form launched back to back
    for `sustain_s` seconds (under the power cap)."""
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    grid = n_sm - (n_sm & 1)
    iters = 16384
    forms = {}
    for variant, name in ((0, "one CTA, M=128 N=256"), (1, "CTA pair, M=256 N=256")):
        r = nb.fp4_mma_probe(variant, iters=iters, grid=grid, repeats=5, device=dev)
        if r["status"] != 0:
            raise RuntimeError(f"FP4 probe variant {variant} status {r['status']}")
        forms[name] = r
    best_name = max(forms, key=lambda n: forms[n]["tflops"])
    best = forms[best_name]
    # sustained: back-to-back launches of the best form
    per_launch_s = min(best["ms"]) / 1e3
    n = max(10, int(sustain_s / per_launch_s))
    cycles = torch.zeros(grid, dtype=torch.int64, device=dev)
    ws = nb._workspace(256, dev)
    s = torch.cuda.Stream(device=dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        a.record(s)
        for _ in range(n):
            nb._check("nvmoe_fp4_mma_probe", nb.lib().nvmoe_fp4_mma_probe(
                best["variant"], iters, grid, nb._ptr(cycles), nb._ptr(ws), ws.numel(),
                s.cuda_stream))
        b.record(s)
    s.synchronize()
    sustained = n * grid * iters * 2.0 * 128 * 256 * 64 / (a.elapsed_time(b) / 1e3) / 1e12
    return {"burst_tflops": best["tflops"], "sustained_tflops": sustained, "form": best_name,
            "cycles_per_mma": best["cycles_per_mma"],
            "forms": {k: {"tflops": v["tflops"], "cycles_per_mma": v["cycles_per_mma"]}
                      for k, v in forms.items()},
            "datasheet_tflops": FP4_DATASHEET_TFLOPS}


def run_peak(args, nb, dev, torch):
    """The probe alone: every variant, one JSON line."""
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    grid = n_sm - (n_sm & 1)
    names = {0: "1cta_n256", 1: "pair_n256", 2: "1cta_n128", 3: "pair_n128",
             4: "1cta_n256_cp32", 5: "pair_n256_cp32", 6: "1cta_n128_cp32",
             7: "pair_n128_cp32", 8: "1cta_n256_cp256", 9: "pair_n256_cp256",
             10: "1cta_n128_cp256", 11: "pair_n128_cp256"}
    out = {}
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for v, name in names.items():
        r = nb.fp4_mma_probe(v, iters=16384, grid=grid, repeats=5, device=dev)
        out[name] = {"tflops": round(r["tflops"], 1), "cycles_per_mma": r["cycles_per_mma"],
                     "status": r["status"]}
    pk = measure_fp4_peak(nb, torch, dev)
    clocks = sampler.stop()
    print(json.dumps({"metric": "dense NVFP4 tensor-core throughput (probe)", "unit": "TFLOP/s",
                      "variants": out, "peak": pk, "clocks": clocks, "grid": grid}), flush=True)


GEMM_SOURCES = ("gemm.cu", "ptx.cuh", "quant.cuh", "internal.h")


def gemm_source_hash():
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "nvfp4_block_scaled_route_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, config: str):
    """DRAM bytes per launch of `kernel` from the committed ncu record, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("source_hash") != gemm_source_hash():
        return None
    return d.get("per_launch_bytes", {}).get(config)


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (every rank gets it); the value itself when
    there is one rank."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time
    (the replicas are independent, so work grows with the rank count)."""
    return world * tokens_per_step * steps / (ms / 1000.0)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding as nb
    from nvfp4_block_scaled_route_gb300 import synthetic as syn

    nb.lib().nvmoe_set_pdl(1 if args.pdl == "on" else 0)
    cfg = syn.CONFIGS[args.config]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.part == "peak":
        if rank == 0:
            run_peak(args, nb, dev, torch)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.part == "router":
        run_router(args, nb, syn, cfg, dev, world, torch)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    # ---- inputs (resident in HBM) ----
    q1s, s1s, g1s, q2s, s2s, g2s, gus = [], [], [], [], [], [], []
    split = args.gate_up_scales == "split"
    for e in range(cfg.E):
        w1 = syn.draw_weight(cfg, 1, e, device=dev)[None]
        w2 = syn.draw_weight(cfg, 2, e, device=dev)[None]
        if split:
            qg, sg, gg = nb.quantize_weights(w1[:, :, :cfg.I].contiguous())
            qu, su, gu = nb.quantize_weights(w1[:, :, cfg.I:].contiguous())
            q1s.append(torch.cat([qg, qu], 2)); s1s.append(torch.cat([sg, su], 2))
            g1s.append(gg); gus.append(gu)
        else:
            q, s, g = nb.quantize_weights(w1)
            q1s.append(q); s1s.append(s); g1s.append(g)
        q, s, g = nb.quantize_weights(w2)
        q2s.append(q); s2s.append(s); g2s.append(g)
        del w1, w2
    pw = nb.PreparedWeights.from_checkpoint(torch.cat(q1s), torch.cat(s1s), torch.cat(g1s),
                                            torch.cat(q2s), torch.cat(s2s), torch.cat(g2s),
                                            gs1_up=torch.cat(gus) if split else None)
    del q1s, s1s, q2s, s2s
    x_h = syn.draw_activations(cfg).pin_memory()
    ids_h, w_h = syn.draw_routing(cfg)
    ids_h, w_h = ids_h.pin_memory(), w_h.pin_memory()
    Layer = nb.FusedLayer if args.api == "layer" else nb.MoELayer
    if args.mid_scale == "static":
        # calibration: one dynamic forward gives the static scale of every expert
        cal = Layer(pw, cfg.T, cfg.k, device=dev, out_dtype=torch.bfloat16)
        gs_h = torch.zeros(1, dtype=torch.float32, device=dev)
        cal.forward(x_h.to(dev), ids_h.to(dev), w_h.to(dev), taps={"gs_h": gs_h})
        torch.cuda.synchronize()
        pw.gs_mid = gs_h.expand(cfg.E).contiguous()
        del cal
    layer = Layer(pw, cfg.T, cfg.k, device=dev, out_dtype=torch.bfloat16)
    staged = None
    if args.api == "layer":
        # the one-call API's pinned staging area: the step's inputs travel in
        # one host-to-device copy, y in one device-to-host copy
        (sx, sids, sw, sy), (x, ids, w) = layer.staging()
        sx.copy_(x_h)
        sids.copy_(ids_h)
        sw.copy_(w_h)
        staged = (sx, sids, sw, sy)
        x_h, ids_h, w_h = sx, sids, sw
        layer.forward_staged()
    else:
        x, ids, w = x_h.to(dev), ids_h.to(dev), w_h.to(dev)
    torch.cuda.synchronize()

    active = sorted(set(ids_h.flatten().tolist()))
    E_act = len(active)
    H, I = cfg.H, cfg.I
    l1_bytes = E_act * (2 * I * H // 2 + 2 * I * H // 16)
    l2_bytes = E_act * (H * I // 2 + H * I // 16)
    S = cfg.T * cfg.k
    flops = 2.0 * S * H * 2 * I + 2.0 * S * I * H
    hbm_gbs, _, peak_src = peaks()

    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    if args.profile_steps:
        with torch.cuda.stream(stream):
            for _ in range(args.profile_steps):
                flush.fill_(1)
                layer.forward(x, ids, w)
        torch.cuda.synchronize()
        print(json.dumps({"profile_steps": args.profile_steps, "workload": workload_desc(cfg)}))
        return

    # ---- CUDA graph of one step ----
    with torch.cuda.stream(stream):
        for _ in range(3):
            layer.forward(x, ids, w)
    stream.synchronize()
    # library kernels per step, counted by the library itself on one eager step
    n0 = nb.lib().nvmoe_kernel_launch_count()
    with torch.cuda.stream(stream):
        layer.forward(x, ids, w)
    stream.synchronize()
    kernels_per_step = int(nb.lib().nvmoe_kernel_launch_count() - n0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer.forward(x, ids, w)
    stream.synchronize()
    assert layer.status() == 0
    # Small batches (decode): consecutive steps alternate two routings whose
    # expert sets are disjoint (expert ids shifted by E/2) instead of flushing
    # L2: a step's weights (its experts', >= 8 x 37 MB) are larger than the
    # L2 and none were read by the step before, while the kernel's code
    # stays cached as it would across the layers of a model.  The flushed
    # timing is reported beside it.  Large batches flush L2 before each step.
    rotate = cfg.T * cfg.k <= 2048
    steps_fns = [graph.replay]
    ids_alt = [ids]
    if rotate:
        ids_b = ((ids.long() + cfg.E // 2) % cfg.E).to(torch.int32)
        graph_b = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            layer.forward(x, ids_b, w)
        stream.synchronize()
        with torch.cuda.graph(graph_b, stream=stream):
            layer.forward(x, ids_b, w)
        stream.synchronize()
        steps_fns.append(graph_b.replay)
        ids_alt.append(ids_b)

    def timed_loop(n, step_fn, flush_l2=True):
        fns = step_fn if isinstance(step_fn, list) else [step_fn]
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(n):
                if flush_l2:
                    flush.fill_(i & 0xFF)
                starts[i].record(stream)
                fns[i % len(fns)]()
                ends[i].record(stream)
        stream.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    timed_loop(args.warmup, steps_fns, flush_l2=not rotate)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    times = timed_loop(args.steps, steps_fns, flush_l2=not rotate)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    flushed_ms = None
    if rotate:
        flushed_ms = sum(timed_loop(args.steps, graph.replay)) / args.steps
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(times), world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, cfg.T, args.steps, total_ms)

    # ---- dominant kernel: L1 GEMM timed alone by library-recorded events ----
    n_prof = min(args.steps, 50)
    stage = {"l1": [], "requant": [], "l2": []}
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            if not rotate:
                flush.fill_(i & 0xFF)
            layer.forward(x, ids_alt[i % len(ids_alt)], w, taps={"stage_events": evs})
            stream.synchronize()
            stage["l1"].append(evs[0].elapsed_time(evs[1]))
            stage["requant"].append(evs[1].elapsed_time(evs[2]))
            stage["l2"].append(evs[2].elapsed_time(evs[3]))
    l1_ms = statistics.mean(stage["l1"])
    # single-kernel paths record events 1..3 together after their kernel
    fused = max(statistics.mean(stage["requant"]), statistics.mean(stage["l2"])) < 0.01
    decode = cfg.T * cfg.k <= 2048
    act_bytes = x.nbytes + ids.nbytes + w.nbytes + layer.y.nbytes
    if decode and fused and kernels_per_step == 1:
        fb = l1_bytes + l2_bytes + act_bytes
        achieved = fb / (l1_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "peak_source": peak_src,
                "kernel": "layer_kernel (route + quantise + L1 + requantise + L2 + reduce, "
                          "one cooperative launch)",
                "algorithmic_bytes_per_launch": fb, "launch_ms": l1_ms}
    elif decode and fused:
        fb = l1_bytes + l2_bytes
        achieved = fb / (l1_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "peak_source": peak_src,
                "kernel": "fused_ffn_kernel (L1 + requantise + L2, one cooperative launch)",
                "algorithmic_bytes_per_launch": fb, "launch_ms": l1_ms}
    elif decode:
        achieved = l1_bytes / (l1_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "peak_source": peak_src,
                "kernel": "grouped_gemm_kernel (L1, mode 1)",
                "algorithmic_bytes_per_launch": l1_bytes, "launch_ms": l1_ms}
    else:
        l1_flops = 2.0 * S * H * 2 * I
        achieved = l1_flops / (l1_ms / 1000.0) / 1e12
        # the library runs L1 over CTA pairs when every routing gives at least
        # 4 tiles per SM: ceil(S / 128) m-tiles x 2I / 256 n-tiles
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        pair = -(-S // 128) * (2 * I // 256) >= 4 * n_sm
        l1_kernel = ("grouped_gemm_pair_kernel (L1, mode 1, CTA pairs)" if pair
                     else "grouped_gemm_kernel (L1, mode 1)")
        fp4 = measure_fp4_peak(nb, torch, dev)
        peak = fp4["burst_tflops"]
        step_tflops = flops / (ms_per_step / 1000.0) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_source": "measured: nvmoe_fp4_mma_probe burst (" + fp4["form"] + ")",
                "peak_sustained": fp4["sustained_tflops"],
                "peak_datasheet": fp4["datasheet_tflops"],
                "frac_of_datasheet": achieved / fp4["datasheet_tflops"],
                "probe": fp4,
                "kernel": l1_kernel,
                "algorithmic_flops_per_launch": l1_flops, "launch_ms": l1_ms,
                "step_tflops": step_tflops, "step_frac": step_tflops / peak}
    roof["traffic"] = profiled_traffic(roof["kernel"].split()[0], args.config)
    step_bytes = l1_bytes + l2_bytes

    # ---- end to end from pinned host buffers through the public API ----
    e2e = None
    if not args.no_e2e and staged is not None:
        # steps fed from pinned host memory through the public API
        # (StagedPipeline over the one-call layer): every step copies its own
        # inputs in and its y out; step i's input copy and step i-1's readback
        # overlap another step's layer.  Timed from before the first input
        # copy to after the last readback (events on the copy streams).  No L2
        # flush can sit between overlapped steps: the two slots route every
        # token to disjoint expert sets (slot 1: expert ids shifted by E/2), so
        # consecutive steps read different weights, and each step's working
        # set (its experts' weights, and at prefill x) is larger than L2.
        pipe = nb.StagedPipeline(layer, depth=2)
        y_want = []
        for slot in range(pipe.depth):
            px, pids, pw = pipe.inputs(slot)
            px.copy_(staged[0])
            pids.copy_((staged[1] + slot * (cfg.E // 2)) % cfg.E)
            pw.copy_(staged[2])
            with torch.cuda.stream(stream):
                y_want.append(layer.forward(px.to(dev), pids.to(dev), pw.to(dev)).cpu().clone())
            stream.synchronize()
        for _ in range(min(args.warmup, 5)):
            pipe.submit()
        pipe.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(pipe.s_in)
        for s_ in (pipe.s_comp, pipe.s_out):
            s_.wait_event(t0)
        for _ in range(args.steps):
            pipe.submit()
        for s_ in (pipe.s_in, pipe.s_comp):
            ev = torch.cuda.Event()
            ev.record(s_)
            pipe.s_out.wait_event(ev)
        t1.record(pipe.s_out)
        pipe.synchronize()
        e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
        for slot in range(pipe.depth):
            assert torch.equal(pipe.output(slot), y_want[slot])
        e2e = {"value": job_throughput(world, cfg.T, args.steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": pipe.h2d_bytes, "d2h_bytes_per_step": pipe.d2h_bytes,
               "ms_per_step": e_ms / args.steps,
               "api": "StagedPipeline(FusedLayer), depth 2: copy-in / layer / copy-out streams",
               "l2": "no flush between overlapped steps; consecutive steps use disjoint "
                     "expert sets and each step's working set is larger than L2"}
    elif not args.no_e2e:
        # the four-call API: each step's inputs in, the captured step, y out
        y_h = torch.empty((cfg.T, H), dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            x.copy_(x_h, non_blocking=True)
            ids.copy_(ids_h, non_blocking=True)
            w.copy_(w_h, non_blocking=True)
            graph.replay()
            y_h.copy_(layer.y, non_blocking=True)

        timed_loop(min(args.warmup, 5), e2e_step)
        et = timed_loop(args.steps, e2e_step)
        e_ms = max_over_ranks(sum(et), world, dev)
        e2e = {"value": job_throughput(world, cfg.T, args.steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": x_h.nbytes + ids_h.nbytes + w_h.nbytes,
               "d2h_bytes_per_step": y_h.nbytes, "ms_per_step": e_ms / args.steps}
    assert layer.status() == 0

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del layer, pw
        torch.cuda.empty_cache()
        n_tok = oracle_tokens(cfg, 4)
        one_pass, cores, desc = oracle_sample(cfg, n_tok, x_h, ids_h, w_h, weight_device=dev)
        t = one_pass()
        cpu = {"value": n_tok / t, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{desc}: {t:.2f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x e4m3 scales), fp32 accumulate", "data": "synthetic",
            "config": {"workload": workload_desc(cfg),
                       "l2_flush": ("none: consecutive steps use disjoint expert sets, whose "
                                    "weights are larger than L2 (ms_per_step with a 256 MiB "
                                    "flush before every step: %.4f)" % flushed_ms) if rotate
                                   else "256 MiB write before every step",
                       "graph": "one CUDA graph per step", "active_experts": E_act,
                       "pdl": args.pdl,
                       "api": "moe_nvfp4_layer_forward" if args.api == "layer"
                              else "route + quantise + forward + reduce",
                       "gate_up_scales": args.gate_up_scales,
                       "mid_scale": args.mid_scale,
                       "algorithmic_bytes_per_step": step_bytes, "flops_per_step": flops,
                       "step_hbm_frac": (step_bytes / (ms_per_step / 1000.0) / 1e9) / hbm_gbs,
                       "stage_ms": {k: statistics.mean(v) for k, v in stage.items()},
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_step * args.steps, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
