"""Benchmark of the batch-invariant MoE hot path on GB300.

One step = one pass of the whole hot path over one batch of M synthetic
tokens: fp32 router GEMM on the bf16 tokens (read as their exact fp32
values), sigmoid top-k, token permute and row gather, gate/up grouped GEMM
with SwiGLU x probability, down grouped GEMM, slot-order combine.  Default
workload: the largest configuration, the DSv4-router-shaped MoE layer
(H=4096, E=256, top-8, I=2048, router K=4096 N=256), M=4096 tokens per GPU
per step, bf16 weights/activations ~ N(0, 0.02), fp32 router.  The expert
weights (12.9 GB) are far larger than L2, so every step streams them from
HBM (no explicit flush).  The Qwen3-30B-A3B-shaped layer (H=2048, E=128,
top-8, I=768) is timed as a secondary workload (--workload qwen makes it
the headline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload qwen|dsv4] [--tokens M] [--no-extras]
                  [--no-cpu-baseline]
  python bench.py --router-sweep | --moe-sweep [--workload ...] | --topk-window-sweep

Prints one JSON line (rank 0).  N > 1: launched by torchrun, one rank per
GPU, every rank runs its own M tokens (weak scaling, no collective on the
data path); the time is the max over ranks.  The sweeps print one JSON
object each (device time vs batch size, CUDA-graph replay).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    "qwen": dict(name="qwen3-30b-a3b-moe-layer", H=2048, E=128, I=768, top_k=8),
    "dsv4": dict(name="dsv4-router-moe-layer", H=4096, E=256, I=2048, top_k=8),
}


# ------------------------------------------------------------ distributed --
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput: tokens processed by all ranks / slowest rank's time."""
    return tokens_per_rank * steps * world / max_seconds


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

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
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def snapshot(self):
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                 timeout=10).stdout.strip()
            if out:
                self.lines.append(out)
        except (OSError, subprocess.TimeoutExpired):
            pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if not self.lines:
            self.snapshot()
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ our GPU arm --
def measured_peaks():
    """(HBM copy GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), \
            d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def code_digest(text):
    """sha256 of C/CUDA source with its comments and all whitespace removed:
    the same for two revisions that differ only in comments or layout."""
    import hashlib
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # a string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return hashlib.sha256("".join("".join(out).split()).encode()).hexdigest()


def captured_traffic(workload, M, kernel):
    """DRAM bytes per full-size launch of an expert GEMM from the committed
    ncu capture of this workload, or None when there is none or the kernel's
    code (comments aside) changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"moe_gemm_{workload}_{M}_traffic.json")
    src = os.path.join(ROOT, "invariant_moe_gb300", "csrc", "moe_gemm.cu")
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    d = json.load(open(path))
    if code_digest(open(src).read()) != d.get("kernel_code_sha256"):
        return None
    k = d.get(kernel, {})
    return k.get("dram_bytes_per_full_launch") or None


def layer_costs(M, H, E, I, k, feed="copy"):
    """Algorithmic bytes and flops of the method, per expert GEMM and for the
    whole step.  'method' bytes are what the layer must move: the touched
    experts' weights (E_t = E (1 - (1 - k/E)^M) experts), the tokens, the
    routing (ids + wts) and the output; the router's fp32 weight and scores.
    'impl' bytes are this implementation's workspace traffic (gathered token
    rows, activations, fp32 per-slot contributions), reported apart."""
    P = M * k
    touched = E * (1.0 - (1.0 - k / E) ** M)
    w13, w2 = touched * 2 * I * H * 2, touched * H * I * 2
    x = out = M * H * 2
    routing = M * k * 8
    router = E * H * 4 + M * E * 4
    xperm = P * H * 2 if feed == "copy" else 0   # the gathered copy, written and read back
    return {
        "gate_up": {"method": w13 + x + routing, "impl": xperm + P * I * 2, "flops": 2.0 * P * 2 * I * H},
        "down": {"method": w2 + out, "impl": P * I * 2 + P * H * 4, "flops": 2.0 * P * H * I},
        "step": {"method": router + x + w13 + w2 + out + routing,
                 "impl": 2 * xperm + P * I * 2 * 2 + P * H * 4 * 2,
                 "flops": 2.0 * P * 3 * I * H, "fp32_flops": 2.0 * M * H * E},
    }


def roofline_entry(kernel, cost, ms, hbm_gbs, tc_burst, peak_src, traffic=None):
    """Achieved method bytes (or flops) per launch over the launch's CUDA-event
    time, against the roof that binds it: the measured copy bandwidth, or the
    measured bf16 burst peak (these kernels run for at most milliseconds
    inside a sub-second timed region), whichever floor is longer."""
    t = ms / 1e3
    gbs, tfs = cost["method"] / t / 1e9, cost["flops"] / t / 1e12
    hbm_bound = cost["method"] / (hbm_gbs * 1e9) >= cost["flops"] / (tc_burst * 1e12)
    r = {"kernel": kernel}
    if hbm_bound:
        r.update({"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
                  "peak_source": f"{peak_src} copy bandwidth"})
    else:
        r.update({"bound": "tensor", "achieved": tfs, "peak": tc_burst, "unit": "TFLOP/s",
                  "frac": tfs / tc_burst, "peak_source": f"{peak_src} bf16 burst"})
    r.update({
        "traffic": traffic,
        "traffic_unit": "bytes per launch (ncu dram read+write)",
        "algorithmic_bytes": cost["method"],
        "implementation_bytes": cost["impl"],
        "algorithmic_flops": cost["flops"],
        "hbm_gbs": gbs, "hbm_frac": gbs / hbm_gbs,
        "tensor_tflops": tfs, "tensor_frac_of_burst": tfs / tc_burst,
        "ms_per_launch": ms,
    })
    return r


def setup_workload(wl, M, dev, x_seed):
    """Weights (on the device), tokens and the step's buffers for one workload."""
    import torch

    import invariant_moe_gb300 as bm
    from tests import synthetic as syn
    H, E, I, k = wl["H"], wl["E"], wl["I"], wl["top_k"]
    P = M * k
    w = syn.moe_weights(H, E, I, seed=11, device=str(dev))
    lib = bm.load_library()
    b = {
        "w": w, "x": syn.moe_tokens(M, H, seed=x_seed, device=str(dev)),
        "scores": torch.empty(M, E, dtype=torch.float32, device=dev),
        "ids": torch.empty(M, k, dtype=torch.int32, device=dev),
        "wts": torch.empty(M, k, dtype=torch.float32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "perm": torch.empty(P, dtype=torch.int32, device=dev),
        "x_perm": torch.empty(P, H, dtype=torch.bfloat16, device=dev),
        "act": torch.empty(P, I, dtype=torch.bfloat16, device=dev),
        "contrib": torch.empty(P, H, dtype=torch.float32, device=dev),
        "out": torch.empty(M, H, dtype=torch.bfloat16, device=dev),
        "ws_perm": torch.empty(max(int(lib.bi_moe_permute_workspace_bytes(M, E)), 256),
                               dtype=torch.uint8, device=dev),
    }
    return b


def launches_per_step(M, E, feed="copy"):
    """Kernels one step launches: router + top-k (2), permutation (one CTA up to 1024 tokens when its shared memory fits,
    else count / scan / scatter), the gather (only with feed "copy"),
    gate/up, down, combine."""
    small = M <= 1024 and E * (8 + ((M + 255) // 256 * 256 // 32 + 1) * 4) <= 48 * 1024
    return 2 + (1 if small else 3) + (4 if feed == "copy" else 3)


def time_steps(wl, M, b, steps, warmup, world, stream, dev, feed="copy"):
    """Times `steps` steps of the whole hot path (device time, CUDA events on
    the launching stream, barrier + synchronize on both sides) and the
    gate/up and down GEMMs inside them.  Returns (seconds, gate/up ms, down
    ms, clocks)."""
    import torch

    import invariant_moe_gb300 as bm
    E, k = wl["E"], wl["top_k"]
    w = b["w"]
    ev = {"gate_up": [], "down": []}

    def step(record=False):
        # router on the bf16 tokens (read as fp32) and top-k selection
        bm.bi_router_topk(b["x"], w.w_router, k, out=b["scores"], ids=b["ids"], wts=b["wts"])
        bm.bi_moe_permute(b["ids"], E, offsets=b["offsets"], perm=b["perm"], workspace=b["ws_perm"])
        if feed == "copy":
            bm.bi_moe_gather(b["x"], b["offsets"], b["perm"], k, x_perm=b["x_perm"])
        if record:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e2 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        if feed == "copy":
            bm.bi_moe_gate_up(b["x_perm"], b["offsets"], b["perm"], b["wts"], w.w13, k, act=b["act"])
        else:  # the GEMM gathers the token rows itself (bi_moe_gate_up_feed 2)
            bm.bi_moe_gate_up_tokens(b["x"], b["offsets"], b["perm"], b["wts"], w.w13, k, act=b["act"])
        if record:
            e1.record(stream)
        bm.bi_moe_down(b["act"], b["offsets"], b["perm"], w.w2, M, k, contrib=b["contrib"])
        if record:
            e2.record(stream)
            ev["gate_up"].append((e0, e1))
            ev["down"].append((e1, e2))
        bm.bi_moe_combine_consume(b["contrib"], M, k, out=b["out"])

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    if bm.device_error() != 0:
        raise RuntimeError("device error during warm-up")
    clocks = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)  # let the sampler come up before the timed region
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    if bm.device_error() != 0:
        raise RuntimeError("device error during the timed region")
    sec = t0.elapsed_time(t1) / 1e3
    gu_ms = statistics.mean(a.elapsed_time(c) for a, c in ev["gate_up"])
    dn_ms = statistics.mean(a.elapsed_time(c) for a, c in ev["down"])
    return sec, gu_ms, dn_ms, clk


def run_ours(args, rank, world, local):
    import torch

    import invariant_moe_gb300 as bm

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    wl = WORKLOADS[args.workload]
    H, E, I, k = wl["H"], wl["E"], wl["I"], wl["top_k"]
    M = args.tokens
    b = setup_workload(wl, M, dev, x_seed=21 + rank)
    w, x = b["w"], b["x"]
    stream = torch.cuda.current_stream(dev)
    sec, gu_ms, dn_ms, clk = time_steps(wl, M, b, args.steps, args.warmup, world, stream, dev, args.feed)
    sec_max = max_over_ranks(sec, world, dev)

    # ---- end to end through the public API from pinned host buffers.  Each
    # step uploads its tokens, runs the layer and downloads its output; the
    # uploads and downloads run on their own streams (two device input
    # buffers in rotation), so step i+1's upload and step i's download
    # overlap step i's layer, as a serving loop would run them.
    nbuf = 2
    x_host = [x.cpu().pin_memory() for _ in range(nbuf)]
    out_host = [torch.empty(M, H, dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    x_dev = [torch.empty_like(x) for _ in range(nbuf)]
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event() for _ in range(nbuf)]
    consumed = [torch.cuda.Event() for _ in range(nbuf)]
    produced = [torch.cuda.Event() for _ in range(nbuf)]
    downloaded = [torch.cuda.Event() for _ in range(nbuf)]
    e2e_steps = max(3, min(args.steps, 200))
    e2e_i = [0]

    def e2e_step():
        i = e2e_i[0] % nbuf
        e2e_i[0] += 1
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(consumed[i])          # the layer that read x_dev[i] is done
            x_dev[i].copy_(x_host[i], non_blocking=True)
            uploaded[i].record(h2d_stream)
        stream.wait_event(uploaded[i])
        o, _, _, _ = bm.moe_layer(x_dev[i], w.w_router, w.w13, w.w2, k)
        consumed[i].record(stream)
        produced[i].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(produced[i])
            o.record_stream(d2h_stream)
            out_host[i].copy_(o, non_blocking=True)
            downloaded[i].record(d2h_stream)

    for _ in range(3):
        e2e_step()
    barrier(world)
    torch.cuda.synchronize(dev)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    h2d_stream.wait_event(a0)
    for _ in range(e2e_steps):
        e2e_step()
    # the timed region ends when the last download has landed in host memory
    for ev_d in downloaded:
        stream.wait_event(ev_d)
    a1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_sec = max_over_ranks(a0.elapsed_time(a1) / 1e3, world, dev)
    if bm.device_error() != 0:
        raise RuntimeError("device error during the timed region")

    hbm, tc_burst, tc_sust, peak_src = measured_peaks()
    costs = layer_costs(M, H, E, I, k, args.feed)
    rl_gu = roofline_entry("moe_gemm_kernel<gate_up> (tcgen05 grouped GEMM + SwiGLU*p epilogue)",
                           costs["gate_up"], gu_ms, hbm, tc_burst, peak_src,
                           captured_traffic(args.workload, M, "gate_up"))
    rl_dn = roofline_entry("moe_gemm_kernel<down> (tcgen05 grouped GEMM, fp32 per-slot contributions)",
                           costs["down"], dn_ms, hbm, tc_burst, peak_src,
                           captured_traffic(args.workload, M, "down"))
    rl_step = roofline_entry(f"whole step ({launches_per_step(M, E, args.feed)} launches: router + top-k, "
                             "permutation, " + ("gather, " if args.feed == "copy" else "") +
                             "gate/up, down, combine)", costs["step"], sec_max / args.steps * 1e3, hbm, tc_burst,
                             peak_src)

    extras, summary = {}, {}
    # the secondary workload and the sweeps characterise one GPU: the N=1
    # run reports them, and a multi-GPU run does not hold the other GPUs idle
    if rank == 0 and world == 1 and not args.no_extras:
        other = "qwen" if args.workload == "dsv4" else "dsv4"
        del b, x_host, out_host, x_dev
        torch.cuda.empty_cache()
        wl2 = WORKLOADS[other]
        b2 = setup_workload(wl2, M, dev, x_seed=21)
        s2_steps = max(3, min(args.steps, 50))
        sec2, gu2, dn2, clk2 = time_steps(wl2, M, b2, s2_steps, args.warmup, 1, stream, dev, args.feed)
        del b2
        torch.cuda.empty_cache()
        c2 = layer_costs(M, wl2["H"], wl2["E"], wl2["I"], wl2["top_k"], args.feed)
        extras["secondary_workload"] = {
            "workload": wl2["name"], "tokens_per_gpu": M, "H": wl2["H"], "E": wl2["E"], "I": wl2["I"],
            "top_k": wl2["top_k"], "steps": s2_steps, "ms_per_step": sec2 / s2_steps * 1e3,
            "tokens_per_s": M * s2_steps / sec2, "clocks": clk2,
            "roofline_gate_up": roofline_entry("gate/up", c2["gate_up"], gu2, hbm, tc_burst, peak_src,
                                               captured_traffic(other, M, "gate_up")),
            "roofline_down": roofline_entry("down", c2["down"], dn2, hbm, tc_burst, peak_src,
                                            captured_traffic(other, M, "down")),
        }
        extras["router_us_vs_M"] = router_sweep(dev)
        extras["moe_layer_us_vs_M"] = moe_sweep(dev, args.workload)
        extras["moe_layer_us_vs_M_" + other] = moe_sweep(dev, other)
        extras["topk_window_us"] = topk_window_sweep(dev)
        summary = summarize(extras, rl_gu, rl_dn, rl_step)

    if rank != 0:
        return None
    line = {
        "metric": "BI MoE-layer tokens/s (whole hot path: router GEMM + top-k + fused experts)",
        "value": aggregate(M, args.steps, world, sec_max),
        "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_max / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 experts / fp32 router", "data": "synthetic (seeded N(0,0.02) weights and tokens)",
        "config": {"workload": wl["name"], "tokens_per_gpu": M, "H": H, "E": E, "top_k": k, "I": I,
                   "router": f"fp32 [{M},{H}] x [{E},{H}]^T", "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (expert weights %.2f GB streamed per step)"
                         % ((E * 3 * I * H * 2) / 1e9)},
        "roofline": rl_gu,
        "rooflines": {"gate_up": rl_gu, "down": rl_dn, "step": rl_step},
        "e2e": {"value": aggregate(M, e2e_steps, world, e2e_sec), "unit": "tokens/s",
                "h2d_bytes_per_step": M * H * 2, "d2h_bytes_per_step": M * H * 2,
                "steps": e2e_steps},
        "gpu_launches": launches_per_step(M, E, args.feed) * args.steps,
        "clocks": clk,
    }
    line.update(extras)
    if summary:
        line["summary"] = summary
    return line


def summarize(extras, rl_gu, rl_dn, rl_step):
    """A short digest of the line (kept last, where a truncated log still
    shows it): kernel rooflines, router and layer time vs M, cuBLAS's row
    flips on the router shape, the secondary workload."""
    def rl(r):
        return {"bound": r["bound"], "frac": round(r["frac"], 3), "achieved": round(r["achieved"], 1),
                "unit": r["unit"], "ms": round(r["ms_per_launch"], 4),
                "tensor_frac_of_burst": round(r["tensor_frac_of_burst"], 3)}
    s = {"rooflines": {"gate_up": rl(rl_gu), "down": rl(rl_dn), "step": rl(rl_step)}}
    r = extras.get("router_us_vs_M", {})
    s["fp32_fma_peak_tflops"] = r.get("fp32_fma_peak_tflops_measured")
    s["router_dsv4_warm_us_fp32frac"] = {m: [r[m]["warm_us"], r[m]["warm_fp32_frac"]]
                                         for m in ("1", "8", "32", "64", "128", "1024", "4096") if m in r}
    s["router_topk_warm_us"] = {m: [r[m].get("fused_router_topk_warm_us"),
                                    r[m].get("chained_router_topk_warm_us")]
                                for m in ("1", "2", "4", "8", "64", "4096") if m in r}
    s["cublas_fp32_rows_changed_vs_M4096"] = {m: r[m].get("cublas_fp32_rows_changed_vs_M4096")
                                              for m in ("1", "8", "64", "128", "256", "1024") if m in r}
    for key, v in extras.items():
        if key.startswith("moe_layer_us_vs_M"):
            s[key.replace("moe_layer_us_vs_M", "layer_cold_us_hbmfrac") or "layer"] = {
                "workload": v.get("workload"),
                **{m: [v[m]["cold_us"], v[m]["cold_hbm_frac"]] for m in ("1", "16", "256", "4096") if m in v}}
    sec = extras.get("secondary_workload")
    if sec:
        s["secondary"] = {"workload": sec["workload"], "tokens_per_s": round(sec["tokens_per_s"]),
                          "ms_per_step": round(sec["ms_per_step"], 4),
                          "gate_up": rl(sec["roofline_gate_up"]), "down": rl(sec["roofline_down"])}
    return s


def fp32_fma_peak(dev):
    """Measured FP32 (non-tensor) FMA throughput of this GPU in TFLOP/s: the
    library's probe kernel (16 independent FMA chains per thread, 8 CTAs of
    256 threads per SM, no memory traffic), timed with CUDA events."""
    import torch

    import invariant_moe_gb300 as bm
    props = torch.cuda.get_device_properties(dev)
    blocks, iters = props.multi_processor_count * 8, 20000
    bm.bi_fp32_fma_probe(blocks, 200)
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        bm.bi_fp32_fma_probe(blocks, iters)
        e1.record()
        e1.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    return blocks * 256 * 16 * 2 * iters / min(ts) / 1e12


def num_sms_of(dev):
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count


def router_sweep(dev, Ms=(1, 2, 3, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048, 4096)):
    """Device us per router call (DSv4 router: K=4096, N=256, fp32, bias) vs M,
    from CUDA-graph replays so host launch cost is excluded.
    warm: a graph of 20 back-to-back calls (W stays in L2);
    cold: a graph of 20 x (256 MB L2-flushing write, call) minus a graph of
    the 20 flushes alone."""
    import torch

    import invariant_moe_gb300 as bm
    from tests import synthetic as syn
    inp = syn.router_inputs()
    x, w, b = inp.x.to(dev), inp.w.to(dev), inp.b.to(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    n = 20

    def graph_time(fn, reps=5):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def flushes():
        for _ in range(n):
            flush.fill_(1.0)

    t_flush = graph_time(flushes)
    fp32_peak = fp32_fma_peak(dev)
    res = {"fp32_fma_peak_tflops_measured": round(fp32_peak, 2)}
    # the floor of one kernel in this measurement: a grid of one 256-thread
    # CTA per SM doing next to nothing (the FP32 probe with one step)
    probe_out = torch.empty(num_sms_of(dev) * 256, dtype=torch.float32, device=dev)

    def empty_calls():
        for _ in range(n):
            bm.bi_fp32_fma_probe(num_sms_of(dev), 1, stream=stream, out=probe_out)

    res["empty_kernel_floor_us"] = round(graph_time(empty_calls) / n, 2)
    for M in Ms:
        xm = x[:M].contiguous()
        y = torch.empty(M, 256, dtype=torch.float32, device=dev)

        def calls():
            for _ in range(n):
                bm.bi_router_gemm(xm, w, b, out=y, stream=stream)

        def cold_calls():
            for _ in range(n):
                flush.fill_(1.0)
                bm.bi_router_gemm(xm, w, b, out=y, stream=stream)

        warm = graph_time(calls) / n
        cold = (graph_time(cold_calls) - t_flush) / n
        xb = xm.to(torch.bfloat16)

        def bf16_calls():
            for _ in range(n):
                bm.bi_router_gemm(xb, w, b, out=y, stream=stream)

        warm_bf16 = graph_time(bf16_calls) / n
        flops = 2.0 * M * 4096 * 256
        bytes_ = 4.0 * (256 * 4096 + 256 + M * (4096 + 256))
        res[str(M)] = {"warm_us": round(warm, 2), "cold_us": round(cold, 2),
                       "cold_hbm_frac": round(bytes_ / (cold * 1e-6) / 1e9 / measured_peaks()[0], 3),
                       "warm_tflops": round(flops / (warm * 1e-6) / 1e12, 2),
                       "warm_fp32_frac": round(flops / (warm * 1e-6) / 1e12 / fp32_peak, 3),
                       "bf16x_warm_us": round(warm_bf16, 2),
                       "bf16x_warm_fp32_frac": round(flops / (warm_bf16 * 1e-6) / 1e12 / fp32_peak, 3)}
        # router + selection: two launches (bi_router_gemm, bi_topk) against
        # the fused bi_router_topk, top-8 of the 256 scores
        ids = torch.empty(M, 8, dtype=torch.int32, device=dev)
        wts = torch.empty(M, 8, dtype=torch.float32, device=dev)

        def two_calls():
            for _ in range(n):
                bm.bi_router_gemm(xm, w, b, out=y, stream=stream)
                bm.bi_topk(y, 8, ids=ids, wts=wts, stream=stream)

        def fused_calls():
            for _ in range(n):
                bm.bi_router_topk(xm, w, 8, bias=b, out=y, stream=stream)

        # every schedule on the same rows (1 rows, 2 sliced, 3 tiled, 4 split
        # with the tile picked from M, 5..8 split with each lane tile, 9 tiled
        # with 7x8 lane tiles)
        sched = {}
        for s_ in ((1,) if M <= 64 else ()) + (2, 3, 4, 5, 6, 7, 8, 9):
            def scalls(s_=s_):
                for _ in range(n):
                    bm.bi_router_gemm(xm, w, b, out=y, schedule=s_, stream=stream)
            sched[str(s_)] = round(graph_time(scalls) / n, 2)
        res[str(M)]["schedule_warm_us"] = sched
        res[str(M)]["router_plus_topk_warm_us"] = round(graph_time(two_calls) / n, 2)
        res[str(M)]["fused_router_topk_warm_us"] = round(graph_time(fused_calls) / n, 2)
        if M <= 4:
            # the one-kernel path forced (the automatic choice at these M),
            # and the router grid chained with the selection grid
            def one_kernel_calls():
                for _ in range(n):
                    bm.bi_router_topk(xm, w, 8, bias=b, out=y, schedule=10, stream=stream)

            def chained_calls():
                for _ in range(n):
                    bm.bi_router_topk(xm, w, 8, bias=b, out=y, schedule=1 if M <= 2 else 4, stream=stream)

            res[str(M)]["one_kernel_router_topk_warm_us"] = round(graph_time(one_kernel_calls) / n, 2)
            res[str(M)]["chained_router_topk_warm_us"] = round(graph_time(chained_calls) / n, 2)
        # the library default on the same shape: cuBLAS through torch.matmul,
        # fp32 and TF32, with the rows whose bits differ from the same rows
        # computed in the M=4096 batch (ours: none, by construction)
        for name, tf32 in (("cublas_fp32", False), ("cublas_tf32", True)):
            prev = torch.backends.cuda.matmul.allow_tf32
            torch.backends.cuda.matmul.allow_tf32 = tf32
            try:
                yt = torch.empty(M, 256, dtype=torch.float32, device=dev)

                def tcalls():
                    for _ in range(n):
                        torch.addmm(b, xm, w.t(), out=yt)

                res[str(M)][name + "_warm_us"] = round(graph_time(tcalls) / n, 2)
                with torch.cuda.stream(stream):
                    full = torch.addmm(b, x, w.t())
                    part = torch.addmm(b, xm, w.t())
                    stream.synchronize()
                res[str(M)][name + "_rows_changed_vs_M4096"] = int(
                    (part.view(torch.int32) != full[:M].view(torch.int32)).any(dim=1).sum().item())
            finally:
                torch.backends.cuda.matmul.allow_tf32 = prev
    # the Qwen3-30B-A3B-shaped router (K=2048, N=128, no bias) on bf16 tokens,
    # as the MoE layer calls it
    g = torch.Generator().manual_seed(5)
    xq = torch.randn(4096, 2048, generator=g).to(torch.bfloat16).to(dev)
    wq = (torch.randn(128, 2048, generator=g) * 0.02).to(dev)
    qres = {}
    for M in (16, 64, 256, 1024, 2048, 4096):
        xm = xq[:M].contiguous()
        yq = torch.empty(M, 128, dtype=torch.float32, device=dev)
        sched = {}
        for s_ in (0, 2, 3, 4, 5, 6, 7, 8, 9):
            def qcalls(s_=s_):
                for _ in range(n):
                    bm.bi_router_gemm(xm, wq, None, out=yq, schedule=s_, stream=stream)
            sched[str(s_)] = round(graph_time(qcalls) / n, 2)
        qres[str(M)] = sched
    res["qwen_bf16_schedule_warm_us"] = qres
    return res


def moe_sweep(dev, workload, Ms=(1, 16, 64, 256, 1024, 4096)):
    """Whole-layer device time (moe_layer: cast, router, top-k, experts) vs
    batch size M, through CUDA-graph replay of 10 calls: warm (weights stay
    in L2 between calls where they fit) and cold (a 256 MB L2-flushing write
    before each call, its time subtracted).  HBM fraction: touched-expert
    weights E(1-(1-k/E)^M)*3*I*H*2 + router weights + x and out, over the cold
    time, against the measured copy bandwidth."""
    import torch

    import invariant_moe_gb300 as bm
    from tests import synthetic as syn
    wl = WORKLOADS[workload]
    H, E, I, k = wl["H"], wl["E"], wl["I"], wl["top_k"]
    w = syn.moe_weights(H, E, I, seed=11, device=str(dev))
    x_all = syn.moe_tokens(max(Ms), H, seed=21, device=str(dev))
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    n = 10

    def graph_time(fn, reps=5):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            g.replay()
            stream.synchronize()
            ts = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    def flushes():
        for _ in range(n):
            flush.fill_(1.0)

    t_flush = graph_time(flushes)
    res = {"workload": wl["name"]}
    for M in Ms:
        xm = x_all[:M].contiguous()

        def calls():
            for _ in range(n):
                bm.moe_layer(xm, w.w_router, w.w13, w.w2, k, stream=stream)

        def cold_calls():
            for _ in range(n):
                flush.fill_(1.0)
                bm.moe_layer(xm, w.w_router, w.w13, w.w2, k, stream=stream)

        warm = graph_time(calls) / n
        cold = (graph_time(cold_calls) - t_flush) / n
        touched = E * (1.0 - (1.0 - k / E) ** M)
        bytes_ = touched * 3 * I * H * 2 + E * H * 4 + M * H * 2 * 2
        res[str(M)] = {"warm_us": round(warm, 2), "cold_us": round(cold, 2),
                       "cold_tokens_per_s": round(M / (cold * 1e-6), 1),
                       "cold_hbm_frac": round(bytes_ / (cold * 1e-6) / 1e9 / measured_peaks()[0], 3)}
        # the same layer with each expert-GEMM variant forced (1 one CTA per
        # tile, 2 CTA pairs, 3 CTA pairs with interleaved gate/up rows, 4 one
        # CTA per tile with interleaved gate/up rows)
        var = {}
        for v in (1, 2, 3, 4):
            prev = bm.bi_moe_gemm_variant(v)
            try:
                var[str(v)] = round((graph_time(cold_calls) - t_flush) / n, 2)
            finally:
                bm.bi_moe_gemm_variant(prev)
        res[str(M)]["gemm_variant_cold_us"] = var
    if bm.device_error() != 0:
        raise RuntimeError("device error in the MoE sweep")
    return res


def topk_window_sweep(dev, ns=(1, 8, 64), ks=(512, 1024, 2048), num_cols=8192):
    """Windowed per-row top-k (the sparse-MLA indexer's selection) device time
    per call, CUDA-graph replay of 20 calls, on relu-plateau rows (about half
    the scores exactly zero) with each row's window the whole row."""
    import torch

    import invariant_moe_gb300 as bm
    g = torch.Generator().manual_seed(77)
    x = torch.randn(max(ns), num_cols, generator=g).clamp_min(0.0).to(dev)
    flat = torch.zeros(max(ns), num_cols, device=dev)  # the worst case: one plateau
    stream = torch.cuda.Stream(dev)
    n_calls = 20
    res = {"num_cols": num_cols, "scores": "relu(N(0,1)): about half exact zeros"}
    for n in ns:
        for k in ks:
            out = torch.empty(n, k, dtype=torch.int32, device=dev)
            xs = x[:n].contiguous()

            def calls():
                for _ in range(n_calls):
                    bm.bi_topk_window(xs, k, out=out, stream=stream)

            with torch.cuda.stream(stream):
                calls()
                stream.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=stream):
                    calls()
                gr.replay()
                stream.synchronize()
                ts = []
                for _ in range(5):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    gr.replay()
                    e1.record(stream)
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3 / n_calls)
            res[f"n{n}_k{k}_us"] = round(statistics.median(ts), 2)
    # every score equal: each radix pass puts the whole row in one bin
    out = torch.empty(max(ns), 1024, dtype=torch.int32, device=dev)
    xs = flat.contiguous()

    def flat_calls():
        for _ in range(n_calls):
            bm.bi_topk_window(xs, 1024, out=out, stream=stream)

    with torch.cuda.stream(stream):
        flat_calls()
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            flat_calls()
        gr.replay()
        stream.synchronize()
        ts = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / n_calls)
    res[f"all_equal_n{max(ns)}_k1024_us"] = round(statistics.median(ts), 2)
    return res


# ------------------------------------------------------ oracle (CPU) arm --
class OracleSample:
    """Times the fp64 oracle (router, top-k, experts; one host thread) on a
    few tokens of a workload.  The weights are the bench's own, generated on
    the GPU with the same seeds, when a GPU is present; the oracle receives
    only the experts the sampled tokens are routed to (copied to the host
    outside the timed part).  Without a GPU the router weight is drawn on
    the host and each routed expert from its own seeded host stream: the same
    shapes and distributions, other values."""

    def __init__(self, workload, dev=None):
        import oracle
        from tests import synthetic as syn
        oracle.build()
        self.wl = WORKLOADS[workload]
        H, E, I = self.wl["H"], self.wl["E"], self.wl["I"]
        self.dev = dev
        if dev is not None:
            self.w = syn.moe_weights(H, E, I, seed=11, device=str(dev))
            self.wr = self.w.w_router.cpu().numpy()
        else:
            self.w = None
            self.wr = syn.normal((E, H), 0.02, 12).numpy()

    def _experts(self, used):
        """(w13 bits [n,2I,H], w2 bits [n,H,I]) of the experts in `used`."""
        import numpy as np
        import torch

        from tests import synthetic as syn
        H, I = self.wl["H"], self.wl["I"]
        if self.w is not None:
            idx = torch.from_numpy(np.asarray(used, np.int64)).to(self.w.w13.device)
            return syn.bf16_bits(self.w.w13[idx]), syn.bf16_bits(self.w.w2[idx])
        w13 = np.stack([syn.bf16_bits(syn.normal((2 * I, H), 0.02, 5000 + 2 * int(e), torch.bfloat16))
                        for e in used])
        w2 = np.stack([syn.bf16_bits(syn.normal((H, I), 0.02, 5001 + 2 * int(e), torch.bfloat16))
                       for e in used])
        return w13, w2

    def run(self, n_tokens, seed):
        """Seconds the oracle takes for n_tokens tokens (routing + experts)."""
        import numpy as np

        import oracle
        from tests import synthetic as syn
        H, I, k = self.wl["H"], self.wl["I"], self.wl["top_k"]
        x = syn.moe_tokens(n_tokens, H, seed=seed)
        xb = syn.bf16_bits(x)
        t = time.perf_counter()
        r = oracle.router(x.float().numpy(), self.wr)
        ids, wts = oracle.topk(r.astype("float32"), k)
        t_route = time.perf_counter() - t
        used = np.unique(ids)
        w13, w2 = self._experts(used)
        remap = np.full(self.wl["E"], -1, np.int32)
        remap[used] = np.arange(len(used), dtype=np.int32)
        t = time.perf_counter()
        oracle.moe(xb, remap[ids], wts.astype("float32"), w13, w2, len(used), I)
        return t_route + time.perf_counter() - t


def cpu_baseline(args, sampler, budget_s=12.0):
    n, total, tok = 2, 0.0, 0
    while total < budget_s:
        total += sampler.run(n, seed=100 + tok)
        tok += n
    return {"value": tok / total, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{tok} tokens of the {WORKLOADS[args.workload]['name']} workload "
                      f"(fp64 router + top-k + experts, single thread, {total:.1f} s)"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    dev = None
    try:
        import torch
        if torch.cuda.is_available():
            dev = torch.device("cuda", 0)
    except ImportError:
        pass
    sampler = OracleSample(args.workload, dev)
    wl = WORKLOADS[args.workload]
    per_step = 1  # tokens per step: a bounded sample of the workload
    for _ in range(args.warmup):
        sampler.run(per_step, seed=900)
    t = 0.0
    for s in range(args.steps):
        t += sampler.run(per_step, seed=1000 + s)
    value = per_step * args.steps / t
    return {
        "impl": "reference",
        "metric": "BI MoE-layer tokens/s (whole hot path: router GEMM + top-k + fused experts)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["name"], "tokens_per_gpu": args.tokens, "H": wl["H"], "E": wl["E"],
                   "top_k": wl["top_k"], "I": wl["I"], "parallelism": "oracle on 1 host core"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} token(s) per step, fp64 single thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(WORKLOADS), default="dsv4")
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--feed", choices=("gemm", "copy"), default="copy",
                    help="how the gate/up GEMM gets the token rows: from the gather kernel's contiguous "
                         "copy (the layer's path) or gathered by the GEMM itself (tile::gather4)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the workload's expert count (a smaller case of the same "
                         "tokens-per-expert load, for ncu captures that must stay small)")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--router-sweep", action="store_true",
                    help="only print the router device-time sweep (DSv4 router shape)")
    ap.add_argument("--router-ms", default=None,
                    help="comma-separated batch sizes for --router-sweep (default: 1 ... 4096)")
    ap.add_argument("--topk-window-sweep", action="store_true",
                    help="only print the windowed top-k device-time sweep")
    ap.add_argument("--moe-sweep", action="store_true",
                    help="only print the whole-layer device-time sweep over M for --workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()
    if args.experts is not None:
        wl = dict(WORKLOADS[args.workload])
        wl["E"] = args.experts
        wl["name"] = f"{wl['name']}-E{args.experts}"
        WORKLOADS[args.workload] = wl
    if args.router_sweep:
        import torch
        torch.cuda.set_device(local)
        kw = {"Ms": tuple(int(m) for m in args.router_ms.split(","))} if args.router_ms else {}
        print(json.dumps({"router_us_vs_M": router_sweep(torch.device("cuda", local), **kw)}), flush=True)
        return
    if args.topk_window_sweep:
        import torch
        torch.cuda.set_device(local)
        print(json.dumps({"topk_window_us": topk_window_sweep(torch.device("cuda", local))}), flush=True)
        return
    if args.moe_sweep:
        import torch
        torch.cuda.set_device(local)
        print(json.dumps({"moe_layer_us_vs_M": moe_sweep(torch.device("cuda", local), args.workload)}),
              flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
        # the oracle's CPU baseline is timed at N=1 only
        if line is not None and world == 1 and not args.no_cpu_baseline:
            import torch
            summary = line.pop("summary", None)
            line["cpu_baseline"] = cpu_baseline(args, OracleSample(args.workload, torch.device("cuda", local)))
            if summary is not None:
                line["summary"] = summary
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
