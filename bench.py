"""Benchmark of the Flint MoE layer on B300 (one JSON line on stdout).

Default workload: the decode sweep -- one Flint-shaped layer (seed-0 weights) run at
T = 1, 2, 4, 8, 16, 32, 64 tokens (x ~ N(0,1) bf16, seed 1000+T).  One step is one forward
at every T of the sweep (127 tokens); L2 is flushed (a 512 MB write) before every forward,
outside the timed spans; each forward is timed with CUDA events on its stream.  value =
tokens of all ranks / max over ranks of the summed forward times.

Other workloads (--workload): single (T=16, seed 0), prefill (T=8192, router bias
~N(0, 0.5)), stack (47 pre-norm residual layers, T=256), adversarial (T=16384, +8/-8 bias
with tied router columns).

Multi-GPU (torchrun, one rank per GPU): independent replicas, no collective on the data
path; ranks only meet at the timing barriers.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
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

SWEEP = (1, 2, 4, 8, 16, 32, 64)
METRIC = "MoE-layer tokens/s on 1 B300; HBM GB/s (decode) / tensor TFLOPS (prefill) vs peak"


def sweep_config(world):
    """The decode-sweep workload's config object (identical on both arms)."""
    return dict(workload="decode sweep: one Flint MoE layer (H2048 E256 top6 I512 shared1024), "
                         "T=1,2,4,8,16,32,64 per step",
                tokens_per_step=sum(SWEEP), parallelism=f"replicas x{world}",
                l2="flushed (512 MB write) before every forward")


def host_cpu():
    """The host's logical core count and CPU model (for the oracle's baseline lines)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return dict(nproc=os.cpu_count(), cpu_model=model)


KERNEL_SOURCES = ("sparse_moe_layer_15_b300/csrc/decode_fused.cuh", "sparse_moe_layer_15_b300/csrc/common.cuh",
                  "sparse_moe_layer_15_b300/csrc/flint_moe.cu")


# The sources the prefill path's tensor-core kernels are built from.
PREFILL_SOURCES = ("sparse_moe_layer_15_b300/csrc/prefill_kernels.cuh", "sparse_moe_layer_15_b300/csrc/tc_gemm.cuh",
                   "sparse_moe_layer_15_b300/csrc/common.cuh", "sparse_moe_layer_15_b300/csrc/flint_moe.cu")


def kernel_sources_sha256(sources=KERNEL_SOURCES):
    import hashlib
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_prefill_traffic(kernel, workload):
    """DRAM bytes per launch of the prefill kernel `kernel` on `workload`, from the committed ncu
    summary profiles/<kernel>_traffic.json, or None when the prefill sources have changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("sources_sha256") != kernel_sources_sha256(PREFILL_SOURCES):
        return None
    return rec.get("dram_bytes_per_launch", {}).get(workload)


def measured_traffic(kernel, sweep):
    """DRAM bytes per launch of `kernel` averaged over the sweep, from the committed ncu
    summary profiles/decode_fused_traffic.json, or None when the kernel sources have changed
    since the counters were taken (or no summary exists)."""
    path = os.path.join(ROOT, "profiles", "decode_fused_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("kernel") != kernel or rec.get("sources_sha256") != kernel_sources_sha256():
        return None
    per = rec["dram_bytes_per_launch"]
    if not all(str(T) in per for T in sweep):
        return None
    return round(sum(per[str(T)] for T in sweep) / len(sweep))


def measured_stack_traffic(T, n_layers):
    """DRAM bytes of one launch of decode_stack over n_layers at T tokens: the committed ncu
    summary profiles/decode_stack_traffic.json holds a small stack's bytes per layer (the
    weights of each layer are streamed once, so the bytes scale with the layers); None when the
    sources changed since or the summary has no entry for T."""
    path = os.path.join(ROOT, "profiles", "decode_stack_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("sources_sha256") != kernel_sources_sha256():
        return None
    per = rec.get("dram_bytes_per_layer", {}).get(str(T))
    return None if per is None else round(per * n_layers)


# The B300's nominal HBM3e bandwidth and dense bf16 rate, for the "spec" fractions next to the
# measured ones.
SPEC_HBM_GBS = 8000.0
SPEC_BF16_TFLOPS = 2250.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                    reasons=sorted(reasons), samples=len(sm))


def dist_setup():
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm
    from sparse_moe_layer_15_b300 import accounting as acc

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(4 * l2, 512 << 20), dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    w = synth.flint_weights(seed=0, device=dev)
    layer = fm.FlintMoE(w, max_tokens=max(SWEEP))
    xs = {T: synth.torch_normal_bf16((T, fm.HIDDEN), 1000 + T, synth.TAG_X, 1.0, device=dev) for T in SWEEP}
    ys = {T: torch.empty_like(xs[T]) for T in SWEEP}
    idx = {T: torch.empty((T, fm.TOP_K), dtype=torch.int32, device=dev) for T in SWEEP}
    gw = {T: torch.empty((T, fm.TOP_K), dtype=torch.float32, device=dev) for T in SWEEP}
    ev = {T: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for T in SWEEP}

    def step(times):
        for T in SWEEP:
            flush()
            a, b = ev[T]
            a.record(stream)
            layer.forward(xs[T], y=ys[T], topk_idx=idx[T], topk_w=gw[T])
            b.record(stream)
        torch.cuda.synchronize()
        for T in SWEEP:
            times[T].append(ev[T][0].elapsed_time(ev[T][1]))

    warm = {T: [] for T in SWEEP}
    for _ in range(args.warmup):
        step(warm)
    if layer.poll_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    # touched experts per T (for the algorithmic bytes)
    U = {}
    for T in SWEEP:
        _, _, c = layer.route(xs[T])
        torch.cuda.synchronize()
        U[T] = int((c > 0).sum().item())

    times = {T: [] for T in SWEEP}
    clocks = ClockSampler(local)
    clocks.start()
    # keep the GPU busy (untimed) long enough for the clock sampler to see it under load
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.5:
        step({T: [] for T in SWEEP})
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        step(times)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    barrier(world)
    if layer.poll_device_status() != 0:
        raise RuntimeError("device status error in the timed region")

    ms_step_local = sum(statistics.mean(times[T]) for T in SWEEP)
    ms_step = max_over_ranks(ms_step_local, world)
    tokens_step = sum(SWEEP)
    value = world * tokens_step / (ms_step * 1e-3)

    sweep = {}
    for T in SWEEP:
        med = statistics.median(times[T])
        q = sorted(times[T])
        b = acc.algorithmic_bytes(U[T], T)
        sweep[str(T)] = dict(us=round(med * 1e3, 2), us_p10=round(q[len(q) // 10] * 1e3, 2),
                             us_p90=round(q[(9 * len(q)) // 10] * 1e3, 2), tokens_per_s=round(T / (med * 1e-3), 1),
                             touched_experts=U[T], alg_bytes=b, gbs=round(b / (med * 1e-3) / 1e9, 1),
                             hbm_frac=round(b / (med * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                             hbm_frac_spec=round(b / (med * 1e-3) / 1e9 / SPEC_HBM_GBS, 4))

    # per-kernel times (second pass with kernel events; same workload, same flushes)
    layer.enable_kernel_timing(True)
    kt = {}
    for _ in range(max(3, min(args.steps, 10))):
        for T in SWEEP:
            flush()
            layer.forward(xs[T], y=ys[T], topk_idx=idx[T], topk_w=gw[T])
            for name, ms in layer.kernel_times():
                kt.setdefault(name, {}).setdefault(T, []).append(ms)
    layer.enable_kernel_timing(False)
    kernels = {}
    for name, per_t in kt.items():
        kernels[name] = {str(T): round(statistics.median(v) * 1e3, 2) for T, v in per_t.items()}
    # dominant kernel: largest summed time over the sweep
    dom = max(kt, key=lambda n: sum(statistics.mean(v) for v in kt[n].values()))

    # The decode kernel runs the whole layer: its algorithmic bytes per launch are the layer's
    # (touched experts x 6 MB + shared 12 MB + router 1 MB + bf16 x and y); averaged over the
    # sweep's launches (one per T).
    dom_bytes = sum(acc.algorithmic_bytes(U[T], T) for T in SWEEP) / len(SWEEP)
    dom_ms = sum(statistics.mean(kt[dom][T]) for T in SWEEP) / len(SWEEP)
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = measured_traffic(dom, SWEEP)
    roofline = dict(bound="hbm", kernel=dom, achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=round(achieved / peaks["hbm_gbs"], 4), traffic=traffic,
                    frac_vs_spec=round(achieved / SPEC_HBM_GBS, 4),
                    alg_bytes_per_launch=round(dom_bytes), peak_source=peaks["source"] + " (hbm_gbs, copy test)",
                    note="per-launch means over the sweep's 7 launches; traffic: DRAM read+write bytes per "
                         "launch from the committed ncu summary (null if the kernel sources changed since)")

    # end to end through the C ABI with host buffers (H2D of x and D2H of y inside the span)
    xh = {T: xs[T].cpu().pin_memory() for T in SWEEP}
    yh = {T: torch.empty_like(xh[T]).pin_memory() for T in SWEEP}
    e2e_t = {T: [] for T in SWEEP}
    for it in range(args.warmup + args.steps):
        for T in SWEEP:
            flush()
            a, b = ev[T]
            a.record(stream)
            layer.forward_host(xh[T], yh[T])
            b.record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            for T in SWEEP:
                e2e_t[T].append(ev[T][0].elapsed_time(ev[T][1]))
    e2e_ms = max_over_ranks(sum(statistics.mean(e2e_t[T]) for T in SWEEP), world)
    e2e = dict(value=round(world * tokens_step / (e2e_ms * 1e-3), 1), unit="tokens/s",
               h2d_bytes_per_step=2 * fm.HIDDEN * tokens_step, d2h_bytes_per_step=2 * fm.HIDDEN * tokens_step)

    out = dict(metric=METRIC, value=round(value, 1), unit="tokens/s", n_gpus=world, steps=args.steps,
               warmup=args.warmup, ms_per_step=round(ms_step, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="bf16", data="synthetic", config=sweep_config(world),
               sweep=sweep, kernels_us=kernels, roofline=roofline, e2e=e2e,
               gpu_launches=args.steps * len(SWEEP), clocks=clk, wall_s=round(wall, 3))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, xs, budget_s=args.cpu_budget)
    layer.close()
    del layer, w
    torch.cuda.empty_cache()
    if not args.no_configs:
        # the other configurations, each measured on its own (own clocks, own roofline, own e2e)
        out["configs"] = {}
        for name in ("single", "prefill", "adversarial", "stack"):
            sub_args = argparse.Namespace(**vars(args))
            sub_args.workload = name
            sub_args.steps = min(args.steps, 20)
            r = run_workload(sub_args, rank, world, local, summary=True)
            out["configs"][name] = r
            torch.cuda.empty_cache()
        # the rows beyond the MoE layer: the dense MLP layers and sliding-window decode attention
        out["extra"] = {}
        for T in (1, 64, 8192):
            out["extra"][f"dense_T{T}"] = run_dense(args, local, T)
        for B in (64, 256):
            out["extra"][f"swa_B{B}"] = run_swa(args, local, B)
        out["extra"]["nvfp4_decode_sweep"] = run_nvfp4_sweep(args, local)
        torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- other workloads

WORKLOADS = {
    "single": dict(T=16, seed_x=0, bias=None, bias_seed=None,
                   desc="single Flint MoE layer, T=16 tokens, seed 0 (x seed 0)"),
    "prefill": dict(T=8192, seed_x=3, bias="normal", bias_seed=3,
                    desc="prefill: one Flint MoE layer, T=8192, router bias ~N(0, 0.5) (seed 3), x seed 3"),
    "adversarial": dict(T=16384, seed_x=5, bias="adversarial", bias_seed=5,
                        desc="adversarial: one Flint MoE layer, T=16384, router bias +8 on 8 hot / -8 on 200 cold "
                             "experts, duplicated router columns (exact ties), x seed 5"),
}

# Algorithmic FLOPs per token of each prefill kernel (2 per multiply-add).
PF_KERNEL_FLOPS_PER_TOKEN = {
    "pf_router": 2 * 2048 * 256,
    "pf_gateup": 6 * 2 * 2 * 2048 * 512 + 2 * 2 * 2048 * 1024,
    "pf_down": 6 * 2 * 512 * 2048 + 2 * 1024 * 2048,  # routed and shared down projections
}


def timed_loop(fn, steps, flush, stream, ev):
    import torch
    out = []
    for _ in range(steps):
        if flush:
            flush()
        a, b = ev
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return out


def summarize(out):
    """The per-configuration entry of the default line: the workload's own line without the
    keys that belong to the whole run."""
    drop = ("metric", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "dtype",
            "data")
    r = {k: v for k, v in out.items() if k not in drop}
    r["tokens_per_s"] = r.pop("value")
    return r


def run_workload(args, rank, world, local, summary=False):
    """One workload other than the decode sweep: a step is one forward of T tokens (the
    47-layer stack: 47 pre-norm residual forwards of T=256 tokens).  summary=True: the entry of
    the default line's `configs` object (no CPU baseline)."""
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm
    from sparse_moe_layer_15_b300 import accounting as acc

    if args.workload == "stack":
        return run_stack(args, rank, world, local, summary=summary)
    cfg = WORKLOADS[args.workload]
    T = cfg["T"]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    w = synth.flint_weights(seed=0, device=dev, bias=cfg["bias"], bias_seed=cfg["bias_seed"])
    layer = fm.FlintMoE(w, max_tokens=T)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), cfg["seed_x"], synth.TAG_X, 1.0, device=dev)
    y = torch.empty_like(x)
    idx = torch.empty((T, fm.TOP_K), dtype=torch.int32, device=dev)
    gw = torch.empty((T, fm.TOP_K), dtype=torch.float32, device=dev)
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def fwd():
        layer.forward(x, y=y, topk_idx=idx, topk_w=gw)

    timed_loop(fwd, args.warmup, flush, stream, ev)
    _, _, c = layer.route(x)
    torch.cuda.synchronize()
    counts = c.cpu().numpy()
    U = int((counts > 0).sum())
    clocks = ClockSampler(local)
    clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.5:
        timed_loop(fwd, 1, flush, stream, ev)
    barrier(world)
    times = timed_loop(fwd, args.steps, flush, stream, ev)
    clk = clocks.stop()
    q = sorted(times)
    barrier(world)
    if layer.poll_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    ms = max_over_ranks(statistics.mean(times), world)
    value = world * T / (ms * 1e-3)
    flop = acc.flops_per_token() * T
    alg_bytes = acc.algorithmic_bytes(U, T)
    # per-kernel times (second pass with kernel events)
    layer.enable_kernel_timing(True)
    kt = {}
    for _ in range(max(3, min(args.steps, 10))):
        flush()
        fwd()
        for name, kms in layer.kernel_times():
            kt.setdefault(name, []).append(kms)
    layer.enable_kernel_timing(False)
    kernels = {k: round(statistics.median(v) * 1e3, 2) for k, v in kt.items()}
    dom = max(kt, key=lambda n: statistics.mean(kt[n]))
    dom_ms = statistics.mean(kt[dom])
    if dom in PF_KERNEL_FLOPS_PER_TOKEN:
        achieved = PF_KERNEL_FLOPS_PER_TOKEN[dom] * T / (dom_ms * 1e-3) / 1e12
        roofline = dict(bound="tensor", kernel=dom, achieved=round(achieved, 1), peak=peaks["bf16_tflops"],
                        unit="TFLOP/s", frac=round(achieved / peaks["bf16_tflops"], 4),
                        traffic=measured_prefill_traffic(dom, args.workload),
                        frac_vs_spec=round(achieved / SPEC_BF16_TFLOPS, 4),
                        alg_flop_per_launch=PF_KERNEL_FLOPS_PER_TOKEN[dom] * T,
                        peak_source=peaks["source"] + " (bf16_tflops, burst)",
                        note="algorithmic FLOPs of the kernel (no tile padding) / its CUDA-event time")
    else:
        achieved = alg_bytes / (dom_ms * 1e-3) / 1e9
        roofline = dict(bound="hbm", kernel=dom, achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                        frac=round(achieved / peaks["hbm_gbs"], 4), traffic=None, alg_bytes_per_launch=alg_bytes,
                        peak_source=peaks["source"] + " (hbm_gbs, copy test)")
    # end to end with host buffers
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e2e_t = timed_loop(lambda: layer.forward_host(xh, yh), args.warmup + args.steps, flush, stream, ev)[args.warmup:]
    e2e_ms = max_over_ranks(statistics.mean(e2e_t), world)
    t_roof_ms = max(alg_bytes / (peaks["hbm_gbs"] * 1e9), flop / (peaks["bf16_tflops"] * 1e12)) * 1e3
    out = dict(metric=METRIC, value=round(value, 1), unit="tokens/s", n_gpus=world, steps=args.steps,
               warmup=args.warmup, ms_per_step=round(ms, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="bf16", data="synthetic",
               config=dict(workload=cfg["desc"], tokens_per_step=T, parallelism=f"replicas x{world}",
                           l2="flushed (512 MB write) before every forward"),
               layer=dict(touched_experts=U, alg_bytes=alg_bytes, alg_flop=flop,
                          tflops=round(flop / (ms * 1e-3) / 1e12, 1), gbs=round(alg_bytes / (ms * 1e-3) / 1e9, 1),
                          roofline_ms=round(t_roof_ms, 4), roofline_frac=round(t_roof_ms / ms, 4),
                          us_median=round(statistics.median(times) * 1e3, 2), us_p10=round(q[len(q) // 10] * 1e3, 2),
                          us_p90=round(q[(9 * len(q)) // 10] * 1e3, 2),
                          hot_share=(round(float(np.sort(counts)[::-1][:8].sum() / counts.sum()), 4)
                                     if args.workload == "adversarial" else None)),
               kernels_us=kernels, roofline=roofline,
               e2e=dict(value=round(world * T / (e2e_ms * 1e-3), 1), unit="tokens/s",
                        h2d_bytes_per_step=2 * fm.HIDDEN * T, d2h_bytes_per_step=2 * fm.HIDDEN * T),
               gpu_launches=args.steps * len(kernels), clocks=clk)
    layer.close()
    if summary:
        return summarize(out)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_tokens(w, x, n=16, what=args.workload)
    return out


def run_stack(args, rank, world, local, summary=False):
    """47 Flint MoE layers (weights seed 100+l, about 76 GB), T=256 tokens (x seed 4); each
    layer x <- x + MoE_l(RMSNorm(x)), eps 1e-6.  One step = the 47 forwards, through the stack
    call (one launch of decode_stack for all layers).  --stack-tokens T measures the same stack at
    T tokens; --stack-layers N < 47 is a small case for the profiler, not the configuration."""
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm
    from sparse_moe_layer_15_b300 import accounting as acc

    L, T = args.stack_layers, args.stack_tokens
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    ws = torch.empty(fm.workspace_bytes(T, flags, 1e-6), dtype=torch.uint8, device=dev)
    weights = [synth.flint_weights(seed=100 + l, device=dev) for l in range(L)]
    layers = [fm.FlintMoE(weights[l], max_tokens=T, flags=flags, rms_eps=1e-6, workspace=ws) for l in range(L)]
    # the public stack call: one launch of decode_stack for all layers
    stack_handle = fm.FlintMoEStack(weights, max_tokens=T, flags=flags, rms_eps=1e-6)
    x0 = synth.torch_normal_bf16((T, fm.HIDDEN), 4, synth.TAG_X, 1.0, device=dev)
    x = x0.clone()
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def stack():
        stack_handle.forward(x)

    timed_loop(stack, args.warmup, None, stream, ev)
    # touched experts per layer on the layer inputs of one pass
    U = []
    x.copy_(x0)
    for lay in layers:
        _, _, c = lay.route(x)
        U.append(int((c > 0).sum().item()))
        lay.forward(x, y=x)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 1.5:
        x.copy_(x0)
        timed_loop(stack, 1, None, stream, ev)
    barrier(world)
    times = []
    for _ in range(args.steps):
        x.copy_(x0)
        times += timed_loop(stack, 1, None, stream, ev)
    clk = clocks.stop()
    barrier(world)
    for lay in layers:
        if lay.poll_device_status() != 0:
            raise RuntimeError("device status error in the timed region")
    if stack_handle.poll_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    ms = max_over_ranks(statistics.mean(times), world)
    alg_bytes = sum(acc.algorithmic_bytes(u, T) for u in U)
    flop = acc.flops_per_token() * T * L
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    roofline = dict(bound="hbm", kernel=f"decode_stack (one launch, {L} layers)", achieved=round(achieved, 1),
                    peak=peaks["hbm_gbs"], unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4),
                    traffic=measured_stack_traffic(T, L), alg_bytes_per_launch=round(alg_bytes),
                    peak_source=peaks["source"] + " (hbm_gbs, copy test)",
                    note="the step is one launch; traffic: DRAM bytes per layer from the committed ncu "
                         "summary of a small stack, times the layers (null if the sources changed)")
    xh = x0.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()

    def e2e_step():
        x.copy_(xh, non_blocking=True)
        stack()
        yh.copy_(x, non_blocking=True)

    e2e_t = timed_loop(e2e_step, args.warmup + args.steps, None, stream, ev)[args.warmup:]
    e2e_ms = max_over_ranks(statistics.mean(e2e_t), world)
    out = dict(metric=METRIC, value=round(world * T / (ms * 1e-3), 1), unit="tokens/s", n_gpus=world,
               steps=args.steps, warmup=args.warmup, ms_per_step=round(ms, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="bf16", data="synthetic",
               config=dict(workload=f"stack: {L} Flint MoE layers (pre-norm RMSNorm eps 1e-6, residual), T={T}, "
                                    f"weights seed 100+l ({L * 1.62:.0f} GB resident), x seed 4"
                                    + ("" if L == acc.N_MOE_LAYERS else " (a small profiling case)"),
                           tokens_per_step=T, parallelism=f"replicas x{world}",
                           l2=f"inputs larger than L2 ({alg_bytes / 1e9:.1f} GB of touched weights streamed per step)"),
               layer=dict(touched_experts_per_layer=U, alg_bytes=alg_bytes, alg_flop=flop,
                          gbs=round(achieved, 1), roofline_ms=round(alg_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3, 3)),
               roofline=roofline,
               e2e=dict(value=round(world * T / (e2e_ms * 1e-3), 1), unit="tokens/s",
                        h2d_bytes_per_step=2 * fm.HIDDEN * T, d2h_bytes_per_step=2 * fm.HIDDEN * T),
               gpu_launches=args.steps, clocks=clk)
    for lay in layers:
        lay.close()
    stack_handle.close()
    if summary:
        return summarize(out)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_tokens(weights[0], x0, n=min(8, T), what="stack layer 0", eps=1e-6)
    return out


def run_dense(args, local, T):
    """One dense SwiGLU MLP layer (width 6144, weights seed 7, x seed 600+T): tokens/s, and the
    roofline of the layer -- weight bytes (75.5 MB) at the copy bandwidth, or its FLOPs
    (75.5 MFLOP per token) at the bf16 peak, whichever is slower."""
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm

    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    w = synth.dense_weights(seed=7, device=dev)
    layer = fm.FlintDense(w, max_tokens=T)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), 600 + T, synth.TAG_X, 1.0, device=dev)
    y = torch.empty_like(x)
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    steps = min(args.steps, 20)
    timed_loop(lambda: layer.forward(x, y=y), args.warmup, lambda: flush_buf.fill_(1), stream, ev)
    times = timed_loop(lambda: layer.forward(x, y=y), steps, lambda: flush_buf.fill_(1), stream, ev)
    if layer.poll_device_status() != 0:
        raise RuntimeError("device status error (dense layer)")
    layer.enable_kernel_timing(True)
    kt = {}
    for _ in range(3):
        flush_buf.fill_(1)
        layer.forward(x, y=y)
        for name, kms in layer.kernel_times():
            kt.setdefault(name, []).append(kms)
    layer.enable_kernel_timing(False)
    layer.close()
    ms = statistics.mean(times)
    wbytes = 3 * fm.HIDDEN * fm.DENSE_INTER * 2
    alg_bytes = wbytes + 2 * 2 * fm.HIDDEN * T
    flop = 2 * 3 * fm.HIDDEN * fm.DENSE_INTER * T
    t_mem, t_flop = alg_bytes / (peaks["hbm_gbs"] * 1e9), flop / (peaks["bf16_tflops"] * 1e12)
    if t_mem >= t_flop:
        roof = dict(bound="hbm", achieved=round(alg_bytes / (ms * 1e-3) / 1e9, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=round(alg_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4), alg_bytes=alg_bytes)
    else:
        roof = dict(bound="tensor", achieved=round(flop / (ms * 1e-3) / 1e12, 1), peak=peaks["bf16_tflops"],
                    unit="TFLOP/s", frac=round(flop / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4), alg_flop=flop)
    roof.update(kernel="+".join(sorted(kt)), traffic=None, note="the whole layer call / its CUDA-event time")
    return dict(workload=f"dense SwiGLU MLP layer (2048 -> 6144 -> 2048), T={T}, L2 flushed before every call",
                tokens_per_s=round(T / (ms * 1e-3), 1), us_median=round(statistics.median(times) * 1e3, 2),
                kernels_us={k: round(statistics.median(v) * 1e3, 2) for k, v in kt.items()}, roofline=roof,
                gpu_launches=steps * len(kt))


# NVFP4 bytes: E2M1 codes (4 bits) + one E4M3 scale per 16 weights = 4.5 bits per weight.
NVFP4_EXPERT_BYTES = 3 * 2048 * 512 // 2 + 3 * 2048 * 512 // 16      # 1,769,472 per routed expert
NVFP4_SHARED_BYTES = 3 * 2048 * 1024 // 2 + 3 * 2048 * 1024 // 16    # 3,538,944


def nvfp4_alg_bytes(U, T):
    """Touched bytes of one layer call on NVFP4 expert weights: U experts' codes and scales, the
    shared expert's, the bf16 router (1 MB) and the bf16 input and output rows."""
    return U * NVFP4_EXPERT_BYTES + NVFP4_SHARED_BYTES + 2048 * 256 * 2 + 2 * 2 * 2048 * T


def run_nvfp4_sweep(args, local):
    """The decode sweep (T = 1..64, x seed 1000+T, L2 flushed before every forward) on NVFP4
    expert weights quantised from the seed-0 layer: tokens/s and the HBM roofline of the 4.5-bit
    weight stream."""
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm

    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    w = synth.flint_weights(seed=0, device=dev)
    q = synth.nvfp4_weights(w)
    wr = w["w_router"]
    del w
    layer = fm.FlintMoE.nvfp4(wr, q, max_tokens=max(SWEEP))
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    steps = min(args.steps, 20)
    per_t, tot_ms, tot_bytes = {}, 0.0, 0
    for T in SWEEP:
        x = synth.torch_normal_bf16((T, fm.HIDDEN), 1000 + T, synth.TAG_X, 1.0, device=dev)
        y = torch.empty_like(x)
        timed_loop(lambda: layer.forward(x, y=y), args.warmup, lambda: flush_buf.fill_(1), stream, ev)
        times = timed_loop(lambda: layer.forward(x, y=y), steps, lambda: flush_buf.fill_(1), stream, ev)
        _, _, c = layer.route(x)
        torch.cuda.synchronize()
        U = int((c > 0).sum().item())
        ms = statistics.mean(times)
        b = nvfp4_alg_bytes(U, T)
        tot_ms += ms
        tot_bytes += b
        per_t[str(T)] = dict(us=round(statistics.median(times) * 1e3, 2), touched_experts=U, alg_bytes=b,
                             hbm_frac=round(b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4))
    if layer.poll_device_status() != 0:
        raise RuntimeError("device status error (nvfp4)")
    layer.close()
    gbs = tot_bytes / (tot_ms * 1e-3) / 1e9
    return dict(workload="decode sweep T=1..64 on NVFP4 expert weights (E2M1 + E4M3 per 16 + fp32 per matrix; "
                         "router bf16), L2 flushed before every forward",
                tokens_per_s=round(sum(SWEEP) / (tot_ms * 1e-3), 1), ms_per_step=round(tot_ms, 4), sweep=per_t,
                roofline=dict(bound="hbm", kernel="decode_fused (NVFP4 stream)", achieved=round(gbs, 1),
                              peak=peaks["hbm_gbs"], unit="GB/s", frac=round(gbs / peaks["hbm_gbs"], 4),
                              traffic=None, note="4.5-bit weights: U x 1,769,472 + 3,538,944 + 1 MB router + x, y"),
                gpu_launches=steps * len(SWEEP))


def run_swa(args, local, B):
    """Sliding-window decode attention with sinks over B sequences (the input recipe's length
    mix, seed 900+B): sequences/s, and HBM bytes (the valid K/V cache slots + q + out) at the
    copy bandwidth."""
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm

    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    attn = fm.SwaAttention(max_batch=B, device=dev)
    inp = synth.swa_inputs(B, seed=900 + B, device=dev)
    out = torch.empty_like(inp["q"])
    ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    steps = min(args.steps, 20)

    def step():
        attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"], out=out)

    timed_loop(step, args.warmup, lambda: flush_buf.fill_(1), stream, ev)
    times = timed_loop(step, steps, lambda: flush_buf.fill_(1), stream, ev)
    if attn.poll_device_status() != 0:
        raise RuntimeError("device status error (swa)")
    ms = statistics.mean(times)
    n_valid = np.minimum(inp["pos"].cpu().numpy().astype(np.int64) + 1, fm.SWA_WINDOW)
    alg_bytes = int(n_valid.sum()) * fm.SWA_KV_HEADS * fm.SWA_HEAD_DIM * 2 * 2 + 2 * B * 32 * 128 * 2 + 32 * 4
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    return dict(workload=f"sliding-window decode attention, 32/4 heads x 128, window 513, sinks, B={B} "
                         "(length mix of the input recipe), L2 flushed before every call",
                sequences_per_s=round(B / (ms * 1e-3), 1), us_median=round(statistics.median(times) * 1e3, 2),
                roofline=dict(bound="hbm", kernel="swa::decode_kernel", achieved=round(gbs, 1), peak=peaks["hbm_gbs"],
                              unit="GB/s", frac=round(gbs / peaks["hbm_gbs"], 4), alg_bytes=alg_bytes, traffic=None),
                gpu_launches=steps)


# ----------------------------------------------------------------------------- oracle timing

def cpu_baseline_tokens(w, x, n=16, what="", eps=None):
    """The fp64 oracle (single thread) on the first n tokens of the workload's input."""
    import oracle
    from tests import parity

    x64 = oracle.bf16_to_f64(parity.to_np_bf16(x[:n]))
    if eps is not None:
        x64 = oracle.prenorm_input(x64, eps)
    experts = parity.touched_experts(w, x64, list(range(n)))
    layer = parity.oracle_layer(w, experts=experts)
    t0 = time.perf_counter()
    oracle.forward(layer, x64, nthreads=1)
    dt = time.perf_counter() - t0
    return dict(value=round(n / dt, 3), unit="tokens/s", cores=1, kind="oracle",
                sample=f"{what}: the first {n} tokens, fp64, one thread", **host_cpu())


def cpu_baseline(w, xs, budget_s=20.0, sample=(1, 2, 4, 8)):
    """The fp64 oracle (single thread) on the first tokens of the sweep, until the budget."""
    import oracle
    from tests import parity

    layer = parity.oracle_layer(w)
    n_tok = 0
    t0 = time.perf_counter()
    done = []
    for T in sample:
        x64 = oracle.bf16_to_f64(parity.to_np_bf16(xs[T]))
        oracle.forward(layer, x64, nthreads=1)
        n_tok += T
        done.append(T)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return dict(value=round(n_tok / dt, 3), unit="tokens/s", cores=1, kind="oracle",
                sample=f"decode-sweep forwards at T={done} ({n_tok} tokens), fp64, one thread", **host_cpu())


def run_reference(args, rank, world, local):
    """--impl reference: the fp64 CPU oracle as the reference arm (rank 0 only), one thread, on
    the same decode sweep as our arm (one step = the forwards at T = 1, 2, 4, 8, 16, 32, 64, 127
    tokens, x seed 1000+T)."""
    import torch

    import synth
    import oracle
    from tests import parity

    sample = SWEEP
    w = synth.flint_weights(seed=0, device="cuda" if torch.cuda.is_available() else "cpu")
    layer = parity.oracle_layer(w)
    xin = {T: oracle.bf16_to_f64(parity.to_np_bf16(synth.torch_normal_bf16((T, 2048), 1000 + T, synth.TAG_X, 1.0,
                                                                          device="cpu"))) for T in sample}

    def step():
        for T in sample:
            oracle.forward(layer, xin[T], nthreads=1)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    tok = sum(sample) * args.steps
    v = tok / dt
    return dict(metric=METRIC, value=round(v, 3), unit="tokens/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(dt / args.steps * 1e3, 3), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=sweep_config(world),
                cpu_baseline=dict(value=round(v, 3), unit="tokens/s", cores=1, kind="oracle",
                                  sample="the whole decode sweep per step (T=1..64, 127 tokens), fp64, one thread",
                                  **host_cpu()),
                e2e=dict(value=round(v, 3), unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))


def decode_phase_trace(layer, fn, flush_buf):
    """Phase stamps of the decode kernel: per slot, min / median / max over CTAs, in us from the
    earliest CTA start; five repetitions, the median of each statistic reported."""
    names = {0: "start", 1: "inputs_ready", 11: "A_first_block", 2: "A_done", 3: "barrier1", 4: "routed",
             5: "tables", 6: "C_issued", 12: "C_first_block", 7: "C_done", 8: "D_start", 13: "D_first_block",
             9: "D_done", 14: "barrier3", 10: "end"}
    layer.enable_phase_trace(True)
    reps = []
    for _ in range(5):
        flush_buf.fill_(1)
        fn()
        rows = layer.read_trace()
        t0 = min(r[0] for r in rows if r[0])
        stat = {}
        for s, nm in names.items():
            v = sorted((r[s] - t0) / 1e3 for r in rows if r[s])
            if v:
                stat[nm] = (v[0], v[len(v) // 2], v[-1])
        reps.append(stat)
    layer.enable_phase_trace(False)
    return {nm: [round(statistics.median(r[nm][i] for r in reps if nm in r), 2) for i in range(3)]
            for nm in names.values() if all(nm in r for r in reps)}


def run_profile_case(args):
    """A small, fixed case for profilers: `steps` forwards at T = --profile tokens, L2
    flushed before each, nothing else (no soak, no timing passes)."""
    import torch

    import synth
    import sparse_moe_layer_15_b300 as fm

    dev = torch.device("cuda", 0)
    T = args.profile
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    if args.workload in ("dense", "swa", "nvfp4"):
        # the dense MLP layer at T tokens, or SWA decode attention over B = T sequences
        if args.workload == "nvfp4":
            w0 = synth.flint_weights(seed=0, device=dev)
            q = synth.nvfp4_weights(w0)
            lay = fm.FlintMoE.nvfp4(w0["w_router"], q, max_tokens=T)
            x = synth.torch_normal_bf16((T, fm.HIDDEN), 1000 + T, synth.TAG_X, 1.0, device=dev)
            fn, poll = (lambda: lay.forward(x)), lay.poll_device_status
        elif args.workload == "dense":
            lay = fm.FlintDense(synth.dense_weights(seed=7, device=dev), max_tokens=T)
            x = synth.torch_normal_bf16((T, fm.HIDDEN), 600 + T, synth.TAG_X, 1.0, device=dev)
            fn, poll = (lambda: lay.forward(x)), lay.poll_device_status
        else:
            attn = fm.SwaAttention(max_batch=T, device=dev)
            inp = synth.swa_inputs(T, seed=900 + T, device=dev)
            fn = lambda: attn.decode(inp["q"], inp["k"], inp["v"], inp["sinks"], inp["pos"])  # noqa: E731
            poll = attn.poll_device_status
        for _ in range(args.warmup + args.steps):
            flush_buf.fill_(1)
            fn()
        torch.cuda.synchronize()
        rc = poll()
        trace = None
        if args.trace and args.workload == "nvfp4":
            trace = decode_phase_trace(lay, fn, flush_buf)
        print(json.dumps(dict(profile_case=T, workload=args.workload, steps=args.steps, device_status=rc,
                              trace=trace)))
        if rc != 0:
            raise SystemExit(1)
        return
    cfg = WORKLOADS.get(args.workload)  # router bias and x seed of that workload, at this T
    w = synth.flint_weights(seed=0, device=dev, bias=cfg["bias"] if cfg else None,
                            bias_seed=cfg["bias_seed"] if cfg else None)
    layer = fm.FlintMoE(w, max_tokens=T)
    x = synth.torch_normal_bf16((T, fm.HIDDEN), cfg["seed_x"] if cfg else 1000 + T, synth.TAG_X, 1.0, device=dev)
    for _ in range(args.warmup + args.steps):
        flush_buf.fill_(1)
        y = layer.forward(x)
    torch.cuda.synchronize()
    rc = layer.poll_device_status()
    trace = None
    if args.trace and T > 256:
        # wait profile of the GEMMs (gate/up: slots 0..7, down: 8..15, router: 16..23):
        # per CTA, SM kcycles spent waiting, median / max over CTAs, one repetition
        layer.enable_phase_trace(True)
        flush_buf.fill_(1)
        layer.forward(x)
        rows = layer.read_trace()
        layer.enable_phase_trace(False)
        fields = ["producer_wait_free_stage", "mma_wait_loaded_stage", "mma_wait_free_accumulator",
                  "epilogue_wait_accumulator", "epilogue_busy"]
        trace = {}
        for base, kern in ((16, "router"), (0, "gateup"), (8, "down")):
            rr = [r for r in rows if r[base + 7]]
            d = {}
            for k, nm in enumerate(fields):
                v = sorted(r[base + k] / 1e3 for r in rr)
                d[nm] = [round(v[len(v) // 2], 1), round(v[-1], 1)]
            span = sorted((r[base + 6] - r[base + 5]) / 1e3 for r in rr)
            d["cta_span_us"] = [round(span[len(span) // 2], 1), round(span[-1], 1)]
            d["tiles"] = [int(statistics.median(r[base + 7] for r in rr)), int(max(r[base + 7] for r in rr))]
            d["first_start_last_end_ns"] = [min(r[base + 5] for r in rr), max(r[base + 6] for r in rr)]
            trace[kern] = d
        # timeline (us from the router's first CTA start): each GEMM's first CTA start and last CTA end
        t0 = trace["router"]["first_start_last_end_ns"][0]
        for d in trace.values():
            a, b = d.pop("first_start_last_end_ns")
            d["span_from_router_start_us"] = [round((a - t0) / 1e3, 1), round((b - t0) / 1e3, 1)]
    elif args.trace:
        trace = decode_phase_trace(layer, lambda: layer.forward(x), flush_buf)
    layer.close()
    print(json.dumps(dict(profile_case=T, steps=args.steps, device_status=rc, y_abs_mean=float(y.float().abs().mean()),
                          trace=trace)))
    if rc != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="default workload only: skip the other four configurations")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--profile", type=int, default=0, help="profiler case: forwards at this T only")
    ap.add_argument("--trace", action="store_true",
                    help="with --profile: print the decode kernel's phase trace (T <= 256) or the grouped GEMMs' "
                         "wait profile (T > 256)")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "single", "prefill", "adversarial", "stack", "dense", "swa", "nvfp4"],
                    help="dense / swa / nvfp4: only with --profile (the default line measures them under 'extra')")
    ap.add_argument("--stack-tokens", type=int, default=256, help="stack workload: tokens per step (1..256)")
    ap.add_argument("--stack-layers", type=int, default=47,
                    help="stack workload: layers (fewer than 47 only as a small profiling case)")
    args = ap.parse_args()
    if args.profile:
        run_profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world, local)), flush=True)
        return
    out = run_ours(args, rank, world, local) if args.workload == "decode" else run_workload(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
