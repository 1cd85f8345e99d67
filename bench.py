#!/usr/bin/env python3
"""Benchmark of the local MoE forward (route -> dispatch -> SwiGLU experts -> combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one moe_forward over the workload's whole batch (all four stages), inputs resident in
HBM.  Prints ONE JSON line on rank 0.  Default workload: the many-expert skewed layer (T=16384,
H=7168, I=2048, E=256, top_k=8, bf16, Zipf(1.2) expert bias) -- the largest full-layer workload;
the route-only sweep is not a full forward.  Inputs and weights are larger than L2 (x 235 MB,
weights 22.5 GB), so no L2 flush is needed between steps.

The path shards only as independent replicas (every token is independent given replicated expert
weights), so under torchrun each rank runs its own batch: weak scaling, no collective on the data
path; the timed region is bracketed by barriers and the max over ranks is reported.

--impl reference times the fp64 CPU oracle (the only reference implementation of this method; the
pages publish no code to install) on rank 0, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_routing_moe_gb300 import workloads as W  # noqa: E402

METRIC = "MoE fwd tokens/s; grouped-GEMM TFLOP/s vs bf16 peak; route/combine GB/s vs HBM"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
def kernels_per_forward(wl) -> int:
    """route 1 + dispatch (2 for <= 4096 slots: fused index kernel + rows; else 4) + experts 2
    + combine 1."""
    return 1 + (2 if wl.T * wl.top_k <= 4096 else 4) + 2 + 1
STAGES = ["route", "dispatch", "gate_up_gemm", "down_gemm", "combine"]
# Measured DRAM traffic per launch of the forward GEMM kernels (ncu dram__bytes_read.sum +
# dram__bytes_write.sum on a small case, scaled to the full workload), recorded together with the
# hash of the kernel sources it was taken on; used only while the sources still have that hash.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="skewed", choices=sorted(W.WORKLOADS),
                    help="a full-layer workload, or route_sweep to time the route stage alone")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads measured after the headline one")
    ap.add_argument("--config-cpu-seconds", type=float, default=3.0,
                    help="target CPU time of the oracle baseline of each other workload")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward chain (combine, experts, dispatch, router) instead")
    ap.add_argument("--router", choices=["softmax", "sigmoid"], default="softmax",
                    help="sigmoid: time group-limited sigmoid routing (8 groups, top 4, top-two "
                         "group scores) alone and in the whole layer")
    return ap.parse_args()


# ------------------------------------------------------------------------------ environment
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            flat = {}

            def walk(o, pre=""):
                if isinstance(o, dict):
                    for k, v in o.items():
                        walk(v, f"{pre}{k}.")
                elif isinstance(o, (int, float)):
                    flat[pre[:-1]] = float(o)
            walk(d)

            def pick(*names):
                for n in names:
                    for k, v in flat.items():
                        if k.split(".")[-1] == n:
                            return v
                return None
            p = {"hbm_gbs": pick("hbm_gbs", "hbm_GBs", "copy_gbs"),
                 "bf16_tflops": pick("bf16_tflops", "bf16_tflops_burst"),
                 "bf16_tflops_sustained": pick("bf16_tflops_sustained")}
            if p["hbm_gbs"] and p["bf16_tflops"]:
                if not p["bf16_tflops_sustained"]:
                    p["bf16_tflops_sustained"] = p["bf16_tflops"]
                return p, "measured"
        except Exception as e:  # malformed file: fall back, say so
            log(f"MEASURED_PEAKS.json unreadable ({e}); using fallback peaks")
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device):
        self.proc = None
        self.path = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}",
               "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            u = self.uuid if self.uuid.startswith("GPU-") else f"GPU-{self.uuid}"
            cmd += ["-i", u]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def replica_throughput(tokens_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s of `world` independent replicas: every rank processes its own batch of
    `tokens_per_step` tokens per step; the job takes the slowest rank's time."""
    return tokens_per_step * steps * world / (max_ms / 1e3)


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ work accounting
def stage_work(wl: W.Workload, n_active: int):
    """Algorithmic bytes / flops of one forward, per stage (the roofline numerators)."""
    es = 2 if wl.dtype != "f32" else 4
    T, E, H, I, k = wl.T, wl.E, wl.H, wl.I, wl.top_k
    R = T * k
    return {
        "route": {"bytes": T * E * es + R * (4 + es)},
        "dispatch": {"bytes": T * H * es + R * H * es + 3 * R * 4},
        "gate_up_gemm": {"flops": 4 * R * H * I,
                         "bytes": R * H * es + 2 * n_active * I * H * es + R * I * es},
        "down_gemm": {"flops": 2 * R * I * H,
                      "bytes": R * I * es + n_active * H * I * es + R * H * es},
        "combine": {"bytes": R * H * es + R * (4 + es) + T * H * es},
    }


def kernel_source_sha256():
    """SHA-256 over the sources the forward GEMM kernels compile from (kernels, tile raster,
    PTX wrappers, helpers)."""
    h = hashlib.sha256()
    for f in ("experts_tc.cu", "gemm_cta.cuh", "tcgen05.cuh", "tiles.cuh", "common.cuh"):
        h.update(open(os.path.join(ROOT, "mixture_experts_routing_moe_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def recorded_traffic(kernel: str, workload: str):
    """Bytes per launch of `kernel` on `workload` from the committed traffic record, or None when
    there is none or the kernel sources have changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_source_sha256():
        return None
    e = rec.get("launches", {}).get(kernel, {}).get(workload)
    return None if e is None else float(e["bytes_per_launch"])


def tensor_peak(pk, clocks, region_s: float):
    """The bf16 tensor peak a GEMM timed in `region_s` seconds is measured against: the burst
    figure when the region is shorter than a second and the sampled SM clock stayed at its
    maximum (the condition the burst GEMM was measured in), else the sustained figure (a
    seconds-long loop under the power cap)."""
    at_max = bool(clocks) and clocks["sm_mhz"] >= 0.97 * clocks["sm_max_mhz"]
    if region_s < 1.0 and at_max:
        return pk["bf16_tflops"], "burst"
    return pk["bf16_tflops_sustained"], "sustained"


# ------------------------------------------------------------------------------ oracle timing
def oracle_sample(wl, host, tokens):
    """Run the fp64 oracle end to end (route + dispatch + experts + combine) on `tokens`."""
    import oracle as O
    name = wl.dtype
    l64 = O.to_f64(host["logits"][tokens], name)
    idx, w = O.route(l64, wl.top_k, wl.renormalize, name)
    x64 = O.to_f64(host["x"][tokens], name)

    def weights(e):
        return tuple(O.to_f64(host[m][e], name) for m in ("gate", "up", "down"))
    return O.forward_rows(x64, idx, w, weights)


def host_storage(inp):
    return {k: W.to_storage_numpy(v)[0] for k, v in inp.items()}


def time_oracle(wl, host, seconds: float, first_token: int = 0):
    """Oracle throughput on a bounded sample: grow the token sample until ~`seconds` of CPU work."""
    n, done, elapsed = 1, 0, 0.0
    t_first = first_token
    while elapsed < seconds and done < wl.T:
        n = min(n, wl.T - done)
        toks = (np.arange(n) + t_first) % wl.T
        t0 = time.perf_counter()
        oracle_sample(wl, host, toks)
        dt = time.perf_counter() - t0
        elapsed += dt
        done += n
        t_first += n
        if dt < seconds / 8:
            n *= 2
    return done, elapsed


# ------------------------------------------------------------------------------ arms
def run_reference(args):
    rank, world, local = dist_setup()
    if rank != 0:
        return
    wl = W.WORKLOADS[args.workload]
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    inp = W.make_layer_inputs(wl, dev)
    host = host_storage(inp)
    del inp
    # per-step sample sized so the whole --warmup + --steps run stays near 90 s of CPU time
    t0 = time.perf_counter()
    oracle_sample(wl, host, np.array([0]))
    per_token = max(time.perf_counter() - t0, 1e-4)
    budget = 90.0 / max(1, args.steps + args.warmup)
    S = int(max(1, min(wl.T, budget // per_token)))
    tok = 0
    for _ in range(args.warmup):
        oracle_sample(wl, host, (np.arange(S) + tok) % wl.T)
        tok += S
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample(wl, host, (np.arange(S) + tok) % wl.T)
        tok += S
    el = time.perf_counter() - t0
    value = S * args.steps / el
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                       "top_k": wl.top_k, "renormalize": wl.renormalize, "storage_dtype": wl.dtype,
                       "sample_tokens_per_step": S, "parallelism": "rank 0 only"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{S} token(s) per step of the {wl.name} workload, fp64 "
                                       f"numpy oracle end to end, BLAS on all {cores} host cores"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class L2Flush:
    """Empties L2 before a timed launch: writes a buffer larger than L2, then reads another one.
    A write alone leaves about an L2's worth of dirty lines, whose write-back to HBM would land
    inside the next (timed) kernel; the read moves that write-back before the timed region."""

    def __init__(self, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum(dtype=torch.int64)
        # keep the GPU busy (about 100 us) while the host enqueues the start event and the timed
        # launch: otherwise the GPU idles on the host's launch overhead and the events time it
        torch.cuda._sleep(200_000)


def run_route_only(args):
    """The route-only workload: moe_route alone, renormalise on and off, against HBM."""
    import mixture_experts_routing_moe_gb300 as moe
    from mixture_experts_routing_moe_gb300 import build as build_mod
    build_mod.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    res, roof, clocks = route_entry(moe, wl, dev, args.steps, args.warmup, L2Flush(dev))
    best = min(res.values(), key=lambda d: d["ms"])
    roof = {**roof, "achieved": best["gbs"], "frac": best["frac"]}
    line = {"metric": "route GB/s vs HBM (route-only workload)", "value": wl.T / (best["ms"] / 1e3),
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": best["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": f"{wl.name}: logits [{wl.T}, {wl.E}] {wl.dtype}, top_k={wl.top_k}",
                       "l2": "L2 emptied before every launch (256 MB written, then 256 MB read)"},
            "roofline": roof, "variants": res, "gpu_launches": 2 * args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def run_backward(args):
    """The backward chain on a layer workload: combine_backward -> experts backward ->
    dispatch_backward -> router backward, inputs from one forward, resident in HBM."""
    import mixture_experts_routing_moe_gb300 as moe
    from mixture_experts_routing_moe_gb300 import build as build_mod
    build_mod.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    inp = W.make_layer_inputs(wl, dev)
    x, logits, gate, up, down = (inp[k] for k in ("x", "logits", "gate", "up", "down"))
    idx, _ = moe.moe_route(logits, wl.top_k, wl.renormalize)
    d = moe.moe_dispatch(x, idx, wl.E)
    y = moe.moe_experts_forward_dispatched(d["x_d"], d["offsets"], gate, up, down)
    wts = moe.moe_selected_router_weights(logits, idx, "softmax", wl.renormalize, 1.0).to(x.dtype)
    dout = torch.randn(wl.T, wl.H, device=dev, generator=torch.Generator(device=dev).manual_seed(1)).to(x.dtype)
    R = wl.T * wl.top_k
    ws = torch.empty(moe.binding.lib().moe_experts_backward_workspace_bytes(R, wl.I),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev: ev[0].record(stream)
        de, dw = moe.moe_combine_backward(y, d["row_of_slot"], wts, dout)
        if ev: ev[1].record(stream)
        dxd, dg, du, dd = moe.moe_experts_backward(d["x_d"], d["offsets"], gate, up, down, de, ws=ws)
        if ev: ev[2].record(stream)
        moe.moe_dispatch_backward(dxd, d["row_of_slot"], wl.T, wl.top_k)
        moe.moe_selected_router_backward(logits, idx, dw, "softmax", wl.renormalize, 1.0)
        if ev: ev[3].record(stream)
    for _ in range(max(3, args.warmup)):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(dev)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)   # let the sampler take its first reading
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st = moe.moe_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    tot = float(np.mean([e[0].elapsed_time(e[3]) for e in evs]))
    exp_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    flops = 16 * R * wl.H * wl.I          # recompute g, u (4) + da (2) + dinput (4) + weight grads (6)
    tensor = x.dtype != torch.float32 and wl.I % 64 == 0   # the library's tensor-core condition
    achieved = flops / (exp_ms / 1e3) / 1e12
    if tensor:
        pk, pk_src = peaks()
        peak, kind = tensor_peak(pk, clocks, tot * args.steps / 1e3)
        roof = {"kernel": "experts backward (tcgen05 GEMMs: dA, gate/up + SwiGLU grad, dinput, "
                          "weight grads)", "bound": "tensor",
                "peak_source": f"{pk_src} bf16 {kind} (dense, cuBLAS; chosen from the timed "
                               f"region's length and sampled clocks); f16 runs at the bf16 rate"}
        launches = 9
    else:
        # FP32 CUDA-core peak from unit counts and clock: SMs x 128 FMA/clk x 2 x max SM clock
        props = torch.cuda.get_device_properties(dev)
        peak = props.multi_processor_count * 128 * 2 * 2.07e9 / 1e12
        roof = {"kernel": "experts backward (FP32 CUDA-core ragged GEMMs)", "bound": "alu",
                "peak_source": "derived: SMs x 128 FP32 FMA/clk x 2 x 2.07 GHz"}
        launches = 10
    line = {"metric": "MoE backward tokens/s (combine, experts, dispatch, router backward)",
            "value": wl.T / (tot / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                       "top_k": wl.top_k},
            "roofline": {**roof, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "algorithmic_flops_per_launch": flops},
            "stages_ms": {"combine_backward": float(np.mean([e[0].elapsed_time(e[1]) for e in evs])),
                          "experts_backward": exp_ms,
                          "dispatch_and_router_backward": float(np.mean([e[2].elapsed_time(e[3]) for e in evs])),
                          "total": tot},
            "gpu_launches": launches * args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def run_sigmoid(args):
    """Group-limited sigmoid routing (8 groups, best 4 by the sum of their two largest corrected
    scores, top_k of the workload, a per-expert FP32 correction bias): the router alone against
    HBM, and the whole layer (moe_forward_sigmoid_grouped) in tokens/s."""
    import mixture_experts_routing_moe_gb300 as moe
    from mixture_experts_routing_moe_gb300 import build as build_mod
    build_mod.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    G, SG = 8, 4
    inp = W.make_layer_inputs(wl, dev)
    x, logits, gate, up, down = (inp[k] for k in ("x", "logits", "gate", "up", "down"))
    bias = (0.01 * torch.randn(wl.E, generator=torch.Generator(device=dev).manual_seed(9),
                               device=dev)).float()
    out = torch.empty_like(x)
    ws = torch.empty(moe.forward_workspace_bytes(wl.T, wl.E, wl.H, wl.I, wl.top_k, logits.dtype,
                                                 x.dtype), dtype=torch.uint8, device=dev)
    idx = torch.empty(wl.T, wl.top_k, dtype=torch.uint32, device=dev)
    w = torch.empty(wl.T, wl.top_k, dtype=logits.dtype, device=dev)
    flush = L2Flush(dev)

    def route():
        moe.moe_route_sigmoid_grouped(logits, wl.top_k, G, SG, True, wl.renormalize, 1.0, bias,
                                      idx=idx, w=w)

    def layer():
        moe.moe_forward_sigmoid_grouped(x, logits, gate, up, down, wl.top_k, G, SG, True,
                                        wl.renormalize, 1.0, bias, out=out, ws=ws)

    def timed(fn, n, flush_l2):
        for _ in range(max(3, args.warmup)):
            fn()
        ms = []
        for _ in range(n):
            if flush_l2:
                flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return float(np.median(ms))
    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.3)
    route_ms = timed(route, args.steps, True)
    layer_ms = timed(layer, args.steps, False)
    clocks = sampler.stop()
    st = moe.moe_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st}")
    es = logits.element_size()
    nbytes = wl.T * wl.E * es + wl.E * 4 + wl.T * wl.top_k * (4 + es)
    pk, pk_src = peaks()
    gbs = nbytes / (route_ms / 1e3) / 1e9
    line = {"metric": "MoE fwd tokens/s with group-limited sigmoid routing; router GB/s vs HBM",
            "value": wl.T / (layer_ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": layer_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                       "top_k": wl.top_k, "groups": G, "selected_groups": SG,
                       "group_top_two": True, "l2": "emptied before each router launch (256 MB written, then 256 MB read)"},
            "roofline": {"kernel": "moe_route_sigmoid_sub (sub-warp rows; FP32 decision, float64 only where a margin fails)",
                         "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "peak_source": f"{pk_src} HBM copy",
                         "traffic": None, "algorithmic_bytes_per_launch": nbytes},
            "stages_ms": {"route_sigmoid": route_ms, "layer": layer_ms},
            "gpu_launches": args.steps * (1 + (1 if moe.moe_forward_fused(
                wl.T, wl.E, wl.H, wl.I, wl.top_k, logits.dtype, x.dtype) else kernels_per_forward(wl))),
            "clocks": clocks}
    print(json.dumps(line), flush=True)


def measure_layer(moe, wl, dev, steps, warmup, world=1, flush=None):
    """Times `steps` moe_forward calls over one batch of `wl`, inputs resident in HBM.

    Stage times come from CUDA events on the launching stream inside the timed region (the
    staged path), or from events around the single launch (the fused short-batch path, whose
    stage kernels are then timed separately for comparison).  With `flush`, L2 is emptied before
    every step and only the forward itself is inside the events.  Returns the measurements and
    the resident tensors (for the end-to-end leg and the CPU baseline)."""
    stream = torch.cuda.current_stream()
    inp = W.make_layer_inputs(wl, dev)
    x, logits, gate, up, down = (inp[k] for k in ("x", "logits", "gate", "up", "down"))
    out = torch.empty_like(x)
    wsb = moe.forward_workspace_bytes(wl.T, wl.E, wl.H, wl.I, wl.top_k, logits.dtype, x.dtype)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    idx, _ = moe.moe_route(logits, wl.top_k, wl.renormalize)
    counts = torch.bincount(idx.view(torch.int32).flatten().long(), minlength=wl.E)
    n_active = int((counts > 0).sum())
    max_load = int(counts.max())
    del idx
    # short batches run as one fused launch; the staged path is then timed only for comparison
    fused = moe.moe_forward_fused(wl.T, wl.E, wl.H, wl.I, wl.top_k, logits.dtype, x.dtype)

    def staged_step(evs=None):
        moe.moe_forward_with_events(x, logits, gate, up, down, wl.top_k, wl.renormalize, out, ws,
                                    evs)

    def step(evs=None):
        if not fused:
            staged_step(evs)
            return
        if evs:
            evs[0].record(stream)
        moe.moe_forward(x, logits, gate, up, down, wl.top_k, wl.renormalize, out=out, ws=ws)
        if evs:
            evs[1].record(stream)

    for _ in range(max(3, warmup)):
        step()
    st = moe.moe_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    n_ev = 2 if fused else 6
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(dev)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)   # let the sampler take its first reading
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            flush()
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    if flush is None:
        el_ms = t_start.elapsed_time(t_end)
    else:   # the forwards alone, without the flushes between them
        el_ms = float(sum(e[0].elapsed_time(e[-1]) for e in evs))
    el_ms = max_over_ranks(el_ms, world, dev)
    st = moe.moe_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")
    fused_ms = None
    if fused:
        fused_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
        # the staged launches on the same inputs, for comparison only (not the timed steps)
        sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(10)]
        for e in sevs:
            if flush is not None:
                flush()
            staged_step(e)
        torch.cuda.synchronize()
        stage_ms = {s: float(np.mean([e[j].elapsed_time(e[j + 1]) for e in sevs]))
                    for j, s in enumerate(STAGES)}
    else:
        stage_ms = {s: float(np.mean([e[j].elapsed_time(e[j + 1]) for e in evs]))
                    for j, s in enumerate(STAGES)}
    return {"el_ms": el_ms, "stage_ms": stage_ms, "fused": fused, "fused_ms": fused_ms,
            "n_active": n_active, "max_load": max_load, "clocks": clocks,
            "tensors": {"x": x, "logits": logits, "gate": gate, "up": up, "down": down,
                        "out": out, "ws": ws}, "inputs": inp}


def layer_roofline(wl, m, pk, pk_src):
    """Per-stage figures and the roofline entry of the dominant kernel of one measured layer."""
    work = stage_work(wl, m["n_active"])
    stage_ms = m["stage_ms"]
    region_s = m["el_ms"] / 1e3
    tpeak, tkind = tensor_peak(pk, m["clocks"], region_s)
    stages = {}
    for s in STAGES:
        d = {"ms": stage_ms[s], "gbs": work[s]["bytes"] / (stage_ms[s] / 1e3) / 1e9}
        if "flops" in work[s]:
            d["tflops"] = work[s]["flops"] / (stage_ms[s] / 1e3) / 1e12
            d["frac"] = d["tflops"] / tpeak
        else:
            d["frac"] = d["gbs"] / pk["hbm_gbs"]
        stages[s] = d
    if m["fused"]:
        x, logits = m["tensors"]["x"], m["tensors"]["logits"]
        es = x.element_size()
        # the layer's own bytes: logits, x, the touched experts' weights, out (x_d, a and y
        # stay in L2 between the phases of the fused launch)
        fbytes = (logits.numel() * logits.element_size() + 2 * wl.T * wl.H * es
                  + 3 * m["n_active"] * wl.H * wl.I * es)
        fms = m["fused_ms"]
        achieved = fbytes / (fms / 1e3) / 1e9
        stages = {"fused_forward": {"ms": fms, "gbs": achieved, "frac": achieved / pk["hbm_gbs"]},
                  "staged_path_for_comparison": stages}
        roof = {"kernel": "moe_decode_fused (route, dispatch, gate/up, down, combine in one "
                          "cooperative launch)",
                "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": f"{pk_src} HBM copy",
                "traffic": None, "algorithmic_bytes_per_launch": fbytes}
        return stages, roof
    dom = "gate_up_gemm"
    pair = wl.rows >= 128 * wl.E
    kname = "moe_experts_tc2<gate/up>" if pair else "moe_experts_tc<gate/up>"
    achieved = stages[dom]["tflops"]
    traffic = recorded_traffic(kname, wl.name)
    roof = {"kernel": kname + (" (CTA-pair tcgen05 grouped GEMM + SwiGLU)" if pair
                               else " (tcgen05 grouped GEMM + SwiGLU)"),
            "bound": "tensor", "achieved": achieved, "peak": tpeak, "unit": "TFLOP/s",
            "frac": achieved / tpeak,
            "peak_source": f"{pk_src} bf16 {tkind} (cuBLAS; {tkind} chosen from a "
                           f"{region_s:.2f} s timed region at a median "
                           f"{(m['clocks'] or {}).get('sm_mhz', 'unknown')} MHz)",
            "traffic": traffic,
            "traffic_over_algorithmic": (traffic / work[dom]["bytes"]) if traffic else None,
            "algorithmic_flops_per_launch": work[dom]["flops"],
            "algorithmic_bytes_per_launch": work[dom]["bytes"]}
    return stages, roof


def route_entry(moe, wl, dev, steps, warmup, flush):
    """moe_route alone on a route-only workload, renormalise on and off, L2 emptied before
    every launch; GB/s of the algorithmic bytes against the HBM peak."""
    logits = W.make_logits(wl, dev)
    idx = torch.empty(wl.T, wl.top_k, dtype=torch.uint32, device=dev)
    w = torch.empty(wl.T, wl.top_k, dtype=logits.dtype, device=dev)
    es = logits.element_size()
    nbytes = wl.T * wl.E * es + wl.T * wl.top_k * (4 + es)
    pk, pk_src = peaks()
    res = {}
    sampler = ClockSampler(dev)
    sampler.start()
    time.sleep(0.3)
    for renorm in (True, False):
        for _ in range(max(3, warmup)):
            moe.moe_route(logits, wl.top_k, renorm, idx=idx, w=w)
        times = []
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            moe.moe_route(logits, wl.top_k, renorm, idx=idx, w=w)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        ms = float(np.mean(times))
        gbs = nbytes / (ms / 1e3) / 1e9
        res["renormalize" if renorm else "plain"] = {"ms": ms, "gbs": gbs,
                                                     "frac": gbs / pk["hbm_gbs"]}
    clocks = sampler.stop()
    kern = ("moe_route16_small" if es == 2 and wl.E <= 64 and wl.E % 8 == 0 and wl.top_k <= 8
            else "moe_route_kernel")
    return res, {"kernel": kern, "bound": "hbm", "peak": pk["hbm_gbs"], "unit": "GB/s",
                 "peak_source": f"{pk_src} HBM copy", "algorithmic_bytes_per_launch": nbytes,
                 "traffic": None}, clocks


def cpu_leg(wl, inputs, seconds):
    """The oracle, as it stands, on the first tokens of a workload for about `seconds` of CPU time
    (the same CPU baseline as the headline's, on a smaller sample)."""
    import oracle as O
    cores = os.cpu_count()
    if wl.H == 0:  # route only: grow the row sample
        arr, name = W.to_storage_numpy(inputs["logits"])
        n, done, elapsed = 1024, 0, 0.0
        while elapsed < seconds and done < wl.T:
            n = min(n, wl.T - done)
            t0 = time.perf_counter()
            O.route(O.to_f64(arr[done:done + n], name), wl.top_k, True, name)
            elapsed += time.perf_counter() - t0
            done += n
            n *= 2
        what = f"route of the first {done} rows"
    else:
        host = host_storage(inputs)
        done, elapsed = time_oracle(wl, host, seconds)
        what = f"the first {done} tokens end to end"
    return {"value": done / elapsed, "unit": "tokens/s" if wl.H else "rows/s", "cores": cores,
            "kind": "oracle", "sample": f"{what} of the {wl.name} workload through the fp64 numpy "
                                        f"oracle ({elapsed:.1f} s; BLAS threads = all {cores} host cores)"}


def other_configs(moe, dev, args):
    """The other workloads, measured in the same process after the headline one: the route-only
    sweep, the decode layer (the fused launch, L2 emptied between steps), the prefill layer
    (staged) and the tiny f32 layer (a correctness workload; its time is reported, its roofline
    is not meaningful)."""
    pk, pk_src = peaks()
    flush = L2Flush(dev)
    out = {}
    wl = W.WORKLOADS["route_sweep"]
    res, roof, clocks = route_entry(moe, wl, dev, max(20, args.steps), args.warmup, flush)
    out["route_sweep"] = {"workload": f"logits [{wl.T}, {wl.E}] {wl.dtype} N(0, 2^2), "
                                      f"top_k={wl.top_k}", "variants": res, "roofline": roof,
                          "l2": "emptied before every launch", "clocks": clocks}
    if not args.no_cpu_baseline:
        out["route_sweep"]["cpu_baseline"] = cpu_leg(wl, {"logits": W.make_logits(wl, dev)},
                                                     args.config_cpu_seconds)
    torch.cuda.empty_cache()
    for name, steps, fl in (("decode", max(50, args.steps), flush), ("prefill", args.steps, None),
                            ("tiny_f32", max(20, args.steps), None)):
        wl = W.WORKLOADS[name]
        m = measure_layer(moe, wl, dev, steps, args.warmup, flush=fl)
        stages, roof = layer_roofline(wl, m, pk, pk_src)
        ms = m["el_ms"] / steps
        e = {"workload": f"T={wl.T} H={wl.H} I={wl.I} E={wl.E} top_k={wl.top_k} {wl.dtype}"
                         + (f" Zipf({wl.zipf_s}) expert bias" if wl.zipf_s else ""),
             "ms": ms, "tokens_per_s": wl.T / (ms / 1e3), "steps": steps,
             "path": "fused single launch" if m["fused"] else "staged launches",
             "active_experts": m["n_active"], "max_rows_per_expert": m["max_load"],
             "l2": "emptied before every step" if fl is not None else
                   "inputs larger than L2; no flush",
             "stages": stages, "roofline": roof, "clocks": m["clocks"]}
        if name == "tiny_f32":
            e["roofline"] = None
            e["note"] = "correctness workload (parity in tests/test_gpu_parity.py::test_layer_tiny_f32)"
        if not args.no_cpu_baseline:
            e["cpu_baseline"] = cpu_leg(wl, m["inputs"], args.config_cpu_seconds)
        out[name] = e
        del m
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import mixture_experts_routing_moe_gb300 as moe
    from mixture_experts_routing_moe_gb300 import build as build_mod
    build_mod.build()
    rank, world, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = W.WORKLOADS[args.workload]
    stream = torch.cuda.current_stream()
    m = measure_layer(moe, wl, dev, args.steps, args.warmup, world=world)
    t = m["tensors"]
    x, logits, gate, up, down, out, ws = (t[k] for k in ("x", "logits", "gate", "up", "down",
                                                         "out", "ws"))
    el_ms = m["el_ms"]
    value = replica_throughput(wl.T, args.steps, world, el_ms)
    pk, pk_src = peaks()
    stages, roof = layer_roofline(wl, m, pk, pk_src)

    # End to end through the public API, as a serving loop runs it: every step copies its own
    # inputs in from pinned host memory and its output back to pinned host memory.  Steps are
    # pipelined over three streams with two device buffer sets: the inputs of step i+1 are copied
    # in and the output of step i-1 copied out while moe_forward runs step i.
    x_h = x.cpu().pin_memory()
    l_h = logits.cpu().pin_memory()
    o_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    xs = [torch.empty_like(x) for _ in range(2)]
    ls = [torch.empty_like(logits) for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(comp_done[b])     # the compute that read this buffer set is done
            xs[b].copy_(x_h, non_blocking=True)
            ls[b].copy_(l_h, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        if started[b]:
            stream.wait_event(out_done[b])        # its previous output has been copied out
        moe.moe_forward(xs[b], ls[b], gate, up, down, wl.top_k, wl.renormalize, out=outs[b],
                        ws=ws)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            o_h[b].copy_(outs[b], non_blocking=True)
            out_done[b].record(s_out)
        started[b] = True
    for i in range(2):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(args.e2e_steps):
        e2e_step(i)
    s_out.wait_stream(stream)
    s_out.wait_stream(s_in)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e = {"value": replica_throughput(wl.T, args.e2e_steps, world, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": x.numel() * x.element_size() + logits.numel() * logits.element_size(),
           "d2h_bytes_per_step": out.numel() * out.element_size(),
           "pipelining": "h2d of step i+1 and d2h of step i-1 overlap moe_forward of step i "
                         "(three streams, two device buffer sets)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = host_storage(m["inputs"])
        done, secs = time_oracle(wl, host, args.cpu_seconds)
        cores = os.cpu_count()
        cpu = {"value": done / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {done} tokens of the {wl.name} workload through the fp64 numpy "
                         f"oracle end to end ({secs:.1f} s; BLAS threads = all {cores} host cores)"}
        del host
    n_active, max_load, clocks, fused = m["n_active"], m["max_load"], m["clocks"], m["fused"]
    x_mb, w_gb = x.numel() * 2 / 1e6, 3 * gate.numel() * 2 / 1e9
    del m, t, x, logits, gate, up, down, out, ws, xs, ls, outs, x_h, l_h, o_h
    torch.cuda.empty_cache()

    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = other_configs(moe, dev, args)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": f"{wl.name}: T={wl.T} H={wl.H} I={wl.I} E={wl.E} "
                                   f"top_k={wl.top_k} renormalize={wl.renormalize} {wl.dtype}"
                                   + (f" Zipf({wl.zipf_s}) expert bias" if wl.zipf_s else ""),
                       "tokens_per_step_per_gpu": wl.T, "active_experts": n_active,
                       "max_rows_per_expert": max_load,
                       "l2": "inputs larger than L2 (x %.0f MB, weights %.1f GB); no flush" % (
                           x_mb, w_gb),
                       "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "stages": stages,
            "hbm_peak_gbs": pk["hbm_gbs"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (1 if fused else kernels_per_forward(wl)) * args.steps,
            "clocks": clocks,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif W.WORKLOADS[args.workload].H == 0:
        run_route_only(args)
    elif args.backward:
        run_backward(args)
    elif args.router == "sigmoid":
        run_sigmoid(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
