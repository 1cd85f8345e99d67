"""Helpers shared by the GPU parity tests (comparison only; no method arithmetic)."""
import numpy as np
import torch

import oracle as O
from mixture_experts_routing_moe_gb300 import workloads as W

DT_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
TORCH_DT = {v: k for k, v in DT_NAME.items()}


def u32(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int32).cpu().numpy().view(np.uint32)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


def storage(t: torch.Tensor):
    return W.to_storage_numpy(t)


def ulp_distance(got: torch.Tensor, ref64: np.ndarray) -> np.ndarray:
    """Distance in representable steps between a 16-bit tensor and exactly representable
    float64 reference values of the same dtype (NaN positions must be checked separately)."""
    dt = got.dtype
    ref = torch.from_numpy(np.nan_to_num(ref64, nan=0.0)).to(dt)
    g = torch.where(torch.isnan(got.cpu()), torch.zeros((), dtype=dt), got.cpu())
    a = g.view(torch.int16).to(torch.int32) & 0xFFFF
    b = ref.view(torch.int16).to(torch.int32) & 0xFFFF
    oa = torch.where(a >= 0x8000, -(a & 0x7FFF), a)
    ob = torch.where(b >= 0x8000, -(b & 0x7FFF), b)
    return (oa - ob).abs().numpy()


def check_weights(w_gpu: torch.Tensor, w_ref: np.ndarray, what=""):
    """Route weights: NaN where the oracle has NaN; else abs 1e-6 (f32) or <= 1 ulp (16-bit)."""
    g = f64(w_gpu)
    nan_ref = np.isnan(w_ref)
    assert (np.isnan(g) == nan_ref).all(), f"{what}: NaN pattern differs"
    if w_gpu.dtype == torch.float32:
        err = np.abs(g[~nan_ref] - w_ref[~nan_ref]).max(initial=0.0)
        assert err <= 1e-6, f"{what}: f32 weight abs error {err}"
    else:
        d = ulp_distance(w_gpu, w_ref)[~nan_ref]
        assert d.max(initial=0) <= 1, f"{what}: weight off by {d.max()} ulp"


def rel_max_err(got: np.ndarray, ref: np.ndarray) -> float:
    fin = np.isfinite(ref)
    assert (np.isnan(got) == np.isnan(ref)).all(), "NaN pattern differs"
    denom = np.abs(ref[fin]).max(initial=0.0)
    if denom == 0:
        return float(np.abs(got[fin]).max(initial=0.0))
    return float(np.abs(got[fin] - ref[fin]).max(initial=0.0) / denom)


def layer_tol(dtype) -> float:
    """max|gpu - oracle| / max|oracle| bound for a layer output: 1e-4 for f32, 2e-2 for 16-bit."""
    return 1e-4 if dtype == torch.float32 else 2e-2


def oracle_expert_weights(gate, up, down, dt):
    """Lazily converted float64 expert weights (one expert at a time, from device tensors)."""
    cache = {}

    def get(e):
        if e not in cache:
            cache.clear()
            cache[e] = tuple(O.to_f64(storage(w[e])[0], dt) for w in (gate, up, down))
        return cache[e]
    return get
