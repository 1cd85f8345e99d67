"""Seeded synthetic inputs for the local MoE forward.

This module only draws random numbers and lays them out in the storage dtype; it holds none of
the method's arithmetic (no softmax, no selection, no grouping, no expert maths).  Both the CUDA
path and the fp64 oracle are fed from the same tensors it returns, so the two sides see the same
bytes.

The five workloads mirror the shapes the ruDNN user guide uses for its MoE contract (§4
"Routing-Vertrag": logits [T, E] in F32/F16/BF16; §5 "Expertengewichte und Verteilung":
x [T, H], gate/up [E, I, H], down [E, H, I]):

  tiny_f32     T=64     H=128  I=256   E=8   k=2  f32   N(0,1) logits with tie / NaN / +inf / -inf rows
  route_sweep  T=2^20   E=64                 k=8  bf16  N(0, 2^2) logits, route only
  decode       T=256    H=2048 I=768   E=128 k=8  bf16  N(0,1) + log Zipf(1.1) expert bias
  prefill      T=8192   H=4096 I=14336 E=8   k=2  bf16  i.i.d.
  skewed       T=16384  H=7168 I=2048  E=256 k=8  bf16  N(0,1) + log Zipf(1.2) expert bias

Weights are N(0, 1/fan_in) with fan_in = H for gate/up and I for down; tokens are N(0, 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    E: int
    top_k: int
    renormalize: bool
    dtype: str            # storage dtype of logits, tokens and expert weights
    seed: int
    H: int = 0            # 0 for route-only workloads
    I: int = 0
    logit_std: float = 1.0
    zipf_s: float = 0.0   # 0: no expert bias
    special_rows: bool = False

    @property
    def rows(self) -> int:
        return self.T * self.top_k

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", T=64, H=128, I=256, E=8, top_k=2, renormalize=True,
                         dtype="f32", seed=0, special_rows=True),
    "route_sweep": Workload("route_sweep", T=1 << 20, E=64, top_k=8, renormalize=True,
                            dtype="bf16", seed=2, logit_std=2.0),
    "decode": Workload("decode", T=256, H=2048, I=768, E=128, top_k=8, renormalize=True,
                       dtype="bf16", seed=3, zipf_s=1.1),
    "prefill": Workload("prefill", T=8192, H=4096, I=14336, E=8, top_k=2, renormalize=True,
                        dtype="bf16", seed=4),
    "skewed": Workload("skewed", T=16384, H=7168, I=2048, E=256, top_k=8, renormalize=True,
                       dtype="bf16", seed=5, zipf_s=1.2),
    # profiling case: the skewed layer's expert shape with 32 experts and 2048 tokens, small
    # enough (2.8 GB of weights) for multi-pass counter captures
    "skewed_e32": Workload("skewed_e32", T=2048, H=7168, I=2048, E=32, top_k=8,
                           renormalize=True, dtype="bf16", seed=6, zipf_s=1.2),
    # profiling cases of the expert backward (about 1.3 GB on the device): every expert with
    # exactly 512 rows (top_k = E), and 16 experts under a steep Zipf bias
    "wgrad_uniform": Workload("wgrad_uniform", T=512, H=4096, I=2048, E=8, top_k=8,
                              renormalize=True, dtype="bf16", seed=7),
    "wgrad_skewed": Workload("wgrad_skewed", T=1024, H=4096, I=2048, E=16, top_k=4,
                             renormalize=True, dtype="bf16", seed=8, zipf_s=1.5),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_log_bias(E: int, s: float, seed: int) -> torch.Tensor:
    """log of a Zipf(s) pmf over ranks 1..E, assigned to experts through a seeded permutation.

    bias[perm[r-1]] = log(r^-s / sum_q q^-s).  float64, CPU.
    """
    g = _gen(seed + 7919, "cpu")
    perm = torch.randperm(E, generator=g)
    r = torch.arange(1, E + 1, dtype=torch.float64)
    pmf = r.pow(-s)
    pmf = pmf / pmf.sum()
    bias = torch.empty(E, dtype=torch.float64)
    bias[perm] = pmf.log()
    return bias


def make_logits(w: Workload, device="cpu") -> torch.Tensor:
    """Router logits [T, E] in the workload's dtype."""
    g = _gen(w.seed, device)
    l = torch.randn(w.T, w.E, generator=g, device=device, dtype=torch.float32) * w.logit_std
    if w.zipf_s > 0:
        l += zipf_log_bias(w.E, w.zipf_s, w.seed).to(device=device, dtype=torch.float32)
    if w.special_rows:
        l = _plant_special_rows(l)
    return l.to(TORCH_DTYPE[w.dtype])


def _plant_special_rows(l: torch.Tensor) -> torch.Tensor:
    """Rows 0-3: exact ties across experts {1,5} and {0,7}; row 4 holds a NaN, row 5 a +inf,
    row 6 is all -inf.  Needs T >= 7 and E >= 8."""
    assert l.shape[0] >= 7 and l.shape[1] >= 8
    l = l.clone()
    # row 0: {1,5} tie at the top;  row 1: {0,7} tie at the top
    l[0, 1] = l[0, 5] = 4.0
    l[1, 0] = l[1, 7] = 4.0
    # row 2: expert 3 on top, {1,5} tie for second place; row 3: {0,7} on top, {1,5} next
    l[2, 3] = 5.0
    l[2, 1] = l[2, 5] = 4.0
    l[3, 0] = l[3, 7] = 5.0
    l[3, 1] = l[3, 5] = 4.0
    l[4, 2] = float("nan")
    l[5, 6] = float("inf")
    l[6, :] = float("-inf")
    return l


def make_layer_inputs(w: Workload, device="cpu") -> dict:
    """x [T,H], logits [T,E], gate/up [E,I,H], down [E,H,I], all in the workload's dtype.

    Large expert tensors are drawn one expert at a time so the float32 temporaries stay small.
    """
    assert w.H > 0 and w.I > 0
    dt = TORCH_DTYPE[w.dtype]
    logits = make_logits(w, device)
    g = _gen(w.seed + 1, device)
    x = torch.randn(w.T, w.H, generator=g, device=device, dtype=torch.float32).to(dt)
    gate = torch.empty(w.E, w.I, w.H, device=device, dtype=dt)
    up = torch.empty(w.E, w.I, w.H, device=device, dtype=dt)
    down = torch.empty(w.E, w.H, w.I, device=device, dtype=dt)
    sh, si = 1.0 / math.sqrt(w.H), 1.0 / math.sqrt(w.I)
    for e in range(w.E):
        gate[e] = (torch.randn(w.I, w.H, generator=g, device=device) * sh).to(dt)
        up[e] = (torch.randn(w.I, w.H, generator=g, device=device) * sh).to(dt)
        down[e] = (torch.randn(w.H, w.I, generator=g, device=device) * si).to(dt)
    return {"x": x, "logits": logits, "gate": gate, "up": up, "down": down}


def to_storage_numpy(t: torch.Tensor):
    """(numpy array, dtype name) holding the exact stored bits: bf16 as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16"), "bf16"
    if t.dtype == torch.float16:
        return t.numpy(), "f16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    raise TypeError(f"unsupported dtype {t.dtype}")
