"""GPU parity of group-limited sigmoid routing (ruDNN user guide §10) against the fp64 oracle:
indices bit-exact, weights within abs 1e-6 (f32) or 1 ulp (f16 / bf16), NaN rows NaN; the
sigmoid-routed forward within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle as O
import mixture_experts_routing_moe_gb300 as moe
from mixture_experts_routing_moe_gb300 import workloads as W
from gpu_helpers import DT_NAME, check_weights, f64, layer_tol, rel_max_err, storage, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [  # E, groups, selected, top_k, top_two
    (256, 8, 4, 8, True), (64, 8, 3, 6, True), (32, 4, 1, 8, False), (48, 1, 1, 5, False),
    (128, 16, 16, 16, True), (8, 4, 2, 3, False), (1024, 128, 8, 64, True), (96, 3, 2, 40, False),
    # sub-warp rows (L lanes x EPL experts): L = 32 with 8 and 16 experts a lane, L = 1, 2, 4,
    # and top_k equal to the candidates of the chosen groups (no (k+1)-th round)
    (256, 32, 8, 8, True), (512, 8, 2, 8, True), (16, 1, 1, 1, False), (32, 2, 1, 2, True),
    (64, 4, 2, 4, False), (64, 8, 1, 8, False),
]


def _logits(T, E, dt, seed):
    g = torch.Generator().manual_seed(seed)
    l = torch.randn(T, E, generator=g) * 2
    if T >= 40:
        l[10:40] = torch.randint(-2, 3, (30, E), generator=g).float()   # exact ties
        l[3, E // 2] = float("nan")
        l[5, 0] = float("inf")
        l[6, :] = float("-inf")
    return l.to(dt)


@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("E,G,SG,k,top2", CASES)
@pytest.mark.parametrize("renorm,with_bias", [(True, True), (False, False), (True, False)])
def test_sigmoid_route_matches_oracle(dt, E, G, SG, k, top2, renorm, with_bias):
    T = 333
    l = _logits(T, E, dt, seed=E + G + SG + k)
    bias = (torch.randn(E, generator=torch.Generator().manual_seed(7)) * 0.05
            if with_bias else None)
    if bias is not None:
        bias[E // 3] = 0.8                                # steers the selection
    idx, w = moe.moe_route_sigmoid_grouped(l.to(DEV), k, G, SG, top2, renorm, 2.5,
                                           None if bias is None else bias.to(DEV))
    torch.cuda.synchronize()
    arr, name = storage(l)
    b64 = None if bias is None else bias.double().numpy()
    ridx, rw = O.route_sigmoid_grouped(O.to_f64(arr, name), b64, k, G, SG, top2, renorm, 2.5, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, f"sigmoid {name} E={E} G={G} k={k}")


@pytest.mark.parametrize("top2", [True, False])
def test_sigmoid_route_near_ties(top2):
    """f32 logits a few ulps apart around a handful of values: most rows fall inside the FP32
    error margin of the first pass and are decided in float64, the rest by the FP32 pass; the
    indices must be the float64 decision either way."""
    T, E, G, SG, k = 2000, 64, 8, 3, 6
    g = torch.Generator().manual_seed(11)
    base = torch.tensor([-1.0, 0.25, 0.5, 1.75], dtype=torch.float32)[
        torch.randint(0, 4, (T, E), generator=g)]
    ulps = torch.randint(-4, 5, (T, E), generator=g).to(torch.int32)
    l = (base.view(torch.int32) + ulps).view(torch.float32)
    l[: T // 2] += torch.randn(T // 2, E, generator=g) * 3          # half the rows well apart
    bias = (torch.randn(E, generator=g) * 1e-7).float()              # corrections of a few ulps
    idx, w = moe.moe_route_sigmoid_grouped(l.to(DEV), k, G, SG, top2, True, 1.0, bias.to(DEV))
    torch.cuda.synchronize()
    ridx, rw = O.route_sigmoid_grouped(O.to_f64(*storage(l)), bias.double().numpy(), k, G, SG,
                                       top2, True, 1.0, "f32")
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, "sigmoid near ties")


def test_sigmoid_route_large_batch():
    T, E = 16384, 256
    wl = W.WORKLOADS["skewed"]
    l = W.make_logits(wl, DEV)
    bias = torch.linspace(-0.1, 0.1, E, device=DEV, dtype=torch.float32)
    idx, w = moe.moe_route_sigmoid_grouped(l, 8, 8, 4, True, True, 2.5, bias)
    torch.cuda.synchronize()
    arr, name = storage(l)
    ridx, rw = O.route_sigmoid_grouped(O.to_f64(arr, name), bias.double().cpu().numpy(), 8, 8, 4,
                                       True, True, 2.5, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, "sigmoid large")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_sigmoid_forward_matches_oracle(dt):
    wl = W.Workload("sig_layer", T=300, H=256, I=384, E=64, top_k=6, renormalize=True,
                    dtype=DT_NAME[dt], seed=31, zipf_s=0.8)
    inp = W.make_layer_inputs(wl, "cpu")
    bias = torch.randn(wl.E, generator=torch.Generator().manual_seed(3)) * 0.1
    g = {k: v.to(DEV) for k, v in inp.items()}
    out = moe.moe_forward_sigmoid_grouped(g["x"], g["logits"], g["gate"], g["up"], g["down"],
                                          wl.top_k, 8, 4, True, True, 1.5, bias.to(DEV))
    torch.cuda.synchronize()
    st = {k: storage(v) for k, v in inp.items()}
    ref = O.forward_sigmoid_grouped(*st["x"], *st["logits"], bias.numpy(), st["gate"][0],
                                    st["up"][0], st["down"][0], st["gate"][1], wl.top_k, 8, 4,
                                    True, True, 1.5)
    err = rel_max_err(f64(out), ref["out_unrounded"])
    assert err <= layer_tol(dt), err
