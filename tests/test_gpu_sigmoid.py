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
@pytest.mark.parametrize("E,G,SG,k", [(64, 8, 3, 6), (256, 8, 4, 8)])
def test_sigmoid_route_near_ties(top2, E, G, SG, k):
    """f32 logits a few ulps apart around a handful of values: most rows fall inside the FP32
    error margin of the first pass and are decided in float64 (the runs of close candidates up to
    the k-th, or the whole row), the rest by the FP32 pass; the indices must be the float64
    decision either way."""
    T = 2000
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


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("E,G,SG,k", [(256, 8, 4, 8), (64, 8, 3, 6), (256, 8, 1, 8)])
@pytest.mark.parametrize("with_bias", [True, False])
def test_sigmoid_route_crowded_rows(dt, E, G, SG, k, with_bias):
    """Rows whose chosen groups hold many candidates at or near the k-th score: constant rows (every
    candidate ties), rows of a few repeated values (dozens of exact ties at the line), and rows with
    one dominant value per group.  They exercise both forms of the top-k inside the chosen groups:
    the ranked compaction of the candidates near the line, and the rounds of sub-warp argmax when
    more candidates sit there than the compaction holds."""
    T = 480
    g = torch.Generator().manual_seed(E + SG + k)
    l = torch.randn(T, E, generator=g)
    l[0:60] = 0.5                                                      # constant rows
    l[60:120] = 0.0
    l[120:240] = torch.randint(0, 3, (120, E), generator=g).float()   # three values
    l[240:300] = torch.randint(0, 2, (60, E), generator=g).float() * 4 - 2
    l[300:360, ::5] = 3.0                                              # a dominant value
    l = l.to(dt)
    bias = None
    if with_bias:
        bias = torch.zeros(E)
        bias[::7] = 0.25                                               # lifts a few experts
    idx, w = moe.moe_route_sigmoid_grouped(l.to(DEV), k, G, SG, True, True, 1.0,
                                           None if bias is None else bias.to(DEV))
    torch.cuda.synchronize()
    arr, name = storage(l)
    b64 = None if bias is None else bias.double().numpy()
    ridx, rw = O.route_sigmoid_grouped(O.to_f64(arr, name), b64, k, G, SG, True, True, 1.0, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, f"sigmoid crowded {name} E={E} SG={SG}")


@pytest.mark.parametrize("E,G,SG,k", [(256, 8, 4, 8), (64, 8, 3, 6)])
def test_sigmoid_route_close_pairs(E, G, SG, k):
    """Rows with a few candidates one or two ulps apart at chosen places of the ranking (inside the
    top k, across the k-th / (k+1)-th boundary, a chain of four), the rest well apart: the FP32
    pass proves all but the close runs, which are ordered by their float64 scores."""
    T = 1000
    g = torch.Generator().manual_seed(E + k)
    l = torch.randn(T, E, generator=g) * 2
    order = l.argsort(dim=1, descending=True)
    rows = torch.arange(T)

    def tie(r, p, q, ulps):  # logit at sorted place q := logit at place p moved by `ulps` ulps
        src = l[r, order[r, p]]
        moved = (src.view(torch.int32) + torch.tensor(ulps, dtype=torch.int32)).view(torch.float32)
        l[r, order[r, q]] = moved

    for r in range(0, 250):
        tie(r, 2, 3, -1)
    for r in range(250, 500):
        tie(r, k - 1, k, 1 if r % 2 else -1)
    for r in range(500, 750):
        for q in range(k - 3, k + 1):
            tie(r, k - 4, q, -(q - k + 4) * (1 if r % 3 else -1))
    assert rows.numel() == T
    idx, w = moe.moe_route_sigmoid_grouped(l.to(DEV), k, G, SG, True, True, 1.0, None)
    torch.cuda.synchronize()
    ridx, rw = O.route_sigmoid_grouped(O.to_f64(*storage(l)), None, k, G, SG, True, True, 1.0,
                                       "f32")
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, "sigmoid close pairs")
