"""GPU parity of fixed-selection router weights and their logits gradient (ruDNN user guide §12)
against the fp64 oracle: FP32 weights within 2e-6 * scale + 1e-5 |ref|; gradients within one
rounding of the logits dtype plus 1e-5 of the row's largest gradient; NaN rows (invalid index,
poisoned softmax row) exactly where the oracle has them."""
import numpy as np
import pytest
import torch

import oracle as O
import mixture_experts_routing_moe_gb300 as moe
from gpu_helpers import f64, storage

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL = {torch.float32: 1e-5, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -10}


def _case(T, E, k, ldt, idt, seed):
    g = torch.Generator().manual_seed(seed)
    l = (torch.randn(T, E, generator=g) * 1.5)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)])
    if k >= 2:
        idx[0, 1] = idx[0, 0]                       # repeated index: gather semantics
    idx[2, k - 1] = E                               # invalid: row 2 becomes NaN
    if idt != torch.uint32:
        idx[3, 0] = -1                              # negative index (signed types)
    l[5, 0] = float("nan")                          # poisoned softmax row
    gw = torch.randn(T, k, generator=g)
    return l.to(ldt), idx, gw


def _to_idx(idx, idt):
    if idt == torch.uint32:
        return torch.from_numpy(idx.numpy().astype(np.uint32).view(np.int32)).view(torch.uint32)
    return idx.to(idt)


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("ldt", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("idt", [torch.uint32, torch.int32, torch.int64])
@pytest.mark.parametrize("T,E,k", [(300, 64, 8), (60, 1000, 64), (40, 7, 7)])
def test_router_weights_and_backward_match_oracle(scoring, renorm, ldt, idt, T, E, k):
    l, idx, gw = _case(T, E, k, ldt, idt, seed=T + E + k)
    gi = _to_idx(idx, idt).to(DEV)
    w = moe.moe_selected_router_weights(l.to(DEV), gi, scoring, renorm, 2.5)
    d = moe.moe_selected_router_backward(l.to(DEV), gi, gw.to(DEV), scoring, renorm, 2.5)
    torch.cuda.synchronize()
    arr, name = storage(l)
    l64 = O.to_f64(arr, name)
    idx64 = idx.numpy().astype(np.int64)
    if idt == torch.uint32:
        idx64 = np.where(idx64 < 0, 2 ** 32 + idx64, idx64)
    rw = O.selected_router_weights(l64, idx64, scoring, renorm, 2.5)
    rd = O.selected_router_backward(l64, idx64, gw.double().numpy(), scoring, renorm, 2.5)
    gw_ = w.double().cpu().numpy()
    assert (np.isnan(gw_) == np.isnan(rw)).all()
    ok = ~np.isnan(rw)
    assert (np.abs(gw_[ok] - rw[ok]) <= 2e-6 * 2.5 + 1e-5 * np.abs(rw[ok])).all()
    gd = f64(d)
    assert (np.isnan(gd) == np.isnan(rd)).all()
    fin = ~np.isnan(rd).any(axis=1)
    rowmax = np.abs(rd[fin]).max(axis=1, keepdims=True)
    err = np.abs(gd[fin] - rd[fin])
    assert (err <= REL[ldt] * np.abs(rd[fin]) + 1e-5 * rowmax + 1e-30).all(), err.max()


def test_backward_is_run_to_run_identical():
    l, idx, gw = _case(500, 256, 16, torch.float32, torch.int32, seed=9)
    args = (l.to(DEV), idx.to(torch.int32).to(DEV), gw.to(DEV), "softmax", True, 1.0)
    a = moe.moe_selected_router_backward(*args)
    b = moe.moe_selected_router_backward(*args)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
