"""Pins of the oracle's MoE backward chain (ruDNN user guide §12) to torch autograd of the float64
forward, stage by stage and end to end (dL/dx, dL/dlogits, dL/dgate, dL/dup, dL/ddown)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _layer(seed, T=23, H=12, I=10, E=5, k=2):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E))
    x = rng.standard_normal((T, H))
    gate = rng.standard_normal((E, I, H)) / np.sqrt(H)
    up = rng.standard_normal((E, I, H)) / np.sqrt(H)
    down = rng.standard_normal((E, H, I)) / np.sqrt(I)
    dout = rng.standard_normal((T, H))
    return l, x, gate, up, down, dout, k


def test_combine_backward_matches_autograd():
    l, x, gate, up, down, dout, k = _layer(1)
    idx, w = O.route(l, k, True, "f32")
    _, _, _, ros = O.dispatch(idx, l.shape[1])
    y = np.random.default_rng(2).standard_normal((x.shape[0] * k, x.shape[1]))
    Y = torch.tensor(y, requires_grad=True)
    Wt = torch.tensor(w, requires_grad=True)
    rs = torch.from_numpy(ros.astype(np.int64)).view(-1, k)
    out = sum(Wt[:, j:j + 1] * Y[rs[:, j]] for j in range(k))
    (out * torch.from_numpy(dout)).sum().backward()
    de, dw = O.combine_backward(y, ros, w, dout)
    np.testing.assert_allclose(de, Y.grad.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dw, Wt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_experts_backward_matches_autograd():
    l, x, gate, up, down, dout, k = _layer(3)
    idx, _ = O.route(l, k, True, "f32")
    _, offsets, tor, _ = O.dispatch(idx, l.shape[1])
    xd = O.gather(x, tor)
    dy = np.random.default_rng(4).standard_normal(xd.shape)
    f32 = lambda a: a.astype(np.float32)  # noqa: E731 - the oracle reads stored (f32) weights
    dx, dg, du, dd = O.experts_backward(xd, offsets, f32(gate), f32(up), f32(down), "f32", dy)
    # autograd on the same stored values
    G2, U2, D2 = (torch.tensor(f32(a).astype(np.float64), requires_grad=True)
                  for a in (gate, up, down))
    X2 = torch.tensor(xd, requires_grad=True)
    ys = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        xe = X2[lo:hi]
        ys.append((F.silu(xe @ G2[e].T) * (xe @ U2[e].T)) @ D2[e].T)
    (torch.cat(ys) * torch.from_numpy(dy)).sum().backward()
    np.testing.assert_allclose(dx, X2.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dg, G2.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(du, U2.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dd, D2.grad.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("renorm", [True, False])
def test_full_chain_matches_autograd(renorm):
    """dispatch_backward(experts_backward(combine_backward)) + the router backward equals autograd
    of the whole float64 forward with the selection held fixed."""
    l, x, gate, up, down, dout, k = _layer(5, k=3)
    T, E = l.shape
    idx, w = O.route(l, k, renorm, "f32")
    w64 = O.selected_router_weights(l, idx, "softmax", renorm, 1.0)   # unrounded weights
    _, offsets, tor, ros = O.dispatch(idx, E)
    xd = O.gather(x, tor)
    gate32, up32, down32 = (a.astype(np.float32) for a in (gate, up, down))
    y = O.experts(xd, offsets, gate32, up32, down32, "f32")
    dexp, dwts = O.combine_backward(y, ros, w64, dout)
    dxd, dg, du, dd = O.experts_backward(xd, offsets, gate32, up32, down32, "f32", dexp)
    dx = O.dispatch_backward(dxd, ros, T, k)
    dl = O.selected_router_backward(l, idx, dwts, "softmax", renorm, 1.0)

    L = torch.tensor(l, requires_grad=True)
    X = torch.tensor(x, requires_grad=True)
    G, U, D = (torch.tensor(a.astype(np.float64), requires_grad=True)
               for a in (gate32, up32, down32))
    P = torch.softmax(L, 1).gather(1, torch.from_numpy(idx.astype(np.int64)))
    if renorm:
        P = P / P.sum(1, keepdim=True)
    out = torch.zeros(T, x.shape[1], dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            xe = X[t]
            out[t] = out[t] + P[t, j] * ((F.silu(G[e] @ xe) * (U[e] @ xe)) @ D[e].T)
    (out * torch.from_numpy(dout)).sum().backward()
    np.testing.assert_allclose(dx, X.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dl, L.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, G.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(du, U.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dd, D.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_dispatch_backward_sums_slots_without_weights():
    idx = np.array([[0, 1], [1, 1], [2, 0]], dtype=np.uint32)
    _, _, _, ros = O.dispatch(idx, 3)
    dinp = np.arange(6 * 2, dtype=np.float64).reshape(6, 2)
    dx = O.dispatch_backward(dinp, ros, 3, 2)
    rs = ros.astype(np.int64).reshape(3, 2)
    np.testing.assert_array_equal(dx, dinp[rs[:, 0]] + dinp[rs[:, 1]])
