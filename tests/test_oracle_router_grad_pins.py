"""Pins of the oracle's fixed-selection router weights and their gradient (ruDNN user guide §12):
central finite differences and torch.autograd (both float64) for the gradient, torch softmax /
sigmoid gathers for the weights, gather semantics of repeated indices, NaN rows for invalid
indices, linearity in `scale`."""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
MODES = [(s, r) for s in ("softmax", "sigmoid") for r in (False, True)]


def _case(seed, T=7, E=9, k=4):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)) * 1.5
    idx = rng.integers(0, E, size=(T, k))
    idx[0, 1] = idx[0, 0]                 # a repeated index (gather semantics)
    g = rng.standard_normal((T, k))
    return l, idx, g


@pytest.mark.parametrize("scoring,renorm", MODES)
def test_gradient_matches_central_differences(scoring, renorm):
    l, idx, g = _case(1)
    an = O.selected_router_backward(l, idx, g, scoring, renorm, 1.7)
    h = 1e-6
    fd = np.zeros_like(l)
    for t in range(l.shape[0]):
        for e in range(l.shape[1]):
            lp, lm = l.copy(), l.copy()
            lp[t, e] += h
            lm[t, e] -= h
            dw = (O.selected_router_weights(lp, idx, scoring, renorm, 1.7)
                  - O.selected_router_weights(lm, idx, scoring, renorm, 1.7))
            fd[t, e] = (dw[t] * g[t]).sum() / (2 * h)
    np.testing.assert_allclose(an, fd, atol=1e-8)


@pytest.mark.parametrize("scoring,renorm", MODES)
def test_weights_and_gradient_match_torch_autograd(scoring, renorm):
    l, idx, g = _case(2, T=50, E=33, k=6)
    L = torch.tensor(l, requires_grad=True)
    P = torch.softmax(L, 1) if scoring == "softmax" else torch.sigmoid(L)
    W = P.gather(1, torch.from_numpy(idx))
    if renorm:
        W = W / W.sum(1, keepdim=True)
    W = W * 2.5
    (W * torch.from_numpy(g)).sum().backward()
    np.testing.assert_allclose(O.selected_router_weights(l, idx, scoring, renorm, 2.5),
                               W.detach().numpy(), rtol=1e-13)
    np.testing.assert_allclose(O.selected_router_backward(l, idx, g, scoring, renorm, 2.5),
                               L.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_invalid_index_gives_nan_row_only():
    l, idx, g = _case(3)
    idx = idx.copy()
    idx[2, 3] = l.shape[1]          # out of range
    idx[4, 0] = -1                  # negative (signed index types)
    for scoring, renorm in MODES:
        w = O.selected_router_weights(l, idx, scoring, renorm, 1.0)
        d = O.selected_router_backward(l, idx, g, scoring, renorm, 1.0)
        assert np.isnan(w[[2, 4]]).all() and np.isnan(d[[2, 4]]).all()
        keep = [0, 1, 3, 5, 6]
        assert np.isfinite(w[keep]).all() and np.isfinite(d[keep]).all()


def test_scale_is_linear():
    l, idx, g = _case(4)
    for scoring, renorm in MODES:
        a = O.selected_router_backward(l, idx, g, scoring, renorm, 1.0)
        b = O.selected_router_backward(l, idx, g, scoring, renorm, 3.0)
        np.testing.assert_allclose(b, 3 * a, rtol=1e-14, atol=1e-300)
