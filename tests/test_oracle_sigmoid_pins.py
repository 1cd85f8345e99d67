"""Pins of the oracle's group-limited sigmoid router (ruDNN user guide §10) to hand-worked cases,
torch's sigmoid / topk on tie-free data, and the invariants the page states (the bias changes
the selection only; renormalised weights sum to `scale`)."""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _num(v):
    return float(eval(v, {"__builtins__": {}}, {"inf": math.inf, "nan": math.nan}))


def _vec(s):
    return np.array([_num(v) for v in s.split(",")])


def test_sigmoid_closed_form_and_torch():
    z = torch.linspace(-30, 30, 241, dtype=torch.float64)
    np.testing.assert_allclose(O.sigmoid(z.numpy()), torch.sigmoid(z).numpy(), rtol=1e-15)
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    assert O.sigmoid(np.array([-np.inf]))[0] == 0.0 and O.sigmoid(np.array([np.inf]))[0] == 1.0


def test_sigmoid_route_golden(golden):
    rows = golden("sigmoid_route_cases.txt")
    assert len(rows) == 9
    for name, dt, k, G, sel, top2, ren, scale, logits, bias, eidx, ew in rows:
        l = O.round_to_dtype(_vec(logits)[None, :], dt)
        b = None if bias == "-" else _vec(bias)
        idx, w = O.route_sigmoid_grouped(l, b, int(k), int(G), int(sel), bool(int(top2)),
                                         bool(int(ren)), float(scale), dt)
        assert list(idx[0]) == [int(v) for v in eidx.split(",")], name
        if ew != "-":
            np.testing.assert_array_equal(w[0], _vec(ew), err_msg=name)


def _torch_reference(l, b, k, G, sel, top2, ren, scale):
    """The same routing written with torch.sigmoid / torch.topk (tie-free inputs only)."""
    L = torch.from_numpy(l)
    s = torch.sigmoid(L)
    c = s + (0 if b is None else torch.from_numpy(b))
    T, E = L.shape
    cg = c.view(T, G, E // G)
    gsc = cg.topk(2, dim=2).values.sum(2) if top2 else cg.max(2).values
    gi = gsc.topk(sel, dim=1).indices
    mask = torch.zeros(T, G, dtype=torch.bool).scatter_(1, gi, True).repeat_interleave(E // G, 1)
    idx = c.masked_fill(~mask, float("-inf")).topk(k, dim=1).indices
    w = s.gather(1, idx)
    if ren:
        w = w / w.sum(1, keepdim=True)
    return idx.numpy(), (w * scale).numpy()


@pytest.mark.parametrize("E,G,sel,k,top2", [(64, 8, 3, 6, True), (256, 8, 4, 8, True),
                                            (32, 4, 1, 8, False), (48, 1, 1, 5, False),
                                            (128, 16, 16, 16, True)])
@pytest.mark.parametrize("ren", [True, False])
def test_sigmoid_route_matches_torch_topk(E, G, sel, k, top2, ren):
    rng = np.random.default_rng(E + G + sel + k)
    l = rng.standard_normal((300, E)) * 2
    b = rng.standard_normal(E) * 0.1
    idx, w = O.route_sigmoid_grouped(l, b, k, G, sel, top2, ren, 2.5, "f32")
    ridx, rw = _torch_reference(l, b, k, G, sel, top2, ren, 2.5)
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2 ** -23)


def test_bias_changes_selection_only():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((200, 32))
    b = np.zeros(32)
    b[7] = 5.0                                    # expert 7 always wins the selection
    idx, w = O.route_sigmoid_grouped(l, b, 2, 1, 1, False, False, 1.0, "f32")
    assert (idx[:, 0] == 7).all()
    np.testing.assert_allclose(w[:, 0], O.round_to_dtype(O.sigmoid(l[:, 7]), "f32"))


def test_renormalised_weights_sum_to_scale():
    l = np.random.default_rng(4).standard_normal((100, 64))
    _, w = O.route_sigmoid_grouped(l, None, 8, 8, 4, True, True, 3.0, "f32")
    np.testing.assert_allclose(w.sum(1), 3.0, rtol=1e-6)
