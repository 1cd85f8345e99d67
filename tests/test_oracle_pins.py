"""Pins of the fp64 oracle to things other than itself (no GPU needed).

Each check is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign or
index, a transposed operand, a wrong tie rule) fails one of them: closed forms, hand-derived
fixtures under tests/golden/, library routines (torch float64 softmax / silu, numpy's and torch's
float casts), brute force on tiny inputs, and invariants of the routing contract in the ruDNN
user guide §4 "Routing-Vertrag" and §5 "Expertengewichte und Verteilung".
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from mixture_experts_routing_moe_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _num(s):
    return float(eval(s, {"__builtins__": {}}, {"inf": math.inf, "nan": math.nan}))


def _vec(s):
    return np.array([_num(v) for v in s.split(",")], dtype=np.float64)


# ------------------------------------------------------------------ storage and rounding
def test_bf16_to_f64_matches_torch():
    g = torch.Generator().manual_seed(1)
    t = (torch.randn(4096, generator=g) * 1e3).to(torch.bfloat16)
    t[:4] = torch.tensor([float("inf"), float("-inf"), 0.0, -0.0])
    arr, dt = W.to_storage_numpy(t)
    np.testing.assert_array_equal(O.to_f64(arr, dt), t.to(torch.float64).numpy())


def test_round_f32_matches_numpy_cast():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-45, 39, 20000),
                        [3.4028235677973366e38, 3.4028235e38 * 1.0000001, 1e-46, -1e-45]])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(O.round_to_dtype(x, "f32"), ref)


@pytest.mark.parametrize("dt,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_round_matches_torch_cast_of_float32(dt, tdt):
    # float32 inputs are exact in float64, so torch's single rounding float32 -> dt is the answer
    g = torch.Generator().manual_seed(3)
    x = torch.randn(50000, generator=g) * torch.exp2(torch.randint(-30, 30, (50000,), generator=g).float())
    # every tie pattern: float32 values whose dropped bits are exactly half
    ties = torch.arange(0, 4096, dtype=torch.int32) << 12 | (1 << 15) | (0x3F800000)
    ties = ties.view(torch.float32)
    x = torch.cat([x, ties, -ties, torch.tensor([65519.0, 65520.0, 65536.0, 3.4e38, 1e-40, 6e-8])])
    ref = x.to(tdt).to(torch.float64).numpy()
    got = O.round_to_dtype(x.double().numpy(), dt)
    np.testing.assert_array_equal(got, ref)


def test_rounding_golden(golden):
    for dt, inp, exp in golden("rounding_cases.txt"):
        got = O.round_to_dtype(np.array([_num(inp)]), dt)[0]
        assert got == _num(exp), (dt, inp, got, exp)


@pytest.mark.parametrize("dt", O.DTYPES)
def test_encode_roundtrip(dt):
    x = np.random.default_rng(4).standard_normal(1000) * 7
    np.testing.assert_array_equal(O.to_f64(O.encode(x, dt), dt), O.round_to_dtype(x, dt))


# ------------------------------------------------------------------ softmax
def test_softmax_matches_torch_and_sums_to_one():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((300, 37)) * 5
    l[0, 3] = -np.inf
    p = O.softmax(l)
    np.testing.assert_allclose(p, torch.softmax(torch.from_numpy(l), dim=1).numpy(), rtol=1e-13,
                               atol=1e-300)
    np.testing.assert_allclose(p.sum(1), 1.0, rtol=1e-13)
    assert p[0, 3] == 0.0


def test_softmax_two_expert_closed_form():
    a, b = 0.3, -1.7
    p = O.softmax(np.array([[a, b]]))[0]
    assert p[0] == pytest.approx(1.0 / (1.0 + math.exp(b - a)), rel=1e-15)
    assert p[1] == pytest.approx(1.0 / (1.0 + math.exp(a - b)), rel=1e-15)


def test_softmax_identical_logits_and_huge_values():
    p = O.softmax(np.full((2, 5), 123.0))
    np.testing.assert_allclose(p, 0.2, rtol=1e-15)
    # large magnitudes need the max subtraction; exp(1000) alone overflows
    p = O.softmax(np.array([[1000.0, 1000.0 + math.log(3.0)]]))[0]
    np.testing.assert_allclose(p, [0.25, 0.75], rtol=1e-12)


# ------------------------------------------------------------------ selection / route
def _brute_topk(row, k):
    """Definition: i precedes u iff l_i > l_u, or l_i == l_u and i < u; take the first k."""
    E = len(row)
    better = lambda i, u: row[i] > row[u] or (row[i] == row[u] and i < u)  # noqa: E731
    chosen = []
    for _ in range(k):
        best = None
        for i in range(E):
            if i in chosen:
                continue
            if best is None or better(i, best):
                best = i
        chosen.append(best)
    return chosen


def test_select_topk_brute_force_with_many_ties():
    rng = np.random.default_rng(6)
    for E in (1, 2, 3, 5, 8, 13):
        l = rng.integers(-2, 3, size=(200, E)).astype(np.float64)  # small ints: ties everywhere
        l[rng.random((200, E)) < 0.1] = -np.inf
        l[np.isneginf(l).all(1), 0] = 0.0
        for k in range(1, E + 1):
            idx = O.select_topk(l, k)
            for t in range(l.shape[0]):
                assert list(idx[t]) == _brute_topk(l[t], k)


def test_route_golden(golden):
    for name, dt, k, renorm, logits, eidx, ew in golden("route_cases.txt"):
        l = O.round_to_dtype(_vec(logits)[None, :], dt)
        idx, w = O.route(l, int(k), bool(int(renorm)), dt)
        assert list(idx[0]) == [int(v) for v in eidx.split(",")], name
        if ew != "-":
            np.testing.assert_array_equal(w[0], _vec(ew), err_msg=name)


def test_route_topk_equals_E_is_full_softmax_sorted():
    rng = np.random.default_rng(7)
    l = rng.standard_normal((64, 16))
    idx, w = O.route(l, 16, True, "f32")
    order = np.argsort(-l, axis=1, kind="stable")
    np.testing.assert_array_equal(idx, order)
    p = torch.softmax(torch.from_numpy(l), 1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(p, order, 1), rtol=2 ** -23)


def test_route_renormalised_weights_sum_to_one_and_ratio_kept():
    rng = np.random.default_rng(8)
    l = rng.standard_normal((500, 64)) * 2
    idx, w = O.route(l, 8, True, "f32")
    np.testing.assert_allclose(w.sum(1), 1.0, atol=8 * 2 ** -24)
    _, wp = O.route(l, 8, False, "f32")
    # renormalising only rescales a row: the ratios between selected weights are unchanged
    np.testing.assert_allclose(w / w[:, :1], wp / wp[:, :1], rtol=4 * 2 ** -24)
    # without renormalisation, weights are the plain softmax values
    p = torch.softmax(torch.from_numpy(l), 1).numpy()
    np.testing.assert_allclose(wp, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=2 ** -24)


def test_route_weights_descending():
    l = np.random.default_rng(9).standard_normal((200, 32))
    for dt in O.DTYPES:
        _, w = O.route(O.round_to_dtype(l, dt), 6, False, dt)
        assert (np.diff(w, axis=1) <= 0).all()


def test_tiny_workload_special_rows():
    w = W.WORKLOADS["tiny_f32"]
    arr, dt = W.to_storage_numpy(W.make_logits(w))
    idx, wt = O.route(O.to_f64(arr, dt), w.top_k, w.renormalize, dt)
    assert [list(r) for r in idx[:7]] == [[1, 5], [0, 7], [3, 1], [0, 7], [0, 1], [0, 1], [0, 1]]
    assert (wt[0] == 0.5).all() and (wt[1] == 0.5).all() and (wt[3] == 0.5).all()
    assert np.isnan(wt[4:7]).all() and not np.isnan(wt[7:]).any()


# ------------------------------------------------------------------ dispatch
def test_dispatch_golden(golden):
    for name, E, k, idx, counts, tor, ros in golden("dispatch_cases.txt"):
        ix = np.array([int(v) for v in idx.split(",")], dtype=np.uint32).reshape(-1, int(k))
        c, off, t_of_r, r_of_s = O.dispatch(ix, int(E))
        assert list(c) == [int(v) for v in counts.split(",")], name
        assert list(t_of_r) == [int(v) for v in tor.split(",")], name
        assert list(r_of_s) == [int(v) for v in ros.split(",")], name
        assert list(off) == [0] + list(np.cumsum(c)), name


@pytest.mark.parametrize("skew", ["uniform", "same_set", "zipf"])
def test_dispatch_invariants(skew):
    rng = np.random.default_rng(10)
    T, E, k = 333, 40, 4
    if skew == "uniform":
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    elif skew == "same_set":
        idx = np.tile(np.arange(k), (T, 1)) * 0 + np.array([7, 0, 1, 2])
    else:
        p = np.arange(1, E + 1) ** -1.5
        idx = np.stack([rng.choice(E, k, replace=False, p=p / p.sum()) for _ in range(T)])
    idx = idx.astype(np.uint32)
    c, off, t_of_r, r_of_s = O.dispatch(idx, E)
    assert c.sum() == T * k                                       # nothing dropped
    assert sorted(r_of_s.tolist()) == list(range(T * k))          # bijection
    flat = idx.reshape(-1)
    for e in range(E):                                            # brute-force group contents
        slots = [s for s in range(T * k) if flat[s] == e]
        rows = list(range(off[e], off[e + 1]))
        assert [int(r_of_s[s]) for s in slots] == rows
        assert [int(t_of_r[r]) for r in rows] == [s // k for s in slots]
    # permutation round trip: scatter then gather back restores slot order
    vals = rng.standard_normal(T * k)
    disp = np.empty(T * k)
    disp[r_of_s] = vals
    np.testing.assert_array_equal(disp[r_of_s], vals)


# ------------------------------------------------------------------ experts / combine / forward
def test_silu_closed_form():
    z = np.array([0.0, 1.0, -1.0, 40.0, -800.0])
    got = O.silu(z)
    exp = [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e), 40.0, -0.0]
    np.testing.assert_allclose(got, exp, rtol=1e-15, atol=0)
    zs = torch.linspace(-9, 9, 101, dtype=torch.float64)
    np.testing.assert_allclose(O.silu(zs.numpy()), F.silu(zs).numpy(), rtol=1e-14)


def _rand_layer(rng, T, H, I, E, k, dt="f32", tie_free=True):
    l = rng.standard_normal((T, E))
    x = rng.standard_normal((T, H))
    gate = rng.standard_normal((E, I, H)) / math.sqrt(H)
    up = rng.standard_normal((E, I, H)) / math.sqrt(H)
    down = rng.standard_normal((E, H, I)) / math.sqrt(I)
    enc = lambda a: O.encode(a, dt)  # noqa: E731
    return enc(x), enc(l), enc(gate), enc(up), enc(down)


def test_single_expert_is_plain_swiglu_mlp():
    rng = np.random.default_rng(11)
    x, l, gate, up, down = _rand_layer(rng, 17, 24, 40, 1, 1)
    r = O.forward(x, "f32", l, "f32", gate, up, down, "f32", 1, True)
    X = torch.from_numpy(x.astype(np.float64))
    G, U, D = (torch.from_numpy(a[0].astype(np.float64)) for a in (gate, up, down))
    ref = (F.silu(X @ G.T) * (X @ U.T)) @ D.T
    np.testing.assert_allclose(r["out_unrounded"], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert (r["w"] == 1.0).all()


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("dt", O.DTYPES)
def test_forward_matches_dense_brute_force(renorm, dt):
    """Every expert on every token densely, then out[t] = sum_e G[t,e] * D[t,e] with G the
    scattered routing weights: independent of dispatch order and of the combine's indexing."""
    rng = np.random.default_rng(12)
    T, H, I, E, k = 29, 16, 12, 6, 3
    x, l, gate, up, down = _rand_layer(rng, T, H, I, E, k, dt)
    r = O.forward(x, dt, l, dt, gate, up, down, dt, k, renorm)
    X = torch.from_numpy(O.to_f64(x, dt))
    dense = np.zeros((T, E, H))
    for e in range(E):
        G, U, D = (torch.from_numpy(O.to_f64(a[e], dt)) for a in (gate, up, down))
        dense[:, e] = ((F.silu(X @ G.T) * (X @ U.T)) @ D.T).numpy()
    Gm = np.zeros((T, E))
    for t in range(T):
        for j in range(k):
            Gm[t, r["idx"][t, j]] += r["w"][t, j]
    ref = np.einsum("te,teh->th", Gm, dense)
    np.testing.assert_allclose(r["out_unrounded"], ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(r["out"], O.round_to_dtype(r["out_unrounded"], dt))


def test_combine_one_hot_and_slot_order():
    T, k, H = 5, 3, 4
    idx = np.array([[0, 1, 2], [2, 1, 0], [1, 1, 1], [0, 0, 0], [2, 0, 1]], dtype=np.uint32)
    _, _, t_of_r, r_of_s = O.dispatch(idx, 3)
    y = np.zeros((T * k, H))
    for r in range(T * k):
        y[r, r % H] = 1.0 + r                                  # tag each row
    w = np.arange(T * k, dtype=np.float64).reshape(T, k) + 0.5
    out = O.combine(y, r_of_s, w)
    for t in range(T):
        ref = np.zeros(H)
        for j in range(k):
            r = r_of_s[t * k + j]
            ref += w[t, j] * y[r]
        np.testing.assert_array_equal(out[t], ref)


def test_combine_nan_weight_poisons_token_only():
    idx = np.array([[0, 1], [1, 0]], dtype=np.uint32)
    _, _, _, r_of_s = O.dispatch(idx, 2)
    y = np.ones((4, 3))
    w = np.array([[np.nan, np.nan], [0.25, 0.75]])
    out = O.combine(y, r_of_s, w)
    assert np.isnan(out[0]).all()
    np.testing.assert_array_equal(out[1], 1.0)


def test_down_weights_scale_output_linearly():
    rng = np.random.default_rng(13)
    x, l, gate, up, down = _rand_layer(rng, 11, 8, 6, 4, 2)
    r1 = O.forward(x, "f32", l, "f32", gate, up, down, "f32", 2, True)
    r2 = O.forward(x, "f32", l, "f32", gate, up, (down.astype(np.float64) * 2).astype(np.float32),
                   "f32", 2, True)
    np.testing.assert_allclose(r2["out_unrounded"], 2 * r1["out_unrounded"], rtol=1e-14)


def test_forward_rows_matches_forward():
    rng = np.random.default_rng(14)
    x, l, gate, up, down = _rand_layer(rng, 40, 16, 24, 5, 2, "bf16")
    r = O.forward(x, "bf16", l, "bf16", gate, up, down, "bf16", 2, True)
    tok = np.array([3, 0, 39, 17])
    f64 = lambda a, e: O.to_f64(a[e], "bf16")  # noqa: E731
    got = O.forward_rows(O.to_f64(x, "bf16")[tok], r["idx"][tok], r["w"][tok],
                         lambda e: (f64(gate, e), f64(up, e), f64(down, e)))
    np.testing.assert_allclose(got, r["out_unrounded"][tok], rtol=1e-13, atol=1e-13)


def test_tiny_workload_full_forward_no_token_dropped():
    w = W.WORKLOADS["tiny_f32"]
    inp = W.make_layer_inputs(w)
    st = {k: W.to_storage_numpy(v) for k, v in inp.items()}
    r = O.forward(*st["x"], *st["logits"], st["gate"][0], st["up"][0], st["down"][0], "f32",
                  w.top_k, w.renormalize)
    assert r["counts"].sum() == w.T * w.top_k
    assert np.isnan(r["out"][4:7]).all() and np.isfinite(r["out"][7:]).all()
    assert np.isfinite(r["out"][:4]).all()
