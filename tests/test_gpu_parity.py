"""GPU parity: every stage of the CUDA path, called through the C ABI, against the fp64 oracle.

Bars (from the routing contract of the ruDNN user guide §4 and the layer definition of §5):
indices, counts, offsets and row maps bit-exact; route weights within abs 1e-6 (f32) or 1 ulp
(f16 / bf16), NaN where the oracle has NaN; layer outputs within max|d| / max|ref| <= 2e-2 for
16-bit layers and 1e-4 for f32 layers; repeated runs bitwise identical.
"""
import numpy as np
import pytest
import torch

import oracle as O
import mixture_experts_routing_moe_gb300 as moe
from mixture_experts_routing_moe_gb300 import workloads as W
from gpu_helpers import (DT_NAME, check_weights, f64, layer_tol, oracle_expert_weights,
                         rel_max_err, storage, u32)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _logits(T, E, dt, seed, std=2.0, ties=True, poison=True):
    g = torch.Generator().manual_seed(seed)
    l = torch.randn(T, E, generator=g) * std
    if ties and T >= 40:
        l[10:40] = torch.randint(-2, 3, (30, E), generator=g).float()   # many exact ties
    if poison and T >= 8:
        l[1, E // 2] = float("nan")
        l[3, E - 1] = float("inf")
        l[5, :] = float("-inf")
        if E > 2:
            l[7, : E - 2] = float("-inf")           # finite row with few finite entries
    l = l.to(dt)
    if poison and T >= 10:
        # a NaN with the sign bit set (bit pattern), which sorts below -inf as raw bits
        bits = {torch.float32: (torch.int32, -4194303), torch.float16: (torch.int16, -511),
                torch.bfloat16: (torch.int16, -63)}[dt]
        l.view(bits[0])[9, E // 3] = bits[1]
    return l


# ------------------------------------------------------------------------------------ route
ROUTE_SHAPES = [(1000, 8, 2), (777, 64, 8), (513, 128, 8), (300, 256, 8), (129, 1000, 16),
                (64, 1, 1), (50, 7, 7), (33, 3, 2), (250, 64, 64), (200, 40, 5)]


@pytest.mark.parametrize("dt", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("T,E,k", ROUTE_SHAPES)
@pytest.mark.parametrize("renorm", [True, False])
def test_route_matches_oracle(dt, T, E, k, renorm):
    l = _logits(T, E, dt, seed=T * 31 + E + k)
    idx, w = moe.moe_route(l.to(DEV), k, renorm)
    torch.cuda.synchronize()
    arr, name = storage(l)
    ridx, rw = O.route(O.to_f64(arr, name), k, renorm, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, f"{name} T={T} E={E} k={k}")


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("k,renorm", [(8, True), (8, False), (3, True)])
def test_route_e64_many_waves(dt, k, renorm):
    """E = 64 at a size where 256-row tiles staged in shared memory run in several waves over
    the SMs (T = 2 x 3 x 152 x 256 + 77 rows), with a ragged last tile (ties, NaN, inf and -inf
    rows included)."""
    T = 2 * 3 * 152 * 256 + 77
    l = _logits(T, 64, dt, seed=6400 + k)
    idx, w = moe.moe_route(l.to(DEV), k, renorm)
    torch.cuda.synchronize()
    arr, name = storage(l)
    ridx, rw = O.route(O.to_f64(arr, name), k, renorm, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, f"{name} T={T} E=64 k={k}")


def test_route_unaligned_rows_take_scalar_path():
    base = _logits(301, 10, torch.bfloat16, seed=5)      # 20-byte rows: no 16-byte loads
    storage_t = torch.empty(301 * 10 + 3, dtype=torch.bfloat16, device=DEV)
    l = storage_t[3:].view(301, 10)
    l.copy_(base.to(DEV))
    idx, w = moe.moe_route(l, 3, True)
    arr, name = storage(base)
    ridx, rw = O.route(O.to_f64(arr, name), 3, True, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, "unaligned")


def _raw16(t):
    """16-bit storage bits from the monotone code t (sign bit set: non-negative value)."""
    t = np.asarray(t, dtype=np.int64)
    return np.where(t & 0x8000, t & 0x7FFF, ~t & 0xFFFF).astype(np.uint16)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("k", [8, 3])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_half_width_boundary(dt, k, renorm):
    """E = 64 rows built in the monotone code t, around the 1024 codes below each row's largest
    value that the one-row-per-thread route ranks on half-width keys: the k-th largest exactly
    1022 or 1023 codes below the top (the last kept code and the first squashed one), ties at
    that place, equal values straddling the k-th place, and rows spread over many binades."""
    rng = np.random.default_rng(11 + k)
    E, T, top = 64, 512, 0xC100                    # top: 8.0 (bf16) / 2.5 (f16)
    t = np.zeros((T, E), dtype=np.int64)
    for r in range(T):
        kind = r % 8
        row = top - 1100 - rng.integers(0, 3000, E)          # every other value well below
        perm = rng.permutation(E)
        row[perm[0]] = top
        near = perm[1:k]
        row[near] = top - rng.integers(0, 1022, len(near))
        if kind == 0:
            row[perm[k - 1]] = top - 1023                     # k-th squashed: decided again
        elif kind == 1:
            row[perm[k - 1]] = top - 1022                     # k-th keeps code 1
            row[perm[k]] = top - 1023
        elif kind == 2:
            row[perm[k - 1]] = row[perm[k]] = top - 1022      # tie across the k-th place
        elif kind == 3:
            row[perm[k - 1:k + 3]] = top - 1023               # ties among squashed codes
        elif kind == 4:
            row[perm[k - 1]] = row[perm[k]] = top - 500       # tie above the boundary
        elif kind == 5:
            row = top - rng.integers(0, 40000, E)             # many binades, both signs
            row[perm[0]] = top
        elif kind == 6:
            row[perm[1:k + 2]] = top                          # all of the top k equal
        else:
            row = top - 1022 + rng.integers(0, 1023, E)       # everything inside the window
        t[r] = row
    raw = _raw16(t)
    l = torch.from_numpy(raw.view(np.int16)).view(dt)
    assert torch.isfinite(l.float()).all()
    idx, w = moe.moe_route(l.to(DEV), k, renorm)
    torch.cuda.synchronize()
    arr, name = storage(l)
    ridx, rw = O.route(O.to_f64(arr, name), k, renorm, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, f"half-width boundary {name} k={k}")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("E,k", [(8, 3), (64, 4), (64, 8), (256, 8), (40, 5)])
def test_route_signed_zero_ties(dt, E, k):
    """+0 and -0 are equal logits: where they meet at the top-k boundary the lower id goes first,
    whatever the signs.  Rows hold six zeros of both signs at random places among negative logits
    (some of them ties at -1), and rows whose largest values are -0 only."""
    g = torch.Generator().manual_seed(E + k)
    rows = []
    for i in range(120):
        r = -1.0 - torch.randint(0, 3, (E,), generator=g).float()
        pos = torch.randperm(E, generator=g)[:min(6, E)]
        signs = torch.randint(0, 2, (len(pos),), generator=g)
        if i % 4 == 0:
            signs[:] = 1                                          # -0 only
        r[pos] = torch.where(signs == 1, torch.tensor(-0.0), torch.tensor(0.0))
        rows.append(r)
    l = torch.stack(rows).to(dt)
    assert (torch.signbit(l.float()) & (l.float() == 0)).any()
    for renorm in (True, False):
        idx, w = moe.moe_route(l.to(DEV), k, renorm)
        torch.cuda.synchronize()
        arr, name = storage(l)
        ridx, rw = O.route(O.to_f64(arr, name), k, renorm, name)
        np.testing.assert_array_equal(u32(idx), ridx)
        check_weights(w, rw, f"signed zeros {name} E={E} k={k}")


@pytest.mark.parametrize("dt,scales", [(torch.bfloat16, [300.0, -300.0, 1e6, 1e20, 1e30, -1e30]),
                                       (torch.float16, [300.0, -300.0, 3e4, -3e4])])
@pytest.mark.parametrize("E,k", [(64, 8), (40, 5), (128, 8)])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_large_logits(dt, scales, E, k, renorm):
    """Logits of large magnitude: the softmax is taken against the row maximum, so exp(x - x0)
    must not lose x0's own term.  Rows hold up to four copies of the maximum (weights 1/m) and
    values a few spacings below it (nonzero weights), at magnitudes up to 1e30 (bf16) and 3e4
    (f16)."""
    g = torch.Generator().manual_seed(E * 7 + k)
    rows = []
    for i in range(96 * len(scales)):
        s = scales[i % len(scales)]
        x0 = torch.tensor(s).to(dt).float()
        spacing = (torch.tensor(abs(s)).to(dt).float().item()) * (2.0 ** -7 if dt == torch.bfloat16
                                                                   else 2.0 ** -10)
        steps = torch.randint(1, 6, (E,), generator=g).float()
        if i % 3 == 0:
            steps = steps * 1024.0                                # far below: exp underflows
        r = torch.clamp(x0 - steps * spacing, min=-torch.finfo(dt).max).to(dt)
        m = 1 + i % 4
        pos = torch.randperm(E, generator=g)[:m]
        r[pos] = x0.to(dt)
        rows.append(r)
    l = torch.stack(rows)
    assert torch.isfinite(l.float()).all()
    idx, w = moe.moe_route(l.to(DEV), k, renorm)
    torch.cuda.synchronize()
    arr, name = storage(l)
    ridx, rw = O.route(O.to_f64(arr, name), k, renorm, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, f"large logits {name} E={E} k={k}")


@pytest.mark.parametrize("renorm", [True, False])
def test_route_sweep_full_size(renorm):
    """The routing-only workload at full size: [1 048 576, 64] bf16, N(0, 2^2), top_k = 8."""
    wl = W.WORKLOADS["route_sweep"]
    l = W.make_logits(wl, DEV)
    idx, w = moe.moe_route(l, wl.top_k, renorm)
    torch.cuda.synchronize()
    arr, name = storage(l)
    ridx, rw = O.route(O.to_f64(arr, name), wl.top_k, renorm, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, "route_sweep")


# ------------------------------------------------------------------------------------ dispatch
def _expected_dispatch(idx_np, E):
    """Oracle dispatch; slots with ids >= E go to a virtual expert E placed after all others,
    so rows of the real experts are exactly the oracle's."""
    flat = idx_np.astype(np.int64)
    bad = flat >= E
    v = np.where(bad, E, flat).astype(np.uint32)
    counts, offsets, t_of_r, r_of_s = O.dispatch(v, E + 1)
    r_of_s = r_of_s.copy()
    r_of_s.reshape(-1)[bad.reshape(-1)] = 0xFFFFFFFF
    return counts[:E], offsets[:E + 1], t_of_r[:offsets[E]], r_of_s


DISPATCH_SEEDS = {"uniform": 101, "zipf": 102, "one_expert": 103, "many_empty": 104,
                  "invalid_ids": 105, "large": 106}


@pytest.mark.parametrize("case", list(DISPATCH_SEEDS))
@pytest.mark.parametrize("T0", [1500, 300])   # 6000 slots: multi-block path; 1200: one block
def test_dispatch_matches_oracle(case, T0):
    rng = np.random.default_rng(DISPATCH_SEEDS[case] * 10 + (T0 == 300))
    T, E, k, H = T0, 64, 4, 96
    if case == "uniform":
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    elif case == "zipf":
        p = np.arange(1, E + 1) ** -1.3
        idx = np.stack([rng.choice(E, k, replace=False, p=p / p.sum()) for _ in range(T)])
    elif case == "one_expert":
        idx = np.full((T, k), 17)
    elif case == "many_empty":
        E = 1024
        idx = rng.integers(0, E, size=(T, k))
    elif case == "invalid_ids":
        idx = rng.integers(0, E + 5, size=(T, k))
        idx[0, 0] = 0xFFFFFFFF
    else:
        T, E, k, H = 40000, 256, 8, 64
        idx = rng.integers(0, E, size=(T, k))
    idx = idx.astype(np.uint32)
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    gidx = torch.from_numpy(idx.view(np.int32)).to(DEV).view(torch.uint32)
    r = moe.moe_dispatch(x.to(DEV), gidx, E)
    st = moe.moe_device_status(r["ws"])
    counts, offsets, t_of_r, r_of_s = _expected_dispatch(idx, E)
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(u32(r["row_of_slot"]), r_of_s.reshape(-1))
    n = int(offsets[E])
    np.testing.assert_array_equal(u32(r["token_of_row"])[:n], t_of_r)
    xd = r["x_d"][:n].cpu()
    assert torch.equal(xd.view(torch.int16), x[torch.from_numpy(t_of_r.astype(np.int64))].view(torch.int16))
    assert st == (8 if case == "invalid_ids" else 0)


# ------------------------------------------------------------------------------------ combine
@pytest.mark.parametrize("ydt,wdt", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32),
                                     (torch.bfloat16, torch.float32), (torch.float16, torch.float16)])
@pytest.mark.parametrize("T,k,H", [(333, 8, 256), (100, 2, 72), (17, 1, 8), (64, 40, 96), (9, 3, 13)])
def test_combine_matches_oracle(ydt, wdt, T, k, H):
    g = torch.Generator().manual_seed(T + k + H)
    E = 2 * k + 1
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).numpy().astype(np.uint32)
    _, _, _, r_of_s = O.dispatch(idx, E)
    y = torch.randn(T * k, H, generator=g).to(ydt)
    w = torch.rand(T, k, generator=g).to(wdt)
    w[min(2, T - 1), 0] = float("nan")
    ros = torch.from_numpy(r_of_s.view(np.int32)).to(DEV).view(torch.uint32)
    out = moe.moe_combine(y.to(DEV), ros, w.to(DEV))
    ref = O.combine(O.to_f64(*storage(y)), r_of_s, O.to_f64(*storage(w)))
    got = f64(out)
    assert (np.isnan(got) == np.isnan(ref)).all()
    fin = np.isfinite(ref)
    rounded = O.round_to_dtype(ref, DT_NAME[ydt])
    if ydt == torch.float32:
        np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-5, atol=1e-5)
    else:
        # FP32 sum then one rounding: within one step of the correctly rounded value, or (where
        # cancellation leaves a result in f16's subnormal range) within the FP32 accumulation
        # error bound k * 2^-23 * sum_j |w_j y_j|
        from gpu_helpers import ulp_distance
        mag = O.combine(np.abs(O.to_f64(*storage(y))), r_of_s, np.abs(O.to_f64(*storage(w))))
        ok = (ulp_distance(out, rounded) <= 1) | (np.abs(got - ref) <= k * 2.0 ** -23 * mag)
        assert ok[fin].all()


# ------------------------------------------------------------------------------------ experts
def _rand_groups(rows_per_expert, seed):
    rng = np.random.default_rng(seed)
    E = len(rows_per_expert)
    ids = np.concatenate([np.full(n, e) for e, n in enumerate(rows_per_expert)])
    rng.shuffle(ids)
    return ids.astype(np.uint32)[:, None]  # top_k = 1 layout: one slot per "token"


EXPERT_CASES = [
    # (rows per expert, H, I)
    ([300, 0, 257, 143], 256, 384),
    ([129, 1, 0, 77, 200], 200, 136),          # K tail (200 = 3*64 + 8), N tails (136, 200)
    ([1000], 128, 256),                       # one expert, 8 m-tiles: a full raster group
    ([37] * 16, 512, 1024),
    ([0, 0, 5, 0], 64, 64),
    ([2100, 3, 250, 0, 0, 640], 384, 1536),    # > 16 m-tiles: two raster groups
    # CTA-pair path (>= 128 rows per expert on average) with every kind of partial m-tile:
    # 1..255 rows (operand-swapped tiles, N = rows rounded up to 16), exactly 256, 257; K tail
    # of the down GEMM (I = 136) and ragged output columns (I = 136, H = 200)
    ([1, 15, 16, 17, 31, 33, 129, 255, 256, 257, 600, 0], 200, 136),
    ([5000, 40, 3, 700, 1], 512, 1024),
]


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("case", range(len(EXPERT_CASES)))
def test_experts_match_oracle(dt, case):
    counts, H, I = EXPERT_CASES[case]
    E = len(counts)
    ids = _rand_groups(counts, seed=case)
    cnt, offsets, t_of_r, _ = O.dispatch(ids, E)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(100 + case)
    x_d = torch.randn(rows, H, generator=g).to(dt)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dt)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    y = moe.moe_experts_forward_dispatched(x_d.to(DEV), off_t, gate.to(DEV), up.to(DEV),
                                           down.to(DEV))
    torch.cuda.synchronize()
    name = DT_NAME[dt]
    ref = O.experts(O.to_f64(*storage(x_d)), offsets, storage(gate)[0], storage(up)[0],
                    storage(down)[0], name)
    err = rel_max_err(f64(y), ref)
    assert err <= layer_tol(dt), f"rel max err {err}"


# K of at least 64 slices of 64 (H >= 4096 for gate/up, I >= 4096 for down) puts the CTA-pair
# GEMMs on dynamic tile claims: each pair's first tile is its index, later ones come from a
# global counter.  Few tiles (most pairs get none), one tile per pair, and more tiles than
# co-resident pairs (claims past the first round).
DYNAMIC_CASES = [
    ([300, 1, 257, 0, 600], 4096, 128),          # gate/up: 8 tiles
    ([700, 300, 2, 0], 256, 4096),                # down: 6 tiles, K = 4096
    ([1500, 3, 0, 900, 129, 600], 4096, 1024),    # gate/up: 15 m-tiles x 8 n-tiles = 120 tiles
]


def _tile_rows(offsets, seed, per_tile=3):
    """Rows of every 128-row m-tile of every expert: each tile's first and last row and a few
    seeded others, so that a wrong tile order or a tile computed twice or not at all shows."""
    rng = np.random.default_rng(seed)
    out = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for m in range(lo, hi, 128):
            end = min(m + 128, hi)
            out += [m, end - 1] + list(rng.integers(m, end, per_tile))
    return np.unique(np.array(out, dtype=np.int64))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", range(len(DYNAMIC_CASES)))
def test_experts_dynamic_tile_claims(dt, case):
    counts, H, I = DYNAMIC_CASES[case]
    E = len(counts)
    _, offsets, _, _ = O.dispatch(_rand_groups(counts, seed=40 + case), E)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(400 + case)
    x_d = torch.randn(rows, H, generator=g).to(dt)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dt)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    y = moe.moe_experts_forward_dispatched(x_d.to(DEV), off_t, gate.to(DEV), up.to(DEV),
                                           down.to(DEV))
    torch.cuda.synchronize()
    # rows are independent: the oracle runs on the sampled rows with their experts' offsets
    sel = _tile_rows(offsets, seed=case)
    sub_off = np.searchsorted(sel, offsets, side="left")
    name = DT_NAME[dt]
    ref = O.experts(O.to_f64(*storage(x_d))[sel], sub_off, storage(gate)[0], storage(up)[0],
                    storage(down)[0], name)
    got = f64(y)[sel]
    assert np.isfinite(got).all()
    err = rel_max_err(got, ref)
    assert err <= layer_tol(dt), f"rel max err {err}"


# ------------------------------------------------------------------------------------ full layer
def _stratified_tokens(offsets, token_of_row, T, n_total, seed):
    """A seeded token sample that puts at least one row in every 128-row m-tile of every expert's
    dispatched group (a random row of each, plus each group's first and last row, so every
    ragged tail tile is reached), topped up with random tokens to n_total."""
    rng = np.random.default_rng(seed)
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            rows += [lo, hi - 1]
            rows += [int(rng.integers(r0, min(r0 + 128, hi))) for r0 in range(lo, hi, 128)]
    tok = set(int(t) for t in token_of_row[np.array(rows, dtype=np.int64)])
    rest = np.setdiff1d(np.arange(T), np.fromiter(tok, dtype=np.int64))
    extra = max(0, n_total - len(tok))
    tok |= set(int(t) for t in rng.choice(rest, min(extra, len(rest)), replace=False))
    return np.array(sorted(tok), dtype=np.int64)


def _run_layer(wl, sample=None, seed=0):
    tok = None
    dev_inputs = W.make_layer_inputs(wl, DEV if sample else "cpu")
    g = {k: v.to(DEV) for k, v in dev_inputs.items()}
    out = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], wl.top_k,
                          wl.renormalize)
    out2 = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], wl.top_k,
                           wl.renormalize)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8)), "not run-to-run identical"
    # stage outputs through the staged API, for bit-exact route / dispatch checks
    idx, w = moe.moe_route(g["logits"], wl.top_k, wl.renormalize)
    d = moe.moe_dispatch(g["x"], idx, wl.E)
    torch.cuda.synchronize()
    larr, lname = storage(dev_inputs["logits"])
    ridx, rw = O.route(O.to_f64(larr, lname), wl.top_k, wl.renormalize, lname)
    np.testing.assert_array_equal(u32(idx), ridx)
    check_weights(w, rw, wl.name)
    counts, offsets, t_of_r, r_of_s = O.dispatch(ridx, wl.E)
    np.testing.assert_array_equal(d["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(u32(d["row_of_slot"]), r_of_s)
    np.testing.assert_array_equal(u32(d["token_of_row"]), t_of_r)
    # moe_forward runs the same kernels as the staged calls: bit for bit the same output
    y = moe.moe_experts_forward_dispatched(d["x_d"], d["offsets"], g["gate"], g["up"], g["down"])
    out_st = moe.moe_combine(y, d["row_of_slot"], w)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), out_st.view(torch.uint8)), \
        f"{wl.name}: moe_forward differs from the staged calls"
    del y, out_st
    wname = DT_NAME[g["x"].dtype]
    if sample == "stratified":
        tok = _stratified_tokens(offsets, t_of_r, wl.T, 2048, seed)
        print(f"{wl.name}: oracle sample of {len(tok)} tokens covering every (expert, 128-row "
              f"m-tile) of {int((np.diff(offsets) > 0).sum())} routed experts")
        sample = len(tok)
    if sample is None:
        st = {k: storage(v) for k, v in dev_inputs.items()}
        ref = O.forward(*st["x"], *st["logits"], st["gate"][0], st["up"][0], st["down"][0],
                        wname, wl.top_k, wl.renormalize)["out_unrounded"]
        got = f64(out)
    else:
        if tok is None:
            tok = np.sort(np.random.default_rng(seed).choice(wl.T, sample, replace=False))
        xs = O.to_f64(storage(g["x"][torch.from_numpy(tok).to(DEV)])[0], wname)
        ref = O.forward_rows(xs, ridx[tok], rw[tok],
                             oracle_expert_weights(g["gate"], g["up"], g["down"], wname))
        got = f64(out)[tok]
    err = rel_max_err(got, ref)
    assert err <= layer_tol(g["x"].dtype), f"{wl.name}: rel max err {err}"
    return err


def test_layer_tiny_f32():
    _run_layer(W.WORKLOADS["tiny_f32"])


def test_layer_small_bf16_full_oracle():
    _run_layer(W.Workload("small_bf16", T=300, H=256, I=512, E=16, top_k=4, renormalize=False,
                          dtype="bf16", seed=21, zipf_s=1.0))


@pytest.mark.parametrize("wl", [
    # CTA-pair experts (at least 128 rows an expert on average) at sizes the oracle runs whole:
    # even experts; ragged experts with idle ones, H = 200 (a K tail) and I = 192 (an N tail);
    # f16 with top_k = 3
    W.Workload("pair_even", T=700, H=256, I=256, E=4, top_k=2, renormalize=True, dtype="bf16",
               seed=41),
    W.Workload("pair_ragged", T=1100, H=200, I=192, E=16, top_k=2, renormalize=False,
               dtype="bf16", seed=42, zipf_s=1.3),
    W.Workload("pair_f16", T=900, H=320, I=384, E=8, top_k=3, renormalize=True, dtype="f16",
               seed=43, zipf_s=0.7),
], ids=lambda w: w.name)
def test_layer_pair_full_oracle(wl):
    _run_layer(wl)


def test_layer_decode_full():
    _run_layer(W.WORKLOADS["decode"])


def test_layer_prefill_sampled():
    """The prefill layer at full size, checked on >= 2048 tokens that cover every m-tile."""
    _run_layer(W.WORKLOADS["prefill"], sample="stratified", seed=4)


def test_layer_skewed_sampled():
    """The skewed layer at full size, checked on >= 2048 tokens that cover every (expert, m-tile),
    including every ragged tail tile and the last tiles of the heaviest expert."""
    _run_layer(W.WORKLOADS["skewed"], sample="stratified", seed=5)


# ------------------------------------------------------------------------------------ edges
def test_empty_batch_and_status():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    l = torch.empty(0, 8, dtype=torch.bfloat16, device=DEV)
    gate = torch.zeros(8, 64, 64, dtype=torch.bfloat16, device=DEV)
    out = moe.moe_forward(x, l, gate, gate, gate, 2)
    assert out.shape == (0, 64)
    idx, w = moe.moe_route(l, 2)
    assert idx.shape == (0, 2)


def test_single_expert_top1_is_plain_mlp():
    wl = W.Workload("e1", T=200, H=128, I=256, E=1, top_k=1, renormalize=True, dtype="bf16", seed=9)
    _run_layer(wl)


def test_topk_equals_E():
    wl = W.Workload("k_eq_e", T=150, H=64, I=128, E=4, top_k=4, renormalize=True, dtype="bf16",
                    seed=10)
    _run_layer(wl)
