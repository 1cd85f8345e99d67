"""Plain fp64 CPU oracle of the local MoE forward: route -> dispatch -> SwiGLU experts -> combine.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import, call or execute this module.  It shares no code with
the CUDA path (no kernels, headers, helpers, tables or constants) and imports nothing from it.

What it computes follows the ruDNN user guide (docs.rs, ruDNN 0.1.72, docs/de/README.md):

* §3 "MoE-Workflow": logits -> softmax/top-k -> compact dispatch -> SwiGLU experts -> weighted
  combine, all local.
* §4 "Routing-Vertrag": logits [T, E] in F32/F16/BF16; 1 <= top_k <= E; softmax over *all*
  experts before the top-k; ties favour the lower expert id; with renormalisation the selected
  weights are renormalised and *then* cast to the logits dtype; rows holding a NaN, a +inf or only
  -inf keep NaN weights (no uniform fallback); indices u32 and weights both [T, top_k].
* §5 "Expertengewichte und Verteilung": x [T, H]; gate, up [E, I, H]; down [E, H, I]; bias-free;
  no token is dropped for a capacity limit; a saved map restores token order.
* §6 "MoE aufrufen": forward(input, logits, options) -> output [T, H]; combine uses the dispatch
  map and the routing weights.

Every value is computed in float64 from the exact values of the stored inputs and rounded once,
round-to-nearest-even, to the output dtype.  The page says FP32 for the softmax; float64 is
stricter, and the comparison tolerances absorb the difference.

Readings taken where the page is silent (each is repeated at the function that applies it):
  R1 selection key: rank experts by the logit itself (exp is increasing, so this is the ranking
     of the exact softmax), equal logits lower id first;
  R2 poisoned rows select experts 0..k-1 and carry NaN weights, so no token is dropped;
  R3 finite rows holding some -inf give those experts p = 0; they are selectable once the
     finite entries are used up;
  R4 the top-k slots are ordered by descending weight, equal weights lower id first;
  R5 rows of one expert are kept in ascending flat slot order s = t*top_k + j (stable);
  R6 SwiGLU: a = silu(x gate^T) * (x up^T), y = a down^T, silu(z) = z / (1 + exp(-z));
  R7 routing weights are applied in the combine, after the down projection, summed over the
     slots j = 0..k-1 of a token in slot order; the output takes the input dtype.

Group-limited sigmoid routing follows §10 "Gruppenbeschränktes Sigmoid-MoE-Routing" of the same
page: sigmoid scores, an optional FP32 correction bias that affects the selection only, groups
scored by their maximum or the sum of their two largest corrected scores, the best
`selected_groups` groups, then the top_k experts inside them; weights are the uncorrected sigmoid
values, optionally renormalised, times `scale`; ties prefer smaller ids.  Readings:
  S1 the selection (sigmoid, correction, group scores, ranking) is decided in float64 on both
     sides of the comparison, so CPU and GPU take the same decision;
  S2 slots are ordered by descending corrected score, equal scores lower id first;
  S3 rows whose corrected scores hold a NaN keep NaN weights and select ids 0..k-1;
  S4 weights are rounded once to the logits dtype after renormalisation and scaling.

Router weights of a fixed selection and their gradient follow §12 "MoE-Training erster Ordnung":
FP32 weights [T, k] for given indices (softmax over all experts, or sigmoid), optional
renormalisation over the k slots, then `scale`; repeated indices gather; an invalid index makes
the whole row NaN; the gradient is with respect to the logits of the continuous weights only.

The backward chain of the same section (combine_backward -> expert backward ->
dispatch_backward, then the router backward above) is the chain rule of the forward written out:
  combine:  dexpert[row(t, j)] = w[t, j] * dout[t];  dweights[t, j] = <dout[t], y[row(t, j)]>
  experts:  da = dy down_e;  du = da * silu(g);  dg = da * u * silu'(g),
            silu'(g) = s (1 + g (1 - s)), s = sigmoid(g);  dx = dg gate_e + du up_e;
            ddown_e = dy^T a;  dgate_e = dg^T x;  dup_e = du^T x
  dispatch: dx[t] = sum_j dinput[row(t, j)]  (the routing weights are not applied again)

Pins (tests/test_oracle_pins.py) tie each function to something other than itself: closed forms,
library routines (torch float64 softmax and silu, numpy's float32 cast), brute force on tiny
inputs, and invariants.  Parity unpinned: R1 for two *different* logits whose FP32 softmax values
round to the same number (the page fixes no rule there beyond "ties to the lower id").
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "DTYPES", "to_f64", "round_to_dtype", "encode", "poisoned_rows", "softmax", "select_topk",
    "route", "dispatch", "gather", "silu", "swiglu", "experts", "combine", "forward",
    "forward_rows", "sigmoid", "route_sigmoid_grouped", "forward_sigmoid_grouped",
    "selected_router_weights", "selected_router_backward", "combine_backward",
    "experts_backward", "dispatch_backward",
]

DTYPES = ("f32", "f16", "bf16")

# (significand bits including the leading one, minimum normal exponent, maximum exponent)
_FORMAT = {"f32": (24, -126, 127), "f16": (11, -14, 15), "bf16": (8, -126, 127)}


# --------------------------------------------------------------------------------------------
# storage <-> exact values
# --------------------------------------------------------------------------------------------
def to_f64(stored, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements.

    bf16 arrives as raw uint16 bit patterns: a bf16 is the upper 16 bits of an IEEE binary32, so
    shifting the pattern into the high half of a 32-bit word gives the same number as a float32.
    """
    if dtype == "bf16":
        bits = np.asarray(stored, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(stored, dtype=np.float16).astype(np.float64)
    if dtype == "f32":
        return np.asarray(stored, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def round_to_dtype(x, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest value of ``dtype`` (ties to even), returned as float64.

    A binary format with p significand bits has spacing 2^(e - p + 1) between neighbours whose
    leading bit is 2^e; below the smallest normal exponent the spacing stays at the subnormal
    step.  Dividing by that spacing is exact in float64, ``np.rint`` rounds half to even, and a
    result past the largest finite value overflows to infinity.
    """
    p, emin, emax = _FORMAT[dtype]
    x = np.array(x, dtype=np.float64, copy=True)
    sel = np.isfinite(x) & (x != 0.0)
    v = x[sel]
    _, e = np.frexp(v)                      # v = m * 2^e with 0.5 <= |m| < 1
    lead = np.maximum(e - 1, emin)          # exponent of the leading bit, clamped at subnormals
    step = np.ldexp(1.0, lead - (p - 1))
    r = np.rint(v / step) * step
    max_finite = (2.0 - 2.0 ** (1 - p)) * 2.0 ** emax
    over = np.abs(r) > max_finite
    r[over] = np.copysign(np.inf, r[over])
    x[sel] = r
    return x


def encode(x, dtype: str) -> np.ndarray:
    """Storage form (bf16: uint16 bit patterns) of float64 values after rounding to ``dtype``."""
    r = round_to_dtype(x, dtype)
    if dtype == "bf16":
        return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    if dtype == "f16":
        return r.astype(np.float16)
    return r.astype(np.float32)


# --------------------------------------------------------------------------------------------
# route (§4 "Routing-Vertrag")
# --------------------------------------------------------------------------------------------
def poisoned_rows(logits: np.ndarray) -> np.ndarray:
    """Rows that keep NaN weights: any NaN, any +inf, or every entry -inf (§4)."""
    return (np.isnan(logits).any(axis=1) | np.isposinf(logits).any(axis=1)
            | np.isneginf(logits).all(axis=1))


def softmax(logits: np.ndarray) -> np.ndarray:
    """p[t, e] = exp(l[t, e] - m_t) / sum_e' exp(l[t, e'] - m_t), m_t the row max, over all experts.

    Poisoned rows are all NaN.  -inf entries of other rows get p = 0 (reading R3).
    """
    bad = poisoned_rows(logits)
    safe = np.where(bad[:, None], 0.0, logits)
    m = safe.max(axis=1, keepdims=True)
    z = np.exp(safe - m)
    p = z / z.sum(axis=1, keepdims=True)
    p[bad] = np.nan
    return p


def select_topk(logits: np.ndarray, top_k: int) -> np.ndarray:
    """Indices [T, top_k] (uint32) of the top_k experts of each row.

    Readings R1/R4: order by descending logit, equal logits lower id first (a stable sort of the
    negated logits keeps ascending ids among equals).  R2: poisoned rows take 0..top_k-1.
    """
    T, E = logits.shape
    assert 1 <= top_k <= E
    bad = poisoned_rows(logits)
    safe = np.where(bad[:, None], 0.0, logits)
    order = np.argsort(-safe, axis=1, kind="stable")
    idx = order[:, :top_k].copy()
    idx[bad] = np.arange(top_k)
    return idx.astype(np.uint32)


def route(logits: np.ndarray, top_k: int, renormalize: bool, out_dtype: str):
    """route(logits, RoutingOptions{top_k, renormalize}) -> (indices u32 [T,k], weights [T,k]).

    Weights are the softmax values of the selected experts; with renormalisation they are divided
    by their sum over the selection; only then are they rounded to ``out_dtype`` (the logits
    dtype).  Returned weights are float64 holding exactly representable ``out_dtype`` values.
    """
    p = softmax(logits)
    idx = select_topk(logits, top_k)
    w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    if renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return idx, round_to_dtype(w, out_dtype)


# --------------------------------------------------------------------------------------------
# dispatch (§5 "Expertengewichte und Verteilung")
# --------------------------------------------------------------------------------------------
def dispatch(idx: np.ndarray, E: int):
    """Capacity-free dispatch of the T*k routed slots, grouped by expert.

    Slot s = t*k + j carries expert idx[t, j].  Returns
      counts [E]          rows per expert (no slot is dropped: sum = T*k),
      offsets [E+1]       exclusive prefix sum of counts,
      token_of_row [T*k]  token feeding dispatched row r,
      row_of_slot [T*k]   dispatched row holding slot s (the saved map that restores order).
    Reading R5: inside one expert the rows keep ascending slot order (a stable sort by expert).
    """
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < E)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    slot_of_row = np.argsort(flat, kind="stable")
    row_of_slot = np.empty_like(slot_of_row)
    row_of_slot[slot_of_row] = np.arange(flat.size)
    token_of_row = slot_of_row // k
    return counts, offsets, token_of_row.astype(np.uint32), row_of_slot.astype(np.uint32)


def gather(x: np.ndarray, token_of_row: np.ndarray) -> np.ndarray:
    """Dispatched input rows: x_d[r] = x[token_of_row[r]]."""
    return x[token_of_row.astype(np.int64)]


# --------------------------------------------------------------------------------------------
# experts (§5, §6: bias-free SwiGLU, gate/up [E,I,H], down [E,H,I])
# --------------------------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(x_rows, gate_e, up_e, down_e) -> np.ndarray:
    """Reading R6: y = (silu(x gate_e^T) * (x up_e^T)) down_e^T for rows x [n, H]."""
    g = x_rows @ gate_e.T
    u = x_rows @ up_e.T
    return (silu(g) * u) @ down_e.T


def experts(x_d: np.ndarray, offsets, gate, up, down, wdtype: str) -> np.ndarray:
    """forward_dispatched: expert e transforms rows offsets[e]:offsets[e+1] of x_d.

    ``x_d`` is float64; gate/up/down are stored arrays of dtype ``wdtype``, converted to float64
    one expert at a time.  Returns float64 [T*k, H], unrounded.
    """
    E = len(offsets) - 1
    y = np.zeros((x_d.shape[0], down.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = swiglu(x_d[lo:hi], to_f64(gate[e], wdtype), to_f64(up[e], wdtype),
                              to_f64(down[e], wdtype))
    return y


# --------------------------------------------------------------------------------------------
# combine (§3, §6)
# --------------------------------------------------------------------------------------------
def combine(y: np.ndarray, row_of_slot: np.ndarray, w: np.ndarray) -> np.ndarray:
    """out[t] = sum_{j=0..k-1} w[t, j] * y[row_of_slot[t*k + j]], summed in slot order (R7)."""
    T, k = w.shape
    rs = row_of_slot.astype(np.int64).reshape(T, k)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y[rs[:, j]]
    return out


# --------------------------------------------------------------------------------------------
# full forward (§6 "MoE aufrufen")
# --------------------------------------------------------------------------------------------
def forward(x, x_dtype, logits, logits_dtype, gate, up, down, w_dtype, top_k, renormalize):
    """SwiGluExperts::forward(input, logits, options): route, dispatch, experts, combine.

    Inputs are stored arrays with their dtype names.  Returns a dict with every intermediate;
    ``out`` is rounded to the input dtype.
    """
    l64 = to_f64(logits, logits_dtype)
    x64 = to_f64(x, x_dtype)
    E = l64.shape[1]
    idx, w = route(l64, top_k, renormalize, logits_dtype)
    counts, offsets, token_of_row, row_of_slot = dispatch(idx, E)
    x_d = gather(x64, token_of_row)
    y = experts(x_d, offsets, gate, up, down, w_dtype)
    out = combine(y, row_of_slot, w)
    return {"idx": idx, "w": w, "counts": counts, "offsets": offsets,
            "token_of_row": token_of_row, "row_of_slot": row_of_slot, "x_d": x_d, "y": y,
            "out_unrounded": out, "out": round_to_dtype(out, x_dtype)}


def forward_rows(x_rows: np.ndarray, idx_rows: np.ndarray, w_rows: np.ndarray, expert_weights):
    """Output rows of selected tokens only (each token's output depends on its own row alone).

    x_rows [n, H] float64, idx_rows [n, k], w_rows [n, k] float64, and
    ``expert_weights(e) -> (gate_e, up_e, down_e)`` in float64.  The same dispatch / experts /
    combine steps restricted to n tokens; returns float64 [n, H], unrounded.
    """
    n, k = idx_rows.shape
    counts, offsets, token_of_row, row_of_slot = dispatch(idx_rows, int(idx_rows.max()) + 1)
    x_d = gather(x_rows, token_of_row)
    y = np.zeros((x_d.shape[0], x_rows.shape[1]), dtype=np.float64)
    for e in range(len(counts)):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = swiglu(x_d[lo:hi], *expert_weights(e))
    return combine(y, row_of_slot, w_rows)


# --------------------------------------------------------------------------------------------
# group-limited sigmoid routing (§10 "Gruppenbeschränktes Sigmoid-MoE-Routing")
# --------------------------------------------------------------------------------------------
def sigmoid(z: np.ndarray) -> np.ndarray:
    """sigmoid(z) = 1 / (1 + exp(-z)); exact limits 0 and 1 at -inf and +inf."""
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def route_sigmoid_grouped(logits: np.ndarray, bias, top_k: int, groups: int, selected_groups: int,
                          group_top_two: bool, renormalize: bool, scale: float, out_dtype: str):
    """route_sigmoid_grouped(logits, bias, GroupRoutingOptions) -> (indices u32 [T,k], weights).

    s = sigmoid(l); c = s + bias (bias: FP32 [E] or None, selection only).  Experts form `groups`
    contiguous groups of E / groups; a group scores max(c) over its experts, or the sum of its two
    largest c with group_top_two.  The `selected_groups` best groups are kept (ties: lower group
    id), then the top_k experts inside them by c (ties: lower id).  Weights are s of the chosen
    experts, divided by their sum when renormalising, times scale, rounded to `out_dtype`.
    """
    T, E = logits.shape
    gs = E // groups
    assert gs * groups == E and 1 <= selected_groups <= groups
    assert 1 <= top_k <= selected_groups * gs and (gs >= 2 or not group_top_two)
    s = sigmoid(logits)
    c = s + (0.0 if bias is None else np.asarray(bias, dtype=np.float64)[None, :])
    bad = np.isnan(c).any(axis=1)
    c = np.where(bad[:, None], 0.0, c)
    srt = -np.sort(-c.reshape(T, groups, gs), axis=2)
    gscore = srt[:, :, 0] + srt[:, :, 1] if group_top_two else srt[:, :, 0]
    gsel = np.argsort(-gscore, axis=1, kind="stable")[:, :selected_groups]
    allowed = np.zeros((T, groups), dtype=bool)
    np.put_along_axis(allowed, gsel, True, axis=1)
    allowed = np.repeat(allowed, gs, axis=1)
    # rank: allowed experts first, then by corrected score descending, then by id ascending
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -c, ~allowed), axis=1)
    idx = order[:, :top_k].copy()
    idx[bad] = np.arange(top_k)
    w = np.take_along_axis(s, idx, axis=1)
    if renormalize:
        with np.errstate(invalid="ignore", divide="ignore"):
            w = w / w.sum(axis=1, keepdims=True)
    w = w * scale
    w[bad] = np.nan
    return idx.astype(np.uint32), round_to_dtype(w, out_dtype)


def forward_sigmoid_grouped(x, x_dtype, logits, logits_dtype, bias, gate, up, down, w_dtype,
                            top_k, groups, selected_groups, group_top_two, renormalize, scale):
    """SwiGluExperts::forward_sigmoid_grouped: sigmoid routing, then dispatch, experts, combine."""
    l64 = to_f64(logits, logits_dtype)
    x64 = to_f64(x, x_dtype)
    E = l64.shape[1]
    b64 = None if bias is None else to_f64(bias, "f32")
    idx, w = route_sigmoid_grouped(l64, b64, top_k, groups, selected_groups, group_top_two,
                                   renormalize, scale, logits_dtype)
    counts, offsets, token_of_row, row_of_slot = dispatch(idx, E)
    y = experts(gather(x64, token_of_row), offsets, gate, up, down, w_dtype)
    out = combine(y, row_of_slot, w)
    return {"idx": idx, "w": w, "counts": counts, "offsets": offsets,
            "out_unrounded": out, "out": round_to_dtype(out, x_dtype)}


# --------------------------------------------------------------------------------------------
# router weights of a fixed selection and their backward (§12 "MoE-Training erster Ordnung")
# --------------------------------------------------------------------------------------------
def _selection_scores(logits, scoring):
    if scoring == "softmax":
        return softmax(logits)
    if scoring == "sigmoid":
        return sigmoid(logits)
    raise ValueError(scoring)


def selected_router_weights(logits: np.ndarray, idx: np.ndarray, scoring: str, renormalize: bool,
                            scale: float) -> np.ndarray:
    """w[t, j] = scale * p[t, idx[t, j]] (divided by sum_j p[t, idx[t, j]] when renormalising),
    p = softmax over all experts or sigmoid.  Repeated indices gather the same p; a row with an
    index outside [0, E) is all NaN.  float64 [T, k]; the page returns FP32."""
    T, E = logits.shape
    idx = np.asarray(idx).astype(np.int64)
    bad = ((idx < 0) | (idx >= E)).any(axis=1)
    p = _selection_scores(logits, scoring)
    w = np.take_along_axis(p, np.where(idx < 0, 0, np.minimum(idx, E - 1)), axis=1)
    if renormalize:
        with np.errstate(invalid="ignore", divide="ignore"):
            w = w / w.sum(axis=1, keepdims=True)
    w = w * scale
    w[bad] = np.nan
    return w


def selected_router_backward(logits: np.ndarray, idx: np.ndarray, grad_w: np.ndarray,
                             scoring: str, renormalize: bool, scale: float) -> np.ndarray:
    """dL/dlogits [T, E] of selected_router_weights given dL/dw [T, k] (chain rule, float64).

    With q_j the selected score (p or s) of slot j, G_e = sum over slots j with idx j = e of g_j,
    and for renormalisation Z = sum_j q_j:
      softmax, plain:  dl_e = scale * p_e * (G_e - sum_j g_j q_j)
      softmax, renorm: the weights are a softmax over the k selected logits, r_j = q_j / Z:
                       dl_e = scale * (sum_{j: idx_j = e} g_j r_j - n_e r_e * sum_j g_j r_j)
                       where n_e counts the slots holding e and r_e = p_e / Z
      sigmoid, plain:  dl_e = scale * s_e (1 - s_e) * G_e
      sigmoid, renorm: dl_e = scale * s_e (1 - s_e) / Z * (G_e - n_e * sum_j g_j q_j / Z)
    Rows with an invalid index are all NaN.
    """
    T, E = logits.shape
    idx = np.asarray(idx).astype(np.int64)
    bad = ((idx < 0) | (idx >= E)).any(axis=1)
    sidx = np.where(idx < 0, 0, np.minimum(idx, E - 1))
    g = np.asarray(grad_w, dtype=np.float64)
    p = _selection_scores(logits, scoring)
    q = np.take_along_axis(p, sidx, axis=1)
    rows = np.arange(T)[:, None]
    G = np.zeros((T, E))
    np.add.at(G, (np.broadcast_to(rows, sidx.shape), sidx), g)
    n = np.zeros((T, E))
    np.add.at(n, (np.broadcast_to(rows, sidx.shape), sidx), 1.0)
    with np.errstate(invalid="ignore", divide="ignore"):
        if scoring == "softmax" and not renormalize:
            out = p * (G - (g * q).sum(axis=1, keepdims=True))
        elif scoring == "softmax":
            Z = q.sum(axis=1, keepdims=True)
            r = q / Z
            Gr = np.zeros((T, E))
            np.add.at(Gr, (np.broadcast_to(rows, sidx.shape), sidx), g * r)
            out = Gr - n * (p / Z) * (g * r).sum(axis=1, keepdims=True)
        elif not renormalize:
            out = p * (1.0 - p) * G
        else:
            Z = q.sum(axis=1, keepdims=True)
            out = p * (1.0 - p) / Z * (G - n * (g * q).sum(axis=1, keepdims=True) / Z)
    out = out * scale
    out[bad] = np.nan
    return out


# --------------------------------------------------------------------------------------------
# backward chain (§12 "MoE-Training erster Ordnung", steps 1-3)
# --------------------------------------------------------------------------------------------
def combine_backward(y: np.ndarray, row_of_slot: np.ndarray, w: np.ndarray, dout: np.ndarray):
    """dexpert [T*k, H] and dweights [T, k] of out[t] = sum_j w[t, j] y[row(t, j)]."""
    T, k = w.shape
    rs = row_of_slot.astype(np.int64).reshape(T, k)
    dexpert = np.zeros_like(y, dtype=np.float64)
    dweights = np.zeros((T, k))
    for j in range(k):
        dexpert[rs[:, j]] = w[:, j:j + 1] * dout
        dweights[:, j] = (dout * y[rs[:, j]]).sum(axis=1)
    return dexpert, dweights


def experts_backward(x_d: np.ndarray, offsets, gate, up, down, wdtype: str, dy: np.ndarray):
    """Gradients of forward_dispatched for dL/dy: (dinput [rows, H], dgate [E, I, H],
    dup [E, I, H], ddown [E, H, I]), all float64, recomputing g = x gate^T and u = x up^T."""
    E = len(offsets) - 1
    I, H = gate.shape[1], gate.shape[2]
    dx = np.zeros_like(x_d, dtype=np.float64)
    dgate = np.zeros((E, I, H))
    dup = np.zeros((E, I, H))
    ddown = np.zeros((E, H, I))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi <= lo:
            continue
        ge, ue, de = (to_f64(wt[e], wdtype) for wt in (gate, up, down))
        x = x_d[lo:hi]
        g = x @ ge.T
        u = x @ ue.T
        with np.errstate(over="ignore"):
            s = 1.0 / (1.0 + np.exp(-g))
        act = g * s
        a = act * u
        da = dy[lo:hi] @ de
        du = da * act
        dg = da * u * (s * (1.0 + g * (1.0 - s)))
        dx[lo:hi] = dg @ ge + du @ ue
        ddown[e] = dy[lo:hi].T @ a
        dgate[e] = dg.T @ x
        dup[e] = du.T @ x
    return dx, dgate, dup, ddown


def dispatch_backward(dinput: np.ndarray, row_of_slot: np.ndarray, T: int, k: int):
    """dx [T, H] = sum over the k slots of each token of its dispatched rows' gradients."""
    rs = row_of_slot.astype(np.int64).reshape(T, k)
    dx = np.zeros((T, dinput.shape[1]))
    for j in range(k):
        dx += dinput[rs[:, j]]
    return dx
