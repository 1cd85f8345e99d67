"""GPU parity of the MoE backward chain (ruDNN user guide §12) against the fp64 oracle:
combine_backward, the expert backward (dinput, FP32 dgate / dup / ddown), dispatch_backward and
the full chain with the router backward.  Bounds (max |d| / max |ref|): f32 layers 1e-4
everywhere (FP32 on CUDA cores); 16-bit layers with I % 64 == 0 run on tensor cores, whose
operands (dy, dg, du, a) are rounded to the layer dtype as the forward rounds a, so every output
gets the 16-bit layer tolerance 2e-2; other 16-bit shapes (CUDA cores, FP32 operands) keep 1e-4
for the FP32 weight gradients."""
import numpy as np
import pytest
import torch

import oracle as O
import mixture_experts_routing_moe_gb300 as moe
from mixture_experts_routing_moe_gb300 import workloads as W
from gpu_helpers import DT_NAME, f64, layer_tol, rel_max_err, storage, u32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _groups(counts, seed):
    rng = np.random.default_rng(seed)
    ids = np.concatenate([np.full(n, e) for e, n in enumerate(counts)])
    rng.shuffle(ids)
    return ids.astype(np.uint32)[:, None]


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("counts,H,I", [([70, 0, 129, 5], 96, 160), ([200], 64, 72),
                                        ([33] * 6, 128, 256), ([0, 0, 3, 0], 40, 24),
                                        ([300, 0, 129, 77], 256, 384), ([1000], 128, 192),
                                        ([0, 40, 0, 513, 2], 200, 128),
                                        # >= 128 rows per expert: dA, g/u and dinput on CTA
                                        # pairs (half tiles of 1, 129 and 44 rows, ragged
                                        # output columns, dinput's K crossing from gate to up)
                                        ([600, 0, 1, 257, 129, 256], 192, 256),
                                        ([2000, 300], 512, 320),
                                        # K of 64 slices: dA and g/u (H = 4096), dinput
                                        # (2 I = 4096) on dynamic tile claims
                                        ([400, 0, 129, 300], 4096, 128),
                                        ([300, 200, 1], 128, 2048)])
def test_experts_backward_matches_oracle(dt, counts, H, I):
    E = len(counts)
    _, offsets, _, _ = O.dispatch(_groups(counts, sum(counts)), E)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(rows + H + I)
    x_d = torch.randn(rows, H, generator=g).to(dt)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dt)
    dy = torch.randn(rows, H, generator=g).to(dt)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    dx, dg, du, dd = moe.moe_experts_backward(x_d.to(DEV), off_t, gate.to(DEV), up.to(DEV),
                                              down.to(DEV), dy.to(DEV))
    torch.cuda.synchronize()
    name = DT_NAME[dt]
    rdx, rdg, rdu, rdd = O.experts_backward(O.to_f64(*storage(x_d)), offsets, storage(gate)[0],
                                            storage(up)[0], storage(down)[0], name,
                                            O.to_f64(*storage(dy)))
    assert rel_max_err(f64(dx), rdx) <= layer_tol(dt)
    wtol = layer_tol(dt) if (dt != torch.float32 and I % 64 == 0) else 1e-4
    for got, ref in ((dg, rdg), (du, rdu), (dd, rdd)):
        assert rel_max_err(f64(got), ref) <= wtol


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,k,H,E", [(150, 3, 96, 7),     # 16-byte rows, k <= 8: vector kernels
                                     (60, 12, 40, 16),    # k > 8: scalar combine backward
                                     (90, 5, 41, 9)])     # 82 / 164-byte rows: scalar kernels
def test_combine_and_dispatch_backward_match_oracle(ydt, T, k, H, E):
    gen = torch.Generator().manual_seed(5)
    idx = torch.stack([torch.randperm(E, generator=gen)[:k] for _ in range(T)]).numpy().astype(np.uint32)
    _, _, _, ros = O.dispatch(idx, E)
    y = torch.randn(T * k, H, generator=gen).to(ydt)
    w = torch.rand(T, k, generator=gen).to(ydt)
    dout = torch.randn(T, H, generator=gen).to(ydt)
    ros_t = torch.from_numpy(ros.view(np.int32)).to(DEV).view(torch.uint32)
    de, dw = moe.moe_combine_backward(y.to(DEV), ros_t, w.to(DEV), dout.to(DEV))
    rde, rdw = O.combine_backward(O.to_f64(*storage(y)), ros, O.to_f64(*storage(w)),
                                  O.to_f64(*storage(dout)))
    assert rel_max_err(f64(de), rde) <= (1e-6 if ydt == torch.float32 else 2.0 ** -8)
    assert rel_max_err(f64(dw), rdw) <= 1e-5
    dx = moe.moe_dispatch_backward(de, ros_t, T, k)
    rdx = O.dispatch_backward(O.to_f64(*storage(de.cpu())), ros, T, k)
    assert rel_max_err(f64(dx), rdx) <= (1e-6 if ydt == torch.float32 else 2.0 ** -8)


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("H", [96, 41])
def test_backward_invalid_slot_gives_nan(ydt, H):
    """A slot whose row_of_slot is 0xFFFFFFFF (an expert id >= E never dispatched): its dweight is
    NaN, its token's dx row is NaN, and the dexpert rows of the other slots are still written."""
    T, k, E = 40, 4, 6
    gen = torch.Generator().manual_seed(8)
    idx = torch.stack([torch.randperm(E, generator=gen)[:k] for _ in range(T)]).numpy().astype(np.uint32)
    _, _, _, ros = O.dispatch(idx, E)
    ros = ros.copy()
    ros[3 * k + 1] = 0xFFFFFFFF
    y = torch.randn(T * k, H, generator=gen).to(ydt)
    w = torch.rand(T, k, generator=gen).to(ydt)
    dout = torch.randn(T, H, generator=gen).to(ydt)
    ros_t = torch.from_numpy(ros.view(np.int32)).to(DEV).view(torch.uint32)
    de, dw = moe.moe_combine_backward(y.to(DEV), ros_t, w.to(DEV), dout.to(DEV))
    dx = moe.moe_dispatch_backward(de, ros_t, T, k)
    torch.cuda.synchronize()
    dw, dx, de = dw.cpu(), dx.float().cpu(), de.float().cpu()
    assert torch.isnan(dw[3, 1]) and not torch.isnan(dw[3, [0, 2, 3]]).any()
    assert torch.isnan(dx[3]).all() and not torch.isnan(dx[torch.arange(T) != 3]).any()
    r0 = int(ros[3 * k])   # a valid slot of the same token: dexpert = w dout
    ref = (w[3, 0].float() * dout[3].float()).to(ydt).float()
    assert torch.equal(de[r0], ref)


@pytest.mark.parametrize("ydt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("H", [96, 41])
def test_combine_backward_writes_every_row(ydt, H):
    """Through the C ABI with an uninitialised dexpert buffer (filled with NaN bytes): ids >= E
    dispatched by moe_dispatch leave the last rows of the [T*k, H] layout unused; the library
    sets exactly those to zero and writes w dout into every other row."""
    from mixture_experts_routing_moe_gb300 import binding as B
    T, k, E = 50, 4, 6
    gen = torch.Generator().manual_seed(9)
    idx = torch.stack([torch.randperm(E + 2, generator=gen)[:k] for _ in range(T)])
    idx_np = idx.numpy().astype(np.uint32)
    n_bad = int((idx_np >= E).sum())
    assert n_bad > 0
    x = torch.randn(T, 64, generator=gen).to(torch.bfloat16).to(DEV)
    d = moe.moe_dispatch(x, torch.from_numpy(idx_np.view(np.int32)).to(DEV).view(torch.uint32), E)
    ros = d["row_of_slot"]
    y = torch.randn(T * k, H, generator=gen).to(ydt).to(DEV)
    w = torch.rand(T, k, generator=gen).to(ydt).to(DEV)
    dout = torch.randn(T, H, generator=gen).to(ydt).to(DEV)
    de = torch.full((T * k, H), float("nan"), dtype=ydt, device=DEV)
    dw = torch.empty(T, k, dtype=torch.float32, device=DEV)
    st = B.lib().moe_combine_backward(y.data_ptr(), B.DTYPE_CODE[ydt], ros.data_ptr(), w.data_ptr(),
                                      B.DTYPE_CODE[ydt], dout.data_ptr(), T, H, k, de.data_ptr(),
                                      dw.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    de = de.float().cpu()
    n_valid = T * k - n_bad
    assert torch.equal(de[n_valid:], torch.zeros(n_bad, H))
    ros_np = ros.view(torch.int32).cpu().numpy().view(np.uint32)
    for s in range(T * k):
        r = int(ros_np[s])
        if r != 0xFFFFFFFF:
            t, j = divmod(s, k)
            ref = (w[t, j].float().cpu() * dout[t].float().cpu()).to(ydt).float()
            assert torch.equal(de[r], ref), f"slot {s}"


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_full_backward_chain_matches_oracle(dt):
    """forward (route, dispatch, experts, combine) then combine_backward -> experts backward ->
    dispatch_backward -> router backward, against the oracle's chain on the same stored values."""
    wl = W.Workload("bwd_layer", T=200, H=128, I=192, E=8, top_k=2, renormalize=True,
                    dtype=DT_NAME[dt], seed=41)
    inp = W.make_layer_inputs(wl, "cpu")
    gdev = {k: v.to(DEV) for k, v in inp.items()}
    dout = torch.randn(wl.T, wl.H, generator=torch.Generator().manual_seed(6)).to(dt)
    idx, w = moe.moe_route(gdev["logits"], wl.top_k, True)
    d = moe.moe_dispatch(gdev["x"], idx, wl.E)
    y = moe.moe_experts_forward_dispatched(d["x_d"], d["offsets"], gdev["gate"], gdev["up"],
                                           gdev["down"])
    wts = moe.moe_selected_router_weights(gdev["logits"], idx, "softmax", True, 1.0)
    de, dwts = moe.moe_combine_backward(y, d["row_of_slot"], wts.to(dt), dout.to(DEV))
    dxd, dg, du, dd = moe.moe_experts_backward(d["x_d"], d["offsets"], gdev["gate"], gdev["up"],
                                               gdev["down"], de)
    dx = moe.moe_dispatch_backward(dxd, d["row_of_slot"], wl.T, wl.top_k)
    dl = moe.moe_selected_router_backward(gdev["logits"], idx, dwts, "softmax", True, 1.0)
    torch.cuda.synchronize()

    name = DT_NAME[dt]
    st = {k: storage(v) for k, v in inp.items()}
    l64 = O.to_f64(*st["logits"])
    ridx, _ = O.route(l64, wl.top_k, True, name)
    np.testing.assert_array_equal(u32(idx), ridx)
    _, offsets, tor, ros = O.dispatch(ridx, wl.E)
    xd = O.gather(O.to_f64(*st["x"]), tor)
    ry = O.experts(xd, offsets, st["gate"][0], st["up"][0], st["down"][0], name)
    rw = O.selected_router_weights(l64, ridx, "softmax", True, 1.0)
    rde, rdw = O.combine_backward(ry, ros, rw, O.to_f64(*storage(dout)))
    rdxd, rdg, rdu, rdd = O.experts_backward(xd, offsets, st["gate"][0], st["up"][0],
                                             st["down"][0], name, rde)
    rdx = O.dispatch_backward(rdxd, ros, wl.T, wl.top_k)
    rdl = O.selected_router_backward(l64, ridx, rdw, "softmax", True, 1.0)
    tol = layer_tol(dt)
    assert rel_max_err(f64(dx), rdx) <= tol
    assert rel_max_err(f64(dl), rdl) <= tol
    for got, ref in ((dg, rdg), (du, rdu), (dd, rdd)):
        assert rel_max_err(f64(got), ref) <= tol


@pytest.mark.parametrize("counts,H,I", [
    ([0, 300, 0, 0, 5, 64, 0, 1], 256, 128),        # tensor cores: idle experts between others
    ([0, 0, 0, 0], 128, 64),                          # no rows at all: every gradient is zero
    ([700, 0, 3, 0, 0, 600], 192, 256),               # CTA pairs for dA, g/u, dinput
    ([0] * 1000 + [200, 0, 0, 64] + [0] * 20, 64, 64),  # E = 1024, 1022 idle experts
])
def test_experts_backward_writes_every_gradient(counts, H, I):
    """Through the C ABI with dinput and the FP32 weight-gradient buffers filled with NaN: the
    library writes every element, the zero gradients of experts without rows included, and the
    rest equals moe_experts_backward's result."""
    from mixture_experts_routing_moe_gb300 import binding as B
    dt = torch.bfloat16
    E = len(counts)
    _, offsets, _, _ = O.dispatch(_groups(counts, 5), E) if sum(counts) else (
        None, np.zeros(E + 1, np.int64), None, None)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(E + H + I)
    x_d = torch.randn(max(rows, 1), H, generator=g).to(dt).to(DEV)[:rows]
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt).to(DEV)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt).to(DEV)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dt).to(DEV)
    dy = torch.randn(max(rows, 1), H, generator=g).to(dt).to(DEV)[:rows]
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    nan = float("nan")
    dx = torch.full((max(rows, 1), H), nan, dtype=dt, device=DEV)
    dg = torch.full((E, I, H), nan, dtype=torch.float32, device=DEV)
    du = torch.full((E, I, H), nan, dtype=torch.float32, device=DEV)
    dd = torch.full((E, H, I), nan, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(B.lib().moe_experts_backward_workspace_bytes(rows, I), 256),
                     dtype=torch.uint8, device=DEV)
    st = B.lib().moe_experts_backward(
        x_d.data_ptr(), off_t.data_ptr(), rows, gate.data_ptr(), up.data_ptr(), down.data_ptr(),
        B.DTYPE_CODE[dt], E, H, I, dy.data_ptr(), dx.data_ptr(), dg.data_ptr(), du.data_ptr(),
        dd.data_ptr(), ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    for name, t in (("dgate", dg), ("dup", du), ("ddown", dd), ("dinput", dx[:rows])):
        assert not torch.isnan(t).any(), f"{name}: elements left unwritten"
    idle = [e for e, n in enumerate(counts) if n == 0]
    for t in (dg, du, dd):
        assert torch.count_nonzero(t[idle]) == 0
    if rows:
        rx, rg, ru, rd = moe.moe_experts_backward(x_d, off_t, gate, up, down, dy)
        torch.cuda.synchronize()
        for got, ref in ((dx[:rows], rx), (dg, rg), (du, ru), (dd, rd)):
            assert torch.equal(got, ref)


def test_experts_backward_in_cuda_graph():
    """Captured into a CUDA graph and replayed.  Under capture the zero gradients of experts
    without rows are written in order on the captured stream, not beside the GEMMs on the
    library's second stream.  The replay into buffers refilled with NaN gives the same bytes as
    an eager call."""
    dt = torch.bfloat16
    counts, H, I = [400, 0, 300, 0, 129], 256, 128   # CTA pairs; two idle experts
    E = len(counts)
    _, offsets, _, _ = O.dispatch(_groups(counts, 7), E)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(77)
    x_d = torch.randn(rows, H, generator=g).to(dt).to(DEV)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt).to(DEV)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt).to(DEV)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dt).to(DEV)
    dy = torch.randn(rows, H, generator=g).to(dt).to(DEV)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    args = (x_d, off_t, gate, up, down, dy)
    ref = moe.moe_experts_backward(*args)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the capture, as torch recommends
        moe.moe_experts_backward(*args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = moe.moe_experts_backward(*args)
    for t in out:
        t.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    for got, want in zip(out, ref):
        iv = torch.int16 if got.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(got.view(iv), want.view(iv))
    for t in out[1:]:
        assert torch.count_nonzero(t[[1, 3]]) == 0


def test_experts_backward_fill_ordered_on_callers_stream():
    """The zero gradients of idle experts are written on the library's second stream and joined
    back into the caller's stream: kernels the caller enqueues on its stream right after the
    call (no device synchronisation in between) read no element of the NaN the buffers held.
    62 of 64 experts are idle, about 1.6 GB of zeros, long after the two active experts' GEMMs."""
    from mixture_experts_routing_moe_gb300 import binding as B
    dt = torch.bfloat16
    counts, H, I = [0] * 64, 2048, 1024
    counts[5], counts[40] = 300, 17
    E = len(counts)
    _, offsets, _, _ = O.dispatch(_groups(counts, 9), E)
    rows = int(offsets[-1])
    g = torch.Generator().manual_seed(99)
    x_d = torch.randn(rows, H, generator=g).to(dt).to(DEV)
    gate = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt).to(DEV)
    up = (torch.randn(E, I, H, generator=g) / H ** 0.5).to(dt).to(DEV)
    down = (torch.randn(E, H, I, generator=g) / I ** 0.5).to(dt).to(DEV)
    dy = torch.randn(rows, H, generator=g).to(dt).to(DEV)
    off_t = torch.from_numpy(offsets.astype(np.int32)).to(DEV)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        nan = float("nan")
        dx = torch.full((rows, H), nan, dtype=dt, device=DEV)
        dg = torch.full((E, I, H), nan, dtype=torch.float32, device=DEV)
        du = torch.full((E, I, H), nan, dtype=torch.float32, device=DEV)
        dd = torch.full((E, H, I), nan, dtype=torch.float32, device=DEV)
        ws = torch.empty(B.lib().moe_experts_backward_workspace_bytes(rows, I),
                         dtype=torch.uint8, device=DEV)
        st = B.lib().moe_experts_backward(
            x_d.data_ptr(), off_t.data_ptr(), rows, gate.data_ptr(), up.data_ptr(),
            down.data_ptr(), B.DTYPE_CODE[dt], E, H, I, dy.data_ptr(), dx.data_ptr(),
            dg.data_ptr(), du.data_ptr(), dd.data_ptr(), ws.data_ptr(), ws.numel(), s.cuda_stream)
        assert st == 0
        left = torch.stack([torch.isnan(t).sum() for t in (dx, dg, du, dd)])
        idle_nonzero = sum(torch.count_nonzero(t[[e for e in range(E) if counts[e] == 0]])
                           for t in (dg, du, dd))
    s.synchronize()
    assert left.tolist() == [0, 0, 0, 0]
    assert int(idle_nonzero) == 0
