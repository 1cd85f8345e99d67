"""GPU parity of the fused short-batch forward (one cooperative launch: route, dispatch, gate/up,
down, combine; ruDNN user guide §3-§6) against the fp64 oracle, and against the staged launches.

The fused route reads a row with one full warp, the staged route with the narrowest lane group
that covers E; for 16-bit logits and 64 < E <= 256 both sum the softmax in the same order, so the
two paths must agree bit for bit.  Elsewhere they agree within the layer tolerance."""
import numpy as np
import pytest
import torch

import oracle as O
import mixture_experts_routing_moe_gb300 as moe
from mixture_experts_routing_moe_gb300 import workloads as W

from gpu_helpers import DT_NAME, f64, layer_tol, oracle_expert_weights, rel_max_err, storage

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    # name, T, E, k, H, I, dtype, logits dtype, renormalize, zipf, special rows
    ("bf16_e96_ragged_i", 48, 96, 6, 256, 192, "bf16", "bf16", True, 1.0, False),
    ("f16_e128_no_renorm", 100, 128, 8, 128, 128, "f16", "f16", False, 1.1, False),
    ("bf16_f32_logits_e64", 64, 64, 4, 192, 256, "bf16", "f32", True, 0.0, False),
    ("bf16_poisoned_rows", 40, 72, 3, 128, 128, "bf16", "bf16", True, 0.5, True),
    ("bf16_max_slots_e256", 512, 256, 8, 128, 128, "bf16", "bf16", True, 1.2, False),
    ("bf16_e16_small", 300, 16, 4, 256, 512, "bf16", "bf16", False, 1.0, False),
]
TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def _inputs(name, T, E, k, H, I, dt, ldt, renorm, zipf, special, seed):
    wl = W.Workload(name, T=T, E=E, top_k=k, renormalize=renorm, dtype=dt, seed=seed, H=H, I=I,
                    zipf_s=zipf, special_rows=special)
    inp = W.make_layer_inputs(wl, "cpu")
    inp["logits"] = W.make_logits(wl, "cpu").float().to(TORCH_DT[ldt]) if ldt != dt else inp["logits"]
    return wl, inp


def _staged(g, wl):
    return moe.moe_forward_with_events(g["x"], g["logits"], g["gate"], g["up"], g["down"],
                                       wl.top_k, wl.renormalize)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_oracle_and_staged(case):
    name, T, E, k, H, I, dt, ldt, renorm, zipf, special = case
    wl, inp = _inputs(name, T, E, k, H, I, dt, ldt, renorm, zipf, special, seed=31)
    assert moe.moe_forward_fused(T, E, H, I, k, TORCH_DT[ldt], TORCH_DT[dt])
    g = {n: v.to(DEV) for n, v in inp.items()}
    ws = torch.empty(moe.forward_workspace_bytes(T, E, H, I, k, g["logits"].dtype, g["x"].dtype),
                     dtype=torch.uint8, device=DEV)
    out = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], k, renorm, ws=ws)
    assert moe.moe_device_status(ws) == 0
    out2 = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], k, renorm, ws=ws)
    staged = _staged(g, wl)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), out2.view(torch.uint8)), "not run-to-run identical"
    if ldt != "f32" and 64 < E <= 256:  # same route arithmetic on both paths
        assert torch.equal(out.view(torch.uint8), staged.view(torch.uint8)), "fused != staged"
    assert rel_max_err(f64(out), f64(staged)) <= layer_tol(g["x"].dtype)
    st = {n: storage(v) for n, v in inp.items()}
    ref = O.forward(*st["x"], *st["logits"], st["gate"][0], st["up"][0], st["down"][0], dt, k,
                    renorm)["out_unrounded"]
    err = rel_max_err(f64(out), ref)
    assert err <= layer_tol(g["x"].dtype), f"{name}: rel max err {err}"


def test_fused_decode_full_size():
    """The decode layer (T=256, E=128, k=8, H=2048, I=768): fused == staged bit for bit, and a
    sample of tokens against the oracle."""
    wl = W.WORKLOADS["decode"]
    assert moe.moe_forward_fused(wl.T, wl.E, wl.H, wl.I, wl.top_k, torch.bfloat16, torch.bfloat16)
    g = W.make_layer_inputs(wl, DEV)
    out = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], wl.top_k,
                          wl.renormalize)
    staged = _staged(g, wl)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), staged.view(torch.uint8)), "fused != staged"
    larr, lname = storage(g["logits"])
    ridx, rw = O.route(O.to_f64(larr, lname), wl.top_k, wl.renormalize, lname)
    tok = np.sort(np.random.default_rng(3).choice(wl.T, 24, replace=False))
    xs = O.to_f64(storage(g["x"][torch.from_numpy(tok).to(DEV)])[0], "bf16")
    ref = O.forward_rows(xs, ridx[tok], rw[tok],
                         oracle_expert_weights(g["gate"], g["up"], g["down"], "bf16"))
    assert rel_max_err(f64(out)[tok], ref) <= layer_tol(torch.bfloat16)


def test_fused_path_selection():
    """Sizes outside the fused path's limits take the staged launches."""
    bf, f32 = torch.bfloat16, torch.float32
    assert not moe.moe_forward_fused(256, 128, 2048, 768, 8, bf, f32)      # f32 experts
    assert not moe.moe_forward_fused(1024, 128, 2048, 768, 8, bf, bf)      # T*k > 4096
    assert not moe.moe_forward_fused(256, 8, 2048, 768, 8, bf, bf)         # >= 128 rows/expert
    assert not moe.moe_forward_fused(256, 512, 2048, 768, 8, bf, bf)       # E > 256
    assert not moe.moe_forward_fused(256, 128, 2040, 768, 8, bf, bf)       # H % 64 != 0
    assert not moe.moe_forward_fused(256, 124, 2048, 768, 8, bf, bf)       # E * 2 % 16 != 0
    assert moe.moe_forward_fused(256, 128, 2048, 768, 8, bf, bf)


@pytest.mark.parametrize("name,T,E,k,H,I,G,SG,top2", [
    ("decode_sigmoid", 256, 128, 8, 2048, 768, 8, 4, True),
    ("small_sigmoid", 60, 96, 4, 256, 192, 6, 2, False),
])
def test_fused_sigmoid_forward_equals_stages(name, T, E, k, H, I, G, SG, top2):
    """moe_forward_sigmoid_grouped on a short batch runs the single fused launch; it equals, bit
    for bit, the stage calls (sigmoid route, dispatch, experts, combine) on the same inputs, and
    a sample of tokens matches the oracle."""
    assert moe.moe_forward_fused(T, E, H, I, k, torch.bfloat16, torch.bfloat16)
    wl = W.Workload(name, T=T, E=E, top_k=k, renormalize=True, dtype="bf16", seed=23, H=H, I=I,
                    zipf_s=1.0)
    g = W.make_layer_inputs(wl, DEV)
    bias = (0.02 * torch.randn(E, generator=torch.Generator(device=DEV).manual_seed(3),
                               device=DEV)).float()
    out = moe.moe_forward_sigmoid_grouped(g["x"], g["logits"], g["gate"], g["up"], g["down"], k, G,
                                          SG, top2, True, 1.5, bias)
    idx, w = moe.moe_route_sigmoid_grouped(g["logits"], k, G, SG, top2, True, 1.5, bias)
    d = moe.moe_dispatch(g["x"], idx, E)
    y = moe.moe_experts_forward_dispatched(d["x_d"], d["offsets"], g["gate"], g["up"], g["down"])
    staged = moe.moe_combine(y, d["row_of_slot"], w)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), staged.view(torch.uint8)), "fused != stages"
    larr, lname = storage(g["logits"])
    ridx, rw = O.route_sigmoid_grouped(O.to_f64(larr, lname), bias.double().cpu().numpy(), k, G,
                                       SG, top2, True, 1.5, lname)
    tok = np.sort(np.random.default_rng(5).choice(T, min(T, 20), replace=False))
    xs = O.to_f64(storage(g["x"][torch.from_numpy(tok).to(DEV)])[0], "bf16")
    ref = O.forward_rows(xs, ridx[tok], rw[tok],
                         oracle_expert_weights(g["gate"], g["up"], g["down"], "bf16"))
    assert rel_max_err(f64(out)[tok], ref) <= layer_tol(torch.bfloat16)


PAIR_CASES = [
    # name, T, E, k, H, I, dtype, zipf: experts average >= 128 rows, so the layer takes the CTA-pair
    # kernels (256-row tiles, 128-row tails)
    ("bf16_e4", 600, 4, 2, 256, 192, "bf16", 1.0),
    ("f16_e16_ragged", 2000, 16, 2, 512, 256, "f16", 1.3),
    ("bf16_e8_k3_steep", 1003, 8, 3, 128, 384, "bf16", 2.0),
]


@pytest.mark.parametrize("case", PAIR_CASES, ids=[c[0] for c in PAIR_CASES])
def test_forward_pair_equals_stages(case):
    """moe_forward on the CTA-pair path equals, bit for bit, the stage calls (route, dispatch,
    experts on x_d, combine) on ragged experts, and a sample of tokens matches the oracle."""
    name, T, E, k, H, I, dt, zipf = case
    assert not moe.moe_forward_fused(T, E, H, I, k, TORCH_DT[dt], TORCH_DT[dt])
    wl = W.Workload(name, T=T, E=E, top_k=k, renormalize=True, dtype=dt, seed=41, H=H, I=I,
                    zipf_s=zipf)
    g = W.make_layer_inputs(wl, DEV)
    out = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], k, True)
    idx, w = moe.moe_route(g["logits"], k, True)
    d = moe.moe_dispatch(g["x"], idx, E)
    y = moe.moe_experts_forward_dispatched(d["x_d"], d["offsets"], g["gate"], g["up"], g["down"])
    staged = moe.moe_combine(y, d["row_of_slot"], w)
    torch.cuda.synchronize()
    counts = np.diff(d["offsets"].cpu().numpy())
    assert counts.max() > 256, counts     # several 256-row tiles in one expert
    if name != "bf16_e4":                 # and experts whose last tile has <= 128 rows
        assert ((counts % 256 > 0) & (counts % 256 <= 128)).any(), counts
    assert torch.equal(out.view(torch.uint8), staged.view(torch.uint8)), "forward != stages"
    larr, lname = storage(g["logits"])
    ridx, rw = O.route(O.to_f64(larr, lname), k, True, lname)
    tok = np.sort(np.random.default_rng(2).choice(T, 24, replace=False))
    xs = O.to_f64(storage(g["x"][torch.from_numpy(tok).to(DEV)])[0], dt)
    ref = O.forward_rows(xs, ridx[tok], rw[tok], oracle_expert_weights(g["gate"], g["up"], g["down"], dt))
    assert rel_max_err(f64(out)[tok], ref) <= layer_tol(g["x"].dtype)
