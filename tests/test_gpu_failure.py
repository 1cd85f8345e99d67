"""Failure detection on the GPU without a fault: a bounded wait that nothing completes gives up,
the status word reports the timeout, and the context keeps working."""
import pytest
import torch

import mixture_experts_routing_moe_gb300 as moe
from mixture_experts_routing_moe_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert moe.moe_device_status(ws) == 0          # reads and clears
    moe.moe_wait_selftest(ws)
    assert moe.moe_device_status(ws) == 7                   # MOE_ERR_TIMEOUT
    assert moe.moe_device_status(ws) == 0          # cleared by the read
    # the context is usable: a forward (the fused launch) runs and reports no error
    wl = W.Workload("after_timeout", T=64, H=256, I=256, E=16, top_k=2, renormalize=True,
                    dtype="bf16", seed=2)
    g = W.make_layer_inputs(wl, "cuda")
    wsf = torch.empty(moe.forward_workspace_bytes(wl.T, wl.E, wl.H, wl.I, wl.top_k,
                                                  g["logits"].dtype, g["x"].dtype),
                      dtype=torch.uint8, device="cuda")
    out = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], wl.top_k, True,
                          ws=wsf)
    assert moe.moe_device_status(wsf) == 0
    assert torch.isfinite(out.float()).all()
