"""moe_dispatch_static: the dispatch entry point that allocates nothing and takes no workspace.

Some callers cannot hand device scratch memory to a library call: a plugin whose interface
passes only inputs and outputs, or a runtime whose memory plan fixes every device allocation at
start-up.  For them moe_dispatch_static keeps its scratch in a file-scope device array.  This
test calls it through the C ABI and checks that it returns exactly what the workspace-taking
moe_dispatch returns, on two calls in a row with different sizes (the array still holds the
first call's contents when the second one runs), on expert ids >= E (not dispatched), at a size
that needs exactly the array's capacity, and that the next larger size is rejected before
anything is enqueued.
"""
import numpy as np
import pytest
import torch

import mixture_experts_routing_moe_gb300 as moe
from mixture_experts_routing_moe_gb300 import binding as B
from mixture_experts_routing_moe_gb300 import build

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _routed(T, E, k, seed):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1) ** -1.2
    p /= p.sum()
    idx = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.uint32)
    return torch.from_numpy(idx.view(np.int32)).to(DEV).view(torch.uint32)


def _dispatch_static(x, idx, E):
    T, H = x.shape
    k = idx.shape[1]
    R = T * k
    x_d = torch.empty(R, H, dtype=x.dtype, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    tor = torch.empty(R, dtype=torch.uint32, device=DEV)
    ros = torch.empty(R, dtype=torch.uint32, device=DEV)
    st = B.lib().moe_dispatch_static(x.data_ptr(), B.DTYPE_CODE[x.dtype], T, H, idx.data_ptr(), E,
                                     k, x_d.data_ptr(), offsets.data_ptr(), tor.data_ptr(),
                                     ros.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, B.STATUS.get(st, st)
    return x_d, offsets, tor, ros


def _i32(t):
    return t.view(torch.int32).cpu()


def test_static_dispatch_matches_workspace_dispatch_on_two_calls():
    build.build()
    for T, E, k, H, seed in [(3000, 64, 8, 256, 1), (700, 128, 4, 96, 2)]:
        g = torch.Generator().manual_seed(seed)
        x = torch.randn(T, H, generator=g).to(torch.bfloat16).to(DEV)
        idx = _routed(T, E, k, seed)
        ref = moe.moe_dispatch(x, idx, E)
        x_d, offsets, tor, ros = _dispatch_static(x, idx, E)
        torch.cuda.synchronize()
        assert torch.equal(offsets.cpu(), ref["offsets"].cpu())
        assert torch.equal(_i32(ros), _i32(ref["row_of_slot"]))
        assert torch.equal(_i32(tor), _i32(ref["token_of_row"]))
        assert torch.equal(x_d.view(torch.int16).cpu(), ref["x_d"].view(torch.int16).cpu())

    # beyond the static capacity (256 B + 1 MiB): T*k = 131072 slots -> 512 chunks x 1024 experts
    st = B.lib().moe_dispatch_static(0x10000, B.MOE_BF16, 16384, 64, 0x10000, 1024, 8, 0x10000,
                                     0x10000, 0x10000, 0x10000, None)
    assert st == 2


def _check_equal(x, idx, E):
    ref = moe.moe_dispatch(x, idx, E)
    x_d, offsets, tor, ros = _dispatch_static(x, idx, E)
    torch.cuda.synchronize()
    assert torch.equal(offsets.cpu(), ref["offsets"].cpu())
    assert torch.equal(_i32(ros), _i32(ref["row_of_slot"]))
    n = int(ref["offsets"][-1])
    assert torch.equal(_i32(tor)[:n], _i32(ref["token_of_row"])[:n])
    assert torch.equal(x_d[:n].view(torch.int16).cpu(), ref["x_d"][:n].view(torch.int16).cpu())
    return ros


def test_static_dispatch_invalid_ids_and_capacity_edge():
    build.build()
    # ids >= E are not dispatched (row_of_slot 0xFFFFFFFF), on both the one-block path (R <= 4096)
    # and the three-kernel path
    for T, E, k, seed in [(400, 64, 4, 3), (5000, 64, 4, 4)]:
        rng = np.random.default_rng(seed)
        idx_np = rng.integers(0, E + 5, size=(T, k)).astype(np.uint32)
        idx_np[0, 0] = 0xFFFFFFFF
        idx = torch.from_numpy(idx_np.view(np.int32)).to(DEV).view(torch.uint32)
        x = torch.randn(T, 128, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
        ros = _check_equal(x.to(DEV), idx, E)
        bad = (idx_np >= E).reshape(-1)
        assert bad.any()
        assert (_i32(ros).numpy().view(np.uint32)[bad] == 0xFFFFFFFF).all()

    # exactly at capacity: E = 1024, top_k = 8, T = 8160 needs 256 + (1023 + 1) * 256 * 4 bytes
    # ... = MOE_STATIC_DISPATCH_SCRATCH_BYTES (the histogram's last word is the array's last word)
    cap = 256 + (1 << 20)
    E, k = 1024, 8
    assert B.lib().moe_dispatch_workspace_bytes(8160, E, k) == cap
    assert B.lib().moe_dispatch_workspace_bytes(8161, E, k) > cap
    x = torch.randn(8160, 64, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    _check_equal(x.to(DEV), _routed(8160, E, k, 5), E)
    # one more token needs one more chunk of histograms: rejected, nothing enqueued
    st = B.lib().moe_dispatch_static(0x10000, B.MOE_BF16, 8161, 64, 0x10000, E, k, 0x10000,
                                     0x10000, 0x10000, 0x10000, None)
    assert st == 2
