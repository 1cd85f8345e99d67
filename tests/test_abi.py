"""The C ABI without a GPU: the library loads, exports what include/moe.h declares, and rejects
bad arguments on the host before anything is enqueued (the error behaviour of §6 "MoE aufrufen"
of the ruDNN user guide: shape, dtype and argument mismatches return an error)."""
import ctypes

import pytest
import torch

from mixture_experts_routing_moe_gb300 import binding as B
from mixture_experts_routing_moe_gb300 import build as build_mod


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


FAKE = 0x10000  # never dereferenced: every call below is rejected (or fails to launch) first
F32, F16, BF16 = B.MOE_F32, B.MOE_F16, B.MOE_BF16


def test_exports_every_header_function(L):
    names = B.header_functions()
    assert len(names) == 23
    for n in names:
        assert hasattr(L, n), n
    assert L.moe_abi_version() == 1
    for code in range(10):
        assert L.moe_status_string(code) not in (None, b"unknown status")


def test_route_rejects(L):
    ok = dict(logits=FAKE, ldt=BF16, T=16, E=8, k=2, r=1, idx=FAKE, w=FAKE)

    def call(**kw):
        a = {**ok, **kw}
        return L.moe_route(a["logits"], a["ldt"], a["T"], a["E"], a["k"], a["r"], a["idx"],
                           a["w"], None)
    assert call(ldt=7) == 3
    assert call(k=0) == 2
    assert call(k=9) == 2           # top_k > E
    assert call(E=0, k=1) == 2
    assert call(E=1025, k=2) == 2
    assert call(T=-1) == 2
    assert call(T=1 << 29, k=8, E=64) == 2   # T * k >= 2^31
    assert call(logits=None) == 1
    assert call(idx=None) == 1
    assert call(w=None) == 1
    assert call(T=0, logits=None, idx=None, w=None) == 0   # empty batch: nothing enqueued


def test_dispatch_rejects(L):
    ws_need = L.moe_dispatch_workspace_bytes(100, 16, 4)
    assert ws_need >= 256 + 16 * 4

    def call(x=FAKE, xdt=BF16, T=100, H=64, idx=FAKE, E=16, k=4, ws=FAKE, wsb=ws_need, xd=FAKE):
        return L.moe_dispatch(x, xdt, T, H, idx, E, k, xd, FAKE, FAKE, FAKE, ws, wsb, None)
    assert call(xdt=9) == 3
    assert call(k=17) == 2
    assert call(H=0) == 2
    assert call(idx=None) == 1
    assert call(x=FAKE + 2) == 4        # misaligned tokens
    assert call(H=12) == 4              # 24-byte rows: not a multiple of 16 bytes
    assert call(ws=None) == 5
    assert call(wsb=ws_need - 1) == 5
    assert call(T=0, x=None, idx=None, xd=None, ws=None) == 0


def test_experts_rejects(L):
    need = L.moe_experts_workspace_bytes(64, 4, 128, 256, BF16)
    assert need >= 256 + 64 * 256 * 2

    def call(xd=FAKE, rows=64, g=FAKE, wdt=BF16, E=4, H=128, I=256, ws=FAKE, wsb=need):
        return L.moe_experts_forward_dispatched(xd, FAKE, rows, g, FAKE, FAKE, wdt, E, H, I, FAKE,
                                                ws, wsb, None)
    assert call(wdt=5) == 3
    assert call(E=0) == 2
    assert call(I=0) == 2
    assert call(g=None) == 1
    assert call(xd=None) == 1
    assert call(ws=FAKE + 16) == 5      # workspace must be 256-byte aligned
    assert call(wsb=need - 1) == 5
    assert call(H=100) == 4             # tensor-core path needs H % 8 == 0
    assert call(I=260, wsb=L.moe_experts_workspace_bytes(64, 4, 128, 260, BF16)) == 4
    assert call(xd=FAKE + 8) == 4
    assert call(rows=0, xd=None) == 0


def test_combine_and_forward_reject(L):
    assert L.moe_combine(FAKE, 4, FAKE, FAKE, F32, 8, 64, 2, FAKE, None) == 3
    assert L.moe_combine(FAKE, F32, FAKE, FAKE, F32, 8, 0, 2, FAKE, None) == 2
    assert L.moe_combine(None, F32, FAKE, FAKE, F32, 8, 64, 2, FAKE, None) == 1
    need = L.moe_forward_workspace_bytes(32, 8, 128, 256, 2, BF16, BF16)
    assert need > 0

    def fwd(x=FAKE, ldt=BF16, wdt=BF16, T=32, E=8, H=128, I=256, k=2, ws=FAKE, wsb=need):
        return L.moe_forward(x, FAKE, ldt, FAKE, FAKE, FAKE, wdt, T, E, H, I, k, 1, FAKE, ws, wsb,
                             None)
    assert fwd(ldt=3) == 3
    assert fwd(k=9) == 2
    assert fwd(x=None) == 1
    assert fwd(H=132) == 4
    assert fwd(wsb=need - 1) == 5
    assert fwd(T=0, x=None) == 0


def test_workspace_queries_grow_with_size(L):
    a = L.moe_forward_workspace_bytes(1024, 64, 512, 1024, 4, BF16, BF16)
    b = L.moe_forward_workspace_bytes(2048, 64, 512, 1024, 4, BF16, BF16)
    assert 0 < a < b
    assert L.moe_forward_workspace_bytes(16, 8, 64, 64, 9, BF16, BF16) == 0   # invalid -> 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_valid_call_without_gpu_fails_loudly(L):
    """No CPU fallback: a well-formed call on a machine without a GPU reports a CUDA error."""
    assert L.moe_route(FAKE, BF16, 16, 8, 2, 1, FAKE, FAKE, None) == 6
    with pytest.raises(Exception):
        B.moe_route(torch.zeros(4, 8), 2)


def test_sigmoid_router_rejects(L):
    def call(ldt=BF16, T=16, E=64, k=8, G=8, SG=4, top2=1, scale=1.0, logits=FAKE):
        return L.moe_route_sigmoid_grouped(logits, ldt, None, T, E, k, G, SG, top2, 1, scale, FAKE,
                                           FAKE, None)
    assert call(ldt=5) == 3
    assert call(G=7) == 2             # E % groups != 0
    assert call(G=256, E=256) == 2    # more than 128 groups
    assert call(SG=9) == 2            # selected_groups > groups
    assert call(k=65, E=128) == 2     # top_k > 64
    assert call(k=9, SG=1) == 2       # top_k > selected_groups * E / groups
    assert call(G=64, top2=1) == 2    # group_top_two needs >= 2 experts per group
    assert call(scale=0.0) == 9
    assert call(scale=float("inf")) == 9
    assert call(scale=float("nan")) == 9
    assert call(logits=None) == 1
    assert call(T=0, logits=None) == 0
    need = L.moe_forward_workspace_bytes(16, 64, 128, 256, 8, BF16, BF16)
    assert L.moe_forward_sigmoid_grouped(FAKE, FAKE, BF16, None, FAKE, FAKE, FAKE, BF16, 16, 64,
                                         128, 256, 8, 8, 4, 1, 1, -1.0, FAKE, FAKE, need,
                                         None) == 9


def test_router_train_rejects(L):
    def fw(ldt=F32, idt=0, T=8, E=16, k=4, sc=0, scale=1.0, logits=FAKE):
        return L.moe_selected_router_weights(logits, ldt, FAKE, idt, T, E, k, sc, 1, scale, FAKE,
                                             None)
    assert fw(ldt=4) == 3
    assert fw(idt=3) == 3
    assert fw(sc=2) == 9
    assert fw(k=17) == 2
    assert fw(k=65, E=128) == 2
    assert fw(scale=-2.0) == 9
    assert fw(logits=None) == 1
    assert fw(T=0, logits=None) == 0
    assert L.moe_selected_router_backward(FAKE, F32, FAKE, 2, None, 8, 16, 4, 1, 0, 1.0, FAKE,
                                          None) == 1


def test_wait_selftest_rejects(L):
    assert L.moe_wait_selftest(None, 256, None) == 1
    assert L.moe_wait_selftest(FAKE + 16, 256, None) == 5
    assert L.moe_wait_selftest(FAKE, 255, None) == 5


def test_backward_chain_rejects(L):
    assert L.moe_combine_backward(FAKE, 5, FAKE, FAKE, F32, FAKE, 4, 8, 2, FAKE, FAKE, None) == 3
    assert L.moe_combine_backward(FAKE, F32, FAKE, FAKE, F32, None, 4, 8, 2, FAKE, FAKE, None) == 1
    assert L.moe_dispatch_backward(FAKE, BF16, FAKE, 4, 0, 2, FAKE, None) == 2
    need = L.moe_experts_backward_workspace_bytes(64, 32)
    assert need >= 256 + 64 * 32 * 20
    assert L.moe_experts_backward(FAKE, FAKE, 64, FAKE, FAKE, FAKE, BF16, 4, 16, 32, FAKE, FAKE,
                                  FAKE, FAKE, FAKE, FAKE, need - 1, None) == 5
    assert L.moe_experts_backward(FAKE, FAKE, 64, FAKE, FAKE, FAKE, BF16, 4, 16, 32, None, FAKE,
                                  FAKE, FAKE, FAKE, FAKE, need, None) == 1
