"""ctypes binding of libmoe (include/moe.h).  Argument marshalling only.

Every function here takes torch CUDA tensors, checks that they are contiguous CUDA tensors,
allocates missing outputs / workspace with torch (device memory is the one thing torch is used
for), and passes raw pointers, sizes and the current stream to the C ABI.  All computation runs
in libmoe's kernels; there is no CPU path.  A missing or unbuilt library raises at first use.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe.h")

MOE_F32, MOE_F16, MOE_BF16 = 0, 1, 2
DTYPE_CODE = {torch.float32: MOE_F32, torch.float16: MOE_F16, torch.bfloat16: MOE_BF16}
STATUS = {0: "MOE_OK", 1: "MOE_ERR_NULL", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_DTYPE",
          4: "MOE_ERR_ALIGN", 5: "MOE_ERR_WORKSPACE", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_TIMEOUT",
          8: "MOE_ERR_INDEX", 9: "MOE_ERR_ARG"}

_i64, _int, _sz, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
_f32 = ctypes.c_float
_SIGS = {
    "moe_abi_version": (_int, []),
    "moe_status_string": (ctypes.c_char_p, [_int]),
    "moe_route": (_int, [_vp, _int, _i64, _i64, _int, _int, _vp, _vp, _vp]),
    "moe_route_sigmoid_grouped": (_int, [_vp, _int, _vp, _i64, _i64, _int, _int, _int, _int, _int,
                                         _f32, _vp, _vp, _vp]),
    "moe_selected_router_weights": (_int, [_vp, _int, _vp, _int, _i64, _i64, _int, _int, _int,
                                           _f32, _vp, _vp]),
    "moe_selected_router_backward": (_int, [_vp, _int, _vp, _int, _vp, _i64, _i64, _int, _int,
                                            _int, _f32, _vp, _vp]),
    "moe_dispatch_workspace_bytes": (_sz, [_i64, _i64, _int]),
    "moe_dispatch": (_int, [_vp, _int, _i64, _i64, _vp, _i64, _int, _vp, _vp, _vp, _vp, _vp, _sz,
                            _vp]),
    "moe_dispatch_static": (_int, [_vp, _int, _i64, _i64, _vp, _i64, _int, _vp, _vp, _vp, _vp,
                                   _vp]),
    "moe_experts_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _int]),
    "moe_experts_forward_dispatched": (_int, [_vp, _vp, _i64, _vp, _vp, _vp, _int, _i64, _i64,
                                              _i64, _vp, _vp, _sz, _vp]),
    "moe_combine": (_int, [_vp, _int, _vp, _vp, _int, _i64, _i64, _int, _vp, _vp]),
    "moe_forward_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64, _int, _int, _int]),
    "moe_forward": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _int, _i64, _i64, _i64, _i64, _int, _int,
                           _vp, _vp, _sz, _vp]),
    "moe_forward_sigmoid_grouped": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _int, _i64, _i64,
                                           _i64, _i64, _int, _int, _int, _int, _int, _f32, _vp,
                                           _vp, _sz, _vp]),
    "moe_forward_with_events": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _int, _i64, _i64, _i64,
                                       _i64, _int, _int, _vp, _vp, _sz, _vp, _vp]),
    "moe_forward_fused": (_int, [_i64, _i64, _i64, _i64, _int, _int, _int]),
    "moe_wait_selftest": (_int, [_vp, _sz, _vp]),
    "moe_combine_backward": (_int, [_vp, _int, _vp, _vp, _int, _vp, _i64, _i64, _int, _vp, _vp,
                                    _vp]),
    "moe_experts_backward_workspace_bytes": (_sz, [_i64, _i64]),
    "moe_experts_backward": (_int, [_vp, _vp, _i64, _vp, _vp, _vp, _int, _i64, _i64, _i64, _vp,
                                    _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_dispatch_backward": (_int, [_vp, _int, _vp, _i64, _i64, _int, _vp, _vp]),
    "moe_device_status": (_int, [_vp, _sz, _vp]),
}

_lib = None


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} "
                         f"({lib().moe_status_string(status).decode()})")


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_routing_moe_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/moe.h declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def _check(st: int, where: str):
    if st != 0:
        raise MoeError(st, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("libmoe takes contiguous CUDA tensors")


def _code(t) -> int:
    try:
        return DTYPE_CODE[t.dtype]
    except KeyError:
        raise MoeError(3, f"dtype {t.dtype}") from None


# ------------------------------------------------------------------------------ entry points
def moe_route(logits, top_k: int, renormalize: bool = True, idx=None, w=None, stream=None):
    """route(logits, RoutingOptions{top_k, renormalize}) -> (idx uint32 [T,k], w [T,k])."""
    _cuda(logits)
    T, E = logits.shape
    if idx is None:
        idx = torch.empty(T, top_k, dtype=torch.uint32, device=logits.device)
    if w is None:
        w = torch.empty(T, top_k, dtype=logits.dtype, device=logits.device)
    _cuda(idx, w)
    _check(lib().moe_route(_ptr(logits), _code(logits), T, E, top_k, int(bool(renormalize)),
                           _ptr(idx), _ptr(w), _stream(stream)), "moe_route")
    return idx, w


def moe_route_sigmoid_grouped(logits, top_k: int, groups: int, selected_groups: int,
                              group_top_two: bool = True, renormalize: bool = True,
                              scale: float = 1.0, bias=None, idx=None, w=None, stream=None):
    """route_sigmoid_grouped(logits, bias, GroupRoutingOptions) -> (idx uint32 [T,k], w [T,k])."""
    _cuda(logits, bias)
    if bias is not None and bias.dtype != torch.float32:
        raise MoeError(3, "bias must be float32")
    T, E = logits.shape
    if idx is None:
        idx = torch.empty(T, top_k, dtype=torch.uint32, device=logits.device)
    if w is None:
        w = torch.empty(T, top_k, dtype=logits.dtype, device=logits.device)
    _cuda(idx, w)
    _check(lib().moe_route_sigmoid_grouped(
        _ptr(logits), _code(logits), _ptr(bias), T, E, top_k, groups, selected_groups,
        int(bool(group_top_two)), int(bool(renormalize)), float(scale), _ptr(idx), _ptr(w),
        _stream(stream)), "moe_route_sigmoid_grouped")
    return idx, w


INDEX_CODE = {torch.uint32: 0, torch.int32: 1, torch.int64: 2}
SCORING = {"softmax": 0, "sigmoid": 1}


def moe_selected_router_weights(logits, idx, scoring: str = "softmax", renormalize: bool = True,
                                scale: float = 1.0, w=None, stream=None):
    """selected_router_weights(logits, indices, options) -> FP32 weights [T, k]."""
    _cuda(logits, idx)
    T, E = logits.shape
    k = idx.shape[1]
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device) if w is None else w
    _cuda(w)
    _check(lib().moe_selected_router_weights(
        _ptr(logits), _code(logits), _ptr(idx), INDEX_CODE[idx.dtype], T, E, k, SCORING[scoring],
        int(bool(renormalize)), float(scale), _ptr(w), _stream(stream)),
        "moe_selected_router_weights")
    return w


def moe_selected_router_backward(logits, idx, grad_w, scoring: str = "softmax",
                                 renormalize: bool = True, scale: float = 1.0, grad=None,
                                 stream=None):
    """selected_router_backward(logits, indices, grad_weights, options) -> dL/dlogits [T, E]."""
    _cuda(logits, idx, grad_w)
    if grad_w.dtype != torch.float32:
        raise MoeError(3, "grad_weights must be float32")
    T, E = logits.shape
    k = idx.shape[1]
    grad = torch.empty_like(logits) if grad is None else grad
    _cuda(grad)
    _check(lib().moe_selected_router_backward(
        _ptr(logits), _code(logits), _ptr(idx), INDEX_CODE[idx.dtype], _ptr(grad_w), T, E, k,
        SCORING[scoring], int(bool(renormalize)), float(scale), _ptr(grad), _stream(stream)),
        "moe_selected_router_backward")
    return grad


def dispatch_workspace_bytes(T: int, E: int, top_k: int) -> int:
    return lib().moe_dispatch_workspace_bytes(T, E, top_k)


def moe_dispatch(x, idx, E: int, x_d=None, offsets=None, token_of_row=None, row_of_slot=None,
                 ws=None, stream=None):
    """RoutingPlan::dispatch -> dict(x_d, offsets, token_of_row, row_of_slot, ws)."""
    _cuda(x, idx)
    T, H = x.shape
    k = idx.shape[1]
    R, dev = T * k, x.device
    x_d = torch.empty(R, H, dtype=x.dtype, device=dev) if x_d is None else x_d
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if offsets is None else offsets
    token_of_row = (torch.empty(R, dtype=torch.uint32, device=dev) if token_of_row is None
                    else token_of_row)
    row_of_slot = (torch.empty(R, dtype=torch.uint32, device=dev) if row_of_slot is None
                   else row_of_slot)
    if ws is None:
        ws = torch.empty(max(dispatch_workspace_bytes(T, E, k), 256), dtype=torch.uint8,
                         device=dev)
    _cuda(x_d, offsets, token_of_row, row_of_slot, ws)
    _check(lib().moe_dispatch(_ptr(x), _code(x), T, H, _ptr(idx), E, k, _ptr(x_d), _ptr(offsets),
                              _ptr(token_of_row), _ptr(row_of_slot), _ptr(ws), ws.numel(),
                              _stream(stream)), "moe_dispatch")
    return {"x_d": x_d, "offsets": offsets, "token_of_row": token_of_row,
            "row_of_slot": row_of_slot, "ws": ws}


def experts_workspace_bytes(rows: int, E: int, H: int, I: int, dtype) -> int:
    return lib().moe_experts_workspace_bytes(rows, E, H, I, DTYPE_CODE[dtype])


def moe_experts_forward_dispatched(x_d, offsets, gate, up, down, y=None, ws=None, stream=None):
    """SwiGluExperts::forward_dispatched -> y [rows, H]."""
    _cuda(x_d, offsets, gate, up, down)
    rows, H = x_d.shape
    E, I, _ = gate.shape
    y = torch.empty(rows, H, dtype=x_d.dtype, device=x_d.device) if y is None else y
    if ws is None:
        ws = torch.empty(max(experts_workspace_bytes(rows, E, H, I, gate.dtype), 256),
                         dtype=torch.uint8, device=x_d.device)
    _cuda(y, ws)
    _check(lib().moe_experts_forward_dispatched(
        _ptr(x_d), _ptr(offsets), rows, _ptr(gate), _ptr(up), _ptr(down), _code(gate), E, H, I,
        _ptr(y), _ptr(ws), ws.numel(), _stream(stream)), "moe_experts_forward_dispatched")
    return y


def moe_combine(y, row_of_slot, w, out=None, stream=None):
    """DispatchedTokens::combine -> out [T, H] in y's dtype."""
    _cuda(y, row_of_slot, w)
    T, k = w.shape
    H = y.shape[1]
    out = torch.empty(T, H, dtype=y.dtype, device=y.device) if out is None else out
    _cuda(out)
    _check(lib().moe_combine(_ptr(y), _code(y), _ptr(row_of_slot), _ptr(w), _code(w), T, H, k,
                             _ptr(out), _stream(stream)), "moe_combine")
    return out


def forward_workspace_bytes(T, E, H, I, top_k, logits_dtype, dtype) -> int:
    return lib().moe_forward_workspace_bytes(T, E, H, I, top_k, DTYPE_CODE[logits_dtype],
                                             DTYPE_CODE[dtype])


def moe_forward(x, logits, gate, up, down, top_k: int, renormalize: bool = True, out=None,
                ws=None, stream=None):
    """SwiGluExperts::forward(input, logits, options) -> out [T, H]."""
    _cuda(x, logits, gate, up, down)
    T, H = x.shape
    E, I, _ = gate.shape
    out = torch.empty_like(x) if out is None else out
    if ws is None:
        ws = torch.empty(max(forward_workspace_bytes(T, E, H, I, top_k, logits.dtype, x.dtype), 256),
                         dtype=torch.uint8, device=x.device)
    _cuda(out, ws)
    _check(lib().moe_forward(_ptr(x), _ptr(logits), _code(logits), _ptr(gate), _ptr(up),
                             _ptr(down), _code(gate), T, E, H, I, top_k, int(bool(renormalize)),
                             _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "moe_forward")
    return out


def moe_forward_sigmoid_grouped(x, logits, gate, up, down, top_k: int, groups: int,
                                selected_groups: int, group_top_two: bool = True,
                                renormalize: bool = True, scale: float = 1.0, bias=None, out=None,
                                ws=None, stream=None):
    """SwiGluExperts::forward_sigmoid_grouped -> out [T, H]."""
    _cuda(x, logits, gate, up, down, bias)
    T, H = x.shape
    E, I, _ = gate.shape
    out = torch.empty_like(x) if out is None else out
    if ws is None:
        ws = torch.empty(max(forward_workspace_bytes(T, E, H, I, top_k, logits.dtype, x.dtype), 256),
                         dtype=torch.uint8, device=x.device)
    _cuda(out, ws)
    _check(lib().moe_forward_sigmoid_grouped(
        _ptr(x), _ptr(logits), _code(logits), _ptr(bias), _ptr(gate), _ptr(up), _ptr(down),
        _code(gate), T, E, H, I, top_k, groups, selected_groups, int(bool(group_top_two)),
        int(bool(renormalize)), float(scale), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
        "moe_forward_sigmoid_grouped")
    return out


def moe_forward_fused(T: int, E: int, H: int, I: int, top_k: int, logits_dtype, dtype) -> bool:
    """Whether moe_forward runs these sizes as the single fused launch (aligned tensors)."""
    return bool(lib().moe_forward_fused(T, E, H, I, top_k, DTYPE_CODE[logits_dtype], DTYPE_CODE[dtype]))


def moe_forward_with_events(x, logits, gate, up, down, top_k: int, renormalize: bool, out=None,
                            ws=None, events=None, stream=None):
    """The staged moe_forward (separate launches), recording six torch.cuda.Event objects at the
    stage boundaries (before route / after route / after dispatch / after gate-up / after down /
    after combine) when `events` is given."""
    _cuda(x, logits, gate, up, down)
    T, H = x.shape
    E, I, _ = gate.shape
    out = torch.empty_like(x) if out is None else out
    if ws is None:
        ws = torch.empty(max(forward_workspace_bytes(T, E, H, I, top_k, logits.dtype, x.dtype), 256),
                         dtype=torch.uint8, device=x.device)
    _cuda(out, ws)
    arr = None
    if events is not None:
        if len(events) != 6:
            raise ValueError("moe_forward_with_events needs six events")
        for ev in events:
            if ev.cuda_event == 0:      # torch creates the CUDA event on its first record
                ev.record(torch.cuda.current_stream() if stream is None else stream)
        arr = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    _check(lib().moe_forward_with_events(
        _ptr(x), _ptr(logits), _code(logits), _ptr(gate), _ptr(up), _ptr(down), _code(gate), T, E,
        H, I, top_k, int(bool(renormalize)), _ptr(out), _ptr(ws), ws.numel(), _stream(stream),
        arr), "moe_forward_with_events")
    return out


def moe_combine_backward(y, row_of_slot, w, dout, stream=None):
    """DispatchedTokens::combine_backward -> (dexpert [T*k, H], dweights [T, k] FP32)."""
    _cuda(y, row_of_slot, w, dout)
    T, k = w.shape
    H = y.shape[1]
    dexpert = torch.empty_like(y)
    dweights = torch.empty(T, k, dtype=torch.float32, device=y.device)
    _check(lib().moe_combine_backward(_ptr(y), _code(y), _ptr(row_of_slot), _ptr(w), _code(w),
                                      _ptr(dout), T, H, k, _ptr(dexpert), _ptr(dweights),
                                      _stream(stream)), "moe_combine_backward")
    return dexpert, dweights


def moe_experts_backward(x_d, offsets, gate, up, down, dy, ws=None, stream=None):
    """cache.backward(dexpert) -> (dinput [rows, H], dgate, dup [E, I, H], ddown [E, H, I] FP32)."""
    _cuda(x_d, offsets, gate, up, down, dy)
    rows, H = x_d.shape
    E, I, _ = gate.shape
    dev = x_d.device
    dinput = torch.empty_like(x_d)
    dgate = torch.empty(E, I, H, dtype=torch.float32, device=dev)
    dup = torch.empty(E, I, H, dtype=torch.float32, device=dev)
    ddown = torch.empty(E, H, I, dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(max(lib().moe_experts_backward_workspace_bytes(rows, I), 256),
                         dtype=torch.uint8, device=dev)
    _check(lib().moe_experts_backward(
        _ptr(x_d), _ptr(offsets), rows, _ptr(gate), _ptr(up), _ptr(down), _code(gate), E, H, I,
        _ptr(dy), _ptr(dinput), _ptr(dgate), _ptr(dup), _ptr(ddown), _ptr(ws), ws.numel(),
        _stream(stream)), "moe_experts_backward")
    return dinput, dgate, dup, ddown


def moe_dispatch_backward(dinput, row_of_slot, T: int, top_k: int, stream=None):
    """DispatchedTokens::dispatch_backward -> dx [T, H] (slot rows summed, no weights)."""
    _cuda(dinput, row_of_slot)
    H = dinput.shape[1]
    dx = torch.empty(T, H, dtype=dinput.dtype, device=dinput.device)
    _check(lib().moe_dispatch_backward(_ptr(dinput), _code(dinput), _ptr(row_of_slot), T, H, top_k,
                                       _ptr(dx), _stream(stream)), "moe_dispatch_backward")
    return dx


def moe_wait_selftest(ws, stream=None) -> None:
    """One bounded wait that nothing completes: the timeout lands in ws's status word."""
    _cuda(ws)
    _check(lib().moe_wait_selftest(_ptr(ws), ws.numel(), _stream(stream)), "moe_wait_selftest")


def moe_device_status(ws, stream=None) -> int:
    """Synchronise, read and clear the workspace status word (0 = MOE_OK)."""
    return lib().moe_device_status(_ptr(ws), ws.numel(), _stream(stream))
