"""W4A8 mixture-of-experts FFN and block-FP8 projection for GB300 (sm_103a).

Thin Python binding over the C ABI in include/w4a8_moe.h: each function has
the C entry point's name, takes torch CUDA tensors, allocates outputs and
workspaces with torch when the caller passes none, and forwards pointers, sizes
and the current CUDA stream. Every arithmetic step runs in the library's CUDA
kernels (libw4a8_moe.so, built in-tree by w4a8_moe_gb300/build.py); there is
no other implementation, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from collections import namedtuple

import torch

__all__ = [
    "w4a8_quantize_experts", "w4a8_quantize_act", "moe_route", "moe_w4a8_forward",
    "fp8_block_linear", "w4a8_device_error", "w4a8_selftest_wait_timeout", "w4a8_set_profile_events", "moe_w4a8_workspace_size",
    "moe_route_workspace_size", "fp8_block_linear_workspace_size", "moe_route_gate",
    "moe_route_gate_workspace_size", "fp8_linear", "fp8_linear_workspace_size",
    "moe_w4a8_forward_dynamic", "moe_w4a8_dynamic_workspace_size", "moe_w4a8_workspace_layout",
    "moe_w4a8_plan",
    "w4a8_quantize_act_workspace_size", "RouteResult", "library_path", "W4A8Error",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libw4a8_moe.so")
_lib = None

RouteResult = namedtuple("RouteResult", "topk_ids topk_w counts offsets sorted_ids inv_perm")


class W4A8Error(RuntimeError):
    pass


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise W4A8Error(f"CUDA library {_LIB_PATH} is not built; run "
                        "`python -m w4a8_moe_gb300.build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "w4a8_status_string": (ctypes.c_char_p, [i32]),
        "w4a8_version": (i32, []),
        "w4a8_quantize_experts": (i32, [P, i32, i32, i32, P, P, P]),
        "w4a8_quantize_act": (i32, [P, i64, P, i32, P, P, sz, P]),
        "w4a8_quantize_act_workspace_size": (sz, [i64]),
        "moe_route": (i32, [P, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]),
        "moe_route_workspace_size": (sz, [i32, i32, i32]),
        "moe_route_gate": (i32, [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, sz, P]),
        "moe_route_gate_workspace_size": (sz, [i32, i32, i32, i32]),
        "moe_w4a8_forward": (i32, [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P,
                                   P, P, P, sz, P]),
        "moe_w4a8_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "moe_w4a8_plan": (i32, [i32, i32, i32, i32, i32, i32, i32, P]),
        "moe_w4a8_workspace_layout": (i32, [i32, i32, i32, i32, i32, P]),
        "moe_w4a8_forward_dynamic": (i32, [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P,
                                           P, P, P, sz, P]),
        "moe_w4a8_dynamic_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "fp8_block_linear": (i32, [P, i32, i32, i32, P, P, P, P, P, P, sz, P]),
        "fp8_block_linear_workspace_size": (sz, [i32, i32, i32]),
        "fp8_linear": (i32, [P, P, i32, i32, i32, P, P, P, P, sz, P]),
        "fp8_linear_workspace_size": (sz, [i32, i32, i32]),
        "w4a8_device_error": (i32, [P, P, P]),
        "w4a8_selftest_wait_timeout": (i32, [P, P]),
        "w4a8_set_profile_events": (i32, [P, i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise W4A8Error(_load().w4a8_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _u8(t):
    return t.view(torch.uint8) if t.dtype != torch.uint8 else t


def _ws(nbytes: int, device, ws=None):
    if ws is not None:
        return ws
    buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    buf[:256].zero_()  # device error word
    return buf


# --------------------------------------------------------------------------- sizes
def moe_w4a8_workspace_size(T, H, I, E, k) -> int:
    return int(_load().moe_w4a8_workspace_size(T, H, I, E, k))


_PLAN_KEYS = ("token_tile", "k_per_stage", "down_ksplit", "down_streamk", "down_slots", "one_launch",
              "launches", "partials")


def moe_w4a8_plan(T, H, I, E, k, dynamic=False, num_sms=None) -> dict:
    """The launch plan of the MoE forward for this shape (host only; see
    moe_w4a8_plan in include/w4a8_moe.h). num_sms defaults to the current
    device's SM count."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    plan = (ctypes.c_int32 * 8)()
    _check(_load().moe_w4a8_plan(T, H, I, E, k, 1 if dynamic else 0, num_sms, plan))
    return dict(zip(_PLAN_KEYS, list(plan)))


def moe_w4a8_workspace_layout(T, H, I, E, k) -> dict:
    """Byte offsets of the intermediate tensors a forward call leaves in its
    workspace (see moe_w4a8_workspace_layout in include/w4a8_moe.h)."""
    off = (ctypes.c_int64 * 2)()
    _check(_load().moe_w4a8_workspace_layout(T, H, I, E, k, off))
    return {"hq": int(off[0]), "xp": int(off[1])}


def moe_w4a8_dynamic_workspace_size(T, H, I, E, k) -> int:
    return int(_load().moe_w4a8_dynamic_workspace_size(T, H, I, E, k))


def moe_route_workspace_size(T, E, k) -> int:
    return int(_load().moe_route_workspace_size(T, E, k))


def moe_route_gate_workspace_size(T, H, E, k) -> int:
    return int(_load().moe_route_gate_workspace_size(T, H, E, k))


def fp8_linear_workspace_size(M, N, K) -> int:
    return int(_load().fp8_linear_workspace_size(M, N, K))


def fp8_block_linear_workspace_size(M, N, K) -> int:
    return int(_load().fp8_block_linear_workspace_size(M, N, K))


def w4a8_quantize_act_workspace_size(numel) -> int:
    return int(_load().w4a8_quantize_act_workspace_size(numel))


# --------------------------------------------------------------------------- calls
def w4a8_quantize_experts(w_bf16: torch.Tensor, packed=None, scale=None, stream=None):
    """bf16 [E, N, K] -> (packed int32 [E, N, K/8], scale fp32 [E, N])."""
    assert w_bf16.dtype == torch.bfloat16 and w_bf16.is_contiguous() and w_bf16.dim() == 3
    E, N, K = w_bf16.shape
    dev = w_bf16.device
    packed = packed if packed is not None else torch.empty(E, N, K // 8, dtype=torch.int32, device=dev)
    scale = scale if scale is not None else torch.empty(E, N, dtype=torch.float32, device=dev)
    _check(_load().w4a8_quantize_experts(_ptr(w_bf16), E, N, K, _ptr(packed), _ptr(scale),
                                         _stream(stream)))
    return packed, scale


def w4a8_quantize_act(x_bf16: torch.Tensor, scale=None, compute_scale: bool = True, out=None,
                      ws=None, stream=None):
    """bf16 tensor -> (E4M3 codes uint8 of the same shape, fp32 scale [1])."""
    assert x_bf16.dtype == torch.bfloat16 and x_bf16.is_contiguous()
    dev = x_bf16.device
    n = x_bf16.numel()
    if scale is None:
        if not compute_scale:
            raise ValueError("a static scale tensor is required when compute_scale=False")
        scale = torch.empty(1, dtype=torch.float32, device=dev)
    out = out if out is not None else torch.empty(x_bf16.shape, dtype=torch.uint8, device=dev)
    nbytes = w4a8_quantize_act_workspace_size(n)
    ws = _ws(nbytes, dev, ws) if compute_scale else ws
    _check(_load().w4a8_quantize_act(_ptr(x_bf16), n, _ptr(scale), int(bool(compute_scale)),
                                     _ptr(_u8(out)), _ptr(ws), 0 if ws is None else ws.numel(),
                                     _stream(stream)))
    return out, scale


def moe_route(logits: torch.Tensor, k: int, renormalize: bool = True, out: RouteResult = None,
              ws=None, stream=None) -> RouteResult:
    """fp32 router logits [T, E] -> RouteResult (top-k ids/weights, histogram, permutation)."""
    assert logits.dtype == torch.float32 and logits.is_contiguous() and logits.dim() == 2
    T, E = logits.shape
    dev = logits.device
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = RouteResult(torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=dev),
                          torch.empty(E, **i32), torch.empty(E + 1, **i32),
                          torch.empty(T * k, **i32), torch.empty(T * k, **i32))
    ws = _ws(moe_route_workspace_size(T, E, k), dev, ws)
    _check(_load().moe_route(_ptr(logits), T, E, k, int(bool(renormalize)), *map(_ptr, out), _ptr(ws),
                             ws.numel(), _stream(stream)))
    return out


def moe_route_gate(hidden: torch.Tensor, gate: torch.Tensor, k: int, renormalize: bool = True,
                   out: RouteResult = None, logits=None, ws=None, stream=None):
    """bf16 hidden [T, H] and bf16 router gate [E, H] -> (RouteResult, fp32 logits [T, E] or None).
    Pass `logits` (an fp32 [T, E] tensor, or True to allocate one) to receive the logits."""
    assert hidden.dtype == torch.bfloat16 and hidden.is_contiguous() and hidden.dim() == 2
    assert gate.dtype == torch.bfloat16 and gate.is_contiguous() and gate.dim() == 2
    T, H = hidden.shape
    E = gate.shape[0]
    dev = hidden.device
    if out is None:
        i32 = dict(dtype=torch.int32, device=dev)
        out = RouteResult(torch.empty(T, k, **i32), torch.empty(T, k, dtype=torch.float32, device=dev),
                          torch.empty(E, **i32), torch.empty(E + 1, **i32),
                          torch.empty(T * k, **i32), torch.empty(T * k, **i32))
    if logits is True:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    ws = _ws(moe_route_gate_workspace_size(T, H, E, k), dev, ws)
    _check(_load().moe_route_gate(_ptr(hidden), _ptr(gate), T, H, E, k, int(bool(renormalize)),
                                  None if logits is None else _ptr(logits), *map(_ptr, out), _ptr(ws),
                                  ws.numel(), _stream(stream)))
    return out, logits


def moe_w4a8_forward(x_e4m3, a1_scale, w_gu, s_gu, w_d, s_d, a2_scale, act: int,
                     route: RouteResult, out=None, ws=None, stream=None):
    """W4A8 MoE FFN: E4M3 x [T, H] -> bf16 [T, H] (act 0 = SiLU-gated, 1 = GELU-tanh-gated)."""
    x = _u8(x_e4m3)
    T, H = x.shape
    E, I2, _ = w_gu.shape
    I = I2 // 2
    k = route.topk_ids.shape[1]
    dev = x.device
    out = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = _ws(moe_w4a8_workspace_size(T, H, I, E, k), dev, ws)
    _check(_load().moe_w4a8_forward(
        _ptr(x), _ptr(a1_scale), T, H, I, E, k, _ptr(w_gu), _ptr(s_gu), _ptr(w_d), _ptr(s_d),
        _ptr(a2_scale), int(act), _ptr(route.topk_ids), _ptr(route.topk_w), _ptr(route.counts),
        _ptr(route.offsets), _ptr(route.sorted_ids), _ptr(route.inv_perm), _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def moe_w4a8_forward_dynamic(x_e4m3, a1_scale, w_gu, s_gu, w_d, s_d, act: int, route: RouteResult,
                             out=None, a2_out=None, ws=None, stream=None):
    """moe_w4a8_forward with the intermediate scale computed from this call's h:
    returns (bf16 out [T, H], fp32 a2 [1])."""
    x = _u8(x_e4m3)
    T, H = x.shape
    E, I2, _ = w_gu.shape
    I = I2 // 2
    k = route.topk_ids.shape[1]
    dev = x.device
    out = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    a2_out = a2_out if a2_out is not None else torch.empty(1, dtype=torch.float32, device=dev)
    ws = _ws(moe_w4a8_dynamic_workspace_size(T, H, I, E, k), dev, ws)
    _check(_load().moe_w4a8_forward_dynamic(
        _ptr(x), _ptr(a1_scale), T, H, I, E, k, _ptr(w_gu), _ptr(s_gu), _ptr(w_d), _ptr(s_d),
        _ptr(a2_out), int(act), _ptr(route.topk_ids), _ptr(route.topk_w), _ptr(route.counts),
        _ptr(route.offsets), _ptr(route.sorted_ids), _ptr(route.inv_perm), _ptr(out), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out, a2_out


def fp8_linear(x_e4m3, x_scale, w_e4m3, w_scale, out=None, ws=None, stream=None):
    """Per-tensor FP8: E4M3 x [M, K] (scale [1]) x E4M3 W [N, K] (scale [1]) -> bf16 y [M, N].
    A workspace passed in must have been zero-filled before its first use here."""
    x = _u8(x_e4m3)
    w = _u8(w_e4m3)
    M, K = x.shape
    N = w.shape[0]
    dev = x.device
    out = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.zeros(max(fp8_linear_workspace_size(M, N, K), 256), dtype=torch.uint8, device=dev)
    _check(_load().fp8_linear(_ptr(x), _ptr(x_scale), M, N, K, _ptr(w), _ptr(w_scale), _ptr(out), _ptr(ws),
                              ws.numel(), _stream(stream)))
    return out


def fp8_block_linear(x_bf16, w_e4m3, w_scale_inv, out=None, xq_out=None, xs_out=None, ws=None,
                     stream=None):
    """bf16 x [M, K] x (E4M3 W [N, K], Wsi [N/128, K/128]) -> bf16 y [M, N]."""
    assert x_bf16.dtype == torch.bfloat16 and x_bf16.is_contiguous()
    M, K = x_bf16.shape
    w = _u8(w_e4m3)
    N = w.shape[0]
    dev = x_bf16.device
    out = out if out is not None else torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = _ws(fp8_block_linear_workspace_size(M, N, K), dev, ws)
    _check(_load().fp8_block_linear(_ptr(x_bf16), M, N, K, _ptr(w), _ptr(w_scale_inv), _ptr(out),
                                    _ptr(None if xq_out is None else _u8(xq_out)), _ptr(xs_out),
                                    _ptr(ws), ws.numel(), _stream(stream)))
    return out


def w4a8_set_profile_events(events) -> None:
    """Measurement hook: torch.cuda.Event objects (up to 4, enable_timing=True)
    that moe_w4a8_forward records before/after its GEMMs on this host thread;
    None or [] switches recording off."""
    events = list(events or [])
    for e in events:
        if e.cuda_event == 0:  # torch creates the CUDA event on first record
            e.record()
    arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_load().w4a8_set_profile_events(arr, len(events)))


def w4a8_selftest_wait_timeout(ws, stream=None):
    """Record a wait timeout in ws from a kernel whose barrier never completes (test hook)."""
    _check(_load().w4a8_selftest_wait_timeout(_ptr(ws), _stream(stream)))


def w4a8_device_error(ws, stream=None) -> int:
    """Read and clear a workspace's device error word (synchronizes the stream)."""
    code = ctypes.c_int(0)
    _check(_load().w4a8_device_error(_ptr(ws), ctypes.byref(code), _stream(stream)))
    return code.value
