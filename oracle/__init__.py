"""CPU oracle for the W4A8 MoE FFN and the block-FP8 dense projection.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the library in
``w4a8_moe_gb300`` never does. The arithmetic lives in ``w4a8_oracle.c``
(plain C, no CUDA), which shares no code with the CUDA path; this module only
compiles it with gcc and marshals numpy arrays into it.

Every function cites the passage of the pages it follows in the C source:
  [P1] "ROCm: enable trillion-parameter MoE models with INT4-FP8 single node"
  [P2] "[AMD][Quantization] Add int4fp8_moe online quantization on ROCm"
  [P3] "qwen4_exp: serve the block-FP8 dense projections natively (+25% decode)"
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_w4a8.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE fp32/fp64 semantics)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
            sig = {
                "orc_e4m3_to_double": (f64, [ctypes.c_uint8]),
                "orc_e4m3_from_float": (ctypes.c_uint8, [f32]),
                "orc_e4m3_encode_array": (None, [P, i64, P]),
                "orc_e4m3_decode_array": (None, [P, i64, P]),
                "orc_bf16_to_float": (f32, [ctypes.c_uint16]),
                "orc_double_to_bf16": (ctypes.c_uint16, [f64]),
                "orc_bf16_array_from_double": (None, [P, i64, P]),
                "orc_quantize_experts": (None, [P, i32, i32, i32, P, P]),
                "orc_unpack_int4": (None, [P, i64, P]),
                "orc_act_scale": (f32, [P, i64]),
                "orc_quantize_act": (None, [P, i64, f32, P]),
                "orc_route": (None, [P, i32, i32, i32, i32, P, P]),
                "orc_gate_logits": (None, [P, P, i32, i32, i32, P]),
                "orc_permute": (None, [P, i32, i32, i32, P, P, P, P]),
                "orc_moe_forward": (None, [P, f32, i32, i32, i32, i32, i32, P, P, P, P, f32, i32,
                                           P, P, P, i32, P, i32]),
                "orc_moe_hidden_codes": (None, [P, f32, i32, i32, i32, i32, i32, P, P, f32, i32, P, P,
                                                i32, P, i32]),
                "orc_moe_hidden_absmax": (f64, [P, f32, i32, i32, i32, i32, i32, P, P, i32, P, P,
                                                i32, i32]),
                "orc_block_quantize_weight": (None, [P, i32, i32, P, P]),
                "orc_block_quantize_act": (None, [P, i32, i32, P, P]),
                "orc_block_linear": (None, [P, P, i32, i32, i32, P, P, P, i32, P, i32]),
                "orc_fp8_linear": (None, [P, f32, i32, i32, i32, P, f32, P, i32, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a) -> np.ndarray:
    """bf16 input as uint16 bit patterns (accepts a torch bf16 tensor or uint16 array)."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        return a.contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
    return _c(a, np.uint16)


def cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


# --- formats -----------------------------------------------------------------

def e4m3_to_double(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e4m3_from_float(v) -> np.ndarray:
    x = _c(v, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def bf16_from_double(d) -> np.ndarray:
    x = _c(d, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_array_from_double(_p(x), x.size, _p(out))
    return out


def bf16_to_float(bits) -> np.ndarray:
    b = _bits16(bits)
    return (b.astype(np.uint32) << 16).view(np.float32)


# --- INT4 experts ------------------------------------------------------------

def quantize_experts(w_bf16):
    """bf16 [E, N, K] -> (packed int32 [E, N, K/8], scale fp32 [E, N])."""
    w = _bits16(w_bf16)
    E, N, K = w.shape
    packed = np.empty((E, N, K // 8), np.int32)
    scale = np.empty((E, N), np.float32)
    _load().orc_quantize_experts(_p(w), E, N, K, _p(packed), _p(scale))
    return packed, scale


def unpack_int4(packed) -> np.ndarray:
    p = _c(packed, np.int32)
    q = np.empty(p.shape[:-1] + (p.shape[-1] * 8,), np.int8)
    _load().orc_unpack_int4(_p(p), p.size, _p(q))
    return q


# --- activations -------------------------------------------------------------

def act_scale(x_bf16) -> float:
    x = _bits16(x_bf16)
    return float(_load().orc_act_scale(_p(x), x.size))


def quantize_act(x_bf16, scale: float) -> np.ndarray:
    x = _bits16(x_bf16)
    out = np.empty(x.shape, np.uint8)
    _load().orc_quantize_act(_p(x), x.size, ctypes.c_float(scale), _p(out))
    return out


# --- routing -----------------------------------------------------------------

def gate_logits(hidden_bf16, gate_bf16) -> np.ndarray:
    """bf16 bits hidden [T, H] and gate [E, H] -> double logits [T, E]."""
    x = _bits16(hidden_bf16)
    g = _bits16(gate_bf16)
    T, H = x.shape
    E = g.shape[0]
    out = np.empty((T, E), np.float64)
    _load().orc_gate_logits(_p(x), _p(g), T, H, E, _p(out))
    return out


def route(logits, k: int, renorm: bool = True):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().orc_route(_p(lg), T, E, k, int(bool(renorm)), _p(ids), _p(w))
    return ids, w


def permute(ids, E: int):
    i = _c(ids, np.int32)
    T, k = i.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_ids = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    _load().orc_permute(_p(i), T, k, E, _p(counts), _p(offsets), _p(sorted_ids), _p(inv))
    return counts, offsets, sorted_ids, inv


# --- MoE forward -------------------------------------------------------------

def moe_forward(xq, s1, w_gu, s_gu, w_d, s_d, s2, act, ids, topk_w, tokens=None, nthreads=1):
    """Exact-integer W4A8 MoE forward for the listed tokens -> float64 [len(tokens), H]."""
    xq = _c(xq, np.uint8)
    T, H = xq.shape
    w_gu = _c(w_gu, np.int32)
    w_d = _c(w_d, np.int32)
    E, I2, _ = w_gu.shape
    I = I2 // 2
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    topk_w = _c(topk_w, np.float64)
    s_gu = _c(s_gu, np.float32)
    s_d = _c(s_d, np.float32)
    tok = _c(np.arange(T) if tokens is None else tokens, np.int32)
    out = np.empty((tok.size, H), np.float64)
    _load().orc_moe_forward(_p(xq), ctypes.c_float(s1), T, H, I, E, k, _p(w_gu), _p(s_gu), _p(w_d),
                            _p(s_d), ctypes.c_float(s2), int(act), _p(ids), _p(topk_w), _p(tok),
                            tok.size, _p(out), int(nthreads))
    return out


def moe_hidden_codes(xq, s1, w_gu, s_gu, s2, act, ids, tokens, nthreads=1) -> np.ndarray:
    """E4M3 codes of the intermediate activation h / s2 for the listed tokens:
    uint8 [len(tokens), k, I], assignment (token, j), i in natural order."""
    xq = _c(xq, np.uint8)
    T, H = xq.shape
    w_gu = _c(w_gu, np.int32)
    E, I2, _ = w_gu.shape
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    s_gu = _c(s_gu, np.float32)
    tok = _c(tokens, np.int32)
    out = np.empty((tok.size, k, I2 // 2), np.uint8)
    _load().orc_moe_hidden_codes(_p(xq), ctypes.c_float(s1), T, H, I2 // 2, E, k, _p(w_gu), _p(s_gu),
                                 ctypes.c_float(s2), int(act), _p(ids), _p(tok), tok.size, _p(out),
                                 int(nthreads))
    return out


def moe_hidden_scale(xq, s1, w_gu, s_gu, act, ids, tokens, nthreads=1) -> float:
    """Static scale of the intermediate activation: max|h| / 448 over the listed tokens."""
    xq = _c(xq, np.uint8)
    T, H = xq.shape
    w_gu = _c(w_gu, np.int32)
    E, I2, _ = w_gu.shape
    ids = _c(ids, np.int32)
    s_gu = _c(s_gu, np.float32)
    tok = _c(tokens, np.int32)
    m = _load().orc_moe_hidden_absmax(_p(xq), ctypes.c_float(s1), T, H, I2 // 2, E, ids.shape[1],
                                      _p(w_gu), _p(s_gu), int(act), _p(ids), _p(tok), tok.size,
                                      int(nthreads))
    return float(np.float32(m) / np.float32(448.0)) if m > 0 else 1.0


# --- block-FP8 ---------------------------------------------------------------

def block_quantize_weight(w_bf16):
    w = _bits16(w_bf16)
    N, K = w.shape
    wq = np.empty((N, K), np.uint8)
    wsi = np.empty((N // 128, K // 128), np.float32)
    _load().orc_block_quantize_weight(_p(w), N, K, _p(wq), _p(wsi))
    return wq, wsi


def block_quantize_act(x_bf16):
    x = _bits16(x_bf16)
    M, K = x.shape
    xq = np.empty((M, K), np.uint8)
    xs = np.empty((M, K // 128), np.float32)
    _load().orc_block_quantize_act(_p(x), M, K, _p(xq), _p(xs))
    return xq, xs


def block_linear(xq, xs, wq, wsi, rows=None, nthreads=1) -> np.ndarray:
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    wq = _c(wq, np.uint8)
    wsi = _c(wsi, np.float32)
    M, K = xq.shape
    N = wq.shape[0]
    r = _c(np.arange(M) if rows is None else rows, np.int32)
    y = np.empty((r.size, N), np.float64)
    _load().orc_block_linear(_p(xq), _p(xs), M, N, K, _p(wq), _p(wsi), _p(r), r.size, _p(y),
                             int(nthreads))
    return y


def fp8_linear(xq, sx: float, wq, sw: float, rows=None) -> np.ndarray:
    """Per-tensor FP8 linear: codes xq [M, K], wq [N, K] with scales sx, sw -> double y [rows, N]."""
    xq = _c(xq, np.uint8)
    wq = _c(wq, np.uint8)
    M, K = xq.shape
    N = wq.shape[0]
    r = _c(np.arange(M) if rows is None else rows, np.int32)
    y = np.empty((r.size, N), np.float64)
    _load().orc_fp8_linear(_p(xq), float(sx), M, N, K, _p(wq), float(sw), _p(r), r.size, _p(y))
    return y
