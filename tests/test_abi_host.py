"""CPU-only checks of the C ABI: the library builds for sm_103a, loads, exports
every symbol include/w4a8_moe.h declares, validates arguments on the host
before touching a device, and refuses to run without an sm_103 GPU."""
import ctypes
import os
import re

import pytest
import torch

from helpers import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "w4a8_moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z][a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in {"if", "while", "sizeof"}))


@pytest.fixture(scope="module")
def lib():
    path = ensure_built()
    return ctypes.CDLL(path)


def test_header_lists_the_entry_points():
    names = declared_functions()
    for required in ["w4a8_quantize_experts", "w4a8_quantize_act", "moe_route", "moe_w4a8_forward",
                     "fp8_block_linear", "moe_w4a8_workspace_size", "w4a8_status_string",
                     "w4a8_device_error", "moe_route_gate", "moe_route_gate_workspace_size"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_targets_sm103a_only():
    from w4a8_moe_gb300 import build as b
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    lib.w4a8_status_string.restype = ctypes.c_char_p
    for code in range(8):
        assert lib.w4a8_status_string(code).startswith(b"W4A8")
    assert lib.w4a8_version() >= 100


def _vp(v):
    return ctypes.c_void_p(v)


def test_validation_happens_before_the_device(lib):
    """Null, shape, alignment and workspace errors come back without a GPU;
    a valid call without a GPU is W4A8_ERR_DEVICE (no CPU fallback)."""
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    f = lib.moe_route
    f.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P, sz, P]
    f.restype = i32
    good = _vp(0x10000)
    ws_need = lib.moe_route_workspace_size(32, 8, 2)
    # NULL
    assert f(None, 32, 8, 2, 1, good, good, good, good, good, good, good, ws_need, None) == 1
    # shape: k > E, E > 256, T < 1
    assert f(good, 32, 8, 9, 1, good, good, good, good, good, good, good, ws_need, None) == 2
    assert f(good, 32, 300, 2, 1, good, good, good, good, good, good, good, 10**9, None) == 2
    assert f(good, 0, 8, 2, 1, good, good, good, good, good, good, good, ws_need, None) == 2
    # alignment
    assert f(_vp(0x10004), 32, 8, 2, 1, good, good, good, good, good, good, good, ws_need, None) == 3
    # workspace too small
    assert f(good, 32, 8, 2, 1, good, good, good, good, good, good, good, 16, None) == 4
    # everything valid, no GPU here (or a GPU that is not sm_103): device error
    if not torch.cuda.is_available():
        assert f(good, 32, 8, 2, 1, good, good, good, good, good, good, good, ws_need, None) == 5


def test_route_gate_validation_before_the_device(lib):
    """moe_route_gate: null, shape, alignment and workspace errors without a GPU;
    valid arguments without an sm_103 GPU give W4A8_ERR_DEVICE."""
    f = lib.moe_route_gate
    P, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
    f.restype = i32
    lib.moe_route_gate_workspace_size.restype = ctypes.c_size_t
    lib.moe_route_gate_workspace_size.argtypes = [i32, i32, i32, i32]
    good = _vp(0x10000)
    need = lib.moe_route_gate_workspace_size(32, 4096, 8, 2)
    assert need > 256

    def call(x=good, T=32, H=4096, E=8, k=2, logits=None, ids=good, ws=good, nbytes=need):
        return f(x, good, T, H, E, k, 1, logits, ids, good, good, good, good, good, ws, nbytes, None)
    assert call(x=None) == 1 and call(ids=None) == 1                 # NULL
    assert call(H=4000) == 2 and call(k=9) == 2 and call(E=300) == 2  # shape (H % 128, k > E, E > 256)
    assert call(T=0) == 2
    assert call(x=_vp(0x10002)) == 3 and call(logits=_vp(0x10004)) == 3   # alignment
    assert call(nbytes=need - 1) == 4 and call(ws=None) == 4             # workspace
    if not torch.cuda.is_available():
        assert call() == 5                                              # no sm_103 device, no fallback


def test_selftest_hook_validates_its_workspace(lib):
    f = lib.w4a8_selftest_wait_timeout
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(None, None) == 1                     # NULL
    assert f(_vp(0x10004), None) == 3             # alignment
    if not torch.cuda.is_available():
        assert f(_vp(0x10000), None) == 5         # no sm_103 device


def test_forward_shape_rules(lib):
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    f = lib.moe_w4a8_forward
    f.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P, P, P, P, sz, P]
    f.restype = i32
    lib.moe_w4a8_workspace_size.restype = sz
    g = _vp(0x10000)
    ws = lib.moe_w4a8_workspace_size(32, 4096, 14336, 8, 2)
    args = lambda T, H, I, E, k, act=0: [g, g, T, H, I, E, k, g, g, g, g, g, act, g, g, g, g, g, g, g,
                                         g, ws, None]
    assert f(*args(32, 4096 + 64, 14336, 8, 2)) == 2       # H not a multiple of 128
    assert f(*args(32, 4096, 14336 + 64, 8, 2)) == 2       # I not a multiple of 128
    assert f(*args(32, 0, 14336, 8, 2)) == 2
    assert f(*args(32, 4096, 14336, 8, 3, act=2)) == 2     # unknown activation
    assert f(*args(32, 4096, 14336, 2, 3)) == 2            # k > E
    bad = args(32, 4096, 14336, 8, 2)
    bad[7] = _vp(0x10008)
    assert f(*bad) == 3


def test_workspace_sizes_are_monotone(lib):
    lib.moe_w4a8_workspace_size.restype = ctypes.c_size_t
    lib.fp8_block_linear_workspace_size.restype = ctypes.c_size_t
    a = lib.moe_w4a8_workspace_size(32, 4096, 14336, 8, 2)
    b = lib.moe_w4a8_workspace_size(64, 4096, 14336, 8, 2)
    assert 256 < a < b
    # decode: hq + gathered x + split-K partials; prefill-sized grows with T
    assert lib.moe_w4a8_workspace_size(32768, 6144, 32768, 8, 2) > 4 * 10**9
    # prefill-sized calls hold the weights unpacked once: E * 3 * I * H bytes more
    assert lib.moe_w4a8_workspace_size(129, 512, 256, 8, 2) - lib.moe_w4a8_workspace_size(128, 512, 256, 8, 2) \
        >= 8 * 3 * 256 * 512
    assert lib.fp8_block_linear_workspace_size(1, 16384, 2560) > 2560


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import w4a8_moe_gb300 as pkg
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(pkg.W4A8Error):
        pkg.moe_route_workspace_size(4, 8, 2)


def _plan(lib, T, H, I, E, k, dynamic=0, sms=152):
    f = lib.moe_w4a8_plan
    f.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    out = (ctypes.c_int32 * 8)()
    st = f(T, H, I, E, k, dynamic, sms, ctypes.cast(out, ctypes.c_void_p))
    return st, list(out)


def test_plan_of_the_decode_and_prefill_layers(lib):
    """The host planner (no GPU needed): decode-sized layers with the static
    scale run both projections in one launch, the dynamic scale and the
    256-token tiles of a prefill run them separately, after unpacking the
    weights once."""
    st, p = _plan(lib, 32, 4096, 14336, 8, 2)                  # Mixtral decode
    assert st == 0 and p[0] == 32 and p[5] == 1 and p[6] == 3
    assert (14336 // p[1]) % p[2] == 0 and p[7] == p[2] and p[3] == 0
    st, p = _plan(lib, 32, 4096, 14336, 8, 2, dynamic=1)
    assert st == 0 and p[5] == 0 and p[6] == 5                  # + the scale's quantizer
    st, p = _plan(lib, 1, 6144, 32768, 8, 2)                   # Grok single token
    assert st == 0 and p[5] == 1 and p[2] > 1                   # the down K is split to fill the SMs
    st, p = _plan(lib, 32768, 6144, 32768, 8, 2)               # Grok prefill
    assert st == 0 and p[0] == 256 and p[5] == 0 and p[6] == 5 and p[7] == 1   # + the weights' unpack


def test_plan_rejects_what_the_forward_rejects(lib):
    assert _plan(lib, 32, 4096 + 64, 14336, 8, 2)[0] == 2
    assert _plan(lib, 32, 4096 + 128, 14336 + 128, 8, 2)[0] == 0   # multiples of 128 are accepted
    assert _plan(lib, 0, 4096, 14336, 8, 2)[0] == 2
    assert _plan(lib, 32, 4096, 14336, 8, 2, sms=0)[0] == 2
    f = lib.moe_w4a8_plan
    f.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p]
    assert f(32, 4096, 14336, 8, 2, 0, 152, None) == 1


def test_plan_fits_the_workspace(lib):
    """Whatever split the planner picks, its fp32 partial sums fit the
    workspace the size query promises, and every K split divides the K blocks
    into at least two stages (the two MMA issuers)."""
    lib.moe_w4a8_workspace_size.restype = ctypes.c_size_t
    for T in (1, 2, 3, 5, 8, 16, 31, 32, 33, 64, 100, 128, 129, 300, 1024):
        for (H, I, E, k) in ((4096, 14336, 8, 2), (6144, 32768, 8, 2), (256, 512, 16, 4), (2048, 1536, 64, 6),
                             (512, 256, 256, 8), (384, 640, 8, 2), (128, 128, 4, 1), (640, 384, 16, 4)):
            for dyn in (0, 1):
                for sms in (152, 148, 7):
                    st, p = _plan(lib, T, H, I, E, k, dyn, sms)
                    assert st == 0
                    kb = -(-I // p[1])          # stages of the down K, the last one possibly partial
                    assert kb % p[2] == 0 and kb // p[2] >= 2 or p[2] == 1
                    ws = lib.moe_w4a8_workspace_size(T, H, I, E, k)
                    assert ws >= p[7] * T * k * H * 4, (T, H, I, E, k, dyn, sms, p)
                    assert p[5] in (0, 1) and (p[5] == 0 or (dyn == 0 and p[0] <= 128))


def test_static_scratch_forward_checks_like_the_regular_one(lib):
    """moe_w4a8_forward_static: the regular entry point's null / shape /
    alignment statuses in the same order, then W4A8_ERR_WORKSPACE for a
    problem larger than the built-in array, all without a device."""
    P, i32 = ctypes.c_void_p, ctypes.c_int
    f = lib.moe_w4a8_forward_static
    f.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P, P, P, P]
    f.restype = i32
    g = _vp(0x10000)
    args = lambda T, H, I, E, k, act=0, x=g: [x, g, T, H, I, E, k, g, g, g, g, g, act, g, g, g, g, g, g, g, None]
    assert f(*args(32, 4096, 14336, 8, 2, x=None)) == 1          # NULL before anything else
    assert f(*args(0, 4096, 14336, 8, 2)) == 2                   # T < 1: shape, as the regular call
    assert f(*args(32, -256, 14336, 8, 2)) == 2
    assert f(*args(32, 4096, 14336, 8, 2, act=5)) == 2
    assert f(*args(32, 4096, 14336, 8, 2, x=_vp(0x10001))) == 3  # alignment
    assert f(*args(32768, 6144, 32768, 8, 2)) == 4               # needs gigabytes of scratch
    if not torch.cuda.is_available():
        assert f(*args(32, 4096, 14336, 8, 2)) == 5              # fits, but no sm_103 device
    e = lib.moe_w4a8_forward_static_error
    e.argtypes = [P, P]
    e.restype = i32
    assert e(None, None) == 1


def test_workspace_layout_hook(lib):
    """The intermediate codes sit inside the workspace the size query promises."""
    i64 = ctypes.c_int64
    f = lib.moe_w4a8_workspace_layout
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    lib.moe_w4a8_workspace_size.restype = ctypes.c_size_t
    for (T, H, I, E, k) in ((16, 256, 512, 8, 2), (32, 4096, 14336, 8, 2), (300, 256, 256, 8, 2)):
        off = (i64 * 2)()
        assert f(T, H, I, E, k, ctypes.cast(off, ctypes.c_void_p)) == 0
        hq, xp = off[0], off[1]
        ws = lib.moe_w4a8_workspace_size(T, H, I, E, k)
        assert 256 <= xp and xp + T * k * H <= hq and hq + T * k * I <= ws
        assert hq % 256 == 0 and xp % 256 == 0
    assert f(0, 256, 512, 8, 2, ctypes.cast((i64 * 2)(), ctypes.c_void_p)) == 2
    assert f(16, 256, 512, 8, 2, None) == 1
