"""moe_w4a8_forward_static: the MoE forward for callers that cannot allocate.

Callers such as plugins inside a host application that owns all device
memory, or hot loops that must never call cudaMalloc, cannot hand the library
a workspace. This entry point uses a scratch array built into the library
instead. The test calls it through the C ABI (ctypes on the shared library)
on several layers in a row and checks each result against the regular entry
point (moe_w4a8_forward with a caller workspace) within the parity tolerance
of the other tests, and against the oracle; it checks that the calls allocate
no device memory, that the array's error word reads clean, and that a problem
too large for the built-in scratch is refused. The layers cover both launch
plans of the forward: both projections in one launch (up to 128 tokens) and
the two-launch plan of prefill-sized calls (256-token tiles, weights unpacked
once into the scratch). This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import MoECase, assert_close, bf16_to_f64, ensure_built

pytestmark = pytest.mark.gpu

W4A8_ERR_WORKSPACE = 4


def _lib():
    lib = ctypes.CDLL(ensure_built())
    P, i32 = ctypes.c_void_p, ctypes.c_int
    f = lib.moe_w4a8_forward_static
    f.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P, P, P, P]
    f.restype = i32
    e = lib.moe_w4a8_forward_static_error
    e.argtypes = [P, P]
    e.restype = i32
    return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(lib, case: MoECase, out: torch.Tensor) -> int:
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    r = case.route
    st = lib.moe_w4a8_forward_static(p(case.xq), p(case.a1), case.T, case.H, case.I, case.E, case.k, p(case.w_gu),
                                     p(case.s_gu), p(case.w_d), p(case.s_d), p(case.a2), case.act, p(r.topk_ids),
                                     p(r.topk_w), p(r.counts), p(r.offsets), p(r.sorted_ids), p(r.inv_perm),
                                     p(out), _stream())
    torch.cuda.synchronize()
    return st


def _static_error(lib) -> int:
    code = ctypes.c_int(-1)
    assert lib.moe_w4a8_forward_static_error(ctypes.byref(code), _stream()) == 0
    return code.value


def test_static_scratch_forward_matches_workspace_forward_and_oracle():
    import w4a8_moe_gb300 as w
    lib = _lib()
    cases = [MoECase(16, 256, 512, 8, 2, 0, seed=1),                   # tiny SiLU layer, one launch
             MoECase(32, 2048, 4096, 8, 2, 1, bias_std=0.5, seed=2),   # decode-shaped GELU layer, one launch
             MoECase(200, 512, 512, 8, 2, 0, seed=3)]                  # 256-token tiles: two launches
    assert [w.moe_w4a8_plan(c.T, c.H, c.I, c.E, c.k)["one_launch"] for c in cases] == [1, 1, 0]
    outs = [torch.empty(c.T, c.H, dtype=torch.bfloat16, device="cuda") for c in cases]
    first = [torch.empty_like(o) for o in outs]
    # first pass: the first call in this context sets up the array's address,
    # and every kernel the layers use gets loaded
    for case, out in zip(cases, first):
        assert _call(lib, case, out) == 0
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    for case, out in zip(cases, outs):                 # calls in a row on the shared array
        assert _call(lib, case, out) == 0
    assert torch.cuda.memory_allocated() == alloc0, "the static entry point allocated through torch"
    assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated during the static calls"
    assert _static_error(lib) == 0
    for a, b in zip(first, outs):                      # same inputs, same bits, whatever ran before
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for case, out in zip(cases, outs):
        ref = case.run_gpu()
        assert_close(bf16_to_f64(out), bf16_to_f64(ref), f"static scratch vs moe_w4a8_forward T{case.T} H{case.H}")
        toks = sorted(set([0, case.T - 1] + list(range(0, case.T, max(1, case.T // 24)))))
        assert_close(bf16_to_f64(out[toks]), case.oracle_out(toks), f"static scratch vs oracle T{case.T} H{case.H}")
    # the array keeps the previous call's contents: a repeat of the first layer
    # after the larger ones must still agree with the first result
    again = torch.empty_like(outs[0])
    assert _call(lib, cases[0], again) == 0
    assert torch.equal(again.view(torch.int16), outs[0].view(torch.int16))


def test_static_scratch_mixtral_sized_128_tokens():
    """128 tokens of a Mixtral-shaped layer (about 21 MiB of scratch, the down
    projection split over several fp32 partial sums) fit."""
    lib = _lib()
    case = MoECase(128, 4096, 14336, 8, 2, 0, bias_std=0.5, seed=4, calib_tokens=16)
    out = torch.empty(case.T, case.H, dtype=torch.bfloat16, device="cuda")
    assert _call(lib, case, out) == 0
    ref = case.run_gpu()
    assert_close(bf16_to_f64(out), bf16_to_f64(ref), "static scratch vs moe_w4a8_forward T128 Mixtral-shaped")
    toks = [0, 5, 64, 127]
    assert_close(bf16_to_f64(out[toks]), case.oracle_out(toks), "static scratch vs oracle T128 Mixtral-shaped")
    assert _static_error(lib) == 0


def test_static_scratch_refuses_oversized_problems():
    lib = _lib()
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    g = ctypes.c_void_p(buf.data_ptr())
    # a 32768-token prefill-sized layer needs gigabytes of scratch
    args = [g, g, 32768, 6144, 32768, 8, 2] + [g] * 5 + [1] + [g] * 7 + [_stream()]
    assert lib.moe_w4a8_forward_static(*args) == W4A8_ERR_WORKSPACE
