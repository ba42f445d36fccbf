"""moe_w4a8_forward_static: the MoE forward for callers that cannot allocate.

Callers such as plugins inside a host application that owns all device
memory, or hot loops that must never call cudaMalloc, cannot hand the library
a workspace. This entry point uses a scratch array built into the library
instead. The test calls it through the C ABI (ctypes on the shared library)
twice in a row, on two different layers, and checks each result against the
regular entry point (moe_w4a8_forward with a caller workspace) within the
parity tolerance of the other tests; it also checks that a problem too large
for the built-in scratch is refused. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from helpers import MoECase, assert_close, bf16_to_f64, ensure_built

pytestmark = pytest.mark.gpu

W4A8_ERR_WORKSPACE = 4


def _entry():
    lib = ctypes.CDLL(ensure_built())
    f = lib.moe_w4a8_forward_static
    P, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, i32, P, P, P, P, P, P, P, P]
    f.restype = i32
    return f


def _call(f, case: MoECase, out: torch.Tensor) -> int:
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    r = case.route
    st = f(p(case.xq), p(case.a1), case.T, case.H, case.I, case.E, case.k, p(case.w_gu), p(case.s_gu),
           p(case.w_d), p(case.s_d), p(case.a2), case.act, p(r.topk_ids), p(r.topk_w), p(r.counts),
           p(r.offsets), p(r.sorted_ids), p(r.inv_perm), p(out),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def test_static_scratch_forward_matches_workspace_forward():
    f = _entry()
    cases = [MoECase(16, 256, 512, 8, 2, 0, seed=1),              # tiny SiLU layer
             MoECase(32, 2048, 4096, 8, 2, 1, bias_std=0.5, seed=2)]  # decode-shaped GELU layer
    for case in cases:                                            # two calls in a row
        ref = case.run_gpu()
        out = torch.empty_like(ref)
        assert _call(f, case, out) == 0
        assert_close(bf16_to_f64(out), bf16_to_f64(ref), f"static scratch T{case.T} H{case.H}")
    # the array keeps the previous call's contents: a repeat of the first layer
    # after the larger one must still agree
    again = torch.empty_like(cases[0].run_gpu())
    assert _call(f, cases[0], again) == 0
    assert_close(bf16_to_f64(again), bf16_to_f64(cases[0].run_gpu()), "static scratch repeat")


def test_static_scratch_refuses_oversized_problems():
    f = _entry()
    none = ctypes.c_void_p(0)
    # a 32768-token prefill-sized layer needs gigabytes of scratch
    args = [none, none, 32768, 6144, 32768, 8, 2] + [none] * 5 + [1] + [none] * 7 + [none]
    assert f(*args) == W4A8_ERR_WORKSPACE
