"""moe_w4a8_forward_dynamic against the oracle: the intermediate scale is
computed on the device as max|h|/448 over every assignment of the call.

The GPU's h is fp32 (the oracle's exact h in double), so its scale is
compared with the oracle's within fp32 rounding, and the output is compared
with the oracle run at the GPU's scale (the scale decides every E4M3 code of
hq, so both sides take those decisions from the same value)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import MoECase, assert_close, bf16_to_f64, ensure_built, oracle_threads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,I,E,k,act,bias", [
    (16, 256, 512, 8, 2, 0, 0.0),        # tiny
    (33, 256, 256, 8, 2, 1, 0.0),        # ragged, GELU
    (32, 4096, 14336, 8, 2, 0, 0.5),     # Mixtral-8x7B decode
    (200, 384, 640, 8, 2, 1, 0.0),       # prefill plan (weights unpacked once), ragged K stages
])
def test_dynamic_scale_forward(T, H, I, E, k, act, bias):
    ensure_built()
    import w4a8_moe_gb300 as lib
    case = MoECase(T, H, I, E, k, act, bias_std=bias, seed=T, calib_tokens=T)   # oracle scale: all tokens
    ws = torch.zeros(lib.moe_w4a8_dynamic_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    out, a2 = lib.moe_w4a8_forward_dynamic(case.xq, case.a1, case.w_gu, case.s_gu, case.w_d, case.s_d,
                                           case.act, case.route, ws=ws)
    torch.cuda.synchronize()
    s2 = a2.item()
    assert abs(s2 - case.s2) <= 1e-4 * case.s2, (s2, case.s2)
    ref = oracle.moe_forward(case.o_xq, case.o_s1, case.o_pgu, case.o_sgu, case.o_pd, case.o_sd,
                             float(np.float32(s2)), case.act, case.o_ids, case.o_w, nthreads=oracle_threads())
    assert_close(bf16_to_f64(out), ref, f"dynamic T{T} H{H} I{I}")
    # a second call on the same workspace recomputes the scale from zero
    out2, a2b = lib.moe_w4a8_forward_dynamic(case.xq, case.a1, case.w_gu, case.s_gu, case.w_d, case.s_d,
                                             case.act, case.route, ws=ws)
    torch.cuda.synchronize()
    assert a2b.item() == s2
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert lib.w4a8_device_error(ws) == 0
