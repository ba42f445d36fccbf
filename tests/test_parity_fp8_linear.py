"""fp8_linear (per-tensor FP8 dense projection) on the GPU against the oracle.

Inputs are quantized on the GPU with w4a8_quantize_act (activations and, once,
the weight) and checked bit-exactly against the oracle's tensor-wise quantizer;
the oracle then evaluates y = sx * sw * sum_k dec(xq) dec(wq) exactly from the
same codes, and the bf16 output must match within the parity tolerance."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_to_f64, ensure_built, to_np_bits

pytestmark = pytest.mark.gpu


def _case(M, N, K, seed=0):
    ensure_built()
    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth
    inp = synth.fp8_linear_inputs(M, N, K, seed=seed, device="cuda")
    xq, sx = lib.w4a8_quantize_act(inp["x"])
    wq, sw = lib.w4a8_quantize_act(inp["w"])
    torch.cuda.synchronize()
    # the quantized inputs are the oracle's, bit for bit
    o_sw = oracle.act_scale(to_np_bits(inp["w"]))
    assert sw.item() == o_sw
    o_wq = oracle.quantize_act(to_np_bits(inp["w"]), o_sw)
    assert np.array_equal(wq.cpu().numpy().reshape(-1), o_wq.reshape(-1))
    o_sx = oracle.act_scale(to_np_bits(inp["x"]))
    assert sx.item() == o_sx
    assert np.array_equal(xq.cpu().numpy().reshape(-1),
                          oracle.quantize_act(to_np_bits(inp["x"]), o_sx).reshape(-1))
    return lib, xq, sx, wq, sw


@pytest.mark.parametrize("N,K", [(8192, 6144), (6144, 6144)])   # Grok-1 qkv_proj, o_proj
@pytest.mark.parametrize("M", [1, 8, 64])
def test_fp8_linear_decode_shapes(M, N, K):
    lib, xq, sx, wq, sw = _case(M, N, K, seed=M)
    y = lib.fp8_linear(xq, sx, wq, sw)
    torch.cuda.synchronize()
    ref = oracle.fp8_linear(xq.cpu().numpy(), sx.item(), wq.cpu().numpy(), sw.item())
    assert_close(bf16_to_f64(y), ref, f"fp8_linear M{M} N{N} K{K}")


@pytest.mark.parametrize("N,K", [(8192, 6144), (6144, 6144)])
def test_fp8_linear_prefill_sampled_rows(N, K):
    M = 4096
    lib, xq, sx, wq, sw = _case(M, N, K, seed=3)
    y = lib.fp8_linear(xq, sx, wq, sw)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 255, 256, 1000, 2047, 2048, 3333, 4094, 4095], np.int32)
    ref = oracle.fp8_linear(xq.cpu().numpy(), sx.item(), wq.cpu().numpy(), sw.item(), rows=rows)
    assert_close(bf16_to_f64(y)[rows], ref, f"fp8_linear M{M} N{N} K{K} sampled rows")


@pytest.mark.parametrize("M,N,K", [(5, 256, 384), (37, 384, 256), (100, 128, 1024),
                                   (200, 256, 512), (300, 384, 384), (17, 1024, 2048),
                                   (10, 2048, 4096)])   # stream-K, ~10 segments per tile
def test_fp8_linear_ragged(M, N, K):
    lib, xq, sx, wq, sw = _case(M, N, K, seed=M + N)
    y = lib.fp8_linear(xq, sx, wq, sw)
    torch.cuda.synchronize()
    ref = oracle.fp8_linear(xq.cpu().numpy(), sx.item(), wq.cpu().numpy(), sw.item())
    assert_close(bf16_to_f64(y), ref, f"fp8_linear M{M} N{N} K{K}")


def test_fp8_linear_reuses_its_workspace_deterministically():
    lib, xq, sx, wq, sw = _case(8, 6144, 6144, seed=9)
    ws = torch.zeros(lib.fp8_linear_workspace_size(8, 6144, 6144), dtype=torch.uint8, device="cuda")
    ys = [lib.fp8_linear(xq, sx, wq, sw, ws=ws) for _ in range(3)]
    torch.cuda.synchronize()
    assert lib.w4a8_device_error(ws) == 0
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
