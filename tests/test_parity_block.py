"""GPU parity of the block-FP8 projection against the oracle: the per-token
128-column activation codes and scales bit-exact, y within the fp tolerance."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_to_f64, ensure_built, oracle_threads, to_np_bits
from w4a8_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


_weights = {}


def block_weights(N, K):
    """Checkpoint-style weights: bf16 N(0, 0.02) quantized per 128x128 block by the
    oracle's input-preparation quantizer (the format the projection consumes)."""
    if (N, K) not in _weights:
        w = synth.block_fp8_inputs(1, N, K, device="cuda")["w"]
        wq, wsi = oracle.block_quantize_weight(to_np_bits(w))
        _weights[(N, K)] = (wq, wsi, torch.from_numpy(wq).cuda(), torch.from_numpy(wsi).cuda())
    return _weights[(N, K)]


def run(M, N, K, rows=None, seed=0):
    import w4a8_moe_gb300 as lib
    wq, wsi, d_wq, d_wsi = block_weights(N, K)
    x = synth.block_fp8_inputs(M, 128, K, seed=seed, device="cuda")["x"]
    xq = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    xs = torch.empty(M, K // 128, dtype=torch.float32, device="cuda")
    y = lib.fp8_block_linear(x, d_wq, d_wsi, xq_out=xq, xs_out=xs)
    torch.cuda.synchronize()
    o_xq, o_xs = oracle.block_quantize_act(to_np_bits(x))
    assert np.array_equal(xq.cpu().numpy(), o_xq)
    assert np.array_equal(xs.cpu().numpy(), o_xs)
    if rows is None:
        rows = list(range(M))
    ref = oracle.block_linear(o_xq, o_xs, wq, wsi, rows=rows, nthreads=oracle_threads())
    return assert_close(bf16_to_f64(y[rows]), ref, f"M{M} N{N} K{K}")


@pytest.mark.parametrize("N,K", synth.BLOCK_FP8_SHAPES)
@pytest.mark.parametrize("M", synth.BLOCK_FP8_M)
def test_block_fp8_configs(M, N, K):
    # sampled rows: every 32-row quadrant of a 128-token tile (its TMEM lane
    # group) appears, in the first, a middle and the last tile
    rows = None if M <= 8 else sorted({r for r in (0, 1, 37, 70, 101, 127, M // 2 + 45, M - 90, M - 1)
                                       if 0 <= r < M})
    run(M, N, K, rows=rows)


@pytest.mark.parametrize("M,N,K", [(3, 128, 128), (17, 256, 384), (100, 384, 1024),
                                   (130, 128, 256), (65, 512, 2560),
                                   (300, 768, 384),     # 256-row weight tiles, 3 token tiles, ragged last
                                   (257, 640, 1024)])   # 128-row weight tiles (N % 256 = 128), a 1-row tile
def test_block_fp8_ragged(M, N, K):
    run(M, N, K, seed=M)


def test_block_fp8_scale_by_power_of_two_is_exact():
    import w4a8_moe_gb300 as lib
    wq, wsi, d_wq, d_wsi = block_weights(256, 512)
    x = synth.block_fp8_inputs(8, 128, 512, device="cuda")["x"]
    y1 = lib.fp8_block_linear(x, d_wq, d_wsi).float()
    y2 = lib.fp8_block_linear(x, d_wq, d_wsi * 4.0).float()
    assert torch.equal(y1 * 4.0, y2)
