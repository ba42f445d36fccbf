"""GPU parity of the quantizers and the router against the oracle: every code,
packed word, scale, index and permutation entry must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built, to_np_bits
from w4a8_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def lib():
    import w4a8_moe_gb300 as m
    return m


@pytest.mark.parametrize("E,N,K", [(3, 40, 256), (2, 128, 4104), (1, 1, 8)])
def test_quantize_experts_bit_exact(E, N, K):
    g = torch.Generator(device="cuda").manual_seed(E * 1000 + K)
    w = (torch.randn(E, N, K, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w[0, 0] = 0                                    # all-zero channel -> scale 1
    if N > 2:
        w[0, 1, :8] = torch.tensor([0.875, 0.3125, 0.4375, -0.3125, 0.0625, 0.1875, 0, 0],
                                   device="cuda").to(torch.bfloat16)   # exact half-way ties
        w[0, 1, 8:] = 0
    packed, scale = lib().w4a8_quantize_experts(w.contiguous())
    o_p, o_s = oracle.quantize_experts(to_np_bits(w))
    assert np.array_equal(packed.cpu().numpy(), o_p)
    assert np.array_equal(scale.cpu().numpy(), o_s)


def test_quantize_experts_mixtral_shape_sampled():
    w = synth.moe_weights(4096, 14336, 1, device="cuda")["w_d"]        # [1, 4096, 14336]
    packed, scale = lib().w4a8_quantize_experts(w)
    rows = [0, 1, 777, 4095]
    sub = to_np_bits(w[0, rows])[None]
    o_p, o_s = oracle.quantize_experts(sub)
    assert np.array_equal(packed[0, rows].cpu().numpy(), o_p[0])
    assert np.array_equal(scale[0, rows].cpu().numpy(), o_s[0])


@pytest.mark.parametrize("T,H", [(16, 256), (32, 4096), (3, 6144), (4096, 6144)])
def test_quantize_act_bit_exact(T, H):
    x = synth.moe_inputs(T, H, 256, 1, device="cuda", weights=False)["x"]
    xq, s = lib().w4a8_quantize_act(x, compute_scale=True)
    hx = to_np_bits(x)
    s_ref = oracle.act_scale(hx)
    assert s.item() == s_ref
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_act(hx, s_ref))
    # static scale: a smaller scale saturates part of the tensor
    st = torch.tensor([s_ref * 0.25], dtype=torch.float32, device="cuda")
    xq2, _ = lib().w4a8_quantize_act(x, scale=st, compute_scale=False)
    assert np.array_equal(xq2.cpu().numpy(), oracle.quantize_act(hx, float(st.item())))


def test_quantize_act_zero_tensor():
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    xq, s = lib().w4a8_quantize_act(x, compute_scale=True)
    assert s.item() == 1.0 and not xq.any()


def _route_check(logits, k, renorm=True):
    r = lib().moe_route(logits, k, renormalize=renorm)
    torch.cuda.synchronize()
    h = logits.cpu().numpy()
    ids, w = oracle.route(h, k, renorm)
    E = logits.shape[1]
    counts, offsets, srt, inv = oracle.permute(ids, E)
    assert np.array_equal(r.topk_ids.cpu().numpy(), ids)
    np.testing.assert_allclose(r.topk_w.cpu().numpy(), w, rtol=3e-6, atol=1e-7)
    assert np.array_equal(r.counts.cpu().numpy(), counts)
    assert np.array_equal(r.offsets.cpu().numpy(), offsets)
    assert np.array_equal(r.sorted_ids.cpu().numpy(), srt)
    assert np.array_equal(r.inv_perm.cpu().numpy(), inv)
    return counts


@pytest.mark.parametrize("T,E,k,bias", [(16, 8, 2, 0.0), (32, 8, 2, 0.5), (1, 8, 2, 0.0),
                                        (1000, 64, 6, 0.0), (2048, 8, 2, 0.0), (2049, 8, 2, 0.0),
                                        (32768, 8, 2, 1.0), (3000, 256, 8, 0.0), (5, 1, 1, 0.0),
                                        (40, 256, 10, 0.0)])
def test_route_bit_exact(T, E, k, bias):
    logits = synth.moe_inputs(T, 256, 256, E, bias_std=bias, device="cuda", weights=False)["logits"]
    counts = _route_check(logits, k)
    assert counts.sum() == T * k


def test_route_ties_and_empty_experts():
    g = torch.Generator(device="cuda").manual_seed(5)
    logits = torch.randint(-2, 2, (777, 16), generator=g, device="cuda").float()
    logits[:, 3] = -100.0                           # expert 3 never chosen
    counts = _route_check(logits.contiguous(), 4)
    assert counts[3] == 0
    _route_check(logits.contiguous(), 4, renorm=False)


def test_route_all_tokens_one_expert():
    logits = torch.zeros(300, 8, device="cuda")
    logits[:, 5] = 10.0
    counts = _route_check(logits, 1)
    assert counts[5] == 300
