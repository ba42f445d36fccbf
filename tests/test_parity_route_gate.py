"""moe_route_gate on the GPU against the oracle.

The logits are floating point: the GPU's fp32 sums are compared with the
oracle's exact (double) logits within a tolerance derived from fp32
accumulation. Routing is decided on the GPU's own fp32 logits, and near-ties
could go either way on logits that differ in the last bits, so the integer
outputs are checked as the unique result of routing those logits: the oracle's
router applied to the GPU logits must give the same ids, histogram and
permutation bit for bit, and the same weights within rounding."""
import numpy as np
import pytest
import torch

import oracle
from helpers import ensure_built

pytestmark = pytest.mark.gpu


def _run(T, H, E, k, renorm=True, seed=0, with_logits=True):
    ensure_built()
    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth
    inp = synth.router_gate_inputs(T, H, E, seed=seed, device="cuda")
    route, logits = lib.moe_route_gate(inp["hidden"], inp["gate"], k, renormalize=renorm,
                                       logits=True if with_logits else None)
    torch.cuda.synchronize()
    return inp, route, logits


def _check(inp, route, logits, E, k, renorm=True):
    H = inp["hidden"].shape[1]
    ref = oracle.gate_logits(inp["hidden"].cpu(), inp["gate"].cpu())
    got = logits.cpu().numpy().astype(np.float64)
    # fp32 accumulation of H exact products: error <= ~H * 2^-24 * sum|x g|
    bound = H * 2.0 ** -24 * (inp["hidden"].float().abs() @ inp["gate"].float().abs().T).cpu().numpy()
    assert np.all(np.abs(got - ref) <= bound + 1e-30), float(np.max(np.abs(got - ref) - bound))
    ids, w = oracle.route(logits.cpu().numpy(), k, renorm)
    cnt, off, srt, inv = oracle.permute(ids, E)
    assert np.array_equal(route.topk_ids.cpu().numpy(), ids)
    np.testing.assert_allclose(route.topk_w.cpu().numpy(), w, rtol=2e-6, atol=1e-7)
    assert np.array_equal(route.counts.cpu().numpy(), cnt)
    assert np.array_equal(route.offsets.cpu().numpy(), off)
    assert np.array_equal(route.sorted_ids.cpu().numpy(), srt)
    assert np.array_equal(route.inv_perm.cpu().numpy(), inv)


@pytest.mark.parametrize("T,H,E,k", [
    (16, 256, 8, 2),      # tiny
    (32, 4096, 8, 2),     # Mixtral-8x7B decode
    (32, 6144, 8, 2),     # Grok-1 decode
    (1, 6144, 8, 2),
    (7, 384, 16, 3),      # ragged token count, 128-wide slices
    (100, 512, 64, 6),    # more experts than lanes
    (3000, 256, 8, 2),    # T*k > 4096: per-token kernel + multi-block permutation
    (2048, 4096, 8, 2),   # partials too large for one launch
])
def test_route_gate_matches_oracle(T, H, E, k):
    inp, route, logits = _run(T, H, E, k, seed=T + E)
    _check(inp, route, logits, E, k)


def test_route_gate_without_renormalization_and_without_logits_out():
    inp, route, logits = _run(24, 1024, 8, 2, renorm=False, seed=7)
    _check(inp, route, logits, 8, 2, renorm=False)
    # the same call without a logits output routes identically
    import w4a8_moe_gb300 as lib
    r2, none = lib.moe_route_gate(inp["hidden"], inp["gate"], 2, renormalize=False)
    torch.cuda.synchronize()
    assert none is None
    for a, b in zip(route, r2):
        assert torch.equal(a, b)


def test_route_gate_is_deterministic_and_reuses_its_workspace():
    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth
    inp = synth.router_gate_inputs(32, 4096, 8, seed=11, device="cuda")
    ws = torch.zeros(lib.moe_route_gate_workspace_size(32, 4096, 8, 2), dtype=torch.uint8, device="cuda")
    outs = [lib.moe_route_gate(inp["hidden"], inp["gate"], 2, logits=True, ws=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for r, lg in outs[1:]:
        assert torch.equal(lg.view(torch.int32), outs[0][1].view(torch.int32))
        for a, b in zip(r, outs[0][0]):
            assert torch.equal(a, b)
    assert int(ws[:256].count_nonzero()) == 0        # the header is left zero
