"""GPU parity of the W4A8 MoE forward against the oracle on the same seeded
inputs: integer stages bit-exact, the bf16 output within rel-L2 <= 2e-3 and
max-abs <= 1e-2 * max|ref| of the oracle's float64 result."""
import numpy as np
import pytest
import torch

from helpers import MoECase, QuantizedWeights, assert_close, bf16_to_f64, compare_codes, ensure_built
from w4a8_moe_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def run_case(case: MoECase, tokens=None, what=""):
    case.check_integer_parts()
    out = case.run_gpu()
    ref = case.oracle_out(tokens)
    got = bf16_to_f64(out if tokens is None else out[list(tokens)])
    return assert_close(got, ref, what)


def test_tiny_layer_all_tokens():
    s = synth.MOE_SHAPES["tiny"]
    case = MoECase(s.T, s.H, s.I, s.E, s.k, s.act)
    case.check_integer_parts()
    ws = _workspace(case)
    out = case.run_gpu(ws=ws)
    check_hidden_codes(case, ws, list(range(s.T)), "tiny")
    assert_close(bf16_to_f64(out), case.oracle_out(), "tiny")


@pytest.mark.parametrize("T,H,I,E,k,act", [
    (1, 256, 256, 8, 2, 0),       # single token
    (3, 256, 512, 2, 1, 1),       # k = 1, two experts, GELU
    (33, 256, 256, 8, 2, 0),      # ragged: 64-token tile
    (100, 512, 256, 4, 2, 1),     # 128-token tile
    (300, 256, 256, 8, 2, 0),     # 256-token tiles, several per expert
    (7, 256, 256, 1, 1, 0),       # E = 1, k = 1: dense W4A8 MLP
    (64, 768, 512, 16, 4, 1),     # k = 4, 16 experts, H not a power of two
    (64, 256, 256, 256, 8, 0),    # the most experts the boundary accepts, top-8
    (5, 128, 128, 4, 2, 0),       # the smallest H and I: one half-filled K stage
    (24, 384, 640, 8, 2, 1),      # H, I = 128 mod 256: a ragged last K stage in both GEMMs
    (40, 640, 384, 8, 2, 0),      # the same, 64-token tile
    (100, 384, 384, 8, 2, 1),     # the same, 128-token tile
    (3, 640, 640, 8, 2, 0),       # the same, stream-K down projection (T*k <= E)
    (150, 384, 640, 8, 2, 0),     # prefill plan (256-token tiles, weights unpacked once), K = 128 stages
])
def test_shapes_and_tails(T, H, I, E, k, act):
    case = MoECase(T, H, I, E, k, act, seed=T + E)
    run_case(case, what=f"T{T} H{H} I{I} E{E} k{k}")


@pytest.mark.parametrize("T,H,I,E,k", [
    (1, 4096, 14336, 8, 2),   # Mixtral-shaped single token: 2 of 8 experts active
    (3, 2048, 4096, 8, 2),    # 6 assignments over 8 experts
    (4, 2048, 4096, 16, 4),   # 16 assignments, 16 experts
])
def test_stream_k_down_projection(T, H, I, E, k):
    """T*k <= E: the down GEMM takes equal K-block ranges per CTA; tiles cut
    by CTA boundaries are summed from several partial slots."""
    case = MoECase(T, H, I, E, k, 0, seed=41 + T)
    run_case(case, what=f"stream-K T{T} H{H} I{I} E{E} k{k}")


def test_empty_experts_and_one_hot_expert():
    T, E = 50, 8
    logits = torch.randn(T, E, generator=torch.Generator().manual_seed(3))
    logits[:, 2] = -50.0           # never routed
    logits[:, 6] = -50.0
    case = MoECase(T, 256, 256, E, 2, 0, logits_override=logits)
    assert case.o_counts[2] == 0 and case.o_counts[6] == 0
    run_case(case, what="empty experts")
    logits1 = torch.zeros(40, E)
    logits1[:, 4] = 20.0           # every token on expert 4 (k = 1)
    case1 = MoECase(40, 256, 256, E, 1, 1, logits_override=logits1)
    assert case1.o_counts[4] == 40
    run_case(case1, what="one expert")


def test_prefill_empty_experts_and_one_hot_expert():
    """The prefill plan (weights unpacked ahead, banded tiles, paced down
    weight streams) with idle experts, and with every token on one expert."""
    T, E = 600, 8
    logits = torch.randn(T, E, generator=torch.Generator().manual_seed(5))
    logits[:, 1] = -50.0           # never routed
    logits[:, 5] = -50.0
    case = MoECase(T, 384, 640, E, 2, 1, logits_override=logits)
    assert case.o_counts[1] == 0 and case.o_counts[5] == 0
    run_case(case, what="prefill empty experts")
    logits1 = torch.zeros(T, E)
    logits1[:, 4] = 20.0           # every token on expert 4 (k = 1)
    case1 = MoECase(T, 384, 640, E, 1, 0, logits_override=logits1)
    assert case1.o_counts[4] == T
    run_case(case1, what="prefill one expert")


def test_deterministic_and_error_word_clean():
    import w4a8_moe_gb300 as lib
    case = MoECase(37, 512, 512, 8, 2, 1, seed=9)
    ws = torch.zeros(lib.moe_w4a8_workspace_size(37, 512, 512, 8, 2), dtype=torch.uint8,
                     device="cuda")
    a = case.run_gpu(ws=ws).clone()
    b = case.run_gpu(ws=ws).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert lib.w4a8_device_error(ws) == 0
    # this shape runs both projections in one launch, whose tile-claim
    # counters (header bytes 192-199) every call leaves zero for the next
    assert lib.moe_w4a8_plan(37, 512, 512, 8, 2)["one_launch"] == 1
    torch.cuda.synchronize()
    assert int(ws[192:200].count_nonzero()) == 0


def test_prefill_deterministic_across_calls():
    """Prefill plan: repeated calls on one workspace give identical bits (the
    down launch's pacing counters are reset by every call) and leave the
    error word clean."""
    import w4a8_moe_gb300 as lib
    T, H, I, E, k = 700, 384, 640, 8, 2
    case = MoECase(T, H, I, E, k, 1, seed=12)
    assert lib.moe_w4a8_plan(T, H, I, E, k)["one_launch"] == 0
    ws = torch.zeros(lib.moe_w4a8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device="cuda")
    outs = [case.run_gpu(ws=ws).clone() for _ in range(3)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert lib.w4a8_device_error(ws) == 0


def covering_sample(case: MoECase, n: int, seed: int = 0):
    """A seeded sample of n tokens that covers every expert with tokens: first
    one token of each expert, least loaded expert first, then random tokens,
    and the last token of the batch."""
    ids, counts = case.o_ids, case.o_counts
    pick = []
    for e in sorted((e for e in range(case.E) if counts[e] > 0), key=lambda e: (counts[e], e)):
        routed = np.nonzero((ids == e).any(1))[0]
        if not any(t in pick for t in routed.tolist()):
            pick.append(int(routed[-1]))
    if case.T - 1 not in pick:
        pick.append(case.T - 1)
    rng = np.random.default_rng(seed)
    for t in rng.permutation(case.T):
        if len(pick) >= n:
            break
        if int(t) not in pick:
            pick.append(int(t))
    toks = sorted(pick)
    covered = set(ids[toks].ravel().tolist())
    assert covered == {e for e in range(case.E) if counts[e] > 0}
    return toks


def check_hidden_codes(case: MoECase, ws, tokens, what, max_rate=1e-3):
    """The kernel's intermediate E4M3 codes against the oracle's, on the
    sampled tokens: a small share may sit one E4M3 step apart (h / a2 within
    fp32 rounding of a midpoint); none further."""
    got = case.gpu_hidden_codes(ws)[tokens]
    ref = case.oracle_hidden_codes(tokens)
    rate, far = compare_codes(got, ref, what)
    assert far == 0, f"{what}: {far} intermediate codes more than one E4M3 step from the oracle's"
    assert rate <= max_rate, f"{what}: intermediate code mismatch rate {rate:.2e}"


def _workspace(case: MoECase):
    import w4a8_moe_gb300 as lib
    return torch.zeros(lib.moe_w4a8_workspace_size(case.T, case.H, case.I, case.E, case.k),
                       dtype=torch.uint8, device="cuda")


def test_mixtral_decode_full_size():
    """All 32 tokens of the Mixtral-shaped decode layer, and every intermediate code."""
    s = synth.MOE_SHAPES["mixtral_decode"]
    case = MoECase(s.T, s.H, s.I, s.E, s.k, s.act, bias_std=s.bias_std)
    case.check_integer_parts()
    ws = _workspace(case)
    out = case.run_gpu(ws=ws)
    toks = list(range(s.T))
    check_hidden_codes(case, ws, toks, "mixtral decode")
    assert_close(bf16_to_f64(out), case.oracle_out(toks), "mixtral decode T32")


@pytest.fixture(scope="module")
def grok_weights():
    s = synth.MOE_SHAPES["grok_decode"]
    w = synth.moe_weights(s.H, s.I, s.E, device="cuda")
    q = QuantizedWeights(w["w_gu"], w["w_d"])
    del w
    torch.cuda.empty_cache()
    return q


@pytest.mark.parametrize("name", ["grok_decode", "grok_decode_t8", "grok_decode_t1"])
def test_grok_decode_full_size(name, grok_weights):
    """Every token of the Grok-1-shaped decode layers (32, 8 and 1 tokens)."""
    s = synth.MOE_SHAPES[name]
    case = MoECase(s.T, s.H, s.I, s.E, s.k, s.act, bias_std=s.bias_std, weights=grok_weights)
    case.check_integer_parts(sample_rows=[(0, 0), (3, 40000), (7, 65535)])
    ws = _workspace(case)
    out = case.run_gpu(ws=ws)
    toks = list(range(s.T))
    check_hidden_codes(case, ws, toks, name)
    assert_close(bf16_to_f64(out), case.oracle_out(toks), name)


def test_grok_prefill_full_size_sampled(grok_weights):
    """The 32768-token Grok-1 prefill layer: route and permutation on every
    token (bit-exact), the output and the intermediate codes on a seeded
    512-token sample that covers every expert, the least loaded included
    (each token's output depends only on that token, given the static scales)."""
    s = synth.MOE_SHAPES["grok_prefill"]
    case = MoECase(s.T, s.H, s.I, s.E, s.k, s.act, bias_std=s.bias_std, weights=grok_weights)
    case.check_integer_parts(sample_rows=[(1, 5)])
    assert case.o_counts.max() > 2 * case.o_counts.min()       # skewed load
    toks = covering_sample(case, 512)
    assert len(toks) == 512
    ws = _workspace(case)
    out = case.run_gpu(ws=ws)
    assert torch.isfinite(out.float()).all()
    check_hidden_codes(case, ws, toks, "grok prefill (512-token sample)")
    assert_close(bf16_to_f64(out[toks]), case.oracle_out(toks), "grok prefill (512-token sample)")


def test_prefill_bands_with_partial_last_bands():
    """The prefill plan's banded tile order across several bands: 9000 tokens
    over 2 experts (k = 1) give each expert 18 token tiles of 256 (gate_up
    bands of 16 + 2 token tiles) and H = 2560 gives 20 down row tiles (bands of
    16 + 4); every token and every intermediate code is compared."""
    import w4a8_moe_gb300 as lib
    T, H, I, E, k = 9000, 2560, 512, 2, 1
    assert lib.moe_w4a8_plan(T, H, I, E, k)["token_tile"] == 256
    case = MoECase(T, H, I, E, k, 1, seed=77)
    assert min(case.o_counts) > 16 * 256                       # more than one token band per expert
    case.check_integer_parts()
    ws = _workspace(case)
    out = case.run_gpu(ws=ws)
    toks = list(range(T))
    check_hidden_codes(case, ws, toks, "prefill bands T9000 H2560")
    assert_close(bf16_to_f64(out), case.oracle_out(toks), "prefill bands T9000 H2560")
