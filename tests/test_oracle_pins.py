"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against a closed form, a value the
format definition fixes (tests/golden/), a library routine (torch's
float8_e4m3fn / bfloat16 conversions, numpy's stable sort, scipy's softmax,
float64 matmul) or brute force on tiny inputs. They run on the CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALL_CODES = np.arange(256, dtype=np.uint8)
NAN_CODES = {0x7F, 0xFF}


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def torch_e4m3_value(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_e4m3_encode(v32):
    """Library RNE fp32 -> e4m3 (valid where |v| <= 448)."""
    t = torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# --------------------------------------------------------------------- e4m3

def test_e4m3_decode_all_codes_match_torch():
    ours = oracle.e4m3_to_double(ALL_CODES)
    ref = torch_e4m3_value(ALL_CODES)
    for c in range(256):
        if c in NAN_CODES:
            assert math.isnan(ours[c]) and math.isnan(ref[c])
        else:
            assert ours[c] == ref[c], hex(c)
            assert math.copysign(1, ours[c]) == math.copysign(1, ref[c])


def test_e4m3_landmarks_golden():
    for code_hex, val in _read_golden("e4m3_landmarks.txt"):
        got = oracle.e4m3_to_double(np.array([int(code_hex, 16)], np.uint8))[0]
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_encode_roundtrips_every_code():
    vals = oracle.e4m3_to_double(ALL_CODES)
    mask = np.array([c not in NAN_CODES for c in range(256)])
    enc = oracle.e4m3_from_float(vals[mask].astype(np.float32))
    assert np.array_equal(enc, ALL_CODES[mask])


def test_e4m3_encode_midpoints_and_neighbours_match_torch():
    pos = np.array([c for c in range(0x7F)], np.uint8)   # 0x00..0x7E, ascending values
    v = oracle.e4m3_to_double(pos)
    mids = (v[:-1] + v[1:]) / 2                            # exact in fp32 (<= 5 significant bits)
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    cases = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)),
                            np.nextafter(m32, np.float32(0))])
    cases = np.concatenate([cases, -cases])
    assert np.array_equal(oracle.e4m3_from_float(cases), torch_e4m3_encode(cases))
    # ties go to the even mantissa: midpoint between 1.0 (0x38) and 1.125 (0x39) -> 0x38,
    # between 1.125 and 1.25 (0x3A) -> 0x3A
    assert oracle.e4m3_from_float(np.array([1.0625, 1.1875], np.float32)).tolist() == [0x38, 0x3A]


def test_e4m3_encode_random_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 2.0 ** -7, 20000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_from_float(v), torch_e4m3_encode(v))


def test_e4m3_encode_saturates_and_nan():
    v = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, np.inf, -449.0, -np.inf, np.nan, -0.0],
                 np.float32)
    assert oracle.e4m3_from_float(v).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE,
                                                  0xFE, 0x7F, 0x80]


def test_int4_codes_golden():
    for q, nib, code in _read_golden("int4_e4m3.txt"):
        q, nib, code = int(q), int(nib, 16), int(code, 16)
        assert oracle.e4m3_from_float(np.array([q], np.float32))[0] == code
        assert oracle.e4m3_to_double(np.array([code], np.uint8))[0] == q
        word = np.array([nib], np.int32)                  # nibble in position 0
        assert oracle.unpack_int4(word)[0] == q


# --------------------------------------------------------------------- bf16

def test_bf16_rounding_of_float32_matches_torch():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.normal(0, 1, 50000), rng.normal(0, 1e-30, 1000),
                        rng.normal(0, 1e30, 1000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_from_double(v.astype(np.float64)), ref)


def test_bf16_single_rounding_from_double():
    rng = np.random.default_rng(3)
    b = rng.integers(0x0080, 0x7F00, 2000).astype(np.uint16)   # positive normal bf16
    lo = oracle.bf16_to_float(b).astype(np.float64)
    hi = oracle.bf16_to_float(b + 1).astype(np.float64)
    mid = (lo + hi) / 2
    eps = (hi - lo) * 2.0 ** -30                              # far below fp32 resolution of mid
    assert np.array_equal(oracle.bf16_from_double(mid + eps), b + 1)
    assert np.array_equal(oracle.bf16_from_double(mid - eps), b)
    tie = oracle.bf16_from_double(mid)
    assert np.array_equal(tie, np.where(b % 2 == 0, b, b + 1))


# --------------------------------------------------------------------- INT4

def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_quantize_experts_known_codes_and_packing():
    rng = np.random.default_rng(4)
    E, N, K = 2, 5, 32
    q_true = rng.integers(-7, 8, (E, N, K))
    q_true[:, :, 3] = 7                                    # amax = 7 * 0.125 in every row
    w = _bf16(q_true * 0.125)
    packed, scale = oracle.quantize_experts(w)
    assert np.all(scale == np.float32(0.125))
    words = np.zeros((E, N, K // 8), np.uint32)
    for i in range(8):
        words |= ((q_true[:, :, i::8] & 0xF).astype(np.uint32) << (4 * i))
    assert np.array_equal(packed.view(np.uint32), words)
    assert np.array_equal(oracle.unpack_int4(packed), q_true)


def test_quantize_experts_half_to_even_and_zero_row():
    # scale 0.125: 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, 0.5 -> 0, 1.5 -> 2
    row = np.zeros(8 * 4, np.float32)
    row[:6] = [7 * 0.125, 2.5 * 0.125, 3.5 * 0.125, -2.5 * 0.125, 0.5 * 0.125, 1.5 * 0.125]
    w = _bf16(np.stack([row, np.zeros_like(row)])[None])
    packed, scale = oracle.quantize_experts(w)
    q = oracle.unpack_int4(packed)
    assert q[0, 0, :6].tolist() == [7, 2, 4, -2, 0, 2]
    assert scale[0, 1] == 1.0 and not q[0, 1].any()


def test_quantize_experts_invariants_random():
    torch.manual_seed(0)
    w = (torch.randn(3, 40, 256) * 0.02).to(torch.bfloat16)
    packed, scale = oracle.quantize_experts(w)
    q = oracle.unpack_int4(packed).astype(np.float64)
    wf = w.float().numpy().astype(np.float64)
    assert np.abs(q).max() <= 7
    assert np.all(np.abs(q).max(axis=2) == 7)
    amax = np.abs(wf).max(axis=2)
    assert np.array_equal(scale, (amax.astype(np.float32) / np.float32(7)))
    err = np.abs(wf - scale[..., None].astype(np.float64) * q)
    assert np.all(err <= scale[..., None] * (0.5 + 1e-6))


# --------------------------------------------------------------------- activations

def test_quantize_act_matches_library_conversion():
    torch.manual_seed(1)
    x = torch.randn(64, 256).to(torch.bfloat16)
    s = oracle.act_scale(x)
    assert s == np.float32(np.abs(x.float().numpy()).max()) / np.float32(448.0)
    xq = oracle.quantize_act(x, s)
    q32 = (x.float().numpy() / np.float32(s)).astype(np.float32)
    assert np.abs(q32).max() <= 448.0 + 1e-3
    ref = torch_e4m3_encode(np.clip(q32, -448, 448))
    assert np.array_equal(xq, ref)
    flat = np.abs(x.float().numpy()).ravel()
    assert xq.ravel()[np.argmax(flat)] & 0x7F == 0x7E     # the largest element maps to 448


def test_act_scale_of_zero_tensor_is_one():
    assert oracle.act_scale(torch.zeros(4, 128, dtype=torch.bfloat16)) == 1.0


# --------------------------------------------------------------------- routing

def test_route_topk_against_sorting_with_ties():
    rng = np.random.default_rng(5)
    T, E, k = 300, 8, 2
    logits = rng.normal(0, 1, (T, E)).astype(np.float32)
    logits[::3, 5] = logits[::3, 2]                        # exact ties
    logits[::7, :] = 0.25                                  # all equal
    ids, w = oracle.route(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        assert ids[t].tolist() == order[:k]
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, ids, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    ids2, w2 = oracle.route(logits, k, renorm=False)
    np.testing.assert_allclose(w2, sel, rtol=1e-12)


def test_route_brute_force_subsets():
    rng = np.random.default_rng(6)
    T, E, k = 50, 6, 3
    logits = rng.integers(-3, 3, (T, E)).astype(np.float32)   # many ties
    ids, _ = oracle.route(logits, k)
    for t in range(T):
        best = None
        for sub in itertools.combinations(range(E), k):
            key = (sorted((-float(logits[t, e]), e) for e in sub))
            if best is None or key < best:
                best = key
        assert ids[t].tolist() == [e for _, e in best]


def test_permute_against_stable_sort():
    rng = np.random.default_rng(7)
    T, E, k = 257, 8, 2
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, sorted_ids, inv = oracle.permute(ids, E)
    flat = ids.ravel()
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(sorted_ids, np.argsort(flat, kind="stable"))
    assert np.array_equal(inv[sorted_ids], np.arange(T * k))
    # an expert with no tokens
    ids0 = np.where(ids == 3, 4, ids).astype(np.int32)
    ids0[:, 1] = np.where(ids0[:, 0] == ids0[:, 1], (ids0[:, 1] + 1) % E, ids0[:, 1])
    ids0 = np.where(ids0 == 3, 5, ids0).astype(np.int32)
    c0, o0, s0, _ = oracle.permute(ids0, E)
    assert c0[3] == 0 and o0[3] == o0[4]
    assert np.array_equal(s0, np.argsort(ids0.ravel(), kind="stable"))


# --------------------------------------------------------------------- MoE forward

def _moe_case(T, H, I, E, k, act, seed, identical=False, bias=0.0):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g).numpy() + bias
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w_gu = (torch.randn(E, 2 * I, H, generator=g) * 0.02).to(torch.bfloat16)
    w_d = (torch.randn(E, H, I, generator=g) * 0.02).to(torch.bfloat16)
    if identical:
        w_gu[:] = w_gu[0:1]
        w_d[:] = w_d[0:1]
    s1 = oracle.act_scale(x)
    xq = oracle.quantize_act(x, s1)
    pgu, sgu = oracle.quantize_experts(w_gu)
    pd, sd = oracle.quantize_experts(w_d)
    ids, tw = oracle.route(logits.astype(np.float32), k)
    return dict(logits=logits.astype(np.float32), x=x, s1=s1, xq=xq, pgu=pgu, sgu=sgu, pd=pd,
                sd=sd, ids=ids, tw=tw, act=act, H=H, I=I, E=E, k=k, T=T)


def _torch_reference(c, s2, topk_w, return_codes=False):
    """Float64 torch reference on dequantized operands; library routines for the
    e4m3 conversion, the activations (silu / gelu-tanh), softmax and matmul."""
    xv = torch.from_numpy(torch_e4m3_value(c["xq"]))                      # [T,H]
    qgu = torch.from_numpy(oracle.unpack_int4(c["pgu"]).astype(np.float64))  # [E,2I,H]
    qd = torch.from_numpy(oracle.unpack_int4(c["pd"]).astype(np.float64))    # [E,H,I]
    I = c["I"]
    out = torch.zeros(c["T"], c["H"], dtype=torch.float64)
    codes = np.zeros((c["T"], c["k"], I), np.uint8)
    hmax = 0.0
    for t in range(c["T"]):
        for j in range(c["k"]):
            e = int(c["ids"][t, j])
            acc = qgu[e] @ xv[t]                                              # [2I]
            sc = torch.from_numpy(c["sgu"][e].astype(np.float64)) * float(c["s1"])
            gu = acc * sc
            g, u = gu[:I], gu[I:]
            a = torch.nn.functional.silu(g) if c["act"] == 0 else \
                torch.nn.functional.gelu(g, approximate="tanh")
            h = a * u
            hmax = max(hmax, float(h.abs().max()))
            h32 = (h / float(s2)).to(torch.float32).clamp(-448, 448)
            h8 = h32.to(torch.float8_e4m3fn)
            codes[t, j] = h8.view(torch.uint8).numpy()
            hv = h8.to(torch.float64)
            y = (qd[e] @ hv) * torch.from_numpy(c["sd"][e].astype(np.float64)) * float(s2)
            out[t] += float(topk_w[t, j]) * y
    if return_codes:
        return out.numpy(), hmax, codes
    return out.numpy(), hmax


@pytest.mark.parametrize("act", [0, 1])
def test_moe_forward_matches_float64_reference(act):
    c = _moe_case(T=6, H=128, I=256, E=4, k=2, act=act, seed=11)
    s2 = oracle.moe_hidden_scale(c["xq"], c["s1"], c["pgu"], c["sgu"], act, c["ids"], [0, 1, 2])
    p = scipy.special.softmax(c["logits"].astype(np.float64), axis=1)
    sel = np.take_along_axis(p, c["ids"], axis=1)
    tw = sel / sel.sum(1, keepdims=True)
    ref, _ = _torch_reference(c, s2, tw)
    _, hmax3 = _torch_reference({**c, "T": 3}, s2, tw)
    assert s2 == np.float32(hmax3) / np.float32(448.0) or abs(s2 - hmax3 / 448) < 1e-6 * s2
    out = oracle.moe_forward(c["xq"], c["s1"], c["pgu"], c["sgu"], c["pd"], c["sd"], s2, act,
                             c["ids"], c["tw"], nthreads=2)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("act", [0, 1])
def test_moe_hidden_codes_match_float64_reference(act):
    """The intermediate E4M3 codes: torch's float64 gating of dequantized
    operands, then torch's fp32 -> float8_e4m3fn conversion of h / s2."""
    c = _moe_case(T=5, H=256, I=128, E=3, k=2, act=act, seed=15)
    # a scale small enough that the largest |h| saturate at +-448
    s2 = oracle.moe_hidden_scale(c["xq"], c["s1"], c["pgu"], c["sgu"], act, c["ids"], [0]) * 0.5
    _, _, ref = _torch_reference(c, s2, np.ones((5, 2)), return_codes=True)
    got = oracle.moe_hidden_codes(c["xq"], c["s1"], c["pgu"], c["sgu"], s2, act, c["ids"],
                                  [0, 1, 2, 3, 4], nthreads=2)
    assert got.shape == (5, 2, 128)
    assert np.array_equal(got, ref)
    assert np.any((got & 0x7F) == 0x7E)                         # saturated codes present
    sub = oracle.moe_hidden_codes(c["xq"], c["s1"], c["pgu"], c["sgu"], s2, act, c["ids"], [3, 1])
    assert np.array_equal(sub, got[[3, 1]])


def test_moe_single_expert_is_dense_mlp():
    c = _moe_case(T=5, H=128, I=128, E=1, k=1, act=0, seed=12)
    s2 = float(np.float32(0.01))
    ref, _ = _torch_reference(c, s2, np.ones((5, 1)))
    out = oracle.moe_forward(c["xq"], c["s1"], c["pgu"], c["sgu"], c["pd"], c["sd"], s2, 0,
                             c["ids"], c["tw"])
    assert np.all(c["tw"] == 1.0)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def test_moe_identical_experts_ignore_routing():
    c = _moe_case(T=4, H=128, I=128, E=4, k=2, act=1, seed=13, identical=True)
    s2 = float(np.float32(0.02))
    out1 = oracle.moe_forward(c["xq"], c["s1"], c["pgu"], c["sgu"], c["pd"], c["sd"], s2, 1,
                              c["ids"], c["tw"])
    ids2, tw2 = oracle.route(c["logits"][:, ::-1].copy(), 2)     # different experts, same layer
    assert not np.array_equal(ids2, c["ids"])
    out2 = oracle.moe_forward(c["xq"], c["s1"], c["pgu"], c["sgu"], c["pd"], c["sd"], s2, 1,
                              ids2, tw2)
    np.testing.assert_allclose(out1, out2, rtol=1e-12, atol=1e-14)
    single = oracle.moe_forward(c["xq"], c["s1"], c["pgu"][:1], c["sgu"][:1], c["pd"][:1],
                                c["sd"][:1], s2, 1, np.zeros((4, 1), np.int32), np.ones((4, 1)))
    np.testing.assert_allclose(out1, single, rtol=1e-12, atol=1e-14)


def test_moe_token_subset_equals_full():
    c = _moe_case(T=7, H=128, I=128, E=3, k=2, act=0, seed=14)
    full = oracle.moe_forward(c["xq"], c["s1"], c["pgu"], c["sgu"], c["pd"], c["sd"], 0.02, 0,
                              c["ids"], c["tw"], nthreads=3)
    sub = oracle.moe_forward(c["xq"], c["s1"], c["pgu"], c["sgu"], c["pd"], c["sd"], 0.02, 0,
                             c["ids"], c["tw"], tokens=[6, 2], nthreads=1)
    assert np.array_equal(sub, full[[6, 2]])


# --------------------------------------------------------------------- block-FP8

def test_block_linear_integer_case_is_exact_integer_gemm():
    rng = np.random.default_rng(8)
    M, N, K = 5, 256, 384
    ints = np.arange(-8, 9)
    codes = oracle.e4m3_from_float(ints.astype(np.float32))
    xi = rng.integers(0, ints.size, (M, K))
    wi = rng.integers(0, ints.size, (N, K))
    y = oracle.block_linear(codes[xi], np.ones((M, K // 128), np.float32), codes[wi],
                            np.ones((N // 128, K // 128), np.float32))
    assert np.array_equal(y, (ints[xi].astype(np.int64) @ ints[wi].T.astype(np.int64)))


def test_block_linear_matches_float64_reference_and_scales():
    torch.manual_seed(2)
    M, N, K = 3, 256, 512
    x = torch.randn(M, K).to(torch.bfloat16)
    w = (torch.randn(N, K) * 0.02).to(torch.bfloat16)
    wq, wsi = oracle.block_quantize_weight(w)
    xq, xs = oracle.block_quantize_act(x)
    y = oracle.block_linear(xq, xs, wq, wsi, nthreads=2)
    xd = torch_e4m3_value(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)
    wd = torch_e4m3_value(wq) * np.kron(wsi.astype(np.float64), np.ones((128, 128)))
    np.testing.assert_allclose(y, xd @ wd.T, rtol=1e-10, atol=1e-13)
    y8 = oracle.block_linear(xq, xs, wq, wsi * np.float32(8.0))
    assert np.array_equal(y8, y * 8.0)
    yrows = oracle.block_linear(xq, xs, wq, wsi, rows=[2, 0])
    assert np.array_equal(yrows, y[[2, 0]])


def test_block_quantizers_invariants():
    torch.manual_seed(3)
    x = torch.randn(4, 256).to(torch.bfloat16)
    xq, xs = oracle.block_quantize_act(x)
    xf = x.float().numpy()
    for m in range(4):
        for g in range(2):
            seg = xf[m, g * 128:(g + 1) * 128]
            assert xs[m, g] == np.float32(np.abs(seg).max()) / np.float32(448.0)
            q32 = (seg / xs[m, g]).astype(np.float32)
            assert np.array_equal(xq[m, g * 128:(g + 1) * 128],
                                  torch_e4m3_encode(np.clip(q32, -448, 448)))
    w = (torch.randn(256, 128) * 0.02).to(torch.bfloat16)
    w[128:] = 0
    wq, wsi = oracle.block_quantize_weight(w)
    assert wsi.shape == (2, 1) and wsi[1, 0] == 1.0 and not wq[128:].any()
    assert (wq[:128] & 0x7F).max() == 0x7E


# --- router gate logits ---------------------------------------------------------

def test_gate_logits_match_float64_matmul():
    """Plain double loop vs numpy's float64 matrix product of the same bf16 values."""
    from w4a8_moe_gb300 import synth
    inp = synth.router_gate_inputs(5, 384, 7, seed=3)
    x = inp["hidden"].float().numpy().astype(np.float64)
    g = inp["gate"].float().numpy().astype(np.float64)
    got = oracle.gate_logits(inp["hidden"], inp["gate"])
    np.testing.assert_allclose(got, x @ g.T, rtol=1e-12, atol=1e-12)


def test_gate_logits_one_hot_rows_pick_gate_columns():
    """Closed form: a one-hot hidden row at h (value v) gives logits v * gate[:, h] exactly."""
    from w4a8_moe_gb300 import synth
    g = synth.router_gate_inputs(1, 256, 9, seed=4)["gate"]
    T, H = 6, 256
    x = torch.zeros(T, H, dtype=torch.bfloat16)
    cols = [0, 17, 100, 128, 200, 255]
    vals = [1.0, -2.0, 0.5, 3.0, -0.25, 1.5]
    for t, (h, v) in enumerate(zip(cols, vals)):
        x[t, h] = v
    got = oracle.gate_logits(x, g)
    gf = g.float().numpy().astype(np.float64)
    for t, (h, v) in enumerate(zip(cols, vals)):
        assert np.array_equal(got[t], v * gf[:, h])


def test_gate_logits_are_linear_in_the_gate():
    """Doubling the gate (exact in bf16) doubles every logit exactly."""
    from w4a8_moe_gb300 import synth
    inp = synth.router_gate_inputs(4, 128, 5, seed=5)
    a = oracle.gate_logits(inp["hidden"], inp["gate"])
    b = oracle.gate_logits(inp["hidden"], (inp["gate"].float() * 2).to(torch.bfloat16))
    assert np.array_equal(b, 2 * a)


# --- per-tensor FP8 linear ------------------------------------------------------

def _fp8_codes(shape, rng):
    """Random finite E4M3 codes (NaN codes 0x7F/0xFF excluded)."""
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)


def test_fp8_linear_equals_block_linear_with_uniform_scales():
    """With every block scale equal to sw and every activation group scale sx,
    the block-FP8 definition (pinned separately) is the per-tensor one."""
    rng = np.random.default_rng(21)
    M, N, K = 5, 256, 384
    xq, wq = _fp8_codes((M, K), rng), _fp8_codes((N, K), rng)
    sx, sw = np.float32(0.013), np.float32(0.0021)
    y = oracle.fp8_linear(xq, sx, wq, sw)
    xs = np.full((M, K // 128), sx, np.float32)
    wsi = np.full((N // 128, K // 128), sw, np.float32)
    yb = oracle.block_linear(xq, xs, wq, wsi)
    np.testing.assert_allclose(y, yb, rtol=1e-13, atol=0)


def test_fp8_linear_integer_codes_unit_scales_is_an_integer_gemm():
    """E4M3 codes of small integers with unit scales: an exact int64 matrix product."""
    rng = np.random.default_rng(22)
    M, N, K = 4, 128, 256
    table = {v: int(oracle.e4m3_from_float(np.float32(v))[0]) for v in range(-8, 9)}
    xi = rng.integers(-8, 9, size=(M, K))
    wi = rng.integers(-8, 9, size=(N, K))
    xq = np.vectorize(table.get)(xi).astype(np.uint8)
    wq = np.vectorize(table.get)(wi).astype(np.uint8)
    y = oracle.fp8_linear(xq, 1.0, wq, 1.0)
    assert np.array_equal(y, (xi.astype(np.int64) @ wi.astype(np.int64).T).astype(np.float64))


def test_fp8_linear_scales_by_powers_of_two_exactly():
    rng = np.random.default_rng(23)
    xq, wq = _fp8_codes((3, 256), rng), _fp8_codes((128, 256), rng)
    a = oracle.fp8_linear(xq, 0.5, wq, 0.25)
    b = oracle.fp8_linear(xq, 0.5 * 2 ** 5, wq, 0.25 * 2 ** -3)
    assert np.array_equal(b, a * 4)
