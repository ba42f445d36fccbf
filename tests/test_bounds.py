"""Out-of-bounds writes: every entry point's outputs and workspace are placed
inside larger buffers whose bytes before and after are filled with a canary
pattern; after the call (and a synchronize) the canaries must be unchanged and
the results identical to the same call on ordinary tensors. Shapes cover the
ragged tails and every launch plan (one-launch decode, stream-K, prefill with
the weights unpacked once, split-K linear layers, the multi-kernel router).
This stands in for a memory checker, which is not available on this machine."""
import pytest
import torch

from helpers import MoECase, ensure_built
from w4a8_moe_gb300 import synth

pytestmark = pytest.mark.gpu

PAD = 4096          # canary bytes on each side (a multiple of 256: keeps alignment)
CANARY = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` inside a canary-padded byte buffer."""

    def __init__(self, shape, dtype, zero=False):
        n = 1
        for d in shape:
            n *= d
        self.nbytes = n * torch.tensor([], dtype=dtype).element_size()
        self.buf = torch.full((PAD + self.nbytes + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        mid = self.buf[PAD:PAD + self.nbytes]
        if zero:
            mid.zero_()
        self.t = mid.view(dtype).view(*shape)

    def check(self, what):
        torch.cuda.synchronize()
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.nbytes:]
        assert bool((head == CANARY).all()), f"{what}: write before the buffer"
        assert bool((tail == CANARY).all()), f"{what}: write past the end of the buffer"


def guarded_route(T, E, k):
    import w4a8_moe_gb300 as lib
    parts = [Guarded((T, k), torch.int32), Guarded((T, k), torch.float32), Guarded((E,), torch.int32),
             Guarded((E + 1,), torch.int32), Guarded((T * k,), torch.int32), Guarded((T * k,), torch.int32)]
    return parts, lib.RouteResult(*[p.t for p in parts])


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("T,H,I,E,k,act", [
    (33, 256, 256, 8, 2, 0),      # one launch, 64-token tiles, ragged
    (3, 2048, 4096, 8, 2, 1),     # stream-K down projection
    (300, 384, 640, 8, 2, 0),     # prefill plan: weights unpacked once, ragged K stages
])
def test_moe_forward_stays_in_bounds(T, H, I, E, k, act):
    import w4a8_moe_gb300 as lib
    case = MoECase(T, H, I, E, k, act, seed=T)
    ref = case.run_gpu()
    out = Guarded((T, H), torch.bfloat16)
    ws = Guarded((lib.moe_w4a8_workspace_size(T, H, I, E, k),), torch.uint8, zero=True)
    lib.moe_w4a8_forward(case.xq, case.a1, case.w_gu, case.s_gu, case.w_d, case.s_d, case.a2, act, case.route,
                         out=out.t, ws=ws.t)
    out.check("moe_w4a8_forward out")
    ws.check("moe_w4a8_forward workspace")
    assert torch.equal(out.t.view(torch.int16), ref.view(torch.int16))


def test_dynamic_forward_stays_in_bounds():
    import w4a8_moe_gb300 as lib
    T, H, I, E, k = 200, 384, 640, 8, 2
    case = MoECase(T, H, I, E, k, 1, seed=5)
    out = Guarded((T, H), torch.bfloat16)
    a2 = Guarded((1,), torch.float32)
    ws = Guarded((lib.moe_w4a8_dynamic_workspace_size(T, H, I, E, k),), torch.uint8, zero=True)
    lib.moe_w4a8_forward_dynamic(case.xq, case.a1, case.w_gu, case.s_gu, case.w_d, case.s_d, 1, case.route,
                                 out=out.t, a2_out=a2.t, ws=ws.t)
    for g, what in ((out, "out"), (a2, "a2_out"), (ws, "workspace")):
        g.check(f"moe_w4a8_forward_dynamic {what}")
    ref, a2_ref = lib.moe_w4a8_forward_dynamic(case.xq, case.a1, case.w_gu, case.s_gu, case.w_d, case.s_d, 1,
                                               case.route)
    torch.cuda.synchronize()
    assert torch.equal(out.t.view(torch.int16), ref.view(torch.int16)) and a2.t.item() == a2_ref.item()


@pytest.mark.parametrize("T,E,k", [(37, 8, 2), (3000, 16, 2)])   # one block; the multi-kernel router
def test_route_stays_in_bounds(T, E, k):
    import w4a8_moe_gb300 as lib
    logits = torch.randn(T, E, generator=torch.Generator(device="cuda").manual_seed(T), device="cuda")
    parts, out = guarded_route(T, E, k)
    ws = Guarded((lib.moe_route_workspace_size(T, E, k),), torch.uint8, zero=True)
    lib.moe_route(logits, k, out=out, ws=ws.t)
    for i, p in enumerate(parts):
        p.check(f"moe_route output {i}")
    ws.check("moe_route workspace")
    ref = lib.moe_route(logits, k)
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)


def test_route_gate_stays_in_bounds():
    import w4a8_moe_gb300 as lib
    T, H, E, k = 40, 512, 8, 2
    inp = synth.router_gate_inputs(T, H, E, seed=3, device="cuda")
    parts, out = guarded_route(T, E, k)
    logits = Guarded((T, E), torch.float32)
    ws = Guarded((lib.moe_route_gate_workspace_size(T, H, E, k),), torch.uint8, zero=True)
    lib.moe_route_gate(inp["hidden"], inp["gate"], k, out=out, logits=logits.t, ws=ws.t)
    for i, p in enumerate(parts):
        p.check(f"moe_route_gate output {i}")
    logits.check("moe_route_gate logits")
    ws.check("moe_route_gate workspace")


def test_quantizers_stay_in_bounds():
    import w4a8_moe_gb300 as lib
    E, N, K = 3, 136, 264
    w = (torch.randn(E, N, K, device="cuda") * 0.02).to(torch.bfloat16)
    packed, scale = Guarded((E, N, K // 8), torch.int32), Guarded((E, N), torch.float32)
    lib.w4a8_quantize_experts(w, packed=packed.t, scale=scale.t)
    packed.check("w4a8_quantize_experts packed")
    scale.check("w4a8_quantize_experts scale")
    p_ref, s_ref = lib.w4a8_quantize_experts(w)
    torch.cuda.synchronize()
    assert torch.equal(packed.t, p_ref) and torch.equal(scale.t, s_ref)

    x = torch.randn(7, 272, device="cuda").to(torch.bfloat16)
    xq, s1 = Guarded((7, 272), torch.uint8), Guarded((1,), torch.float32)
    ws = Guarded((lib.w4a8_quantize_act_workspace_size(x.numel()),), torch.uint8, zero=True)
    lib.w4a8_quantize_act(x, scale=s1.t, compute_scale=True, out=xq.t, ws=ws.t)
    for g, what in ((xq, "codes"), (s1, "scale"), (ws, "workspace")):
        g.check(f"w4a8_quantize_act {what}")


@pytest.mark.parametrize("M,N,K", [(1, 256, 1024), (17, 384, 512), (130, 256, 384)])
def test_block_fp8_linear_stays_in_bounds(M, N, K):
    import oracle
    import w4a8_moe_gb300 as lib
    inp = synth.block_fp8_inputs(M, N, K, seed=M, device="cuda")
    wq, wsi = oracle.block_quantize_weight(inp["w"].cpu())
    wq, wsi = torch.from_numpy(wq).cuda(), torch.from_numpy(wsi).cuda()
    y, xq, xs = Guarded((M, N), torch.bfloat16), Guarded((M, K), torch.uint8), Guarded((M, K // 128), torch.float32)
    ws = Guarded((lib.fp8_block_linear_workspace_size(M, N, K),), torch.uint8, zero=True)
    lib.fp8_block_linear(inp["x"], wq, wsi, out=y.t, xq_out=xq.t, xs_out=xs.t, ws=ws.t)
    for g, what in ((y, "y"), (xq, "xq_out"), (xs, "xs_out"), (ws, "workspace")):
        g.check(f"fp8_block_linear {what}")
    ref = lib.fp8_block_linear(inp["x"], wq, wsi)
    torch.cuda.synchronize()
    assert torch.equal(y.t.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(5, 256, 2048), (37, 384, 256), (300, 384, 384)])
def test_fp8_linear_stays_in_bounds(M, N, K):
    import w4a8_moe_gb300 as lib
    inp = synth.fp8_linear_inputs(M, N, K, seed=M, device="cuda")
    xq, sx = lib.w4a8_quantize_act(inp["x"])
    wq, sw = lib.w4a8_quantize_act(inp["w"])
    y = Guarded((M, N), torch.bfloat16)
    ws = Guarded((lib.fp8_linear_workspace_size(M, N, K),), torch.uint8, zero=True)
    lib.fp8_linear(xq, sx, wq, sw, out=y.t, ws=ws.t)
    y.check("fp8_linear y")
    ws.check("fp8_linear workspace")
    ref = lib.fp8_linear(xq, sx, wq, sw)
    torch.cuda.synchronize()
    assert torch.equal(y.t.view(torch.int16), ref.view(torch.int16))


def _sweep_cases(n=48, seed=2024):
    """A seeded sample of the small-shape grid T in {1,2,3,7,16,33},
    E in {1,2,8}, k in {1,2} (k <= E), H, I in {128, 256, 384}."""
    import itertools
    import random
    grid = [c for c in itertools.product((1, 2, 3, 7, 16, 33), (1, 2, 8), (1, 2), (128, 256, 384), (128, 256, 384))
            if c[2] <= c[1]]
    return random.Random(seed).sample(grid, n)


@pytest.mark.parametrize("T,E,k,H,I", _sweep_cases())
def test_small_shape_sweep(T, E, k, H, I):
    """Every token against the oracle, with the output and workspace guarded."""
    import w4a8_moe_gb300 as lib
    from helpers import assert_close, bf16_to_f64
    act = (T + H + I) % 2
    case = MoECase(T, H, I, E, k, act, seed=T * 1000 + H + I + E)
    case.check_integer_parts()
    out = Guarded((T, H), torch.bfloat16)
    ws = Guarded((lib.moe_w4a8_workspace_size(T, H, I, E, k),), torch.uint8, zero=True)
    lib.moe_w4a8_forward(case.xq, case.a1, case.w_gu, case.s_gu, case.w_d, case.s_d, case.a2, act, case.route,
                         out=out.t, ws=ws.t)
    out.check("sweep out")
    ws.check("sweep workspace")
    assert lib.w4a8_device_error(ws.t) == 0
    assert_close(bf16_to_f64(out.t), case.oracle_out(), f"sweep T{T} E{E} k{k} H{H} I{I}")
