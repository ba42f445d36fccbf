"""Seeded synthetic inputs for the W4A8 MoE layer and the block-FP8 projection.

This module draws random numbers only; it holds none of the method's
arithmetic (no quantization, routing or GEMM). The tests, the oracle and the
benchmark all take their inputs from here, so both sides of every comparison
see identical tensors.

Workload shapes follow the layers the pages describe: Grok-1 (hidden 6144,
intermediate 32768, 8 experts, 2 per token, bf16; "ROCm: enable
trillion-parameter MoE models with INT4-FP8 single node", config.json),
Mixtral-8x7B ("[AMD][Quantization] Add int4fp8_moe online quantization on
ROCm", run command), and the block-FP8 dense projections [16384,2560],
[13312,2560] ("qwen4_exp: serve the block-FP8 dense projections natively",
description) plus an o_proj-shaped [2560,6144].

Distributions: weights N(0, 0.02) rounded to bf16; activations N(0, 1) in bf16;
router logits N(0, 1) in fp32, plus an optional per-expert logit bias that
skews the expert load. Each tensor kind has its own generator seeded with
seed * 16 + a fixed offset (logits 1, bias 2, x 3, gate_up 4, down 5), so the
weights of a layer do not depend on the number of tokens drawn with them.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    act: int            # 0 = SiLU-gated, 1 = GELU(tanh)-gated
    bias_std: float     # std of the per-expert logit bias (0 = none)


MOE_SHAPES = {
    "tiny": MoEShape("tiny T16 H256 I512 E8 k2 SiLU", 16, 256, 512, 8, 2, 0, 0.0),
    "mixtral_decode": MoEShape("Mixtral-8x7B MoE layer decode T32 H4096 I14336 E8 k2 SiLU", 32,
                               4096, 14336, 8, 2, 0, 0.5),
    "grok_decode": MoEShape("Grok-1 MoE layer decode T32 H6144 I32768 E8 k2 GELU-tanh", 32, 6144,
                            32768, 8, 2, 1, 0.0),
    "grok_decode_t8": MoEShape("Grok-1 MoE layer decode T8 H6144 I32768 E8 k2 GELU-tanh", 8, 6144,
                               32768, 8, 2, 1, 0.0),
    "grok_decode_t1": MoEShape("Grok-1 MoE layer decode T1 H6144 I32768 E8 k2 GELU-tanh", 1, 6144,
                               32768, 8, 2, 1, 0.0),
    "grok_prefill": MoEShape("Grok-1 MoE layer prefill T32768 H6144 I32768 E8 k2 GELU-tanh skewed",
                             32768, 6144, 32768, 8, 2, 1, 1.0),
    # a prefill-shaped layer small enough for detailed profiling (a few GB on the device)
    "grok_prefill_8k": MoEShape("Grok-1 MoE layer prefill T8192 H6144 I32768 E8 k2 GELU-tanh skewed",
                                8192, 6144, 32768, 8, 2, 1, 1.0),
}

BLOCK_FP8_SHAPES = [(16384, 2560), (13312, 2560), (2560, 6144)]
BLOCK_FP8_M = [1, 8, 64, 4096]


def _gen(seed: int, device, offset: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + offset)
    return g


def moe_inputs(T: int, H: int, I: int, E: int, bias_std: float = 0.0, seed: int = 0,
               device="cpu", weights: bool = True, weight_std: float = 0.02):
    """Router logits fp32 [T,E] (bias added), x bf16 [T,H], W_gu bf16 [E,2I,H], W_d bf16 [E,H,I]."""
    logits = torch.randn(T, E, generator=_gen(seed, device, 1), device=device, dtype=torch.float32)
    if bias_std:
        bias = torch.randn(E, generator=_gen(seed, device, 2), device=device, dtype=torch.float32)
        logits = logits + bias * bias_std
    x = torch.randn(T, H, generator=_gen(seed, device, 3), device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    out = {"logits": logits.contiguous(), "x": x.contiguous()}
    if weights:
        out.update(moe_weights(H, I, E, seed=seed, device=device, weight_std=weight_std))
    return out


def moe_weights(H: int, I: int, E: int, seed: int = 0, device="cpu", weight_std: float = 0.02):
    """W_gu bf16 [E,2I,H] (rows [0,I) gate, [I,2I) up) and W_d bf16 [E,H,I]."""
    g_gu = _gen(seed, device, 4)
    g_d = _gen(seed, device, 5)
    w_gu = torch.empty(E, 2 * I, H, device=device, dtype=torch.bfloat16)
    w_d = torch.empty(E, H, I, device=device, dtype=torch.bfloat16)
    for e in range(E):  # per expert keeps the fp32 temporary small
        w_gu[e] = (torch.randn(2 * I, H, generator=g_gu, device=device) * weight_std).to(torch.bfloat16)
    for e in range(E):
        w_d[e] = (torch.randn(H, I, generator=g_d, device=device) * weight_std).to(torch.bfloat16)
    return {"w_gu": w_gu, "w_d": w_d}


def block_fp8_inputs(M: int, N: int, K: int, seed: int = 0, device="cpu", weight_std: float = 0.02):
    """Activations x bf16 [M,K] and a dense weight bf16 [N,K] to be block-quantized."""
    x = torch.randn(M, K, generator=_gen(seed, device, 6), device=device).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=_gen(seed, device, 7), device=device) * weight_std).to(torch.bfloat16)
    return {"x": x.contiguous(), "w": w.contiguous()}


def router_gate_inputs(T: int, H: int, E: int, seed: int = 0, device="cpu", gate_std: float = 0.02):
    """Hidden states bf16 [T, H] ~ N(0, 1) and a router gate bf16 [E, H] ~ N(0, gate_std)."""
    x = torch.randn(T, H, generator=_gen(seed, device, 8), device=device).to(torch.bfloat16)
    g = (torch.randn(E, H, generator=_gen(seed, device, 9), device=device) * gate_std).to(torch.bfloat16)
    return {"hidden": x.contiguous(), "gate": g.contiguous()}


# Per-tensor FP8 dense projections of a Grok-1-shaped attention block
# (hidden 6144, 48 query heads and 8 key/value heads of 128): qkv_proj and o_proj.
FP8_LINEAR_SHAPES = [(8192, 6144), (6144, 6144)]
FP8_LINEAR_M = [1, 8, 64, 4096]


def fp8_linear_inputs(M: int, N: int, K: int, seed: int = 0, device="cpu", weight_std: float = 0.02):
    """Activations x bf16 [M, K] ~ N(0, 1) and a dense weight bf16 [N, K] ~ N(0, weight_std)."""
    x = torch.randn(M, K, generator=_gen(seed, device, 10), device=device).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=_gen(seed, device, 11), device=device) * weight_std).to(torch.bfloat16)
    return {"x": x.contiguous(), "w": w.contiguous()}


def calibration_tokens(T: int, n: int = 256):
    """Tokens the static intermediate scale is calibrated on: the first min(T, n)."""
    return list(range(min(T, n)))
