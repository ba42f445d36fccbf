"""Shared helpers for the parity tests: build/load the library, run the GPU path
and the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from w4a8_moe_gb300 import synth  # noqa: E402

# Floating-point parity bar (relative L2 and max-abs relative to max|ref|).
REL_L2_TOL = 2e-3
MAX_ABS_TOL = 1e-2


def gpu_ok() -> bool:
    return torch.cuda.is_available()


def ensure_built():
    from w4a8_moe_gb300 import build as b
    return b.build()


def to_np_bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU output"
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got - ref)
    mref = np.abs(ref).max()
    mabs = np.abs(got - ref).max() / mref if mref > 0 else np.abs(got - ref).max()
    return float(rel), float(mabs)


def assert_close(got, ref, what=""):
    rel, mabs = compare(got, ref)
    assert rel <= REL_L2_TOL and mabs <= MAX_ABS_TOL, f"{what}: rel_l2={rel:.3e} max_abs/max|ref|={mabs:.3e}"
    return rel, mabs


def oracle_threads() -> int:
    return max(1, min(16, oracle.cores()))


class QuantizedWeights:
    """Expert weights quantized once by each side: the library on the GPU and the
    oracle on host copies of the same bf16 tensors."""

    def __init__(self, w_gu_bf16: torch.Tensor, w_d_bf16: torch.Tensor):
        import w4a8_moe_gb300 as lib
        self.gpu = (*lib.w4a8_quantize_experts(w_gu_bf16), *lib.w4a8_quantize_experts(w_d_bf16))
        torch.cuda.synchronize()
        self.oracle = (*oracle.quantize_experts(to_np_bits(w_gu_bf16)),
                       *oracle.quantize_experts(to_np_bits(w_d_bf16)))


class MoECase:
    """One MoE layer run through both sides on the same seeded inputs."""

    def __init__(self, T, H, I, E, k, act, bias_std=0.0, seed=0, logits_override=None,
                 calib_tokens=8, weights=None):
        import w4a8_moe_gb300 as lib
        self.T, self.H, self.I, self.E, self.k, self.act = T, H, I, E, k, act
        inp = synth.moe_inputs(T, H, I, E, bias_std=bias_std, seed=seed, device="cuda",
                               weights=weights is None)
        if logits_override is not None:
            inp["logits"] = logits_override.to("cuda", torch.float32).contiguous()
        self.inp = inp
        if weights is None:
            weights = QuantizedWeights(inp["w_gu"], inp["w_d"])
        self.weights = weights
        # GPU side
        self.w_gu, self.s_gu, self.w_d, self.s_d = weights.gpu
        self.xq, self.a1 = lib.w4a8_quantize_act(inp["x"], compute_scale=True)
        self.route = lib.moe_route(inp["logits"], k)
        torch.cuda.synchronize()
        # oracle side, from host copies of the same inputs
        self.h_logits = inp["logits"].cpu().numpy()
        self.h_x = to_np_bits(inp["x"])
        self.o_pgu, self.o_sgu, self.o_pd, self.o_sd = weights.oracle
        self.o_s1 = oracle.act_scale(self.h_x)
        self.o_xq = oracle.quantize_act(self.h_x, self.o_s1)
        self.o_ids, self.o_w = oracle.route(self.h_logits, k)
        self.o_counts, self.o_offsets, self.o_sorted, self.o_inv = oracle.permute(self.o_ids, E)
        cal = synth.calibration_tokens(T, calib_tokens)
        self.s2 = oracle.moe_hidden_scale(self.o_xq, self.o_s1, self.o_pgu, self.o_sgu, act,
                                          self.o_ids, cal, nthreads=oracle_threads())
        self.a2 = torch.tensor([self.s2], dtype=torch.float32, device="cuda")

    def run_gpu(self, ws=None):
        import w4a8_moe_gb300 as lib
        out = lib.moe_w4a8_forward(self.xq, self.a1, self.w_gu, self.s_gu, self.w_d, self.s_d,
                                   self.a2, self.act, self.route, ws=ws)
        torch.cuda.synchronize()
        return out

    def oracle_out(self, tokens=None):
        return oracle.moe_forward(self.o_xq, self.o_s1, self.o_pgu, self.o_sgu, self.o_pd, self.o_sd,
                                  self.s2, self.act, self.o_ids, self.o_w, tokens=tokens,
                                  nthreads=oracle_threads())

    def check_integer_parts(self, sample_rows=None):
        """Quantized codes, packed words, scales, top-k ids and permutation: bit-exact."""
        if sample_rows is None:
            assert np.array_equal(self.w_gu.cpu().numpy(), self.o_pgu)
            assert np.array_equal(self.w_d.cpu().numpy(), self.o_pd)
            assert np.array_equal(self.s_gu.cpu().numpy(), self.o_sgu)
            assert np.array_equal(self.s_d.cpu().numpy(), self.o_sd)
        else:
            for e, r in sample_rows:
                assert np.array_equal(self.w_gu[e, r].cpu().numpy(), self.o_pgu[e, r])
                assert self.s_gu[e, r].item() == self.o_sgu[e, r]
            assert np.array_equal(self.w_gu.view(-1)[::9973].cpu().numpy(),
                                  self.o_pgu.reshape(-1)[::9973])
            assert np.array_equal(self.w_d.view(-1)[::9973].cpu().numpy(),
                                  self.o_pd.reshape(-1)[::9973])
            assert np.array_equal(self.s_gu.cpu().numpy(), self.o_sgu)
            assert np.array_equal(self.s_d.cpu().numpy(), self.o_sd)
        assert self.a1.item() == self.o_s1
        assert np.array_equal(self.xq.cpu().numpy(), self.o_xq)
        r = self.route
        assert np.array_equal(r.topk_ids.cpu().numpy(), self.o_ids)
        np.testing.assert_allclose(r.topk_w.cpu().numpy(), self.o_w, rtol=2e-6, atol=1e-7)
        assert np.array_equal(r.counts.cpu().numpy(), self.o_counts)
        assert np.array_equal(r.offsets.cpu().numpy(), self.o_offsets)
        assert np.array_equal(r.sorted_ids.cpu().numpy(), self.o_sorted)
        assert np.array_equal(r.inv_perm.cpu().numpy(), self.o_inv)
