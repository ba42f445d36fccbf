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


# Every comparison made by assert_close, for the margin table that
# tests/conftest.py prints at the end of the session.
MARGINS = []


def assert_close(got, ref, what="", bf16_out=True):
    """rel-L2 and max-abs of `got` against the oracle's float64 `ref`, within
    the parity bar. For a bf16 output also reports the same two measures
    against the oracle result rounded once to bf16: that part of the error is
    the kernel's own (the output format's rounding is no longer in it)."""
    rel, mabs = compare(got, ref)
    row = {"what": what, "rel_l2": rel, "max_abs": mabs, "n": int(np.asarray(ref).size)}
    if bf16_out:
        ref_b = oracle.bf16_to_float(oracle.bf16_from_double(np.asarray(ref, np.float64)))
        rb, mb = compare(got, ref_b)
        row.update(rel_l2_vs_bf16_ref=rb, max_abs_vs_bf16_ref=mb,
                   bf16_flips=float(np.mean(np.asarray(got, np.float64) != ref_b.astype(np.float64))))
    MARGINS.append(row)
    print(f"[margin] {what}: rel_l2={rel:.3e} (bar {REL_L2_TOL:.0e}) max_abs/max|ref|={mabs:.3e} "
          f"(bar {MAX_ABS_TOL:.0e})"
          + (f"; vs bf16(ref): rel_l2={row['rel_l2_vs_bf16_ref']:.3e} "
             f"flips={row['bf16_flips']:.3%}" if bf16_out else ""))
    assert rel <= REL_L2_TOL and mabs <= MAX_ABS_TOL, f"{what}: rel_l2={rel:.3e} max_abs/max|ref|={mabs:.3e}"
    return rel, mabs


def kperm_index(n: int) -> np.ndarray:
    """Column of element i in the library's stored K order: inside every group
    of 8, elements 0,2,4,6 then 1,3,5,7 (include/w4a8_moe.h,
    moe_w4a8_workspace_layout)."""
    i = np.arange(n)
    return (i & ~7) | ((i & 7) >> 1) | ((i & 1) << 2)


def e4m3_step_index(codes: np.ndarray) -> np.ndarray:
    """Signed position of an E4M3 code on the ordered grid of finite values
    (+0 and -0 both 0): two codes are neighbours iff positions differ by 1."""
    c = np.asarray(codes, np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def compare_codes(got: np.ndarray, ref: np.ndarray, what=""):
    """E4M3 codes of the intermediate activation: the share that differ and
    whether every difference is one step of the E4M3 grid (a value of h / a2
    near a rounding midpoint, decided on either side of it by the kernel's fp32
    arithmetic and the oracle's exact sums)."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got != ref
    rate = float(diff.mean())
    far = int((np.abs(e4m3_step_index(got) - e4m3_step_index(ref)) > 1).sum())
    MARGINS.append({"what": what + " (hq codes)", "code_mismatch_rate": rate, "non_adjacent": far,
                    "n": int(ref.size)})
    print(f"[margin] {what}: hq code mismatches {int(diff.sum())} of {ref.size} ({rate:.2e}), "
          f"non-adjacent {far}")
    return rate, far


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
                 calib_tokens=256, weights=None):
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

    def gpu_hidden_codes(self, ws) -> np.ndarray:
        """The kernel's E4M3 intermediate codes left in `ws` by the last forward
        call, as uint8 [T, k, I] in natural i order."""
        import w4a8_moe_gb300 as lib
        off = lib.moe_w4a8_workspace_layout(self.T, self.H, self.I, self.E, self.k)["hq"]
        A = self.T * self.k
        rows = ws[off:off + A * self.I].view(A, self.I).cpu().numpy()
        nat = rows[:, kperm_index(self.I)]
        out = np.empty((A, self.I), np.uint8)
        out[self.o_sorted] = nat
        return out.reshape(self.T, self.k, self.I)

    def oracle_hidden_codes(self, tokens):
        return oracle.moe_hidden_codes(self.o_xq, self.o_s1, self.o_pgu, self.o_sgu, self.s2, self.act,
                                       self.o_ids, tokens, nthreads=oracle_threads())

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
