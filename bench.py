"""Benchmark of the W4A8 MoE layer on GB300.

One step = one pass of the whole hot path over one batch of tokens: moe_route
(softmax top-k, histogram, permutation) + moe_w4a8_forward (gather, grouped
gate_up GEMM with gating and E4M3 requantization, grouped down GEMM, weighted
combine), with the E4M3 activations and router logits resident in HBM.

The headline workload is the largest single-GPU layer of the suite, the
Grok-1-shaped prefill layer: 32768 tokens (32 sequences of 1024), hidden 6144,
intermediate 32768, 8 experts, top-2, GELU(tanh)-gated, skewed routing
(per-expert logit bias N(0, 1)); 7.92e13 FLOP per step, bound by the FP8
tensor cores. The same JSON line carries, under "suite", the decode-shaped
layers (Mixtral-8x7B T32; Grok-1 T32, T8, T1; bound by weight bytes) and the
block-FP8 dense projections, each measured in the same run. --config picks
another headline layer.

Timed steps are replayed from captured CUDA graphs (no per-kernel events
inside them); per-kernel durations come from separate eager steps that carry
CUDA events. `e2e` times the same step through the public Python API with the
step's inputs copied from pinned host memory and its output copied back.

`python bench.py --impl reference` times the CPU oracle, as it stands, on the
same workload: every step runs the oracle's routing on all tokens and its
exact-integer MoE forward on a bounded sample of tokens.

Multi-GPU (torchrun): every rank runs its own replica of the layer on its own
tokens (the path has no exchange step), timed between barriers; value is the
total tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W4A8 MoE layer tokens/s"
UNIT = "tokens/s"
HEADLINE = "grok_prefill"
GRAPH_STEPS = 50          # steps captured per CUDA graph
PROFILE_STEPS = {"decode": 16, "prefill": 3}   # eager steps that carry per-kernel events


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--cpu-sample-tokens", type=int, default=0,
                    help="tokens in the oracle sample (0: sized for about 15 s of CPU work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-suite", action="store_true", help="headline layer only")
    ap.add_argument("--extra", action="store_true",
                    help="also measure the router gate, the dynamic intermediate scale and the "
                         "per-tensor FP8 linear (into the suite)")
    ap.add_argument("--only", default=None,
                    help="skip the headline layer and print only the suite entries whose workload "
                         "name contains this text (for profiling one workload)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- dist
def dist_setup(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, tokens_per_rank: int, steps: int, ms_slowest: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms_slowest / 1e3)


# DRAM bytes (read + write) per launch of a GEMM kernel from ncu captures
# (summarized with their commands under profiles/), valid only for the GEMM
# sources they were taken on: moe.cu without its row kernels (gather,
# intermediate quantizer, combine: the part from "// Gather:" up to
# "// Host side"), the PTX and scheduling headers the GEMM includes, and the
# moe.cu section of internal.h, comments left out. A changed GEMM reports
# null.
NCU_TRAFFIC = {
    "sources": ["w4a8_moe_gb300/csrc/moe.cu", "w4a8_moe_gb300/csrc/ptx.cuh", "w4a8_moe_gb300/csrc/sched.cuh",
                "w4a8_moe_gb300/csrc/internal.h"],
    "sha256": "53d58d5cfe022ee6aa66c4e0bab6853ec02489eb9603ebc8109b957d6fa66c93",
    "grok_prefill:gate_up": 11414465792 + 2116776192,
    "mixtral_decode:one_launch": 705904640 + 4985856,
}


def gemm_source_digest(read=None) -> str:
    """sha256 over the GEMM's sources (see NCU_TRAFFIC), comments and blank
    lines left out (they do not change the kernel)."""
    import hashlib
    import re
    read = read or (lambda f: open(os.path.join(ROOT, f), "rb").read())
    h = hashlib.sha256()
    for f in NCU_TRAFFIC["sources"]:
        data = read(f)
        if f.endswith("moe.cu"):
            a, b = data.index(b"// Gather: "), data.index(b"// Host side")
            data = data[:a] + data[b:]
        if f.endswith("internal.h"):
            a = data.index(b"// ---- moe.cu")
            data = data[a:data.index(b"// ---- ", a + 1)]
        text = re.sub(r"/\*.*?\*/", "", data.decode(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()


def ncu_traffic(key: str):
    if NCU_TRAFFIC.get(key) is None or gemm_source_digest() != NCU_TRAFFIC["sha256"]:
        return None
    return NCU_TRAFFIC[key]


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi SM clock and throttle reasons, sampled from before the warm-up
    to after the timed region; summary() keeps the samples taken inside the
    timed region (the one nearest to it if none fell inside)."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []     # (host time, fields)
        self.window = None
        self._stop = threading.Event()
        self._th = None

    def _query(self):
        cmd = ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits"]
        try:
            t = time.perf_counter()
            out = subprocess.run(cmd, capture_output=True, text=True, timeout=5).stdout.strip()
            if out:
                self.rows.append((t, [c.strip() for c in out.split(",")]))
        except Exception:
            pass

    def _poll(self):
        while not self._stop.is_set():
            self._query()
            self._stop.wait(0.05)

    def start(self):
        self._th = threading.Thread(target=self._poll, daemon=True)
        self._th.start()
        return self

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        self._stop.set()
        if self._th:
            self._th.join(timeout=10)

    def summary(self):
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        rows = self.rows
        if self.window and rows:
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
            if not inside:
                mid = 0.5 * (self.window[0] + self.window[1])
                inside = [min(rows, key=lambda r: abs(r[0] - mid))]
            rows = inside
        rows = [r[1] for r in rows]
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if len(r) > 2 and num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 3 + i and r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w": statistics.median(pw) if pw else None}


def load_peaks():
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(pp)) if os.path.exists(pp) else {}


def peaks():
    p = load_peaks()
    src = "of measured (MEASURED_PEAKS.json)" if p else "of fallback"
    return {"hbm": p.get("hbm_gbs", 6800.0), "hbm_src": f"hbm_gbs, burst copy, {src}",
            # FP8 dense peak: the measured bf16 burst peak times the nominal fp8/bf16 ratio (2)
            "fp8": 2.0 * p.get("bf16_tflops", 1900.0),
            "fp8_src": f"2 x bf16_tflops (burst; nominal fp8/bf16 ratio 2), {src}"}


# ----------------------------------------------------------------------------- workload
def algorithmic_bytes(shape, counts):
    """Weight bytes the layer must read (experts with tokens only) plus activation I/O."""
    H, I = shape.H, shape.I
    active = sum(1 for c in counts if c > 0)
    gate_up = active * (2 * I * H // 2 + 2 * I * 4)
    down = active * (H * I // 2 + H * 4)
    act_io = shape.T * H * (1 + 2)
    return gate_up, down, act_io


def layer_flops(shape):
    """2 * assignments * (gate_up 2I*H + down H*I): routed assignments only."""
    A = shape.T * shape.k
    return 2.0 * A * 2 * shape.I * shape.H, 2.0 * A * shape.H * shape.I


def make_weights(H, I, E, seed, dev):
    """Seeded bf16 expert weights and their library quantization."""
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth
    w = synth.moe_weights(H, I, E, seed=seed, device=dev)
    w_gu, s_gu = lib.w4a8_quantize_experts(w["w_gu"])
    w_d, s_d = lib.w4a8_quantize_experts(w["w_d"])
    torch.cuda.synchronize()
    return {"bf16_gu": w["w_gu"], "bf16_d": w["w_d"], "w_gu": w_gu, "s_gu": s_gu, "w_d": w_d, "s_d": s_d}


def static_hidden_scale(x_bf16, logits, w_gu_bf16, shape, tokens=256):
    """Static scale of the intermediate activation for the synthetic layer:
    max|h| / 448 over the first min(T, 256) tokens, calibrated in float32 on
    the unquantized bf16 weights (the offline calibration a static scheme
    implies; input preparation, not a timed step)."""
    import torch
    n = min(shape.T, tokens)
    x = x_bf16[:n].float()
    top = torch.topk(logits[:n], shape.k, dim=1).indices
    hmax = 0.0
    for e in range(shape.E):
        rows = (top == e).any(1).nonzero().flatten()
        if rows.numel() == 0:
            continue
        gu = x[rows] @ w_gu_bf16[e].float().t()
        g, u = gu[:, :shape.I], gu[:, shape.I:]
        a = torch.nn.functional.silu(g) if shape.act == 0 else torch.nn.functional.gelu(g, approximate="tanh")
        hmax = max(hmax, float((a * u).abs().max()))
        del gu, g, u, a
    return hmax / 448.0 if hmax > 0 else 1.0


def prepare_moe(shape, seed, dev, weights):
    """Seeded synthetic layer on the device: routing inputs, E4M3 activations
    with their calibrated scale, the calibrated static intermediate scale,
    workspaces, and one routing of the logits."""
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth

    inp = synth.moe_inputs(shape.T, shape.H, shape.I, shape.E, bias_std=shape.bias_std, seed=seed,
                           device=dev, weights=False)
    xq, a1 = lib.w4a8_quantize_act(inp["x"], compute_scale=True)      # calibration of a1
    s2 = static_hidden_scale(inp["x"], inp["logits"], weights["bf16_gu"], shape)
    st = {k_: weights[k_] for k_ in ("w_gu", "s_gu", "w_d", "s_d")}
    st.update({"xq": xq, "a1": a1, "a2": torch.tensor([s2], dtype=torch.float32, device=dev),
               "logits": inp["logits"], "x": inp["x"]})
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    st["route_ws"] = torch.zeros(lib.moe_route_workspace_size(T, E, k), dtype=torch.uint8, device=dev)
    st["ws"] = torch.zeros(lib.moe_w4a8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    st["out"] = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    st["route"] = lib.moe_route(st["logits"], k, ws=st["route_ws"])
    torch.cuda.synchronize()
    return st


def moe_step(lib, shape, st):
    """One step of the hot path: route + forward, inputs resident on the device."""
    lib.moe_route(st["logits"], shape.k, out=st["route"], ws=st["route_ws"])
    lib.moe_w4a8_forward(st["xq"], st["a1"], st["w_gu"], st["s_gu"], st["w_d"], st["s_d"], st["a2"],
                         shape.act, st["route"], out=st["out"], ws=st["ws"])


def capture(fn, n):
    """A CUDA graph of n consecutive calls of fn (None for n = 0)."""
    import torch
    if n == 0:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(n):
            fn()
    return g


def time_graph_steps(fn, steps, warmup, world, clock=None, per=None):
    """Exactly `steps` calls of fn, replayed from CUDA graphs of `per` (default
    up to GRAPH_STEPS) calls, between barriers, timed with CUDA events on the
    launching stream; returns the slowest rank's total milliseconds."""
    import torch
    for _ in range(max(3, warmup)):
        fn()
    torch.cuda.synchronize()
    per = min(steps, per or GRAPH_STEPS)
    full, rem = divmod(steps, per)
    g_main, g_rem = capture(fn, per), capture(fn, rem)
    g_main.replay()                                  # one untimed replay of each graph
    if g_rem is not None:
        g_rem.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    start.record(stream)
    for _ in range(full):
        g_main.replay()
    if g_rem is not None:
        g_rem.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if clock is not None:
        clock.mark(t0, t1)
    barrier(world)
    return max_over_ranks(start.elapsed_time(stop), world)


def kernel_times(lib, fn, n):
    """Mean per-kernel milliseconds of the forward over n eager steps that carry
    the library's profile events: [0]-[1] the gate_up GEMM launch (both
    projections when they share one launch), [1]-[2] the down launch, [2]-[3]
    the combine. Not part of any timed region."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for e4 in ev:
        for e in e4:
            e.record()
    torch.cuda.synchronize()
    for e4 in ev:
        lib.w4a8_set_profile_events(e4)
        fn()
        lib.w4a8_set_profile_events(None)
    torch.cuda.synchronize()
    return [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ev) for i in range(3)]


def measure_moe(lib, shape, st, steps, warmup, world, clock=None):
    """Layer step time (graph replay), per-kernel times, and the roofline
    bookkeeping of one MoE layer."""
    import torch
    fn = lambda: moe_step(lib, shape, st)
    ms_total = time_graph_steps(fn, steps, warmup, world, clock)
    err = lib.w4a8_device_error(st["ws"])
    assert err == 0, "device error word set"
    counts = st["route"].counts.cpu().tolist()
    kind = "prefill" if shape.T > 256 else "decode"
    ms_gu, ms_dn, ms_fin = kernel_times(lib, fn, PROFILE_STEPS[kind])
    plan = lib.moe_w4a8_plan(shape.T, shape.H, shape.I, shape.E, shape.k)
    gu_b, dn_b, act_b = algorithmic_bytes(shape, counts)
    torch.cuda.synchronize()
    return {"ms_per_step": ms_total / steps, "ms_total": ms_total, "plan": plan,
            "one_launch": bool(plan["one_launch"]), "ms_gu": ms_gu, "ms_dn": ms_dn, "ms_fin": ms_fin,
            "gu_bytes": gu_b, "dn_bytes": dn_b, "act_bytes": act_b,
            "active_experts": sum(1 for c in counts if c > 0)}


def moe_e2e(lib, shape, st, steps, world):
    """The step through the public API from host buffers, as a serving loop
    runs it: every step copies its inputs (bf16 x, fp32 logits) from pinned
    host memory, quantizes the activations with the static scale, routes,
    runs the forward and copies its bf16 output back to pinned host memory.
    The upload of step i+1 and the readback of step i run on two copy streams
    while step i+1 computes (double-buffered device inputs and outputs); the
    host waits for each step's output one step behind, and for the last at
    the end. Wall clock."""
    import torch
    T, H, k = shape.T, shape.H, shape.k
    hx = st["x"].cpu().pin_memory()
    hl = st["logits"].cpu().pin_memory()
    hout = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx = [torch.empty_like(st["x"]) for _ in range(2)]
    dl = [torch.empty_like(st["logits"]) for _ in range(2)]
    dout = [st["out"], torch.empty_like(st["out"])]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    for e in in_free + out_free:
        e.record(comp)

    def step(i):
        s = i % 2
        with torch.cuda.stream(up):
            up.wait_event(in_free[s])                 # step i-2 has consumed dx[s], dl[s]
            dx[s].copy_(hx, non_blocking=True)
            dl[s].copy_(hl, non_blocking=True)
            in_ready[s].record(up)
        comp.wait_event(in_ready[s])
        lib.w4a8_quantize_act(dx[s], scale=st["a1"], compute_scale=False, out=st["xq"])
        lib.moe_route(dl[s], k, out=st["route"], ws=st["route_ws"])
        in_free[s].record(comp)
        comp.wait_event(out_free[s])                  # step i-2's output has been read back
        lib.moe_w4a8_forward(st["xq"], st["a1"], st["w_gu"], st["s_gu"], st["w_d"], st["s_d"], st["a2"],
                             shape.act, st["route"], out=dout[s], ws=st["ws"])
        out_ready[s].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(out_ready[s])
            hout[s].copy_(dout[s], non_blocking=True)
            out_free[s].record(down)

    # the pipelined step gives what a device-resident step gives, bit for bit
    moe_step(lib, shape, st)
    torch.cuda.synchronize()
    ref = st["out"].cpu()
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    assert torch.equal(hout[0].view(torch.int16), ref.view(torch.int16)), "e2e step differs from a device step"
    barrier(world)
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
        if i >= 1:
            out_free[(i - 1) % 2].synchronize()       # step i-1's output is on the host
    out_free[(steps - 1) % 2].synchronize()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    return {"value": world * T * steps / e2e_s, "unit": UNIT,
            "h2d_bytes_per_step": hx.numel() * 2 + hl.numel() * 4,
            "d2h_bytes_per_step": hout[0].numel() * 2,
            "mode": "pipelined: upload of step i+1 and readback of step i overlap step i+1's compute",
            "steps": steps}


def moe_roofline(shape, m, pk, traffic_key=None):
    """Roofline of the dominant kernel: the GEMM launch that carries gate_up
    (both projections when they share one launch). Prefill-sized layers are
    bound by the FP8 tensor cores (FLOP/s), decode-sized ones by weight bytes."""
    fl_gu, fl_dn = layer_flops(shape)
    traffic = ncu_traffic(traffic_key) if traffic_key else None
    common = {"traffic": traffic,
              "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
              "per_launch_ms": m["ms_gu"]}
    if shape.T > 256:
        tf = fl_gu / (m["ms_gu"] * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": "moe_gemm_kernel<gate_up>", "achieved": tf, "peak": pk["fp8"],
                "unit": "TFLOP/s", "frac": tf / pk["fp8"], "peak_source": pk["fp8_src"],
                "algorithmic_flops": fl_gu, **common,
                "down": {"kernel": "moe_gemm_kernel<down>", "per_launch_ms": m["ms_dn"],
                         "achieved": fl_dn / (m["ms_dn"] * 1e-3) / 1e12, "unit": "TFLOP/s"},
                "step_breakdown_ms": {"gate_up": m["ms_gu"], "down": m["ms_dn"], "finalize": m["ms_fin"],
                                      "rest_net_of_overlap": m["ms_per_step"] - m["ms_gu"] - m["ms_dn"]
                                      - m["ms_fin"]}}
    w_bytes = m["gu_bytes"] + (m["dn_bytes"] if m["one_launch"] else 0)
    gbs = w_bytes / (m["ms_gu"] * 1e-3) / 1e9
    name = "moe_gemm_kernel<gate_up+down, one launch>" if m["one_launch"] else "moe_gemm_kernel<gate_up>"
    out = {"bound": "hbm", "kernel": name, "achieved": gbs, "peak": pk["hbm"], "unit": "GB/s",
           "frac": gbs / pk["hbm"], "peak_source": pk["hbm_src"], "algorithmic_bytes": w_bytes, **common}
    if m["one_launch"]:
        out["step_breakdown_ms"] = {"gate_up+down": m["ms_gu"], "finalize": m["ms_fin"],
                                    "rest_net_of_overlap": m["ms_per_step"] - m["ms_gu"] - m["ms_fin"]}
    else:
        out["step_breakdown_ms"] = {"gate_up": m["ms_gu"], "down": m["ms_dn"], "finalize": m["ms_fin"],
                                    "rest_net_of_overlap": m["ms_per_step"] - m["ms_gu"] - m["ms_dn"]
                                    - m["ms_fin"]}
    return out


def layer_fields(shape, m, pk):
    """Whole-layer throughput against the layer's bound."""
    if shape.T > 256:
        fl = sum(layer_flops(shape))
        tf = fl / (m["ms_per_step"] * 1e-3) / 1e12
        return {"layer_tflops": tf, "layer_fp8_frac": tf / pk["fp8"]}
    b = m["gu_bytes"] + m["dn_bytes"] + m["act_bytes"]
    gbs = b / (m["ms_per_step"] * 1e-3) / 1e9
    return {"layer_weight_gbs": gbs, "layer_hbm_frac": gbs / pk["hbm"], "active_experts": m["active_experts"]}


def config_dict(shape, world):
    return {"workload": shape.name, "tokens_per_step": shape.T, "hidden": shape.H,
            "intermediate": shape.I, "experts": shape.E, "top_k": shape.k,
            "activation": "SiLU-gated" if shape.act == 0 else "GELU-tanh-gated",
            "global_batch": shape.T * world, "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (packed expert weights stream from HBM every step); no flush"}


# ----------------------------------------------------------------------------- suite
def suite_moe_entry(lib, shape, st, steps, pk, traffic_key=None):
    m = measure_moe(lib, shape, st, steps, 10, 1)
    return {"workload": shape.name, "ms_per_step": m["ms_per_step"], "tokens_per_s": shape.T / (m["ms_per_step"] * 1e-3),
            "steps": steps, "timing": f"{steps} steps replayed from CUDA graphs", **layer_fields(shape, m, pk),
            "roofline": moe_roofline(shape, m, pk, traffic_key), "plan": m["plan"]}


def rotating_copies(weight_bytes, l2_bytes, at_least=4):
    """Weight copies to rotate through so that the set exceeds twice the L2."""
    return max(at_least, math.ceil(2.2 * l2_bytes / weight_bytes))


def wanted(name, only):
    return only is None or only in name


def suite_block_fp8(lib, dev, pk, l2_bytes, only=None):
    """Block-FP8 dense projections: every call reads its weights from HBM
    (rotating copies totalling more than twice the L2)."""
    import torch

    from w4a8_moe_gb300 import synth
    out = []
    for (N, K) in synth.BLOCK_FP8_SHAPES:
        if not any(wanted(f"block-FP8 linear N{N} K{K} M{M}", only) for M in synth.BLOCK_FP8_M):
            continue
        w = synth.block_fp8_inputs(1, N, K, seed=0, device=dev)["w"].float()
        blk = w.view(N // 128, 128, K // 128, 128).abs().amax(dim=(1, 3))
        wsi = torch.where(blk > 0, blk / 448.0, torch.ones_like(blk))
        q = (w / wsi.repeat_interleave(128, 0).repeat_interleave(128, 1)).to(torch.float8_e4m3fn)
        q = q.view(torch.uint8).contiguous()
        del w
        ncopy = rotating_copies(N * K, l2_bytes)
        wl = [q.clone() for _ in range(ncopy)]
        sl = [wsi.clone() for _ in range(ncopy)]
        for M in synth.BLOCK_FP8_M:
            if not wanted(f"block-FP8 linear N{N} K{K} M{M}", only):
                continue
            x = synth.block_fp8_inputs(M, N, K, seed=9, device=dev)["x"]
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsp = torch.zeros(lib.fp8_block_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            per = ncopy * max(1, GRAPH_STEPS // ncopy)    # every graph holds whole rotations
            iters = per * max(1, (400 if M <= 64 else 40) // per)
            state = {"i": 0}

            def call():
                i = state["i"] % ncopy
                state["i"] += 1
                lib.fp8_block_linear(x, wl[i], sl[i], out=y, ws=wsp)
            ms = time_graph_steps(call, iters, 2 * ncopy, 1, per=per) / iters
            assert lib.w4a8_device_error(wsp) == 0, "device error word set"
            nbytes = N * K + 4 * (N // 128) * (K // 128) + 2 * M * K + 2 * M * N
            flops = 2.0 * M * N * K
            e = {"workload": f"block-FP8 linear N{N} K{K} M{M}", "ms_per_call": ms,
                 "gbs": nbytes / (ms * 1e-3) / 1e9, "tflops": flops / (ms * 1e-3) / 1e12,
                 "l2": f"{ncopy} rotating weight copies ({ncopy * N * K / 1e6:.0f} MB > 2 x L2)"}
            if M <= 64:
                e.update({"bound": "hbm", "frac": e["gbs"] / pk["hbm"], "peak": pk["hbm"], "unit": "GB/s"})
            else:
                e.update({"bound": "tensor", "frac": e["tflops"] / pk["fp8"], "peak": pk["fp8"],
                          "unit": "TFLOP/s"})
            out.append(e)
        del wl, sl
        torch.cuda.empty_cache()
    return out


def suite_extra(lib, dev, pk, l2_bytes, st_mix, mix, only=None):
    """The rows beyond the hot path proper: per-tensor FP8 linear, router gate
    fused with routing, and the dynamic intermediate scale."""
    import torch

    from w4a8_moe_gb300 import synth
    out = []
    for (N, K) in synth.FP8_LINEAR_SHAPES:
        if not any(wanted(f"per-tensor FP8 linear N{N} K{K} M{M}", only) for M in synth.FP8_LINEAR_M):
            continue
        ncopy = rotating_copies(N * K, l2_bytes)
        wl, swl = [], []
        w = synth.fp8_linear_inputs(1, N, K, seed=0, device=dev)["w"]
        q, s_ = lib.w4a8_quantize_act(w)
        del w
        wl = [q.clone() for _ in range(ncopy)]
        swl = [s_.clone() for _ in range(ncopy)]
        for M in synth.FP8_LINEAR_M:
            if not wanted(f"per-tensor FP8 linear N{N} K{K} M{M}", only):
                continue
            x = synth.fp8_linear_inputs(M, N, K, seed=9, device=dev)["x"]
            xq, sx = lib.w4a8_quantize_act(x)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsp = torch.zeros(lib.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            per = ncopy * max(1, GRAPH_STEPS // ncopy)
            iters = per * max(1, (400 if M <= 64 else 40) // per)
            state = {"i": 0}

            def call():
                i = state["i"] % ncopy
                state["i"] += 1
                lib.fp8_linear(xq, sx, wl[i], swl[i], out=y, ws=wsp)
            ms = time_graph_steps(call, iters, 2 * ncopy, 1, per=per) / iters
            assert lib.w4a8_device_error(wsp) == 0, "device error word set"
            nbytes = N * K + M * K + 2 * M * N
            flops = 2.0 * M * N * K
            e = {"workload": f"per-tensor FP8 linear N{N} K{K} M{M}", "ms_per_call": ms,
                 "gbs": nbytes / (ms * 1e-3) / 1e9, "tflops": flops / (ms * 1e-3) / 1e12,
                 "l2": f"{ncopy} rotating weight copies"}
            if M <= 64:
                e.update({"bound": "hbm", "frac": e["gbs"] / pk["hbm"]})
            else:
                e.update({"bound": "tensor", "frac": e["tflops"] / pk["fp8"]})
            out.append(e)
        del wl, swl
        torch.cuda.empty_cache()

    for (T, H, E, k) in ((32, 4096, 8, 2), (32, 6144, 8, 2)):
        if not wanted(f"router gate + routing T{T} H{H} E{E} k{k}", only):
            continue
        inp = synth.router_gate_inputs(T, H, E, seed=0, device=dev)
        ws_g = torch.zeros(lib.moe_route_gate_workspace_size(T, H, E, k), dtype=torch.uint8, device=dev)
        r_out, _ = lib.moe_route_gate(inp["hidden"], inp["gate"], k, ws=ws_g)
        ms = time_graph_steps(lambda: lib.moe_route_gate(inp["hidden"], inp["gate"], k, out=r_out, ws=ws_g),
                              500, 20, 1) / 500
        out.append({"workload": f"router gate + routing T{T} H{H} E{E} k{k}", "us_per_call": ms * 1e3,
                    "launches": 1})

    if st_mix is None or not wanted(mix.name + ", intermediate scale calibrated per call (dynamic)", only):
        return out
    T, H, I, E, k = mix.T, mix.H, mix.I, mix.E, mix.k
    wsd = torch.zeros(lib.moe_w4a8_dynamic_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    a2d = torch.empty(1, dtype=torch.float32, device=dev)

    def dyn_step():
        lib.moe_route(st_mix["logits"], k, out=st_mix["route"], ws=st_mix["route_ws"])
        lib.moe_w4a8_forward_dynamic(st_mix["xq"], st_mix["a1"], st_mix["w_gu"], st_mix["s_gu"], st_mix["w_d"],
                                     st_mix["s_d"], mix.act, st_mix["route"], out=st_mix["out"], a2_out=a2d,
                                     ws=wsd)
    ms = time_graph_steps(dyn_step, 500, 20, 1) / 500
    assert lib.w4a8_device_error(wsd) == 0, "device error word set"
    out.append({"workload": mix.name + ", intermediate scale calibrated per call (dynamic)",
                "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3), "dynamic_a2": a2d.item()})
    return out


# ----------------------------------------------------------------------------- oracle side
def oracle_layer(shape, seed=0):
    """The same seeded layer for the oracle: inputs drawn by the shared
    generators (on the GPU when there is one, for speed; no library call),
    then quantized, routed and calibrated by the oracle on the host. Expert
    slices are quantized on parallel host threads (the oracle's own function,
    called once per expert)."""
    import numpy as np
    import torch

    import oracle
    from w4a8_moe_gb300 import synth
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.moe_inputs(shape.T, shape.H, shape.I, shape.E, bias_std=shape.bias_std, seed=seed, device=dev)
    inp = {k_: v.cpu() for k_, v in inp.items()}
    if dev == "cuda":
        torch.cuda.empty_cache()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    threads = oracle.cores()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(shape.E, threads))) as ex:
        gu = list(ex.map(lambda e: oracle.quantize_experts(bits(inp["w_gu"][e:e + 1])), range(shape.E)))
        dn = list(ex.map(lambda e: oracle.quantize_experts(bits(inp["w_d"][e:e + 1])), range(shape.E)))
    pgu = np.concatenate([g[0] for g in gu]), np.concatenate([g[1] for g in gu])
    pd = np.concatenate([d[0] for d in dn]), np.concatenate([d[1] for d in dn])
    s1 = oracle.act_scale(bits(inp["x"]))
    xq = oracle.quantize_act(bits(inp["x"]), s1)
    logits = inp["logits"].numpy()
    ids, w = oracle.route(logits, shape.k)
    cal = synth.calibration_tokens(shape.T)
    s2 = oracle.moe_hidden_scale(xq, s1, pgu[0], pgu[1], shape.act, ids, cal, nthreads=threads)
    return {"xq": xq, "s1": s1, "pgu": pgu, "pd": pd, "logits": logits, "s2": s2, "threads": threads}


def oracle_step(shape, L, tokens, nthreads):
    """One oracle step on the sample: routing of every token's logits, the
    permutation, and the exact-integer MoE forward of the sampled tokens."""
    import oracle
    ids, w = oracle.route(L["logits"], shape.k)
    oracle.permute(ids, shape.E)
    return oracle.moe_forward(L["xq"], L["s1"], L["pgu"][0], L["pgu"][1], L["pd"][0], L["pd"][1], L["s2"],
                              shape.act, ids, w, tokens=tokens, nthreads=nthreads)


def sample_size(shape, L, target_s, requested):
    """Tokens per oracle step for about target_s seconds on all host cores."""
    if requested:
        return min(shape.T, requested), None
    t0 = time.perf_counter()
    oracle_step(shape, L, [0], 1)
    one = time.perf_counter() - t0
    return max(1, min(shape.T, int(target_s * L["threads"] / max(one, 1e-6)))), one


def cpu_baseline(args, shape):
    """The oracle, as it stands, on a bounded sample of the same layer."""
    L = oracle_layer(shape)
    n, one = sample_size(shape, L, 15.0, args.cpu_sample_tokens)
    t0 = time.perf_counter()
    oracle_step(shape, L, list(range(n)), L["threads"])
    dt = time.perf_counter() - t0
    out = {"value": n / dt, "unit": UNIT, "cores": L["threads"], "kind": "oracle",
           "sample": f"tokens 0..{n - 1} of the {shape.T}-token {shape.name} layer: routing and permutation of "
                     f"all {shape.T} tokens + exact-integer MoE forward of the {n} sampled tokens, "
                     f"{L['threads']} threads, {dt:.1f} s"}
    if n < shape.T:
        # every token costs the same (k assignments of the full H x I work)
        out["extrapolated_full_layer_s"] = shape.T / out["value"]
        out["extrapolation"] = "full-layer time extrapolated from the sample by token count (equal flops per token)"
    if one is not None:
        out["single_thread"] = {"value": 1.0 / one, "unit": UNIT,
                                "sample": "token 0 of the same layer, 1 thread"}
    return out


def run_reference(args, shape, world):
    """The reference arm: the oracle on the host cores, `warmup` untimed and
    `steps` timed steps, each one the oracle's routing of all tokens plus its
    forward on a fixed sample of tokens."""
    L = oracle_layer(shape)
    n, _ = sample_size(shape, L, 1.0, args.cpu_sample_tokens)
    toks = list(range(n))
    for _ in range(args.warmup):
        oracle_step(shape, L, toks, L["threads"])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(shape, L, toks, L["threads"])
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n * args.steps / total
    sample = (f"tokens 0..{n - 1} of the {shape.T}-token {shape.name} layer per step: routing and permutation "
              f"of all {shape.T} tokens + exact-integer MoE forward of the sample, {L['threads']} threads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "tokens_per_step": n, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int64+f64", "data": "synthetic", "config": config_dict(shape, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": L["threads"], "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- main
def run_ours(args, rank, world):
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth

    shape = synth.MOE_SHAPES[args.config]
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    weights = make_weights(shape.H, shape.I, shape.E, rank, dev)
    st = prepare_moe(shape, rank, dev, weights)
    # the Grok-1 decode layers of the suite share the headline's weights
    suite_on = (not args.no_suite) and world == 1
    grok = [n for n in ("grok_decode", "grok_decode_t8", "grok_decode_t1")
            if suite_on and synth.MOE_SHAPES[n].H == shape.H and synth.MOE_SHAPES[n].I == shape.I
            and synth.MOE_SHAPES[n].E == shape.E]
    grok_st = {n: prepare_moe(synth.MOE_SHAPES[n], 0, dev, weights) for n in grok}
    del weights["bf16_gu"], weights["bf16_d"]
    torch.cuda.empty_cache()

    clock = ClockSampler(torch.cuda.current_device()).start()
    m = measure_moe(lib, shape, st, args.steps, args.warmup, world, clock)
    clock.stop()
    e2e = moe_e2e(lib, shape, st, max(3, min(args.steps, 20)), world)
    res = {"m": m, "e2e": e2e, "clocks": clock.summary(), "shape": shape, "pk": pk}
    if not suite_on:
        return res

    suite = []
    for n in grok:
        s = synth.MOE_SHAPES[n]
        suite.append(suite_moe_entry(lib, s, grok_st.pop(n), max(args.steps, 500), pk))
    del st, grok_st
    torch.cuda.empty_cache()
    mix = synth.MOE_SHAPES["mixtral_decode"]
    if args.config != "mixtral_decode":
        wm = make_weights(mix.H, mix.I, mix.E, 0, dev)
        st_mix = prepare_moe(mix, 0, dev, wm)
        del wm
        torch.cuda.empty_cache()
        suite.append(suite_moe_entry(lib, mix, st_mix, max(args.steps, 2000), pk, "mixtral_decode:one_launch"))
    else:
        st_mix = None
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    suite += suite_block_fp8(lib, dev, pk, l2)
    if args.extra:
        suite += suite_extra(lib, dev, pk, l2, st_mix, mix)
    res["suite"] = suite
    return res


def run_only(args):
    """Only the suite entries whose workload contains args.only (one JSON line
    each), e.g. to profile one workload under ncu."""
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = []
    for n in ("grok_decode", "grok_decode_t8", "grok_decode_t1", "mixtral_decode"):
        s = synth.MOE_SHAPES[n]
        if wanted(s.name, args.only):
            w = make_weights(s.H, s.I, s.E, 0, dev)
            st = prepare_moe(s, 0, dev, w)
            del w
            torch.cuda.empty_cache()
            out.append(suite_moe_entry(lib, s, st, max(args.steps, 50), pk))
            del st
            torch.cuda.empty_cache()
    out += suite_block_fp8(lib, dev, pk, l2, args.only)
    out += suite_extra(lib, dev, pk, l2, None, synth.MOE_SHAPES["mixtral_decode"], args.only)
    for e in out:
        print(json.dumps(e), flush=True)


def main(argv=None):
    args = parse(argv)
    rank, world = dist_setup(args.gpus)
    from w4a8_moe_gb300 import synth
    shape = synth.MOE_SHAPES[args.config]

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, shape, world)), flush=True)
        return

    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    if args.only is not None:
        if rank == 0:
            run_only(args)
        return
    res = run_ours(args, rank, world)
    if rank != 0:
        return
    m, pk = res["m"], res["pk"]
    plan = m["plan"]
    key = {"grok_prefill": "grok_prefill:gate_up", "mixtral_decode": "mixtral_decode:one_launch"}.get(args.config)
    line = {"metric": METRIC, "value": throughput(world, shape.T, args.steps, m["ms_total"]), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xint4->f32",
            "data": "synthetic", "config": config_dict(shape, world),
            "timing": f"{args.steps} steps replayed from CUDA graphs of up to {GRAPH_STEPS} steps, "
                      "CUDA events on the launching stream",
            **layer_fields(shape, m, pk),
            "roofline": moe_roofline(shape, m, pk, key), "e2e": res["e2e"], "clocks": res["clocks"],
            # moe_route (one kernel up to 4096 assignments, else four) plus the
            # forward's launches (gather, GEMM launch(es), combine)
            "gpu_launches": ((1 if shape.T * shape.k <= 4096 else 4) + plan["launches"]) * args.steps,
            "plan": plan}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, shape)
    if "suite" in res:
        line["suite"] = res["suite"]
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
