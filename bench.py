"""Benchmark of the W4A8 MoE layer on GB300.

One step = one pass of the whole hot path over one batch of tokens: moe_route
(softmax top-k, histogram, permutation) + moe_w4a8_forward (gather, grouped
gate_up GEMM with gating and E4M3 requantization, grouped down GEMM, weighted
combine), with the E4M3 activations and router logits resident in HBM. The
default workload is the Mixtral-8x7B-shaped decode layer (32 tokens, hidden
4096, intermediate 14336, 8 experts, top-2, SiLU-gated, per-expert logit bias
N(0, 0.5)); --config selects another layer shape. Weights (705.7 MB packed for
8 active experts) are far larger than L2, so every step streams them from HBM.

Prints one JSON line (rank 0). `python bench.py --impl reference` times the CPU
oracle on a bounded sample of the same workload instead. `--suite` adds one
line per secondary workload (Grok-1-shaped layers, block-FP8 linear) after the
headline line.

Multi-GPU (torchrun): every rank runs its own replica of the layer on its own
tokens (the path has no exchange step), timed between barriers; value is the
total tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
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
PROFILE_EVERY = 16   # timed steps per step that carries the per-kernel events


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral_decode")
    ap.add_argument("--cpu-sample-tokens", type=int, default=0,
                    help="tokens in the oracle sample (0: sized for ~15 s of CPU work)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--suite", action="store_true",
                    help="also print one line per secondary workload (Grok-1 layers, block-FP8)")
    return ap.parse_args()


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


# DRAM bytes (read + write) per launch of the GEMM kernel from one ncu capture
# of the Mixtral decode layer (summarized with its command under profiles/), valid only
# for the GEMM sources they were taken on: moe.cu without its row kernels
# (gather, intermediate quantizer, combine: the part from "// Gather:" up to
# "// Host side"), and the headers the GEMM includes, comments left out. A
# changed GEMM reports null.
NCU_TRAFFIC = {
    "sources": ["w4a8_moe_gb300/csrc/moe.cu", "w4a8_moe_gb300/csrc/ptx.cuh", "w4a8_moe_gb300/csrc/sched.cuh",
                "w4a8_moe_gb300/csrc/internal.h"],
    "sha256": "4130b854d288ead709d5c50d9e6e356976508b372508691037cea4cf94121a5a",
    "one_launch": 705919744 + 4460544,
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
        text = re.sub(r"/\*.*?\*/", "", data.decode(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()


def ncu_traffic(kernel: str):
    return NCU_TRAFFIC.get(kernel) if gemm_source_digest() == NCU_TRAFFIC["sha256"] else None


def throughput(world: int, tokens_per_rank: int, steps: int, ms_slowest: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms_slowest / 1e3)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi SM clock and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self._stop = threading.Event()
        self._th = None

    def _poll(self):
        cmd = ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits"]
        while not self._stop.is_set():
            try:
                out = subprocess.run(cmd, capture_output=True, text=True, timeout=5).stdout.strip()
                if out:
                    self.rows.append([c.strip() for c in out.split(",")])
            except Exception:
                pass
            self._stop.wait(0.1)

    def __enter__(self):
        self._th = threading.Thread(target=self._poll, daemon=True)
        self._th.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._th.join(timeout=10)
        if not self.rows:  # region shorter than one poll: take one sample now
            self._stop.clear()
            self._stop.set()
            cmd = ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                   "--format=csv,noheader,nounits"]
            try:
                out = subprocess.run(cmd, capture_output=True, text=True, timeout=5).stdout.strip()
                if out:
                    self.rows.append([c.strip() for c in out.split(",")])
            except Exception:
                pass

    def summary(self):
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 3 + i and r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- workload
def algorithmic_bytes(shape, counts):
    """Weight bytes the layer must read (experts with tokens only) plus activation I/O."""
    H, I = shape.H, shape.I
    active = sum(1 for c in counts if c > 0)
    gate_up = active * (2 * I * H // 2 + 2 * I * 4)
    down = active * (H * I // 2 + H * 4)
    act_io = shape.T * H * (1 + 2)
    return gate_up, down, act_io


def static_hidden_scale(inp, shape, tokens=8):
    """Static scale of the intermediate activation for the synthetic layer,
    calibrated in float32 on the unquantized bf16 weights over the first tokens
    (the offline calibration a static scheme implies)."""
    import torch
    x = inp["x"][:tokens].float()
    top = torch.topk(inp["logits"][:tokens], shape.k, dim=1).indices
    hmax = 0.0
    for t in range(x.shape[0]):
        for e in top[t].tolist():
            gu = inp["w_gu"][e].float() @ x[t]
            g, u = gu[:shape.I], gu[shape.I:]
            a = torch.nn.functional.silu(g) if shape.act == 0 else \
                torch.nn.functional.gelu(g, approximate="tanh")
            hmax = max(hmax, float((a * u).abs().max()))
    return hmax / 448.0 if hmax > 0 else 1.0


def prepare_moe(shape, seed, dev):
    """Seeded synthetic layer: packed weights, calibrated static scales, routing."""
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth

    inp = synth.moe_inputs(shape.T, shape.H, shape.I, shape.E, bias_std=shape.bias_std,
                           seed=seed, device=dev)
    w_gu, s_gu = lib.w4a8_quantize_experts(inp["w_gu"])
    w_d, s_d = lib.w4a8_quantize_experts(inp["w_d"])
    xq, a1 = lib.w4a8_quantize_act(inp["x"], compute_scale=True)      # calibration of a1
    s2 = static_hidden_scale(inp, shape)
    a2 = torch.tensor([s2], dtype=torch.float32, device=dev)
    st = {"w_gu": w_gu, "s_gu": s_gu, "w_d": w_d, "s_d": s_d, "xq": xq, "a1": a1, "a2": a2,
          "logits": inp["logits"], "x": inp["x"]}
    del inp
    torch.cuda.empty_cache()
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    st["route_ws"] = torch.zeros(lib.moe_route_workspace_size(T, E, k), dtype=torch.uint8, device=dev)
    st["ws"] = torch.zeros(lib.moe_w4a8_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    st["out"] = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    st["route"] = lib.moe_route(st["logits"], k, ws=st["route_ws"])
    return st


def moe_step(lib, shape, st):
    """One step of the hot path: route + forward, inputs resident on the device."""
    lib.moe_route(st["logits"], shape.k, out=st["route"], ws=st["route_ws"])
    lib.moe_w4a8_forward(st["xq"], st["a1"], st["w_gu"], st["s_gu"], st["w_d"], st["s_d"], st["a2"],
                         shape.act, st["route"], out=st["out"], ws=st["ws"])


def time_moe_steps(lib, shape, st, steps, warmup, world, clock_index=None):
    """K timed steps between barriers, CUDA events on the launching stream.
    Per-kernel events (recorded by the library around the two GEMMs and the
    combine) go into every PROFILE_EVERY-th step only: an event between two
    kernels stops the next one from launching early, so recording them in
    every step would slow the step it measures."""
    import torch

    stream = torch.cuda.current_stream()
    for _ in range(max(3, warmup)):
        moe_step(lib, shape, st)
    torch.cuda.synchronize()
    counts = st["route"].counts.cpu().tolist()
    sampled = list(range(0, steps, PROFILE_EVERY))
    ev = {i: [torch.cuda.Event(enable_timing=True) for _ in range(4)] for i in sampled}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e4 in ev.values():  # materialize the CUDA events before the timed region
        for e in e4:
            e.record(stream)
    barrier(world)
    torch.cuda.synchronize()
    clk = ClockSampler(clock_index if clock_index is not None else torch.cuda.current_device())
    with clk:
        start.record(stream)
        for i in range(steps):
            if i in ev:
                lib.w4a8_set_profile_events(ev[i])
                moe_step(lib, shape, st)
                lib.w4a8_set_profile_events(None)
            else:
                moe_step(lib, shape, st)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(start.elapsed_time(stop), world)
    assert lib.w4a8_device_error(st["ws"]) == 0, "device error word set"
    ms_gu = statistics.mean(e[0].elapsed_time(e[1]) for e in ev.values())
    ms_dn = statistics.mean(e[1].elapsed_time(e[2]) for e in ev.values())
    ms_fin = statistics.mean(e[2].elapsed_time(e[3]) for e in ev.values())
    gu_bytes, d_bytes, act_bytes = algorithmic_bytes(shape, counts)
    plan = lib.moe_w4a8_plan(shape.T, shape.H, shape.I, shape.E, shape.k)
    return {"ms_per_step": ms_total / steps, "clocks": clk.summary(), "plan": plan,
            # with one launch for both projections, events 0-1 bracket it and 1-2 nothing
            "kernels": {"gate_up_ms": ms_gu, "down_ms": ms_dn, "finalize_ms": ms_fin,
                        "one_launch": bool(plan["one_launch"]),
                        "route_gather_gaps_ms": ms_total / steps - ms_gu - ms_dn - ms_fin,
                        "gate_up_bytes": gu_bytes, "down_bytes": d_bytes, "act_bytes": act_bytes,
                        "active_experts": sum(1 for c in counts if c > 0)}}


def run_ours(args, rank, world):
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth

    shape = synth.MOE_SHAPES[args.config]
    dev = torch.device("cuda", torch.cuda.current_device())
    st = prepare_moe(shape, rank, dev)
    T, H, k = shape.T, shape.H, shape.k
    tm = time_moe_steps(lib, shape, st, args.steps, args.warmup, world)

    # the static-scale activation quantization that precedes the layer,
    # timed on its own (it is not part of the layer step)
    n_aq = 200
    for _ in range(5):
        lib.w4a8_quantize_act(st["x"], scale=st["a1"], compute_scale=False, out=st["xq"])
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s_ev.record()
    for _ in range(n_aq):
        lib.w4a8_quantize_act(st["x"], scale=st["a1"], compute_scale=False, out=st["xq"])
    e_ev.record()
    torch.cuda.synchronize()
    act_quant_ms = s_ev.elapsed_time(e_ev) / n_aq

    # end to end through the public API with host buffers: H2D of the step's
    # inputs (bf16 x, fp32 logits) from pinned memory, static-scale quantization,
    # route, forward, D2H of the bf16 output
    hx = st["x"].cpu().pin_memory()
    hl = st["logits"].cpu().pin_memory()
    hout = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    dx = torch.empty_like(st["x"])
    dl = torch.empty_like(st["logits"])

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dl.copy_(hl, non_blocking=True)
        lib.w4a8_quantize_act(dx, scale=st["a1"], compute_scale=False, out=st["xq"])
        lib.moe_route(dl, k, out=st["route"], ws=st["route_ws"])
        lib.moe_w4a8_forward(st["xq"], st["a1"], st["w_gu"], st["s_gu"], st["w_d"], st["s_d"], st["a2"],
                             shape.act, st["route"], out=st["out"], ws=st["ws"])
        hout.copy_(st["out"], non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    # Decode steps are replayed from a captured CUDA graph (the copies of the
    # step's inputs and output included), as a serving loop would; if capture
    # is not available the same calls run eagerly.
    run = e2e_step
    e2e_mode = "eager"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            e2e_step()
        graph.replay()
        torch.cuda.synchronize()
        run = graph.replay
        e2e_mode = "cuda_graph"
    except Exception as exc:   # noqa: BLE001 -- report and fall back
        print(f"graph capture unavailable ({exc}); timing the eager loop", file=sys.stderr)
        torch.cuda.synchronize()
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e_steps = max(10, min(args.steps, 500))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e_steps):
        run()
        torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    # the replayed step must give what an eager step gives, bit for bit
    got = hout.clone()
    e2e_step()
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), hout.view(torch.int16)), "e2e replay differs from an eager step"

    return {
        "ms_per_step": tm["ms_per_step"],
        "value": throughput(world, T, args.steps, tm["ms_per_step"] * args.steps),
        "e2e": {"value": world * T * e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": hx.numel() * 2 + hl.numel() * 4,
                "d2h_bytes_per_step": hout.numel() * 2, "mode": e2e_mode},
        "clocks": tm["clocks"],
        "kernels": tm["kernels"],
        "plan": tm["plan"],
        "act_quant_static_ms": act_quant_ms,
        "shape": shape,
    }


def load_peaks():
    pp = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(pp)) if os.path.exists(pp) else {}


def run_suite(args):
    """Secondary workloads, one JSON line each (not the headline): the Grok-1
    shaped layers (decode at 32, 8 and 1 tokens: weight GB/s against HBM;
    prefill at 32768 tokens: FP8 TFLOP/s against the dense FP8 peak) and the
    block-FP8 linear (GB/s at M <= 64, TFLOP/s at M = 4096)."""
    import torch

    import w4a8_moe_gb300 as lib
    from w4a8_moe_gb300 import synth

    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    # FP8 dense peak: the measured bf16 peak times the nominal fp8/bf16 ratio (2)
    fp8_burst = 2.0 * peaks.get("bf16_tflops", 1900.0)
    fp8_sust = 2.0 * peaks.get("bf16_tflops_sustained", 1700.0)
    src = "MEASURED_PEAKS.json" if peaks else "fallback"
    dev = torch.device("cuda", torch.cuda.current_device())
    for name, steps, warm in (("grok_decode", 200, 10), ("grok_decode_t8", 200, 10),
                              ("grok_decode_t1", 200, 10), ("grok_prefill", 6, 2)):
        shape = synth.MOE_SHAPES[name]
        st = prepare_moe(shape, 0, dev)
        tm = time_moe_steps(lib, shape, st, steps, warm, 1)
        kk = tm["kernels"]
        ms = tm["ms_per_step"]
        line = {"suite": True, "workload": shape.name, "ms_per_step": ms,
                "tokens_per_s": shape.T / (ms * 1e-3), "steps": steps, "warmup": warm,
                "kernels_ms": ({"gate_up+down": kk["gate_up_ms"], "finalize": kk["finalize_ms"]}
                               if kk["one_launch"] else
                               {"gate_up": kk["gate_up_ms"], "down": kk["down_ms"], "finalize": kk["finalize_ms"]}),
                "plan": tm["plan"],
                "active_experts": kk["active_experts"], "clocks": tm["clocks"]}
        wbytes = kk["gate_up_bytes"] + kk["down_bytes"] + kk["act_bytes"]
        if shape.T <= 256:
            gbs = wbytes / (ms * 1e-3) / 1e9
            line.update({"bound": "hbm", "layer_gbs": gbs, "peak_gbs": hbm, "frac": gbs / hbm,
                         "peak_source": src + " hbm_gbs"})
        else:
            flops = 2.0 * shape.T * shape.k * 3 * shape.H * shape.I
            tf = flops / (ms * 1e-3) / 1e12
            line.update({"bound": "tensor", "tflops": tf, "peak_tflops": fp8_sust,
                         "frac": tf / fp8_sust,
                         "peak_source": src + " bf16_tflops_sustained x 2 (nominal fp8/bf16)",
                         "gate_up_tflops": 2.0 * shape.T * shape.k * 2 * shape.H * shape.I
                         / (kk["gate_up_ms"] * 1e-3) / 1e12,
                         "down_tflops": 2.0 * shape.T * shape.k * shape.H * shape.I
                         / (kk["down_ms"] * 1e-3) / 1e12})
        print(json.dumps(line), flush=True)
        del st
        torch.cuda.empty_cache()

    # Mixtral decode with the intermediate scale calibrated on the device per call
    shape = synth.MOE_SHAPES["mixtral_decode"]
    st = prepare_moe(shape, 0, dev)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    wsd = torch.zeros(lib.moe_w4a8_dynamic_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    a2d = torch.empty(1, dtype=torch.float32, device=dev)

    def dyn_step():
        lib.moe_route(st["logits"], k, out=st["route"], ws=st["route_ws"])
        lib.moe_w4a8_forward_dynamic(st["xq"], st["a1"], st["w_gu"], st["s_gu"], st["w_d"], st["s_d"],
                                     shape.act, st["route"], out=st["out"], a2_out=a2d, ws=wsd)

    res = {}
    for name, fn in (("static", lambda: moe_step(lib, shape, st)), ("dynamic", dyn_step)):
        for _ in range(20):
            fn()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s_ev.record()
        for _ in range(1000):
            fn()
        e_ev.record()
        torch.cuda.synchronize()
        res[name] = s_ev.elapsed_time(e_ev) / 1000
    assert lib.w4a8_device_error(wsd) == 0, "device error word set"
    print(json.dumps({"suite": True, "workload": shape.name + ", intermediate scale static vs dynamic",
                      "ms_per_step": res, "tokens_per_s": {n: T / (v * 1e-3) for n, v in res.items()},
                      "dynamic_a2": a2d.item()}), flush=True)
    del st
    torch.cuda.empty_cache()

    # router gate fused with routing (one launch at decode) against the gate
    # product as a separate library matmul followed by moe_route
    for (T, H, E, k) in ((32, 4096, 8, 2), (32, 6144, 8, 2)):
        inp = synth.router_gate_inputs(T, H, E, seed=0, device=dev)
        ws_g = torch.zeros(lib.moe_route_gate_workspace_size(T, H, E, k), dtype=torch.uint8, device=dev)
        ws_r = torch.zeros(lib.moe_route_workspace_size(T, E, k), dtype=torch.uint8, device=dev)
        r_out, _ = lib.moe_route_gate(inp["hidden"], inp["gate"], k, ws=ws_g)
        lg = torch.empty(T, E, dtype=torch.float32, device=dev)

        def fused():
            lib.moe_route_gate(inp["hidden"], inp["gate"], k, out=r_out, ws=ws_g)

        def unfused():
            torch.matmul(inp["hidden"].float(), inp["gate"].float().t(), out=lg)
            lib.moe_route(lg, k, out=r_out, ws=ws_r)

        res = {}
        for name, fn in (("fused", fused), ("matmul_then_route", unfused)):
            for _ in range(20):
                fn()
            s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s_ev.record()
            for _ in range(500):
                fn()
            e_ev.record()
            torch.cuda.synchronize()
            res[name] = s_ev.elapsed_time(e_ev) / 500 * 1e3
        print(json.dumps({"suite": True, "workload": f"router gate + routing T{T} H{H} E{E} k{k}",
                          "us_per_call": res, "launches": {"fused": 1, "matmul_then_route": "2 + casts"}}),
              flush=True)

    # per-tensor FP8 linear (Grok-1 attention projections), four rotating
    # weight copies (> L2)
    for (N, K) in synth.FP8_LINEAR_SHAPES:
        wl, swl = [], []
        for c in range(4):
            w = synth.fp8_linear_inputs(1, N, K, seed=c, device=dev)["w"]
            q, s_ = lib.w4a8_quantize_act(w)
            wl.append(q)
            swl.append(s_)
            del w
        for M in synth.FP8_LINEAR_M:
            x = synth.fp8_linear_inputs(M, N, K, seed=9, device=dev)["x"]
            xq, sx = lib.w4a8_quantize_act(x)
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsp = torch.zeros(lib.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            iters = 400 if M <= 64 else 40
            for i in range(8):
                lib.fp8_linear(xq, sx, wl[i % 4], swl[i % 4], out=y, ws=wsp)
            torch.cuda.synchronize()
            s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_ev.record()
            for i in range(iters):
                lib.fp8_linear(xq, sx, wl[i % 4], swl[i % 4], out=y, ws=wsp)
            e_ev.record()
            torch.cuda.synchronize()
            assert lib.w4a8_device_error(wsp) == 0, "device error word set"
            ms = s_ev.elapsed_time(e_ev) / iters
            nbytes = N * K + M * K + 2 * M * N
            flops = 2.0 * M * N * K
            line = {"suite": True, "workload": f"per-tensor FP8 linear N{N} K{K} M{M}", "ms_per_call": ms,
                    "gbs": nbytes / (ms * 1e-3) / 1e9, "tflops": flops / (ms * 1e-3) / 1e12,
                    "l2": "4 rotating weight copies"}
            if M <= 64:
                line.update({"bound": "hbm", "frac": line["gbs"] / hbm, "peak_gbs": hbm,
                             "peak_source": src + " hbm_gbs"})
            else:
                line.update({"bound": "tensor", "frac": line["tflops"] / fp8_burst, "peak_tflops": fp8_burst,
                             "peak_source": src + " bf16_tflops x 2 (nominal fp8/bf16)"})
            print(json.dumps(line), flush=True)
        del wl, swl
        torch.cuda.empty_cache()

    # block-FP8 linear: four rotating weight copies (> L2) so that every call
    # reads its weights from HBM
    for (N, K) in synth.BLOCK_FP8_SHAPES:
        ws_list, wsi_list = [], []
        for c in range(4):
            w = synth.block_fp8_inputs(1, N, K, seed=c, device=dev)["w"].float()
            blk = w.view(N // 128, 128, K // 128, 128).abs().amax(dim=(1, 3))
            wsi = torch.where(blk > 0, blk / 448.0, torch.ones_like(blk))
            q = (w / wsi.repeat_interleave(128, 0).repeat_interleave(128, 1)).to(torch.float8_e4m3fn)
            ws_list.append(q.view(torch.uint8).contiguous())
            wsi_list.append(wsi.contiguous())
            del w
        for M in synth.BLOCK_FP8_M:
            x = synth.block_fp8_inputs(M, N, K, seed=9, device=dev)["x"]
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            wsp = torch.zeros(lib.fp8_block_linear_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            iters = 400 if M <= 64 else 40
            for i in range(8):
                lib.fp8_block_linear(x, ws_list[i % 4], wsi_list[i % 4], out=y, ws=wsp)
            torch.cuda.synchronize()
            s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_ev.record()
            for i in range(iters):
                lib.fp8_block_linear(x, ws_list[i % 4], wsi_list[i % 4], out=y, ws=wsp)
            e_ev.record()
            torch.cuda.synchronize()
            assert lib.w4a8_device_error(wsp) == 0, "device error word set"
            ms = s_ev.elapsed_time(e_ev) / iters
            nbytes = N * K + 4 * (N // 128) * (K // 128) + 2 * M * K + 2 * M * N
            flops = 2.0 * M * N * K
            line = {"suite": True, "workload": f"block-FP8 linear N{N} K{K} M{M}", "ms_per_call": ms,
                    "gbs": nbytes / (ms * 1e-3) / 1e9, "tflops": flops / (ms * 1e-3) / 1e12,
                    "l2": "4 rotating weight copies"}
            if M <= 64:
                line.update({"bound": "hbm", "frac": line["gbs"] / hbm, "peak_gbs": hbm,
                             "peak_source": src + " hbm_gbs"})
            else:
                line.update({"bound": "tensor", "frac": line["tflops"] / fp8_burst,
                             "peak_tflops": fp8_burst,
                             "peak_source": src + " bf16_tflops x 2 (nominal fp8/bf16)"})
            print(json.dumps(line), flush=True)
        del ws_list, wsi_list
        torch.cuda.empty_cache()


def cpu_baseline(args, shape):
    """The oracle, as it stands, on a bounded sample of the same layer."""
    import numpy as np
    import torch

    import oracle
    from w4a8_moe_gb300 import synth

    # same seeded layer as rank 0 of the GPU arm (drawn on the GPU when there is one)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.moe_inputs(shape.T, shape.H, shape.I, shape.E, bias_std=shape.bias_std, seed=0,
                           device=dev)
    inp = {k_: v.cpu() for k_, v in inp.items()}
    if dev == "cuda":
        torch.cuda.empty_cache()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    pgu, sgu = oracle.quantize_experts(bits(inp["w_gu"]))
    pd, sd = oracle.quantize_experts(bits(inp["w_d"]))
    s1 = oracle.act_scale(bits(inp["x"]))
    xq = oracle.quantize_act(bits(inp["x"]), s1)
    threads = oracle.cores()
    ids, w = oracle.route(inp["logits"].numpy(), shape.k)
    oracle.permute(ids, shape.E)
    s2 = oracle.moe_hidden_scale(xq, s1, pgu, sgu, shape.act, ids, [0], nthreads=threads)
    # size the sample for ~15 s of CPU work: time one token first
    t0 = time.perf_counter()
    oracle.moe_forward(xq, s1, pgu, sgu, pd, sd, s2, shape.act, ids, w, tokens=[0], nthreads=1)
    one = time.perf_counter() - t0
    n = args.cpu_sample_tokens or max(1, min(shape.T, int(15.0 * threads / max(one, 1e-6))))
    toks = list(range(n))
    t0 = time.perf_counter()
    oracle.route(inp["logits"].numpy()[:n], shape.k)
    oracle.moe_forward(xq, s1, pgu, sgu, pd, sd, s2, shape.act, ids, w, tokens=toks, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} of {shape.T} tokens of the {shape.name} layer (route + exact-integer "
                      f"MoE forward), {threads} threads",
            "single_thread": {"value": 1.0 / one, "unit": UNIT,
                              "sample": "token 0 of the same layer (MoE forward), 1 thread"}}


def config_dict(shape, world):
    return {"workload": shape.name, "tokens_per_step": shape.T, "hidden": shape.H,
            "intermediate": shape.I, "experts": shape.E, "top_k": shape.k,
            "activation": "SiLU-gated" if shape.act == 0 else "GELU-tanh-gated",
            "global_batch": shape.T * world, "parallelism": f"replicas{world}",
            "l2": "weights (packed) larger than L2; no flush needed"}


def main():
    args = parse()
    rank, world = dist_setup(args.gpus)
    from w4a8_moe_gb300 import synth
    shape = synth.MOE_SHAPES[args.config]

    if args.impl == "reference":
        if rank == 0:
            cb = cpu_baseline(args, shape)
            line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT,
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": shape.T / cb["value"] * 1e3, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64",
                    "data": "synthetic", "config": config_dict(shape, 1),
                    "cpu_baseline": cb,
                    "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return

    import json as _json  # noqa: F401
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    res = run_ours(args, rank, world)
    if rank != 0:
        return
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    kk = res["kernels"]
    peak_src = "MEASURED_PEAKS.json hbm_gbs (burst copy)" if peaks else "fallback 6.8 TB/s"
    traffic_unit = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
    on_bench_layer = args.config == "mixtral_decode"
    if kk["one_launch"]:
        # gate_up and down in one persistent launch: the roofline is that launch's
        w_bytes = kk["gate_up_bytes"] + kk["down_bytes"]
        gbs = w_bytes / (kk["gate_up_ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "moe_gemm_kernel<gate_up+down, one launch>", "achieved": gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak, "peak_source": peak_src,
                "traffic": ncu_traffic("one_launch") if on_bench_layer else None, "traffic_unit": traffic_unit,
                "per_launch_ms": kk["gate_up_ms"], "algorithmic_bytes": w_bytes,
                "step_breakdown_ms": {"gate_up+down": kk["gate_up_ms"], "finalize": kk["finalize_ms"],
                                      "rest_net_of_overlap": kk["route_gather_gaps_ms"] + kk["down_ms"]}}
    else:
        gu_gbs = kk["gate_up_bytes"] / (kk["gate_up_ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "moe_gemm_kernel<gate_up>", "achieved": gu_gbs,
                "peak": hbm_peak, "unit": "GB/s", "frac": gu_gbs / hbm_peak, "peak_source": peak_src,
                "traffic": None, "traffic_unit": traffic_unit,
                "per_launch_ms": kk["gate_up_ms"], "algorithmic_bytes": kk["gate_up_bytes"],
                "down": {"per_launch_ms": kk["down_ms"], "algorithmic_bytes": kk["down_bytes"],
                         "achieved": kk["down_bytes"] / (kk["down_ms"] * 1e-3) / 1e9},
                "step_breakdown_ms": {"gate_up": kk["gate_up_ms"], "down": kk["down_ms"],
                                      "finalize": kk["finalize_ms"],
                                      "rest_net_of_overlap": kk["route_gather_gaps_ms"]}}
    layer_bytes = kk["gate_up_bytes"] + kk["down_bytes"] + kk["act_bytes"]
    line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xint4->f32",
            "data": "synthetic", "config": config_dict(shape, world),
            "layer_weight_gbs": layer_bytes / (res["ms_per_step"] * 1e-3) / 1e9,
            "layer_hbm_frac": layer_bytes / (res["ms_per_step"] * 1e-3) / 1e9 / hbm_peak,
            "roofline": roof, "e2e": res["e2e"], "clocks": res["clocks"],
            # moe_route plus the forward's launches (gather, GEMM launch(es), combine)
            "gpu_launches": (1 + res["plan"]["launches"]) * args.steps,
            "plan": res["plan"],
            "act_quant_static_ms": res["act_quant_static_ms"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, shape)
    print(json.dumps(line), flush=True)
    if args.suite and world == 1:
        run_suite(args)


if __name__ == "__main__":
    main()
